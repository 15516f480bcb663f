"""GPU parity: the CUDA library through its C ABI against the fp64 oracle.

Every case draws seeded synthetic inputs, runs ``dflash_block_attn`` on the
GPU and the oracle on the host, and checks the bar in ``_gpu_cases``.
"""

import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_draft_paged_gb300 as dflash
from speculative_decoding_draft_paged_gb300 import workloads as W
from tests._gpu_cases import (assert_parity, check_case, compact_requests, metrics, run_lib,
                              run_oracle)

pytestmark = pytest.mark.gpu


def test_tiny_config(cuda_device):
    m, _, _ = check_case(W.tiny(), cuda_device)
    assert m["rel_l2"] < 5e-3


@pytest.mark.parametrize("K", [1, 3, 7])
@pytest.mark.parametrize("L", [100, 2048, 5000, 9000])
def test_minimax_shape(cuda_device, K, L):
    check_case(W.minimax(B=3, K=K, ctx_lens=[L, max(0, L - 77), L // 2 + 5]), cuda_device)


@pytest.mark.parametrize("K", [3, 7])
@pytest.mark.parametrize("L", [3000, 8200])
def test_adp_shape_with_outliers(cuda_device, K, L):
    check_case(W.adp(B=2, K=K, ctx_lens=[L, L - 1000]), cuda_device)


@pytest.mark.parametrize("Hq", [8, 12])
@pytest.mark.parametrize("L", [5000, 20000])
def test_longctx_shape(cuda_device, Hq, L):
    check_case(W.longctx(B=2, L=L, Hq=Hq), cuda_device)


def test_ragged_shape(cuda_device):
    spec = W.ragged(B=5, lo=1, hi=20000)
    check_case(spec, cuda_device)


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
@pytest.mark.parametrize("D,P", [(64, 16), (64, 32), (128, 64), (128, 16)])
@pytest.mark.parametrize("window,fk", [(0, 1), (0, 0), (300, 1), (300, 0)])
def test_edge_lengths(cuda_device, D, P, window, fk, path):
    K = 5
    lens = [0, 1, P - 1, P, P + 1, 2 * P - K, 2 * P - K + 1, 63, 64, 65, 127, 128]
    if window:
        lens += [window - 1, window, window + K, window + P + 3]
    spec = W.CaseSpec(f"edges_D{D}_P{P}_W{window}_fk{fk}", B=len(lens), Hq=8, Hkv=2, D=D, K=K, P=P,
                      window=window, future_keys=fk, ctx_lens=lens, seed=77, poison=True,
                      extra_pages=3, extra_table_slots=2)
    check_case(spec, cuda_device, force_path=path)


@pytest.mark.parametrize("G,K", [(1, 1), (4, 3), (4, 7), (13, 5), (6, 11)])
@pytest.mark.parametrize("D", [64, 128])
def test_tcgen05_small_row_counts(cuda_device, G, K, D):
    """The tcgen05 tile with most of its 128 rows padding."""
    spec = W.CaseSpec(f"tc_rows_G{G}_K{K}_D{D}", B=2, Hq=2 * G, Hkv=2, D=D, K=K, P=32, window=0,
                      future_keys=1, ctx_lens=[900, 61], seed=6, poison=True)
    check_case(spec, cuda_device, force_path=dflash.PATH_TCGEN05)


def test_paths_agree(cuda_device):
    """Both split kernels against the oracle and against each other."""
    spec = W.minimax(B=2, K=7, ctx_lens=[6000, 2500])
    _, o1, l1 = check_case(spec, cuda_device, force_path=dflash.PATH_MMA)
    _, o2, l2 = check_case(spec, cuda_device, force_path=dflash.PATH_TCGEN05)
    d = (o1.double() - o2.double()).abs().max().item()
    assert d <= 2 * 2.0 ** -7 * max(1.0, o1.double().abs().max().item())
    assert (l1 - l2).abs().max().item() < 1e-3


@pytest.mark.parametrize("n_tiles", [1, 3, 0])
def test_mma_two_ctas_per_sm(cuda_device, n_tiles):
    """The mma.sync kernel's two-CTAs-per-SM form (a plan of more than one
    wave at 8/2 heads, D = 64): boundary lengths, poisoned slots, forced and
    planned unit lengths."""
    lens = [0, 1, 6, 7, 31, 32, 33, 127, 128, 129, 255, 256, 1000, 2047, 2048, 2049, 3001, 4095, 4096, 4097,
            4500, 4999, 5000, 321]
    spec = W.CaseSpec(f"two_ctas_{n_tiles}", B=len(lens), Hq=8, Hkv=2, D=64, K=7, P=32, window=0,
                      future_keys=1, ctx_lens=lens, seed=91, poison=True, extra_pages=3, extra_table_slots=2)
    p = dflash.make_params(batch=spec.B, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=32,
                           max_pages_per_req=(spec.max_ctx_len + spec.K + 31) // 32 + 2,
                           num_pages=spec.B * 200, block_size=7, window=0, future_keys=1, scale=0.125,
                           max_ctx_len=spec.max_ctx_len, force_split_tiles=n_tiles)
    if n_tiles:
        assert dflash.plan(p)["ctas_per_sm"] == 2
    check_case(spec, cuda_device, force_path=dflash.PATH_MMA, force_split_tiles=n_tiles)


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 4, 5, 9])
def test_tcgen05_unit_tile_counts(cuda_device, n_tiles):
    """Units of 1..9 tiles: both softmax groups, one of them empty, uneven."""
    spec = W.minimax(B=2, K=7, ctx_lens=[3000, 700])
    check_case(spec, cuda_device, force_path=dflash.PATH_TCGEN05, force_split_tiles=n_tiles)


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
@pytest.mark.parametrize("win,r", [(0, 0), (0, 2), (0, 6), (300, 3), (3, 0), (3, 2), (1, 0), (5, 6)])
def test_right_window(cuda_device, path, win, r):
    """A right window r (row i sees block keys up to i+r) and windows shorter
    than the block, on both kernels."""
    lens = [0, 1, 6, 63, 64, 65, 700, 2049]
    spec = W.CaseSpec(f"rw_W{win}_r{r}", B=len(lens), Hq=16, Hkv=1, D=128, K=7, P=64, window=win,
                      future_keys=0, right_window=r, ctx_lens=lens, seed=41, poison=True)
    check_case(spec, cuda_device, force_path=path)


@pytest.mark.parametrize("win,r", [(0, 1), (2, 4)])
def test_right_window_d64(cuda_device, win, r):
    lens = [0, 3, 31, 32, 33, 1000]
    spec = W.CaseSpec(f"rw64_W{win}_r{r}", B=len(lens), Hq=8, Hkv=2, D=64, K=5, P=32, window=win,
                      future_keys=0, right_window=r, ctx_lens=lens, seed=42, poison=True)
    check_case(spec, cuda_device)


@pytest.mark.parametrize("kind", ["many_short", "one_long", "max_batch"])
def test_tcgen05_flat_split_batches(cuda_device, kind):
    """The flat split over many pairs: ranges holding many whole pairs
    (direct outputs), one long pair cut over many CTAs among short ones, and
    the largest batch the tcgen05 kernel takes."""
    rng = np.random.default_rng({"many_short": 21, "one_long": 22, "max_batch": 23}[kind])
    if kind == "many_short":
        lens = [int(x) for x in rng.integers(0, 300, size=200)]
        window = 0
    elif kind == "one_long":
        lens = [12000] + [int(x) for x in rng.integers(0, 200, size=39)]
        window = 4096
    else:
        lens = [int(x) for x in rng.integers(0, 64, size=768)]
        window = 0
    spec = W.CaseSpec(f"tc_flat_{kind}", B=len(lens), Hq=16, Hkv=1, D=128, K=7, P=64, window=window,
                      future_keys=1, ctx_lens=lens, seed=31, poison=True)
    check_case(spec, cuda_device, force_path=dflash.PATH_TCGEN05)


@pytest.mark.parametrize("G,K", [(1, 1), (4, 3), (16, 1), (3, 5), (4, 7), (6, 7), (16, 3), (5, 13),
                                 (16, 7), (8, 16)])
@pytest.mark.parametrize("D", [64, 128])
def test_packed_row_counts(cuda_device, G, K, D):
    spec = W.CaseSpec(f"rows_G{G}_K{K}_D{D}", B=2, Hq=2 * G, Hkv=2, D=D, K=K, P=32, window=0,
                      future_keys=1, ctx_lens=[700, 261], seed=5)
    check_case(spec, cuda_device)


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
def test_forced_path_and_tiny_splits(cuda_device, path):
    """force_split_tiles=1 gives one tile per unit: many empty units for the
    short requests of a ragged batch, and the combine over many partials."""
    spec = W.CaseSpec("empty_splits", B=4, Hq=8, Hkv=2, D=64, K=7, P=32, window=0, future_keys=1,
                      ctx_lens=[3000, 0, 130, 1000], seed=9, poison=True)
    m1, o1, l1 = check_case(spec, cuda_device, force_path=path, force_split_tiles=1)
    m2, o2, l2 = check_case(spec, cuda_device, force_path=path, force_split_tiles=5)
    assert m1["rel_l2"] < 5e-3 and m2["rel_l2"] < 5e-3


@pytest.mark.parametrize("D,L", [(64, 9000), (128, 5000), (128, 1500), (64, 2041)])
@pytest.mark.parametrize("window", [0, 1000])
def test_combine_many_partials(cuda_device, D, L, window):
    """One tile per unit on the mma.sync path: 16 (L = 2041 at D = 64) to 141
    partials per pair for the combine kernel, with partials that see no key
    (LSE -inf) under the window."""
    spec = W.CaseSpec(f"many_partials_D{D}", B=3, Hq=8, Hkv=2, D=D, K=7, P=32, window=window,
                      future_keys=1, ctx_lens=[L, 200, L // 3], seed=13, poison=True)
    check_case(spec, cuda_device, force_path=dflash.PATH_MMA, force_split_tiles=1)


@pytest.mark.parametrize("window", [0, 1000])
def test_page_permutation_bitwise(cuda_device, window):
    spec = W.CaseSpec("perm", B=3, Hq=16, Hkv=2, D=64, K=7, P=32, window=window, future_keys=1,
                      ctx_lens=[2500, 777, 4000], seed=11, extra_pages=5)
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    out1, lse1 = run_lib(spec, inp)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(spec.num_pages, generator=g).to(cuda_device)
    kp = torch.empty_like(inp["k_pages"])
    vp = torch.empty_like(inp["v_pages"])
    kp[perm] = inp["k_pages"]
    vp[perm] = inp["v_pages"]
    tab = inp["page_table"].clone()
    m = tab >= 0
    tab[m] = perm[tab[m].long()].to(torch.int32)
    inp2 = dict(inp, k_pages=kp, v_pages=vp, page_table=tab)
    out2, lse2 = run_lib(spec, inp2)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    assert torch.equal(lse1, lse2)


def test_deterministic(cuda_device):
    spec = W.longctx(B=2, L=9000, Hq=12)
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    a = run_lib(spec, inp)
    b = run_lib(spec, inp)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
def test_guard_bands_untouched(cuda_device, path):
    """No byte before or after out, lse2 or the workspace is written, on
    either path (the tcgen05 path's TMA stores included)."""
    spec = W.CaseSpec("guards", B=3, Hq=16, Hkv=2, D=128, K=7, P=64, window=0, future_keys=1,
                      ctx_lens=[1500, 64, 3333], seed=12)
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=spec.K,
                          window=0, future_keys=1, scale=spec.softmax_scale,
                          max_ctx_len=spec.max_ctx_len, force_path=path)
    ws_bytes = dflash.workspace_size(p)
    G = 4096
    out_buf = torch.full((G + inp["q"].numel() * 2 + G,), 0xA5, dtype=torch.uint8, device=cuda_device)
    lse_buf = torch.full((G + spec.B * spec.K * spec.Hq * 4 + G,), 0x5A, dtype=torch.uint8,
                         device=cuda_device)
    ws_buf = torch.full((G + ws_bytes + G,), 0x3C, dtype=torch.uint8, device=cuda_device)
    ws_buf[G:G + 4] = 0
    rc = dflash.block_attn_raw(p, inp["q"].data_ptr(), inp["k_pages"].data_ptr(),
                               inp["v_pages"].data_ptr(), inp["page_table"].data_ptr(),
                               inp["ctx_lens"].data_ptr(), out_buf.data_ptr() + G,
                               lse_buf.data_ptr() + G, ws_buf.data_ptr() + G, ws_bytes,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == dflash.DFLASH_OK
    torch.cuda.synchronize()
    for buf, val, n in ((out_buf, 0xA5, inp["q"].numel() * 2), (lse_buf, 0x5A, spec.B * spec.K * spec.Hq * 4),
                        (ws_buf, 0x3C, ws_bytes)):
        assert bool((buf[:G] == val).all()), "guard band before the buffer was written"
        assert bool((buf[G + n:] == val).all()), "guard band after the buffer was written"
    out = out_buf[G:G + inp["q"].numel() * 2].view(torch.bfloat16).view(inp["q"].shape)
    lse = lse_buf[G:G + spec.B * spec.K * spec.Hq * 4].view(torch.float32).view(spec.B, spec.K, spec.Hq)
    ro, rl = run_oracle(spec, {k: v.cpu() for k, v in inp.items()})
    assert_parity(metrics(out, lse, ro, rl), "guards")


def test_workspace_too_small_refused(cuda_device):
    spec = W.tiny()
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=3, window=0,
                          future_keys=1, scale=spec.softmax_scale, max_ctx_len=100)
    need = dflash.workspace_size(p)
    ws = torch.zeros(need, dtype=torch.uint8, device=cuda_device)
    out = torch.full_like(inp["q"], 7.0)
    lse = torch.full((1, 3, 4), 7.0, device=cuda_device)
    rc = dflash.block_attn_raw(p, inp["q"].data_ptr(), inp["k_pages"].data_ptr(),
                               inp["v_pages"].data_ptr(), inp["page_table"].data_ptr(),
                               inp["ctx_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
                               ws.data_ptr(), need - 256, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == dflash.DFLASH_ERR_WORKSPACE
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())


def test_bad_device_data_flags_status_without_fault(cuda_device):
    spec = W.CaseSpec("baddata", B=3, Hq=8, Hkv=2, D=64, K=3, P=32, window=0, future_keys=1,
                      ctx_lens=[500, 300, 900], seed=13)
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=3, window=0,
                          future_keys=1, scale=spec.softmax_scale, max_ctx_len=900)
    ws = torch.zeros(dflash.workspace_size(p), dtype=torch.uint8, device=cuda_device)
    run_lib(spec, inp, workspace=ws)
    assert dflash.read_device_status(ws) == 0
    bad = dict(inp)
    bad["page_table"] = inp["page_table"].clone()
    bad["page_table"][1, 2] = spec.num_pages + 1000
    bad["page_table"][2, 0] = -7
    out, lse = run_lib(spec, bad, workspace=ws)
    st = dflash.read_device_status(ws)
    assert st & dflash.DFLASH_STATUS_BAD_PAGE
    assert not (st & dflash.DFLASH_STATUS_TIMEOUT)
    assert not torch.isnan(out[0].float()).any()
    dflash.clear_device_status(ws)
    assert dflash.read_device_status(ws) == 0
    bad2 = dict(inp, ctx_lens=torch.tensor([500, 5000, -4], dtype=torch.int32, device=cuda_device))
    run_lib(spec, bad2, workspace=ws)
    st = dflash.read_device_status(ws)
    assert st & dflash.DFLASH_STATUS_BAD_CTX_LEN
    assert not (st & dflash.DFLASH_STATUS_TIMEOUT)
    torch.cuda.synchronize()
    # Request 0 was untouched by the bad data of the others.
    ro, rl = run_oracle(spec, {k: v.cpu() for k, v in inp.items()}, req_ids=np.array([0], np.int32))
    assert_parity(metrics(out[:1], lse[:1], ro, rl), "bad-data neighbour")


def test_cuda_graph_replay_with_new_lengths(cuda_device):
    # Tables cover 5000 context tokens for every request; the lengths change
    # between replays of one captured graph.
    spec = W.CaseSpec("graph", B=4, Hq=16, Hkv=2, D=64, K=7, P=32, window=2048, future_keys=1,
                      ctx_lens=[5000] * 4, seed=14)
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    inp["ctx_lens"].copy_(torch.tensor([5000, 4000, 3000, 100], dtype=torch.int32))
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=7, window=2048,
                          future_keys=1, scale=spec.softmax_scale, max_ctx_len=5000)
    ws = torch.zeros(dflash.workspace_size(p), dtype=torch.uint8, device=cuda_device)
    out = torch.empty_like(inp["q"])
    lse = torch.empty(inp["q"].shape[:3], dtype=torch.float32, device=cuda_device)
    lens = inp["ctx_lens"]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_lib(spec, inp, out=out, lse2=lse, workspace=ws)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_lib(spec, inp, out=out, lse2=lse, workspace=ws)
    for new in ([5000, 4000, 3000, 100], [17, 4999, 2048, 0], [3333, 64, 4567, 2047]):
        lens.copy_(torch.tensor(new, dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ro, rl = run_oracle(spec, {k: v.cpu() for k, v in inp.items()}, ctx_lens=np.array(new, np.int32))
        assert_parity(metrics(out, lse, ro, rl), f"graph replay {new}")


def test_mma_unit_grid_large_batch(cuda_device):
    """800 short requests, more than the tcgen05 flat split takes: the
    mma.sync unit grid (one CTA per (request, kv head, split))."""
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(0, 700, size=800)]
    spec = W.CaseSpec("mma_grid_B800", B=len(lens), Hq=8, Hkv=2, D=64, K=7, P=32, window=0, future_keys=1,
                      ctx_lens=lens, seed=13, poison=True)
    p = dflash.make_params(batch=spec.B, num_q_heads=spec.Hq, num_kv_heads=spec.Hkv, head_dim=spec.D,
                           page_size=spec.P, max_pages_per_req=spec.max_pages, num_pages=spec.num_pages,
                           block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
                           scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len)
    pl = dflash.plan(p)
    assert pl["path"] == dflash.PATH_MMA and pl["flat"] == 0
    check_case(spec, cuda_device)


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
def test_bounded_wait_runs_out_and_device_recovers(cuda_device, path):
    """The failure path: with the producers withholding every K/V load
    (DFLASH_TEST_WITHHOLD_LOADS) each pipeline wait runs out after its bound,
    the call finishes with DFLASH_STATUS_TIMEOUT set and nothing in flight,
    and the next normal call on the same device is parity-green."""
    import time

    spec = W.minimax(B=2, K=7, ctx_lens=[3000, 700])
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=spec.K, window=spec.window,
                          future_keys=spec.future_keys, scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len,
                          force_path=path)
    ws = torch.zeros(dflash.workspace_size(p), dtype=torch.uint8, device=cuda_device)
    t0 = time.perf_counter()
    run_lib(spec, inp, force_path=path, workspace=ws, test_flags=dflash.DFLASH_TEST_WITHHOLD_LOADS)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    st = dflash.read_device_status(ws)
    assert st & dflash.DFLASH_STATUS_TIMEOUT, st
    assert waited < 60.0
    # The context is usable and the same workspace serves a correct call.
    dflash.clear_device_status(ws)
    out, lse = run_lib(spec, inp, force_path=path, workspace=ws)
    torch.cuda.synchronize()
    assert dflash.read_device_status(ws) == 0
    host = {k: v.cpu() for k, v in inp.items()}
    ro, rl = run_oracle(spec, host)
    assert_parity(metrics(out, lse, ro, rl), f"after the timeout, path {path}")
