"""GPU parity of the block placement, the K/V append and the fused
append + attention, through the C ABI, against the oracle.

Placement and append are integer and byte work: the bar is bit-exact.  The
fused call's attention output meets the same bar as ``dflash_block_attn``.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_paged_gb300 as dflash
from speculative_decoding_draft_paged_gb300 import workloads as W
from tests._gpu_cases import assert_parity, metrics, run_oracle, to_bits

pytestmark = pytest.mark.gpu

NAN = 0x7FC0


def _block_rows(spec, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (spec.B, spec.K, spec.Hkv, spec.D)
    kb = torch.randn(shape, generator=g).to(torch.bfloat16)
    vb = torch.randn(shape, generator=g).to(torch.bfloat16)
    return kb, vb


def _stale_block_slots(inp, placement, value_bits=NAN):
    """Overwrite the block's slots in the (device) pools, as a recycled page would."""
    pl = torch.as_tensor(placement, device=inp["k_pages"].device).long()
    fill = torch.tensor(value_bits, dtype=torch.int16).view(torch.bfloat16).item()
    for b in range(pl.shape[0]):
        for j in range(pl.shape[1]):
            inp["k_pages"][pl[b, j, 0], :, pl[b, j, 1], :] = fill
            inp["v_pages"][pl[b, j, 0], :, pl[b, j, 1], :] = fill


def _spec(name, lens, **kw):
    args = dict(B=len(lens), Hq=8, Hkv=2, D=64, K=5, P=16, window=0, future_keys=1, ctx_lens=lens,
                seed=61, poison=True, extra_pages=2)
    args.update(kw)
    return W.CaseSpec(name, **args)


@pytest.mark.parametrize("P", [16, 32, 64])
def test_block_placement_bitexact(cuda_device, P):
    lens = [0, 1, P - 3, P - 1, P, 2 * P + 7, 700]
    spec = _spec(f"place_P{P}", lens, P=P)
    inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    got = dflash.block_placement(inp["page_table"], inp["ctx_lens"], inp["k_pages"],
                                 block_size=spec.K, max_ctx_len=spec.max_ctx_len, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.block_placement(inp["page_table"].cpu().numpy(), np.asarray(lens, np.int32),
                                 block_size=spec.K, page_size=P, num_pages=spec.num_pages)
    np.testing.assert_array_equal(got.cpu().numpy(), ref)
    assert dflash.read_device_status(ws) == 0


@pytest.mark.parametrize("D,P,Hkv", [(64, 16, 2), (128, 64, 1), (128, 32, 4)])
def test_append_bitexact(cuda_device, D, P, Hkv):
    lens = [0, 3, P - 2, 2 * P - 5, 333]
    spec = _spec(f"append_D{D}_P{P}", lens, D=D, P=P, Hkv=Hkv, Hq=4 * Hkv, K=7)
    cpu = W.make_inputs(spec, "cpu")
    kb, vb = _block_rows(spec, 5)
    ref_k, ref_v = oracle.append_block_kv(to_bits(kb), to_bits(vb), to_bits(cpu["k_pages"]),
                                          to_bits(cpu["v_pages"]), cpu["page_table"].numpy(),
                                          np.asarray(lens, np.int32))
    inp = {k: v.to(cuda_device) for k, v in cpu.items()}
    dflash.append_block_kv(kb.to(cuda_device), vb.to(cuda_device), inp["k_pages"], inp["v_pages"],
                           inp["page_table"], inp["ctx_lens"], max_ctx_len=spec.max_ctx_len)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(inp["k_pages"]), ref_k)
    np.testing.assert_array_equal(to_bits(inp["v_pages"]), ref_v)


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
@pytest.mark.parametrize("shape", ["gqa8", "minimax"])
def test_fused_append_then_attention(cuda_device, path, shape):
    """The block's slots hold NaN (a recycled page) before the call; the fused
    call writes them and attends over the result."""
    if shape == "gqa8":
        spec = _spec("fused_gqa8", [0, 5, 16, 31, 700, 2000], Hq=16, Hkv=2, K=7, P=32)
    else:
        spec = W.minimax(B=3, K=7, ctx_lens=[5000, 64, 0])
    cpu = W.make_inputs(spec, "cpu")
    kb, vb = _block_rows(spec, 9)
    lens = np.asarray(spec.ctx_lens, np.int32)
    place = oracle.block_placement(cpu["page_table"].numpy(), lens, block_size=spec.K,
                                   page_size=spec.P, num_pages=spec.num_pages)
    inp = {k: v.to(cuda_device) for k, v in cpu.items()}
    _stale_block_slots(inp, place)
    ref_k, ref_v = oracle.append_block_kv(to_bits(kb), to_bits(vb), to_bits(inp["k_pages"]),
                                          to_bits(inp["v_pages"]), cpu["page_table"].numpy(), lens)
    out, lse = dflash.block_attn_append(inp["q"], kb.to(cuda_device), vb.to(cuda_device),
                                        inp["k_pages"], inp["v_pages"], inp["page_table"],
                                        inp["ctx_lens"], block_size=spec.K, window=spec.window,
                                        future_keys=spec.future_keys, scale=spec.softmax_scale,
                                        max_ctx_len=spec.max_ctx_len, force_path=path)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(inp["k_pages"]), ref_k)
    np.testing.assert_array_equal(to_bits(inp["v_pages"]), ref_v)
    ref_inp = dict(cpu)
    ref_inp["k_pages"] = torch.from_numpy(ref_k.view(np.int16)).view(torch.bfloat16)
    ref_inp["v_pages"] = torch.from_numpy(ref_v.view(np.int16)).view(torch.bfloat16)
    ro, rl = run_oracle(spec, ref_inp)
    assert_parity(metrics(out, lse, ro, rl), spec.name)


def test_bad_block_page_is_flagged_and_skipped(cuda_device):
    lens = [10, 40]
    spec = _spec("bad_block_page", lens, K=5, P=16)
    cpu = W.make_inputs(spec, "cpu")
    tab = cpu["page_table"].clone()
    slot = (lens[1] + 2) // spec.P            # the slot of block token 2 of request 1
    tab[1, slot] = spec.num_pages + 5
    inp = {k: v.to(cuda_device) for k, v in cpu.items()}
    inp["page_table"] = tab.to(cuda_device)
    kb, vb = _block_rows(spec, 3)
    before_k = to_bits(inp["k_pages"]).copy()
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    dflash.append_block_kv(kb.to(cuda_device), vb.to(cuda_device), inp["k_pages"], inp["v_pages"],
                           inp["page_table"], inp["ctx_lens"], max_ctx_len=spec.max_ctx_len,
                           workspace=ws)
    torch.cuda.synchronize()
    assert dflash.read_device_status(ws) & dflash.DFLASH_STATUS_BAD_PAGE
    # Request 0 was written in full.
    place = oracle.block_placement(cpu["page_table"].numpy(), np.asarray(lens, np.int32),
                                   block_size=spec.K, page_size=spec.P, num_pages=spec.num_pages)
    after_k = to_bits(inp["k_pages"])
    kbits = to_bits(kb)
    for j in range(spec.K):
        np.testing.assert_array_equal(after_k[place[0, j, 0], :, place[0, j, 1]], kbits[0, j])
    # Nothing outside the block slots changed.
    mask = np.ones(after_k.shape[:3], bool)
    for b in range(2):
        for j in range(spec.K):
            mask[place[b, j, 0], :, place[b, j, 1]] = False
    np.testing.assert_array_equal(after_k[mask], before_k[mask])


# ----------------------------------------------------------------------------
# Dense-suffix form: block rows from dense tensors, context from the pages
# ----------------------------------------------------------------------------

def _dense_suffix_case(spec, device, seed):
    """Inputs whose pages hold the context only: the block's slots are NaN and
    every table entry past the context's last page names no page."""
    cpu = W.make_inputs(spec, "cpu")
    kb, vb = _block_rows(spec, seed)
    lens = np.asarray(spec.ctx_lens, np.int32)
    place = oracle.block_placement(cpu["page_table"].numpy(), lens, block_size=spec.K,
                                   page_size=spec.P, num_pages=spec.num_pages)
    inp = {k: v.to(device) for k, v in cpu.items()}
    _stale_block_slots(inp, place)
    tab = inp["page_table"].cpu()
    for b, L in enumerate(spec.ctx_lens):
        first_unused = (L + spec.P - 1) // spec.P
        tab[b, first_unused:] = spec.num_pages + 1000
    inp["page_table"] = tab.to(device)
    return inp, kb, vb


@pytest.mark.parametrize("path", [dflash.PATH_MMA, dflash.PATH_TCGEN05])
@pytest.mark.parametrize("shape,win,fk,r,split", [
    ("gqa8", 0, 1, 0, 0), ("gqa8", 300, 1, 0, 0), ("gqa8", 3, 0, 2, 0),
    ("minimax", 4096, 1, 0, 0), ("minimax", 0, 0, 0, 0), ("minimax", 0, 1, 0, 1),
    ("minimax", 2, 0, 4, 3), ("gqa4", 0, 1, 0, 1),
])
def test_dense_suffix(cuda_device, path, shape, win, fk, r, split):
    if shape in ("gqa8", "gqa4"):
        # gqa4 with one-tile units: a plan of more than one wave, which the
        # mma.sync kernel runs two CTAs per SM.
        spec = _spec(f"dense_{shape}", [0, 5, 25, 32, 33, 700, 2000], Hq=16 if shape == "gqa8" else 8,
                     Hkv=2, K=7, P=32, window=win, future_keys=fk, right_window=r)
    else:
        spec = W.CaseSpec("dense_minimax", B=4, Hq=16, Hkv=1, D=128, K=7, P=64, window=win,
                          future_keys=fk, right_window=r, ctx_lens=[5000, 64, 0, 121], seed=71,
                          poison=True)
    inp, kb, vb = _dense_suffix_case(spec, cuda_device, 13)
    ws_bytes = dflash.workspace_size(dflash.params_for(
        inp["q"], inp["k_pages"], inp["page_table"], block_size=spec.K, window=spec.window,
        future_keys=spec.future_keys, scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len,
        force_path=path, force_split_tiles=split, right_window=spec.right_window))
    if shape == "gqa4" and path == dflash.PATH_MMA:
        assert dflash.plan(dflash.params_for(
            inp["q"], inp["k_pages"], inp["page_table"], block_size=spec.K, window=spec.window,
            future_keys=spec.future_keys, scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len,
            force_path=path, force_split_tiles=split, right_window=spec.right_window))["ctas_per_sm"] == 2
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda_device)
    out, lse = dflash.block_attn_dense_suffix(
        inp["q"], kb.to(cuda_device), vb.to(cuda_device), inp["k_pages"], inp["v_pages"],
        inp["page_table"], inp["ctx_lens"], block_size=spec.K, window=spec.window,
        future_keys=spec.future_keys, scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len,
        force_path=path, force_split_tiles=split, right_window=spec.right_window, workspace=ws)
    torch.cuda.synchronize()
    assert dflash.read_device_status(ws) == 0, "a page-table slot past the context was read"
    ro, rl = oracle.block_attn(to_bits(inp["q"]), to_bits(inp["k_pages"]), to_bits(inp["v_pages"]),
                               inp["page_table"].cpu().numpy(), np.asarray(spec.ctx_lens, np.int32),
                               block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
                               right_window=spec.right_window, scale=spec.softmax_scale,
                               k_block=to_bits(kb), v_block=to_bits(vb))
    assert_parity(metrics(out, lse, ro, rl), spec.name)
