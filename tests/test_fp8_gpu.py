"""GPU parity of the fp8-context form (dense suffix over E4M3 context pages)
through the C ABI, against the oracle's fp8 reading of the same codes.

The pools hold E4M3 codes of the seeded normal samples (torch's float8 cast
of the bf16 draws; every slot no visible key uses holds the NaN code), the
block rows are bf16 from their own seed, and the per-tensor scales are not
powers of two.  The bar is the one of ``dflash_block_attn`` (the widening to
bf16 is exact; only the fp32 scale products round differently), with the
absolute bound scaled by v_scale when the values are larger than unit
variance.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_paged_gb300 as dflash
from speculative_decoding_draft_paged_gb300 import workloads as W
from tests._gpu_cases import assert_parity, metrics, to_bits

pytestmark = pytest.mark.gpu

NAN_CODE = 0x7F


def _fp8_case(spec, device, seed):
    """(q, k_block, v_block, k_pages8, v_pages8, page_table) on `device`: the
    pages hold the context only (block slots hold the NaN code, table entries
    past the context's last page name no page)."""
    cpu = W.make_inputs(spec, "cpu")
    g = torch.Generator().manual_seed(seed)
    shape = (spec.B, spec.K, spec.Hkv, spec.D)
    kb = torch.randn(shape, generator=g).to(torch.bfloat16)
    vb = torch.randn(shape, generator=g).to(torch.bfloat16)
    kp8 = cpu["k_pages"].float().to(torch.float8_e4m3fn).view(torch.uint8)
    vp8 = cpu["v_pages"].float().to(torch.float8_e4m3fn).view(torch.uint8)
    tab = cpu["page_table"].clone()
    for b, L in enumerate(spec.ctx_lens):
        for p in range(L, L + spec.K):
            pg = int(tab[b, p // spec.P])
            if pg >= 0:
                kp8[pg, :, p % spec.P] = NAN_CODE
                vp8[pg, :, p % spec.P] = NAN_CODE
        tab[b, (L + spec.P - 1) // spec.P:] = spec.num_pages + 1000
    dev = {"q": cpu["q"].to(device), "kb": kb.to(device), "vb": vb.to(device), "kp8": kp8.to(device),
           "vp8": vp8.to(device), "tab": tab.to(device), "lens": cpu["ctx_lens"].to(device)}
    return dev


def _run(spec, device, k_scale, v_scale, path, split=0, seed=17, mutate=None):
    """(out, lse, device status, inputs) of one fp8-context call on `path`."""
    d = _fp8_case(spec, device, seed)
    if mutate is not None:
        mutate(d)
    p = dflash.params_for(d["q"], d["kp8"], d["tab"], block_size=spec.K, window=spec.window,
                          future_keys=spec.future_keys, scale=spec.softmax_scale,
                          max_ctx_len=spec.max_ctx_len, force_path=path, force_split_tiles=split,
                          right_window=spec.right_window, kv_dtype=dflash.KV_FP8_E4M3)
    if dflash.workspace_size(p) == 0:
        pytest.skip("no such plan (the mma.sync code ring would not fit)")
    assert dflash.plan(p)["path"] == path
    ws = torch.zeros(dflash.workspace_size(p), dtype=torch.uint8, device=device)
    out, lse = dflash.block_attn_fp8_context(
        d["q"], d["kb"], d["vb"], d["kp8"], d["vp8"], d["tab"], d["lens"], k_scale=k_scale,
        v_scale=v_scale, block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
        scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len, force_path=path,
        force_split_tiles=split, right_window=spec.right_window, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, dflash.read_device_status(ws), d


def _oracle_check(spec, d, out, lse, k_scale, v_scale):
    ro, rl = oracle.block_attn_fp8(
        to_bits(d["q"]), d["kp8"].cpu().numpy(), d["vp8"].cpu().numpy(), d["tab"].cpu().numpy(),
        np.asarray(spec.ctx_lens, np.int32), k_scale=k_scale, v_scale=v_scale, k_block=to_bits(d["kb"]),
        v_block=to_bits(d["vb"]), block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
        right_window=spec.right_window, scale=spec.softmax_scale)
    assert_parity(metrics(out, lse, ro, rl), spec.name, value_scale=v_scale)


def _check(spec, device, k_scale, v_scale, path, split=0, seed=17):
    out, lse, status, d = _run(spec, device, k_scale, v_scale, path, split, seed)
    assert status == 0, "a page-table slot past the context was read"
    _oracle_check(spec, d, out, lse, k_scale, v_scale)


def _minimax(win=0, fk=1, r=0, lens=(5000, 64, 0, 121, 63, 65)):
    return W.CaseSpec("fp8_minimax", B=len(lens), Hq=16, Hkv=1, D=128, K=7, P=64, window=win,
                      future_keys=fk, right_window=r, ctx_lens=list(lens), seed=81, poison=True)


def _gqa(D, P, K, Hq, Hkv, win=0, fk=1, r=0, lens=(0, 5, 25, 32, 33, 700, 2000)):
    return W.CaseSpec(f"fp8_gqa_D{D}_P{P}", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, K=K, P=P, window=win,
                      future_keys=fk, right_window=r, ctx_lens=list(lens), seed=83, poison=True,
                      extra_pages=2)


PATHS = [dflash.PATH_MMA, dflash.PATH_TCGEN05]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("win,fk,r", [(0, 1, 0), (4096, 1, 0), (0, 0, 0), (2, 0, 4), (300, 0, 3)])
def test_fp8_minimax(cuda_device, path, win, fk, r):
    _check(_minimax(win, fk, r), cuda_device, k_scale=0.0431, v_scale=1.73, path=path)


@pytest.mark.parametrize("D,P,K,Hq,Hkv", [
    (64, 32, 7, 16, 2),    # R = 56: the tcgen05 path although R <= 64
    (64, 16, 5, 8, 2),     # four pages per tile
    (128, 16, 3, 4, 2),    # R = 6
    (128, 32, 4, 64, 4),   # R = 64
    (64, 64, 16, 8, 1),    # K = 16, R = 128
    (128, 64, 8, 32, 2),   # R = 128 at D = 128: the largest code ring of the mma.sync grid
])
@pytest.mark.parametrize("path", PATHS)
def test_fp8_shapes(cuda_device, path, D, P, K, Hq, Hkv):
    _check(_gqa(D, P, K, Hq, Hkv), cuda_device, k_scale=0.27, v_scale=0.0113, path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("split", [1, 3])
def test_fp8_cut_ranges(cuda_device, path, split):
    """Forced short splits: every pair is cut into many partials."""
    _check(_gqa(128, 64, 7, 16, 1, win=1000), cuda_device, k_scale=3.5, v_scale=0.6, path=path, split=split)


@pytest.mark.parametrize("path", PATHS)
def test_fp8_many_requests(cuda_device, path):
    lens = [int(x) for x in np.random.default_rng(5).integers(0, 3000, size=150)]
    lens[:4] = [0, 1, 63, 64]
    _check(_gqa(128, 64, 7, 16, 1, lens=lens), cuda_device, k_scale=0.05, v_scale=2.0, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_fp8_window_smaller_than_block(cuda_device, path):
    _check(_gqa(64, 32, 7, 16, 2, win=3, fk=0, r=6), cuda_device, k_scale=1.0 / 3.0, v_scale=7.0, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_fp8_long_context_d64(cuda_device, path):
    """The 12/2-head D = 64 shape at 20K context (R = 42: three row groups)."""
    spec = W.CaseSpec("fp8_longctx", B=2, Hq=12, Hkv=2, D=64, K=7, P=32, window=0, future_keys=1,
                      ctx_lens=[20000, 777], seed=87, poison=True)
    _check(spec, cuda_device, k_scale=0.19, v_scale=1.3, path=path)


def test_fp8_block_row_outside_f16_range(cuda_device):
    """The PV product runs on f16 operands on both paths: a block value row
    element with v / v_scale = 70000 is flagged in the device status.  Block
    keys are f16 on the mma.sync path only: a key of 1e5 is flagged there,
    and the tcgen05 path (bf16 keys) takes it without a flag."""
    spec = _gqa(64, 32, 7, 16, 2, lens=(100, 300))

    def big_value(d):
        d["vb"][1, 3, 0, 5] = 70.0

    def big_key(d):
        d["kb"][1, 3, 0, 5] = 1.0e5

    for path in PATHS:
        _, _, status, _ = _run(spec, cuda_device, 0.27, 0.001, path, mutate=big_value)
        assert status == dflash.DFLASH_STATUS_FP8_RANGE, (path, status)
    _, _, status, _ = _run(spec, cuda_device, 0.27, 0.5, dflash.PATH_MMA, mutate=big_key)
    assert status == dflash.DFLASH_STATUS_FP8_RANGE
    out, lse, status, _ = _run(spec, cuda_device, 0.27, 0.5, dflash.PATH_TCGEN05, mutate=big_key)
    assert status == 0
    assert not torch.isnan(out.float()).any() and not torch.isnan(lse).any()
