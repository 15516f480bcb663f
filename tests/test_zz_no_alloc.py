"""The entry point without a caller workspace, against the regular one.

dflash_block_attn_static_ws serves callers that cannot allocate device
memory where they call the attention (stream capture that forbids cudaMalloc,
plugins whose framework owns all device memory, allocator-free latency
paths): it keeps its scratch in an array compiled into the library.  These
checks call it through the C ABI twice in a row, with different shapes, and
compare each result with dflash_block_attn on the same inputs, within the
tolerances the parity tests use; and they check that a parameter set needing
more scratch than the array holds is refused without a launch.
"""

import ctypes

import pytest
import torch

import speculative_decoding_draft_paged_gb300 as dflash
from speculative_decoding_draft_paged_gb300 import _lib
from speculative_decoding_draft_paged_gb300 import workloads as W
from tests._gpu_cases import assert_parity, run_lib

pytestmark = pytest.mark.gpu

STATIC_BYTES = _lib.STATIC_SCRATCH_BYTES


def call_static(spec, inp, out, lse):
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=spec.K,
                          window=spec.window, future_keys=spec.future_keys,
                          scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len)
    return _lib.load().dflash_block_attn_static_ws(
        ctypes.byref(p), inp["q"].data_ptr(), inp["k_pages"].data_ptr(), inp["v_pages"].data_ptr(),
        inp["page_table"].data_ptr(), inp["ctx_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream), p


def compare(out, lse, ref_out, ref_lse):
    """Same bar as the oracle comparisons, with the regular entry point's
    result as the reference."""
    a = out.detach().cpu().double()
    b = ref_out.detach().cpu().double()
    rel = float((a - b).norm() / b.norm())
    m = {"rel_l2": rel,
         "max_abs_excess": float((a - b).abs().max()),
         "max_abs_raw": float((a - b).abs().max()),
         "ulp_at_max": 1.0,
         "lse_abs": float((lse.cpu().double() - ref_lse.cpu().double()).abs().max()),
         "nan": bool(torch.isnan(a).any() or torch.isnan(lse).any())}
    assert_parity(m, "static scratch")


def test_static_scratch_matches_regular_entry_point_twice(cuda_device):
    cases = [W.minimax(B=4, K=7, ctx_lens=[9000, 4100, 300, 16384]),
             W.longctx(B=3, L=20000, Hq=12)]
    for spec in cases:   # two calls in a row, different shapes, same scratch
        inp = {k: v.to(cuda_device) for k, v in W.make_inputs(spec, "cpu").items()}
        ref_out, ref_lse = run_lib(spec, inp)
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full(inp["q"].shape[:3], float("nan"), dtype=torch.float32, device=cuda_device)
        rc, p = call_static(spec, inp, out, lse)
        assert rc == dflash.DFLASH_OK, _lib.status_string(rc)
        assert dflash.workspace_size(p) <= STATIC_BYTES
        torch.cuda.synchronize()
        compare(out, lse, ref_out, ref_lse)


def test_static_scratch_refuses_oversized_plans(cuda_device):
    # Candidates from small to large: the persistent splits need little
    # partial state; one-tile ranges over a long batch, or the unit grid of
    # a batch too large for the flat split, need far more than the array
    # holds.
    cands = [(W.adp(B=64, K=7, L=16384), 0), (W.ragged(B=64, lo=120000, hi=131072), 1),
             (W.ragged(B=800, lo=120000, hi=131072), 0)]
    for s, force in cands:
        p = dflash.make_params(batch=s.B, num_q_heads=s.Hq, num_kv_heads=s.Hkv, head_dim=s.D,
                               page_size=s.P, max_pages_per_req=s.max_pages, num_pages=s.num_pages,
                               block_size=s.K, window=s.window, future_keys=s.future_keys,
                               scale=s.softmax_scale, max_ctx_len=s.max_ctx_len, force_split_tiles=force)
        need = dflash.workspace_size(p)
        if need <= STATIC_BYTES:
            continue
        out = torch.full((s.B, s.K, s.Hq, s.D), 3.0, dtype=torch.bfloat16, device=cuda_device)
        lse = torch.full((s.B, s.K, s.Hq), 3.0, dtype=torch.float32, device=cuda_device)
        dummy = torch.zeros(16, dtype=torch.int32, device=cuda_device)
        rc = _lib.load().dflash_block_attn_static_ws(
            ctypes.byref(p), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
            dummy.data_ptr(), out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rc == dflash.DFLASH_ERR_WORKSPACE
        assert bool((out == 3.0).all()) and bool((lse == 3.0).all())
        return
    pytest.fail("expected at least one parameter set above the static scratch size")
