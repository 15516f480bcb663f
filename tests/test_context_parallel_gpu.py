"""Context-parallel parts and their merge on the GPU, through the C ABI.

Ranks are run one after another on one GPU (no kernel waits on another): each
computes its part of every request's keys with ``dflash_block_attn_partial``;
the parts are stacked as the all-gather lays them out and merged with
``dflash_combine_partials``.  Each part is compared with the oracle's part
(fp32 output: rel L2 < 5e-3, max abs <= 1e-2, LSE within 1e-3, empty rows 0
and -inf), and the merge with the oracle's whole attention at the usual bar.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_paged_gb300 as dflash
from speculative_decoding_draft_paged_gb300 import workloads as W
from speculative_decoding_draft_paged_gb300.context_parallel import split_ranges
from tests._gpu_cases import (LSE_ABS_MAX, MAX_ABS_MAX, REL_L2_MAX, assert_parity, compact_requests, metrics,
                              run_oracle, to_bits)

pytestmark = pytest.mark.gpu


def oracle_part(spec, host, kb, ke):
    return oracle.block_attn_part(to_bits(host["q"]), to_bits(host["k_pages"]), to_bits(host["v_pages"]),
                                  host["page_table"].numpy(), host["ctx_lens"].numpy(), kb, ke,
                                  block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
                                  right_window=spec.right_window, scale=spec.softmax_scale)


def assert_part(po, pl, ro, rl, what):
    g = po.detach().cpu().double().numpy()
    gl = pl.detach().cpu().double().numpy()
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(gl), empty), f"{what}: empty rows differ"
    assert np.all(g[empty] == 0.0), f"{what}: an empty row is not zero"
    seen = ~empty
    if not seen.any():
        return
    d = g[seen] - ro[seen]
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ro[seen]), 1e-300))
    mx = float(np.abs(d).max())
    le = float(np.abs(gl[seen] - rl[seen]).max())
    assert rel < REL_L2_MAX and mx <= MAX_ABS_MAX and le <= LSE_ABS_MAX, (what, rel, mx, le)


def run_ranks(spec, dev_inp, ranges, tables=None, **kw):
    """Each rank's part, then the merge.  Returns (parts, merged)."""
    kb_all, ke_all = ranges
    parts = []
    for r in range(kb_all.shape[0]):
        kb = torch.from_numpy(kb_all[r]).to(dev_inp["q"].device)
        ke = torch.from_numpy(ke_all[r]).to(dev_inp["q"].device)
        tab = dev_inp["page_table"] if tables is None else tables[r]
        p = dflash.params_for(dev_inp["q"], dev_inp["k_pages"], tab, block_size=spec.K, window=spec.window,
                              future_keys=spec.future_keys, scale=spec.softmax_scale,
                              max_ctx_len=spec.max_ctx_len, right_window=spec.right_window)
        ws = torch.zeros(dflash.partial_workspace_size(p), dtype=torch.uint8, device=dev_inp["q"].device)
        po, pl = dflash.block_attn_partial(dev_inp["q"], dev_inp["k_pages"], dev_inp["v_pages"], tab,
                                           dev_inp["ctx_lens"], kb, ke, block_size=spec.K, window=spec.window,
                                           future_keys=spec.future_keys, scale=spec.softmax_scale,
                                           max_ctx_len=spec.max_ctx_len, right_window=spec.right_window,
                                           workspace=ws, **kw)
        torch.cuda.synchronize()
        assert dflash.read_device_status(ws) == 0, f"rank {r}: device status flags set"
        parts.append((po, pl))
    out, lse = dflash.combine_partials(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]))
    torch.cuda.synchronize()
    return parts, (out, lse)


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("window,fk", [(0, 1), (300, 1), (0, 0)])
def test_parts_and_merge(cuda_device, world, window, fk):
    lens = [0, 1, 5, 31, 32, 33, 700, 2049]
    spec = W.CaseSpec(f"cp_w{world}_W{window}_fk{fk}", B=len(lens), Hq=8, Hkv=2, D=64, K=7, P=32,
                      window=window, future_keys=fk, ctx_lens=lens, seed=61, poison=True)
    host = W.make_inputs(spec, "cpu")
    dev = {k: v.to(cuda_device) for k, v in host.items()}
    ranges = split_ranges(spec.ctx_lens, spec.K, world)
    parts, (out, lse) = run_ranks(spec, dev, ranges)
    for r, (po, pl) in enumerate(parts):
        ro, rl = oracle_part(spec, host, ranges[0][r], ranges[1][r])
        assert_part(po, pl, ro, rl, f"{spec.name} rank {r}")
    ro, rl = run_oracle(spec, host)
    assert_parity(metrics(out, lse, ro, rl), spec.name + " merged")


@pytest.mark.parametrize("D", [64, 128])
def test_uneven_and_degenerate_parts(cuda_device, D):
    """Ranges that hold the block only, nothing, one key, or cut the window;
    plus a part that holds the whole sequence (equal to the whole call)."""
    lens = [3, 64, 129, 1000]
    spec = W.CaseSpec(f"cp_uneven_D{D}", B=len(lens), Hq=16, Hkv=1, D=D, K=5, P=64 if D == 128 else 16,
                      window=100, future_keys=1, ctx_lens=lens, seed=62, poison=True)
    host = W.make_inputs(spec, "cpu")
    dev = {k: v.to(cuda_device) for k, v in host.items()}
    L = np.asarray(lens, np.int64)
    T = L + spec.K
    # Per request, three ranks' ranges that tile [0, T):
    #   request 0: empty, empty, everything;
    #   request 1: [0, 10), one key [10, 11), the rest;
    #   request 2: a cut through the window's context [0, L-50), the rest of
    #              the context [L-50, L), the block only [L, T);
    #   request 3: all context, empty, the block only.
    kb = np.array([[0, 0, 0, 0],
                   [0, 10, L[2] - 50, L[3]],
                   [0, 11, L[2], L[3]]], np.int32)
    ke = np.array([[0, 10, L[2] - 50, L[3]],
                   [0, 11, L[2], L[3]],
                   [T[0], T[1], T[2], T[3]]], np.int32)
    assert np.all(kb[0] == 0) and np.all(ke[-1] == T) and np.all(ke[:-1] == kb[1:])
    parts, (out, lse) = run_ranks(spec, dev, (kb, ke))
    for r, (po, pl) in enumerate(parts):
        ro, rl = oracle_part(spec, host, kb[r], ke[r])
        assert_part(po, pl, ro, rl, f"{spec.name} rank {r}")
    ro, rl = run_oracle(spec, host)
    assert_parity(metrics(out, lse, ro, rl), spec.name + " merged")
    # One part holding every key is the whole attention.
    whole = (np.zeros((1, len(lens)), np.int32), T[None, :].astype(np.int32))
    parts1, (out1, lse1) = run_ranks(spec, dev, whole)
    assert_parity(metrics(out1, lse1, ro, rl), spec.name + " one part")


def test_rank_tables_name_only_their_pages(cuda_device):
    """Each rank's page table keeps only the slots its part reads; the others
    are -1 (a rank holds those pages nowhere), and no bad page is read."""
    lens = [40, 400, 3000]
    spec = W.CaseSpec("cp_own_pages", B=len(lens), Hq=12, Hkv=2, D=64, K=7, P=32, window=0, future_keys=1,
                      ctx_lens=lens, seed=63)
    host = W.make_inputs(spec, "cpu")
    dev = {k: v.to(cuda_device) for k, v in host.items()}
    world = 3
    ranges = split_ranges(spec.ctx_lens, spec.K, world)
    tables = []
    for r in range(world):
        t = host["page_table"].clone()
        for b in range(spec.B):
            first, last = ranges[0][r, b] // spec.P, (ranges[1][r, b] + spec.P - 1) // spec.P
            keep = torch.zeros(t.shape[1], dtype=torch.bool)
            keep[first:last] = True
            t[b, ~keep] = -1
        tables.append(t.to(cuda_device))
    parts, (out, lse) = run_ranks(spec, dev, ranges, tables=tables)
    ro, rl = run_oracle(spec, host)
    assert_parity(metrics(out, lse, ro, rl), spec.name)


def test_long_context_two_ranks_sampled(cuda_device):
    """8/2 heads, 32K context, 4 requests split over two ranks; the oracle
    checks two requests of the merge."""
    spec = W.longctx(B=4, L=32768, Hq=8)
    inp = W.make_inputs(spec, cuda_device)
    ranges = split_ranges(spec.ctx_lens, spec.K, 2)
    parts, (out, lse) = run_ranks(spec, inp, ranges)
    ids = [0, 3]
    sub = compact_requests(inp, ids)
    ro, rl = run_oracle(spec, sub)
    assert_parity(metrics(out[ids], lse[ids], ro, rl), spec.name + " two ranks")
