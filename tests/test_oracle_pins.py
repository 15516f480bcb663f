"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

None of these compares the oracle with itself re-typed: the dense cases use
torch's own ``scaled_dot_product_attention`` and ``logsumexp`` (float64, CPU)
over contiguous sequences with no page table; the merge pin composes two
independent attentions; the closed forms are counted or averaged directly;
the hand fixtures in ``tests/golden`` were derived on paper.
"""

import glob
import json
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from tests._paged import permute_pool, random_bf16, scatter_to_pages

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LN2 = math.log(2.0)


# ----------------------------------------------------------------------------
# Dense library references (torch float64 on CPU, contiguous keys, no paging)
# ----------------------------------------------------------------------------

def visible_mask(L, K, W, future_keys, right_window=0):
    """Boolean [K, L+K] mask of the pages' visible set, by position.

    Query i sits at position L+i.  Causal window: (L+i-W, L+i] (all of
    [0, L+i] when W = 0).  Later block keys: positions in (L+i, L+i+r], r =
    K-1 in the non-causal form (every later block key) else the right window.
    """
    pos = np.arange(L + K)[None, :]
    qpos = L + np.arange(K)[:, None]
    causal = pos <= qpos
    if W > 0:
        causal &= pos > qpos - W
    r = K - 1 if future_keys else right_window
    later = (pos > qpos) & (pos <= qpos + r)
    return causal | later


def dense_attention(q_bits, k_bits, v_bits, scale, mask):
    """torch SDPA + logsumexp in float64.  q [K,Hq,D], k/v [T,Hkv,D], mask [K,T]."""
    import oracle

    return dense_attention_f64(oracle.bf16_bits_to_float(q_bits), oracle.bf16_bits_to_float(k_bits),
                               oracle.bf16_bits_to_float(v_bits), scale, mask)


def dense_attention_f64(q, k, v, scale, mask):
    """dense_attention over real-valued rows (numpy, any float dtype)."""
    q = torch.from_numpy(np.asarray(q, dtype=np.float64))
    k = torch.from_numpy(np.asarray(k, dtype=np.float64))
    v = torch.from_numpy(np.asarray(v, dtype=np.float64))
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    qh = q.permute(1, 0, 2)                                  # [Hq, K, D]
    kh = k.permute(1, 0, 2).repeat_interleave(G, dim=0)      # [Hq, T, D]
    vh = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
    m = torch.from_numpy(mask)
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=m, scale=scale)
    logits = (qh @ kh.transpose(1, 2)) * scale
    logits = logits.masked_fill(~m, float("-inf"))
    lse2 = torch.logsumexp(logits, dim=-1) / LN2              # [Hq, K]
    return out.permute(1, 0, 2).numpy(), lse2.T.numpy()      # [K,Hq,D], [K,Hq]


def make_case(rng, B, Hq, Hkv, D, K, P, lens, sigma=1.0, extra_pages=2, extra_slots=1):
    q = random_bf16(rng, (B, K, Hq, D), sigma)
    dk = [random_bf16(rng, (L + K, Hkv, D), sigma) for L in lens]
    dv = [random_bf16(rng, (L + K, Hkv, D), sigma) for L in lens]
    kp, vp, tab = scatter_to_pages(rng, dk, dv, P, Hkv, D, extra_pages, extra_slots)
    return q, dk, dv, kp, vp, tab, np.asarray(lens, dtype=np.int32)


TINY_SHAPES = [  # (Hq, Hkv, D, P)
    (1, 1, 4, 1), (2, 1, 8, 4), (4, 2, 4, 8), (6, 3, 8, 3), (4, 4, 8, 5),
]


@pytest.mark.parametrize("shape", TINY_SHAPES)
@pytest.mark.parametrize("K", [1, 2, 4])
def test_unwindowed_equals_dense_full_attention(oracle_mod, shape, K):
    """Unwindowed non-causal = textbook full attention over context + block."""
    Hq, Hkv, D, P = shape
    rng = np.random.default_rng(100 + 7 * K + D + P)
    lens = [0, 1, 5, 17, 40][: 3 + K % 3]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    scale = 0.37
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=0, future_keys=1,
                                      scale=scale)
    for b, L in enumerate(lens):
        mask = np.ones((K, L + K), dtype=bool)
        ro, rl = dense_attention(q[b], dk[b], dv[b], scale, mask)
        np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("W", [0, 1, 3, 6, 50])
@pytest.mark.parametrize("K", [1, 3, 4])
def test_causal_block_equals_windowed_decode(oracle_mod, W, K):
    """future_keys=0 (and K=1 in any form) is causal windowed decode, by position mask."""
    rng = np.random.default_rng(200 + W * 5 + K)
    Hq, Hkv, D, P = 4, 2, 8, 4
    lens = [0, 2, 7, 23, 31]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    forms = [0] + ([1] if K == 1 else [])
    for fk in forms:
        out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W,
                                          future_keys=fk, scale=0.5)
        for b, L in enumerate(lens):
            ro, rl = dense_attention(q[b], dk[b], dv[b], 0.5, visible_mask(L, K, W, 0))
            np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("W", [4, 5, 9, 64])
@pytest.mark.parametrize("K", [2, 4])
def test_noncausal_window_equals_masked_dense(oracle_mod, W, K):
    """Non-causal windowed: window (L+i-W, L+i] plus every block key."""
    rng = np.random.default_rng(300 + W + K)
    Hq, Hkv, D, P = 6, 2, 8, 4
    lens = [0, 3, 9, 21, 40]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=1,
                                      scale=0.41)
    for b, L in enumerate(lens):
        ro, rl = dense_attention(q[b], dk[b], dv[b], 0.41, visible_mask(L, K, W, 1))
        np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("W", [0, 1, 2, 3, 9])
@pytest.mark.parametrize("r", [0, 1, 2, 3])
def test_right_window_equals_masked_dense(oracle_mod, W, r):
    """A right window r: the causal window (L+i-W, L+i] plus block keys
    L+i+1 .. L+i+r; with 0 < W < K the window also drops block keys."""
    K = 4
    rng = np.random.default_rng(310 + 10 * W + r)
    Hq, Hkv, D, P = 4, 2, 8, 3
    lens = [0, 1, 4, 13, 26]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=0,
                                      right_window=r, scale=0.53)
    for b, L in enumerate(lens):
        ro, rl = dense_attention(q[b], dk[b], dv[b], 0.53, visible_mask(L, K, W, 0, r))
        np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)
    if r == K - 1:
        full = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=1,
                                     scale=0.53)
        np.testing.assert_array_equal(full[0], out)
        np.testing.assert_array_equal(full[1], lse2)


def test_window_one_right_zero_is_own_key(oracle_mod):
    """W = 1, r = 0: every row sees its own key only: out = v, lse2 = s/ln 2."""
    import oracle

    rng = np.random.default_rng(330)
    K, Hq, Hkv, D, P = 3, 2, 1, 4, 2
    lens = [0, 3, 8]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=1, future_keys=0,
                                      right_window=0, scale=0.25)
    for b, L in enumerate(lens):
        qf = oracle.bf16_bits_to_float(q[b]).astype(np.float64)
        kf = oracle.bf16_bits_to_float(dk[b]).astype(np.float64)
        vf = oracle.bf16_bits_to_float(dv[b]).astype(np.float64)
        for i in range(K):
            for hq in range(Hq):
                np.testing.assert_array_equal(out[b, i, hq], vf[L + i, 0])
                s = 0.25 * float(np.dot(qf[i, hq], kf[L + i, 0]))
                assert abs(lse2[b, i, hq] - s / LN2) < 1e-12


@pytest.mark.parametrize("W", [0, 5, 12])
def test_lse_merge_of_disjoint_key_sets(oracle_mod, W):
    """Non-causal = causal part merged with the later block keys by base-2 LSE.

    Checks both the log-sum-exp form and the sigmoid/lerp form of the same
    two-way merge (PR #21130, formulation table: einsum + sigmoid/lerp).
    """
    rng = np.random.default_rng(400 + W)
    Hq, Hkv, D, P, K = 4, 1, 8, 4, 4
    lens = [1, 6, 19, 30]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    s = 0.6
    full, full_lse = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W,
                                           future_keys=1, scale=s)
    part, part_lse = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W,
                                           future_keys=0, scale=s)
    for b, L in enumerate(lens):
        for i in range(K - 1):
            fmask = np.zeros((K, L + K), dtype=bool)
            fmask[:, L + i + 1:] = True
            ob, lb = dense_attention(q[b], dk[b], dv[b], s, fmask)
            oa, la = part[b, i], part_lse[b, i]
            ob, lb = ob[i], lb[i]
            lse = np.logaddexp2(la, lb)
            merged = oa * np.exp2(la - lse)[:, None] + ob * np.exp2(lb - lse)[:, None]
            np.testing.assert_allclose(full[b, i], merged, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(full_lse[b, i], lse, rtol=1e-12, atol=1e-12)
            sig = 1.0 / (1.0 + np.exp(-(lb - la) * LN2))
            lerp = oa + sig[:, None] * (ob - oa)
            np.testing.assert_allclose(full[b, i], lerp, rtol=1e-10, atol=1e-11)
        # The last row has no later key: both forms agree exactly.
        np.testing.assert_array_equal(full[b, K - 1], part[b, K - 1])
        np.testing.assert_array_equal(full_lse[b, K - 1], part_lse[b, K - 1])


@pytest.mark.parametrize("W", [0, 7])
def test_page_permutation_invariance_bitwise(oracle_mod, W):
    rng = np.random.default_rng(500 + W)
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 3, 8, 2, 8, 3, 4, [5, 13, 22], extra_pages=5)
    a = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=3, window=W, future_keys=1, scale=0.3)
    kp2, vp2, tab2 = permute_pool(rng, kp, vp, tab)
    b = oracle_mod.block_attn(q, kp2, vp2, tab2, ctx, block_size=3, window=W, future_keys=1,
                              scale=0.3)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_thread_count_invariance_bitwise(oracle_mod):
    rng = np.random.default_rng(600)
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 5, 6, 3, 8, 2, 4, [0, 4, 9, 15, 33])
    a = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=2, window=6, future_keys=1,
                              scale=0.3, nthreads=1)
    b = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=2, window=6, future_keys=1,
                              scale=0.3, nthreads=7)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_request_subset_matches_full_batch(oracle_mod):
    rng = np.random.default_rng(601)
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 5, 4, 2, 8, 3, 4, [3, 4, 9, 15, 33])
    full = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=3, window=0, future_keys=1,
                                 scale=0.3)
    ids = np.array([4, 1], dtype=np.int32)
    sub = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=3, window=0, future_keys=1,
                                scale=0.3, req_ids=ids)
    np.testing.assert_array_equal(sub[0], full[0][ids])
    np.testing.assert_array_equal(sub[1], full[1][ids])


# ----------------------------------------------------------------------------
# Closed forms
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("W,fk", [(0, 1), (0, 0), (6, 1), (6, 0), (3, 1)])
def test_zero_query_gives_mean_and_log2_count(oracle_mod, W, fk):
    """q = 0: uniform weights, out = mean of the visible V rows, lse2 = log2(count)."""
    rng = np.random.default_rng(700 + W + fk)
    K, Hq, Hkv, D, P = 3, 2, 1, 4, 4
    lens = [0, 2, 5, 11]
    _, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    q = np.zeros((len(lens), K, Hq, D), dtype=np.uint16)
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W,
                                      future_keys=fk, scale=1.0)
    import oracle

    for b, L in enumerate(lens):
        vals = oracle.bf16_bits_to_float(dv[b]).astype(np.float64)   # [L+K, Hkv, D]
        for i in range(K):
            lo = max(0, L + i - W + 1) if W > 0 else 0
            block = list(range(L, L + K)) if fk else list(range(L, L + i + 1))
            rows = list(range(lo, L)) + block
            n = (L - lo) + (K if fk else i + 1)
            assert len(rows) == n
            np.testing.assert_allclose(out[b, i, :, :], np.broadcast_to(vals[rows, 0].mean(0), (Hq, D)),
                                       rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse2[b, i], np.full(Hq, math.log2(n)), rtol=0, atol=1e-12)


def test_constant_values_give_constant_output(oracle_mod):
    rng = np.random.default_rng(800)
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 3, 4, 2, 8, 3, 4, [0, 6, 17])
    import oracle

    c = oracle.bf16_bits_from_float(np.float32(1.5))
    vp = np.where(vp == 0x7FC0, vp, c).astype(np.uint16)
    out, _ = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=3, window=5, future_keys=1,
                                   scale=0.7)
    np.testing.assert_allclose(out, 1.5, rtol=1e-14, atol=0)


def test_short_context_window_equals_unwindowed(oracle_mod):
    """With L <= W-K no window edge is inside the sequence: the two forms coincide."""
    rng = np.random.default_rng(900)
    K, W = 3, 12
    lens = [0, 4, 9]                     # all <= W - K
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 3, 4, 1, 8, K, 4, lens)
    a = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=1, scale=0.5)
    b = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=0, future_keys=1, scale=0.5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_empty_context_is_attention_over_the_block(oracle_mod):
    rng = np.random.default_rng(901)
    K = 4
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 1, 4, 2, 8, K, 3, [0])
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=7, future_keys=1,
                                      scale=0.9)
    ro, rl = dense_attention(q[0], dk[0], dv[0], 0.9, np.ones((K, K), dtype=bool))
    np.testing.assert_allclose(out[0], ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse2[0], rl, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------
# Hand-derived fixtures
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "*.json"))))
def test_hand_derived_fixture(oracle_mod, path):
    import oracle

    fx = json.load(open(path))
    P, Hkv, D = fx["P"], fx["Hkv"], fx["D"]
    table = np.asarray(fx["page_table"], dtype=np.int32)
    num_pages = int(table.max()) + 1
    kp = np.full((num_pages, Hkv, P, D), 0x7FC0, dtype=np.uint16)   # unused slots are NaN
    vp = kp.copy()
    kpos = np.asarray(fx["kv_positions"]["k"], dtype=np.float32)
    vpos = np.asarray(fx["kv_positions"]["v"], dtype=np.float32)
    for p in range(kpos.shape[0]):
        pg = table[0, p // P]
        kp[pg, 0, p % P] = oracle.bf16_bits_from_float(kpos[p])
        vp[pg, 0, p % P] = oracle.bf16_bits_from_float(vpos[p])
    q = oracle.bf16_bits_from_float(np.asarray(fx["q"], dtype=np.float32))
    out, lse2 = oracle_mod.block_attn(q, kp, vp, table, np.asarray(fx["ctx_lens"], dtype=np.int32),
                                      block_size=fx["K"], window=fx["window"],
                                      future_keys=fx["future_keys"], scale=fx["scale"])
    np.testing.assert_allclose(out, np.asarray(fx["expected_out"]), rtol=0, atol=fx["tolerance"])
    np.testing.assert_allclose(lse2, np.asarray(fx["expected_lse2"]), rtol=0, atol=fx["tolerance"])


# ----------------------------------------------------------------------------
# Block placement and K/V append (plain data movement)
# ----------------------------------------------------------------------------

def _tagged_case(rng, lens, K, Hkv, D, P):
    """Dense K/V whose rows carry their (request, position) in the first two
    columns (exact small integers in bf16), scattered into shuffled pages."""
    import oracle

    dk, dv = [], []
    for b, L in enumerate(lens):
        k = random_bf16(rng, (L + K, Hkv, D), 1.0)
        v = random_bf16(rng, (L + K, Hkv, D), 1.0)
        pos = np.arange(L + K, dtype=np.float32)
        k[:, :, 0] = oracle.bf16_bits_from_float(np.broadcast_to(pos[:, None], (L + K, Hkv)))
        k[:, :, 1] = oracle.bf16_bits_from_float(np.float32(b))
        dk.append(k)
        dv.append(v)
    kp, vp, tab = scatter_to_pages(rng, dk, dv, P, Hkv, D, extra_pages=3, extra_slots=2)
    return dk, dv, kp, vp, tab


@pytest.mark.parametrize("P", [1, 3, 4, 16])
def test_block_placement_points_at_the_block_rows(oracle_mod, P):
    rng = np.random.default_rng(960 + P)
    K, Hkv, D = 5, 2, 8
    lens = [0, 1, P - 1 if P > 1 else 2, P, 2 * P + 3, 37]
    dk, dv, kp, vp, tab = _tagged_case(rng, lens, K, Hkv, D, P)
    pl = oracle_mod.block_placement(tab, np.asarray(lens, np.int32), block_size=K, page_size=P,
                                    num_pages=kp.shape[0])
    for b, L in enumerate(lens):
        for j in range(K):
            page, off = pl[b, j]
            np.testing.assert_array_equal(kp[page, :, off, :], dk[b][L + j])


def test_append_then_gather_is_the_dense_sequence(oracle_mod):
    """Pages holding the context only, then the append: reading every position
    through the table gives context + block, and no other row changes."""
    rng = np.random.default_rng(970)
    K, Hkv, D, P = 4, 2, 8, 3
    lens = [0, 2, 3, 7, 11]
    dk, dv, kp_full, vp_full, tab = _tagged_case(rng, lens, K, Hkv, D, P)
    kp, vp = kp_full.copy(), vp_full.copy()
    kb = np.zeros((len(lens), K, Hkv, D), np.uint16)
    vb = np.zeros_like(kb)
    for b, L in enumerate(lens):          # blank the block rows, keep them aside
        kb[b], vb[b] = dk[b][L:], dv[b][L:]
        for p in range(L, L + K):
            kp[tab[b, p // P], :, p % P, :] = 0x7FC0
            vp[tab[b, p // P], :, p % P, :] = 0x7FC0
    ka, va = oracle_mod.append_block_kv(kb, vb, kp, vp, tab, np.asarray(lens, np.int32))
    np.testing.assert_array_equal(ka, kp_full)
    np.testing.assert_array_equal(va, vp_full)
    np.testing.assert_array_equal(kp[tab[0, 0], :, 0, :], np.full((Hkv, D), 0x7FC0, np.uint16))


def test_append_then_attention_equals_dense(oracle_mod):
    rng = np.random.default_rng(980)
    K, Hq, Hkv, D, P = 3, 4, 2, 8, 4
    lens = [0, 5, 14]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    kb = np.stack([dk[b][L:] for b, L in enumerate(lens)])
    vb = np.stack([dv[b][L:] for b, L in enumerate(lens)])
    for b, L in enumerate(lens):          # overwrite the block rows with garbage first
        for p in range(L, L + K):
            kp[tab[b, p // P], :, p % P, :] = 0x3F80
            vp[tab[b, p // P], :, p % P, :] = 0x3F80
    ka, va = oracle_mod.append_block_kv(kb, vb, kp, vp, tab, ctx)
    out, lse2 = oracle_mod.block_attn(q, ka, va, tab, ctx, block_size=K, window=0, future_keys=1,
                                      scale=0.4)
    for b, L in enumerate(lens):
        ro, rl = dense_attention(q[b], dk[b], dv[b], 0.4, np.ones((K, L + K), dtype=bool))
        np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("W,fk,r", [(0, 1, 0), (5, 1, 0), (0, 0, 1), (2, 0, 2)])
def test_dense_suffix_equals_dense_attention(oracle_mod, W, fk, r):
    """Dense-suffix form: the pages hold the context only (block slots are NaN),
    the block rows come from dense tensors; the result is the masked dense
    attention over context + block, and equals appending then reading paged."""
    rng = np.random.default_rng(1100 + 10 * W + r)
    K, Hq, Hkv, D, P = 4, 4, 2, 8, 3
    lens = [0, 2, 5, 16]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    kb = np.stack([dk[b][L:] for b, L in enumerate(lens)])
    vb = np.stack([dv[b][L:] for b, L in enumerate(lens)])
    for b, L in enumerate(lens):
        for p in range(L, L + K):
            kp[tab[b, p // P], :, p % P, :] = 0x7FC0
            vp[tab[b, p // P], :, p % P, :] = 0x7FC0
    out, lse2 = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=fk,
                                      right_window=r, scale=0.47, k_block=kb, v_block=vb)
    for b, L in enumerate(lens):
        ro, rl = dense_attention(q[b], dk[b], dv[b], 0.47, visible_mask(L, K, W, fk, r))
        np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)
    ka, va = oracle_mod.append_block_kv(kb, vb, kp, vp, tab, ctx)
    o2, l2 = oracle_mod.block_attn(q, ka, va, tab, ctx, block_size=K, window=W, future_keys=fk,
                                   right_window=r, scale=0.47)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(lse2, l2)


# ----------------------------------------------------------------------------
# fp8 (E4M3) context storage
# ----------------------------------------------------------------------------

def torch_e4m3(codes):
    """torch's own float8_e4m3fn decoding of uint8 codes, as float64."""
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def random_e4m3(rng, shape, sigma=1.0):
    """E4M3 codes of normal samples, rounded by torch's float8_e4m3fn cast."""
    x = torch.from_numpy(rng.normal(0.0, sigma, size=shape).astype(np.float32))
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch(oracle_mod):
    """Every one of the 256 codes decodes as torch's float8_e4m3fn does (NaN
    for S.1111.111 only; 448 the largest finite value; 2^-9 the smallest)."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.e4m3_to_float64(codes)
    ref = torch_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert set(np.flatnonzero(np.isnan(got))) == {0x7F, 0xFF}
    np.testing.assert_array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0 and got[0xB8] == -1.0


def _fp8_case(rng, lens, Hq, Hkv, D, K, P, sigma=1.0):
    """Queries, dense block rows (bf16 bits), fp8 context codes scattered to
    pages (unused slots hold the NaN code), and the context codes per request."""
    B = len(lens)
    q = random_bf16(rng, (B, K, Hq, D), sigma)
    kb = random_bf16(rng, (B, K, Hkv, D), sigma)
    vb = random_bf16(rng, (B, K, Hkv, D), sigma)
    ck = [random_e4m3(rng, (L, Hkv, D), sigma) for L in lens]
    cv = [random_e4m3(rng, (L, Hkv, D), sigma) for L in lens]
    kp, vp, tab = scatter_to_pages(rng, ck, cv, P, Hkv, D, extra_pages=2, extra_slots=1,
                                   fill_bits=0x7F, dtype=np.uint8)
    return q, kb, vb, ck, cv, kp, vp, tab, np.asarray(lens, dtype=np.int32)


@pytest.mark.parametrize("W,fk,r", [(0, 1, 0), (6, 1, 0), (0, 0, 2), (3, 0, 0)])
def test_fp8_context_power_of_two_scales_is_the_bf16_form(oracle_mod, W, fk, r):
    """With power-of-two scales every dequantised context value is a bf16
    value: the fp8 form must equal, bit for bit, the bf16 dense-suffix form
    over pages holding those values (a scale applied to the block rows, the
    K scale used for V, or a decoding slip all break this)."""
    rng = np.random.default_rng(2100 + W + 10 * r)
    K, Hq, Hkv, D, P = 4, 4, 2, 8, 3
    lens = [0, 2, 5, 17]
    q, kb, vb, ck, cv, kp8, vp8, tab, ctx = _fp8_case(rng, lens, Hq, Hkv, D, K, P)
    ks, vs = 0.25, 8.0
    kp16 = oracle_mod.bf16_bits_from_float((torch_e4m3(kp8) * ks).astype(np.float32))
    vp16 = oracle_mod.bf16_bits_from_float((torch_e4m3(vp8) * vs).astype(np.float32))
    args = dict(block_size=K, window=W, future_keys=fk, right_window=r, scale=0.41)
    out8, lse8 = oracle_mod.block_attn_fp8(q, kp8, vp8, tab, ctx, k_scale=ks, v_scale=vs, k_block=kb,
                                           v_block=vb, **args)
    out16, lse16 = oracle_mod.block_attn(q, kp16, vp16, tab, ctx, k_block=kb, v_block=vb, **args)
    np.testing.assert_array_equal(out8, out16)
    np.testing.assert_array_equal(lse8, lse16)


@pytest.mark.parametrize("W,fk,r", [(0, 1, 0), (5, 1, 0), (2, 0, 1)])
def test_fp8_context_equals_dense_attention(oracle_mod, W, fk, r):
    """General scales: torch SDPA in float64 over the contiguous sequence of
    (torch-decoded context codes x scale) followed by the bf16 block rows."""
    import oracle

    rng = np.random.default_rng(2200 + W + 10 * r)
    K, Hq, Hkv, D, P = 3, 6, 3, 8, 4
    lens = [0, 1, 7, 21]
    q, kb, vb, ck, cv, kp8, vp8, tab, ctx = _fp8_case(rng, lens, Hq, Hkv, D, K, P)
    ks, vs = 0.0371, 1.7
    out, lse2 = oracle_mod.block_attn_fp8(q, kp8, vp8, tab, ctx, k_scale=ks, v_scale=vs, k_block=kb,
                                          v_block=vb, block_size=K, window=W, future_keys=fk,
                                          right_window=r, scale=0.52)
    for b, L in enumerate(lens):
        k = np.concatenate([torch_e4m3(ck[b]) * ks, oracle.bf16_bits_to_float(kb[b]).astype(np.float64)])
        v = np.concatenate([torch_e4m3(cv[b]) * vs, oracle.bf16_bits_to_float(vb[b]).astype(np.float64)])
        qf = oracle.bf16_bits_to_float(q[b]).astype(np.float64)
        ro, rl = dense_attention_f64(qf, k, v, 0.52, visible_mask(L, K, W, fk, r))
        np.testing.assert_allclose(out[b], ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse2[b], rl, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------
# Errors
# ----------------------------------------------------------------------------

def test_errors(oracle_mod):
    rng = np.random.default_rng(950)
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, 2, 2, 1, 4, 2, 4, [3, 6])
    bad = tab.copy()
    bad[1, 0] = kp.shape[0] + 3
    with pytest.raises(ValueError, match="-3"):
        oracle_mod.block_attn(q, kp, vp, bad, ctx, block_size=2, window=0, future_keys=1, scale=1.0)
    with pytest.raises(ValueError, match="-2"):
        oracle_mod.block_attn(q, kp, vp, tab, np.array([3, -1], np.int32), block_size=2, window=0,
                              future_keys=1, scale=1.0)
    # A table entry only outside the window is never read.
    tw = tab.copy()
    tw[1, 0] = -1          # positions 0..3 of request 1 (L=6); W=2 reads from position 5 on
    oracle_mod.block_attn(q, kp, vp, tw, ctx, block_size=2, window=2, future_keys=1, scale=1.0)


# ----------------------------------------------------------------------------
# Sensitivity: plausible mistakes planted in a copy of the oracle must fail a pin
# ----------------------------------------------------------------------------

MUTANTS = [
    ("window off by one", "L + i - pr.W + 1", "L + i - pr.W"),
    ("later keys skip the first", "for (int j = i + 1; j <= j_last; ++j)", "for (int j = i + 2; j <= j_last; ++j)"),
    ("right window ignored", "const int r = pr.future_keys ? pr.K - 1 : pr.right_window;",
     "const int r = pr.future_keys ? pr.K - 1 : 0;"),
    ("causal window stops before the query", "for (int64_t p = lo; p <= L + i; ++p)",
     "for (int64_t p = lo; p < L + i; ++p)"),
    ("wrong GQA head map", "const int h = hq / G;", "const int h = hq % pr.Hkv;"),
    ("page slot / offset swapped", "(p % pr.P)) * pr.D", "(p / pr.P) % pr.P) * pr.D"),
    ("scale dropped", "s[t] = pr.scale * acc;", "s[t] = acc;"),
    ("natural-log LSE", "/ std::log(2.0)", "/ 1.0"),
    ("max not subtracted in numerator", "const double w = std::exp(s[t] - m);",
     "const double w = std::exp(s[t]);"),
]

# Planted mistakes in the placement / append, each caught by a pin above.
MOVE_MUTANTS = [
    ("placement offset off by one", "static_cast<int32_t>(p % P);", "static_cast<int32_t>((p + 1) % P);"),
    ("placement from the context end", "const int64_t p = L + j;", "const int64_t p = L + j - 1;"),
    ("append writes K into V", "v_pages[dst + d] = v_block[src + d];", "v_pages[dst + d] = k_block[src + d];"),
]


def _pins_pass(lib) -> bool:
    """A compact set of the pins above, run against an arbitrary oracle build."""
    import oracle

    rng = np.random.default_rng(1234)
    try:
        for (Hq, Hkv, D, P, K, W, fk, rw, lens) in [
            (4, 2, 8, 4, 3, 0, 1, 0, [0, 5, 14]),
            (4, 2, 8, 4, 3, 5, 0, 0, [2, 9, 20]),
            (6, 3, 8, 3, 4, 6, 1, 0, [1, 7, 25]),
            (4, 2, 8, 4, 4, 2, 0, 2, [0, 6, 11]),
        ]:
            q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
            out, lse2 = oracle.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W,
                                          future_keys=fk, right_window=rw, scale=0.45, lib=lib)
            for b, L in enumerate(lens):
                ro, rl = dense_attention(q[b], dk[b], dv[b], 0.45, visible_mask(L, K, W, fk, rw))
                if not (np.allclose(out[b], ro, rtol=1e-10, atol=1e-11) and
                        np.allclose(lse2[b], rl, rtol=1e-10, atol=1e-11)):
                    return False
        # closed form: q = 0, large-magnitude keys do not matter, lse2 = log2(count)
        q = np.zeros((1, 2, 2, 4), dtype=np.uint16)
        kbig = oracle.bf16_bits_from_float(np.full((12, 1, 4), 40.0, np.float32))
        kp, vp, tab = scatter_to_pages(rng, [kbig], [kbig], 4, 1, 4)
        out, lse2 = oracle.block_attn(q, kp, vp, tab, np.array([10], np.int32), block_size=2,
                                      window=0, future_keys=1, scale=1.0, lib=lib)
        if not (np.allclose(lse2, math.log2(12), atol=1e-12) and np.allclose(out, 40.0)):
            return False
    except ValueError:
        return False
    return True


def test_pins_reject_planted_mistakes(oracle_mod, tmp_path):
    import oracle

    src = open(os.path.join(os.path.dirname(oracle.__file__), "dflash_oracle.cpp")).read()
    assert _pins_pass(oracle._load()), "the unmodified oracle must pass the compact pins"
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name
        path = tmp_path / (name.replace(" ", "_").replace("/", "") + ".cpp")
        path.write_text(src.replace(old, new))
        so = str(path) + ".so"
        subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(path), "-o", so],
                       check=True)
        lib = oracle.load_library(so)
        assert not _pins_pass(lib), f"planted mistake not caught: {name}"


def _move_pins_pass(lib) -> bool:
    import oracle

    try:
        rng = np.random.default_rng(990)
        K, Hkv, D, P = 4, 2, 8, 3
        lens = [0, 2, 5, 9]
        dk, dv, kp_full, vp_full, tab = _tagged_case(rng, lens, K, Hkv, D, P)
        pl = oracle.block_placement(tab, np.asarray(lens, np.int32), block_size=K, page_size=P,
                                    num_pages=kp_full.shape[0], lib=lib)
        for b, L in enumerate(lens):
            for j in range(K):
                if not np.array_equal(kp_full[pl[b, j, 0], :, pl[b, j, 1], :], dk[b][L + j]):
                    return False
        kb = np.stack([dk[b][L:] for b, L in enumerate(lens)])
        vb = np.stack([dv[b][L:] for b, L in enumerate(lens)])
        ka, va = oracle.append_block_kv(kb, vb, kp_full * 0, vp_full * 0, tab,
                                        np.asarray(lens, np.int32), lib=lib)
        for b, L in enumerate(lens):
            for p in range(L, L + K):
                pg = tab[b, p // P]
                if not (np.array_equal(ka[pg, :, p % P], dk[b][p]) and
                        np.array_equal(va[pg, :, p % P], dv[b][p])):
                    return False
    except ValueError:
        return False
    return True


# Planted mistakes in the fp8 context reading, each caught by an fp8 pin.
FP8_MUTANTS = [
    ("e4m3 bias off by one", "std::ldexp(static_cast<double>(8 + m), e - 10)",
     "std::ldexp(static_cast<double>(8 + m), e - 9)"),
    ("e4m3 subnormals read as normals", "e == 0 ? std::ldexp(static_cast<double>(m), -9)",
     "e == 0 ? std::ldexp(static_cast<double>(8 + m), -10)"),
    ("k scale dropped", "RowRef{nullptr, pr.k_pages8 + o, pr.k_scale}", "RowRef{nullptr, pr.k_pages8 + o, 1.0}"),
    ("v read with the k scale", "RowRef{nullptr, pr.v_pages8 + o, pr.v_scale}",
     "RowRef{nullptr, pr.v_pages8 + o, pr.k_scale}"),
    ("block rows scaled too", "krow[t] = RowRef{pr.k_block + o, nullptr, 1.0};",
     "krow[t] = RowRef{pr.k_block + o, nullptr, pr.k_pages8 ? pr.k_scale : 1.0};"),
]


def _fp8_pins_pass(lib) -> bool:
    """The decoding pin and one power-of-two-scale reduction, against a build."""
    import oracle

    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_float64(codes, lib=lib)
    ref = torch_e4m3(codes)
    if not (np.array_equal(np.isnan(got), np.isnan(ref)) and
            np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])):
        return False
    rng = np.random.default_rng(77)
    K, Hq, Hkv, D, P = 3, 4, 2, 8, 4
    q, kb, vb, ck, cv, kp8, vp8, tab, ctx = _fp8_case(rng, [0, 6, 13], Hq, Hkv, D, K, P)
    ks, vs = 0.5, 4.0
    kp16 = oracle.bf16_bits_from_float((torch_e4m3(kp8) * ks).astype(np.float32))
    vp16 = oracle.bf16_bits_from_float((torch_e4m3(vp8) * vs).astype(np.float32))
    args = dict(block_size=K, window=0, future_keys=1, scale=0.5)
    try:
        o8, l8 = oracle.block_attn_fp8(q, kp8, vp8, tab, ctx, k_scale=ks, v_scale=vs, k_block=kb,
                                       v_block=vb, lib=lib, **args)
    except ValueError:
        return False
    o16, l16 = oracle.block_attn(q, kp16, vp16, tab, ctx, k_block=kb, v_block=vb, **args)
    return np.array_equal(o8, o16) and np.array_equal(l8, l16)


def test_fp8_pins_reject_planted_mistakes(oracle_mod, tmp_path):
    import oracle

    src = open(os.path.join(os.path.dirname(oracle.__file__), "dflash_oracle.cpp")).read()
    assert _fp8_pins_pass(oracle._load())
    for name, old, new in FP8_MUTANTS:
        assert src.count(old) == 1, name
        path = tmp_path / (name.replace(" ", "_") + ".cpp")
        path.write_text(src.replace(old, new))
        so = str(path) + ".so"
        subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(path), "-o", so],
                       check=True)
        assert not _fp8_pins_pass(oracle.load_library(so)), f"planted mistake not caught: {name}"


def test_move_pins_reject_planted_mistakes(oracle_mod, tmp_path):
    import oracle

    src = open(os.path.join(os.path.dirname(oracle.__file__), "dflash_oracle.cpp")).read()
    assert _move_pins_pass(oracle._load())
    for name, old, new in MOVE_MUTANTS:
        assert src.count(old) == 1, name
        path = tmp_path / (name.replace(" ", "_") + ".cpp")
        path.write_text(src.replace(old, new))
        so = str(path) + ".so"
        subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(path), "-o", so],
                       check=True)
        assert not _move_pins_pass(oracle.load_library(so)), f"planted mistake not caught: {name}"


# ----------------------------------------------------------------------------
# Context-parallel parts: a part covers logical keys [kb, ke) of L + K
# ----------------------------------------------------------------------------

def range_mask(L, K, kb, ke):
    pos = np.arange(L + K)[None, :]
    return np.broadcast_to((pos >= kb) & (pos < ke), (K, L + K))


def _check_part_against_dense(out, lse2, q, dk, dv, scale, L, K, W, fk, kb, ke, rtol=1e-11, atol=1e-12):
    """Rows that see a key of [kb, ke): torch SDPA over the masked sequence;
    rows that see none: out 0, lse2 -inf."""
    mask = visible_mask(L, K, W, fk) & range_mask(L, K, kb, ke)
    seen = mask.any(axis=1)
    if seen.any():
        ro, rl = dense_attention(q, dk, dv, scale, np.where(seen[:, None], mask, True))
        np.testing.assert_allclose(out[seen], ro[seen], rtol=rtol, atol=atol)
        np.testing.assert_allclose(lse2[seen], rl[seen], rtol=rtol, atol=atol)
    assert np.all(out[~seen] == 0.0) and np.all(np.isneginf(lse2[~seen]))


def _part_ranges(rng, L, K):
    """Ranges covering the interesting cases for a request of L + K keys."""
    T = L + K
    cuts = sorted(int(x) for x in rng.integers(0, T + 1, size=3))
    out = [(0, T), (0, 0), (L, T), (0, L), (T, T + 5)]
    out += [(a, b) for a, b in zip([0] + cuts, cuts + [T])]
    return out


@pytest.mark.parametrize("W,fk", [(0, 1), (6, 1), (0, 0), (4, 0)])
def test_part_equals_masked_dense(oracle_mod, W, fk):
    """A part is the attention over the visible keys inside its range."""
    rng = np.random.default_rng(700 + W + 10 * fk)
    Hq, Hkv, D, P, K = 4, 2, 8, 4, 3
    lens = [0, 3, 9, 22]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    s = 0.55
    per_req = [_part_ranges(rng, L, K) for L in lens]
    for t in range(len(per_req[0])):
        kb = np.array([r[t][0] for r in per_req], np.int32)
        ke = np.array([r[t][1] for r in per_req], np.int32)
        out, lse2 = oracle_mod.block_attn_part(q, kp, vp, tab, ctx, kb, ke, block_size=K, window=W,
                                               future_keys=fk, scale=s)
        for b, L in enumerate(lens):
            _check_part_against_dense(out[b], lse2[b], q[b], dk[b], dv[b], s, L, K, W, fk, kb[b], ke[b])


@pytest.mark.parametrize("n_parts", [1, 2, 3, 5])
@pytest.mark.parametrize("W", [0, 7])
def test_parts_merge_into_whole_attention(oracle_mod, n_parts, W):
    """Parts that tile [0, L+K), merged by the base-2 LSE combine, give the
    whole attention; the combine agrees with a plain logaddexp2 merge."""
    rng = np.random.default_rng(800 + 11 * n_parts + W)
    Hq, Hkv, D, P, K = 6, 2, 8, 3, 4
    lens = [0, 1, 8, 19, 33]
    q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
    s = 0.5
    full, full_lse = oracle_mod.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=1,
                                           scale=s)
    bounds = []
    for L in lens:
        inner = sorted(int(x) for x in rng.integers(0, L + K + 1, size=n_parts - 1))
        bounds.append([0] + inner + [L + K])
    outs, lses = [], []
    for r in range(n_parts):
        kb = np.array([bd[r] for bd in bounds], np.int32)
        ke = np.array([bd[r + 1] for bd in bounds], np.int32)
        o, l = oracle_mod.block_attn_part(q, kp, vp, tab, ctx, kb, ke, block_size=K, window=W,
                                          future_keys=1, scale=s)
        outs.append(o)
        lses.append(l)
    mo, ml = oracle_mod.combine_parts(np.stack(outs), np.stack(lses))
    np.testing.assert_allclose(mo, full, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ml, full_lse, rtol=1e-12, atol=1e-12)
    # The same merge written with numpy's logaddexp2, part by part.
    acc_l = np.full(full_lse.shape, -np.inf)
    for l in lses:
        acc_l = np.logaddexp2(acc_l, l)
    acc_o = sum(o * np.exp2(l - acc_l)[..., None] for o, l in zip(outs, lses))
    np.testing.assert_allclose(mo, acc_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ml, acc_l, rtol=1e-13, atol=1e-13)


def test_combine_parts_of_nothing_is_empty(oracle_mod):
    out, lse2 = oracle_mod.combine_parts(np.zeros((3, 2, 5, 4)), np.full((3, 2, 5), -np.inf))
    assert np.all(out == 0.0) and np.all(np.isneginf(lse2))


PART_MUTANTS = [
    ("part range end inclusive", "p < pr.key_end[b]", "p <= pr.key_end[b]"),
    ("part range begin exclusive", "p >= pr.key_begin[b]", "p > pr.key_begin[b]"),
    ("merge weights from the max, not the sum", "std::exp2(part_lse2[s * rows + r] - lse)",
     "std::exp2(part_lse2[s * rows + r] - m)"),
    ("merge LSE natural log", "const double lse = m + std::log2(z);", "const double lse = m + std::log(z);"),
]


def _part_pins_pass(lib) -> bool:
    import oracle

    rng = np.random.default_rng(4321)
    try:
        Hq, Hkv, D, P, K, W = 4, 2, 8, 4, 3, 6
        lens = [2, 9, 17]
        q, dk, dv, kp, vp, tab, ctx = make_case(rng, len(lens), Hq, Hkv, D, K, P, lens)
        full, full_lse = oracle.block_attn(q, kp, vp, tab, ctx, block_size=K, window=W, future_keys=1,
                                           scale=0.5, lib=lib)
        mid = np.array([L // 2 + 1 for L in lens], np.int32)
        zero = np.zeros(len(lens), np.int32)
        end = np.array([L + K for L in lens], np.int32)
        o1, l1 = oracle.block_attn_part(q, kp, vp, tab, ctx, zero, mid, block_size=K, window=W,
                                        future_keys=1, scale=0.5, lib=lib)
        o2, l2 = oracle.block_attn_part(q, kp, vp, tab, ctx, mid, end, block_size=K, window=W,
                                        future_keys=1, scale=0.5, lib=lib)
        for b, L in enumerate(lens):
            _check_part_against_dense(o1[b], l1[b], q[b], dk[b], dv[b], 0.5, L, K, W, 1, 0, mid[b],
                                      rtol=1e-10, atol=1e-11)
        mo, ml = oracle.combine_parts(np.stack([o1, o2]), np.stack([l1, l2]), lib=lib)
        if not (np.allclose(mo, full, rtol=1e-10, atol=1e-11) and np.allclose(ml, full_lse, rtol=1e-10,
                                                                              atol=1e-11)):
            return False
    except (ValueError, AssertionError):
        return False
    return True


def test_part_pins_reject_planted_mistakes(oracle_mod, tmp_path):
    import oracle

    src = open(os.path.join(os.path.dirname(oracle.__file__), "dflash_oracle.cpp")).read()
    assert _part_pins_pass(oracle._load()), "the unmodified oracle must pass the part pins"
    for name, old, new in PART_MUTANTS:
        assert src.count(old) == 1, name
        path = tmp_path / (name.replace(" ", "_").replace(",", "") + ".cpp")
        path.write_text(src.replace(old, new))
        so = str(path) + ".so"
        subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(path), "-o", so],
                       check=True)
        assert not _part_pins_pass(oracle.load_library(so)), f"planted mistake not caught: {name}"
