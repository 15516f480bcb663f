"""Test helpers: build paged pools from dense per-request sequences.

Layout only (scatter of contiguous rows into permuted HND pages); no attention
arithmetic lives here.
"""

import numpy as np

import oracle


def random_bf16(rng, shape, sigma=1.0):
    return oracle.bf16_bits_from_float(rng.normal(0.0, sigma, size=shape).astype(np.float32))


def scatter_to_pages(rng, dense_k, dense_v, P, Hkv, D, extra_pages=0, extra_slots=0, fill_bits=0x7FC0,
                     dtype=np.uint16):
    """Scatter per-request dense rows ``[T_b, Hkv, D]`` into shuffled pages.

    Returns ``k_pages, v_pages, page_table`` with every unused slot set to
    ``fill_bits`` (bf16 NaN by default) and unused table entries -1.  ``dtype``
    is the element type of the pools (uint16 bf16 bits, or uint8 fp8 codes).
    """
    B = len(dense_k)
    npg = [(dk.shape[0] + P - 1) // P for dk in dense_k]
    num_pages = sum(npg) + extra_pages
    perm = rng.permutation(num_pages)
    max_pages = max(max(npg), 1) + extra_slots
    table = np.full((B, max_pages), -1, dtype=np.int32)
    kp = np.full((num_pages, Hkv, P, D), fill_bits, dtype=dtype)
    vp = np.full((num_pages, Hkv, P, D), fill_bits, dtype=dtype)
    cur = 0
    for b in range(B):
        T = dense_k[b].shape[0]
        for s in range(npg[b]):
            pg = perm[cur]
            cur += 1
            table[b, s] = pg
            lo, hi = s * P, min(T, (s + 1) * P)
            kp[pg, :, : hi - lo, :] = np.transpose(dense_k[b][lo:hi], (1, 0, 2))
            vp[pg, :, : hi - lo, :] = np.transpose(dense_v[b][lo:hi], (1, 0, 2))
    return kp, vp, table


def permute_pool(rng, k_pages, v_pages, table):
    """Move every physical page to a new slot and remap the table to match."""
    n = k_pages.shape[0]
    perm = rng.permutation(n)          # new position of old page j is perm[j]
    kp = np.empty_like(k_pages)
    vp = np.empty_like(v_pages)
    kp[perm] = k_pages
    vp[perm] = v_pages
    t = table.copy()
    m = t >= 0
    t[m] = perm[t[m]]
    return kp, vp, t
