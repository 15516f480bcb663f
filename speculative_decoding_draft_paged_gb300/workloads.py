"""Seeded synthetic inputs for paged draft-block attention.

This module only draws numbers and lays out a paged KV pool; it holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Shapes follow the drafter configurations the source pages measure:

* ``tiny``      -- B=1, Hq=4, Hkv=1, D=64, K=3, page 16, context 100, unwindowed.
* ``minimax``   -- Hq=16, Hkv=1, D=128, K in {1,3,7}, W=4096, page 64: the
  MiniMax-M3.1 drafter TP4 rank (PR #21130, per-layer sweep table).
* ``adp``       -- Hq=64, Hkv=4, D=128, K in {3,7}, W=4096, page 64, 1 % of key
  rows scaled by 8: the attention-DP rank of the same sweep.
* ``longctx``   -- Hq/Hkv in {8/2, 12/2}, D=64, K=7, page 32, unwindowed, 32K or
  128K context (PR #20374, kernel-level batch sweep).
* ``ragged``    -- Hq=64, Hkv=16, D=64, K=7, page 32, per-request context
  uniform in [1K, 128K], values N(0, 0.5).

Layouts: ``q [B, K, Hq, D]`` bf16; ``k_pages``/``v_pages`` ``[num_pages, Hkv, P, D]``
bf16 (HND pages); ``page_table [B, max_pages]`` int32 (unused entries -1);
``ctx_lens [B]`` int32 = context tokens before the block.  The block's own K/V
rows sit at positions ``L_b .. L_b+K-1`` of the same pages.  Every request gets
disjoint pages drawn from one random permutation of the pool.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class CaseSpec:
    """Sizes and distribution of one synthetic draft-block attention call."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    K: int
    P: int
    window: int              # 0: unwindowed; W > 0: causal window (L+i-W, L+i]
    future_keys: int         # 1: non-causal block; 0: causal block (+ right_window keys)
    ctx_lens: Sequence[int]  # context tokens before the block, per request
    right_window: int = 0    # with future_keys = 0: later block keys each row sees
    sigma: float = 1.0
    outlier_frac: float = 0.0   # fraction of (token, kv head) key rows scaled by 8
    seed: int = 1001
    extra_pages: int = 0        # unreferenced pool pages (poisoned when poison=True)
    extra_table_slots: int = 0  # unused page-table columns per request
    poison: bool = False        # NaN in every slot no visible position uses
    scale: Optional[float] = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def R(self) -> int:
        return self.G * self.K

    @property
    def softmax_scale(self) -> float:
        s = self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)
        return float(torch.tensor(s, dtype=torch.float32).item())

    def pages_for(self, L: int) -> int:
        return (L + self.K + self.P - 1) // self.P

    @property
    def max_pages(self) -> int:
        return max(self.pages_for(L) for L in self.ctx_lens) + self.extra_table_slots

    @property
    def num_pages(self) -> int:
        return sum(self.pages_for(L) for L in self.ctx_lens) + self.extra_pages

    @property
    def max_ctx_len(self) -> int:
        return max(self.ctx_lens)

    def visible_ctx(self, L: int) -> int:
        """Context keys the union of the block's rows reads (for byte counts)."""
        return min(L, self.window - 1) if self.window > 0 else L

    def kv_bytes(self, ctx_elem_bytes: int = 2) -> int:
        """Algorithmic K+V bytes of one call: each visible row read once; the
        context rows at ``ctx_elem_bytes`` per element (1 for fp8 pages), the
        block rows at 2 (bf16)."""
        return sum(2 * self.Hkv * self.D * (ctx_elem_bytes * self.visible_ctx(L) + 2 * self.K)
                   for L in self.ctx_lens)

    def flops(self) -> int:
        return sum(self.Hkv * (self.visible_ctx(L) + self.K) * 4 * self.R * self.D for L in self.ctx_lens)

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv, "D": self.D,
                "K": self.K, "page": self.P, "window": self.window, "future_keys": self.future_keys,
                "right_window": self.right_window,
                "ctx_min": min(self.ctx_lens), "ctx_max": max(self.ctx_lens), "sigma": self.sigma}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, sigma, seed, device, chunk_elems=1 << 28):
    """N(0, sigma) rounded to bf16, drawn in chunks to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = _gen(seed, device)
    for s in range(0, flat.numel(), chunk_elems):
        n = min(chunk_elems, flat.numel() - s)
        t = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        if sigma != 1.0:
            t.mul_(sigma)
        flat[s:s + n].copy_(t)
    return out


def make_inputs(spec: CaseSpec, device="cpu") -> dict:
    """Draw one call's inputs.  Sub-seeds: q +1, k +2, v +3, pages +4, outliers +5."""
    dev = torch.device(device)
    B, K, Hq, Hkv, D, P = spec.B, spec.K, spec.Hq, spec.Hkv, spec.D, spec.P
    assert len(spec.ctx_lens) == B and Hq % Hkv == 0
    q = _normal_bf16((B, K, Hq, D), spec.sigma, spec.seed * 10 + 1, dev)
    k_pages = _normal_bf16((spec.num_pages, Hkv, P, D), spec.sigma, spec.seed * 10 + 2, dev)
    v_pages = _normal_bf16((spec.num_pages, Hkv, P, D), spec.sigma, spec.seed * 10 + 3, dev)

    perm = torch.randperm(spec.num_pages, generator=_gen(spec.seed * 10 + 4, "cpu"))
    table = torch.full((B, spec.max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, L in enumerate(spec.ctx_lens):
        n = spec.pages_for(L)
        table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n
    ctx = torch.tensor(list(spec.ctx_lens), dtype=torch.int32)

    if spec.outlier_frac > 0:
        # One Bernoulli draw per (page, kv head, slot) key row; scaling by 8 is
        # exact in bf16.
        g = _gen(spec.seed * 10 + 5, dev)
        mask = torch.rand((spec.num_pages, Hkv, P, 1), generator=g, device=dev) < spec.outlier_frac
        k_pages.mul_(torch.where(mask, 8.0, 1.0).to(torch.bfloat16))

    if spec.poison:
        poison_unused_slots(spec, k_pages, v_pages, table)

    return {"q": q, "k_pages": k_pages, "v_pages": v_pages,
            "page_table": table.to(dev), "ctx_lens": ctx.to(dev)}


def poison_unused_slots(spec: CaseSpec, k_pages, v_pages, table) -> None:
    """Write bf16 NaN into every pool slot that no visible key occupies.

    That is the tail of each request's last page (positions >= L+K), the
    unreferenced pages, and -- with a window -- the slots before the earliest
    window start ``max(0, L-W+1)``.  Table entries of pages that hold only
    such positions are set to -1, as a cache that recycles them would.
    """
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=k_pages.device)
    tab = table.clone()
    referenced = set()
    for b, L in enumerate(spec.ctx_lens):
        n = spec.pages_for(L)
        lo = max(0, L - spec.window + 1) if spec.window > 0 else 0
        first = lo // spec.P
        for s in range(first):
            table[b, s] = -1
        for s in range(first, n):
            referenced.add(int(tab[b, s]))
        head = lo - first * spec.P
        if head > 0:
            pg = int(tab[b, first])
            k_pages[pg, :, :head, :] = nan
            v_pages[pg, :, :head, :] = nan
        tail = (L + spec.K) - (n - 1) * spec.P
        if tail < spec.P:
            pg = int(tab[b, n - 1])
            k_pages[pg, :, tail:, :] = nan
            v_pages[pg, :, tail:, :] = nan
    for pg in range(spec.num_pages):
        if pg not in referenced:
            k_pages[pg] = nan
            v_pages[pg] = nan


# --------------------------------------------------------------------------
# Presets for the five drafter configurations.
# --------------------------------------------------------------------------

def tiny(seed: int = 1001, **kw) -> CaseSpec:
    return CaseSpec("tiny", B=1, Hq=4, Hkv=1, D=64, K=3, P=16, window=0, future_keys=1,
                    ctx_lens=[100], seed=seed, **kw)


def minimax(B: int = 64, K: int = 7, L: int = 16384, seed: int = 1002, ctx_lens=None, **kw) -> CaseSpec:
    lens = list(ctx_lens) if ctx_lens is not None else [L] * B
    return CaseSpec(f"minimax_B{B}_K{K}_L{max(lens)}", B=B, Hq=16, Hkv=1, D=128, K=K, P=64,
                    window=4096, future_keys=1, ctx_lens=lens, seed=seed, **kw)


def adp(B: int = 64, K: int = 7, L: int = 16384, seed: int = 1003, ctx_lens=None, **kw) -> CaseSpec:
    lens = list(ctx_lens) if ctx_lens is not None else [L] * B
    return CaseSpec(f"adp_B{B}_K{K}_L{max(lens)}", B=B, Hq=64, Hkv=4, D=128, K=K, P=64,
                    window=4096, future_keys=1, ctx_lens=lens, outlier_frac=0.01, seed=seed, **kw)


def longctx(B: int = 32, L: int = 131072, Hq: int = 8, seed: int = 1004, **kw) -> CaseSpec:
    return CaseSpec(f"longctx_{Hq}x2_B{B}_L{L}", B=B, Hq=Hq, Hkv=2, D=64, K=7, P=32, window=0,
                    future_keys=1, ctx_lens=[L] * B, seed=seed, **kw)


def ragged_lens(B: int, seed: int, lo: int = 1024, hi: int = 131072) -> list:
    g = _gen(seed * 10 + 6, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def ragged(B: int = 256, seed: int = 1005, lo: int = 1024, hi: int = 131072, **kw) -> CaseSpec:
    return CaseSpec(f"ragged_B{B}", B=B, Hq=64, Hkv=16, D=64, K=7, P=32, window=0, future_keys=1,
                    ctx_lens=ragged_lens(B, seed, lo, hi), sigma=0.5, seed=seed, **kw)
