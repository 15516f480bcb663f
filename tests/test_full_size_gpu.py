"""Full-size parity: every point of the five drafter configurations, in the
launch configuration the benchmark times (the planner's choice of kernel and
split), against the fp64 oracle.

Where the oracle would take long over the whole batch, a seeded sample of
requests (always the shortest, the longest, the first and the last) is
compared: their pages are copied to the host through the page table.
Shapes (the five configurations of the benchmark):
* windowed 16/1 heads, D=128, W=4096, page 64: K in {1,3,7} x B in {1,8,64}
  x L in {2K, 8K, 16K} -- every row compared;
* windowed 64/4 heads, D=128, W=4096, page 64, 1 % of key rows x8 (the
  outliers stress the LSE bound): K in {3,7} x B in {1,8,16,64} x L in
  {2K, 8K, 16K} -- every row up to 16 requests, 10+ sampled at 64;
* unwindowed 8/2 and 12/2 heads, D=64, page 32: L in {32K, 128K} x B in
  {1,2,4,8,16,32} -- three requests sampled per point;
* ragged 64/16 heads, D=64, page 32, contexts uniform in [1K, 128K]: B in
  {64, 128, 256} -- twelve requests sampled per batch.
"""

import numpy as np
import pytest
import torch

from speculative_decoding_draft_paged_gb300 import workloads as W
from tests._gpu_cases import assert_parity, compact_requests, metrics, run_lib, run_oracle

pytestmark = pytest.mark.gpu


def sampled_check(spec, device, n_random=None, seed=0):
    """Runs the whole batch on the GPU; compares every request (n_random is
    None) or the shortest, longest, first, last and n_random seeded others."""
    inp = W.make_inputs(spec, device)
    out, lse = run_lib(spec, inp)
    torch.cuda.synchronize()
    if n_random is None or n_random + 4 >= spec.B:
        ids = list(range(spec.B))
    else:
        lens = np.asarray(spec.ctx_lens)
        rng = np.random.default_rng(seed)
        ids = sorted(set([int(lens.argmin()), int(lens.argmax()), 0, spec.B - 1] +
                         rng.choice(spec.B, n_random, replace=False).tolist()))
    sub = compact_requests(inp, ids) if len(ids) < spec.B else {k: v.cpu() for k, v in inp.items()}
    ro, rl = run_oracle(spec, sub)
    m = metrics(out[ids], lse[ids], ro, rl)
    del inp, out, lse
    torch.cuda.empty_cache()
    assert_parity(m, f"{spec.name} ({len(ids)} of {spec.B} requests)")


@pytest.mark.parametrize("L", [2048, 8192, 16384])
@pytest.mark.parametrize("B", [1, 8, 64])
@pytest.mark.parametrize("K", [1, 3, 7])
def test_full_minimax(cuda_device, K, B, L):
    sampled_check(W.minimax(B=B, K=K, L=L), cuda_device)


@pytest.mark.parametrize("L", [2048, 8192, 16384])
@pytest.mark.parametrize("B", [1, 8, 16, 64])
@pytest.mark.parametrize("K", [3, 7])
def test_full_adp_with_outliers(cuda_device, K, B, L):
    sampled_check(W.adp(B=B, K=K, L=L), cuda_device, n_random=None if B <= 16 else 8, seed=K * L + B)


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("L", [32768, 131072])
@pytest.mark.parametrize("Hq", [8, 12])
def test_full_longctx(cuda_device, Hq, L, B):
    sampled_check(W.longctx(B=B, L=L, Hq=Hq), cuda_device, n_random=1, seed=Hq + B)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_full_ragged(cuda_device, B):
    sampled_check(W.ragged(B=B), cuda_device, n_random=8, seed=5 + B)
