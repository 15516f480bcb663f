"""Context-parallel split on CPU: the range split and the one exchange.

Two gloo ranks each compute their part of every request's keys with the fp64
oracle, exchange the parts' (out, lse2) through ``exchange_partials`` (the
all-gather the GPU path uses), merge them with the oracle's base-2 LSE
combine, and must recover the whole attention.  The GPU kernels for a part
and for the merge are checked against the oracle in
``tests/test_context_parallel_gpu.py``.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_draft_paged_gb300.context_parallel import split_ranges


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_split_ranges_tile_every_request():
    lens = [0, 1, 5, 100, 7777]
    for world in (1, 2, 3, 8):
        kb, ke = split_ranges(lens, 7, world)
        assert kb.shape == ke.shape == (world, len(lens)) and kb.dtype == np.int32
        for b, L in enumerate(lens):
            assert kb[0, b] == 0 and ke[-1, b] == L + 7
            assert np.all(ke[:-1, b] == kb[1:, b]) and np.all(ke[:, b] >= kb[:, b])
            assert ke[:, b].max() - kb[:, b].min() == L + 7
            sizes = ke[:, b] - kb[:, b]
            assert sizes.max() - sizes.min() <= 1


def _case():
    from tests._paged import random_bf16, scatter_to_pages

    rng = np.random.default_rng(2024)
    B, Hq, Hkv, D, K, P = 3, 8, 2, 16, 4, 8
    lens = [0, 13, 61]
    q = random_bf16(rng, (B, K, Hq, D), 1.0)
    dk = [random_bf16(rng, (L + K, Hkv, D), 1.0) for L in lens]
    dv = [random_bf16(rng, (L + K, Hkv, D), 1.0) for L in lens]
    kp, vp, tab = scatter_to_pages(rng, dk, dv, P, Hkv, D, 2, 1)
    return q, kp, vp, tab, np.asarray(lens, np.int32), K


def _worker(rank, world, port, window, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from speculative_decoding_draft_paged_gb300.context_parallel import exchange_partials

    q, kp, vp, tab, ctx, K = _case()
    kb, ke = split_ranges(ctx, K, world)
    po, pl = oracle.block_attn_part(q, kp, vp, tab, ctx, kb[rank], ke[rank], block_size=K, window=window,
                                    future_keys=1, scale=0.3)
    outs, lses = exchange_partials(torch.from_numpy(po), torch.from_numpy(pl))
    mo, ml = oracle.combine_parts(outs.numpy(), lses.numpy())
    fo, fl = oracle.block_attn(q, kp, vp, tab, ctx, block_size=K, window=window, future_keys=1, scale=0.3)
    results[rank] = (float(np.abs(mo - fo).max()), float(np.abs(ml - fl).max()),
                     float(np.abs(outs[rank].numpy() - po).max()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("window", [0, 9])
def test_two_ranks_recover_the_whole_attention(window):
    import oracle

    oracle.build()
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), window, results), nprocs=world, join=True)
    for r in range(world):
        d_out, d_lse, d_own = results[r]
        assert d_own == 0.0                   # the exchange keeps each part in rank order
        assert d_out < 1e-12 and d_lse < 1e-12
