"""Context-parallel split of one draft-block attention call over ranks.

Every rank holds part of each request's keys.  A part covers the logical key
positions ``[key_begin[b], key_end[b])`` of request ``b``'s ``L_b + K``
positions (context, then the block).  Each rank computes its part
(``dflash_block_attn_partial``: the output normalised over the part's keys
and their base-2 LSE), the ranks exchange the parts' ``(out, lse2)`` in one
all-gather, and each merges them (``dflash_combine_partials``): the base-2
log-sum-exp merge of partial softmax states (TensorRT-LLM PR #21130, change
1), applied across ranks.  With one GPU per rank the exchange is the only
cross-rank step; a rank's page table need only name the pages of its part.
"""

from __future__ import annotations

import numpy as np


def split_ranges(ctx_lens, block_size: int, world_size: int):
    """Cut each request's ``L_b + K`` keys into ``world_size`` contiguous,
    near-equal ranges.  Returns int32 ``key_begin``, ``key_end`` of shape
    ``[world_size, B]``: rank ``r`` takes ``[key_begin[r], key_end[r])``; the
    ranges of the ranks tile ``[0, L_b + K)``."""
    if world_size < 1:
        raise ValueError("world_size must be at least 1")
    total = np.asarray(ctx_lens, dtype=np.int64) + int(block_size)
    cuts = (total[None, :] * np.arange(world_size + 1, dtype=np.int64)[:, None]) // world_size
    return cuts[:-1].astype(np.int32), cuts[1:].astype(np.int32)


def exchange_partials(part_out, part_lse2, group=None):
    """The one exchange: all-gather the parts' ``(out, lse2)`` over ``group``.

    Returns ``[world, *part_out.shape]`` and ``[world, *part_lse2.shape]``
    tensors, rank order, as ``combine_partials`` takes them."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    outs = [torch.empty_like(part_out) for _ in range(world)]
    lses = [torch.empty_like(part_lse2) for _ in range(world)]
    dist.all_gather(outs, part_out.contiguous(), group=group)
    dist.all_gather(lses, part_lse2.contiguous(), group=group)
    return torch.stack(outs), torch.stack(lses)


def block_attn_context_parallel(q, k_pages, v_pages, page_table, ctx_lens, key_begin, key_end, *,
                                group=None, **kw):
    """This rank's part, the exchange, and the merge: every rank returns the
    whole call's ``(out, lse2)``.  ``key_begin``/``key_end`` are this rank's
    int32 ``[B]`` device tensors (see ``split_ranges``); other keyword
    arguments as ``block_attn``."""
    from . import block_attn_partial, combine_partials

    part_out, part_lse2 = block_attn_partial(q, k_pages, v_pages, page_table, ctx_lens, key_begin, key_end,
                                             **kw)
    outs, lses = exchange_partials(part_out, part_lse2, group=group)
    return combine_partials(outs, lses)
