"""Paged draft-block attention for block speculative decoding on GB300.

Thin Python binding over the C ABI of ``include/dflash.h`` (``libdflash.so``):
it marshals torch tensors' device pointers and the current stream; every step
of the computation runs in the library's CUDA kernels.  torch is used for
device memory and streams only.

    out, lse2 = block_attn(q, k_pages, v_pages, page_table, ctx_lens,
                           block_size=K, window=W, future_keys=1, scale=s,
                           max_ctx_len=Lmax)
"""

from __future__ import annotations

import ctypes
from typing import Optional

from . import _lib
from ._lib import (DFLASH_ERR_DEVICE, DFLASH_ERR_INVALID, DFLASH_ERR_LAUNCH, DFLASH_ERR_WORKSPACE,
                   DFLASH_OK, DFLASH_STATUS_BAD_CTX_LEN, DFLASH_STATUS_BAD_PAGE,
                   DFLASH_STATUS_TIMEOUT, DFLASH_STATUS_FP8_RANGE, DFLASH_TEST_WITHHOLD_LOADS, KV_BF16, KV_FP8_E4M3, PATH_AUTO, PATH_MMA, PATH_TCGEN05,
                   Params, PlanInfo)

__all__ = [
    "Params", "PlanInfo", "DflashError", "make_params", "workspace_size", "plan", "block_attn",
    "block_attn_raw", "block_attn_timed_raw", "read_device_status", "clear_device_status", "version", "PATH_AUTO",
    "block_placement", "append_block_kv", "block_attn_append", "block_attn_append_raw",
    "block_attn_dense_suffix", "block_attn_dense_suffix_raw",
    "block_attn_fp8_context", "block_attn_fp8_context_raw", "block_attn_fp8_context_timed_raw",
    "partial_workspace_size", "block_attn_partial", "combine_partials",
    "KV_BF16", "KV_FP8_E4M3",
    "PATH_MMA", "PATH_TCGEN05", "DFLASH_OK", "DFLASH_ERR_INVALID", "DFLASH_ERR_WORKSPACE",
    "DFLASH_ERR_DEVICE", "DFLASH_ERR_LAUNCH", "DFLASH_STATUS_BAD_PAGE",
    "DFLASH_STATUS_BAD_CTX_LEN", "DFLASH_STATUS_TIMEOUT", "DFLASH_STATUS_FP8_RANGE",
    "DFLASH_TEST_WITHHOLD_LOADS",
]


class DflashError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"dflash_block_attn: {_lib.status_string(code)} ({code})")


def make_params(*, batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_req,
                num_pages, block_size, window, future_keys, scale, max_ctx_len, force_path=0,
                force_split_tiles=0, right_window=0, kv_dtype=0, test_flags=0) -> Params:
    p = Params()
    p.batch = batch
    p.num_q_heads = num_q_heads
    p.num_kv_heads = num_kv_heads
    p.head_dim = head_dim
    p.page_size = page_size
    p.max_pages_per_req = max_pages_per_req
    p.num_pages = num_pages
    p.block_size = block_size
    p.window = window
    p.future_keys = future_keys
    p.scale = scale
    p.max_ctx_len = max_ctx_len
    p.force_path = force_path
    p.force_split_tiles = force_split_tiles
    p.right_window = right_window
    p.kv_dtype = kv_dtype
    p.test_flags = test_flags
    return p


def params_for(q, k_pages, page_table, *, block_size, window, future_keys, scale, max_ctx_len,
               force_path=0, force_split_tiles=0, right_window=0, kv_dtype=0, test_flags=0) -> Params:
    B, K, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    if K != block_size:
        raise ValueError(f"q has {K} block tokens, block_size is {block_size}")
    return make_params(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                       max_pages_per_req=page_table.shape[1], num_pages=num_pages,
                       block_size=block_size, window=window, future_keys=future_keys, scale=scale,
                       max_ctx_len=max_ctx_len, force_path=force_path,
                       force_split_tiles=force_split_tiles, right_window=right_window,
                       kv_dtype=kv_dtype, test_flags=test_flags)


def workspace_size(p: Params) -> int:
    return int(_lib.load().dflash_workspace_size(ctypes.byref(p)))


def plan(p: Params) -> dict:
    info = PlanInfo()
    rc = _lib.load().dflash_plan(ctypes.byref(p), ctypes.byref(info))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_ if f != "reserved"}


def version() -> int:
    return int(_lib.load().dflash_version())


def _stream_handle(stream) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def block_attn_raw(p: Params, q_ptr, k_ptr, v_ptr, table_ptr, lens_ptr, out_ptr, lse_ptr, ws_ptr,
                   ws_bytes, stream_handle) -> int:
    """Direct C-ABI call with integer device pointers; returns the status code."""
    return int(_lib.load().dflash_block_attn(ctypes.byref(p), q_ptr, k_ptr, v_ptr, table_ptr,
                                             lens_ptr, out_ptr, lse_ptr, ws_ptr, ws_bytes,
                                             stream_handle))


def block_attn_timed_raw(p: Params, q_ptr, k_ptr, v_ptr, table_ptr, lens_ptr, out_ptr, lse_ptr,
                         ws_ptr, ws_bytes, stream_handle, start_event, done_event) -> int:
    """C-ABI call that records ``start_event``/``done_event`` (torch.cuda.Event)
    around the split kernel; returns the status code."""
    return int(_lib.load().dflash_block_attn_timed(
        ctypes.byref(p), q_ptr, k_ptr, v_ptr, table_ptr, lens_ptr, out_ptr, lse_ptr, ws_ptr,
        ws_bytes, stream_handle, start_event.cuda_event, done_event.cuda_event))


def block_attn(q, k_pages, v_pages, page_table, ctx_lens, *, block_size: int, window: int,
               future_keys: int, scale: float, max_ctx_len: int, out=None, lse2=None,
               workspace=None, stream=None, force_path: int = 0, force_split_tiles: int = 0,
               right_window: int = 0, test_flags: int = 0):
    """Draft-block attention over a paged bf16 KV cache.  Returns ``(out, lse2)``.

    ``q [B,K,Hq,D]`` bf16, ``k_pages``/``v_pages [num_pages,Hkv,P,D]`` bf16,
    ``page_table [B,max_pages]`` int32, ``ctx_lens [B]`` int32 (device),
    all contiguous on the current CUDA device.  ``out``/``lse2``/``workspace``
    are allocated when not given (``workspace``: uint8, ``workspace_size``
    bytes).
    """
    import torch

    p = params_for(q, k_pages, page_table, block_size=block_size, window=window,
                   future_keys=future_keys, scale=scale, max_ctx_len=max_ctx_len,
                   force_path=force_path, force_split_tiles=force_split_tiles,
                   right_window=right_window, test_flags=test_flags)
    for name, t, dt in (("q", q, torch.bfloat16), ("k_pages", k_pages, torch.bfloat16),
                        ("v_pages", v_pages, torch.bfloat16), ("page_table", page_table, torch.int32),
                        ("ctx_lens", ctx_lens, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages differ in shape")
    if out is None:
        out = torch.empty_like(q)
    if lse2 is None:
        lse2 = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        raise DflashError(DFLASH_ERR_INVALID)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    rc = block_attn_raw(p, q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                        page_table.data_ptr(), ctx_lens.data_ptr(), out.data_ptr(),
                        lse2.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return out, lse2


def partial_workspace_size(p: Params) -> int:
    """Workspace bytes of ``block_attn_partial`` for ``p`` (0: invalid)."""
    return int(_lib.load().dflash_partial_workspace_size(ctypes.byref(p)))


def block_attn_partial(q, k_pages, v_pages, page_table, ctx_lens, key_begin, key_end, *, block_size: int,
                       window: int, future_keys: int, scale: float, max_ctx_len: int, right_window: int = 0,
                       part_out=None, part_lse2=None, workspace=None, stream=None, force_split_tiles: int = 0):
    """One context-parallel part: the attention over the keys at logical
    positions ``[key_begin[b], key_end[b])`` (int32 ``[B]`` device tensors) of
    each request's ``L + K`` positions.  Returns ``(part_out, part_lse2)``,
    fp32 ``[B,K,Hq,D]`` and ``[B,K,Hq]``; other arguments as ``block_attn``."""
    import torch

    p = params_for(q, k_pages, page_table, block_size=block_size, window=window,
                   future_keys=future_keys, scale=scale, max_ctx_len=max_ctx_len,
                   force_split_tiles=force_split_tiles, right_window=right_window)
    for name, t, dt in (("q", q, torch.bfloat16), ("k_pages", k_pages, torch.bfloat16),
                        ("v_pages", v_pages, torch.bfloat16), ("page_table", page_table, torch.int32),
                        ("ctx_lens", ctx_lens, torch.int32), ("key_begin", key_begin, torch.int32),
                        ("key_end", key_end, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if part_out is None:
        part_out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if part_lse2 is None:
        part_lse2 = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    need = partial_workspace_size(p)
    if need == 0:
        raise DflashError(DFLASH_ERR_INVALID)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    rc = _lib.load().dflash_block_attn_partial(
        ctypes.byref(p), q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), page_table.data_ptr(),
        ctx_lens.data_ptr(), key_begin.data_ptr(), key_end.data_ptr(), part_out.data_ptr(),
        part_lse2.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return part_out, part_lse2


def combine_partials(part_out, part_lse2, *, out=None, lse2=None, stream=None):
    """Merge of ``n`` parts: ``part_out [n,B,K,Hq,D]`` and ``part_lse2
    [n,B,K,Hq]`` (fp32, contiguous, CUDA) -> ``(out bf16 [B,K,Hq,D], lse2 fp32
    [B,K,Hq])``."""
    import torch

    if part_out.dtype != torch.float32 or part_lse2.dtype != torch.float32 or not part_out.is_cuda:
        raise ValueError("part_out / part_lse2 must be fp32 CUDA tensors")
    if part_out.dim() != 5 or part_lse2.shape != part_out.shape[:4]:
        raise ValueError("part_out [n,B,K,Hq,D] and part_lse2 [n,B,K,Hq] expected")
    part_out = part_out.contiguous()
    part_lse2 = part_lse2.contiguous()
    n, B, K, Hq, D = part_out.shape
    p = make_params(batch=B, num_q_heads=Hq, num_kv_heads=1, head_dim=D, page_size=16, max_pages_per_req=K,
                    num_pages=1, block_size=K, window=0, future_keys=1, scale=1.0, max_ctx_len=0)
    if out is None:
        out = torch.empty((B, K, Hq, D), dtype=torch.bfloat16, device=part_out.device)
    if lse2 is None:
        lse2 = torch.empty((B, K, Hq), dtype=torch.float32, device=part_out.device)
    rc = _lib.load().dflash_combine_partials(ctypes.byref(p), int(n), part_out.data_ptr(), part_lse2.data_ptr(),
                                             out.data_ptr(), lse2.data_ptr(), _stream_handle(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return out, lse2


def _check_block(name, t, q_like):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if tuple(t.shape) != tuple(q_like):
        raise ValueError(f"{name} must have shape {tuple(q_like)}")


def _params_from_pool(k_pages, page_table, ctx_lens, *, block_size, max_ctx_len, Hq=None):
    num_pages, Hkv, P, D = k_pages.shape
    B = ctx_lens.shape[0]
    return make_params(batch=B, num_q_heads=Hq or Hkv, num_kv_heads=Hkv, head_dim=D, page_size=P,
                       max_pages_per_req=page_table.shape[1], num_pages=num_pages,
                       block_size=block_size, window=0, future_keys=1, scale=1.0,
                       max_ctx_len=max_ctx_len)


def block_placement(page_table, ctx_lens, k_pages, *, block_size: int, max_ctx_len: int,
                    workspace=None, stream=None):
    """int32 ``[B, K, 2]`` (page, offset) of every block token's K/V slot."""
    import torch

    p = _params_from_pool(k_pages, page_table, ctx_lens, block_size=block_size,
                          max_ctx_len=max_ctx_len)
    placement = torch.empty((ctx_lens.shape[0], block_size, 2), dtype=torch.int32,
                            device=page_table.device)
    rc = int(_lib.load().dflash_block_placement(
        ctypes.byref(p), page_table.data_ptr(), ctx_lens.data_ptr(), placement.data_ptr(),
        workspace.data_ptr() if workspace is not None else None, _stream_handle(stream)))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return placement


def append_block_kv(k_block, v_block, k_pages, v_pages, page_table, ctx_lens, *, max_ctx_len: int,
                    workspace=None, stream=None):
    """Write the block's K/V rows ``[B, K, Hkv, D]`` into their page slots, in place."""
    B, K, Hkv, D = k_block.shape
    _check_block("k_block", k_block, (B, K, Hkv, D))
    _check_block("v_block", v_block, (B, K, Hkv, D))
    p = _params_from_pool(k_pages, page_table, ctx_lens, block_size=K, max_ctx_len=max_ctx_len)
    rc = int(_lib.load().dflash_append_block_kv(
        ctypes.byref(p), k_block.data_ptr(), v_block.data_ptr(), k_pages.data_ptr(),
        v_pages.data_ptr(), page_table.data_ptr(), ctx_lens.data_ptr(),
        workspace.data_ptr() if workspace is not None else None, _stream_handle(stream)))
    if rc != DFLASH_OK:
        raise DflashError(rc)


def block_attn_append_raw(p: Params, q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, table_ptr, lens_ptr,
                          out_ptr, lse_ptr, ws_ptr, ws_bytes, stream_handle) -> int:
    """Direct C-ABI call of the fused append + attention; returns the status code."""
    return int(_lib.load().dflash_block_attn_append(ctypes.byref(p), q_ptr, kb_ptr, vb_ptr, k_ptr,
                                                    v_ptr, table_ptr, lens_ptr, out_ptr, lse_ptr,
                                                    ws_ptr, ws_bytes, stream_handle))


def block_attn_append(q, k_block, v_block, k_pages, v_pages, page_table, ctx_lens, *,
                      block_size: int, window: int, future_keys: int, scale: float,
                      max_ctx_len: int, out=None, lse2=None, workspace=None, stream=None,
                      force_path: int = 0, right_window: int = 0):
    """Append the block's K/V to the pages, then the attention (one launch
    sequence).  Returns ``(out, lse2)``; the pools are updated in place."""
    import torch

    B, K, Hq, D = q.shape
    _check_block("k_block", k_block, (B, K, k_pages.shape[1], D))
    _check_block("v_block", v_block, (B, K, k_pages.shape[1], D))
    p = params_for(q, k_pages, page_table, block_size=block_size, window=window,
                   future_keys=future_keys, scale=scale, max_ctx_len=max_ctx_len,
                   force_path=force_path, right_window=right_window)
    if out is None:
        out = torch.empty_like(q)
    if lse2 is None:
        lse2 = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        raise DflashError(DFLASH_ERR_INVALID)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    rc = block_attn_append_raw(p, q.data_ptr(), k_block.data_ptr(), v_block.data_ptr(),
                               k_pages.data_ptr(), v_pages.data_ptr(), page_table.data_ptr(),
                               ctx_lens.data_ptr(), out.data_ptr(), lse2.data_ptr(),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_handle(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return out, lse2


def block_attn_dense_suffix_raw(p: Params, q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, table_ptr, lens_ptr,
                                out_ptr, lse_ptr, ws_ptr, ws_bytes, stream_handle) -> int:
    """Direct C-ABI call of the dense-suffix form; returns the status code."""
    return int(_lib.load().dflash_block_attn_dense_suffix(
        ctypes.byref(p), q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, table_ptr, lens_ptr, out_ptr, lse_ptr,
        ws_ptr, ws_bytes, stream_handle))


def block_attn_dense_suffix(q, k_block, v_block, k_pages, v_pages, page_table, ctx_lens, *,
                            block_size: int, window: int, future_keys: int, scale: float,
                            max_ctx_len: int, out=None, lse2=None, workspace=None, stream=None,
                            force_path: int = 0, force_split_tiles: int = 0,
                            right_window: int = 0):
    """Attention with the block's K/V rows ``[B, K, Hkv, D]`` from dense
    tensors and the context from the pages.  Returns ``(out, lse2)``."""
    import torch

    B, K, Hq, D = q.shape
    _check_block("k_block", k_block, (B, K, k_pages.shape[1], D))
    _check_block("v_block", v_block, (B, K, k_pages.shape[1], D))
    p = params_for(q, k_pages, page_table, block_size=block_size, window=window,
                   future_keys=future_keys, scale=scale, max_ctx_len=max_ctx_len,
                   force_path=force_path, force_split_tiles=force_split_tiles,
                   right_window=right_window)
    if out is None:
        out = torch.empty_like(q)
    if lse2 is None:
        lse2 = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        raise DflashError(DFLASH_ERR_INVALID)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    rc = block_attn_dense_suffix_raw(p, q.data_ptr(), k_block.data_ptr(), v_block.data_ptr(),
                                     k_pages.data_ptr(), v_pages.data_ptr(), page_table.data_ptr(),
                                     ctx_lens.data_ptr(), out.data_ptr(), lse2.data_ptr(),
                                     workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     _stream_handle(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return out, lse2


def block_attn_fp8_context_raw(p: Params, q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, k_scale, v_scale,
                               table_ptr, lens_ptr, out_ptr, lse_ptr, ws_ptr, ws_bytes,
                               stream_handle) -> int:
    """Direct C-ABI call of the fp8-context form; returns the status code."""
    return int(_lib.load().dflash_block_attn_fp8_context(
        ctypes.byref(p), q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, float(k_scale), float(v_scale),
        table_ptr, lens_ptr, out_ptr, lse_ptr, ws_ptr, ws_bytes, stream_handle))


def block_attn_fp8_context_timed_raw(p: Params, q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, k_scale, v_scale,
                                     table_ptr, lens_ptr, out_ptr, lse_ptr, ws_ptr, ws_bytes,
                                     stream_handle, split_start=None, split_done=None) -> int:
    """The fp8-context call with timing marks (torch.cuda.Event or None)."""
    def handle(e):
        return None if e is None else ctypes.c_void_p(e.cuda_event)

    return int(_lib.load().dflash_block_attn_fp8_context_timed(
        ctypes.byref(p), q_ptr, kb_ptr, vb_ptr, k_ptr, v_ptr, float(k_scale), float(v_scale),
        table_ptr, lens_ptr, out_ptr, lse_ptr, ws_ptr, ws_bytes, stream_handle, handle(split_start),
        handle(split_done)))


def block_attn_fp8_context(q, k_block, v_block, k_pages, v_pages, page_table, ctx_lens, *,
                           k_scale: float, v_scale: float, block_size: int, window: int,
                           future_keys: int, scale: float, max_ctx_len: int, out=None, lse2=None,
                           workspace=None, stream=None, force_path: int = 0, force_split_tiles: int = 0,
                           right_window: int = 0):
    """Dense-suffix form over fp8 context pages: ``k_pages``/``v_pages`` are
    uint8 E4M3 codes ``[num_pages, Hkv, P, D]`` dequantised by the per-tensor
    scales; the block rows ``[B, K, Hkv, D]`` are bf16.  Returns ``(out, lse2)``."""
    import torch

    B, K, Hq, D = q.shape
    if k_pages.dtype != torch.uint8 or v_pages.dtype != torch.uint8:
        raise ValueError("fp8 pages are uint8 E4M3 codes")
    _check_block("k_block", k_block, (B, K, k_pages.shape[1], D))
    _check_block("v_block", v_block, (B, K, k_pages.shape[1], D))
    p = params_for(q, k_pages, page_table, block_size=block_size, window=window,
                   future_keys=future_keys, scale=scale, max_ctx_len=max_ctx_len,
                   force_path=force_path, force_split_tiles=force_split_tiles,
                   right_window=right_window, kv_dtype=KV_FP8_E4M3)
    if out is None:
        out = torch.empty_like(q)
    if lse2 is None:
        lse2 = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        raise DflashError(DFLASH_ERR_INVALID)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    rc = block_attn_fp8_context_raw(p, q.data_ptr(), k_block.data_ptr(), v_block.data_ptr(),
                                    k_pages.data_ptr(), v_pages.data_ptr(), k_scale, v_scale,
                                    page_table.data_ptr(), ctx_lens.data_ptr(), out.data_ptr(),
                                    lse2.data_ptr(), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream))
    if rc != DFLASH_OK:
        raise DflashError(rc)
    return out, lse2


def read_device_status(workspace, stream=None) -> int:
    rc = int(_lib.load().dflash_read_device_status(workspace.data_ptr(), _stream_handle(stream)))
    if rc < 0:
        raise DflashError(rc)
    return rc


def clear_device_status(workspace, stream=None) -> None:
    rc = int(_lib.load().dflash_clear_device_status(workspace.data_ptr(), _stream_handle(stream)))
    if rc != DFLASH_OK:
        raise DflashError(rc)
