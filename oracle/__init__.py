"""fp64 CPU oracle for paged draft-block attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product library never
imports, links or calls it, and it imports nothing from the product package.

The arithmetic lives in ``dflash_oracle.cpp`` (plain C++, double precision,
one ``std::thread`` worker per host core); this module only compiles it with
the host C++ compiler and marshals numpy arrays.  Semantics (TensorRT-LLM
PR #21130 "Non-causal windowed DSpark draft block", description and change 2;
PR #20374 "Non-causal unwindowed DFlash draft block", description):

* query token ``i`` of request ``b`` (position ``L+i``, ``L = ctx_lens[b]``)
  sees the causal window ``(L+i-W, L+i]`` when ``window = W > 0`` (every
  position up to ``L+i`` when ``W = 0``) plus the later block keys
  ``L+j``, ``i < j <= i+r``, with ``r = K-1`` for ``future_keys=1`` and
  ``r = right_window`` otherwise;
* every key/value row is read through ``page_table`` from HND pages
  ``[num_pages, Hkv, P, D]``; query head ``hq`` reads kv head ``hq // G``;
* ``out`` is the softmax-weighted mean of the visible values and ``lse2`` the
  base-2 log-sum-exp of ``scale * q.k`` over the visible keys.

The dense-suffix form may read fp8 context pages: OCP E4M3 codes with one
dequantisation scale per tensor (``k = k_scale * e4m3(code)``, likewise V;
the bf16 block rows take no scale) -- PR #16150: the drafter's context may
be stored as fp8.

Also the block placement and the K/V append (the block's rows written into
the pool slots of positions ``L .. L+K-1``), plain data movement; and the
context-parallel form: one part of a request's keys (logical positions
``[key_begin[b], key_end[b])``) and the base-2 log-sum-exp merge of parts.

Pinned by ``tests/test_oracle_pins.py`` (dense brute force, causal decode,
LSE merge of disjoint key sets, page-permutation invariance, closed forms,
placement and append round trips, parts against the masked dense attention
and their merge against the whole).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (host C++ only)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle (``liboracle.so`` or a test's variant of it)."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_block_attn
    f.restype = ctypes.c_int
    i32, vp = ctypes.c_int, ctypes.c_void_p
    f.argtypes = [i32] * 11 + [ctypes.c_double] + [vp] * 8 + [i32] + [vp, vp, i32]
    f = lib.oracle_block_attn_fp8
    f.restype = ctypes.c_int
    dbl = ctypes.c_double
    f.argtypes = [i32] * 11 + [dbl] + [vp] * 3 + [dbl, dbl] + [vp] * 5 + [i32] + [vp, vp, i32]
    f = lib.oracle_e4m3_to_double
    f.restype = ctypes.c_double
    f.argtypes = [i32]
    f = lib.oracle_block_placement
    f.restype = ctypes.c_int
    f.argtypes = [i32] * 5 + [vp] * 3
    f = lib.oracle_append_block_kv
    f.restype = ctypes.c_int
    f.argtypes = [i32] * 7 + [vp] * 6
    f = lib.oracle_block_attn_part
    f.restype = ctypes.c_int
    f.argtypes = [i32] * 11 + [dbl] + [vp] * 8 + [i32] + [vp, vp, i32]
    f = lib.oracle_combine_parts
    f.restype = ctypes.c_int
    f.argtypes = [i32, ctypes.c_int64, i32] + [vp] * 4
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def block_attn(q, k_pages, v_pages, page_table, ctx_lens, *, block_size, window, future_keys,
               scale, right_window=0, k_block=None, v_block=None, req_ids=None, nthreads=0,
               lib=None):
    """Return ``(out, lse2)`` in float64 for requests ``req_ids`` (all when None).

    ``q``: uint16 bf16 bits ``[B, K, Hq, D]``; ``k_pages``/``v_pages``: uint16
    ``[num_pages, Hkv, P, D]``; ``page_table``: int32 ``[B, max_pages]``;
    ``ctx_lens``: int32 ``[B]``.  ``out`` is ``[n, K, Hq, D]``, ``lse2``
    ``[n, K, Hq]`` with ``n = len(req_ids)`` (or B).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    B, K, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    if K != block_size or D2 != D or v_pages.shape != k_pages.shape:
        raise ValueError("inconsistent shapes")
    if page_table.shape[0] != B or ctx_lens.shape != (B,):
        raise ValueError("inconsistent batch")
    if (k_block is None) != (v_block is None):
        raise ValueError("k_block and v_block go together")
    if k_block is not None:
        k_block = np.ascontiguousarray(k_block, dtype=np.uint16)
        v_block = np.ascontiguousarray(v_block, dtype=np.uint16)
        if k_block.shape != (B, K, Hkv, D) or v_block.shape != k_block.shape:
            raise ValueError("k_block / v_block must be [B, K, Hkv, D]")
    if req_ids is not None:
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        n = int(req_ids.shape[0])
    else:
        n = B
    out = np.zeros((n, K, Hq, D), dtype=np.float64)
    lse2 = np.zeros((n, K, Hq), dtype=np.float64)
    rc = (lib or _load()).oracle_block_attn(
        B, Hq, Hkv, D, P, page_table.shape[1], num_pages, K, int(window), int(future_keys),
        int(right_window), float(scale), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(ctx_lens),
        _ptr(k_block), _ptr(v_block), _ptr(req_ids), n, _ptr(out), _ptr(lse2), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_block_attn failed with status {rc}")
    return out, lse2


def block_attn_part(q, k_pages, v_pages, page_table, ctx_lens, key_begin, key_end, *, block_size,
                    window, future_keys, scale, right_window=0, req_ids=None, nthreads=0, lib=None):
    """One context-parallel part: ``(out, lse2)`` in float64 over the visible
    keys at logical positions ``[key_begin[b], key_end[b])`` (int32 ``[B]``);
    rows that see none get 0 and -inf.  Arguments as ``block_attn``."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    key_begin = np.ascontiguousarray(key_begin, dtype=np.int32)
    key_end = np.ascontiguousarray(key_end, dtype=np.int32)
    B, K, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    if K != block_size or D2 != D or v_pages.shape != k_pages.shape:
        raise ValueError("inconsistent shapes")
    if page_table.shape[0] != B or ctx_lens.shape != (B,) or key_begin.shape != (B,) or \
            key_end.shape != (B,):
        raise ValueError("inconsistent batch")
    if req_ids is not None:
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        n = int(req_ids.shape[0])
    else:
        n = B
    out = np.zeros((n, K, Hq, D), dtype=np.float64)
    lse2 = np.zeros((n, K, Hq), dtype=np.float64)
    rc = (lib or _load()).oracle_block_attn_part(
        B, Hq, Hkv, D, P, page_table.shape[1], num_pages, K, int(window), int(future_keys),
        int(right_window), float(scale), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
        _ptr(ctx_lens), _ptr(key_begin), _ptr(key_end), _ptr(req_ids), n, _ptr(out), _ptr(lse2),
        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_block_attn_part failed with status {rc}")
    return out, lse2


def combine_parts(part_out, part_lse2, lib=None):
    """Merge of context-parallel parts: ``part_out [n, ..., D]`` and
    ``part_lse2 [n, ...]`` (float64) -> ``(out [..., D], lse2 [...])`` by the
    base-2 log-sum-exp combine."""
    part_out = np.ascontiguousarray(part_out, dtype=np.float64)
    part_lse2 = np.ascontiguousarray(part_lse2, dtype=np.float64)
    n = part_out.shape[0]
    D = part_out.shape[-1]
    if part_lse2.shape != part_out.shape[:-1]:
        raise ValueError("part_lse2 must match part_out without its last axis")
    rows = int(np.prod(part_lse2.shape[1:])) if part_lse2.ndim > 1 else 1
    out = np.zeros(part_out.shape[1:], dtype=np.float64)
    lse2 = np.zeros(part_lse2.shape[1:], dtype=np.float64)
    rc = (lib or _load()).oracle_combine_parts(int(n), rows, int(D), _ptr(part_out), _ptr(part_lse2),
                                               _ptr(out), _ptr(lse2))
    if rc != 0:
        raise ValueError(f"oracle_combine_parts failed with status {rc}")
    return out, lse2


def block_attn_fp8(q, k_pages8, v_pages8, page_table, ctx_lens, *, k_scale, v_scale, k_block,
                   v_block, block_size, window, future_keys, scale, right_window=0, req_ids=None,
                   nthreads=0, lib=None):
    """Dense-suffix form over fp8 context pages; returns ``(out, lse2)`` in float64.

    ``k_pages8``/``v_pages8``: uint8 E4M3 codes ``[num_pages, Hkv, P, D]``
    (positions < ``ctx_lens[b]`` only are read); ``k_scale``/``v_scale``: the
    per-tensor dequantisation scales; ``k_block``/``v_block``: uint16 bf16
    bits ``[B, K, Hkv, D]`` of the block rows.  Other arguments as
    :func:`block_attn`.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages8 = np.ascontiguousarray(k_pages8, dtype=np.uint8)
    v_pages8 = np.ascontiguousarray(v_pages8, dtype=np.uint8)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    k_block = np.ascontiguousarray(k_block, dtype=np.uint16)
    v_block = np.ascontiguousarray(v_block, dtype=np.uint16)
    B, K, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages8.shape
    if K != block_size or D2 != D or v_pages8.shape != k_pages8.shape:
        raise ValueError("inconsistent shapes")
    if page_table.shape[0] != B or ctx_lens.shape != (B,):
        raise ValueError("inconsistent batch")
    if k_block.shape != (B, K, Hkv, D) or v_block.shape != k_block.shape:
        raise ValueError("k_block / v_block must be [B, K, Hkv, D]")
    if req_ids is not None:
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        n = int(req_ids.shape[0])
    else:
        n = B
    out = np.zeros((n, K, Hq, D), dtype=np.float64)
    lse2 = np.zeros((n, K, Hq), dtype=np.float64)
    rc = (lib or _load()).oracle_block_attn_fp8(
        B, Hq, Hkv, D, P, page_table.shape[1], num_pages, K, int(window), int(future_keys),
        int(right_window), float(scale), _ptr(q), _ptr(k_pages8), _ptr(v_pages8), float(k_scale),
        float(v_scale), _ptr(page_table), _ptr(ctx_lens), _ptr(k_block), _ptr(v_block), _ptr(req_ids),
        n, _ptr(out), _ptr(lse2), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_block_attn_fp8 failed with status {rc}")
    return out, lse2


def e4m3_to_float64(codes, lib=None) -> np.ndarray:
    """The oracle's value of each E4M3 code (uint8 array)."""
    codes = np.asarray(codes, dtype=np.uint8)
    f = (lib or _load()).oracle_e4m3_to_double
    return np.array([f(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def block_placement(page_table, ctx_lens, *, block_size, page_size, num_pages, lib=None):
    """int32 ``[B, K, 2]``: (page, offset) of block token j of request b, the
    pool slot of logical position ``ctx_lens[b] + j``."""
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    B, max_pages = page_table.shape
    out = np.zeros((B, block_size, 2), dtype=np.int32)
    rc = (lib or _load()).oracle_block_placement(B, block_size, page_size, max_pages, num_pages,
                                                 _ptr(page_table), _ptr(ctx_lens), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_block_placement failed with status {rc}")
    return out


def append_block_kv(k_block, v_block, k_pages, v_pages, page_table, ctx_lens, lib=None):
    """Copies of the pools with the block's K/V rows (uint16 bf16 bits
    ``[B, K, Hkv, D]``) written at their placement."""
    k_block = np.ascontiguousarray(k_block, dtype=np.uint16)
    v_block = np.ascontiguousarray(v_block, dtype=np.uint16)
    kp = np.array(k_pages, dtype=np.uint16, copy=True)
    vp = np.array(v_pages, dtype=np.uint16, copy=True)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    B, K, Hkv, D = k_block.shape
    num_pages, Hkv2, P, D2 = kp.shape
    if Hkv2 != Hkv or D2 != D or v_block.shape != k_block.shape or vp.shape != kp.shape:
        raise ValueError("inconsistent shapes")
    rc = (lib or _load()).oracle_append_block_kv(B, K, Hkv, D, P, page_table.shape[1], num_pages,
                                                 _ptr(k_block), _ptr(v_block), _ptr(kp), _ptr(vp),
                                                 _ptr(page_table), _ptr(ctx_lens))
    if rc != 0:
        raise ValueError(f"oracle_append_block_kv failed with status {rc}")
    return kp, vp


def bf16_bits_from_float(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the bits.

    Used by tests to build exactly representable inputs; not part of the
    attention arithmetic.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(f)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_float(bits) -> np.ndarray:
    """Widen bf16 bit patterns exactly to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
