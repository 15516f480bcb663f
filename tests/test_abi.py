"""Host-side checks of the C ABI: exports, struct layout, validation, planner.

No kernel is launched here; these run without a GPU.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(dflash_lib):
    from speculative_decoding_draft_paged_gb300 import _lib

    lib = ctypes.CDLL(_lib.library_path())
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dflash.h but not exported"
    assert set(names) == set(_lib.EXPORTS)


def test_header_constants_match_binding():
    """Every status, error, path and pool-type constant of dflash.h has the
    same value in the Python binding."""
    from speculative_decoding_draft_paged_gb300 import _lib

    defs = dict((n, int(v)) for n, v in re.findall(r"#define\s+(DFLASH_[A-Z0-9_]+)\s+(-?\d+)", open(HEADER).read()))
    assert "DFLASH_STATUS_FP8_RANGE" in defs
    alias = {"DFLASH_PATH_": "PATH_", "DFLASH_KV_": "KV_"}
    for n, v in defs.items():
        py = n
        for pre, rep in alias.items():
            if n.startswith(pre):
                py = rep + n[len(pre):]
        if n == "DFLASH_VERSION" or not hasattr(_lib, py):
            assert n.startswith(("DFLASH_VERSION", "DFLASH_MAX")), f"{n} has no binding constant"
            continue
        assert getattr(_lib, py) == v, n


def test_struct_layout_matches_header(dflash_lib, tmp_path):
    """Compile a C program against the header and compare sizes/offsets."""
    from speculative_decoding_draft_paged_gb300 import _lib

    prog = tmp_path / "layout.c"
    fields_p = [f for f, _ in _lib.Params._fields_]
    fields_i = [f for f, _ in _lib.PlanInfo._fields_]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dflash.h"', "int main(void){",
             'printf("%zu\\n", sizeof(dflash_params));',
             'printf("%zu\\n", sizeof(dflash_plan_info));']
    lines += [f'printf("%zu\\n", offsetof(dflash_params, {f}));' for f in fields_p]
    lines += [f'printf("%zu\\n", offsetof(dflash_plan_info, {f}));' for f in fields_i]
    lines += ["return 0;}"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(_lib.Params)
    assert vals[1] == ctypes.sizeof(_lib.PlanInfo)
    off = vals[2:]
    assert off[: len(fields_p)] == [getattr(_lib.Params, f).offset for f in fields_p]
    assert off[len(fields_p):] == [getattr(_lib.PlanInfo, f).offset for f in fields_i]


def base_params(**kw):
    import speculative_decoding_draft_paged_gb300 as d

    args = dict(batch=4, num_q_heads=16, num_kv_heads=2, head_dim=64, page_size=32,
                max_pages_per_req=40, num_pages=200, block_size=7, window=0, future_keys=1,
                scale=0.125, max_ctx_len=1200)
    args.update(kw)
    return d.make_params(**args)


@pytest.mark.parametrize("bad", [
    dict(batch=0), dict(num_kv_heads=0), dict(num_q_heads=12, num_kv_heads=5),
    dict(head_dim=96), dict(head_dim=256), dict(page_size=8), dict(page_size=48),
    dict(block_size=0), dict(block_size=17), dict(num_q_heads=64, num_kv_heads=2, block_size=5),
    dict(window=-1), dict(future_keys=2), dict(scale=float("inf")),
    dict(future_keys=0, right_window=-1), dict(future_keys=0, right_window=7),
    dict(future_keys=1, right_window=2),
    dict(scale=float("nan")), dict(scale=0.0), dict(scale=-0.125), dict(max_ctx_len=-1), dict(max_ctx_len=40 * 32 - 6),
    dict(num_pages=0), dict(force_path=3), dict(force_split_tiles=-1), dict(force_split_tiles=257),
    dict(kv_dtype=2), dict(kv_dtype=-1), dict(test_flags=2), dict(test_flags=-1),
])
def test_invalid_params_rejected(dflash_lib, bad):
    d = dflash_lib
    p = base_params(**bad)
    assert d.workspace_size(p) == 0
    with pytest.raises(d.DflashError) as e:
        d.plan(p)
    assert e.value.code == d.DFLASH_ERR_INVALID
    rc = d.block_attn_raw(p, 16, 16, 16, 16, 16, 16, 16, 256, 1 << 30, 0)
    assert rc == d.DFLASH_ERR_INVALID


def test_reserved_must_be_zero(dflash_lib):
    p = base_params()
    p.reserved[0] = 1
    assert dflash_lib.workspace_size(p) == 0


def test_boundary_params_accepted(dflash_lib):
    d = dflash_lib
    for kw in [dict(max_ctx_len=40 * 32 - 7), dict(window=7), dict(window=4096), dict(window=3),
               dict(window=1), dict(future_keys=0, right_window=6), dict(future_keys=0, right_window=2),
               dict(num_q_heads=128, num_kv_heads=8, block_size=8), dict(block_size=1, window=1),
               dict(head_dim=128, page_size=64, max_pages_per_req=30), dict(page_size=16,
                                                                            max_pages_per_req=90)]:
        assert d.workspace_size(base_params(**kw)) > 0, kw


def test_null_and_misaligned_pointers_rejected(dflash_lib):
    d = dflash_lib
    p = base_params()
    ws = d.workspace_size(p)
    good = [1 << 20] * 8
    for i in range(8):
        ptrs = list(good)
        ptrs[i] = 0
        assert d.block_attn_raw(p, *ptrs, ws, 0) == d.DFLASH_ERR_INVALID
    for i, off in [(0, 8), (1, 2), (2, 4), (3, 2), (4, 1), (5, 8), (6, 2), (7, 128)]:
        ptrs = list(good)
        ptrs[i] += off
        assert d.block_attn_raw(p, *ptrs, ws, 0) == d.DFLASH_ERR_INVALID


def test_fp8_context_plan_and_validation(dflash_lib):
    """fp8 pools take the path bf16 pools would (the mma.sync plan also needs
    room for its code ring: R = 128 at D = 128 forced onto it is refused);
    the fp8 entry point takes fp8 parameters and positive finite scales only,
    and the bf16 entry points refuse fp8 parameters (all checked before any
    device is touched)."""
    d = dflash_lib
    p8 = base_params(kv_dtype=d.KV_FP8_E4M3, num_q_heads=4, num_kv_heads=2, block_size=3)
    assert d.plan(p8)["path"] == d.PATH_MMA
    assert d.plan(base_params(num_q_heads=4, num_kv_heads=2, block_size=3))["path"] == d.PATH_MMA
    big = dict(head_dim=128, page_size=64, num_q_heads=16, num_kv_heads=1, block_size=8, max_pages_per_req=30,
               batch=64)
    assert d.plan(base_params(kv_dtype=d.KV_FP8_E4M3, **big))["path"] == d.PATH_TCGEN05
    few = dict(big, batch=8, block_size=7)  # R = 112 over 8 pairs: mma.sync for both pool types
    assert d.plan(base_params(**few))["path"] == d.PATH_MMA
    assert d.plan(base_params(kv_dtype=d.KV_FP8_E4M3, **few))["path"] == d.PATH_MMA
    for path in (d.PATH_MMA, d.PATH_TCGEN05):
        assert d.workspace_size(base_params(kv_dtype=d.KV_FP8_E4M3, force_path=path)) > 0
    ws = d.workspace_size(p8)
    assert ws > 0
    ptr = 1 << 20
    args = [ptr] * 5
    tail = [ptr, ptr, ptr, ptr, ptr, ws, 0]
    for ks, vs in [(0.0, 1.0), (1.0, -2.0), (float("nan"), 1.0), (1.0, float("inf"))]:
        assert d.block_attn_fp8_context_raw(p8, *args, ks, vs, *tail) == d.DFLASH_ERR_INVALID
    p16 = base_params()
    assert d.block_attn_fp8_context_raw(p16, *args, 1.0, 1.0, *tail) == d.DFLASH_ERR_INVALID
    assert d.block_attn_raw(p8, *[ptr] * 8, ws, 0) == d.DFLASH_ERR_INVALID
    assert d.block_attn_dense_suffix_raw(p8, *[ptr] * 10, ws, 0) == d.DFLASH_ERR_INVALID
    assert d.block_attn_fp8_context_raw(p8, ptr, 0, ptr, ptr, ptr, 1.0, 1.0, *tail) == d.DFLASH_ERR_INVALID
    from speculative_decoding_draft_paged_gb300 import _lib
    assert _lib.load().dflash_append_block_kv(ctypes.byref(p8), *[ptr] * 6, 0, 0) == d.DFLASH_ERR_INVALID


def test_status_strings(dflash_lib):
    from speculative_decoding_draft_paged_gb300 import _lib

    assert _lib.status_string(0) == "ok"
    assert "workspace" in _lib.status_string(-2)
    assert "10.3" in _lib.status_string(-3)
    assert _lib.status_string(123) == "unknown status"
    assert dflash_lib.version() >= 100


def test_two_ctas_per_sm_plan(dflash_lib):
    """The mma.sync plan takes its two-CTAs-per-SM form (3-stage ring, both
    CTAs' shared memory in one SM) only for bf16 pages at D = 64 with R in
    17..32 and more than one wave of units; every other plan holds one CTA
    per SM."""
    d = dflash_lib
    sm_bytes = 228 * 1024
    big = dict(num_q_heads=64, num_kv_heads=16, batch=256, max_ctx_len=131072, max_pages_per_req=4100)
    pl = d.plan(base_params(**big))
    assert pl["path"] == d.PATH_MMA and pl["threads"] == 288 and pl["ctas_per_sm"] == 2
    assert 2 * (pl["smem_bytes"] + 1024) <= sm_bytes
    one_wave = dict(num_q_heads=8, num_kv_heads=2, batch=1, max_ctx_len=32768, max_pages_per_req=1030)
    assert d.plan(base_params(**one_wave))["ctas_per_sm"] == 1
    for kw in (dict(big, num_q_heads=96),                 # R = 42: 416 threads
               dict(big, kv_dtype=d.KV_FP8_E4M3),         # fp8 pages
               dict(big, head_dim=128, page_size=64, max_pages_per_req=2060),
               dict(big, force_path=d.PATH_TCGEN05, batch=64)):
        pl = d.plan(base_params(**kw))
        assert pl["ctas_per_sm"] == 1, kw
        assert pl["smem_bytes"] + 1024 <= sm_bytes
    # A forced unit length follows the same rule.
    pl = d.plan(base_params(num_q_heads=8, num_kv_heads=2, batch=24, max_ctx_len=5000,
                            max_pages_per_req=160, force_split_tiles=1))
    assert pl["ctas_per_sm"] == 2 and pl["split_tiles"] == 1


def test_every_plan_fits_its_sm(dflash_lib):
    """Over a seeded sample of valid parameter sets: the split kernel's
    shared memory fits one CTA (227 KB) and, as many CTAs as the plan says an
    SM holds, the SM (228 KB, 1 KB reserved per CTA); the two-CTA form only
    where the kernel has it."""
    import random
    d = dflash_lib
    rng = random.Random(20260)
    checked = 0
    for _ in range(400):
        D = rng.choice([64, 128])
        Hkv = rng.choice([1, 2, 4, 16])
        G = rng.choice([1, 2, 4, 6, 8, 16])
        K = rng.choice([1, 3, 5, 7, 8, 16])
        if G * K > 128:
            continue
        P = rng.choice([16, 32, 64])
        L = rng.choice([100, 2048, 16384, 32768, 131072])
        kw = dict(batch=rng.choice([1, 2, 8, 16, 32, 64, 256]), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                  head_dim=D, page_size=P, block_size=K, max_ctx_len=L,
                  max_pages_per_req=(L + K + P - 1) // P + 1, num_pages=10 ** 6,
                  window=rng.choice([0, 0, 4096]), kv_dtype=rng.choice([0, 0, 1]),
                  force_split_tiles=rng.choice([0, 0, 0, 1, 7]))
        p = base_params(**kw)
        if d.workspace_size(p) == 0:
            continue  # a shape no kernel takes (e.g. an fp8 code ring that does not fit)
        pl = d.plan(p)
        checked += 1
        assert pl["smem_bytes"] <= 227 * 1024, kw
        assert pl["ctas_per_sm"] * (pl["smem_bytes"] + 1024) <= 228 * 1024, (kw, pl)
        if pl["ctas_per_sm"] == 2:
            assert (pl["path"], D, pl["rows_padded"], pl["threads"], kw["kv_dtype"]) == \
                (d.PATH_MMA, 64, 32, 288, 0), (kw, pl)
        else:
            assert pl["ctas_per_sm"] == 1, (kw, pl)
    assert checked > 100


def touched_tiles(L, K, W, T):
    lo = max(0, L - W + 1) if W > 0 else 0
    return (L + K + T - 1) // T - lo // T


@pytest.mark.parametrize("kw", [
    dict(), dict(window=4096, head_dim=128, page_size=64, num_q_heads=16, num_kv_heads=1,
                 max_ctx_len=16384, max_pages_per_req=260, batch=64),
    dict(window=100, max_ctx_len=1000), dict(batch=1, max_ctx_len=32768, max_pages_per_req=1030),
    dict(force_split_tiles=1), dict(force_split_tiles=3, window=50),
    dict(num_q_heads=64, num_kv_heads=16, batch=256, max_ctx_len=131072, max_pages_per_req=4100),
    dict(num_q_heads=64, num_kv_heads=4, batch=96, max_ctx_len=8192, max_pages_per_req=260),
    dict(num_q_heads=16, num_kv_heads=1, force_path=2, force_split_tiles=3, window=50),
    dict(num_q_heads=16, num_kv_heads=1, batch=900, max_ctx_len=100, max_pages_per_req=4),
    dict(kv_dtype=1), dict(kv_dtype=1, num_q_heads=4, num_kv_heads=2, block_size=3, window=33),
])
def test_planner_covers_every_length(dflash_lib, kw):
    """For every context length up to max_ctx_len the units cover all tiles,
    and the workspace holds every unit's partial state."""
    d = dflash_lib
    p = base_params(**kw)
    pl = d.plan(p)
    T, C, S = pl["tile_keys"], pl["split_tiles"], pl["max_splits"]
    worst = max(touched_tiles(L, p.block_size, p.window, T) for L in range(0, p.max_ctx_len + 1))
    R = p.num_q_heads // p.num_kv_heads * p.block_size
    assert pl["rows"] == R and pl["rows_padded"] >= R
    ws = d.workspace_size(p)
    # Per partial row: D output values and two log-sums.
    if pl["path"] == d.PATH_TCGEN05:
        assert pl["flat"] == 1
    if pl["flat"]:
        # Flat split: `units` CTAs of C tiles cover every pair at max_ctx_len,
        # two partial slots per CTA, at most one CTA per SM unless forced.
        assert S == 2
        assert pl["units"] * C >= p.batch * p.num_kv_heads * worst
        if not kw.get("force_split_tiles"):
            assert pl["units"] <= pl["num_sms"]
        assert ws >= 256 + 2 * pl["units"] * R * (p.head_dim + 2) * 4
    else:
        assert pl["units"] == p.batch * p.num_kv_heads * S
        assert S * C >= worst
        assert (S - 1) * C < worst + C
        assert ws >= 256 + pl["units"] * R * (p.head_dim + 2) * 4
    if kw.get("force_split_tiles"):
        assert C == kw["force_split_tiles"]


def test_plan_independent_of_lengths_and_pool_contents(dflash_lib):
    """The grid is a function of the parameters only (graph capture)."""
    d = dflash_lib
    a = d.plan(base_params())
    b = d.plan(base_params(num_pages=5000))
    assert a == b
