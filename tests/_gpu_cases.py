"""Helpers for the GPU parity tests: run the library and the oracle on the same
seeded inputs and compare them.

Tolerances (the stated bar for bf16 outputs, read as follows):
* relative L2 error of ``out`` against the unrounded fp64 oracle < 5e-3;
* max abs error of ``out`` beyond the bf16 format's own rounding <= 1e-2
  (times the value scale where the values are not unit-variance: fp8 context
  with v_scale > 1):
  ``max_i (|gpu_i - oracle_i| - ulp_bf16(oracle_i) / 2) <= 1e-2``.  Any bf16
  output is off by up to half an ulp from the exact value (0.0078 at
  |x| in [2, 4)), and a value near a rounding midpoint may round either way,
  so the bound is applied to the error the computation adds;
* the pages' own form, max abs <= 8 bf16 ulp of the biggest reference
  magnitude (PR #20374, test coverage), on the raw error;
* max abs error of the base-2 LSE <= 1e-3.
"""

import json
import os

import numpy as np
import torch

import oracle
import speculative_decoding_draft_paged_gb300 as dflash
from speculative_decoding_draft_paged_gb300 import workloads

REL_L2_MAX = 5e-3
MAX_ABS_MAX = 1e-2
LSE_ABS_MAX = 1e-3


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_lib(spec, inp, **kw):
    kw.setdefault("max_ctx_len", spec.max_ctx_len)
    return dflash.block_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                             inp["ctx_lens"], block_size=spec.K, window=spec.window,
                             future_keys=spec.future_keys, scale=spec.softmax_scale,
                             right_window=spec.right_window, **kw)


def run_oracle(spec, inp, req_ids=None, ctx_lens=None):
    lens = ctx_lens if ctx_lens is not None else inp["ctx_lens"]
    return oracle.block_attn(to_bits(inp["q"]), to_bits(inp["k_pages"]), to_bits(inp["v_pages"]),
                             inp["page_table"].cpu().numpy(), np.asarray(lens.cpu() if
                                                                         torch.is_tensor(lens) else lens,
                                                                         dtype=np.int32),
                             block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
                             right_window=spec.right_window,
                             scale=spec.softmax_scale, req_ids=req_ids)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits); 2^-133 below the normals."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


def metrics(gpu_out, gpu_lse, ora_out, ora_lse) -> dict:
    g = gpu_out.detach().cpu().to(torch.float64).numpy()
    gl = gpu_lse.detach().cpu().to(torch.float64).numpy()
    diff = np.abs(g - ora_out)
    if g.size == 0:
        return {"rel_l2": 0.0, "max_abs_excess": 0.0, "max_abs_vs_bf16": 0.0, "max_abs_raw": 0.0,
                "ulp_at_max": 0.0, "lse_abs": 0.0, "nan": False}
    return {
        "rel_l2": float(np.linalg.norm(g - ora_out) / max(np.linalg.norm(ora_out), 1e-300)),
        "max_abs_excess": float(np.max(diff - ulp_bf16(ora_out) / 2)),
        "max_abs_vs_bf16": float(np.max(np.abs(g - bf16_round(ora_out)))),
        "max_abs_raw": float(np.max(diff)),
        "ulp_at_max": float(ulp_bf16(np.array([np.max(np.abs(ora_out))]))[0]),
        "lse_abs": float(np.max(np.abs(gl - ora_lse))),
        "nan": bool(np.isnan(g).any() or np.isnan(gl).any()),
    }


def log_parity(m: dict, what: str, value_scale: float = 1.0) -> None:
    """Appends the achieved error figures of one comparison, with the share
    of each bound they use, to the JSON-lines file named by
    ``DFLASH_PARITY_LOG`` (when set), so that the headroom left under the
    bounds can be tabulated per case."""
    path = os.environ.get("DFLASH_PARITY_LOG")
    if not path:
        return
    bound_abs = MAX_ABS_MAX * max(1.0, value_scale)
    rec = {"case": what, **{k: v for k, v in m.items()},
           "use_rel_l2": m["rel_l2"] / REL_L2_MAX, "use_max_abs": m["max_abs_excess"] / bound_abs,
           "use_ulp8": m["max_abs_raw"] / (8 * m["ulp_at_max"]) if m["ulp_at_max"] else 0.0,
           "use_lse": m["lse_abs"] / LSE_ABS_MAX, "value_scale": value_scale}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def assert_parity(m: dict, what: str = "", value_scale: float = 1.0):
    """``value_scale``: the magnitude of the values relative to unit variance
    (the fp8 form's v_scale); the absolute bound scales with it, as the bf16
    rounding of the probabilities contributes an error proportional to |v|."""
    log_parity(m, what, value_scale)
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["rel_l2"] < REL_L2_MAX, f"{what}: {m}"
    assert m["max_abs_excess"] <= MAX_ABS_MAX * max(1.0, value_scale), f"{what}: {m}"
    assert m["max_abs_raw"] <= 8 * m["ulp_at_max"], f"{what}: {m}"
    assert m["lse_abs"] <= LSE_ABS_MAX, f"{what}: {m}"


def check_case(spec, device, **kw):
    inp = workloads.make_inputs(spec, "cpu")
    dev = {k: v.to(device) for k, v in inp.items()}
    out, lse = run_lib(spec, dev, **kw)
    torch.cuda.synchronize()
    ref_out, ref_lse = run_oracle(spec, inp)
    m = metrics(out, lse, ref_out, ref_lse)
    assert_parity(m, spec.name)
    return m, out, lse


def compact_requests(inp: dict, req_ids) -> dict:
    """Copy the pages of the chosen requests to the host as a compact pool."""
    table = inp["page_table"].cpu()
    rows = table[list(req_ids)]
    used = sorted(set(int(x) for x in rows.flatten().tolist() if x >= 0))
    remap = {pg: n for n, pg in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=inp["k_pages"].device)
    kp = inp["k_pages"].index_select(0, idx).cpu()
    vp = inp["v_pages"].index_select(0, idx).cpu()
    new_rows = rows.clone()
    for i in range(new_rows.shape[0]):
        for j in range(new_rows.shape[1]):
            x = int(new_rows[i, j])
            new_rows[i, j] = remap[x] if x >= 0 else -1
    return {"q": inp["q"][list(req_ids)].cpu(), "k_pages": kp, "v_pages": vp,
            "page_table": new_rows, "ctx_lens": inp["ctx_lens"].cpu()[list(req_ids)]}
