"""Helpers for the GPU parity tests: run the library and the oracle on the same
seeded inputs and compare them.

Tolerances (from the stated bar for bf16 outputs, with the readings recorded
in the design doc): relative L2 error of ``out`` against the unrounded fp64 oracle
< 5e-3; max abs error of ``out`` against the oracle rounded once to bf16
(nearest-even) <= 1e-2; max abs error of the base-2 LSE <= 1e-3.
"""

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
                             future_keys=spec.future_keys, scale=spec.softmax_scale, **kw)


def run_oracle(spec, inp, req_ids=None, ctx_lens=None):
    lens = ctx_lens if ctx_lens is not None else inp["ctx_lens"]
    return oracle.block_attn(to_bits(inp["q"]), to_bits(inp["k_pages"]), to_bits(inp["v_pages"]),
                             inp["page_table"].cpu().numpy(), np.asarray(lens.cpu() if
                                                                         torch.is_tensor(lens) else lens,
                                                                         dtype=np.int32),
                             block_size=spec.K, window=spec.window, future_keys=spec.future_keys,
                             scale=spec.softmax_scale, req_ids=req_ids)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


def metrics(gpu_out, gpu_lse, ora_out, ora_lse) -> dict:
    g = gpu_out.detach().cpu().to(torch.float64).numpy()
    gl = gpu_lse.detach().cpu().to(torch.float64).numpy()
    diff = g - ora_out
    return {
        "rel_l2": float(np.linalg.norm(diff) / max(np.linalg.norm(ora_out), 1e-300)),
        "max_abs_vs_bf16": float(np.max(np.abs(g - bf16_round(ora_out)))) if g.size else 0.0,
        "max_abs_raw": float(np.max(np.abs(diff))) if g.size else 0.0,
        "lse_abs": float(np.max(np.abs(gl - ora_lse))) if gl.size else 0.0,
        "nan": bool(np.isnan(g).any() or np.isnan(gl).any()),
    }


def assert_parity(m: dict, what: str = ""):
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["rel_l2"] < REL_L2_MAX, f"{what}: {m}"
    assert m["max_abs_vs_bf16"] <= MAX_ABS_MAX, f"{what}: {m}"
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
