"""Parity criteria between the CUDA path and the fp64 oracle.

Tolerances: O max-abs <= 2e-2 and relative L2 <= 5e-3 over all elements; LSE
abs <= 2e-3 on rows with at least one selected key; the sets of empty rows
(LSE = -inf) identical, and O exactly 0 there; plans bit-exact.
"""
import numpy as np
import torch

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 2e-3


def attention_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o = o_gpu.detach().float().cpu().double().numpy() if torch.is_tensor(o_gpu) else np.asarray(o_gpu)
    l = lse_gpu.detach().cpu().double().numpy() if torch.is_tensor(lse_gpu) else np.asarray(lse_gpu)
    diff = o - o_ref
    fin = np.isfinite(lse_ref)
    return {
        "max_abs": float(np.abs(diff).max()) if diff.size else 0.0,
        "rel_l2": float(np.linalg.norm(diff) / max(np.linalg.norm(o_ref), 1e-30)),
        "lse_max_abs": float(np.abs(l[fin] - lse_ref[fin]).max()) if fin.any() else 0.0,
        "empty_rows_match": bool(np.array_equal(np.isneginf(l), np.isneginf(lse_ref))),
        "empty_rows_zero": bool(np.all(o[~fin] == 0.0)),
        "nan": bool(np.isnan(o).any() or np.isnan(l).any()),
    }


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    e = attention_errors(o_gpu, lse_gpu, o_ref, lse_ref)
    ok = (not e["nan"] and e["max_abs"] <= O_MAX_ABS and e["rel_l2"] <= O_REL_L2
          and e["lse_max_abs"] <= LSE_ABS and e["empty_rows_match"] and e["empty_rows_zero"])
    assert ok, f"{what}: {e}"
    return e
