"""Parity criteria between the CUDA path and the fp64 oracle.

Tolerances (from the target statement), applied to raw values on every
element:
  * O: |o_gpu - o_ref| <= 2e-2 + half a bf16 ulp of |o_ref|, where a bf16 ulp
    of x is 2^(floor(log2 x) - 7).  The second term is the rounding that
    storing the result as bf16 itself costs (the oracle's value is exact,
    the kernel's output is a bf16 number); nothing is divided by any
    property of the inputs;
  * relative L2 of O over all elements <= 5e-3;
  * LSE: abs <= 2e-3 on rows with at least one selected key;
  * the sets of empty rows (LSE = -inf) identical, and O exactly 0 there;
  * plans bit-exact (compared array by array in the plan tests).
"""
import numpy as np
import torch

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 2e-3


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (0 at x = 0): 2^(floor(log2|x|) - 8),
    with the subnormal spacing 2^-134 below the smallest normal."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def o_bound(o_ref):
    """Per-element bound on |o_gpu - o_ref|."""
    return O_MAX_ABS + bf16_half_ulp(o_ref)


def _np(x):
    if torch.is_tensor(x):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def attention_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o = _np(o_gpu)
    l = _np(lse_gpu)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    diff = np.abs(o - o_ref)
    fin = np.isfinite(lse_ref)
    if diff.size:
        excess = diff - o_bound(o_ref)
        i = np.unravel_index(int(np.argmax(excess)), excess.shape)
        worst = {"excess": float(excess[i]), "diff": float(diff[i]), "o_ref": float(o_ref[i]),
                 "index": [int(x) for x in i]}
    else:
        worst = {"excess": -O_MAX_ABS, "diff": 0.0, "o_ref": 0.0, "index": []}
    return {
        "max_abs": float(diff.max()) if diff.size else 0.0,
        "worst": worst,
        "rel_l2": float(np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)),
        "lse_max_abs": float(np.abs(l[fin] - lse_ref[fin]).max()) if fin.any() else 0.0,
        "empty_rows_match": bool(np.array_equal(np.isneginf(l), np.isneginf(lse_ref))),
        "empty_rows_zero": bool(np.all(o[~fin] == 0.0)),
        "nan": bool(np.isnan(o).any() or np.isnan(l).any()),
    }


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", record=False):
    """Assert the criteria above; with ``record`` the error summary is
    recorded (record_errors) before the assertion, pass or fail."""
    e = attention_errors(o_gpu, lse_gpu, o_ref, lse_ref)
    if record:
        record_errors(what, e)
    ok = (not e["nan"] and e["worst"]["excess"] <= 0.0 and e["rel_l2"] <= O_REL_L2
          and e["lse_max_abs"] <= LSE_ABS and e["empty_rows_match"] and e["empty_rows_zero"])
    assert ok, f"{what}: {e}"
    return e


def record_errors(name, errors):
    """Print the error summary of a parity check and, when the environment
    variable BSA_PARITY_LOG names a file, append it there as one JSON line."""
    import json
    import os
    line = json.dumps({"case": name, **errors})
    print(line)
    path = os.environ.get("BSA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")
