"""Parity criteria between the CUDA path and the fp64 oracle.

Tolerances: O max-abs <= 2e-2 and relative L2 <= 5e-3 over all elements; LSE
abs <= 2e-3 on rows with at least one selected key; the sets of empty rows
(LSE = -inf) identical, and O exactly 0 there; plans bit-exact.

The max-abs bound is read in units of the value scale: output channels whose
V channel was multiplied by an outlier factor s (workloads with outlier
channels) are divided by s before the max-abs check, since bf16 storage alone
moves an output of magnitude |o| by up to |o|*2^-9.  Relative L2 is
scale-free and is applied unchanged.
"""
import numpy as np
import torch

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 2e-3


def channel_scale(w):
    """Per (query head, channel) factor of the output scale: the product of the
    outlier factors applied to that channel of the head's V (1 elsewhere)."""
    sc = np.ones((w.Hq, w.d))
    pairs = w.meta.get("outlier_pairs")
    if pairs:
        g = w.Hq // w.Hkv
        vs = np.ones((w.Hkv, w.d))
        for p in pairs:
            h, c = divmod(int(p), w.d)
            vs[h // g, c] *= 8.0
        sc = vs[np.arange(w.Hq) // g]
    return sc


def attention_errors(o_gpu, lse_gpu, o_ref, lse_ref, scale=None):
    """``scale``: array broadcastable to O of per-element value-scale factors."""
    o = o_gpu.detach().float().cpu().double().numpy() if torch.is_tensor(o_gpu) else np.asarray(o_gpu)
    l = lse_gpu.detach().cpu().double().numpy() if torch.is_tensor(lse_gpu) else np.asarray(lse_gpu)
    diff = o - o_ref
    fin = np.isfinite(lse_ref)
    nd = diff / scale if scale is not None else diff
    return {
        "max_abs": float(np.abs(nd).max()) if diff.size else 0.0,
        "rel_l2": float(np.linalg.norm(diff) / max(np.linalg.norm(o_ref), 1e-30)),
        "lse_max_abs": float(np.abs(l[fin] - lse_ref[fin]).max()) if fin.any() else 0.0,
        "empty_rows_match": bool(np.array_equal(np.isneginf(l), np.isneginf(lse_ref))),
        "empty_rows_zero": bool(np.all(o[~fin] == 0.0)),
        "nan": bool(np.isnan(o).any() or np.isnan(l).any()),
    }


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", scale=None):
    e = attention_errors(o_gpu, lse_gpu, o_ref, lse_ref, scale)
    ok = (not e["nan"] and e["max_abs"] <= O_MAX_ABS and e["rel_l2"] <= O_REL_L2
          and e["lse_max_abs"] <= LSE_ABS and e["empty_rows_match"] and e["empty_rows_zero"])
    assert ok, f"{what}: {e}"
    return e
