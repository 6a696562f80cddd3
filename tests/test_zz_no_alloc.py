"""bsa_attention_static: the one-call entry point that allocates nothing.

Some callers cannot allocate device memory (an inference-engine plugin whose
execute step must not call cudaMalloc, or a component that only receives
device pointers).  For them the library keeps the plan in a scratch area
compiled into it (a file-scope __device__ array).  These tests call that entry
point through the C ABI and compare it with the ordinary plan + forward path.
This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_plan_gb300 import workloads as W
from compare import assert_attention_close, channel_scale


def _static_call(lib, w, dev_inputs, o, lse):
    mask, q, k, v = dev_inputs
    B, H, NQB, NKB = w.mask.shape
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.bsa_attention_static(P(mask), B, H, NQB, NKB, w.bq, w.bk, w.gqa_group, P(q), P(k),
                                    P(v), P(o), P(lse), w.d, ctypes.c_float(0.0), s)


@pytest.mark.gpu
def test_static_entry_matches_plan_forward_on_two_calls(bsa):
    lib = bsa.library()
    for name in ("video_dit_small", "chunked_prefill_small"):  # two calls in a row
        w = W.make_workload(name)
        dev = [w.mask.cuda(), w.q.cuda(), w.k.cuda(), w.v.cuda()]
        o_ref, l_ref = bsa.forward(bsa.plan(dev[0], w.bq, w.bk, w.gqa_group), *dev[1:])
        o = torch.full_like(dev[1], float("nan"))
        lse = torch.full(dev[1].shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        assert _static_call(lib, w, dev, o, lse) == 0
        torch.cuda.synchronize()
        assert_attention_close(o, lse, o_ref.float().cpu().double().numpy(),
                               l_ref.cpu().double().numpy(), f"static vs plan+forward ({name})",
                               scale=channel_scale(w)[None, :, None, :])


def test_static_entry_rejects_oversized_problem(bsa):
    # long video-DiT geometry: its plan needs far more than the built-in scratch
    lib = bsa.library()
    p = ctypes.c_void_p(256)
    assert lib.bsa_attention_static(p, 1, 40, 592, 592, 128, 128, 1, p, p, p, p, p, 128,
                                    ctypes.c_float(0.0), None) == -5
