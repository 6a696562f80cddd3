"""bsa_attention_static: the one-call entry point that allocates nothing.

Some callers cannot allocate device memory: an inference-engine plugin whose
execute step must not call cudaMalloc, or a component that only ever receives
device pointers for its inputs and outputs.  For them the library keeps the
plan in a scratch area compiled into it (a file-scope __device__ array).
These tests call that entry point through the C ABI and compare it with the
ordinary plan + forward path (which runs the same kernels on a caller
workspace, so the results must be bit-identical) and once with the fp64
oracle.  Every call shares the one scratch area, so the sequence below also
runs a larger plan before a smaller one and a rejected call in between.
This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from oracle import attention as OA
from block_sparse_attention_plan_gb300 import workloads as W
from compare import assert_attention_close


def _static_call(lib, w, dev_inputs, o, lse):
    mask, q, k, v = dev_inputs
    B, H, NQB, NKB = w.mask.shape
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.bsa_attention_static(P(mask), B, H, NQB, NKB, w.bq, w.bk, w.gqa_group, P(q), P(k),
                                    P(v), P(o), P(lse), w.d, ctypes.c_float(0.0), s)


def _static_status(lib):
    det = ctypes.c_int32(0)
    st = lib.bsa_attention_static_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(det))
    return st, det.value


def _loose_bound_problem():
    # Rows whose Cauchy-Schwarz bound is far above their scores: the bounded
    # pass queues them for the exact pass (as in the forward tests).
    w = W.random_problem(21, 1, 4, 2, 512, 1024, 128, 128, 128, 0.7)
    q, k = w.q.float(), w.k.float()
    q[:, :2, :, 0] = 150.0
    k[:, :1, :, 1] = 150.0
    w.q, w.k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    return w


def _workspace(bsa, w):
    return int(bsa.plan_layout(*w.mask.shape, w.bq, w.bk, w.gqa_group, bsa.PLAN_NO_UNION).workspace_bytes)


@pytest.mark.gpu
def test_static_entry_matches_plan_forward_on_calls_in_a_row(bsa):
    lib = bsa.library()
    ws = [W.make_workload(n) for n in ("video_dit_small", "chunked_prefill_small", "regular_small",
                                       "tiny")] + [_loose_bound_problem()]
    # the third and fourth calls run smaller plans than the one before them
    sizes = [_workspace(bsa, w) for w in ws]
    assert sizes[1] > sizes[2] > sizes[3], sizes
    for i, w in enumerate(ws):
        dev = [w.mask.cuda(), w.q.cuda(), w.k.cuda(), w.v.cuda()]
        pl = bsa.plan(dev[0], w.bq, w.bk, w.gqa_group)
        o_ref, l_ref = bsa.forward(pl, *dev[1:])
        queued = int(pl.control()[3].item())  # rows the bounded pass left to the exact pass
        o = torch.full_like(dev[1], float("nan"))
        lse = torch.full(dev[1].shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        assert _static_call(lib, w, dev, o, lse) == 0
        assert _static_status(lib) == (0, 0)
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), w.name
        if i == 0:
            O, L = OA.block_gather(w.q, w.k, w.v, w.mask, w.bq, w.bk)
            assert_attention_close(o, lse, O, L, "static vs oracle")
        if i == 1:
            # A rejected call (plan too large for the scratch area) enqueues
            # nothing: the previous outputs stay as they are.
            o_keep, l_keep = o.clone(), lse.clone()
            P = lambda t: ctypes.c_void_p(t.data_ptr())
            assert lib.bsa_attention_static(P(dev[0]), 1, 40, 592, 592, 128, 128, 1, P(dev[1]),
                                            P(dev[2]), P(dev[3]), P(o), P(lse), 128,
                                            ctypes.c_float(0.0), None) == -5
            torch.cuda.synchronize()
            assert torch.equal(o, o_keep) and torch.equal(lse, l_keep)
        if i == len(ws) - 1:
            # this problem's rows went through the exact pass (on both paths)
            assert queued > 0
        else:
            assert queued == 0


def test_static_entry_rejects_oversized_problem(bsa):
    # long video-DiT geometry: its plan needs far more than the built-in scratch
    lib = bsa.library()
    p = ctypes.c_void_p(256)
    assert lib.bsa_attention_static(p, 1, 40, 592, 592, 128, 128, 1, p, p, p, p, p, 128,
                                    ctypes.c_float(0.0), None) == -5
