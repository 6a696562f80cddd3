"""Failure detection on the GPU without faulting it: the watchdog's bounded
wait gives up by itself; out-of-range plan entries are caught by the kernel's
own bounds checks; argument errors are rejected on the host."""
import pytest
import torch

from block_sparse_attention_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_watchdog_wait_times_out(bsa):
    # The self-test kernel waits on a barrier nothing completes (limit 20 ms).
    assert bsa.watchdog_selftest(20000) == -6


def test_poisoned_plan_is_reported_not_trapped(bsa):
    w = W.make_workload("video_dit_small")
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, 1)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    bsa.forward(p, q, k, v)
    assert bsa.sync_status(p)[0] == 0
    assert bsa.plan_check(p) == 0
    L = p.layout
    ku = p.workspace[L.off_slot_ku:L.off_slot_ku + 16].view(torch.int32)
    ku[0] = 1 << 20                       # k-unit far out of range
    assert bsa.plan_check(p) == -7
    bsa.forward(p, q, k, v)
    st, det = bsa.sync_status(p)
    assert st == -7, (st, hex(det))
    rp = p.workspace[L.off_row_ptr:L.off_row_ptr + 16].view(torch.int32)
    ku[0] = 0
    rp[1] = 1 << 30                       # row pointer past the slot capacity
    bsa.forward(p, q, k, v)
    assert bsa.sync_status(p)[0] == -7


def test_forward_argument_errors(bsa):
    w = W.make_workload("tiny")
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, 1)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    lib = bsa.library()
    import ctypes
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.bsa_forward(p.handle, P(q, 2), P(k), P(v), P(o), P(lse), 64, 0.0, s) == -1
    assert lib.bsa_forward(p.handle, P(q), P(k), P(v), P(o), P(lse), 96, 0.0, s) == -2
    assert lib.bsa_forward(p.handle, P(q), P(k), P(v), P(o), P(lse), 64, float("nan"), s) == -1
    assert lib.bsa_forward(p.handle, P(q), P(k), P(v), P(o), P(lse), 64, 0.0, s) == 0
    assert bsa.sync_status(p)[0] == 0
