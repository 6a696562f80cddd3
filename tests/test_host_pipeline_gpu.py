"""GPU tests of bsa_attention_host: plan + forward from host buffers with the
copies overlapped with the computation, chunk by chunk of (batch, K/V head)
units.  Every row must equal, bit for bit, the device-resident path
(bsa_plan_create + bsa_forward), which the forward parity tests pin to the
oracle; one case is also compared with the oracle directly."""
import ctypes

import pytest
import torch

from oracle import attention as OA
from block_sparse_attention_plan_gb300 import workloads as W
from compare import assert_attention_close

pytestmark = pytest.mark.gpu


def device_path(bsa, w):
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda())
    assert bsa.sync_status(p)[0] == 0
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("name", ["tiny", "video_dit_small", "chunked_prefill_small", "regular_small"])
@pytest.mark.parametrize("chunks", [1, 2, 3, 64])
def test_host_pipeline_equals_device_path(bsa, name, chunks):
    w = W.make_workload(name)
    o_ref, l_ref = device_path(bsa, w)
    pin = [t.pin_memory() for t in (w.mask, w.q, w.k, w.v)]
    o, lse = bsa.attention(*pin, w.bq, w.bk, chunks=chunks)
    assert not o.is_cuda and not lse.is_cuda
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, l_ref)


def test_host_pipeline_pageable_inputs_and_oracle(bsa):
    w = W.random_problem(41, 2, 4, 2, 256, 512, 64, 64, 128, 0.4)
    o, lse = bsa.attention(w.mask, w.q, w.k, w.v, 64, 128, chunks=3)  # pageable host memory
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 128)
    assert_attention_close(o.cuda(), lse.cuda(), O, L, "host pipeline")


def test_host_pipeline_argument_errors(bsa):
    from block_sparse_attention_plan_gb300 import _lib as L
    w = W.make_workload("tiny")
    B, H, NQB, NKB = w.mask.shape
    d = w.q.shape[3]
    lib = L.library()
    need = L.host_buffer_bytes(B, H, NQB, NKB, w.bq, w.bk, 1, d, 2)
    buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(w.q).pin_memory()
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32).pin_memory()
    VP = ctypes.c_void_p
    args = (VP(w.mask.data_ptr()), B, H, NQB, NKB, w.bq, w.bk, 1, VP(w.q.data_ptr()),
            VP(w.k.data_ptr()), VP(w.v.data_ptr()), VP(o.data_ptr()), VP(lse.data_ptr()), d, 0.0)
    assert lib.bsa_attention_host(*args, 2, VP(buf.data_ptr()), need - 1, None) == -5  # too small
    assert lib.bsa_attention_host(*args, 0, VP(buf.data_ptr()), need, None) == -1      # chunks < 1
    assert lib.bsa_attention_host(*args, 2, VP(buf.data_ptr() + 16), need - 256, None) == -1  # misaligned
    assert lib.bsa_attention_host(*args, 2, VP(buf.data_ptr()), need, None) == 0
