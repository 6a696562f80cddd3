"""GPU tests of bsa_forward_ex: paged K/V, per-sequence key lengths and
intra-block causal masking ("CompactAttention: Accelerating Chunked Prefill
with Block-Union KV Selection", summary: zero-copy paged execution of chunked
prefill).  Parity is against the fp64 oracle (``oracle.attention`` with its
element mask) and, for paging alone, bit-exactness against the contiguous
path on the same inputs."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as OA
from block_sparse_attention_plan_gb300 import workloads as W
from compare import assert_attention_close

pytestmark = pytest.mark.gpu

FALLBACK_COUNT = 3  # control word: rows the bounded pass queued for the exact pass


def make_pool(k, v, page_size, seed, extra_pages=3, kv_lens=None):
    """Scatter contiguous K/V [B, Hkv, Nk, d] into shuffled pages of pools
    [num_pages, Hkv, page_size, d]; returns (k_pool, v_pool, block_table).
    Logical pages wholly past kv_lens[b] are left unallocated (-1)."""
    B, Hkv, Nk, d = k.shape
    lp_count = (Nk + page_size - 1) // page_size
    g = torch.Generator().manual_seed(seed)
    num_pages = B * lp_count + extra_pages
    perm = torch.randperm(num_pages, generator=g)
    table = torch.full((B, lp_count), -1, dtype=torch.int32)
    k_pool = torch.randn(num_pages, Hkv, page_size, d, generator=g).to(torch.bfloat16)
    v_pool = torch.randn(num_pages, Hkv, page_size, d, generator=g).to(torch.bfloat16)
    nxt = 0
    for b in range(B):
        for lp in range(lp_count):
            if kv_lens is not None and lp * page_size >= int(kv_lens[b]):
                continue
            phys = int(perm[nxt])
            nxt += 1
            table[b, lp] = phys
            lo, hi = lp * page_size, min((lp + 1) * page_size, Nk)
            k_pool[phys, :, :hi - lo] = k[b, :, lo:hi]
            v_pool[phys, :, :hi - lo] = v[b, :, lo:hi]
    return k_pool.cuda(), v_pool.cuda(), table.cuda()


def test_paged_rows_taking_the_exact_pass(bsa):
    """Rows whose bound is far above their scores go to the exact pass; with
    paged K/V (no element mask) both passes run the paged kernels and give
    the contiguous result bit for bit, and the oracle's within tolerance."""
    w = W.random_problem(21, 1, 4, 2, 512, 1024, 128, 128, 128, 0.7)
    q, k = w.q.float(), w.k.float()
    q[:, :2, :, 0] = 150.0
    k[:, :1, :, 1] = 150.0
    w.q, w.k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    qd = w.q.cuda()
    o1, l1 = bsa.forward(p, qd, w.k.cuda(), w.v.cuda())
    kp, vp, table = make_pool(w.k, w.v, 128, seed=5)
    o2, l2 = bsa.forward(p, qd, kp, vp, block_table=table)
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    assert int(p.control()[FALLBACK_COUNT].item()) > 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128)
    assert_attention_close(o2, l2, O, L, "paged, exact pass")


@pytest.mark.parametrize("name,page_mult", [("video_dit_small", 1), ("video_dit_small", 2),
                                            ("chunked_prefill_small", 1), ("chunked_prefill_small", 4),
                                            ("regular_small", 4)])
def test_paged_equals_contiguous(bsa, name, page_mult):
    w = W.make_workload(name)
    page_size = page_mult * min(w.bk, 128)
    if w.k.shape[2] % page_size:
        pytest.skip("sequence not a whole number of pages")
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    q = w.q.cuda()
    o1, l1 = bsa.forward(p, q, w.k.cuda(), w.v.cuda())
    kp, vp, table = make_pool(w.k, w.v, page_size, seed=7)
    o2, l2 = bsa.forward(p, q, kp, vp, block_table=table)
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


def test_causal_chunk_vs_oracle(bsa):
    # A 512-query chunk at the end of a 2048-key sequence, 64x64 blocks, a
    # block mask that already respects causality at block level (so the
    # element mask acts on the diagonal blocks) plus random blocks below it.
    w = W.random_problem(31, 1, 4, 2, 512, 2048, 128, 64, 64, 0.5)
    NQB, NKB = 512 // 64, 2048 // 64
    off_b = NKB - NQB
    kb = torch.arange(NKB).view(1, NKB)
    qb = torch.arange(NQB).view(NQB, 1)
    causal_blocks = (kb <= qb + off_b).to(torch.uint8)
    w.mask = (w.mask * causal_blocks).contiguous()
    w.mask[:, :, :, 0] = 1
    idx = torch.arange(NQB)
    w.mask[:, :, idx, idx + off_b] = 1  # diagonal blocks always selected
    p = bsa.plan(w.mask.cuda(), 64, 64, w.gqa_group)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda(), causal=True)
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64, causal=True)
    assert_attention_close(o, lse, O, L, "causal chunk")


def test_kv_lens_vs_oracle(bsa):
    w = W.random_problem(32, 3, 2, 2, 256, 1024, 128, 128, 128, 0.7)
    lens = torch.tensor([1024 - 77, 300, 0], dtype=torch.int32)
    p = bsa.plan(w.mask.cuda(), 128, 128, w.gqa_group)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda(), kv_lens=lens.cuda())
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128, kv_lens=lens.tolist())
    assert_attention_close(o, lse, O, L, "kv_lens")
    assert torch.all(o[2] == 0) and torch.all(torch.isneginf(lse[2]))


@pytest.mark.parametrize("bq,bk,d", [(128, 128, 128), (64, 32, 64)])
def test_paged_causal_kv_lens_vs_oracle(bsa, bq, bk, d):
    # Pages past each sequence's key length are unallocated (-1 in the block
    # table): the kernel must neither read them nor report them.
    w = W.random_problem(33, 2, 4, 2, 256, 1536, d, bq, bk, 0.6)
    lens = torch.tensor([1536 - 200, 700], dtype=torch.int32)
    page_size = 256
    p = bsa.plan(w.mask.cuda(), bq, bk, w.gqa_group)
    kp, vp, table = make_pool(w.k, w.v, page_size, seed=11, kv_lens=lens)
    assert int((table == -1).sum()) > 0
    o, lse = bsa.forward(p, w.q.cuda(), kp, vp, block_table=table, kv_lens=lens.cuda(),
                         causal=True)
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk, causal=True, kv_lens=lens.tolist())
    assert_attention_close(o, lse, O, L, f"paged causal kv_lens {bq}x{bk} d{d}")


def test_forward_ex_argument_errors(bsa):
    from block_sparse_attention_plan_gb300 import _lib as L
    w = W.make_workload("chunked_prefill_small")  # bk = 64: K unit 64
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    lib = L.library()
    VP = ctypes.c_void_p
    args = (VP(q.data_ptr()), VP(k.data_ptr()), VP(v.data_ptr()))
    outs = (VP(o.data_ptr()), VP(lse.data_ptr()), 128, 0.0, None)
    assert lib.bsa_forward_ex(p.handle, *args, None, None, 0x4, *outs) == -1  # unknown flag
    table = torch.zeros(w.q.shape[0], 64, dtype=torch.int32, device="cuda")
    bad = L.KVPagesC(table.data_ptr(), 64, 96, 8)  # 96 is not a multiple of the K unit 64
    assert lib.bsa_forward_ex(p.handle, *args, ctypes.byref(bad), None, 0, *outs) == -2
    short = L.KVPagesC(table.data_ptr(), 1, 64, 8)  # 1 page of 64 keys cannot hold Nk
    assert lib.bsa_forward_ex(p.handle, *args, ctypes.byref(short), None, 0, *outs) == -1
    null_table = L.KVPagesC(None, 64, 64, 8)
    assert lib.bsa_forward_ex(p.handle, *args, ctypes.byref(null_table), None, 0, *outs) == -1
