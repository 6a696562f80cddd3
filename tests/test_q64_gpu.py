"""64-row q-tiles (BSA_PLAN_Q64): GPU plans bit-exact against the plan oracle
with tile = 64, and the forward (the kernel that puts a slot's 128 keys on the
MMA's M dimension and the tile's 64 queries on N) against the fp64 attention
oracle, through the C ABI."""
import itertools

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import plan as OP
from block_sparse_attention_plan_gb300 import workloads as W
from compare import assert_attention_close
from test_plan_gpu import assert_plan_equal

pytestmark = pytest.mark.gpu

# Control word holding the number of rows the bounded pass queued for the
# exact pass (index 3 of the plan's control words).
FALLBACK_COUNT = 3


def q64_plan(bsa, mask, bq, bk, g, remap=False):
    flags = bsa.PLAN_Q64 | (bsa.PLAN_REMAP if remap else 0)
    p = bsa.plan(mask.cuda(), bq, bk, g, flags=flags)
    assert bsa.plan_check(p) == 0
    return p


def gpu_arrays(p):
    a = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    a["slot_mask"] = a["slot_mask"].astype(np.int64) & 0xFFFFFFFF
    return a


@pytest.mark.parametrize("bq,bk", list(itertools.product((32, 64), (32, 64, 128, 256))))
def test_q64_plan_random_masks(bsa, bq, bk):
    for g in (1, 2):
        w = W.random_problem(200 + bq + bk + g, 2, 4, 4 // g, 1024, 1536, 16, bq, bk, 0.23, values=True)
        p = q64_plan(bsa, w.mask, bq, bk, g)
        assert p.layout.NQT == 1024 // 64 and p.layout.qu * p.layout.rq == 64
        assert_plan_equal(gpu_arrays(p), OP.build_plan(w.mask.numpy(), bq, bk, g, tile=64))
    w = W.random_problem(300 + bq + bk, 2, 4, 4, 1024, 1536, 16, bq, bk, 0.1)
    x = torch.arange(w.mask.shape[2]).view(-1, 1)
    w.mask[:, 1] |= ((torch.arange(w.mask.shape[3]).view(1, -1) % 2) == (x % 2)).to(torch.uint8)
    p = q64_plan(bsa, w.mask, bq, bk, 1, remap=True)
    assert_plan_equal(gpu_arrays(p), OP.build_plan(w.mask.numpy(), bq, bk, 1, remap=True, tile=64))


@pytest.mark.parametrize("name", ["chunked_prefill", "regular", "chunked_prefill_small", "regular_small"])
def test_q64_plan_workloads(bsa, name):
    w = W.make_workload(name, data=False)
    remap = w.gqa_group == 1
    p = q64_plan(bsa, w.mask, w.bq, w.bk, w.gqa_group, remap=remap)
    ref = OP.build_plan(w.mask.numpy(), w.bq, w.bk, w.gqa_group, remap=remap, tile=64)
    assert_plan_equal(gpu_arrays(p), ref)
    if name == "chunked_prefill":
        assert int(p.arrays()["totals"][0]) == 67584  # 33 slots per 64-row q-block


def test_q64_plan_rejects_large_blocks_and_odd_lengths(bsa):
    with pytest.raises(bsa.BsaError):
        bsa.plan_layout(1, 2, 4, 4, 128, 64, 1, bsa.PLAN_Q64)
    with pytest.raises(bsa.BsaError):
        bsa.plan_layout(1, 2, 3, 4, 32, 64, 1, bsa.PLAN_Q64)   # Nq = 96
    assert bsa.plan_layout(1, 2, 3, 4, 64, 64, 1, bsa.PLAN_Q64).NQT == 3


def run_q64(bsa, w, remap=False, **kw):
    p = q64_plan(bsa, w.mask, w.bq, w.bk, w.gqa_group, remap=remap)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda(), **kw)
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    return p, o, lse


@pytest.mark.parametrize("bq,bk,d,g", [
    (64, 64, 128, 1), (64, 64, 64, 2), (32, 32, 64, 1), (32, 32, 128, 4), (64, 128, 128, 1),
    (32, 256, 64, 1), (64, 32, 128, 2), (32, 64, 64, 1), (64, 256, 128, 1), (32, 128, 128, 1),
])
def test_q64_forward_mappings(bsa, bq, bk, d, g):
    w = W.random_problem(41 + bq + bk + d, 1, 4, 4 // g, 1024, 1536, d, bq, bk, 0.3)
    w.mask[0, 1, 0, :] = 0   # an empty logical q-block row
    _, o, lse = run_q64(bsa, w)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    assert_attention_close(o, lse, O, L, f"q64 bq={bq} bk={bk} d={d} g={g}")


@pytest.mark.parametrize("name", ["chunked_prefill_small", "regular_small"])
def test_q64_forward_small_workloads(bsa, name):
    w = W.make_workload(name)
    for remap in ((False, True) if w.gqa_group == 1 else (False,)):
        p, o, lse = run_q64(bsa, w, remap=remap)
        assert int(p.control()[FALLBACK_COUNT].item()) == 0
        O, L = OA.block_gather(w.q, w.k, w.v, w.mask, w.bq, w.bk)
        assert_attention_close(o, lse, O, L, f"q64 {name} remap={remap}", record=True)


@pytest.mark.parametrize("d", [64, 128])
def test_q64_forward_all_ones_all_zero_and_scale(bsa, d):
    w = W.random_problem(7 + d, 1, 2, 2, 512, 768, d, 64, 64, 1.1)
    _, o, lse = run_q64(bsa, w, scale=0.07)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64, scale=0.07)
    assert_attention_close(o, lse, O, L, "q64 all ones")
    w.mask.zero_()
    _, o, lse = run_q64(bsa, w)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_q64_loose_bound_rows_take_exact_pass(bsa):
    # As for 128-row tiles: |q||k| far above every score of heads 0-1 makes
    # the bounded pass underflow there, and the exact pass (two sweeps: the
    # exact per-query maximum, then split weights) recomputes those rows.
    w = W.random_problem(23, 1, 4, 2, 512, 1024, 128, 64, 64, 0.5)
    q, k = w.q.float(), w.k.float()
    q[:, :2, :, 0] = 150.0
    k[:, :1, :, 1] = 150.0
    w.q, w.k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    p, o, lse = run_q64(bsa, w)
    queued = int(p.control()[FALLBACK_COUNT].item())
    nonempty = int((w.mask[0, :2].reshape(2, 8, -1).sum(-1) > 0).sum())
    assert nonempty <= queued <= 2 * 8, (queued, nonempty)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64)
    assert_attention_close(o, lse, O, L, "q64 loose bound")


@pytest.mark.parametrize("bq,bk,d", [(64, 64, 128), (32, 32, 64), (32, 128, 128)])
def test_q64_split_weights_through_exact_pass(bsa, bq, bk, d):
    # Large V values: every row goes to the exact pass (split weights);
    # forcing split weights gives the same bits.
    w = W.random_problem(51 + bq + d, 1, 4, 2, 1024, 1024, d, bq, bk, 0.3)
    w.mask[0, 3, 1, :] = 0
    v = w.v.float()
    v[:, :, :, :3] *= 16.0
    w.v = v.to(torch.bfloat16)
    p, o, lse = run_q64(bsa, w)
    nonempty_rows = int((w.mask[0].reshape(4, 1024 // 64, -1).sum(-1) > 0).sum()) if bq == 64 else None
    queued = int(p.control()[FALLBACK_COUNT].item())
    assert queued > 0 and (nonempty_rows is None or queued == nonempty_rows)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    assert_attention_close(o, lse, O, L, f"q64 large V {bq}x{bk} d{d}")
    _, o2, l2 = run_q64(bsa, w, split=True)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_q64_same_result_as_128_row_tiles_within_tolerance_and_repeatable(bsa):
    w = W.make_workload("chunked_prefill_small")
    _, o1, l1 = run_q64(bsa, w)
    _, o2, l2 = run_q64(bsa, w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    o3, l3 = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda())
    assert (o1.float() - o3.float()).abs().max().item() < 1e-2
    assert (l1 - l3).abs().max().item() < 1e-3


def test_q64_rejects_pages_and_element_masks(bsa):
    w = W.make_workload("chunked_prefill_small")
    p = q64_plan(bsa, w.mask, w.bq, w.bk, w.gqa_group)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    with pytest.raises(bsa.BsaError):
        bsa.forward(p, q, k, v, causal=True)
    with pytest.raises(bsa.BsaError):
        bsa.forward(p, q, k, v, kv_lens=torch.full((1,), 100, dtype=torch.int32, device="cuda"))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["chunked_prefill", "regular"])
def test_q64_forward_full_configs(bsa, name):
    w = W.make_workload(name)
    p, o, lse = run_q64(bsa, w, remap=w.gqa_group == 1)
    assert int(p.control()[FALLBACK_COUNT].item()) == 0
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, w.bq, w.bk)
    assert_attention_close(o, lse, O, L, f"{name} (64-row q-tiles)", record=True)
