"""GPU plan kernels vs the plan oracle: every array bit-exact."""
import itertools

import numpy as np
import pytest
import torch

from oracle import plan as OP
from block_sparse_attention_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def gpu_plan_arrays(bsa, mask, bq, bk, g):
    p = bsa.plan(mask.cuda(), bq, bk, g)
    a = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    a["slot_mask"] = a["slot_mask"].astype(np.int64) & 0xFFFFFFFF
    assert bsa.plan_check(p) == 0
    return p, a


def assert_plan_equal(a, ref):
    assert int(a["totals"][3]) == 0  # reserved word
    keys = ["row_ptr", "slot_ku", "slot_mask", "urow_ptr", "ukb", "order", "totals"]
    if "plane_sigma" in a and "plane_sigma" in ref:
        keys.append("plane_sigma")
    for k in keys:
        got = np.asarray(a[k]).astype(np.int64)
        want = np.asarray(ref[k]).astype(np.int64)
        if k == "totals":
            got = got[:3]
        assert got.shape == want.shape, (k, got.shape, want.shape)
        if not np.array_equal(got, want):
            bad = np.flatnonzero(got != want)[:10]
            raise AssertionError(f"{k} differs at {bad.tolist()}: got {got[bad].tolist()} want {want[bad].tolist()}")


@pytest.mark.parametrize("name", list(W.SMALL_CONFIGS) + list(W.CONFIGS))
def test_plan_workloads_bit_exact(bsa, name):
    w = W.make_workload(name, data=False)
    _, a = gpu_plan_arrays(bsa, w.mask, w.bq, w.bk, w.gqa_group)
    ref = OP.build_plan(w.mask.numpy(), w.bq, w.bk, w.gqa_group)
    assert_plan_equal(a, ref)
    assert int(a["totals"][1]) == w.active_blocks


@pytest.mark.parametrize("bq,bk", list(itertools.product((32, 64, 128, 256), repeat=2)))
def test_plan_random_masks_all_mappings(bsa, bq, bk):
    g = 2 if (bq + bk) % 3 else 1
    w = W.random_problem(100 + bq + bk, 2, 4, 4 // g, 1024, 1536, 16, bq, bk, 0.23, values=True)
    _, a = gpu_plan_arrays(bsa, w.mask, bq, bk, g)
    assert_plan_equal(a, OP.build_plan(w.mask.numpy(), bq, bk, g))


def test_plan_exhaustive_3x3(bsa):
    for bits in range(512):
        m = torch.tensor([(bits >> t) & 1 for t in range(9)], dtype=torch.uint8).reshape(1, 1, 3, 3)
        for bq, bk in ((128, 128), (256, 64), (128, 32)):
            _, a = gpu_plan_arrays(bsa, m, bq, bk, 1)
            assert_plan_equal(a, OP.build_plan(m.numpy(), bq, bk, 1))


def test_plan_empty_and_full_masks(bsa):
    for fill in (0, 1):
        m = torch.full((2, 4, 8, 12), fill, dtype=torch.uint8)
        _, a = gpu_plan_arrays(bsa, m, 64, 64, 2)
        assert_plan_equal(a, OP.build_plan(m.numpy(), 64, 64, 2))


def test_plan_many_rows_sort_segments(bsa):
    # > 256 rows: the schedule sort spans several segments with equal keys
    w = W.random_problem(7, 1, 8, 8, 8192, 4096, 16, 128, 128, 0.05)
    _, a = gpu_plan_arrays(bsa, w.mask, 128, 128, 1)
    assert_plan_equal(a, OP.build_plan(w.mask.numpy(), 128, 128, 1))


@pytest.mark.parametrize("bq,bk", [(128, 64), (64, 256), (32, 32)])
def test_plan_long_rows_and_unaligned_mask(bsa, bq, bk):
    # More than 1024 k-units per row (several 32-word stretches, a partial
    # last word), non-binary bytes; then the same mask at an odd address,
    # which the plan must read byte by byte.
    g = 2
    NKB = 1040 if bk <= 64 else 528
    gen = torch.Generator().manual_seed(bq * 7 + bk)
    vals = torch.randint(0, 256, (1, 4, 256 // bq * 2, NKB), generator=gen, dtype=torch.int32)
    keep = torch.rand(vals.shape, generator=gen) < 0.15
    m = torch.where(keep, vals.clamp(min=1), torch.zeros_like(vals)).to(torch.uint8).contiguous()
    ref = OP.build_plan(m.numpy(), bq, bk, g)
    _, a = gpu_plan_arrays(bsa, m, bq, bk, g)
    assert_plan_equal(a, ref)
    buf = torch.zeros(m.numel() + 16, dtype=torch.uint8, device="cuda")
    off = buf[1:1 + m.numel()].view(m.shape)
    off.copy_(m.cuda())
    assert off.data_ptr() % 16 == 1
    p = bsa.plan(off, bq, bk, g)
    a2 = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    a2["slot_mask"] = a2["slot_mask"].astype(np.int64) & 0xFFFFFFFF
    assert bsa.plan_check(p) == 0
    assert_plan_equal(a2, ref)



@pytest.mark.parametrize("name", ["tiny", "regular_small", "regular", "chunked_prefill_small"])
def test_plan_remap_workloads_bit_exact(bsa, name):
    w = W.make_workload(name, data=False)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group, flags=bsa.PLAN_REMAP)
    a = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    a["slot_mask"] = a["slot_mask"].astype(np.int64) & 0xFFFFFFFF
    assert bsa.plan_check(p) == 0
    ref = OP.build_plan(w.mask.numpy(), w.bq, w.bk, w.gqa_group, remap=True)
    assert_plan_equal(a, ref)
    if w.gqa_group > 1 or w.bq >= 128:
        assert set(a["plane_sigma"].tolist()) == {1}


@pytest.mark.parametrize("bq,bk,g", [(32, 32, 1), (32, 128, 1), (64, 64, 1), (64, 256, 1), (32, 64, 2)])
def test_plan_remap_random_masks(bsa, bq, bk, g):
    # strided rows (query block x selects key blocks = x mod 4, plus noise):
    # grouping strides other than 1 win on some planes
    B, H, Nq, Nk = 2, 4, 2048, 2048
    NQB, NKB = Nq // bq, Nk // bk
    gen = torch.Generator().manual_seed(bq * 5 + bk + g)
    m = (torch.rand(B, H, NQB, NKB, generator=gen) < 0.04).to(torch.uint8)
    x = torch.arange(NQB).view(NQB, 1)
    kb = torch.arange(NKB).view(1, NKB)
    m[:, 1] |= ((kb % 4) == (x % 4)).to(torch.uint8)
    m[:, 2] |= ((kb % 2) == (x % 2)).to(torch.uint8)
    p = bsa.plan(m.cuda(), bq, bk, g, flags=bsa.PLAN_REMAP)
    a = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    a["slot_mask"] = a["slot_mask"].astype(np.int64) & 0xFFFFFFFF
    assert bsa.plan_check(p) == 0
    ref = OP.build_plan(m.numpy(), bq, bk, g, remap=True)
    assert_plan_equal(a, ref)
    if g == 1:
        assert max(a["plane_sigma"].tolist()) > 1


@pytest.mark.parametrize("name,flags", [("chunked_prefill_small", 0), ("regular_small", 2)])
def test_plan_export_host_copies(bsa, name, flags):
    # bsa_plan_export: the same arrays as the device views, and the oracle's
    w = W.make_workload(name, data=False)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group, flags=flags)
    host = p.export()
    dev = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    for k in ("row_ptr", "slot_ku", "urow_ptr", "ukb", "order", "plane_sigma"):
        assert np.array_equal(host[k], dev[k]), k
    assert np.array_equal(host["slot_mask"].astype(np.int64), dev["slot_mask"].astype(np.int64) & 0xFFFFFFFF)
    ref = OP.build_plan(w.mask.numpy(), w.bq, w.bk, w.gqa_group, remap=bool(flags))
    host["slot_mask"] = host["slot_mask"].astype(np.int64)
    assert_plan_equal(host, ref)
    # a buffer too small: BSA_ERR_WORKSPACE, totals still written
    from block_sparse_attention_plan_gb300 import _lib as L
    import ctypes
    c = L.PlanArraysC()
    small = np.empty(1, np.int32)
    c.row_ptr, c.row_ptr_cap = ctypes.c_void_p(small.ctypes.data), 1
    assert L.library().bsa_plan_export(p.handle, None, ctypes.byref(c)) == -5
    assert list(c.totals)[:3] == host["totals"][:3].tolist()
