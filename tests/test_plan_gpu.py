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
    for k in ("row_ptr", "slot_ku", "slot_mask", "urow_ptr", "ukb", "order", "totals"):
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
