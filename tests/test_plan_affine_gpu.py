"""GPU tests of bsa_plan_create_affine: plans of affine row descriptors
(SPLAT's ACSR reading: key blocks a*qb + b + stride*t) must equal, array by
array, the plan oracle of the expanded mask (oracle.plan.affine_mask), with
and without mask bytes OR-ed in; and the forward on such a plan must equal
the forward on the plan of the expanded mask."""
import itertools

import numpy as np
import pytest
import torch

from oracle import plan as OP
from block_sparse_attention_plan_gb300 import workloads as W
from test_plan_gpu import assert_plan_equal

pytestmark = pytest.mark.gpu


def arrays(bsa, p):
    a = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in p.arrays().items()}
    a["slot_mask"] = a["slot_mask"].astype(np.int64) & 0xFFFFFFFF
    assert bsa.plan_check(p) == 0
    return a


def mixed_segments(NKB):
    return [
        [(1, -2, 1, 5)],                                   # sliding window
        [(1, -3, 1, 7), (1, -4 * 40, 4, 81)],              # strided (most of it off the grid)
        [(1, 6, -2, 7)],                                   # dilated, negative stride
        [(0, 0, 1, 2), (1, -1, 1, 3), (1, NKB - 5, 1, 10), (0, 7, 0, 3), (1, 0, 1, 0)],
    ]


@pytest.mark.parametrize("bq,bk", list(itertools.product((32, 64, 128, 256), repeat=2)))
def test_affine_plan_all_mappings(bsa, bq, bk):
    B, H, g = 2, 4, (2 if (bq + bk) % 3 else 1)
    NQB, NKB = 1024 // bq, 1536 // bk
    segs = mixed_segments(NKB)
    p = bsa.plan_affine(segs, B, NQB, NKB, bq, bk, g)
    assert_plan_equal(arrays(bsa, p), OP.build_plan(OP.affine_mask(segs, B, H, NQB, NKB), bq, bk, g))
    # heads 1 and 3 as explicit mask rows; the mask rows of heads 0 and 2 are ignored
    gen = torch.Generator().manual_seed(bq * 3 + bk)
    base = (torch.rand(B, H, NQB, NKB, generator=gen) < 0.05).to(torch.uint8) * 7
    hyb = [segs[0], [], segs[2], []]
    p2 = bsa.plan_affine(hyb, B, NQB, NKB, bq, bk, g, mask=base.cuda())
    assert_plan_equal(arrays(bsa, p2),
                      OP.build_plan(OP.affine_mask(hyb, B, H, NQB, NKB, base=base.numpy()), bq, bk, g))


@pytest.mark.parametrize("name", ["regular_small", "regular"])
def test_affine_regular_workload_plan_and_forward(bsa, name):
    w = W.make_workload(name)
    B, H, NQB, NKB = w.mask.shape
    kw = {} if name == "regular" else dict(window=4, stride=4, dil_reach=20, glob=2, bb_window=3)
    segs, mask_heads = W.regular_segments(H, NKB, **kw)
    assert all(not segs[h] for h in mask_heads)
    pa = bsa.plan_affine(segs, B, NQB, NKB, w.bq, w.bk, w.gqa_group, mask=w.mask.cuda())
    pm = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    a, m = arrays(bsa, pa), arrays(bsa, pm)
    assert_plan_equal(a, {k: m[k] for k in ("row_ptr", "slot_ku", "slot_mask", "urow_ptr", "ukb", "order")}
                      | {"totals": np.asarray(m["totals"])[:3]})
    if name == "regular":
        return
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    oa, la = bsa.forward(pa, q, k, v)
    om, lm = bsa.forward(pm, q, k, v)
    assert bsa.sync_status(pa)[0] == 0 and bsa.sync_status(pm)[0] == 0
    assert torch.equal(oa, om) and torch.equal(la, lm)


def test_affine_plan_argument_errors(bsa):
    import ctypes
    from block_sparse_attention_plan_gb300 import _lib as L
    lib = L.library()
    seg, ptr, n = L.affine_segments([[(1, 0, 1, 3)]])
    Lay = bsa.plan_layout(1, 1, 8, 8, 128, 128)
    ws = torch.empty(int(Lay.workspace_bytes), dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p()
    VP = ctypes.c_void_p
    args = (1, 1, 8, 8, 128, 128, 1, VP(ws.data_ptr()), ws.numel(), 0, None, ctypes.byref(h))
    assert lib.bsa_plan_create_affine(None, VP(seg.data_ptr()), None, n, *args) == -1       # no seg_ptr
    assert lib.bsa_plan_create_affine(None, VP(seg.data_ptr() + 4), VP(ptr.data_ptr()), n, *args) == -1  # misaligned
    assert lib.bsa_plan_create_affine(None, None, VP(ptr.data_ptr()), 1, *args) == -1       # segments missing
    assert lib.bsa_plan_create_affine(None, VP(seg.data_ptr()), VP(ptr.data_ptr()), n, *args) == 0
    lib.bsa_plan_destroy(h)
