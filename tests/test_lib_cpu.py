"""The C-ABI library builds, loads and exports every symbol of include/bsa.h;
host-side argument validation and layout arithmetic (no GPU needed)."""
import ctypes
import os
import re

import pytest

from oracle import plan as OP
from block_sparse_attention_plan_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsa.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(bsa_[a-z_]+)\s*\(",
                                 src, flags=re.M)))


def test_exports_every_declared_symbol(bsa_lib):
    names = declared_functions()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(bsa_lib, n), f"libbsa.so does not export {n}"
    assert bsa_lib.bsa_version() == 1


def test_status_strings(bsa_lib):
    assert bsa_lib.bsa_status_string(0) == b"BSA_OK"
    assert bsa_lib.bsa_status_string(-6) == b"BSA_ERR_TIMEOUT"
    assert bsa_lib.bsa_status_string(-99) == b"BSA_ERR_UNKNOWN"


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_layout_matches_mapping_rule(bsa, name):
    w = W.make_workload(name, data=False)
    B, H, NQB, NKB = w.mask.shape
    L = bsa.plan_layout(B, H, NQB, NKB, w.bq, w.bk, w.gqa_group)
    mp = OP.mapping(w.bq, w.bk)
    assert (L.qu, L.rq, L.sq, L.ku, L.rk, L.sk) == (mp.qu, mp.rq, mp.sq, mp.ku, mp.rk, mp.sk)
    assert L.NQT == w.Nq // 128 and L.NKU == w.Nk // mp.ku
    assert L.rows == B * H * L.NQT
    assert L.urows == (B * w.Hkv * L.NQT if w.gqa_group > 1 else 0)
    assert L.max_row_slots == -(-L.NKU // L.rk)
    offs = [L.off_row_ptr, L.off_slot_ku, L.off_slot_mask, L.off_urow_ptr, L.off_ukb, L.off_order,
            L.off_totals, L.off_control, L.off_sigma, L.off_scratch]
    assert L.off_scratch - L.off_sigma >= 4 * B * H
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.off_slot_ku - L.off_slot_mask <= 0 and L.workspace_bytes > L.off_scratch
    assert L.off_slot_mask - L.off_slot_ku >= 4 * L.slot_capacity * L.rk


def test_layout_errors(bsa):
    with pytest.raises(bsa.BsaError) as e:
        bsa.plan_layout(1, 1, 3, 4, 64, 64)          # Nq = 192, not a multiple of 128
    assert e.value.status == -1
    with pytest.raises(bsa.BsaError) as e:
        bsa.plan_layout(1, 2, 4, 4, 48, 64)          # unsupported block size
    assert e.value.status == -2
    with pytest.raises(bsa.BsaError) as e:
        bsa.plan_layout(1, 3, 4, 4, 64, 64, gqa_group=2)  # H not a multiple of g
    assert e.value.status == -1
    with pytest.raises(bsa.BsaError) as e:
        bsa.plan_layout(1, 1, 4, 200000, 128, 32)    # too many slots per row for the sort
    assert e.value.status == -2


def test_create_and_forward_argument_errors_without_device(bsa_lib, bsa):
    L = bsa.plan_layout(1, 2, 4, 4, 128, 128)
    out = ctypes.c_void_p()
    buf = (ctypes.c_uint8 * 1024)()
    base = ctypes.addressof(buf)
    aligned = (base + 255) & ~255
    # null mask
    assert bsa_lib.bsa_plan_create(None, 1, 2, 4, 4, 128, 128, 1, ctypes.c_void_p(aligned),
                                   L.workspace_bytes, 0, None, ctypes.byref(out)) == -1
    # misaligned workspace
    assert bsa_lib.bsa_plan_create(ctypes.c_void_p(aligned), 1, 2, 4, 4, 128, 128, 1,
                                   ctypes.c_void_p(aligned + 16), L.workspace_bytes, 0, None,
                                   ctypes.byref(out)) == -1
    # workspace too small
    assert bsa_lib.bsa_plan_create(ctypes.c_void_p(aligned), 1, 2, 4, 4, 128, 128, 1,
                                   ctypes.c_void_p(aligned), L.workspace_bytes - 1, 0, None,
                                   ctypes.byref(out)) == -5
    # null out-parameter, bad flags
    assert bsa_lib.bsa_plan_create(ctypes.c_void_p(aligned), 1, 2, 4, 4, 128, 128, 1,
                                   ctypes.c_void_p(aligned), L.workspace_bytes, 0, None, None) == -1
    assert bsa_lib.bsa_plan_create(ctypes.c_void_p(aligned), 1, 2, 4, 4, 128, 128, 1,
                                   ctypes.c_void_p(aligned), L.workspace_bytes, 0x10, None,
                                   ctypes.byref(out)) == -1
    # forward: NULL plan, then a foreign object posing as a plan
    p = ctypes.c_void_p(aligned)
    assert bsa_lib.bsa_forward(None, p, p, p, p, p, 128, 0.0, None) == -1
    fake = (ctypes.c_uint32 * 64)()
    assert bsa_lib.bsa_forward(ctypes.c_void_p(ctypes.addressof(fake)), p, p, p, p, p, 128, 0.0,
                               None) == -7
    assert bsa_lib.bsa_sync_status(None, None, None) == -1
    assert bsa_lib.bsa_plan_check(None, None) == -1
    assert bsa_lib.bsa_watchdog_selftest(None, 1000, None) == -1
    bsa_lib.bsa_plan_destroy(None)  # no-op



def test_plan_flags_and_layout_independent_of_remap(bsa):
    L0 = bsa.plan_layout(2, 16, 256, 256, 32, 32, 1)
    L1 = bsa.plan_layout(2, 16, 256, 256, 32, 32, 1, bsa.PLAN_REMAP)
    assert L0.as_dict() == L1.as_dict()  # regrouping needs no extra workspace
    with pytest.raises(bsa.BsaError) as e:
        bsa.plan_layout(2, 16, 256, 256, 32, 32, 1, 0x8)  # unknown flag
    assert e.value.status == -1
    # 64-row q-tiles: twice the q-tiles (plan rows); two 32-row blocks per tile
    L2 = bsa.plan_layout(2, 16, 256, 256, 32, 32, 1, bsa.PLAN_Q64)
    assert (L2.NQT, L2.rq, L2.qu, L2.rows) == (2 * L0.NQT, 2, 32, 2 * L0.rows)
    with pytest.raises(bsa.BsaError) as e:
        bsa.plan_layout(2, 16, 64, 64, 128, 32, 1, bsa.PLAN_Q64)  # blocks of more than 64 rows
    assert e.value.status == -2


def test_host_pipeline_buffer_sizes(bsa):
    from block_sparse_attention_plan_gb300 import _lib as L
    # video-DiT geometry: 24 units; chunks clamp to [1, units]; two slots
    # from two chunks on; each slot holds one chunk's inputs, outputs and plan.
    one = L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 128, 1)
    two = L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 128, 2)
    eight = L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 128, 8)
    many = L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 128, 1000)
    per_unit = 3 * 16384 * 128 * 2 + 16384 * 128 * 2 + 16384 * 4 + 128 * 128  # Q, K, V, O, LSE, mask
    assert one >= 24 * per_unit
    assert two >= 2 * 12 * per_unit and two < one * 1.2
    assert eight >= 2 * 3 * per_unit and eight < two
    assert many == L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 128, 24)
    for bad in ((0,), (-3,)):
        with pytest.raises(bsa.BsaError):
            L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 128, *bad)
    with pytest.raises(bsa.BsaError):
        L.host_buffer_bytes(1, 24, 128, 128, 128, 128, 1, 96, 8)  # d not 64 / 128


def test_affine_stage_and_host_argument_errors_without_device(bsa_lib, bsa):
    # Every check below returns before the library touches a device: the
    # pointers are host addresses that are never dereferenced.
    L = bsa.plan_layout(1, 2, 4, 4, 128, 128)
    out = ctypes.c_void_p()
    buf = (ctypes.c_uint8 * 4096)()
    aligned = (ctypes.addressof(buf) + 255) & ~255
    VP = ctypes.c_void_p
    geo = (1, 2, 4, 4, 128, 128, 1)
    ws = (VP(aligned), L.workspace_bytes)
    # affine plans: no seg_ptr; segments missing or misaligned; bad workspace
    assert bsa_lib.bsa_plan_create_affine(None, VP(aligned), None, 1, *geo, *ws, 0, None,
                                          ctypes.byref(out)) == -1
    assert bsa_lib.bsa_plan_create_affine(None, None, VP(aligned), 1, *geo, *ws, 0, None,
                                          ctypes.byref(out)) == -1
    assert bsa_lib.bsa_plan_create_affine(None, VP(aligned + 4), VP(aligned), 1, *geo, *ws, 0,
                                          None, ctypes.byref(out)) == -1
    assert bsa_lib.bsa_plan_create_affine(None, VP(aligned), VP(aligned), -1, *geo, *ws, 0, None,
                                          ctypes.byref(out)) == -1
    assert bsa_lib.bsa_plan_create_affine(None, VP(aligned), VP(aligned), 1, *geo, VP(aligned),
                                          L.workspace_bytes - 1, 0, None, ctypes.byref(out)) == -5
    # staged forward: empty or unknown stage sets are rejected first
    p = VP(aligned)
    for bad in (0, -1, 0x20, 0x40):
        assert bsa_lib.bsa_forward_stage(None, p, p, p, None, None, 0, p, p, 128, 0.0, bad,
                                         None) == -1
    assert bsa_lib.bsa_forward_stage(None, p, p, p, None, None, 0, p, p, 128, 0.0,
                                     bsa.STAGE_ALL, None) == -1       # NULL plan
    # host pipeline: NULL buffers, misaligned device buffer, too small, bad chunks
    n = ctypes.c_size_t(0)
    assert bsa_lib.bsa_attention_host_buffer_bytes(1, 2, 4, 4, 128, 128, 1, 64, 2, ctypes.byref(n)) == 0
    args = (p, 1, 2, 4, 4, 128, 128, 1, p, p, p, p, p, 64, 0.0)
    assert bsa_lib.bsa_attention_host(None, *args[1:], 2, p, n.value, None) == -1
    assert bsa_lib.bsa_attention_host(*args, 2, VP(aligned + 16), n.value, None) == -1
    assert bsa_lib.bsa_attention_host(*args, 2, p, n.value - 1, None) == -5
    assert bsa_lib.bsa_attention_host(*args, 0, p, n.value, None) == -1


def test_plan_workspace_bytes_matches_layout(bsa):
    for geo in ((1, 24, 128, 128, 128, 128, 1), (1, 32, 64, 1024, 64, 64, 4), (2, 16, 256, 256, 32, 32, 1)):
        assert bsa.plan_workspace_bytes(*geo) == bsa.plan_layout(*geo).workspace_bytes
        assert bsa.plan_workspace_bytes(*geo) == bsa.plan_layout(*geo, bsa.PLAN_REMAP).workspace_bytes
    assert bsa.plan_workspace_bytes(1, 1, 3, 4, 64, 64, 1) == 0     # Nq = 192
    assert bsa.plan_workspace_bytes(1, 2, 4, 4, 48, 64, 1) == 0     # unsupported block


def test_plan_export_argument_errors_without_device(bsa_lib):
    from block_sparse_attention_plan_gb300 import _lib as L
    c = L.PlanArraysC()
    assert bsa_lib.bsa_plan_export(None, None, ctypes.byref(c)) == -1
    fake = (ctypes.c_uint32 * 64)()
    assert bsa_lib.bsa_plan_export(ctypes.c_void_p(ctypes.addressof(fake)), None, ctypes.byref(c)) == -1


def test_plan_select_flags_from_table(bsa):
    from block_sparse_attention_plan_gb300 import regime_sweep as RS
    table = {}
    for line in open(RS.TABLE_H):
        m = re.match(r"\s*\{(\d+), (\d+), (\d+), (\d+)\},", line)
        if m:
            bq, bk, d, tile = map(int, m.groups())
            table[(bq, bk, d)] = tile
    for (bq, bk, d) in [(32, 32, 64), (64, 64, 128), (64, 128, 128), (32, 64, 64), (128, 128, 128)]:
        for g in (1, 2):
            f = bsa.select_flags(1, 4, 4096 // bq, 4096 // bk, bq, bk, g, d)
            tile = table.get((bq, bk, d), 128) if bq <= 64 else 128
            assert bool(f & bsa.PLAN_Q64) == (tile == 64), (bq, bk, d, g, f)
            rq = tile // min(bq, tile)
            assert bool(f & bsa.PLAN_REMAP) == (rq > 1 and g == 1), (bq, bk, d, g, f)
            L = bsa.plan_layout(1, 4, 4096 // bq, 4096 // bk, bq, bk, g, f)  # a valid plan layout
            assert L.qu * L.rq == tile
    with pytest.raises(bsa.BsaError):
        bsa.select_flags(1, 2, 4, 4, 48, 64, 1, 128)   # unsupported block size
    with pytest.raises(bsa.BsaError):
        bsa.select_flags(1, 2, 4, 4, 64, 64, 1, 96)    # unsupported head dim


def test_regime_choice_rule():
    # the sweep keeps, per (bq, bk, d), the tile with the smaller geometric-mean time
    from block_sparse_attention_plan_gb300 import regime_sweep as RS
    rows = [{"bq": 64, "bk": 64, "d": 128, "tile": t, "kernel_ms": ms}
            for t, ms in ((128, 1.0), (128, 4.0), (64, 1.5), (64, 2.5))]   # gm 2.0 vs 1.94
    rows += [{"bq": 32, "bk": 32, "d": 64, "tile": t, "kernel_ms": ms} for t, ms in ((128, 1.0), (64, 3.0))]
    best = RS.choose(rows)
    assert best[(64, 64, 128)][0] == 64 and best[(32, 32, 64)][0] == 128
