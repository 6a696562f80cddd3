"""Pins for the plan oracle (CPU only).

The plan oracle is checked against hand-derived examples
(tests/golden/plan_hand_examples.json), against a token-level reconstruction
(the set of (query, key) token pairs the plan covers with a set sub-mask bit
must equal the token-level expansion of the logical mask: Tessera abstract,
"preserving specified attention interactions"), by exhaustive enumeration of
every mask on small logical grids for every mapping, against Python set unions
for the GQA table (CompactAttention summary), and against closed-form counts of
the chunked-prefill workload.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

from oracle import plan as OP
from block_sparse_attention_plan_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_hand_examples.json")
KEYS = ("row_ptr", "slot_ku", "slot_mask", "urow_ptr", "ukb", "order", "totals")


def tile_rows(qt: int, sigma: int, rq: int):
    """Plan format: the q-units row qt of a plane with grouping stride sigma
    covers (runs of sigma tiles; tile run*sigma + r holds q-units
    run*sigma*rq + r + i*sigma)."""
    run, r = qt // sigma, qt % sigma
    return [run * sigma * rq + r + i * sigma for i in range(rq)]


def check_plan_invariants(mask: np.ndarray, bq: int, bk: int, g: int, p: dict, tile: int = 128):
    """Structural checks written independently of the oracle's construction
    (``tile``: q-tile height; K/V slots hold 128 keys)."""
    B, H, NQB, NKB = mask.shape
    Nq, Nk = NQB * bq, NKB * bk
    qu, ku = min(bq, tile), min(bk, 128)
    rq, rk = tile // qu, 128 // ku
    NQT = Nq // tile
    R = B * H * NQT
    rp, sk, sm = p["row_ptr"].astype(np.int64), p["slot_ku"].reshape(-1, rk), p["slot_mask"]
    assert rp[0] == 0 and rp.size == R + 1 and np.all(np.diff(rp) >= 0)
    assert p["totals"][0] == rp[-1] == sk.shape[0] == sm.size
    assert p["totals"][1] == int((mask != 0).sum())
    # token-level coverage
    want = np.zeros((B, H, Nq, Nk), dtype=bool)
    sel = mask != 0
    for b, h, qb, kb in zip(*np.nonzero(sel)):
        want[b, h, qb * bq:(qb + 1) * bq, kb * bk:(kb + 1) * bk] = True
    got = np.zeros_like(want)
    sig = p.get("plane_sigma", np.ones(B * H, dtype=np.int32))
    for bh in range(B * H):  # every plane's tiles partition its q-units
        units = sorted(x for qt in range(NQT) for x in tile_rows(qt, int(sig[bh]), rq))
        assert units == list(range(NQT * rq))
    for r in range(R):
        b, rem = divmod(r, H * NQT)
        h, qt = divmod(rem, NQT)
        xs = tile_rows(qt, int(sig[b * H + h]), rq)
        ks = sk[rp[r]:rp[r + 1]].ravel()
        valid = ks[ks >= 0]
        # ascending, unique, padding only at the tail of the last slot
        assert np.all(np.diff(valid) > 0)
        assert np.all(ks[:valid.size] == valid)
        assert rp[r + 1] - rp[r] == -(-valid.size // rk)  # ceil
        for s in range(rp[r], rp[r + 1]):
            bits = int(sm[s])
            assert bits >> (rq * rk) == 0
            for j in range(rk):
                y = int(sk[s, j])
                if y < 0:
                    assert all(((bits >> (i * rk + j)) & 1) == 0 for i in range(rq))
                    continue
                assert 0 <= y < Nk // ku
                col_on = False
                for i in range(rq):
                    if (bits >> (i * rk + j)) & 1:
                        col_on = True
                        q0 = xs[i] * qu
                        got[b, h, q0:q0 + qu, y * ku:(y + 1) * ku] = True
                assert col_on, "a listed k-unit must be selected by some q-unit of the tile"
    np.testing.assert_array_equal(got, want)
    # schedule: a permutation; KV-head groups contiguous, heaviest group first
    # (ties by group id); inside a group slots non-increasing, ties by row id
    order = p["order"].astype(np.int64)
    assert sorted(order.tolist()) == list(range(R))
    nsl = np.diff(rp)
    Hkv = H // g
    gid = lambda r: (r // (H * NQT)) * Hkv + ((r // NQT) % H) // g
    gsz = g * NQT
    groups = [gid(int(r)) for r in order]
    seq = [groups[i] for i in range(0, R, gsz)]
    for i in range(0, R, gsz):
        assert len(set(groups[i:i + gsz])) == 1            # contiguous
    work = {gg: int(sum(nsl[r] for r in range(R) if gid(r) == gg)) for gg in set(groups)}
    for a, c in zip(seq[:-1], seq[1:]):
        assert work[a] > work[c] or (work[a] == work[c] and a < c)
    for i in range(0, R, gsz):
        blk = order[i:i + gsz]
        for a, c in zip(blk[:-1], blk[1:]):
            assert nsl[a] > nsl[c] or (nsl[a] == nsl[c] and a < c)
    # GQA union table against Python sets
    if g > 1:
        Hkv = H // g
        urp, ukb = p["urow_ptr"].astype(np.int64), p["ukb"]
        assert urp.size == B * Hkv * NQT + 1 and p["totals"][2] == urp[-1]
        for b in range(B):
            for hk in range(Hkv):
                for qt in range(NQT):
                    s = set()
                    for h in range(hk * g, (hk + 1) * g):
                        r = (b * H + h) * NQT + qt
                        s |= set(int(y) for y in sk[rp[r]:rp[r + 1]].ravel() if y >= 0)
                    ur = (b * Hkv + hk) * NQT + qt
                    assert ukb[urp[ur]:urp[ur + 1]].tolist() == sorted(s)
    else:
        assert p["urow_ptr"].tolist() == [0] and p["ukb"].size == 0 and p["totals"][2] == 0


def test_hand_worked_examples():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        mask = np.array(c["mask"], dtype=np.uint8)
        tile = c.get("tile", 128)
        p = OP.build_plan(mask, c["bq"], c["bk"], c["gqa_group"], tile=tile)
        for k in KEYS:
            assert p[k].tolist() == c[k], (c["name"], k, p[k].tolist(), c[k])
        check_plan_invariants(mask, c["bq"], c["bk"], c["gqa_group"], p, tile)


GRIDS = {32: 4, 64: 2, 128: 3, 256: 3}  # NQB so that Nq is a multiple of 128


@pytest.mark.parametrize("bq,bk", list(itertools.product((32, 64, 128, 256), repeat=2)))
def test_exhaustive_small_grids(bq, bk):
    nqb = GRIDS[bq]
    nkb = max(1, 9 // nqb) if nqb != 4 else 2
    n = nqb * nkb
    for bits in range(1 << n):
        m = np.array([(bits >> t) & 1 for t in range(n)], dtype=np.uint8).reshape(1, 1, nqb, nkb)
        p = OP.build_plan(m, bq, bk, 1)
        check_plan_invariants(m, bq, bk, 1, p)


@pytest.mark.parametrize("bq,bk", list(itertools.product((32, 64), (32, 64, 128, 256))))
def test_exhaustive_small_grids_tile64(bq, bk):
    # 64-row q-tiles: a 64-row q-block is a tile of its own, two 32-row
    # q-blocks share one
    nqb = 4 if bq == 32 else 3
    nkb = 2 if bq == 32 else 3
    n = nqb * nkb
    for bits in range(1 << n):
        m = np.array([(bits >> t) & 1 for t in range(n)], dtype=np.uint8).reshape(1, 1, nqb, nkb)
        p = OP.build_plan(m, bq, bk, 1, tile=64)
        check_plan_invariants(m, bq, bk, 1, p, tile=64)


@pytest.mark.parametrize("bq,bk,g", [(64, 32, 2), (32, 64, 4), (128, 256, 2), (256, 64, 1)])
def test_random_masks_nonbinary_bytes(bq, bk, g):
    w = W.random_problem(11, 2, 4, 4 // g, 512, 768, 16, bq, bk, 0.3, values=True)
    m = w.mask.numpy()
    assert m.max() > 1
    p = OP.build_plan(m, bq, bk, g)
    check_plan_invariants(m, bq, bk, g, p)


def test_chunked_prefill_closed_form_counts():
    w = W.make_workload("chunked_prefill", data=False)
    m = w.mask.numpy()
    assert np.all((m != 0).sum(-1) == 65)            # sink + 16-block window + top-48
    assert int((m != 0).sum()) == 32 * 64 * 65 == 133120
    p = OP.build_plan(m, 64, 64, 4)
    assert p["totals"][1] == 133120
    rp = p["row_ptr"].astype(np.int64)
    sk = p["slot_ku"].reshape(-1, 2)
    # each q-tile covers q-blocks 2t, 2t+1: its unit count is the size of the
    # union of their two 65-block sets
    for h in (0, 17, 31):
        for qt in (0, 13, 31):
            r = h * 32 + qt
            s = set(np.flatnonzero(m[0, h, 2 * qt])) | set(np.flatnonzero(m[0, h, 2 * qt + 1]))
            ks = sk[rp[r]:rp[r + 1]].ravel()
            assert sorted(s) == ks[ks >= 0].tolist()


def test_chunked_prefill_closed_form_tile64():
    # one 64-row q-block per tile: each row lists exactly its q-block's 65
    # selected k-blocks, in ceil(65 / 2) = 33 slots
    w = W.make_workload("chunked_prefill", data=False)
    m = w.mask.numpy()
    p = OP.build_plan(m, 64, 64, 4, tile=64)
    rp = p["row_ptr"].astype(np.int64)
    assert np.all(np.diff(rp) == 33) and p["totals"][0] == 32 * 64 * 33 == 67584
    sk = p["slot_ku"].reshape(-1, 2)
    for h in (0, 9, 31):
        for qb in (0, 40, 63):
            r = h * 64 + qb
            ks = sk[rp[r]:rp[r + 1]].ravel()
            assert ks[ks >= 0].tolist() == np.flatnonzero(m[0, h, qb]).tolist()
            assert ks[-1] == -1   # 65 units: the last slot is half padding


def test_random_masks_tile64_gqa_and_remap():
    for bq, bk, g in ((64, 32, 2), (32, 64, 4), (32, 128, 1), (64, 256, 1)):
        w = W.random_problem(17 + bq + bk, 2, 4, 4 // g, 512, 768, 16, bq, bk, 0.3, values=True)
        m = w.mask.numpy()
        check_plan_invariants(m, bq, bk, g, OP.build_plan(m, bq, bk, g, tile=64), tile=64)
        if g == 1 and bq == 32:
            check_plan_invariants(m, bq, bk, g, OP.build_plan(m, bq, bk, g, remap=True, tile=64), tile=64)


def test_mapping_rule():
    assert (OP.mapping(128, 128).rq, OP.mapping(128, 128).rk) == (1, 1)
    mp = OP.mapping(32, 64)
    assert (mp.qu, mp.rq, mp.sq, mp.ku, mp.rk, mp.sk) == (32, 4, 1, 64, 2, 1)
    mp = OP.mapping(256, 256)
    assert (mp.qu, mp.rq, mp.sq, mp.ku, mp.rk, mp.sk) == (128, 1, 2, 128, 1, 2)
    mp = OP.mapping(32, 64, tile=64)
    assert (mp.qu, mp.rq, mp.sq, mp.ku, mp.rk, mp.sk) == (32, 2, 1, 64, 2, 1)
    mp = OP.mapping(64, 256, tile=64)
    assert (mp.qu, mp.rq, mp.sq, mp.ku, mp.rk, mp.sk) == (64, 1, 1, 128, 1, 2)
    with pytest.raises(ValueError):
        OP.mapping(128, 64, tile=64)   # the 64-row tile is for blocks of at most 64 rows
    with pytest.raises(ValueError):
        OP.mapping(48, 64)
    with pytest.raises(ValueError):
        OP.build_plan(np.ones((1, 1, 3, 2), np.uint8), 64, 64)  # Nq = 192


# ---- affine row descriptors (SPLAT's ACSR reading) -------------------------
# Each expansion is checked against the pattern's plain definition written
# with numpy broadcasting over D = qb - kb, not against another expansion.

def _D(NQB, NKB):
    return np.subtract.outer(np.arange(NQB), np.arange(NKB))


def test_affine_sliding_window_is_a_band():
    NQB, NKB, W = 37, 41, 5
    m = OP.affine_mask([[(1, -(W - 1), 1, 2 * W - 1)]], 1, 1, NQB, NKB)
    assert np.array_equal(m[0, 0] != 0, np.abs(_D(NQB, NKB)) < W)


def test_affine_strided_pattern():
    NB, s = 64, 8
    K = -(-NB // s)
    segs = [[(1, -(s - 1), 1, 2 * s - 1), (1, -s * K, s, 2 * K + 1)]]
    m = OP.affine_mask(segs, 2, 1, NB, NB)
    D = _D(NB, NB)
    want = (np.abs(D) < s) | (D % s == 0)
    assert np.array_equal(m[0, 0] != 0, want) and np.array_equal(m[1, 0], m[0, 0])


def test_affine_dilated_and_negative_stride():
    NB, R = 50, 13
    half = R // 2
    fwd = OP.affine_mask([[(1, -2 * half, 2, 2 * half + 1)]], 1, 1, NB, NB)
    rev = OP.affine_mask([[(1, 2 * half, -2, 2 * half + 1)]], 1, 1, NB, NB)
    D = _D(NB, NB)
    assert np.array_equal(fwd[0, 0] != 0, (np.abs(D) <= R) & (D % 2 == 0))
    assert np.array_equal(fwd, rev)


def test_affine_global_columns_zero_stride_and_explicit_heads():
    NQB, NKB, G = 9, 20, 3
    base = np.zeros((2, 3, NQB, NKB), dtype=np.uint8)
    base[0, 1, 4, 17] = 9          # ignored: head 1 has segments
    base[1, 2, 5, 6] = 1           # head 2 has none: its rows come from base
    base[0, 2, 0, 0] = 200
    segs = [[(0, 0, 1, G)], [(0, 11, 0, 4), (1, 100, 1, 3)], []]  # head 1: one column (stride 0), one segment off the grid
    m = OP.affine_mask(segs, 2, 3, NQB, NKB, base=base)
    want0 = np.zeros((NQB, NKB), dtype=bool)
    want0[:, :G] = True
    want1 = np.zeros((NQB, NKB), dtype=bool)
    want1[:, 11] = True
    for b in range(2):
        assert np.array_equal(m[b, 0] != 0, want0)
        assert np.array_equal(m[b, 1] != 0, want1)
    assert np.array_equal(m[:, 2] != 0, base[:, 2] != 0)
    assert OP.affine_mask([[], [(1, 0, 1, 0)]], 1, 2, 4, 4).sum() == 0  # no base, count 0: nothing


# ---- per-plane q-unit grouping (physical mapping chosen at plan time) -----

def test_remap_hand_example():
    # 8 query blocks of 32 rows (four q-units per tile), 8 key blocks of 128
    # (one unit per slot).  Query block x selects key block x % 2.
    # Stride 1: tiles {0,1,2,3} and {4,5,6,7} each need key blocks {0,1}: 4 slots.
    # Stride 2: tiles {0,2,4,6} -> {0} and {1,3,5,7} -> {1}: 2 slots.
    # Stride 4 would need 16 q-units.  So stride 2: rows [0], [1], each slot's
    # sub-mask has all four q-units (bits 0..3).
    m = np.zeros((1, 1, 8, 8), dtype=np.uint8)
    for x in range(8):
        m[0, 0, x, x % 2] = 1
    p = OP.build_plan(m, 32, 128, 1, remap=True)
    assert p["plane_sigma"].tolist() == [2]
    assert p["row_ptr"].tolist() == [0, 1, 2]
    assert p["slot_ku"].tolist() == [0, 1]
    assert p["slot_mask"].tolist() == [0b1111, 0b1111]
    assert OP.build_plan(m, 32, 128, 1)["plane_sigma"].tolist() == [1]
    check_plan_invariants(m, 32, 128, 1, p)


def test_remap_tie_keeps_stride_one():
    m = np.ones((1, 2, 16, 4), dtype=np.uint8)  # every grouping needs the same slots
    assert OP.build_plan(m, 32, 128, 1, remap=True)["plane_sigma"].tolist() == [1, 1]


def _slots_by_sets(sel, sigma, rq, rk):
    NQT = sel.shape[0] // rq
    total = 0
    for qt in range(NQT):
        cols = set()
        for x in tile_rows(qt, sigma, rq):
            cols |= set(np.flatnonzero(sel[x]).tolist())
        total += -(-len(cols) // rk)
    return total


@pytest.mark.parametrize("bq,bk", [(32, 32), (64, 128), (32, 256), (64, 64)])
def test_remap_choice_is_minimal_and_plan_valid(bq, bk):
    W_ = W.regular_mask(torch.Generator().manual_seed(bq + bk), 1, 4, 64 if bq == 32 else 32,
                        window=3, stride=4, dil_reach=9, glob=2, bb_window=2, bb_p=0.1)
    m = W_.numpy()
    if bk != bq:  # reshape the key axis to bk-sized blocks: keep NKB = Nk / bk
        NKB = m.shape[2] * bq // bk
        m = m[..., :NKB]
    p = OP.build_plan(m, bq, bk, 1, remap=True)
    check_plan_invariants(m, bq, bk, 1, p)
    mp = OP.mapping(bq, bk)
    U = OP.unit_mask(m, mp)
    for h in range(m.shape[1]):
        cand = {s: _slots_by_sets(U[0, h], s, mp.rq, mp.rk) for s in OP.SIGMA_CANDIDATES
                if U.shape[2] % (s * mp.rq) == 0}
        best = min(cand, key=lambda s: (cand[s], s))
        assert int(p["plane_sigma"][h]) == best, (h, cand)
    assert int(np.diff(p["row_ptr"]).sum()) <= int(np.diff(OP.build_plan(m, bq, bk, 1)["row_ptr"]).sum())
