"""Oracle of the BSA plan (logical mask -> physical tiles) -- TEST INFRASTRUCTURE ONLY.

Source: "Decoupling Logical Masks from GPU Execution for Dynamic Block-Sparse
Attention" (Tessera), abstract: a physical mapping layer retains, combines or
subdivides logical attention blocks into physical tiles, and a task
organisation layer groups and schedules tiles within GPU tasks.
"CompactAttention: Accelerating Chunked Prefill with Block-Union KV Selection",
summary: a Q-block union plus an intra-group union give a GQA-aware per-group
KV block table.  The pages give no concrete rule; the plainest reading, used
here and by the CUDA path (which implements it independently), is:

Mapping (physical q-tile = T query rows, T = 128 or, for bq <= 64, 64;
physical K/V slot = 128 key rows):
  qu = min(bq,T) rows per q-unit, rq = T/qu q-units per q-tile,
  sq = bq/qu q-units per logical q-block (2 when bq = 256: subdivide);
  ku = min(bk,128) rows per k-unit, rk = 128/ku k-units per slot,
  sk = bk/ku k-units per logical k-block.
  bq = T / bk = 128 retains; smaller blocks are combined rq (rk) to a tile
  (slot); bq = 256 / bk = 256 are subdivided into two 128-row units.
  NQT = Nq/T q-tiles, NKU = Nk/ku k-units.  The 64-row tile is a second
  physical mapping of small query blocks: a 64-row q-block is a tile of its
  own instead of sharing a 128-row tile (and the union of selections) with a
  neighbour.
  Unit mask U[b,h,x,y] = mask[b,h,x // sq, y // sk] != 0.

Per plan row r = (b*H + h)*NQT + qt:
  u[y]   = OR over the rq q-units x in the tile of U[b,h,x,y]  (Q-block union)
  cnt    = |{y : u[y]}|,  slots = ceil(cnt / rk)
  row_ptr = exclusive prefix sum of slots (length R+1)
  slot_ku: the y with u[y], ascending, rk per slot, last slot padded with -1
  slot_mask[s]: bit (i*rk + j) = U[b, h, qt*rq + i, slot_ku[s, j]] (0 for padding)
GQA union (only when g = H/Hkv > 1), per union row (b*Hkv + hk)*NQT + qt:
  uu[y] = OR over the g query heads of the group of u[y]  (intra-group union)
  urow_ptr = exclusive prefix sum of |uu|; ukb = the y with uu[y], ascending
Schedule (task organisation for data reuse): rows are grouped by KV head --
  group id = (b*Hkv + hk), i.e. the g*NQT consecutive rows of the g query heads
  sharing one K/V head -- so that the rows running at one time share the K/V
  they gather.  Groups come in order of total slots descending (ties by group
  id); inside a group rows come by slots descending (longest row first), ties
  by ascending row id.
Totals: [total slots, selected logical blocks (mask != 0), union entries].

Pins (tests/test_oracle_plan.py): a hand-worked example written out in the
test; exhaustive enumeration of every mask on 3x3 logical grids for each
mapping; token-level round trip (the set of token pairs the plan covers with
sub-mask bits set equals the token-level expansion of the logical mask);
closed-form counts of the chunked-prefill workload (65 blocks per logical row);
permutation/monotonicity of the schedule.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

SUPPORTED_BLOCKS = (32, 64, 128, 256)
TILE = 128
TILES = (64, 128)   # physical q-tile heights


@dataclass
class Mapping:
    bq: int
    bk: int
    qu: int
    rq: int
    sq: int
    ku: int
    rk: int
    sk: int


def mapping(bq: int, bk: int, tile: int = TILE) -> Mapping:
    """Retain / combine / subdivide rule for one (bq, bk) pair and q-tile
    height ``tile`` (128, or 64 for bq <= 64); K/V slots are always 128 keys."""
    if bq not in SUPPORTED_BLOCKS or bk not in SUPPORTED_BLOCKS:
        raise ValueError(f"unsupported block sizes bq={bq} bk={bk}")
    if tile not in TILES or (tile == 64 and bq > 64):
        raise ValueError(f"unsupported q-tile height {tile} for bq={bq}")
    qu = min(bq, tile)
    ku = min(bk, TILE)
    return Mapping(bq, bk, qu, tile // qu, bq // qu, ku, TILE // ku, bk // ku)


def unit_mask(mask: np.ndarray, mp: Mapping) -> np.ndarray:
    """Boolean unit-level mask U [B,H,NQU,NKU]."""
    sel = np.asarray(mask) != 0
    return np.repeat(np.repeat(sel, mp.sq, axis=2), mp.sk, axis=3)


SIGMA_CANDIDATES = (1, 2, 4, 8, 16)


def tile_qunits(t: int, sigma: int, rq: int):
    """The rq q-units of q-tile t when a plane groups q-units with stride
    sigma: tiles come in runs of sigma; tile t = run*sigma + r holds q-units
    run*sigma*rq + r + i*sigma, i = 0 .. rq-1 (sigma = 1: t*rq + i)."""
    run, r = divmod(t, sigma)
    return [run * sigma * rq + r + i * sigma for i in range(rq)]


def plane_slots(Up: np.ndarray, sigma: int, rq: int, rk: int) -> int:
    """Slots a (b, h) plane needs (Up: bool [NQU, NKU]) with grouping stride
    sigma: the sum over its q-tiles of ceil(|union of the tile's q-units| / rk)."""
    NQT = Up.shape[0] // rq
    total = 0
    for t in range(NQT):
        n = int(Up[tile_qunits(t, sigma, rq)].any(axis=0).sum())
        total += -(-n // rk)
    return total


def choose_sigma(Up: np.ndarray, rq: int, rk: int) -> int:
    """Physical-mapping choice of one plane (Tessera, abstract: logical blocks
    are combined into physical tiles; reading: which q-units share a tile is
    chosen per plane).  Among the strides that tile the plane exactly
    (NQU divisible by sigma*rq), the one whose tiles need the fewest slots,
    ties to the smaller stride."""
    best, best_slots = 1, None
    for sigma in SIGMA_CANDIDATES:
        if Up.shape[0] % (sigma * rq):
            continue
        n = plane_slots(Up, sigma, rq, rk)
        if best_slots is None or n < best_slots:
            best, best_slots = sigma, n
    return best


def build_plan(mask, bq: int, bk: int, gqa_group: int = 1, remap: bool = False,
               tile: int = TILE) -> dict:
    """Return every plan array as numpy (int32 / uint32 / int64).

    remap: choose each (b, h) plane's q-unit grouping stride (choose_sigma);
    only when tiles combine several q-units (rq > 1) and without GQA
    grouping (gqa_group = 1), otherwise every plane keeps stride 1.  The
    strides are returned as plane_sigma [B*H].
    tile: q-tile height (see the mapping rule above)."""
    if hasattr(mask, "detach"):
        mask = mask.detach().cpu().numpy()
    mask = np.asarray(mask)
    mp = mapping(bq, bk, tile)
    B, H, NQB, NKB = mask.shape
    if H % gqa_group:
        raise ValueError("H must be a multiple of gqa_group")
    U = unit_mask(mask, mp)
    NQU, NKU = U.shape[2], U.shape[3]
    if NQU % mp.rq:
        raise ValueError(f"Nq must be a multiple of {tile}")
    NQT = NQU // mp.rq
    R = B * H * NQT

    # Grouping stride of each plane, then the q-units of each plane's tiles.
    sigma = np.ones(B * H, dtype=np.int64)
    if remap and mp.rq > 1 and gqa_group == 1:
        for bh in range(B * H):
            sigma[bh] = choose_sigma(U[bh // H, bh % H], mp.rq, mp.rk)
    Ut = np.empty((B, H, NQT, mp.rq, NKU), dtype=bool)
    for bh in range(B * H):
        for t in range(NQT):
            Ut[bh // H, bh % H, t] = U[bh // H, bh % H, tile_qunits(t, int(sigma[bh]), mp.rq)]
    # Q-block union over the q-units of each q-tile.
    u = Ut.any(axis=3)                                         # [B,H,NQT,NKU]
    cnt = u.sum(axis=3).reshape(R)
    slots = (cnt + mp.rk - 1) // mp.rk
    row_ptr = np.zeros(R + 1, dtype=np.int64)
    row_ptr[1:] = np.cumsum(slots)
    S = int(row_ptr[-1])
    slot_ku = np.full((S, mp.rk), -1, dtype=np.int64)
    slot_mask = np.zeros(S, dtype=np.uint64)
    ur = u.reshape(R, NKU)
    Ur = Ut.reshape(R, mp.rq, NKU)
    for r in range(R):
        ys = np.flatnonzero(ur[r])
        n = int(slots[r])
        if n == 0:
            continue
        padded = np.full(n * mp.rk, -1, dtype=np.int64)
        padded[:ys.size] = ys
        blk = padded.reshape(n, mp.rk)
        slot_ku[row_ptr[r]:row_ptr[r] + n] = blk
        bits = np.zeros(n, dtype=np.uint64)
        for i in range(mp.rq):
            for j in range(mp.rk):
                y = blk[:, j]
                on = np.zeros(n, dtype=bool)
                valid = y >= 0
                on[valid] = Ur[r, i, y[valid]]
                bits |= on.astype(np.uint64) << np.uint64(i * mp.rk + j)
        slot_mask[row_ptr[r]:row_ptr[r] + n] = bits

    # Schedule: KV-head groups heaviest first; longest row first inside a group.
    grows = gqa_group * NQT                       # rows per group (contiguous)
    G = R // grows
    work = [int(slots[gi * grows:(gi + 1) * grows].sum()) for gi in range(G)]
    order = []
    for gi in sorted(range(G), key=lambda x: (-work[x], x)):
        rows_g = range(gi * grows, (gi + 1) * grows)
        order.extend(sorted(rows_g, key=lambda r: (-int(slots[r]), r)))
    order = np.array(order, dtype=np.int64)

    # GQA per-group union table.
    if gqa_group > 1:
        Hkv = H // gqa_group
        uu = u.reshape(B, Hkv, gqa_group, NQT, NKU).any(axis=2).reshape(B * Hkv * NQT, NKU)
        ucnt = uu.sum(axis=1)
        urow_ptr = np.zeros(uu.shape[0] + 1, dtype=np.int64)
        urow_ptr[1:] = np.cumsum(ucnt)
        ukb = np.concatenate([np.flatnonzero(x) for x in uu]) if uu.shape[0] else np.zeros(0, np.int64)
    else:
        urow_ptr = np.zeros(1, dtype=np.int64)
        ukb = np.zeros(0, dtype=np.int64)

    totals = np.array([S, int((mask != 0).sum()), int(urow_ptr[-1])], dtype=np.int64)
    return {
        "mapping": mp,
        "NQT": NQT,
        "NKU": NKU,
        "rows": R,
        "row_ptr": row_ptr.astype(np.int32),
        "slot_ku": slot_ku.reshape(-1).astype(np.int32),
        "slot_mask": slot_mask.astype(np.uint32),
        "urow_ptr": urow_ptr.astype(np.int32),
        "ukb": ukb.astype(np.int32),
        "order": order.astype(np.int32),
        "totals": totals,
        "plane_sigma": sigma.astype(np.int32),
    }


def affine_mask(segments, B: int, H: int, NQB: int, NKB: int, base=None) -> np.ndarray:
    """Logical mask [B,H,NQB,NKB] (u8) of affine row descriptors.

    Source: "SPLAT: A framework for optimised GPU code-generation for SParse
    reguLar ATtention", abstract: the affine-compressed-sparse-row format
    describes the regular geometry of sparse attention patterns so that it can
    be analysed just in time.  The page gives no field layout; the reading
    used here and by the CUDA path (which implements it independently) is:
    each head h has a list of segments (a, b, stride, count) and query block
    qb selects the key blocks

        a*qb + b + stride*t,   t = 0 .. count-1,   kept when in [0, NKB),

    a = 1 placing the segment relative to the query block (sliding windows,
    strided and dilated patterns), a = 0 at fixed key blocks (global
    columns); stride may be negative, stride 0 repeats one block.  A head
    with segments selects their union, the same for every batch entry; a
    head without any takes its rows of ``base`` ([B,H,NQB,NKB], any non-zero
    byte selects; nothing when ``base`` is None), so irregular heads stay
    explicit rows of a compressed-sparse-row mask.
    ``segments[h]`` is the list of (a, b, stride, count) of head h.
    """
    m = np.zeros((B, H, NQB, NKB), dtype=np.uint8)
    for h in range(H):
        if not segments[h]:
            if base is not None:
                m[:, h] = (np.asarray(base)[:, h] != 0).astype(np.uint8)
            continue
        for (a, b, stride, count) in segments[h]:
            for qb in range(NQB):
                for t in range(count):
                    kb = a * qb + b + stride * t
                    if 0 <= kb < NKB:
                        m[:, h, qb, kb] = 1
    return m
