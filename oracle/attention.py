"""fp64 oracle of block-sparse attention forward -- TEST INFRASTRUCTURE ONLY.

What BSA computes ("Decoupling Logical Masks from GPU Execution for Dynamic
Block-Sparse Attention" (Tessera), abstract): attention restricted to the
(query-block, key-block) pairs a logical mask selects; the pairs it does not
select are not computed, and the selected interactions are preserved exactly.
The pages print no formula, so the plainest reading is written out here:

    for each batch b, query head h and query row i (kv head hk = h // g):
      J  = { j : mask[b, h, i // bq, j // bk] != 0 }          (allowed keys)
      J empty  ->  O[i] = 0,  LSE[i] = -inf
      else     ->  s_j = scale * <Q[b,h,i], K[b,hk,j]>,  scale = 1/sqrt(d)
                   m = max_j s_j,  l = sum_j exp(s_j - m)
                   O[i] = sum_j exp(s_j - m) V[b,hk,j] / l,  LSE[i] = m + ln l

Inputs are bf16 values, which fp64 represents exactly; everything is computed
in fp64.  Any non-zero mask byte selects.

Element mask (optional; the paged/chunked-prefill path of "CompactAttention:
Accelerating Chunked Prefill with Block-Union KV Selection", summary, where
the queries of a chunk are the last positions of the sequence): inside the
selected blocks, key j is dropped for query i when ``causal`` and
j > i + (Nk - Nq), and when ``kv_lens`` is given and j >= kv_lens[b].  A row
left with no key is an empty row (O = 0, LSE = -inf).  Without these options
causality, if any, is expressed at block level by the mask alone.

Two forms:

* ``dense_masked`` -- brute force: builds the full token-level allowed matrix
  and takes a row-wise softmax (tiny shapes only).
* ``block_gather`` -- per (b, h, q-block): gathers the rows of the selected K/V
  blocks and applies the same softmax to them with BLAS matmuls (the mask rows
  of a q-block are shared by its query rows).  Used for the large configs and
  for sampled rows.

Pins (tests/test_oracle_attention.py): agreement with torch's fp64
``scaled_dot_product_attention`` under the equivalent boolean mask on
non-empty rows (library special case); an all-ones mask equals dense SDPA;
empty rows give O = 0 and LSE = -inf; identical keys give the mean of the
selected V rows with LSE = s + ln|J| (closed form); a single selected block
equals dense attention on that block alone; sum_j exp(s_j - LSE) = 1 and
LSE = logsumexp of the selected scores (library routine); affine equivariance
in V; GQA against SDPA on explicitly repeated K/V heads; the two forms agree.
Element mask: with an all-ones block mask, ``causal`` equals SDPA with
``is_causal`` (Nq = Nk) and with torch's lower-triangular mask shifted by
Nk - Nq (Nq < Nk); ``kv_lens`` equals SDPA on K/V sliced to the length; the
two forms agree under both options.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np


def _as_f64(x) -> np.ndarray:
    """torch (any float dtype) or numpy -> float64 numpy (exact for bf16)."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _as_u8(m) -> np.ndarray:
    if hasattr(m, "detach"):
        return m.detach().to("cpu").numpy().astype(np.uint8)
    return np.asarray(m, dtype=np.uint8)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _softmax_rows(S: np.ndarray, Vs: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Row-wise softmax(S) @ Vs with -inf entries excluded; rows with no finite
    entry give (0, -inf)."""
    n, dv = S.shape[0], Vs.shape[1]
    O = np.zeros((n, dv), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    if S.shape[1] == 0:
        return O, lse
    m = S.max(axis=1)
    ok = np.isfinite(m)
    if not ok.any():
        return O, lse
    P = np.exp(S[ok] - m[ok, None])
    l = P.sum(axis=1)
    O[ok] = (P @ Vs) / l[:, None]
    lse[ok] = m[ok] + np.log(l)
    return O, lse


def _element_keep(qpos: np.ndarray, kpos: np.ndarray, Nq: int, Nk: int, causal: bool,
                  kv_len: Optional[int]) -> np.ndarray:
    """Boolean [len(qpos), len(kpos)]: which (query, key) pairs the element
    mask keeps (all of them without options)."""
    keep = np.ones((qpos.size, kpos.size), dtype=bool)
    if causal:
        keep &= kpos[None, :] <= qpos[:, None] + (Nk - Nq)
    if kv_len is not None:
        keep &= kpos[None, :] < kv_len
    return keep


def dense_masked(q, k, v, mask, bq: int, bk: int, scale: Optional[float] = None,
                 causal: bool = False, kv_lens=None):
    """Brute-force form.  q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d], mask [B,Hq,Nq/bq,Nk/bk];
    ``causal`` / ``kv_lens`` ([B] ints) as in the module docstring.
    Returns (O [B,Hq,Nq,d], LSE [B,Hq,Nq]) in fp64."""
    Q, K, V, M = _as_f64(q), _as_f64(k), _as_f64(v), _as_u8(mask)
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    g = Hq // Hkv
    sc = default_scale(d) if scale is None else scale
    O = np.zeros((B, Hq, Nq, V.shape[3]))
    L = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            allowed = np.zeros((Nq, Nk), dtype=bool)
            for i in range(Nq):
                for kb in range(Nk // bk):
                    if M[b, h, i // bq, kb] != 0:
                        allowed[i, kb * bk:(kb + 1) * bk] = True
            allowed &= _element_keep(np.arange(Nq), np.arange(Nk), Nq, Nk, causal,
                                     None if kv_lens is None else int(kv_lens[b]))
            S = (Q[b, h] @ K[b, hk].T) * sc
            S = np.where(allowed, S, -np.inf)
            O[b, h], L[b, h] = _softmax_rows(S, V[b, hk])
    return O, L


def qblock_rows(q64, k64, v64, mask_row, qb: int, bq: int, bk: int, sc: float,
                causal: bool = False, kv_len: Optional[int] = None):
    """One (b, h, q-block): gather the selected K/V blocks, then softmax.
    q64 [Nq,d] (this head), k64/v64 [Nk,d] (its kv head), mask_row [NKB];
    ``causal`` / ``kv_len`` (this sequence) as in the module docstring."""
    sel = np.flatnonzero(mask_row != 0)
    rows = slice(qb * bq, (qb + 1) * bq)
    if sel.size == 0:
        return _softmax_rows(np.zeros((bq, 0)), np.zeros((0, v64.shape[1])))
    keys = (sel[:, None] * bk + np.arange(bk)[None, :]).ravel()
    S = (q64[rows] @ k64[keys].T) * sc
    if causal or kv_len is not None:
        keep = _element_keep(np.arange(qb * bq, (qb + 1) * bq), keys, q64.shape[0],
                             k64.shape[0], causal, kv_len)
        S = np.where(keep, S, -np.inf)
    return _softmax_rows(S, v64[keys])


def block_gather(q, k, v, mask, bq: int, bk: int, scale: Optional[float] = None,
                 heads: Optional[Iterable[Tuple[int, int]]] = None, causal: bool = False,
                 kv_lens=None):
    """Per-q-block gather form over all rows (or over the (b, h) pairs in
    ``heads``; other heads are left 0 / -inf).  Returns fp64 (O, LSE)."""
    M = _as_u8(mask)
    B, Hq, NQB, NKB = M.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    d = q.shape[3]
    sc = default_scale(d) if scale is None else scale
    Nq = NQB * bq
    O = np.zeros((B, Hq, Nq, v.shape[3]))
    L = np.full((B, Hq, Nq), -np.inf)
    pairs = list(heads) if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    cache = {}
    for b, h in pairs:
        hk = h // g
        q64 = _as_f64(q[b, h])
        if (b, hk) not in cache:
            cache.clear()
            cache[(b, hk)] = (_as_f64(k[b, hk]), _as_f64(v[b, hk]))
        k64, v64 = cache[(b, hk)]
        for qb in range(NQB):
            o, l = qblock_rows(q64, k64, v64, M[b, h, qb], qb, bq, bk, sc, causal,
                               None if kv_lens is None else int(kv_lens[b]))
            O[b, h, qb * bq:(qb + 1) * bq] = o
            L[b, h, qb * bq:(qb + 1) * bq] = l
    return O, L


def sampled_qblocks(q, k, v, mask, bq: int, bk: int, samples: Iterable[Tuple[int, int, int]],
                    scale: Optional[float] = None, causal: bool = False, kv_lens=None):
    """Oracle rows for a list of (b, h, qb) samples; returns {(b,h,qb): (O, LSE)}."""
    M = _as_u8(mask)
    Hq, Hkv = M.shape[1], k.shape[1]
    g = Hq // Hkv
    d = q.shape[3]
    sc = default_scale(d) if scale is None else scale
    out = {}
    by_head = {}
    for b, h, qb in samples:
        by_head.setdefault((b, h), []).append(qb)
    for (b, h), qbs in by_head.items():
        hk = h // g
        q64 = _as_f64(q[b, h])
        k64, v64 = _as_f64(k[b, hk]), _as_f64(v[b, hk])
        for qb in qbs:
            out[(b, h, qb)] = qblock_rows(q64, k64, v64, M[b, h, qb], qb, bq, bk, sc, causal,
                                          None if kv_lens is None else int(kv_lens[b]))
    return out
