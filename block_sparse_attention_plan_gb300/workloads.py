"""Seeded synthetic inputs for block-sparse attention (masks and Q/K/V).

This module only *generates inputs*: logical block masks shaped like the
workloads the source pages evaluate on, and bf16 Q/K/V tensors.  It holds none
of the method's arithmetic (no mapping, no planning, no attention), so both the
CUDA path and the fp64 oracle can consume exactly the same bytes.

Workload families (stand-ins for data the pages use but do not publish):

* video-DiT 3D-local masks -- "Decoupling Logical Masks from GPU Execution for
  Dynamic Block-Sparse Attention" (Tessera), abstract: vDiT BSA masks; and
  "Veda", summary: tile geometry of video DiT attention.
* chunked-prefill top-k masks with GQA -- "CompactAttention: Accelerating
  Chunked Prefill with Block-Union KV Selection", summary.
* regular moderately sparse patterns (10-50% non-zero: sliding, strided,
  dilated, global+window+random) -- "SPLAT: A framework for optimised GPU
  code-generation for SParse reguLar ATtention", abstract.

Recipe (shared by every family): one ``torch.Generator('cpu')`` seeded with
``seed``; mask randomness is drawn first, then Q, then K, then V.  Q/K/V are
drawn per (batch, head) chunk as fp32 ``randn(N, d)`` and rounded to bf16 by
round-to-nearest-even (``Tensor.to(torch.bfloat16)``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np
import torch

__all__ = [
    "Workload", "CONFIGS", "SMALL_CONFIGS", "make_workload", "random_block_mask",
    "tiny_mask", "video_dit_mask", "chunked_prefill_mask", "regular_mask",
    "long_video_dit_mask", "make_qkv",
]


@dataclass
class Workload:
    """One synthetic BSA problem: mask u8 [B,H,Nq/bq,Nk/bk]; Q bf16 [B,Hq,Nq,d];
    K, V bf16 [B,Hkv,Nk,d].  All tensors live on the CPU."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    bq: int
    bk: int
    mask: torch.Tensor
    q: Optional[torch.Tensor] = None
    k: Optional[torch.Tensor] = None
    v: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def gqa_group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def active_blocks(self) -> int:
        return int((self.mask != 0).sum().item())

    @property
    def density(self) -> float:
        return self.active_blocks / float(self.mask.numel())

    @property
    def active_flop(self) -> float:
        """4*bq*bk*d FLOP per selected logical block (QK^T and PV)."""
        return 4.0 * self.bq * self.bk * self.d * self.active_blocks


# --------------------------------------------------------------------------
# mask families
# --------------------------------------------------------------------------

def random_block_mask(gen: torch.Generator, B: int, H: int, NQB: int, NKB: int,
                      p: float, values: bool = False) -> torch.Tensor:
    """Bernoulli(p) block mask.  With ``values`` the selected entries get random
    non-zero bytes 1..255 (any non-zero byte selects)."""
    sel = torch.rand(B, H, NQB, NKB, generator=gen) < p
    if not values:
        return sel.to(torch.uint8)
    vals = torch.randint(1, 256, (B, H, NQB, NKB), generator=gen, dtype=torch.int32)
    return torch.where(sel, vals, torch.zeros_like(vals)).to(torch.uint8)


def tiny_mask(gen: torch.Generator, B: int = 1, H: int = 2, NB: int = 8, p: float = 0.3) -> torch.Tensor:
    """Bernoulli(p) square block mask with the diagonal forced on."""
    m = (torch.rand(B, H, NB, NB, generator=gen) < p).to(torch.uint8)
    idx = torch.arange(NB)
    m[:, :, idx, idx] = 1
    return m


def _block_centres(n_blocks: int, blk: int, n_real: int, latent: Tuple[int, int, int]) -> np.ndarray:
    """(t, h, w) latent coordinates of each block's centre token (raster order
    t-major), clipped to the last real token."""
    T, Hl, W = latent
    c = np.minimum(np.arange(n_blocks, dtype=np.int64) * blk + blk // 2, n_real - 1)
    return np.stack([c // (Hl * W), (c // W) % Hl, c % W], axis=1)


def video_dit_mask(gen: torch.Generator, B: int, H: int, latent: Tuple[int, int, int],
                   blk: int = 128, window: Tuple[int, int, int] = (2, 8, 8),
                   p_random: float = 0.05) -> torch.Tensor:
    """3D-local window between block-centre coordinates, |dt|<=wt, |dh|<=wh,
    |dw|<=ww (same for every head), united with Bernoulli(p_random) blocks drawn
    independently per (b, h, q-block, k-block)."""
    T, Hl, W = latent
    N = T * Hl * W
    assert N % blk == 0
    nb = N // blk
    c = _block_centres(nb, blk, N, latent)
    d = np.abs(c[:, None, :] - c[None, :, :])
    local = (d[..., 0] <= window[0]) & (d[..., 1] <= window[1]) & (d[..., 2] <= window[2])
    rnd = torch.rand(B, H, nb, nb, generator=gen) < p_random
    return (torch.from_numpy(local)[None, None] | rnd).to(torch.uint8)


def chunked_prefill_mask(gen: torch.Generator, B: int, H: int, NQB: int, NKB: int,
                         window: int = 16, topk: int = 48) -> torch.Tensor:
    """Query chunk at the end of a causal KV prefix.  Query block qb sits at the
    absolute block a = NKB - NQB + qb and selects: block 0 (sink), the local
    window [a-window+1, a], and the top-``topk`` of [1, a-window] by an
    independent uniform score per (b, h, qb, kb), ties to the lower kb."""
    score = torch.rand(B, H, NQB, NKB, generator=gen)
    m = torch.zeros(B, H, NQB, NKB, dtype=torch.uint8)
    m[..., 0] = 1
    for qb in range(NQB):
        a = NKB - NQB + qb
        lo = max(a - window + 1, 0)
        m[:, :, qb, lo:a + 1] = 1
        cand_hi = a - window  # inclusive
        if cand_hi >= 1:
            s = score[:, :, qb, 1:cand_hi + 1]
            kk = min(topk, s.shape[-1])
            idx = torch.sort(s, dim=-1, descending=True, stable=True).indices[..., :kk] + 1
            m[:, :, qb].scatter_(-1, idx, 1)
    return m


def regular_mask(gen: torch.Generator, B: int, H: int, NB: int, window: int = 16,
                 stride: int = 8, dil_reach: int = 192, glob: int = 8,
                 bb_window: int = 16, bb_p: float = 0.15) -> torch.Tensor:
    """Per head h one of four regular patterns (h mod 4), with D = qb - kb:
    0 sliding |D| < window; 1 strided |D| < stride or D = 0 (mod stride);
    2 dilated |D| <= dil_reach and D even; 3 BigBird-style qb < glob or
    kb < glob or |D| <= bb_window or Bernoulli(bb_p).  Identical for every
    batch entry."""
    rnd = torch.rand(H, NB, NB, generator=gen) < bb_p
    qb = torch.arange(NB)[:, None]
    kb = torch.arange(NB)[None, :]
    D = qb - kb
    pats = [
        D.abs() < window,
        (D.abs() < stride) | (D % stride == 0),
        (D.abs() <= dil_reach) & (D % 2 == 0),
        None,
    ]
    m = torch.zeros(B, H, NB, NB, dtype=torch.uint8)
    for h in range(H):
        kind = h % 4
        if kind == 3:
            sel = (qb < glob) | (kb < glob) | (D.abs() <= bb_window) | rnd[h]
        else:
            sel = pats[kind]
        m[:, h] = sel.to(torch.uint8)
    return m


def regular_segments(H: int, NB: int, window: int = 16, stride: int = 8, dil_reach: int = 192,
                     glob: int = 8, bb_window: int = 16):
    """The regular patterns of ``regular_mask`` as affine row segments
    (a, b, stride, count) per head -- key blocks a*qb + b + stride*t -- plus
    the heads that stay explicit mask rows: the BigBird-style heads
    (h mod 4 = 3), whose random blocks have no affine form, get no segments.
    Same parameters as ``regular_mask``; ``glob`` and ``bb_window`` are
    accepted for symmetry with it."""
    K = -(-NB // stride)
    half = dil_reach // 2
    per_kind = [
        [(1, -(window - 1), 1, 2 * window - 1)],                                  # |D| < window
        [(1, -(stride - 1), 1, 2 * stride - 1), (1, -stride * K, stride, 2 * K + 1)],  # |D| < s or s | D
        [(1, -2 * half, 2, 2 * half + 1)],                                        # |D| <= reach, D even
        [],                                                                       # explicit mask rows
    ]
    segs = [per_kind[h % 4] for h in range(H)]
    mask_heads = [h for h in range(H) if h % 4 == 3]
    return segs, mask_heads


def long_video_dit_mask(gen: torch.Generator, B: int, H: int, latent: Tuple[int, int, int],
                        n_pad: int, blk: int = 128, rho: Tuple[float, float] = (0.05, 0.40),
                        aspect: Tuple[float, float] = (0.5, 2.0)):
    """Per-head 3D-local masks with per-head window shapes.

    Per head: target density rho_h ~ U(rho), aspect ratios r ~ U(aspect)^3.  A
    pair of real blocks is selected when |dt| <= s*r_t/4, |dh| <= s*r_h and
    |dw| <= 2*s*r_w (block-centre coordinates); equivalently when
    max(4|dt|/r_t, |dh|/r_h, |dw|/(2 r_w)) <= s.  The scale s is the smallest
    value whose density over the real-block grid is >= rho_h (the exact
    quantile, which is what a bisection on s converges to).  Blocks made only
    of padding tokens are never selected, so their query rows are empty.
    Returns (mask, per-head realised density)."""
    T, Hl, W = latent
    n_real = T * Hl * W
    assert n_pad % blk == 0 and n_pad >= n_real
    nb = n_pad // blk
    nb_real = (n_real + blk - 1) // blk
    c = _block_centres(nb_real, blk, n_real, latent).astype(np.float64)
    d = np.abs(c[:, None, :] - c[None, :, :])
    rho_h = (torch.rand(H, generator=gen, dtype=torch.float64) * (rho[1] - rho[0]) + rho[0]).numpy()
    r = (torch.rand(H, 3, generator=gen, dtype=torch.float64) * (aspect[1] - aspect[0]) + aspect[0]).numpy()
    m = torch.zeros(B, H, nb, nb, dtype=torch.uint8)
    realised = []
    P = nb_real * nb_real
    for h in range(H):
        need = np.maximum(np.maximum(4.0 * d[..., 0] / r[h, 0], d[..., 1] / r[h, 1]), d[..., 2] / (2.0 * r[h, 2]))
        k = int(math.ceil(rho_h[h] * P))
        s = np.partition(need.ravel(), k - 1)[k - 1]
        sel = need <= s
        realised.append(float(sel.mean()))
        m[:, h, :nb_real, :nb_real] = torch.from_numpy(sel.astype(np.uint8))
    return m, realised


# --------------------------------------------------------------------------
# Q / K / V
# --------------------------------------------------------------------------

def _draw(gen: torch.Generator, B: int, H: int, N: int, d: int) -> torch.Tensor:
    out = torch.empty(B, H, N, d, dtype=torch.bfloat16)
    for b in range(B):
        for h in range(H):
            out[b, h] = torch.randn(N, d, generator=gen).to(torch.bfloat16)
    return out


def make_qkv(gen: torch.Generator, B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
             outlier_pairs: Optional[torch.Tensor] = None, outlier_scale: float = 8.0):
    """Q [B,Hq,Nq,d], K/V [B,Hkv,Nk,d] bf16 ~ N(0,1).  ``outlier_pairs`` is an
    int tensor of flat (head*d + channel) indices whose channels are multiplied
    by ``outlier_scale`` (a power of two, so exact after bf16 rounding) in Q, K
    and V; a K/V head gets the outliers of the query heads that map to it."""
    q = _draw(gen, B, Hq, Nq, d)
    k = _draw(gen, B, Hkv, Nk, d)
    v = _draw(gen, B, Hkv, Nk, d)
    if outlier_pairs is not None:
        g = Hq // Hkv
        for p in outlier_pairs.tolist():
            h, ch = divmod(int(p), d)
            q[:, h, :, ch] *= outlier_scale
            k[:, h // g, :, ch] *= outlier_scale
            v[:, h // g, :, ch] *= outlier_scale
    return q, k, v


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------

def _wl(name, B, Hq, Hkv, Nq, Nk, d, bq, bk, mask_fn, data, seed, outliers=None, meta=None):
    gen = torch.Generator("cpu").manual_seed(seed)
    res = mask_fn(gen)
    meta = dict(meta or {})
    if isinstance(res, tuple):
        mask, realised = res
        meta["head_density"] = realised
    else:
        mask = res
    pairs = None
    if outliers:
        n_pairs = int(math.ceil(0.01 * Hq * d))
        pairs = torch.randperm(Hq * d, generator=gen)[:n_pairs]
        meta["outlier_pairs"] = pairs.tolist()
    w = Workload(name, B, Hq, Hkv, Nq, Nk, d, bq, bk, mask.contiguous(), meta=meta)
    if data:
        w.q, w.k, w.v = make_qkv(gen, B, Hq, Hkv, Nq, Nk, d, pairs)
    return w


def _tiny(data, seed):
    return _wl("tiny", 1, 2, 2, 512, 512, 64, 64, 64,
               lambda g: tiny_mask(g, 1, 2, 8, 0.3), data, seed)


def _video_dit(data, seed):
    return _wl("video_dit", 1, 24, 24, 16384, 16384, 128, 128, 128,
               lambda g: video_dit_mask(g, 1, 24, (16, 32, 32)), data, seed)


def _chunked_prefill(data, seed):
    return _wl("chunked_prefill", 1, 32, 8, 4096, 65536, 128, 64, 64,
               lambda g: chunked_prefill_mask(g, 1, 32, 64, 1024), data, seed)


def _regular(data, seed):
    return _wl("regular", 2, 16, 16, 8192, 8192, 64, 32, 32,
               lambda g: regular_mask(g, 2, 16, 256), data, seed)


def _long_video_dit(data, seed):
    return _wl("long_video_dit", 1, 40, 40, 75776, 75776, 128, 128, 128,
               lambda g: long_video_dit_mask(g, 1, 40, (21, 45, 80), 75776), data, seed,
               outliers=True)


# Reduced versions of the same families: same structure, sizes the fp64 oracle
# finishes in seconds while still spanning several tiles and a ragged tail.
def _video_dit_small(data, seed):
    return _wl("video_dit_small", 1, 3, 3, 4096, 4096, 128, 128, 128,
               lambda g: video_dit_mask(g, 1, 3, (4, 32, 32), window=(1, 8, 8), p_random=0.1),
               data, seed)


def _chunked_prefill_small(data, seed):
    return _wl("chunked_prefill_small", 1, 8, 2, 512, 4096, 128, 64, 64,
               lambda g: chunked_prefill_mask(g, 1, 8, 8, 64, window=8, topk=12), data, seed)


def _regular_small(data, seed):
    return _wl("regular_small", 2, 4, 4, 1024, 1024, 64, 32, 32,
               lambda g: regular_mask(g, 2, 4, 32, window=4, stride=4, dil_reach=20,
                                      glob=2, bb_window=3, bb_p=0.15),
               data, seed)


def _long_video_dit_small(data, seed):
    # 5*12*20 = 1200 real tokens padded to 1408 (11 blocks): block 9 is part
    # padding, block 10 is all padding.
    return _wl("long_video_dit_small", 1, 4, 4, 1408, 1408, 128, 128, 128,
               lambda g: long_video_dit_mask(g, 1, 4, (5, 12, 20), 1408), data, seed,
               outliers=True)


CONFIGS = {
    "tiny": _tiny,
    "video_dit": _video_dit,
    "chunked_prefill": _chunked_prefill,
    "regular": _regular,
    "long_video_dit": _long_video_dit,
}

SMALL_CONFIGS = {
    "tiny": _tiny,
    "video_dit_small": _video_dit_small,
    "chunked_prefill_small": _chunked_prefill_small,
    "regular_small": _regular_small,
    "long_video_dit_small": _long_video_dit_small,
}


def sweep_mask(gen: torch.Generator, B: int, H: int, NQB: int, NKB: int, bq: int, bk: int,
               density: float, skew: float) -> torch.Tensor:
    """Mask family of the mapping sweep: every (b, h, q-block) row gets its
    own density rho * (1 + skew * u), u ~ U(-1, 1) (clipped to [0.01, 1]),
    and selects each key block independently with it (no correlation between
    neighbouring q-blocks: the case where combining them costs most), plus
    the key blocks covering the q-block's own token range, so that no row is
    empty."""
    u = torch.rand(B, H, NQB, 1, generator=gen) * 2.0 - 1.0
    rho = (density * (1.0 + skew * u)).clamp(0.01, 1.0)
    m = (torch.rand(B, H, NQB, NKB, generator=gen) < rho).to(torch.uint8)
    for qb in range(NQB):
        lo, hi = qb * bq // bk, ((qb + 1) * bq - 1) // bk
        m[:, :, qb, lo:hi + 1] = 1
    return m


def _sweep(spec: str, data: bool, seed: int) -> Workload:
    """``sweep:bq=64,bk=128,d=128,density=0.2,skew=0.5`` (defaults: B=1, H=16,
    N=16384, density 0.2, skew 0)."""
    kv = dict(x.split("=") for x in spec.split(":", 1)[1].split(",") if x)
    bq, bk, d = int(kv.get("bq", 64)), int(kv.get("bk", 64)), int(kv.get("d", 128))
    B, H, N = int(kv.get("B", 1)), int(kv.get("H", 16)), int(kv.get("N", 16384))
    density, skew = float(kv.get("density", 0.2)), float(kv.get("skew", 0.0))
    return _wl(spec, B, H, H, N, N, d, bq, bk,
               lambda g: sweep_mask(g, B, H, N // bq, N // bk, bq, bk, density, skew), data, seed)


def make_workload(name: str, seed: int = 0, data: bool = True) -> Workload:
    """Build a named workload (``CONFIGS`` or ``SMALL_CONFIGS``), or one of the
    mapping sweep (``sweep:...``, see ``_sweep``)."""
    if name.startswith("sweep:"):
        return _sweep(name, data, seed)
    fn = CONFIGS.get(name) or SMALL_CONFIGS.get(name)
    if fn is None:
        raise KeyError(f"unknown workload {name!r}")
    return fn(data, seed)


def random_problem(seed: int, B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
                   bq: int, bk: int, p: float, values: bool = False) -> Workload:
    """Bernoulli(p) mask on an arbitrary geometry (for mapping edge cases)."""
    return _wl(f"random_{bq}x{bk}_d{d}", B, Hq, Hkv, Nq, Nk, d, bq, bk,
               lambda g: random_block_mask(g, B, Hq, Nq // bq, Nk // bk, p, values), True, seed)
