// Plan construction kernels: logical block mask -> physical tiles.
//
// Physical mapping ("Decoupling Logical Masks from GPU Execution for Dynamic
// Block-Sparse Attention" (Tessera), abstract: logical blocks are retained,
// combined or subdivided into physical tiles) and task organisation (tiles
// grouped per 128-row q-tile; rows scheduled so that rows sharing a K/V head
// run together, heaviest group first, longest row first inside a group), plus
// the GQA per-group union table ("CompactAttention", summary: Q-block union and
// intra-group union).
//
// Three launches, no host synchronisation:
//   count  one warp per plan row (and per union row).  Lane l owns bitmap word
//          l of every 32-word stretch of k-units (units 32w .. 32w+31): it reads
//          the 32 (16 when a logical block is two units) mask bytes of that
//          word for each of the rq q-units with 16-byte loads, turns nonzero
//          bytes into bits and stores the word in a per-q-unit bitmap; the
//          union over q-units gives the row's unit count.  Union rows OR the
//          g query heads' words the same way.
//   scan   one CTA: exclusive prefix sums (row pointers, union pointers),
//          totals, and the rank of every K/V-head group by its total slots.
//   fill   one warp per row: a warp prefix sum over the words' popcounts
//          places the ascending k-units into slots; the per-slot sub-masks
//          are read off the per-q-unit bitmaps; union rows likewise; and one
//          CTA per K/V-head group places the group's rows in the schedule
//          with a stable counting sort (slots descending, row id ascending).
#include <cstdint>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kScanThreads = 1024;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Nonzero bytes of a 32-bit word -> 4 bits (byte k -> bit k).
__device__ __forceinline__ uint32_t nz4(uint32_t v) {
  const uint32_t m = __vcmpne4(v, 0u);  // 0xff for each nonzero byte
  return ((m >> 7) & 1u) | ((m >> 14) & 2u) | ((m >> 21) & 4u) | ((m >> 28) & 8u);
}

// Mask bytes behind one bitmap word: 32 bytes (sk = 1) or 16 (sk = 2).
struct Raw {
  uint4 a, b;
};

// Mask row of q-unit x in the (b, h) plane mbh ([NQB][NKB] bytes).
__device__ __forceinline__ const uint8_t* qunit_row(const uint8_t* mbh, const PlanDev& p, int x) {
  return mbh + (size_t)(x >> (p.sq >> 1)) * p.NKB;
}

// 16-byte loads of word w of a mask row (the word lies wholly inside the row,
// the row is 16-byte aligned).
__device__ __forceinline__ Raw raw_load(const uint8_t* row, int w, int sk_sh) {
  Raw r;
  if (sk_sh == 0) {
    const uint4* s = reinterpret_cast<const uint4*>(row + 32 * (size_t)w);
    r.a = __ldg(s);
    r.b = __ldg(s + 1);
  } else {
    r.a = __ldg(reinterpret_cast<const uint4*>(row + 16 * (size_t)w));
    r.b = make_uint4(0u, 0u, 0u, 0u);
  }
  return r;
}

__device__ __forceinline__ uint32_t raw_bits(const Raw& r, int sk_sh) {
  const uint32_t lo = nz4(r.a.x) | (nz4(r.a.y) << 4) | (nz4(r.a.z) << 8) | (nz4(r.a.w) << 12);
  if (sk_sh == 0)
    return lo | (nz4(r.b.x) << 16) | (nz4(r.b.y) << 20) | (nz4(r.b.z) << 24) | (nz4(r.b.w) << 28);
  // 16 logical blocks, each two k-units: bit b -> bits 2b and 2b + 1.
  uint32_t t = lo;
  t = (t | (t << 8)) & 0x00ff00ffu;
  t = (t | (t << 4)) & 0x0f0f0f0fu;
  t = (t | (t << 2)) & 0x33333333u;
  t = (t | (t << 1)) & 0x55555555u;
  return t | (t << 1);
}

// Word w of a mask row one byte at a time (unaligned masks, the last word).
__device__ uint32_t slow_bits(const uint8_t* row, const PlanDev& p, int w, int sk_sh) {
  uint32_t bits = 0;
  for (int t = 0; t < 32; ++t) {
    const int y = 32 * w + t;
    if (y < p.NKU && __ldg(row + (y >> sk_sh)) != 0) bits |= 1u << t;
  }
  return bits;
}

// Selected-unit words (k-units 32w .. 32w+31) of up to four mask rows, all
// loads issued before any is used.  Rows with index >= n (and every row when
// the plan has no mask bytes) give 0.
__device__ __forceinline__ void row_words(const uint8_t* const (&rows)[4], int n, const PlanDev& p,
                                          int w, uint32_t (&out)[4]) {
  const int sk_sh = p.sk >> 1;
  if (p.mask == nullptr) n = 0;
  const bool fast = p.vec && 32 * (w + 1) <= p.NKU;
  Raw raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < n && fast) raw[i] = raw_load(rows[i], w, sk_sh);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[i] = 0u;
    if (i < n && w < p.W) out[i] = fast ? raw_bits(raw[i], sk_sh) : slow_bits(rows[i], p, w, sk_sh);
  }
}

// Segments of head h: [s0, s1) clamped to the array (empty: the head's
// selection is its mask rows).
__device__ __forceinline__ void head_segments(const PlanDev& p, int h, int& s0, int& s1) {
  s0 = 0;
  s1 = 0;
  if (p.seg_ptr == nullptr) return;
  s0 = max(__ldg(p.seg_ptr + h), 0);
  s1 = min(__ldg(p.seg_ptr + h + 1), p.nseg);
}

__device__ __forceinline__ int floor_div(int a, int b) {  // b > 0
  return a >= 0 ? a / b : -((b - 1 - a) / b);
}

// Word w (k-units 32w .. 32w+31) of the k-units that segments [s0, s1)
// select for logical query block qb ("SPLAT", abstract: the
// affine-compressed-sparse-row format).  Segment (a, b, stride, count)
// selects key blocks a*qb + b + stride*t, t = 0 .. count-1, inside
// [0, NKB).  A negative stride is turned around (same set), stride 0 is one
// block.  Only the t whose block falls in this word are visited: by 32-bit
// arithmetic when the segment starts at or after -2^28 with a stride of at
// most 2^28 (so no intermediate value leaves int), else by stepping from the
// first block at or after the word in 64 bits.
__device__ uint32_t segment_word(const PlanDev& p, int s0, int s1, int qb, int w) {
  const int sk_sh = p.sk >> 1;
  const int kb_lo = (32 * w) >> sk_sh;
  const int kb_hi = min((32 * w + 31) >> sk_sh, p.NKB - 1);
  const uint32_t unit_bits = sk_sh ? 3u : 1u;
  uint32_t bits = 0u;
  for (int s = s0; s < s1; ++s) {
    const int4 sg = __ldg(reinterpret_cast<const int4*>(p.seg) + s);  // a, b, stride, count
    if (sg.w <= 0) continue;
    long long start = (long long)sg.x * qb + sg.y;
    long long stride = sg.z, count = sg.w;
    if (stride == 0) {
      count = 1;
      stride = 1;
    } else if (stride < 0) {
      start += stride * (count - 1);
      stride = -stride;
    }
    if (start + stride * (count - 1) < kb_lo || start > kb_hi) continue;  // misses this word
    if (start < -(1ll << 28) || stride > (1ll << 28)) {
      const long long t = start < kb_lo ? (kb_lo - start + stride - 1) / stride : 0;
      for (long long x = start + stride * t, n = count - t; n > 0 && x <= kb_hi; x += stride, --n)
        bits |= unit_bits << (int)((x << sk_sh) - 32ll * w);
      continue;
    }
    const int st = (int)start, sd = (int)stride;
    int t0 = -floor_div(st - kb_lo, sd);  // ceil((kb_lo - start) / stride)
    int t1 = floor_div(kb_hi - st, sd);
    t0 = max(t0, 0);
    if ((long long)t1 > count - 1) t1 = (int)(count - 1);
    for (int t = t0; t <= t1; ++t) bits |= unit_bits << (((st + sd * t) << sk_sh) - 32 * w);
  }
  return bits;
}

__global__ void __launch_bounds__(kThreads) plan_count_kernel(const PlanDev p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row_ctas = (p.rows + kWarps - 1) / kWarps;
  if ((int)blockIdx.x < row_ctas) {
    const int r = blockIdx.x * kWarps + warp;
    if (r >= p.rows) return;
    const int bh = r / p.NQT, qt = r % p.NQT;
    const uint8_t* mbh = p.mask + (size_t)bh * p.NQB * p.NKB;
    const uint8_t* rows[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rows[i] = qunit_row(mbh, p, qt * p.rq + (i < p.rq ? i : 0));
    // A logical block is counted once: at its first q-unit (x even when
    // sq = 2) and its first k-unit (even units when sk = 2).
    const uint32_t kfirst = p.sk == 2 ? 0x55555555u : 0xffffffffu;
    int seg0, seg1;  // a head with segments is generated from them, else read from the mask
    head_segments(p, bh % p.H, seg0, seg1);
    int cnt = 0, own = 0;
    for (int w0 = 0; w0 < p.W; w0 += 32) {
      const int w = w0 + lane;
      uint32_t words[4];
      row_words(rows, seg1 > seg0 ? 0 : p.rq, p, w, words);
      uint32_t u = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i >= p.rq) break;
        if (seg1 > seg0 && w < p.W) words[i] = segment_word(p, seg0, seg1, (qt * p.rq + i) >> (p.sq >> 1), w);
        if (w < p.W) p.qbits[((size_t)r * p.rq + i) * p.W + w] = words[i];
        u |= words[i];
        if (((qt * p.rq + i) & (p.sq >> 1)) == 0) own += __popc(words[i] & kfirst);
      }
      cnt += __popc(u);
    }
    for (int s = 16; s > 0; s >>= 1) {
      cnt += __shfl_xor_sync(0xffffffffu, cnt, s);
      own += __shfl_xor_sync(0xffffffffu, own, s);
    }
    if (lane == 0) {
      p.slots[r] = (cnt + p.rk - 1) / p.rk;  // grouping stride 1 (the choose kernel may redo it)
      p.lcnt[r] = own;
      if (qt == 0) p.sigma[bh] = 1;
    }
  } else {
    const int ur = (blockIdx.x - row_ctas) * kWarps + warp;
    if (ur >= p.urows) return;
    const int bhk = ur / p.NQT, qt = ur % p.NQT;
    const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
    const int nsrc = p.g * p.rq;  // (head, q-unit) mask rows OR-ed into the union
    int cnt = 0;
    for (int w0 = 0; w0 < p.W; w0 += 32) {
      const int w = w0 + lane;
      uint32_t u = 0u;
      for (int k0 = 0; k0 < nsrc; k0 += 4) {
        const uint8_t* rows[4] = {p.mask, p.mask, p.mask, p.mask};
        int nmask = 0;  // sources read from the mask (heads without segments)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = k0 + i < nsrc ? k0 + i : k0;
          const int hh = k / p.rq, ii = k % p.rq;
          int s0, s1;
          head_segments(p, hk * p.g + hh, s0, s1);
          if (k0 + i < nsrc && s1 > s0) {
            if (w < p.W) u |= segment_word(p, s0, s1, (qt * p.rq + ii) >> (p.sq >> 1), w);
          } else if (k0 + i < nsrc) {
            const uint8_t* mbh = p.mask + ((size_t)(b * p.H + hk * p.g + hh)) * p.NQB * p.NKB;
            rows[nmask++] = qunit_row(mbh, p, qt * p.rq + ii);
          }
        }
        uint32_t words[4];
        row_words(rows, nmask, p, w, words);
        u |= words[0] | words[1] | words[2] | words[3];
      }
      if (w < p.W) p.ubits[(size_t)ur * p.W + w] = u;
      cnt += __popc(u);
    }
    for (int s = 16; s > 0; s >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, s);
    if (lane == 0) p.ucnt[ur] = cnt;
  }
}

// q-unit i of q-tile qt in a plane grouped with stride s: tiles come in runs
// of s, tile run*s + r holding q-units run*s*rq + r + i*s.
__device__ __forceinline__ int tile_qunit(int qt, int s, int rq, int i) {
  return (qt / s) * s * rq + qt % s + i * s;
}

// Grouping stride of a plane as the plan stores it (1 if out of range).
__device__ __forceinline__ int plane_sigma(const PlanDev& p, int bh) {
  const int s = p.sigma[bh];
  return (s == 1 || s == 2 || s == 4 || s == 8 || s == 16) && p.NQT % s == 0 ? s : 1;
}

// Block-wide sum of one value per thread; every thread gets the total.
__device__ long long block_sum(long long v, long long* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long t = 0;
  for (int w = 0; w < (int)blockDim.x / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

// Per-plane choice of the q-unit grouping stride (physical mapping of
// combined blocks, "Decoupling Logical Masks from GPU Execution for Dynamic
// Block-Sparse Attention" (Tessera), abstract: logical blocks are combined
// into physical tiles).  One CTA per (b, h) plane: for each stride s in
// {1, 2, 4, 8, 16} dividing the plane's q-tiles, the slots its tiles need
// (the sum over tiles of ceil(|OR of the tile's q-unit bitmaps| / rk)); the
// fewest wins, ties to the smaller stride.  Writes the stride and the plane's
// per-row slot counts for it.  Launched only with BSA_PLAN_REMAP.
__global__ void __launch_bounds__(kThreads) plan_choose_kernel(const PlanDev p) {
  extern __shared__ int tile_cnt[];  // [NQT] set bits of each tile's union
  __shared__ long long red[kWarps];
  const int bh = blockIdx.x;
  const int NQU = p.NQT * p.rq;
  const uint32_t* qb = p.qbits + (size_t)bh * NQU * p.W;
  const long long pairs = (long long)p.NQT * p.W;
  auto count_tiles = [&](int s) {
    for (int t = threadIdx.x; t < p.NQT; t += kThreads) tile_cnt[t] = 0;
    __syncthreads();
    for (long long k = threadIdx.x; k < pairs; k += kThreads) {
      const int t = (int)(k / p.W), w = (int)(k % p.W);
      uint32_t u = 0u;
      for (int i = 0; i < p.rq; ++i) u |= qb[(size_t)tile_qunit(t, s, p.rq, i) * p.W + w];
      if (u) atomicAdd(&tile_cnt[t], __popc(u));
    }
    __syncthreads();
  };
  int best = 1;
  long long best_slots = -1;
  for (int s = 1; s <= 16; s <<= 1) {
    if (p.NQT % s) continue;
    count_tiles(s);
    long long mine = 0;
    for (int t = threadIdx.x; t < p.NQT; t += kThreads) mine += (tile_cnt[t] + p.rk - 1) / p.rk;
    const long long total = block_sum(mine, red);
    if (best_slots < 0 || total < best_slots) {
      best = s;
      best_slots = total;
    }
  }
  count_tiles(best);
  for (int t = threadIdx.x; t < p.NQT; t += kThreads)
    p.slots[(size_t)bh * p.NQT + t] = (tile_cnt[t] + p.rk - 1) / p.rk;
  if (threadIdx.x == 0) p.sigma[bh] = best;
}

// Block-wide exclusive scan of one value per thread (blockDim.x = 32 * nwarps);
// returns the block total.  Every thread must call it.
template <typename T>
__device__ T block_exclusive_scan(T v, T* excl_out, T* warp_sums) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int nwarps = blockDim.x / 32;
  T x = v;
  for (int s = 1; s < 32; s <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, s);
    if (lane >= s) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nwarps ? warp_sums[lane] : T(0);
    for (int s = 1; s < 32; s <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, w, s);
      if (lane >= s) w += y;
    }
    if (lane < nwarps) warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const T before = (warp > 0) ? warp_sums[warp - 1] : T(0);
  *excl_out = before + x - v;
  const T total = warp_sums[nwarps - 1];
  __syncthreads();
  return total;
}

// Exclusive prefix sum of in[0..n) into out[0..n] (out[n] = total) by one
// block: each thread sums a contiguous run (loads issued kRun at a time), the
// run sums are scanned once, then each thread writes its run's prefixes --
// from the values still in registers when its run fits in one batch.  With
// in2, the sum of in2[0..n) is taken in the same load pass (*sum2).
constexpr int kRun = 16;
template <typename TIn>
__device__ long long block_scan_array(const TIn* in, int32_t* out, int n, long long* wsum,
                                      const TIn* in2 = nullptr, long long* sum2 = nullptr) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = threadIdx.x * per;
  const int i1 = min(i0 + per, n);
  long long local = 0, local2 = 0;
  TIn t[kRun] = {};
  for (int b = i0; b < i1; b += kRun) {
#pragma unroll
    for (int k = 0; k < kRun; ++k) t[k] = (b + k < i1) ? in[b + k] : TIn(0);
    if (in2 != nullptr) {
#pragma unroll
      for (int k = 0; k < kRun; ++k) local2 += (b + k < i1) ? (long long)in2[b + k] : 0ll;
    }
#pragma unroll
    for (int k = 0; k < kRun; ++k) local += (long long)t[k];
  }
  long long ex;
  const long long total = block_exclusive_scan<long long>(local, &ex, wsum);
  if (in2 != nullptr) {
    long long ex2;
    const long long total2 = block_exclusive_scan<long long>(local2, &ex2, wsum);
    if (sum2) *sum2 = total2;
  }
  if (out) {
    long long run = ex;
    if (per <= kRun) {  // the run is still in t[]
#pragma unroll
      for (int k = 0; k < kRun; ++k) {
        if (i0 + k < i1) out[i0 + k] = (int32_t)run;
        run += (long long)t[k];
      }
    } else {
      for (int b = i0; b < i1; b += kRun) {
#pragma unroll
        for (int k = 0; k < kRun; ++k) t[k] = (b + k < i1) ? in[b + k] : TIn(0);
#pragma unroll
        for (int k = 0; k < kRun; ++k) {
          if (b + k < i1) out[b + k] = (int32_t)run;
          run += (long long)t[k];
        }
      }
    }
    if (threadIdx.x == 0) out[n] = (int32_t)total;
  }
  return total;
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(const PlanDev p) {
  __shared__ long long wsum[32];
  extern __shared__ int work_s[];  // [groups] total slots per K/V-head group
  long long A = 0;  // selected logical blocks: summed in the row-pointer scan's load pass
  const long long S = block_scan_array<int32_t>(p.slots, p.row_ptr, p.rows, wsum, p.lcnt, &A);
  long long U = 0;
  if (p.urows > 0) {
    U = block_scan_array<int32_t>(p.ucnt, p.urow_ptr, p.urows, wsum);
  } else if (threadIdx.x == 0) {
    p.urow_ptr[0] = 0;
  }
  if (threadIdx.x == 0) {
    p.totals[0] = S;
    p.totals[1] = A;
    p.totals[2] = U;
    p.totals[3] = 0;
  }
  __syncthreads();  // row_ptr visible to the whole block
  const int gsz = p.g * p.NQT;
  for (int gi = threadIdx.x; gi < p.groups; gi += blockDim.x)
    work_s[gi] = p.row_ptr[(gi + 1) * gsz] - p.row_ptr[gi * gsz];
  __syncthreads();
  // Groups heaviest first, ties by group id: rank = number of groups before.
  for (int gi = threadIdx.x; gi < p.groups; gi += blockDim.x) {
    const int w = work_s[gi];
    int rank = 0;
    for (int gj = 0; gj < p.groups; ++gj) {
      const int x = work_s[gj];
      rank += (x > w) || (x == w && gj < gi);
    }
    p.gstart[gi] = rank * gsz;
  }
}

// Writes the set bits of `u` (bitmap word w of the warp's lane) as ascending
// k-units at out[pos + ...] (entries at or beyond cap are dropped); returns
// the number of set bits over the warp.
__device__ __forceinline__ int compact_word(uint32_t u, int w, int lane, int32_t* out, int pos,
                                            int cap) {
  const int c = __popc(u);
  int incl = c;
  for (int s = 1; s < 32; s <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, s);
    if (lane >= s) incl += y;
  }
  int idx = pos + incl - c;
  while (u) {
    const int bit = __ffs(u) - 1;
    u &= u - 1u;
    if (idx < cap) out[idx] = 32 * w + bit;
    ++idx;
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

__device__ void fill_row(const PlanDev& p, int r, int lane) {
  const int s0 = p.row_ptr[r];
  const int n = p.row_ptr[r + 1] - s0;
  const int cap = n * p.rk;
  int32_t* out = p.slot_ku + (size_t)s0 * p.rk;
  // Bitmaps of the tile's q-units (the plane's grouping stride decides which).
  const int bh = r / p.NQT, qt = r % p.NQT, sig = plane_sigma(p, bh);
  const uint32_t* qb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    qb[i] = p.qbits + ((size_t)bh * p.NQT * p.rq + tile_qunit(qt, sig, p.rq, i < p.rq ? i : 0)) * p.W;
  int pos = 0;
  for (int w0 = 0; w0 < p.W; w0 += 32) {
    const int w = w0 + lane;
    uint32_t u = 0u;
    if (w < p.W) {
      for (int i = 0; i < p.rq; ++i) u |= qb[i][w];
    }
    pos += compact_word(u, w, lane, out, pos, cap);
  }
  for (int idx = pos + lane; idx < cap; idx += 32) out[idx] = -1;
  __syncwarp();
  // Sub-mask of each slot: bit i*rk + j when q-unit i selects the unit at
  // position j (read off the q-unit bitmaps).
  for (int s = lane; s < n; s += 32) {
    uint32_t bits = 0;
    for (int j = 0; j < p.rk; ++j) {
      const int y = out[s * p.rk + j];
      if (y < 0) continue;
      for (int i = 0; i < p.rq; ++i)
        if ((qb[i][y >> 5] >> (y & 31)) & 1u) bits |= 1u << (i * p.rk + j);
    }
    p.slot_mask[s0 + s] = bits;
  }
}

__device__ void fill_union_row(const PlanDev& p, int ur, int lane) {
  const int s0 = p.urow_ptr[ur];
  const int cap = p.urow_ptr[ur + 1] - s0;
  const uint32_t* ub = p.ubits + (size_t)ur * p.W;
  int pos = 0;
  for (int w0 = 0; w0 < p.W; w0 += 32) {
    const int w = w0 + lane;
    pos += compact_word(w < p.W ? ub[w] : 0u, w, lane, p.ukb + s0, pos, cap);
  }
}

__device__ void order_group(const PlanDev& p, int gi, int* start_s) {
  __shared__ int wsum[32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int gsz = p.g * p.NQT;
  const int r0 = gi * gsz;
  for (int k = threadIdx.x; k < p.nkeys; k += kThreads) start_s[k] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < gsz; i += kThreads) atomicAdd(&start_s[p.slots[r0 + i]], 1);
  __syncthreads();
  // exclusive scan over keys in descending order
  int carry = 0;
  for (int base = 0; base < p.nkeys; base += kThreads) {
    const int key = p.nkeys - 1 - (base + (int)threadIdx.x);
    const int v = (key >= 0) ? start_s[key] : 0;
    int ex;
    const int tot = block_exclusive_scan<int>(v, &ex, wsum);
    if (key >= 0) start_s[key] = carry + ex;
    carry += tot;
    __syncthreads();
  }
  const int base_pos = p.gstart[gi];
  for (int c0 = 0; c0 < gsz; c0 += kThreads) {
    const int i = c0 + (int)threadIdx.x;
    const bool valid = i < gsz;
    const int key = valid ? p.slots[r0 + i] : -1;
    for (int w = 0; w < kWarps; ++w) {
      __syncthreads();
      if (warp == w) {
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        int pos = 0;
        if (valid) pos = start_s[key] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (valid) {
          p.order[base_pos + pos] = r0 + i;
          if (lane == __ffs(peers) - 1) start_s[key] += __popc(peers);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads) plan_fill_kernel(const PlanDev p) {
  extern __shared__ int start_s[];  // [nkeys]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row_ctas = (p.rows + kWarps - 1) / kWarps;
  const int union_ctas = (p.urows + kWarps - 1) / kWarps;
  const int cta = blockIdx.x;
  if (cta < row_ctas) {
    const int r = cta * kWarps + warp;
    if (r < p.rows) fill_row(p, r, lane);
  } else if (cta < row_ctas + union_ctas) {
    const int ur = (cta - row_ctas) * kWarps + warp;
    if (ur < p.urows) fill_union_row(p, ur, lane);
  } else {
    order_group(p, cta - row_ctas - union_ctas, start_s);
  }
}

}  // namespace

cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream) {
  const int row_ctas = (p.rows + kWarps - 1) / kWarps;
  const int union_ctas = (p.urows + kWarps - 1) / kWarps;
  const size_t keys_smem = (size_t)p.nkeys * sizeof(int);
  const size_t groups_smem = (size_t)p.groups * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(plan_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMaxKeys * (int)sizeof(int));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(plan_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxGroups * (int)sizeof(int));
  if (e != cudaSuccess) return e;
  plan_count_kernel<<<row_ctas + union_ctas, kThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.remap) {
    const size_t tiles_smem = (size_t)p.NQT * sizeof(int);
    e = cudaFuncSetAttribute(plan_choose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxRemapTiles * (int)sizeof(int));
    if (e != cudaSuccess) return e;
    plan_choose_kernel<<<p.B * p.H, kThreads, tiles_smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  plan_scan_kernel<<<1, kScanThreads, groups_smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  plan_fill_kernel<<<row_ctas + union_ctas + p.groups, kThreads, keys_smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bsa
