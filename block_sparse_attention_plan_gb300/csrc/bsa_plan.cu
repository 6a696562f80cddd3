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
//   count  one warp per plan row (and per union row): per 32 k-units, each
//          lane ORs the rq q-unit mask bytes of its k-unit; __ballot_sync +
//          __popc give the row's unit count.
//   scan   one CTA: exclusive prefix sums (row pointers, union pointers),
//          totals, and the rank of every K/V-head group by its total slots.
//   fill   one warp per row: ballot + prefix-popcount compaction writes the
//          ascending k-units into slots, then the per-slot sub-masks; union
//          rows likewise; and one CTA per K/V-head group places the group's
//          rows in the schedule with a stable counting sort (slots
//          descending, row id ascending).
#include <cstdint>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kScanThreads = 1024;
constexpr int kBatch = 8;  // 32-unit chunks whose mask loads are issued together

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Mask bytes of kBatch consecutive 32-unit chunks (k-units y0 + c*32 + lane)
// for the rq q-units of q-tile qt of mask plane mbh ([NQB][NKB] of one
// (b, h)).  Every load of the batch is issued before any is used (fully
// unrolled, predicated on rq <= 4), so a warp waits for one round trip per
// batch instead of one per byte.
struct UnitBatch {
  int u[kBatch];    // k-unit selected by some q-unit of the tile
  int own[kBatch];  // logical blocks first-owned here (see count kernel)
};

__device__ __forceinline__ UnitBatch unit_batch(const uint8_t* __restrict__ mbh, const PlanDev& p,
                                                int qt, int y0, int lane) {
  const int sk_sh = p.sk >> 1, sq_sh = p.sq >> 1;  // sk, sq are 1 or 2
  uint8_t v[kBatch][4];
#pragma unroll
  for (int c = 0; c < kBatch; ++c) {
    const int y = y0 + c * 32 + lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int x = qt * p.rq + i;
      v[c][i] = (i < p.rq && y < p.NKU) ? __ldg(mbh + (size_t)(x >> sq_sh) * p.NKB + (y >> sk_sh))
                                        : (uint8_t)0;
    }
  }
  UnitBatch r;
#pragma unroll
  for (int c = 0; c < kBatch; ++c) {
    const int y = y0 + c * 32 + lane;
    const bool first_k = (y & sk_sh) == 0;
    int u = 0, o = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int x = qt * p.rq + i;
      const int sel = v[c][i] != 0;
      u |= sel;
      o += (sel && first_k && (x & sq_sh) == 0);
    }
    r.u[c] = u;
    r.own[c] = o;
  }
  return r;
}

// GQA union over the g query heads of K/V head hk: for each head the same
// hoisted batch of loads, OR-ed together.
__device__ __forceinline__ void union_batch(const PlanDev& p, int b, int hk, int qt, int y0,
                                            int lane, int (&u)[kBatch]) {
#pragma unroll
  for (int c = 0; c < kBatch; ++c) u[c] = 0;
  for (int hh = 0; hh < p.g; ++hh) {
    const uint8_t* mbh = p.mask + ((size_t)(b * p.H + hk * p.g + hh)) * p.NQB * p.NKB;
    const UnitBatch r = unit_batch(mbh, p, qt, y0, lane);
#pragma unroll
    for (int c = 0; c < kBatch; ++c) u[c] |= r.u[c];
  }
}

__global__ void __launch_bounds__(kThreads) plan_count_kernel(const PlanDev p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row_ctas = (p.rows + kWarps - 1) / kWarps;
  if ((int)blockIdx.x < row_ctas) {
    const int r = blockIdx.x * kWarps + warp;
    if (r >= p.rows) return;
    const int bh = r / p.NQT, qt = r % p.NQT;
    const uint8_t* mbh = p.mask + (size_t)bh * p.NQB * p.NKB;
    int cnt = 0, own = 0;
    for (int y0 = 0; y0 < p.NKU; y0 += 32 * kBatch) {
      const UnitBatch r = unit_batch(mbh, p, qt, y0, lane);
#pragma unroll
      for (int c = 0; c < kBatch; ++c) {
        cnt += __popc(__ballot_sync(0xffffffffu, r.u[c]));
        own += r.own[c];
      }
    }
    for (int s = 16; s > 0; s >>= 1) own += __shfl_xor_sync(0xffffffffu, own, s);
    if (lane == 0) {
      p.slots[r] = (cnt + p.rk - 1) / p.rk;
      p.lcnt[r] = own;
    }
  } else {
    const int ur = (blockIdx.x - row_ctas) * kWarps + warp;
    if (ur >= p.urows) return;
    const int bhk = ur / p.NQT, qt = ur % p.NQT;
    const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
    int cnt = 0;
    for (int y0 = 0; y0 < p.NKU; y0 += 32 * kBatch) {
      int u[kBatch];
      union_batch(p, b, hk, qt, y0, lane, u);
#pragma unroll
      for (int c = 0; c < kBatch; ++c) cnt += __popc(__ballot_sync(0xffffffffu, u[c]));
    }
    if (lane == 0) p.ucnt[ur] = cnt;
  }
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
// run sums are scanned once, then each thread writes its run's prefixes.
constexpr int kRun = 16;
template <typename TIn>
__device__ long long block_scan_array(const TIn* in, int32_t* out, int n, long long* wsum) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = threadIdx.x * per;
  const int i1 = min(i0 + per, n);
  long long local = 0;
  for (int b = i0; b < i1; b += kRun) {
    TIn t[kRun];
#pragma unroll
    for (int k = 0; k < kRun; ++k) t[k] = (b + k < i1) ? in[b + k] : TIn(0);
#pragma unroll
    for (int k = 0; k < kRun; ++k) local += (long long)t[k];
  }
  long long ex;
  const long long total = block_exclusive_scan<long long>(local, &ex, wsum);
  if (out) {
    long long run = ex;
    for (int b = i0; b < i1; b += kRun) {
      TIn t[kRun];
#pragma unroll
      for (int k = 0; k < kRun; ++k) t[k] = (b + k < i1) ? in[b + k] : TIn(0);
#pragma unroll
      for (int k = 0; k < kRun; ++k) {
        if (b + k < i1) out[b + k] = (int32_t)run;
        run += (long long)t[k];
      }
    }
    if (threadIdx.x == 0) out[n] = (int32_t)total;
  }
  return total;
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(const PlanDev p) {
  __shared__ long long wsum[32];
  extern __shared__ int work_s[];  // [groups] total slots per K/V-head group
  const long long S = block_scan_array<int32_t>(p.slots, p.row_ptr, p.rows, wsum);
  const long long A = block_scan_array<int32_t>(p.lcnt, nullptr, p.rows, wsum);
  const long long U = block_scan_array<int32_t>(p.ucnt, p.urow_ptr, p.urows, wsum);
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

__device__ void fill_row(const PlanDev& p, int r, int lane) {
  const int bh = r / p.NQT, qt = r % p.NQT;
  const uint8_t* mbh = p.mask + (size_t)bh * p.NQB * p.NKB;
  const int s0 = p.row_ptr[r];
  const int n = p.row_ptr[r + 1] - s0;
  const int cap = n * p.rk;
  int32_t* out = p.slot_ku + (size_t)s0 * p.rk;
  int pos = 0;
  for (int y0 = 0; y0 < p.NKU; y0 += 32 * kBatch) {
    const UnitBatch r = unit_batch(mbh, p, qt, y0, lane);
#pragma unroll
    for (int c = 0; c < kBatch; ++c) {  // ascending k-units: chunk by chunk
      const uint32_t bal = __ballot_sync(0xffffffffu, r.u[c]);
      if (r.u[c]) {
        const int idx = pos + __popc(bal & lanemask_lt());
        if (idx < cap) out[idx] = y0 + c * 32 + lane;
      }
      pos += __popc(bal);
    }
  }
  for (int idx = pos + lane; idx < cap; idx += 32) out[idx] = -1;
  __threadfence_block();
  __syncwarp();
  for (int s = lane; s < n; s += 32) {
    uint32_t bits = 0;
    for (int j = 0; j < p.rk; ++j) {
      const int y = out[s * p.rk + j];
      if (y < 0) continue;
      const int kb = y >> (p.sk >> 1);
      for (int ii = 0; ii < p.rq; ++ii) {
        const int x = qt * p.rq + ii;
        if (__ldg(mbh + (size_t)(x >> (p.sq >> 1)) * p.NKB + kb) != 0) bits |= 1u << (ii * p.rk + j);
      }
    }
    p.slot_mask[s0 + s] = bits;
  }
}

__device__ void fill_union_row(const PlanDev& p, int ur, int lane) {
  const int bhk = ur / p.NQT, qt = ur % p.NQT;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int s0 = p.urow_ptr[ur];
  const int cap = p.urow_ptr[ur + 1] - s0;
  int pos = 0;
  for (int y0 = 0; y0 < p.NKU; y0 += 32 * kBatch) {
    int u[kBatch];
    union_batch(p, b, hk, qt, y0, lane, u);
#pragma unroll
    for (int c = 0; c < kBatch; ++c) {
      const uint32_t bal = __ballot_sync(0xffffffffu, u[c]);
      if (u[c]) {
        const int idx = pos + __popc(bal & lanemask_lt());
        if (idx < cap) p.ukb[s0 + idx] = y0 + c * 32 + lane;
      }
      pos += __popc(bal);
    }
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
  plan_scan_kernel<<<1, kScanThreads, groups_smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  plan_fill_kernel<<<row_ctas + union_ctas + p.groups, kThreads, keys_smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bsa
