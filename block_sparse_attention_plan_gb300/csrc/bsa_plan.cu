// Plan construction kernels: logical block mask -> physical tiles.
//
// Physical mapping ("Decoupling Logical Masks from GPU Execution for Dynamic
// Block-Sparse Attention" (Tessera), abstract: logical blocks are retained,
// combined or subdivided into physical tiles) and task organisation (tiles
// grouped per 128-row q-tile and scheduled longest-row-first), plus the GQA
// per-group union table ("CompactAttention", summary: Q-block union and
// intra-group union).
//
// Three launches, no host synchronisation:
//   count  one warp per plan row: per 32 k-units, each lane ORs the rq
//          q-unit mask bytes of its k-unit; __ballot_sync + __popc give the
//          row's unit count.  Per-segment histogram of slots-per-row.
//   scan   one CTA: exclusive prefix sums (row pointers, union pointers, sort
//          bases) and totals.
//   fill   one warp per row: ballot + prefix-popcount compaction writes the
//          ascending k-units into slots; sub-mask bits per slot; then a stable
//          counting-sort scatter of the rows (slots descending, row id
//          ascending).
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

// Whether k-unit y is selected by any q-unit of q-tile qt of mask plane mbh
// ([NQB][NKB] of one (b, h)).  `own` counts the logical blocks whose first
// q-unit and first k-unit fall here (so every selected logical block is
// counted exactly once over the whole plan).
__device__ __forceinline__ int unit_union(const uint8_t* __restrict__ mbh, const PlanDev& p, int qt,
                                          int y, int* own) {
  const int kb = y / p.sk;
  const bool first_k = (y % p.sk) == 0;
  int u = 0, o = 0;
  for (int i = 0; i < p.rq; ++i) {
    const int x = qt * p.rq + i;
    const int v = __ldg(mbh + (size_t)(x / p.sq) * p.NKB + kb) != 0;
    u |= v;
    o += (v && first_k && (x % p.sq) == 0);
  }
  *own = o;
  return u;
}

__device__ __forceinline__ int union_unit(const PlanDev& p, int b, int hk, int qt, int y) {
  const int kb = y / p.sk;
  int u = 0;
  for (int hh = 0; hh < p.g && !u; ++hh) {
    const uint8_t* mbh = p.mask + ((size_t)(b * p.H + hk * p.g + hh)) * p.NQB * p.NKB;
    for (int i = 0; i < p.rq; ++i) {
      const int x = qt * p.rq + i;
      u |= __ldg(mbh + (size_t)(x / p.sq) * p.NKB + kb) != 0;
    }
  }
  return u;
}

__global__ void __launch_bounds__(kThreads) plan_count_kernel(const PlanDev p) {
  extern __shared__ int hist_s[];  // [nkeys]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cta = blockIdx.x;
  if (cta < p.segments) {
    for (int k = threadIdx.x; k < p.nkeys; k += kThreads) hist_s[k] = 0;
    __syncthreads();
    for (int i = 0; i < 32; ++i) {
      const int r = cta * kPlanSegRows + warp * 32 + i;
      if (r >= p.rows) break;
      const int bh = r / p.NQT, qt = r % p.NQT;
      const uint8_t* mbh = p.mask + (size_t)bh * p.NQB * p.NKB;
      int cnt = 0, own = 0;
      for (int y0 = 0; y0 < p.NKU; y0 += 32) {
        const int y = y0 + lane;
        int u = 0, o = 0;
        if (y < p.NKU) u = unit_union(mbh, p, qt, y, &o);
        cnt += __popc(__ballot_sync(0xffffffffu, u));
        own += o;
      }
      for (int s = 16; s > 0; s >>= 1) own += __shfl_xor_sync(0xffffffffu, own, s);
      if (lane == 0) {
        const int slots = (cnt + p.rk - 1) / p.rk;
        p.slots[r] = slots;
        p.lcnt[r] = own;
        atomicAdd(&hist_s[slots], 1);
      }
    }
    __syncthreads();
    int* h = p.hist + (size_t)cta * p.nkeys;
    for (int k = threadIdx.x; k < p.nkeys; k += kThreads) h[k] = hist_s[k];
  } else {
    const int useg = cta - p.segments;
    for (int i = 0; i < 32; ++i) {
      const int ur = useg * kPlanSegRows + warp * 32 + i;
      if (ur >= p.urows) break;
      const int bhk = ur / p.NQT, qt = ur % p.NQT;
      const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
      int cnt = 0;
      for (int y0 = 0; y0 < p.NKU; y0 += 32) {
        const int y = y0 + lane;
        const int u = (y < p.NKU) ? union_unit(p, b, hk, qt, y) : 0;
        cnt += __popc(__ballot_sync(0xffffffffu, u));
      }
      if (lane == 0) p.ucnt[ur] = cnt;
    }
  }
}

// Block-wide exclusive scan of one 1024-element chunk; returns the chunk sum.
template <typename T>
__device__ T block_exclusive_scan(T v, T* excl_out, T* warp_sums) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  T x = v;
  for (int s = 1; s < 32; s <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, s);
    if (lane >= s) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = warp_sums[lane];
    for (int s = 1; s < 32; s <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, w, s);
      if (lane >= s) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const T before = (warp > 0) ? warp_sums[warp - 1] : T(0);
  *excl_out = before + x - v;
  const T total = warp_sums[31];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(const PlanDev p) {
  __shared__ long long wsum64[32];
  __shared__ int wsum[32];
  // row pointers
  int carry = 0;
  for (int base = 0; base < p.rows; base += kScanThreads) {
    const int i = base + threadIdx.x;
    const int v = (i < p.rows) ? p.slots[i] : 0;
    int ex;
    const int tot = block_exclusive_scan<int>(v, &ex, wsum);
    if (i < p.rows) p.row_ptr[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    p.row_ptr[p.rows] = carry;
    p.totals[0] = carry;
  }
  // selected logical blocks
  long long acc = 0;
  for (int base = 0; base < p.rows; base += kScanThreads) {
    const int i = base + threadIdx.x;
    long long ex;
    acc += block_exclusive_scan<long long>((i < p.rows) ? (long long)p.lcnt[i] : 0ll, &ex, wsum64);
  }
  if (threadIdx.x == 0) {
    p.totals[1] = acc;
    p.totals[3] = 0;
  }
  // union pointers
  carry = 0;
  for (int base = 0; base < p.urows; base += kScanThreads) {
    const int i = base + threadIdx.x;
    const int v = (i < p.urows) ? p.ucnt[i] : 0;
    int ex;
    const int tot = block_exclusive_scan<int>(v, &ex, wsum);
    if (i < p.urows) p.urow_ptr[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    p.urow_ptr[p.urows] = carry;
    p.totals[2] = carry;
  }
  // sort bases: rows with more slots first; within one slot count, earlier
  // segments first.  Flattened index f = (nkeys-1-key)*segments + seg.
  const int nf = p.nkeys * p.segments;
  carry = 0;
  for (int base = 0; base < nf; base += kScanThreads) {
    const int f = base + threadIdx.x;
    int idx = 0, v = 0;
    if (f < nf) {
      const int key = p.nkeys - 1 - f / p.segments;
      const int seg = f % p.segments;
      idx = seg * p.nkeys + key;
      v = p.hist[idx];
    }
    int ex;
    const int tot = block_exclusive_scan<int>(v, &ex, wsum);
    if (f < nf) p.hist[idx] = carry + ex;
    carry += tot;
  }
}

__global__ void __launch_bounds__(kThreads) plan_fill_kernel(const PlanDev p) {
  extern __shared__ int start_s[];  // [nkeys]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cta = blockIdx.x;
  if (cta < p.segments) {
    for (int i = 0; i < 32; ++i) {
      const int r = cta * kPlanSegRows + warp * 32 + i;
      if (r >= p.rows) break;
      const int bh = r / p.NQT, qt = r % p.NQT;
      const uint8_t* mbh = p.mask + (size_t)bh * p.NQB * p.NKB;
      const int s0 = p.row_ptr[r];
      const int n = p.row_ptr[r + 1] - s0;
      const int cap = n * p.rk;
      int32_t* out = p.slot_ku + (size_t)s0 * p.rk;
      int pos = 0;
      for (int y0 = 0; y0 < p.NKU; y0 += 32) {
        const int y = y0 + lane;
        int o;
        const int u = (y < p.NKU) ? unit_union(mbh, p, qt, y, &o) : 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, u);
        if (u) {
          const int idx = pos + __popc(bal & lanemask_lt());
          if (idx < cap) out[idx] = y;
        }
        pos += __popc(bal);
      }
      for (int idx = pos + lane; idx < cap; idx += 32) out[idx] = -1;
      __threadfence_block();
      __syncwarp();
      for (int s = lane; s < n; s += 32) {
        uint32_t bits = 0;
        for (int j = 0; j < p.rk; ++j) {
          const int y = out[s * p.rk + j];
          if (y < 0) continue;
          const int kb = y / p.sk;
          for (int ii = 0; ii < p.rq; ++ii) {
            const int x = qt * p.rq + ii;
            if (__ldg(mbh + (size_t)(x / p.sq) * p.NKB + kb) != 0) bits |= 1u << (ii * p.rk + j);
          }
        }
        p.slot_mask[s0 + s] = bits;
      }
    }
    // Stable counting-sort scatter of this segment's rows.
    for (int k = threadIdx.x; k < p.nkeys; k += kThreads)
      start_s[k] = p.hist[(size_t)cta * p.nkeys + k];
    const int r = cta * kPlanSegRows + threadIdx.x;
    const bool valid = r < p.rows;
    const int key = valid ? p.slots[r] : -1;
    for (int w = 0; w < kWarps; ++w) {
      __syncthreads();
      if (warp == w) {
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        int pos = 0;
        if (valid) pos = start_s[key] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (valid) {
          p.order[pos] = r;
          if (lane == __ffs(peers) - 1) start_s[key] += __popc(peers);
        }
      }
    }
  } else {
    const int useg = cta - p.segments;
    for (int i = 0; i < 32; ++i) {
      const int ur = useg * kPlanSegRows + warp * 32 + i;
      if (ur >= p.urows) break;
      const int bhk = ur / p.NQT, qt = ur % p.NQT;
      const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
      const int s0 = p.urow_ptr[ur];
      const int cap = p.urow_ptr[ur + 1] - s0;
      int pos = 0;
      for (int y0 = 0; y0 < p.NKU; y0 += 32) {
        const int y = y0 + lane;
        const int u = (y < p.NKU) ? union_unit(p, b, hk, qt, y) : 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, u);
        if (u) {
          const int idx = pos + __popc(bal & lanemask_lt());
          if (idx < cap) p.ukb[s0 + idx] = y;
        }
        pos += __popc(bal);
      }
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream) {
  const int grid = p.segments + p.usegments;
  const size_t smem = (size_t)p.nkeys * sizeof(int);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(plan_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kMaxKeys * (int)sizeof(int));
    cudaFuncSetAttribute(plan_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kMaxKeys * (int)sizeof(int));
    attr_set = true;
  }
  plan_count_kernel<<<grid, kThreads, smem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  plan_scan_kernel<<<1, kScanThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  plan_fill_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bsa
