// Preparation passes of a forward over a plan, launched by launch_forward
// before the bounded pass (bsa_forward_stage can enqueue them separately):
//   key-norm pass   kmax_kernel: the largest |k| and the largest |v| element
//                   of every K/V unit (reads K and V once);
//   row-bound pass  rowbound_kernel: per plan row, the largest of each over
//                   its units (and, for paged K/V, each slot position's pool
//                   row).
// The row's key bound gives the bounded pass its reference maximum
// |q| max|k| scale log2(e) (the Cauchy-Schwarz bound of every score of the
// row); the row's |v| bound decides whether it applies split weights.
#include <cstdint>

#include "bsa_fwd_common.cuh"

namespace bsa {
namespace {

// Largest key norm of every K unit (ku rows) of every K/V head, i.e. a bound
// on |k| for the Cauchy-Schwarz reference of the bounded pass, and largest
// |v| element of every V unit (which decides whether a row applies split
// weights); also clears the fallback flags.  The K units come first, then
// the V units: each CTA streams groups of kKmaxGroupBytes / (ku*d*2)
// consecutive units of one tensor through shared-memory stages with bulk
// copies (one thread issues them, completion on the stage's mbarrier), so
// many bytes are in flight per SM with few registers; each thread then
// reduces the rows it owns (16-byte reads rotated across the row so the
// threads of a warp hit different banks).  One stage per CTA and
// kKmaxCtasPerSm CTAs per SM: more CTAs reducing side by side beat deeper
// rings in a CTA (video-DiT, same bytes in flight: 3 stages x 2 CTAs
// 46.4 us, 2 x 3 42.0 us, 1 x 6 38.3 us with the cache hint below).  The
// copies carry an L2 evict-first hint: K and V are streamed once here, and
// the plan kernels running beside this pass keep their small working set in
// L2 (their time in the step: 60 -> 50 us).  Units wholly past the
// sequence's key length (or, paged, without a valid page) get 0 and are not
// read: their keys are masked.  A wait that runs out is recorded in the
// pass's own status words (its stage may run on another stream beside the
// plan kernels).
constexpr int kKmaxThreads = 128;
constexpr int kKmaxStages = 1;
constexpr int kKmaxCtasPerSm = 6;
constexpr uint32_t kKmaxGroupBytes = 32768;
constexpr int kKmaxSmem = kKmaxStages * (int)kKmaxGroupBytes + 1024;
static_assert(kKmaxStages <= 4, "the stage flags end where the row maxima begin");

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

template <int D>
__global__ void __launch_bounds__(kKmaxThreads) kmax_kernel(const FwdParams p) {
  extern __shared__ __align__(1024) uint8_t kmax_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = blockIdx.x * kKmaxThreads + tid; i < p.rows; i += gridDim.x * kKmaxThreads)
    p.fb_flag[i] = 0;
  const uint32_t base = smem_u32(kmax_smem);
  const uint32_t bars = base + kKmaxStages * kKmaxGroupBytes;  // kKmaxStages mbarriers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(kmax_smem + kKmaxStages * kKmaxGroupBytes + 64);
  int* skip_s = reinterpret_cast<int*>(kmax_smem + kKmaxStages * kKmaxGroupBytes + 128);  // [stages][32]
  float* rmax_s = reinterpret_cast<float*>(kmax_smem + kKmaxStages * kKmaxGroupBytes + 640);  // [8]
  const Watchdog wd{abort_flag, p.control + kCtlKnormStatus, p.control + kCtlKnormDetail, p.watchdog_ns};
  const uint32_t ubytes = (uint32_t)p.ku * D * 2;
  const int G = (int)(kKmaxGroupBytes / ubytes);  // units per stage (1 .. 8)
  const long long units = (long long)p.B * p.Hkv * p.NKU;
  const long long groups = (units + G - 1) / G;   // per tensor
  const long long total = 2 * groups;             // K groups, then V groups
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kKmaxStages; ++s) mbar_init(bars + 8u * s, 1);
    fence_barrier_init();
  }
  __syncthreads();

  // Thread 0: start the copies of group gi (of K below `groups`, else of V)
  // into stage s.
  auto issue = [&](long long gi, int s) {
    const bool isv = gi >= groups;
    const long long g0 = (isv ? gi - groups : gi) * G;
    const uint16_t* src = isv ? p.V : p.K;
    uint32_t bytes = 0;
    for (int k = 0; k < G; ++k) {
      const long long unit = g0 + k;
      int skip = 1;
      if (unit < units) {
        const int head = (int)(unit / p.NKU), y = (int)(unit % p.NKU);  // head = b * Hkv + hkv
        const int b = head / p.Hkv;
        const int key = y * p.ku;
        skip = (p.kv_lens != nullptr && key >= __ldg(p.kv_lens + b)) ? 1 : 0;
        if (p.block_table != nullptr && !skip) {
          const int lp = key / p.page_size;
          const int phys = (lp < p.max_pages) ? __ldg(p.block_table + (size_t)b * p.max_pages + lp) : -1;
          if (phys < 0 || phys >= p.num_pages) skip = 1;
        }
      }
      skip_s[s * 32 + k] = skip;
      if (!skip) bytes += ubytes;
    }
    mbar_arrive_expect_tx(bars + 8u * s, bytes);
    for (int k = 0; k < G; ++k) {
      if (skip_s[s * 32 + k]) continue;
      const long long unit = g0 + k;
      const int head = (int)(unit / p.NKU), y = (int)(unit % p.NKU);
      long long row0 = unit * p.ku;  // contiguous: units in row order
      if (p.block_table != nullptr) {
        const int b = head / p.Hkv, hkv = head % p.Hkv, key = y * p.ku, lp = key / p.page_size;
        const int phys = __ldg(p.block_table + (size_t)b * p.max_pages + lp);
        row0 = ((long long)phys * p.Hkv + hkv) * p.page_size + (key - lp * p.page_size);
      }
      bulk_load(base + s * kKmaxGroupBytes + k * ubytes, src + (size_t)row0 * D, ubytes, bars + 8u * s);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < kKmaxStages; ++s) {
      const long long gi = blockIdx.x + (long long)s * gridDim.x;
      if (gi < total) issue(gi, s);
    }
  }
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  const int rows = G * p.ku;      // rows per stage: 32768 / (2 D)
  uint32_t it = 0;
  for (long long gi = blockIdx.x; gi < total; gi += gridDim.x, ++it) {
    const bool isv = gi >= groups;
    const int s = (int)(it % kKmaxStages);
    const bool waited = mbar_wait(bars + 8u * s, (it / kKmaxStages) & 1u, wd, kSiteKvFull);
    if (!__syncthreads_and(waited)) break;  // uniform: no thread left behind at a barrier
    // Rows tid, tid + 128, ... of the stage; row r at byte r * 2D.  K: the
    // row's squared norm; V: the row's largest |v|.
    for (int rb = 0; rb * kKmaxThreads < rows; ++rb) {
      const int r = rb * kKmaxThreads + tid;
      const uint32_t rowp = base + s * kKmaxGroupBytes + (uint32_t)r * (D * 2);
      float s2a = 0.f, s2b = 0.f;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint4 x = ld_shared_v4(rowp + (uint32_t)(((c + tid) % kChunks) * 16));
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
          if (isv) {
            s2a = fmaxf(s2a, fabsf(lo));
            s2b = fmaxf(s2b, fabsf(hi));
          } else {
            s2a = fmaf(lo, lo, s2a);
            s2b = fmaf(hi, hi, s2b);
          }
        }
      }
      float m = isv ? fmaxf(s2a, s2b) : s2a + s2b;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) rmax_s[rb * (kKmaxThreads / 32) + warp] = m;  // rows 32*(rb*4+warp) ..
    }
    __syncthreads();
    if (tid < G) {
      const long long unit = (isv ? gi - groups : gi) * G + tid;
      if (unit < units) {
        float m = 0.f;
        if (!skip_s[s * 32 + tid]) {
          const int b0 = tid * p.ku / 32, b1 = (tid + 1) * p.ku / 32;  // 32-row blocks of the unit
          for (int q = b0; q < b1; ++q) m = fmaxf(m, rmax_s[q]);
        }
        if (isv) p.vmax[unit] = m;
        else p.kmax[unit] = sqrtf(m);
      }
    }
    __syncthreads();  // stage s and rmax_s free again
    if (tid == 0) {
      const long long gn = gi + (long long)kKmaxStages * gridDim.x;
      if (gn < total) issue(gn, s);
    }
  }
  if (*abort_flag && tid == 0) {
    // Let copies already issued land before the CTA's shared memory goes away.
    for (int s = 0; s < kKmaxStages; ++s) {
      const long long gi = blockIdx.x + (long long)(it + s) * gridDim.x;
      if (gi < total) drain_wait(bars + 8u * ((it + s) % kKmaxStages), ((it + s) / kKmaxStages) & 1u, wd);
    }
  }
}

// Largest key norm over the K units of each plan row's slots (one warp per
// row), the |k| factor of the row's Cauchy-Schwarz reference, and the largest
// |v| element over the same units.  Paged K/V: also
// the pool row of each slot position's unit, (page*Hkv + hkv)*page_size +
// key % page_size with the page from the block table, so the producers read
// rows as they would plan entries.  A page outside the table is an error only
// when the unit holds keys within the sequence's key length (beyond it the
// keys are masked, so page 0 serves).
__global__ void __launch_bounds__(256) rowbound_kernel(const FwdParams p) {
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  const int s0 = __ldg(p.row_ptr + row), s1 = __ldg(p.row_ptr + row + 1);
  float km = 0.f, vm = 0.f;
  if (s0 >= 0 && s1 >= s0 && (long long)s1 <= p.slot_capacity) {  // else the forward reports it
    const int bh = row / p.NQT, b = bh / p.H, h = bh % p.H, hkv = h / p.g;
    const float* kh = p.kmax + (size_t)(b * p.Hkv + hkv) * p.NKU;
    const float* vh = p.vmax + (size_t)(b * p.Hkv + hkv) * p.NKU;
    const int kvl = (p.prow && p.kv_lens) ? __ldg(p.kv_lens + b) : 0x7fffffff;
    for (long long i = (long long)s0 * p.rk + lane; i < (long long)s1 * p.rk; i += 32) {
      const int y = __ldg(p.slot_ku + i);
      const bool valid = y >= 0 && y < p.NKU;
      if (valid) {
        km = fmaxf(km, __ldg(kh + y));
        vm = fmaxf(vm, __ldg(vh + y));
      }
      if (p.prow) {
        int prow = -1;  // padding, or an entry out of range (reported here)
        if (valid) {
          const int key = y * p.ku;
          const int lp = key / p.page_size;
          int phys = (lp < p.max_pages) ? __ldg(p.block_table + (size_t)b * p.max_pages + lp) : -1;
          if (phys < 0 || phys >= p.num_pages) {
            if (key < kvl) record_status(p.control, -7, kSitePlanRange + 4);
            phys = 0;
          }
          prow = (phys * p.Hkv + hkv) * p.page_size + (key - lp * p.page_size);
        } else if (y != -1) {
          record_status(p.control, -7, kSitePlanRange + 3);
        }
        p.prow[i] = prow;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
  }
  if (lane == 0) {
    p.rowk[row] = km;
    p.rowv[row] = vm;
  }
}

}  // namespace

cudaError_t launch_prep(const FwdParams& p, int d, int stages, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (stages & (BSA_STAGE_PREPARE | BSA_STAGE_KNORM)) {
    const long long units = (long long)p.B * p.Hkv * p.NKU;
    const long long per = kKmaxGroupBytes / ((long long)p.ku * d * 2);  // units per stage
    const long long kgroups = 2 * ((units + per - 1) / per);
    long long kgrid = (long long)kKmaxCtasPerSm * (p.sms > 0 ? p.sms : 1);
    if (kgrid > kgroups) kgrid = kgroups;
    if (kgrid < 1) kgrid = 1;
    if (d == 64) {
      e = cudaFuncSetAttribute(kmax_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKmaxSmem);
      if (e == cudaSuccess) kmax_kernel<64><<<(unsigned)kgrid, kKmaxThreads, kKmaxSmem, stream>>>(p);
    } else {
      e = cudaFuncSetAttribute(kmax_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKmaxSmem);
      if (e == cudaSuccess) kmax_kernel<128><<<(unsigned)kgrid, kKmaxThreads, kKmaxSmem, stream>>>(p);
    }
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & (BSA_STAGE_PREPARE | BSA_STAGE_ROWBOUND)) {
    rowbound_kernel<<<(unsigned)((p.rows + 7) / 8), 256, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace bsa
