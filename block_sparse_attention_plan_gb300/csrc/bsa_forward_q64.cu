// Block-sparse attention forward over 64-row q-tiles (plans built with
// BSA_PLAN_Q64) for sm_103a.
//
// A second physical mapping of small query blocks ("Decoupling Logical Masks
// from GPU Execution for Dynamic Block-Sparse Attention" (Tessera), abstract:
// logical blocks are combined into physical tiles): a 64-row query block is a
// q-tile of its own (two 32-row blocks share one) instead of sharing a
// 128-row tile, and the union of selections, with its neighbour.  The
// tensor-core MMA takes M = 128 rows, so the q-tile goes on the N dimension:
// for every slot of 128 keys the kernel computes the transposed scores
//     S^T = K Q^T        (M = 128 keys, N = 64 queries, K = d)
// and accumulates the transposed output
//     O^T += V^T P^T     (M = d channels, N = 64 queries, K = 128 keys),
// both in tensor memory with lane = key (S^T) or channel (O^T) and column =
// query.  P^T goes through shared memory (the B operand of the second MMA),
// written by the softmax threads in the 128-byte-swizzled layout the MMA
// reads.  d = 64 runs the second MMA with M = 128 as well: the upper 64
// lanes of O^T are never read.
//
// Passes (launched by bsa_forward.cu's launch_passes after the key-norm and
// row-bound passes, which are the same as for 128-row tiles):
//   bounded pass  every plan row with each query's reference maximum
//                 m_q = |q| max|k| scale log2(e) (no score exceeds it, so no
//                 running maximum is needed); rows whose weights would
//                 underflow, and rows that need split weights (K/V units
//                 holding a |v| above kSplitV), are queued instead;
//   exact pass    the queued rows, in two sweeps over the row's slots: the
//                 first takes each query's exact maximum score, the second
//                 computes P against it with split weights (hi + lo bf16
//                 terms, a second P V product for lo) and normalises O by the
//                 fp32 sum of the weights.
//
// One CTA (384 threads) per SM, looping over plan rows in schedule order:
//   warp 0   K producer: work items, the row's 64-row Q tile, K tiles (once
//            per sweep);   warp 3   V producer;
//   warp 1   S issuer: S^T of every slot into S^T buffer g mod 2;
//   warp 2   owns tensor memory (256 columns); P V issuer: O^T += V^T P^T;
//   warps 4-11 softmax: warp w has key lanes [32(w%4), 32(w%4)+32) of every
//            slot and queries [32h, 32h+32), h = (w-4)/4, so each thread holds
//            one key's scores for 32 queries.  The per-query weight sums are
//            kept per thread over all of a row's slots and reduced over the
//            row's keys once, at the row's end.
// Tensor memory: [0,64) [64,128) S^T buffers, [128,192) O^T.
//
// Every wait is bounded (watchdog), including the softmax-wide exchange at a
// row's end (an mbarrier, not a named barrier, so that a warp that gives up
// cannot leave the others waiting).
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>

#include "bsa_fwd_common.cuh"

namespace bsa {
namespace {

constexpr int kQ64Threads = 384;
constexpr int kQ64TmemCols = 256;
constexpr uint32_t kQColS = 0;    // S^T buffer b at kQColS + 64 b
constexpr uint32_t kQColO = 128;  // O^T
constexpr int kQRegsControl = 72;
constexpr int kQRegsSoftmax = 208;
static_assert(128 * kQRegsControl + 256 * kQRegsSoftmax <= kQ64Threads * 168, "register split");

template <int D_, bool kExact_>
struct QCfg {
  static constexpr int D = D_;
  static constexpr int kTileBytes = 128 * D * 2;    // K/V tile: 128 keys x d bf16
  static constexpr int kChunks = D / 64;            // 64-column (128-byte) swizzle blocks
  static constexpr int kChunkBytes = 128 * 128;     // one block of a 128-row tile
  static constexpr int kQBytes = 64 * D * 2;        // Q tile: 64 queries x d
  static constexpr int kQChunkBytes = 64 * 128;     // one block of the 64-row Q tile
  static constexpr int kQBufs = (D == 128) ? 1 : 2;
  // Two P^T buffers, so that the softmax of slot g writes while the P V of
  // slot g - 1 still reads; at d = 128 that costs a V ring stage (3 K + 2 V
  // and 2 K + 3 V measured the same).
  static constexpr int kStagesK = (D == 128) ? (kExact_ ? 2 : 3) : (kExact_ ? 4 : 5);
  static constexpr int kStagesV = (D == 128) ? 2 : (kExact_ ? 4 : 5);
  static constexpr int kKSweeps = kExact_ ? 2 : 1;
  static constexpr bool kQueueSplit = !kExact_;
  static constexpr int kPBufs = 2;                   // P^T buffers (slot g uses g mod 2)
  static constexpr int kPTerms = kExact_ ? 2 : 1;    // hi (+ lo) tiles per buffer
  static constexpr int kPBytes = 128 * 128;          // P^T: 128 keys x 64 queries bf16
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBufs * kQBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffP = kOffV + kStagesV * kTileBytes;
  static constexpr int kOffBar = kOffP + kPBufs * kPTerms * kPBytes;
  // barriers
  static constexpr int kBarQFull = 0, kBarQEmpty = 2;
  static constexpr int kBarKFull = 4;
  static constexpr int kBarKEmpty = kBarKFull + kStagesK;
  static constexpr int kBarVFull = kBarKEmpty + kStagesK;
  static constexpr int kBarVEmpty = kBarVFull + kStagesV;
  static constexpr int kBarSFull = kBarVEmpty + kStagesV;  // [2]
  static constexpr int kBarSFree = kBarSFull + 2;          // [2]
  static constexpr int kBarPFull = kBarSFree + 2;          // [kPBufs]
  static constexpr int kBarPFree = kBarPFull + kPBufs;     // [kPBufs]
  static constexpr int kBarOFull = kBarPFree + kPBufs;
  static constexpr int kBarOFree = kBarOFull + 1;
  static constexpr int kBarSync = kBarOFree + 1;           // softmax-wide exchange
  static constexpr int kBarDrain = kBarSync + 1;
  static constexpr int kBarSchedFull = kBarDrain + 1;
  static constexpr int kBarSchedEmpty = kBarSchedFull + kSchedSlots;
  static constexpr int kNumBars = kBarSchedEmpty + kSchedSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kOffSched = kOffMisc + 16;           // int [kSchedSlots][8] work items
  static constexpr int kOffM = kOffSched + 32 * kSchedSlots;  // float [64] reference per query
  static constexpr int kOffRed = kOffM + 64 * 4;            // float [4 quads][64] partials
  static constexpr int kOffInv = kOffRed + 4 * 64 * 4;      // float [64] 1 / row sum
  static constexpr int kOffFlag = kOffInv + 64 * 4;         // int [2 halves][4 quads]
  static constexpr int kSmemBytes = kOffFlag + 8 * 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffP % 1024 == 0 && kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle alignment");
};

// Sum (or maximum) over the 32 lanes of a warp of 32 values per lane: lane l
// returns the reduction of everyone's v[l].  Recursive halving: at each step
// a lane keeps the half of its values selected by one bit of its lane index
// and adds its partner's copy of that half.
template <bool kMax>
__device__ __forceinline__ float xpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int n = 16; n >= 1; n >>= 1) {
    const bool up = (lane & n) != 0;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float keep = up ? v[k + n] : v[k];
      const float send = up ? v[k] : v[k + n];
      const float got = __shfl_xor_sync(0xffffffffu, send, n);
      v[k] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// ------------------------------------------------------------------ MMA issuers
// S issuer: S^T = K Q^T (M=128 keys, N=64 queries, K=16 per instruction) of
// every slot (of every sweep) into S^T buffer g mod 2, once the softmax has
// read that buffer's previous tile and the K tile has landed.
template <class C>
__device__ __noinline__ void q64_s_issuer(const FwdParams& p, const uint8_t* smem, const Smem<C> sm,
                                          uint32_t tmem, const Watchdog wd) {
  constexpr int D = C::D;
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 64, false);  // A = K, B = Q: both K-major
  const uint64_t kdesc0 = smem_desc_sw128(sm.kst(0), 16, 1024);
  const uint64_t qdesc[2] = {smem_desc_sw128(sm.q(0), 16, 1024),
                             smem_desc_sw128(sm.q(C::kQBufs - 1), 16, 1024)};
  uint32_t kc = 0, sg = 0, q_it = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const Item m = sched_take<C>(sm, smem, t, true, false, wd);
    if (m.it < 0) break;
    if (m.n == 0) continue;
    const int qb = q_buf<C>(q_it);
    if (!mbar_wait(sm.bar(C::kBarQFull + qb), q_par<C>(q_it), wd, kSiteQFull)) break;
    tc_fence_after();
    const int ns = C::kKSweeps * m.n;
    for (int j = 0; j < ns; ++j) {
      const int b = (int)(sg & 1u);
      const uint32_t u = sg >> 1;
      if (u > 0 && !mbar_wait(sm.bar(C::kBarSFree + b), (u - 1) & 1u, wd, kSiteSFull)) {
        ok = false;
        break;
      }
      const uint32_t stage = kc % (uint32_t)C::kStagesK;
      if (!mbar_wait(sm.bar(C::kBarKFull + (int)stage), (kc / C::kStagesK) & 1u, wd, kSiteKvFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t kd = kdesc0 + (uint64_t)stage * (uint64_t)(C::kTileBytes >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t aoff = (uint64_t)(((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4);
        const uint64_t boff = (uint64_t)(((kk / 4) * C::kQChunkBytes + (kk % 4) * 32) >> 4);
        mma_ss(tmem + kQColS + 64u * (uint32_t)b, kd + aoff, qdesc[qb] + boff, kIdesc, kk > 0 ? 1u : 0u);
      }
      mma_commit(sm.bar(C::kBarKEmpty + (int)stage));
      mma_commit(sm.bar(C::kBarSFull + b));
      ++kc;
      ++sg;
    }
    if (ok) mma_commit(sm.bar(C::kBarQEmpty + qb));  // Q is free once the row's S MMAs are done
    ++q_it;
  }
  mma_commit(sm.bar(C::kBarDrain));
  drain_wait(sm.bar(C::kBarDrain), 0, wd);
}

// P V issuer: O^T (+)= V^T P^T (M=128, N=64 queries, K=16 keys per
// instruction, 8 instructions; split weights: 8 more with the lo tile) of
// every slot once its P^T is in shared memory and its V tile has landed; the
// first of a row also waits until the previous row's epilogue has read O^T.
// A = the V tile read MN-major (channels contiguous; LBO = next 64
// channels; for d = 64 the upper 64 rows of A read the next 16 KB of shared
// memory and only fill O^T lanes that are never read).
template <class C>
__device__ __noinline__ void q64_pv_issuer(const FwdParams& p, const uint8_t* smem, const Smem<C> sm,
                                           uint32_t tmem, const Watchdog wd) {
  constexpr uint32_t kIdesc = idesc_bf16_f32_mn(128, 64, true, true);
  const uint64_t vdesc0 = smem_desc_sw128(sm.vst(0), C::D == 128 ? C::kChunkBytes : C::kTileBytes, 1024);
  const uint64_t pdesc0 = smem_desc_sw128(sm.base + C::kOffP, C::kPBytes, 1024);
  uint32_t vc = 0, pg = 0, rows = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const Item m = sched_take<C>(sm, smem, t, true, false, wd);
    if (m.it < 0) break;
    const int n = m.n;
    if (n == 0) continue;
    for (int j = 0; j < n; ++j) {
      const int pb = (int)(pg % (uint32_t)C::kPBufs);
      if (!mbar_wait(sm.bar(C::kBarPFull + pb), (pg / C::kPBufs) & 1u, wd, kSitePFull)) {
        ok = false;
        break;
      }
      const uint32_t stage = vc % (uint32_t)C::kStagesV;
      if (!mbar_wait(sm.bar(C::kBarVFull + (int)stage), (vc / C::kStagesV) & 1u, wd, kSiteKvFull)) {
        ok = false;
        break;
      }
      if (j == 0 && rows > 0 && !mbar_wait(sm.bar(C::kBarOFree), (rows - 1) & 1u, wd, kSiteODone)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t vd = vdesc0 + (uint64_t)stage * (uint64_t)(C::kTileBytes >> 4);
      const uint64_t pd = pdesc0 + (uint64_t)(pb * C::kPTerms) * (uint64_t)(C::kPBytes >> 4);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + kQColO, vd + (uint64_t)(kk * (2048 >> 4)), pd + (uint64_t)(kk * (2048 >> 4)), kIdesc,
               (j > 0 || kk > 0) ? 1u : 0u);
      if constexpr (C::kPTerms == 2) {
        const uint64_t pl = pd + (uint64_t)(C::kPBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kQColO, vd + (uint64_t)(kk * (2048 >> 4)), pl + (uint64_t)(kk * (2048 >> 4)), kIdesc, 1u);
      }
      mma_commit(sm.bar(C::kBarVEmpty + (int)stage));
      mma_commit(sm.bar(C::kBarPFree + pb));
      if (j == n - 1) mma_commit(sm.bar(C::kBarOFull));
      ++vc;
      ++pg;
    }
    ++rows;
  }
  mma_commit(sm.bar(C::kBarDrain));
  drain_wait(sm.bar(C::kBarDrain), 0, wd);
}

// ------------------------------------------------------------------ softmax
template <class C, bool kExact>
__device__ __forceinline__ void q64_softmax(const FwdParams& p, uint8_t* smem, const Smem<C>& sm,
                                            uint32_t tmem, const Watchdog& wd) {
  constexpr int D = C::D;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int st = (int)threadIdx.x - 128;  // 0 .. 255 among the softmax threads
  const int h = (warp - 4) >> 2;          // queries [32h, 32h + 32) of the tile
  const int quad = warp & 3;              // TMEM lane quadrant
  const int kl = quad * 32 + lane;        // this thread's key within a slot (S^T lane)
  const uint32_t tl = (uint32_t)(quad * 32) << 16;
  const bool submask = (p.rq * p.rk) > 1;
  const int qi = (p.qu == 64) ? 0 : h;    // q-unit of this thread's queries
  const int ku_shift = p.ku == 32 ? 0 : (p.ku == 64 ? 1 : 2);  // log2(ku / 32)
  const int kj = quad >> ku_shift;        // k-unit position of this thread's key in a slot
  const int my_bit = qi * p.rk + kj;      // its bit in a slot's sub-mask
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_make(sl2, sl2);
  float* m_s = reinterpret_cast<float*>(smem + C::kOffM);
  float* red_s = reinterpret_cast<float*>(smem + C::kOffRed);
  float* inv_s = reinterpret_cast<float*>(smem + C::kOffInv);
  volatile int* flag_s = reinterpret_cast<volatile int*>(smem + C::kOffFlag);
  uint32_t sg = 0, pg = 0, rows = 0, q_it = 0, xc = 0;

  // All eight softmax warps meet (bounded wait on an mbarrier).
  auto sm_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarSync));
    const bool ok = __all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarSync), xc & 1u, wd, kSiteXchg));
    ++xc;
    return ok;
  };

  for (uint32_t t = 0;; ++t) {
    const Item m = sched_take<C>(sm, smem, t, lane == 0, true, wd);
    if (m.it < 0) break;
    if (!m.valid) continue;
    // Tile column q (0..63) is q-unit q / qu of the tile, i.e. q-unit
    // qx + (q / qu) * qs of the head, row q % qu of it.
    auto orow = [&](int q) -> size_t {
      return (size_t)m.bh * p.Nq + (size_t)((m.qx + (q / p.qu) * m.qs) * p.qu + (q & (p.qu - 1)));
    };
    if (m.n == 0) {  // no selected key: O = 0, LSE = -inf
      const int q = st >> 2, part = st & 3;
      uint4* dst = reinterpret_cast<uint4*>(p.O + orow(q) * D + part * (D / 4));
#pragma unroll
      for (int c = 0; c < D / 32; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
      if (part == 0) p.LSE[orow(q)] = -INFINITY;
      continue;
    }
    const int qb = q_buf<C>(q_it);
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarQFull + qb), q_par<C>(q_it), wd, kSiteQFull)))
      break;
    if constexpr (!kExact) {
      // Reference of tile row st / 4: |q| from the 128B-swizzled Q tile (a
      // quarter of the row per thread; 16-byte unit u of row r sits at unit
      // position u ^ (r % 8)), times the row's largest key norm.
      const int q = st >> 2, part = st & 3;
      const uint32_t qrow = sm.q(qb) + (uint32_t)q * 128u;
      float a2 = 0.f, b2 = 0.f;
#pragma unroll
      for (int uu = 0; uu < D / 32; ++uu) {
        const int e0 = part * (D / 4) + uu * 8;  // first element of the 16-byte unit
        const uint4 x = ld_shared_v4(qrow + (uint32_t)((e0 / 64) * C::kQChunkBytes) +
                                     ((uint32_t)(((e0 % 64) / 8) ^ (q & 7)) << 4));
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
          a2 = fmaf(lo, lo, a2);
          b2 = fmaf(hi, hi, b2);
        }
      }
      float s2 = a2 + b2;
      s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
      if (part == 0) m_s[q] = sqrtf(s2) * m.kb * sl2;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarQEmpty + qb));
    ++q_it;

    bool ok = true;
    bool kept = false;  // some slot selected this warp's (q-unit, k-unit) chunk
    // One sweep over the row's slots.  kMaxOnly: the exact pass's first
    // sweep, each query's largest score into mx; otherwise the weights
    // against the references nm2 (negated, pairs) into P^T, with the sums.
    auto sweep = [&](auto max_only, float (&mx)[32], const uint64_t (&nm2)[16], uint64_t (&acc_e)[16]) {
      constexpr bool kMaxOnly = decltype(max_only)::value;
      uint32_t wnext = submask ? __ldg(p.slot_mask + m.s0) : 0u;
      for (int j = 0; j < m.n; ++j) {
        const uint32_t word = wnext;
        if (submask && j + 1 < m.n) wnext = __ldg(p.slot_mask + m.s0 + j + 1);
        const bool on = !submask || ((word >> my_bit) & 1u);  // warp-uniform
        const int b = (int)(sg & 1u);
        const uint32_t u = sg >> 1;
        if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarSFull + b), u & 1u, wd, kSiteSFull))) {
          ok = false;
          return;
        }
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + tl + kQColS + 64u * (uint32_t)b + 32u * (uint32_t)h, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.bar(C::kBarSFree + b));
        ++sg;
        kept |= on;
        if constexpr (kMaxOnly) {
          if (on) {
#pragma unroll
            for (int i = 0; i < 32; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(v[i]));
          }
          continue;
        } else {
          uint32_t pk[16], lo[16];
          if (on) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              f2_split(ffma2(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2x2, nm2[e]),
                       x0, x1);
              const uint64_t p2 = f2_make(ex2_approx(x0), ex2_approx(x1));
              float p0, p1;
              f2_split(p2, p0, p1);
              pk[e] = pack_bf16x2(p0, p1);
              acc_e[e] = fadd2(acc_e[e], p2);
              if constexpr (kExact) {
                // split weights: lo = bf16(p - hi), p - hi exact in fp32
                float r0, r1;
                f2_split(ffma2(f2_make(__uint_as_float(pk[e] << 16), __uint_as_float(pk[e] & 0xffff0000u)),
                               f2_make(-1.f, -1.f), p2),
                         r0, r1);
                lo[e] = pack_bf16x2(r0, r1);
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              pk[e] = 0u;
              lo[e] = 0u;
            }
          }
          // Row kl of the P^T tile (64 queries, 128 bytes): this thread's 32
          // queries are 16-byte units 4h .. 4h+3, stored at unit positions
          // (4h + c) ^ (kl % 8) (the 128-byte swizzle the MMA reads).
          const int pb = (int)(pg % (uint32_t)C::kPBufs);
          const uint32_t pu = pg / C::kPBufs;
          if (pu > 0 && !__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + pb), (pu - 1) & 1u, wd, kSitePFull))) {
            ok = false;
            return;
          }
          const uint32_t prow = sm.base + (uint32_t)(C::kOffP + pb * C::kPTerms * C::kPBytes) + (uint32_t)kl * 128u;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t off = (uint32_t)(((4 * h + c) ^ (kl & 7)) << 4);
            st_shared_v4(prow + off, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            if constexpr (kExact)
              st_shared_v4(prow + (uint32_t)C::kPBytes + off, lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
          }
          fence_proxy_async_smem();  // the MMA reads P^T through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.bar(C::kBarPFull + pb));
          ++pg;
        }
      }
    };

    float mx[32];
    uint64_t nm2[16];
    uint64_t acc_e[16];
#pragma unroll
    for (int i = 0; i < 32; ++i) mx[i] = -INFINITY;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc_e[e] = 0ull;
    if constexpr (kExact) {
      // First sweep: each query's largest score over the row's selected keys.
      sweep(std::true_type{}, mx, nm2, acc_e);
      if (!ok) break;
      red_s[quad * 64 + 32 * h + lane] = xpose_reduce<true>(mx, lane);
      if (!sm_sync()) break;
      if (quad == 0) {
        const int q = 32 * h + lane;
        float x = red_s[q];
#pragma unroll
        for (int q4 = 1; q4 < 4; ++q4) x = fmaxf(x, red_s[q4 * 64 + q]);
        m_s[q] = x * sl2;  // -inf when the query has no selected key
      }
    }
    if (!sm_sync()) break;  // references in m_s
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a = m_s[32 * h + 2 * e], b = m_s[32 * h + 2 * e + 1];
      a = (a == -INFINITY) ? 0.f : a;
      b = (b == -INFINITY) ? 0.f : b;
      nm2[e] = f2_make(-a, -b);
    }
    sweep(std::false_type{}, mx, nm2, acc_e);
    if (!ok) break;

    // ------------------------------------------------------------ epilogue
    // Per-query sums over the row's keys: over this warp's 32 key lanes,
    // then over the four lane quadrants.
    float ce[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) f2_split(acc_e[e], ce[2 * e], ce[2 * e + 1]);
    const float se = xpose_reduce<false>(ce, lane);
    if (lane == 0) flag_s[h * 4 + quad] = kept ? 1 : 0;
    red_s[quad * 64 + 32 * h + lane] = se;
    if (!sm_sync()) break;
    if (quad == 0) {
      // The fp32 sum of p normalises O as well as giving the log-sum-exp.
      const int q = 32 * h + lane;
      const float L = red_s[q] + red_s[64 + q] + red_s[128 + q] + red_s[192 + q];
      const bool keys = flag_s[h * 4] | flag_s[h * 4 + 1] | flag_s[h * 4 + 2] | flag_s[h * 4 + 3];
      if constexpr (!kExact) {
        // weights underflowed although the query has selected keys
        const bool need = keys && !(L >= kFallbackPerKey * (float)(m.n * 128));
        if (__any_sync(0xffffffffu, need) && lane == 0) {
          if (atomicExch(p.fb_flag + m.row, 1) == 0)
            p.fb_list[atomicAdd(p.control + kCtlFallbackCount, 1)] = m.row;
        }
      }
      inv_s[q] = (L > 0.f) ? 1.f / L : 0.f;
      p.LSE[orow(q)] = (L > 0.f) ? (m_s[q] + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    if (!sm_sync()) break;  // inv_s
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarOFull), rows & 1u, wd, kSiteODone))) break;
    tc_fence_after();
    if (quad * 32 < D) {
      // O^T lane kl = channel kl; columns 32h .. 32h+31 = this half's queries.
      uint32_t o[32];
      tmem_ld32(tmem + tl + kQColO + 32u * (uint32_t)h, o);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int q = 32 * h + i;
        const float val = __uint_as_float(o[i]) * inv_s[q];
        p.O[orow(q) * D + kl] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
      }
    }
    // O^T has been read: the next row's first P V may overwrite it.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarOFree));
    ++rows;
  }
}

template <int D, bool kExact>
__global__ void __launch_bounds__(kQ64Threads, 1) bsa_fwd_q64_kernel(const __grid_constant__ FwdParams p) {
  using C = QCfg<D, kExact>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Smem<C> sm{smem_u32(smem)};
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Watchdog wd{abort_flag, p.control + kCtlStatus, p.control + kCtlDetail, p.watchdog_ns};
  // A pass over a queue (the exact pass) with nothing queued: leave before
  // any setup.  The count was written by the previous kernel in the stream.
  if (p.work_count != nullptr && *reinterpret_cast<const volatile int32_t*>(p.work_count) <= 0) return;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    if (sm.base & 1023u) record_failure(wd, -4, 0);  // layout assumption violated
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.bar(C::kBarQFull + i), 1);
      mbar_init(sm.bar(C::kBarQEmpty + i), 1 + 8);  // S issuer commit + softmax warps
      mbar_init(sm.bar(C::kBarSFull + i), 1);
      mbar_init(sm.bar(C::kBarSFree + i), 8);       // one arrival per softmax warp
    }
    for (int i = 0; i < C::kPBufs; ++i) {
      mbar_init(sm.bar(C::kBarPFull + i), 8);       // one arrival per softmax warp
      mbar_init(sm.bar(C::kBarPFree + i), 1);
    }
    for (int s = 0; s < C::kStagesK; ++s) {
      mbar_init(sm.bar(C::kBarKFull + s), 1);
      mbar_init(sm.bar(C::kBarKEmpty + s), 1);
    }
    for (int s = 0; s < C::kStagesV; ++s) {
      mbar_init(sm.bar(C::kBarVFull + s), 1);
      mbar_init(sm.bar(C::kBarVEmpty + s), 1);
    }
    mbar_init(sm.bar(C::kBarOFull), 1);
    mbar_init(sm.bar(C::kBarOFree), 8);
    mbar_init(sm.bar(C::kBarSync), 8);
    mbar_init(sm.bar(C::kBarDrain), 2);  // both MMA threads
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(sm.bar(C::kBarSchedFull + i), 1);
      mbar_init(sm.bar(C::kBarSchedEmpty + i), kSchedConsumers);
    }
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(sm.base + C::kOffMisc, kQ64TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp >= 4) {
    regs_inc<kQRegsSoftmax>();
    q64_softmax<C, kExact>(p, smem, sm, tmem, wd);
  } else {
    regs_dec<kQRegsControl>();
    if (p.rk > 1 && (warp == 0 || warp == 3)) {
      // Slots of several units: the producers run on their whole warp (lane
      // u issues the copies of a slot's unit u).
      if (__shfl_sync(0xffffffffu, *abort_flag == 0 ? 1 : 0, 0)) producer_role_warp<C, false>(p, smem, sm, wd, warp == 0);
    } else if (lane == 0 && !*abort_flag) {
      if (warp == 0) producer_role<C, false>(p, smem, sm, wd, true);
      else if (warp == 1) q64_s_issuer<C>(p, smem, sm, tmem, wd);
      else if (warp == 2) q64_pv_issuer<C>(p, smem, sm, tmem, wd);
      else if (warp == 3) producer_role<C, false>(p, smem, sm, wd, false);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kQ64TmemCols);
  }
}

template <int D, bool kExact>
cudaError_t launch_q64_d(const FwdParams& p, int grid, cudaStream_t stream) {
  const int smem = QCfg<D, kExact>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(bsa_fwd_q64_kernel<D, kExact>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bsa_fwd_q64_kernel<D, kExact><<<grid, kQ64Threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_q64(const FwdParams& p, int d, int grid, cudaStream_t stream, bool exact) {
  if (d == 64) return exact ? launch_q64_d<64, true>(p, grid, stream) : launch_q64_d<64, false>(p, grid, stream);
  return exact ? launch_q64_d<128, true>(p, grid, stream) : launch_q64_d<128, false>(p, grid, stream);
}

}  // namespace bsa
