// Block-sparse attention forward for sm_103a: a persistent, warp-specialised
// flash-style kernel that computes only the K/V tiles a plan lists.
//
// Source of the method: "Decoupling Logical Masks from GPU Execution for
// Dynamic Block-Sparse Attention" (Tessera), abstract -- compute only the
// blocks a logical mask selects, with tiles grouped per GPU task so that data
// movement overlaps computation.  The softmax over tiles is the
// FlashAttention fusion the pages refer to ("Sol-Attn" summary: online
// softmax), with a reading of its reference maximum described below.
//
// Passes of one forward (bsa_forward_stage can enqueue them separately):
//   key-norm pass   the largest |k| and the largest |v| element of every K/V
//                   unit (reads K and V once; bsa_prep.cu);
//   row-bound pass  per plan row, the largest of each over its units (and,
//                   for paged K/V, each slot position's pool row; bsa_prep.cu);
//   bounded pass    this kernel over every plan row with the row's reference
//                   maximum m = |q| max|k| scale log2(e): no score exceeds
//                   it, so no running maximum, exchange or rescale is needed;
//                   a row whose weights would underflow is queued;
//   exact pass      this kernel over the queued rows with a running maximum.
//
// One CTA (384 threads) per SM, looping over plan rows (one 128-row q-tile of
// one head each, possibly of regrouped q-units) in schedule order:
//   warp 0   takes the work items, publishes them to the other roles, loads
//            each row's Q tile and the K tiles of its slots into the K ring
//            (shared-memory stages guarded by full/empty mbarriers);
//   warp 3   loads the V tiles into the V ring.  A slot of 128 keys is
//            gathered as rk units of ku rows (ku = 128 / rk); the producers
//            run on one thread when a slot is one unit, on the whole warp
//            (one TMA box per lane) when it holds several;
//   warp 1   (one thread) issues S = Q K^T (tcgen05.mma, operands in shared
//            memory, result in tensor memory) for every slot, up to two slots
//            ahead of the softmax (S is double-buffered);
//   warp 2   owns the tensor-memory allocation (512 columns); one thread
//            issues O += P V with P read from tensor memory.  Two issuing
//            threads in different warps keep the tensor pipe fed while either
//            one waits on a barrier or is slowed by the softmax warps sharing
//            its scheduler;
//   warps 4-11 the softmax: each row of a slot is shared by two threads, one
//            in warps 4-7 (keys 0-63 of the slot) and one in warps 8-11 (keys
//            64-127); they combine their row sums at the row's end (and, in
//            the exact pass, their maxima while it runs).
//
// Tensor memory (512 x 32-bit columns x 128 lanes; lane = q-tile row):
//   [0,128) S buffer 0   [128,256) S buffer 1   [256,256+d) O
//   [384,448) P buffer 0 [448,512) P buffer 1   (P: bf16 pairs, keys 2c, 2c+1
//   in column c).  Slot g of the CTA uses S and P buffer g mod 2.  A row with
//   split weights writes the low-order terms of slot g into the other P
//   buffer (same layout), which the P V of slot g - 1 must have finished
//   reading first; so such a slot waits for the P V of the slot before it
//   as well as for the one two slots back, and the first slot after such a
//   row waits for the P V of the row's last slot.  The S buffers are
//   released by the softmax after loading in every row.
//
// Split weights.  P V on the tensor cores applies P rounded to bf16, i.e.
// each weight with a relative error of up to 2^-8, which moves O by up to
// 2^-8 times the spread of the V values the row attends.  For rows whose K/V
// units hold a value with |v| > kSplitV (and for every row with
// BSA_FWD_SPLIT_P) each weight p is applied as hi + lo, hi = bf16(p) and
// lo = bf16(p - hi), with a second P V product for lo: the weights are then
// exact to about 2^-16, and O is normalised by the fp32 sum of the weights.
//
// Every wait is bounded (watchdog): on expiry the CTA records
// BSA_ERR_TIMEOUT in the plan's status word, lets its in-flight copies and
// MMAs land, frees tensor memory and exits.
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>

#include "bsa_fwd_common.cuh"

namespace bsa {
namespace {

constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
// Register split: 384 threads x 168 at launch = 64,512 registers =
// 128 x kRegsControl (warps 0-3) + 256 x kRegsSoftmax (warps 4-11).
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 208;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr uint32_t kColS = 0;    // S buffer b at kColS + 128 b
constexpr uint32_t kColO = 256;  // O accumulator, d columns
constexpr uint32_t kColP = 384;  // P buffer b at kColP + 64 b
// Lazy rescale: O and the row sums keep the reference maximum m of the row
// until some score exceeds it by more than kRescaleThreshold (log2 units),
// so weights stay <= 2^16 (bf16 and fp32 hold them exactly as well as 1).
// A half-row whose weight sum is <= 2^16 cannot hold such a score, which
// is what is checked per slot; only then are the exact maxima compared.
constexpr float kRescaleThreshold = 16.0f;
constexpr float kRescaleSumBound = 65536.0f;  // 2^kRescaleThreshold
template <int D_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int kTileBytes = 128 * D * 2;   // 128 rows x d bf16
  static constexpr int kChunks = D / 64;           // 64-column (128-byte) swizzle blocks
  static constexpr int kChunkBytes = 128 * 128;    // one block of 128 rows
  static constexpr int kQBytes = kTileBytes;       // the Q tile is a 128-row tile too
  static constexpr int kQChunkBytes = kChunkBytes;
  static constexpr int kKSweeps = 1;
  static constexpr bool kQueueSplit = false;
  static constexpr int kQBufs = (D == 128) ? 1 : 2;
  static constexpr int kStagesK = (D == 128) ? 3 : 6;
  static constexpr int kStagesV = (D == 128) ? 3 : 6;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBufs * kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
  // barriers
  static constexpr int kBarQFull = 0, kBarQEmpty = 2;
  static constexpr int kBarKFull = 4;
  static constexpr int kBarKEmpty = kBarKFull + kStagesK;
  static constexpr int kBarVFull = kBarKEmpty + kStagesK;
  static constexpr int kBarVEmpty = kBarVFull + kStagesV;
  static constexpr int kBarSFull = kBarVEmpty + kStagesV;   // [2]
  static constexpr int kBarSFree = kBarSFull + 2;           // [2]
  static constexpr int kBarPFull = kBarSFree + 2;           // [2]
  static constexpr int kBarPFree = kBarPFull + 2;           // [2]
  static constexpr int kBarOFull = kBarPFree + 2;
  static constexpr int kBarOFree = kBarOFull + 1;
  static constexpr int kBarXchg = kBarOFree + 1;            // [4 lane quadrants][2 parities]
  static constexpr int kBarDrain = kBarXchg + 8;
  static constexpr int kBarSchedFull = kBarDrain + 1;
  static constexpr int kBarSchedEmpty = kBarSchedFull + kSchedSlots;
  static constexpr int kNumBars = kBarSchedEmpty + kSchedSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kOffSched = kOffMisc + 16;          // int [kSchedSlots][8] work items
  static constexpr int kOffX = kOffSched + 32 * kSchedSlots;  // float [2 parities][2 halves][128 rows]
  static constexpr int kSmemBytes = kOffX + 2 * 2 * 128 * 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// ------------------------------------------------------------------ MMA issuer
// Descriptors are built once; per instruction only a compile-time offset is
// added (the start-address field is the low 14 bits of the descriptor and
// shared-memory offsets here never carry out of it).
template <int D>
struct MmaState {
  using C = Cfg<D>;
  uint64_t qdesc[2];  // K-major SW128 descriptor of each Q buffer
  uint64_t kdesc0;    // K-major SW128 descriptor of K stage 0
  uint64_t vdesc0;    // MN-major SW128 descriptor of V stage 0 (LBO = next 64 columns)
  uint32_t kc = 0;    // K tiles consumed
  uint32_t vc = 0;    // V tiles consumed
  uint32_t sg = 0;    // S tiles issued (slot g of the CTA uses S/P buffer g mod 2)
  uint32_t pg = 0;    // P V products issued
  static constexpr uint64_t kStageStep = (uint64_t)(C::kTileBytes >> 4);
};

// S = Q K^T into S buffer sg mod 2 (M=128, N=128, K=16 per instruction, d/16
// instructions), once that buffer's previous tile has been read out (by the
// softmax, or for split weights by that slot's P V).
template <int D>
__device__ __forceinline__ bool issue_s(const Smem<Cfg<D>>& sm, MmaState<D>& st, uint32_t tmem, int qb,
                                        const Watchdog& wd) {
  using C = Cfg<D>;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);
  const int b = (int)(st.sg & 1u);
  const uint32_t u = st.sg >> 1;
  if (u > 0 && !mbar_wait(sm.bar(C::kBarSFree + b), (u - 1) & 1u, wd, kSiteSFull)) return false;
  const uint32_t stage = st.kc % (uint32_t)C::kStagesK;
  if (!mbar_wait(sm.bar(C::kBarKFull + (int)stage), (st.kc / C::kStagesK) & 1u, wd, kSiteKvFull))
    return false;
  tc_fence_after();
  const uint64_t kd = st.kdesc0 + (uint64_t)stage * MmaState<D>::kStageStep;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4);
    mma_ss(tmem + kColS + 128u * (uint32_t)b, st.qdesc[qb] + off, kd + off, kIdescS,
           kk > 0 ? 1u : 0u);
  }
  mma_commit(sm.bar(C::kBarKEmpty + (int)stage));
  mma_commit(sm.bar(C::kBarSFull + b));
  ++st.kc;
  ++st.sg;
  return true;
}

// O (+)= P V: M=128, N=d, K=16 keys per instruction, 8 instructions; P from
// tensor memory (columns [8kk, 8kk+8) hold keys [16kk, 16kk+16)), V rows
// [16kk, 16kk+16) start 2048 bytes apart.  Split weights: 8 more
// instructions with the low-order terms, which sit in the slot's S buffer
// (keys [16kk, 16kk+16) in columns 64(kk/4) + 8(kk%4) .. +8), against the
// same V rows.
template <int D>
__device__ __forceinline__ void issue_pv(MmaState<D>& st, uint32_t tmem, uint32_t stage,
                                         bool accumulate, bool split) {
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);
  const uint32_t pcol = tmem + kColP + 64u * (st.pg & 1u);
  const uint64_t vd = st.vdesc0 + (uint64_t)stage * MmaState<D>::kStageStep;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(tmem + kColO, pcol + 8u * (uint32_t)kk, vd + (uint64_t)(kk * (2048 >> 4)), kIdescPV,
           (accumulate || kk > 0) ? 1u : 0u);
  if (split) {
    const uint32_t lcol = tmem + kColP + 64u * ((st.pg & 1u) ^ 1u);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(tmem + kColO, lcol + 8u * (uint32_t)kk, vd + (uint64_t)(kk * (2048 >> 4)), kIdescPV, 1u);
  }
}

// S issuer: S of every slot, in slot order, as soon as its S buffer has been
// read out (two slots back) and its K tile has landed.
template <int D>
__device__ __noinline__ void s_issuer_role(const FwdParams& p, const uint8_t* smem, const Smem<Cfg<D>> sm,
                                           uint32_t tmem, const Watchdog wd) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.qdesc[0] = smem_desc_sw128(sm.q(0), 16, 1024);
  st.qdesc[1] = smem_desc_sw128(sm.q(C::kQBufs - 1), 16, 1024);
  st.kdesc0 = smem_desc_sw128(sm.kst(0), 16, 1024);
  uint32_t q_it = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const Item m = sched_take<Cfg<D>>(sm, smem, t, true, false, wd);
    if (m.it < 0) break;
    if (m.n == 0) continue;
    const int qb = q_buf<Cfg<D>>(q_it);
    if (!mbar_wait(sm.bar(C::kBarQFull + qb), q_par<Cfg<D>>(q_it), wd, kSiteQFull)) break;
    tc_fence_after();
    for (int j = 0; j < m.n && ok; ++j) ok = issue_s<D>(sm, st, tmem, qb, wd);
    if (ok) mma_commit(sm.bar(C::kBarQEmpty + qb));  // Q is free once the row's S MMAs are done
    ++q_it;
  }
  mma_commit(sm.bar(C::kBarDrain));
  drain_wait(sm.bar(C::kBarDrain), 0, wd);
}

// P V issuer: O (+)= P V of every slot once its P is in tensor memory and its
// V tile has landed; the first of a row also waits until the previous row's
// epilogue has read O out.  Runs in its own warp so that its waits and
// commits never leave the tensor pipe without queued S work.
template <int D>
__device__ __noinline__ void pv_issuer_role(const FwdParams& p, const uint8_t* smem, const Smem<Cfg<D>> sm,
                                            uint32_t tmem, const Watchdog wd) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.vdesc0 = smem_desc_sw128(sm.vst(0), C::kChunkBytes, 1024);
  uint32_t rows = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const Item m = sched_take<Cfg<D>>(sm, smem, t, true, false, wd);
    if (m.it < 0) break;
    const int n = m.n;
    if (n == 0) continue;
    for (int j = 0; j < n && ok; ++j) {
      const int b = (int)(st.pg & 1u);
      if (!mbar_wait(sm.bar(C::kBarPFull + b), (st.pg >> 1) & 1u, wd, kSitePFull)) {
        ok = false;
        break;
      }
      const uint32_t stage = st.vc % (uint32_t)C::kStagesV;
      if (!mbar_wait(sm.bar(C::kBarVFull + (int)stage), (st.vc / C::kStagesV) & 1u, wd,
                     kSiteKvFull)) {
        ok = false;
        break;
      }
      if (j == 0 && rows > 0 &&
          !mbar_wait(sm.bar(C::kBarOFree), (rows - 1) & 1u, wd, kSiteODone)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv<D>(st, tmem, stage, j > 0, m.split);
      mma_commit(sm.bar(C::kBarVEmpty + (int)stage));
      mma_commit(sm.bar(C::kBarPFree + b));  // also frees the other buffer's low-order terms
      if (j == n - 1) mma_commit(sm.bar(C::kBarOFull));
      ++st.vc;
      ++st.pg;
    }
    ++rows;
  }
  mma_commit(sm.bar(C::kBarDrain));
  drain_wait(sm.bar(C::kBarDrain), 0, wd);
}

// ------------------------------------------------------------------ softmax
// Bounded pass (kExact = false): every row takes as its reference maximum the
// Cauchy-Schwarz bound |q| * max|k| * scale * log2(e) over the K units of its
// slots, which no score of the row exceeds, so each weight is <= 1, no
// rescale is ever due and the two threads of a row need no exchange until
// the epilogue.  A row whose weights then sum to less than 2^-64 (the bound
// was far above its scores) is queued for the exact pass.
// Exact pass (kExact = true): the running row maximum, agreed between the
// two threads of a row, with a lazy rescale of O.
template <int D, bool kExact, bool kElem>
__device__ __forceinline__ void softmax_role(const FwdParams& p, uint8_t* smem, const Smem<Cfg<D>>& sm,
                                             uint32_t tmem, const Watchdog& wd) {
  using C = Cfg<D>;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int h = (warp - 4) >> 2;          // key half of each slot: [64h, 64h + 64)
  const int quad = warp & 3;              // TMEM lane quadrant of this warp
  const int rloc = quad * 32 + lane;      // row within the q-tile
  const uint32_t tl = (uint32_t)(quad * 32) << 16;
  const int qi = rloc / p.qu;
  const bool submask = (p.rq * p.rk) > 1;
  const int ku_shift = p.ku == 32 ? 0 : (p.ku == 64 ? 1 : 2);  // log2(ku / 32)
  const uint32_t my_bits_mask = (1u << p.rk) - 1u;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_make(sl2, sl2);
  float* xbuf = reinterpret_cast<float*>(smem + C::kOffX);
  uint32_t sg = 0, rows = 0, xc = 0, q_it = 0;
  bool lo_prev = false;  // the last row with slots applied split weights
  uint32_t bits = 0xffffffffu;  // this row's sub-mask bits for the current slot
  // Element mask (causal / key lengths): key position of the first key of each
  // of this thread's two 32-key chunks of the current slot (-1: padding), the
  // last key position this row keeps, and the smallest of that over the warp.
  int cbase[2] = {0, 0};
  int lim_row = 0x7fffffff, lim_warp = 0x7fffffff, lim_warp_hi = 0x7fffffff;
  bool live = false;  // some key of this thread's columns kept in the current slot
  // Bit c: 32-key chunk c of this thread's columns may hold a kept key for
  // some row of the warp (warp-uniform).  The exponentials of a chunk without
  // one are skipped: its weights are +0 either way.
  uint32_t chunks = 3u;

  // One float per row with the thread of the other key half that owns the
  // same row (warp quad + 4 <-> quad + 8); double-buffered by round parity.
  // post() hands this thread's value over; collect() waits for the
  // partner's value of the same round.
  auto post = [&](float mine) {
    const int par = (int)(xc & 1u);
    xbuf[(par * 2 + h) * 128 + rloc] = mine;
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarXchg + quad * 2 + par));
  };
  auto collect = [&](float& theirs) -> bool {
    const int par = (int)(xc & 1u);
    const uint32_t bar = sm.bar(C::kBarXchg + quad * 2 + par);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, (xc >> 1) & 1u, wd, kSiteXchg));
    if (ok) theirs = xbuf[(par * 2 + (h ^ 1)) * 128 + rloc];
    ++xc;
    return ok;
  };
  auto exchange = [&](float mine, float& theirs) -> bool {
    post(mine);
    return collect(theirs);
  };
  // This thread's 64 scores of the slot in S buffer `sbuf` (masked -> -inf).
  auto load_s = [&](uint32_t sbuf, uint32_t (&v)[64]) {
    tmem_ld32_at<0>(sbuf + 64u * (uint32_t)h, v);
    tmem_ld32_at<32>(sbuf + 64u * (uint32_t)h + 32u, v);
    tmem_wait_ld();
    chunks = 3u;
    if (submask) {
      // 32-key chunk 2h + c lies in k-unit (2h + c) >> ku_shift; a warp's rows
      // share one q-unit, so the branch is warp-uniform.  The bounded pass
      // never reads a dropped chunk's scores; the exact pass takes maxima
      // over all 64, so there they become -inf.
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!((bits >> ((2 * h + c) >> ku_shift)) & 1u)) {
          chunks &= ~(1u << c);
          if constexpr (kExact) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[c * 32 + e] = __float_as_uint(-INFINITY);
          }
        }
      }
    }
    live = !submask || bits != 0u;  // the row keeps a key of this slot (block level)
    if constexpr (kElem) {
      if (p.elem_mask) {
        live = false;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (submask && !((bits >> ((2 * h + c) >> ku_shift)) & 1u)) continue;
          // Keys base .. base+31 (ascending): all kept for every row of the
          // warp when the last one is within the warp's smallest limit
          // (warp-uniform); otherwise per element.
          const int base = cbase[c];
          live |= (base >= 0 && base <= lim_row);
          if (base >= 0 && base + 31 <= lim_warp) continue;
          if (base < 0 || base > lim_warp_hi) {  // no row of the warp keeps a key of it
            chunks &= ~(1u << c);
            if constexpr (!kExact) continue;
          }
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (base < 0 || base + e > lim_row) v[c * 32 + e] = __float_as_uint(-INFINITY);
        }
      }
    }
  };
  // p = 2^(s*scale*log2e - m) as bf16 pairs into pk (keys 2e, 2e+1 -> pk[e]).
  // Returns the fp32 sum of the 64 values of p, which both the log-sum-exp
  // and the normalisation of O use (the bf16 weights the P V product applies
  // differ from p by at most 2^-8 relatively, in unbiased round-to-nearest
  // steps).  Chunks dropped from `chunks` get +0 weights without
  // exponentials (adding +0 leaves the sum as it is).
  auto exp_pack = [&](const uint32_t (&v)[64], uint32_t (&pk)[32], float m) -> float {
    const float mb = (m == -INFINITY) ? 0.f : m;
    const uint64_t nmbx2 = f2_make(-mb, -mb);
    uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (chunks & (1u << c)) {
#pragma unroll
        for (int e = 16 * c; e < 16 * c + 16; ++e) {
          float x0, x1;
          f2_split(ffma2(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2x2, nmbx2),
                   x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          pk[e] = pack_bf16x2(p0, p1);
          acc2[e & 1] = fadd2(acc2[e & 1], f2_make(p0, p1));
        }
      } else {
#pragma unroll
        for (int e = 16 * c; e < 16 * c + 16; ++e) pk[e] = 0u;
      }
    }
    float s0, s1, s2, s3;
    f2_split(acc2[0], s0, s1);
    f2_split(acc2[1], s2, s3);
    return (s0 + s1) + (s2 + s3);
  };
  // Split weights: pk gets hi = bf16(p), lo gets bf16(p - hi) (p - hi is
  // exact in fp32: hi is within a factor of two of p).  The weights applied,
  // hi + lo, are within 2^-16 of p; the fp32 sum of p normalises them.
  auto exp_pack_split = [&](const uint32_t (&v)[64], uint32_t (&pk)[32], uint32_t (&lo)[32],
                            float m) -> float {
    const float mb = (m == -INFINITY) ? 0.f : m;
    const uint64_t nmbx2 = f2_make(-mb, -mb);
    const uint64_t neg1x2 = f2_make(-1.f, -1.f);
    uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (chunks & (1u << c)) {
#pragma unroll
        for (int e = 16 * c; e < 16 * c + 16; ++e) {
          float x0, x1;
          f2_split(ffma2(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2x2, nmbx2),
                   x0, x1);
          const uint64_t p2 = f2_make(ex2_approx(x0), ex2_approx(x1));
          float p0, p1;
          f2_split(p2, p0, p1);
          const uint32_t hi = pack_bf16x2(p0, p1);
          pk[e] = hi;
          acc2[e & 1] = fadd2(acc2[e & 1], p2);
          float r0, r1;
          f2_split(ffma2(f2_make(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u)),
                         neg1x2, p2),
                   r0, r1);
          lo[e] = pack_bf16x2(r0, r1);
        }
      } else {
#pragma unroll
        for (int e = 16 * c; e < 16 * c + 16; ++e) {
          pk[e] = 0u;
          lo[e] = 0u;
        }
      }
    }
    float s0, s1, s2, s3;
    f2_split(acc2[0], s0, s1);
    f2_split(acc2[1], s2, s3);
    return (s0 + s1) + (s2 + s3);
  };
  for (uint32_t t = 0;; ++t) {
    const Item m = sched_take<Cfg<D>>(sm, smem, t, lane == 0, true, wd);
    if (m.it < 0) break;
    if (!m.valid) continue;
    // Query position of this thread's row: q-unit qi of the tile is q-unit
    // qx + qi*qs of the head.
    const int qpos = (m.qx + qi * m.qs) * p.qu + (rloc & (p.qu - 1));
    const size_t orow = (size_t)m.bh * p.Nq + qpos;
    uint4* optr = reinterpret_cast<uint4*>(p.O + orow * D + h * (D / 2));
    if (m.n == 0) {  // no selected key: O = 0, LSE = -inf
#pragma unroll
      for (int c = 0; c < D / 16; ++c) optr[c] = make_uint4(0u, 0u, 0u, 0u);
      if (h == 0) p.LSE[orow] = -INFINITY;
      continue;
    }
    // The row's Q tile: (bounded pass) this row's query norm; then release
    // it (with the S issuer's commit, the buffer can be refilled).
    const int qb = q_buf<Cfg<D>>(q_it);
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarQFull + qb), q_par<Cfg<D>>(q_it), wd, kSiteQFull)))
      break;
    float m_ref = -INFINITY;
    if constexpr (!kExact) {
      // |q|^2 from the 128B-swizzled tile: 16-byte unit u of row r in a
      // 64-column chunk sits at unit position u ^ (r % 8).
      float q2a = 0.f, q2b = 0.f;
      const uint32_t qrow = sm.q(qb) + (uint32_t)rloc * 128u;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          const uint4 x = ld_shared_v4(qrow + (uint32_t)(c * C::kChunkBytes) + ((u4 ^ (rloc & 7)) << 4));
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
            q2a = fmaf(lo, lo, q2a);
            q2b = fmaf(hi, hi, q2b);
          }
        }
      }
      m_ref = sqrtf(q2a + q2b) * m.kb * sl2;  // m.kb: largest key norm of the row's K units
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarQEmpty + qb));
    ++q_it;
    if (kElem && p.elem_mask) {
      const int qmin = qpos - lane;  // the warp's 32 rows lie in one q-unit (qu >= 32)
      const int kvl = p.kv_lens ? __ldg(p.kv_lens + m.bh / p.H) : 0x7fffffff;
      lim_row = min(p.causal ? qpos + p.causal_off : 0x7fffffff, kvl - 1);
      lim_warp = min(p.causal ? qmin + p.causal_off : 0x7fffffff, kvl - 1);
      lim_warp_hi = min(p.causal ? qmin + 31 + p.causal_off : 0x7fffffff, kvl - 1);
    }
    float l_run = 0.f;                // the row sum of p (this thread's keys)
    bool has_keys = false;            // (bounded pass) some key of this thread's columns is kept
    bool ok = true;
    // The slot loop, instantiated per kind of row (split weights or not): a
    // row runs one of them, so the hot loop holds one exponential path.
    auto slot_loop = [&](auto split_c) {
    constexpr bool kSplit = decltype(split_c)::value;
    for (int j = 0; j < m.n; ++j) {
      const int b = (int)(sg & 1u);
      const uint32_t u = sg >> 1;
      if (submask) bits = (__ldg(p.slot_mask + m.s0 + j) >> (qi * p.rk)) & my_bits_mask;
      if (kElem && p.elem_mask) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * h + 32 * c;  // ku = 32 << ku_shift
          const int y = __ldg(p.slot_ku + (size_t)(m.s0 + j) * p.rk + (col0 >> (5 + ku_shift)));
          cbase[c] = (y < 0) ? -1 : (y << (5 + ku_shift)) + (col0 & (p.ku - 1));
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarSFull + b), u & 1u, wd, kSiteSFull))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[64];
      load_s(tmem + tl + kColS + 128u * (uint32_t)b, v);
      // The scores are in registers: hand the S buffer back for the next S.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(C::kBarSFree + b));
      uint32_t pk[32];
      uint32_t lo[kSplit ? 32 : 1];
      float sum, factor = 1.f;
      const uint32_t pcol = tmem + tl + kColP + 64u * (uint32_t)b + 32u * (uint32_t)h;
      // Split weights: the low-order terms go to the same columns of the
      // other P buffer (the slot's P V reads both).
      const uint32_t lcol = tmem + tl + kColP + 64u * (uint32_t)(b ^ 1) + 32u * (uint32_t)h;
      // Weights against reference `mr` into pk (and, split, lo); their sum.
      auto exps = [&](float mr) -> float {
        if constexpr (kSplit) return exp_pack_split(v, pk, lo, mr);
        else return exp_pack(v, pk, mr);
      };
      // Until the P V of slot g has finished (both threads of a row ask
      // together, so the warp waits together).
      auto wait_pv = [&](uint32_t g) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + (int)(g & 1u)), (g >> 1) & 1u, wd,
                                                 kSitePFull));
      };
      // P buffer b was last read by the P V of slot sg - 2.  With split
      // weights the other buffer, where this slot writes its low-order terms,
      // is read by the P V of slot sg - 1: wait for that one too.
      auto store_p = [&]() -> bool {
        if (u > 0 && !wait_pv(sg - 2)) return false;
        if constexpr (kSplit) {
          if (sg > 0 && !wait_pv(sg - 1)) return false;
        }
        tmem_st32(pcol, pk);
        if constexpr (kSplit) tmem_st32(lcol, lo);
        return true;
      };
      if constexpr (!kExact) {
        has_keys |= live;  // (set by load_s)
        sum = exps(m_ref);
        if (!store_p()) {
          ok = false;
          break;
        }
      } else if (m_ref == -INFINITY) {
        // No reference yet in this row: the whole-row maximum first (both
        // threads of a row get the same value and so the same reference).
        float mx4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) mx4[c] = fmaxf(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
#pragma unroll
        for (int e = 8; e < 64; e += 8) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            mx4[c] = fmax3(mx4[c], __uint_as_float(v[e + 2 * c]), __uint_as_float(v[e + 2 * c + 1]));
        }
        float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        float mo = -INFINITY;
        if (!exchange(mx, mo)) {
          ok = false;
          break;
        }
        m_ref = fmaxf(mx, mo) * sl2;  // stays -inf while every key so far is masked
        sum = exps(m_ref);
        if (!store_p()) {
          ok = false;
          break;
        }
      } else {
        // Exponentials against the current reference right away; whether a
        // rescale is due is settled while P is being written.
        sum = exps(m_ref);
        post(sum);
        if (!store_p()) {
          ok = false;
          break;
        }
        float sw_other = 0.f;
        if (!collect(sw_other)) {
          ok = false;
          break;
        }
        // Both threads of a row see the same two sums, and the two warps of a
        // lane quadrant hold the same rows: they take this branch together.
        if (__any_sync(0xffffffffu, sum > kRescaleSumBound || sw_other > kRescaleSumBound)) {
          float mx4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) mx4[c] = fmaxf(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
#pragma unroll
          for (int e = 8; e < 64; e += 8) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              mx4[c] = fmax3(mx4[c], __uint_as_float(v[e + 2 * c]), __uint_as_float(v[e + 2 * c + 1]));
          }
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          float mo = -INFINITY;
          if (!exchange(mx, mo)) {
            ok = false;
            break;
          }
          const float m_new = fmaxf(mx, mo) * sl2;
          if (__any_sync(0xffffffffu, m_new > m_ref + kRescaleThreshold)) {
            if (m_new > m_ref + kRescaleThreshold) {
              factor = ex2_approx(m_ref - m_new);
              m_ref = m_new;
            }
            tmem_wait_st();  // the first stores of this slot's terms are done
            sum = exps(m_ref);
            // O changes scale: the P V of slot g - 1 must have finished with
            // it (the one of slot g starts only after this slot's P is
            // published).
            const uint32_t g1 = sg - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + (int)(g1 & 1u)), (g1 >> 1) & 1u, wd, kSitePFull))) {
              ok = false;
              break;
            }
            tc_fence_after();
            tmem_wait_st();
            tmem_st32(pcol, pk);
            if constexpr (kSplit) tmem_st32(lcol, lo);
            const uint32_t o_addr = tmem + tl + kColO + (uint32_t)(h * (D / 2));
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              uint32_t o[32];
              tmem_ld32(o_addr + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
              tmem_st32(o_addr + c * 32, o);
            }
          }
        }
      }
      tmem_wait_st();
      l_run = l_run * factor + sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(C::kBarPFull + b));  // one arrival per warp
      ++sg;
    }
    };
    // After a row with split weights, the low-order terms of its last slot
    // sit in the P buffer this row's first slot writes: wait for the P V
    // that reads them (once per such row, outside the slot loop).
    if (lo_prev && sg > 0 &&
        !__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + (int)((sg - 1) & 1u)), ((sg - 1) >> 1) & 1u,
                                           wd, kSitePFull)))
      break;
    lo_prev = m.split;
    if (m.split) slot_loop(std::true_type{});
    else slot_loop(std::false_type{});
    if (!ok) break;
    // ------------------------------------------------------------ epilogue
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarOFull), rows & 1u, wd, kSiteODone))) break;
    tc_fence_after();
    float l_other = 0.f;
    if (!exchange(l_run, l_other)) break;
    const float L = l_run + l_other;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    if constexpr (!kExact) {
      // Whether the row keeps any key: without an element mask both threads
      // see the same sub-mask bits; with one, they combine their columns.
      float hk_other = has_keys ? 1.f : 0.f;
      if (kElem && p.elem_mask && !exchange(has_keys ? 1.f : 0.f, hk_other)) break;
      const bool row_keys = has_keys || hk_other > 0.f;
      // Both threads of a row compute the same L and row_keys.
      const bool need = row_keys && !(L >= kFallbackPerKey * (float)(m.n * 128));
      if (__any_sync(0xffffffffu, need) && lane == 0) {
        if (atomicExch(p.fb_flag + m.row, 1) == 0)
          p.fb_list[atomicAdd(p.control + kCtlFallbackCount, 1)] = m.row;
      }
    }
    const uint32_t o_addr = tmem + tl + kColO + (uint32_t)(h * (D / 2));
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {  // this thread's half of the row, 32 columns at a time
      uint32_t o[32];
      tmem_ld32(o_addr + c * 32, o);
      tmem_wait_ld();
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
      if (p.o_v8) {  // whole 32-byte sectors: half the store instructions
#pragma unroll
        for (int q8 = 0; q8 < 2; ++q8) {
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w8[e] = pk[8 * q8 + e];
          st_global_v8(optr + c * 4 + 2 * q8, w8);
        }
      } else {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          optr[c * 4 + q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
      }
    }
    // O has been read: the next row's first P V may overwrite it.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarOFree));
    if (h == 0) p.LSE[orow] = (L > 0.f) ? (m_ref + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    ++rows;
  }
}

// kMode: 0 plain; 1 paged K/V (the producers read pool rows, the softmax is
// the plain one); 2 element masks (causal / key lengths), with or without
// pages (runtime-selected inside).  The softmax's element-mask code alone
// costs 3.5-10 % where no mask is set, so only mode 2 carries it.
// kMulti: slots of several K/V units (p.rk > 1), gathered by whole producer
// warps; a separate instantiation, so that the kernels of one-unit slots keep
// the single-thread producers alone (about 1 % faster than with both forms in
// one binary).
template <int D, bool kExact, int kMode, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1) bsa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  constexpr bool kPaged = kMode != 0;  // producers: keys may be pool rows
  constexpr bool kElem = kMode == 2;   // softmax: element masks
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Smem<Cfg<D>> sm{smem_u32(smem)};
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
      // one arrival per softmax warp
      mbar_init(sm.bar(C::kBarSFree + i), 8);
      mbar_init(sm.bar(C::kBarPFull + i), 8);  // one arrival per softmax warp
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
    for (int i = 0; i < 8; ++i) mbar_init(sm.bar(C::kBarXchg + i), 2);  // the two warps of a quadrant
    mbar_init(sm.bar(C::kBarDrain), 2);  // both MMA threads
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(sm.bar(C::kBarSchedFull + i), 1);
      mbar_init(sm.bar(C::kBarSchedEmpty + i), kSchedConsumers);
    }
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(sm.base + C::kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp >= 4) {
    regs_inc<kRegsSoftmax>();
    softmax_role<D, kExact, kElem>(p, smem, sm, tmem, wd);
  } else {
    regs_dec<kRegsControl>();
    if (kMulti && (warp == 0 || warp == 3)) {
      // Slots of several units: the producers run on their whole warp (lane
      // u issues the copies of a slot's unit u).
      if (__shfl_sync(0xffffffffu, *abort_flag == 0 ? 1 : 0, 0))
        producer_role_warp<Cfg<D>, kPaged>(p, smem, sm, wd, warp == 0);
    } else if (lane == 0 && !*abort_flag) {
      if (!kMulti && warp == 0) producer_role<Cfg<D>, kPaged>(p, smem, sm, wd, true);
      else if (warp == 1) s_issuer_role<D>(p, smem, sm, tmem, wd);
      else if (warp == 2) pv_issuer_role<D>(p, smem, sm, tmem, wd);
      else if (!kMulti && warp == 3) producer_role<Cfg<D>, kPaged>(p, smem, sm, wd, false);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void watchdog_selftest_kernel(int32_t* status, long long limit_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t bar = smem_u32(&b);
  mbar_init(bar, 1);
  fence_barrier_init();
  Watchdog wd{&abort_flag, status + kCtlStatus, status + kCtlDetail, limit_ns};
  // Nothing ever arrives on this barrier: the wait must give up by itself.
  if (mbar_wait(bar, 0, wd, kSiteSelftest)) status[3] = 1;
}

template <int D, bool kExact, int kMode, bool kMulti>
cudaError_t launch_dm(const FwdParams& p, int grid, cudaStream_t stream) {
  const int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(bsa_fwd_kernel<D, kExact, kMode, kMulti>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bsa_fwd_kernel<D, kExact, kMode, kMulti><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}
template <int D, bool kExact, int kMode>
cudaError_t launch_dk(const FwdParams& p, int grid, cudaStream_t stream) {
  return p.rk > 1 ? launch_dm<D, kExact, kMode, true>(p, grid, stream)
                  : launch_dm<D, kExact, kMode, false>(p, grid, stream);
}
template <int D, bool kExact>
cudaError_t launch_d(const FwdParams& p, int grid, cudaStream_t stream) {
  if (p.elem_mask) return launch_dk<D, kExact, 2>(p, grid, stream);
  if (p.block_table != nullptr) return launch_dk<D, kExact, 1>(p, grid, stream);
  return launch_dk<D, kExact, 0>(p, grid, stream);
}

template <int D>
cudaError_t launch_passes(const FwdParams& p, int grid, cudaStream_t stream, int stages) {
  cudaError_t e = cudaSuccess;
  // Key-norm and row-bound passes (bsa_prep.cu).
  e = launch_prep(p, D, stages, stream);
  if (e != cudaSuccess) return e;
  // Plans with 64-row q-tiles run the kernels of bsa_forward_q64.cu (plain
  // path only; the host rejects pages and element masks for them).
  const bool q64 = p.qu * p.rq == 64;
  if (stages & BSA_STAGE_BOUNDED) {
    FwdParams a = p;
    a.work_counter = p.control + kCtlWorkCounter;
    a.work_count = nullptr;
    e = q64 ? launch_forward_q64(a, D, grid, stream, false)
            : launch_d<D, false>(a, grid, stream);
    if (e != cudaSuccess) return e;
  }
  if (stages & BSA_STAGE_EXACT) {
    // Exact pass over the queued rows (exits at once when none was queued).
    FwdParams x = p;
    x.order = p.fb_list;
    x.work_counter = p.control + kCtlFallbackWork;
    x.work_count = p.control + kCtlFallbackCount;
    e = q64 ? launch_forward_q64(x, D, grid, stream, true)
            : launch_d<D, true>(x, grid, stream);
  }
  return e;
}

}  // namespace

int forward_smem_bytes(int d) { return d == 64 ? Cfg<64>::kSmemBytes : Cfg<128>::kSmemBytes; }

cudaError_t launch_forward(const FwdParams& p, int d, int grid, cudaStream_t stream, int stages) {
  if (d == 64) return launch_passes<64>(p, grid, stream, stages);
  return launch_passes<128>(p, grid, stream, stages);
}

cudaError_t launch_watchdog_selftest(int32_t* status, long long limit_ns, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace bsa
