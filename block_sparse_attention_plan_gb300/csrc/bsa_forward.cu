// Block-sparse attention forward for sm_103a: a persistent, warp-specialised
// flash-style kernel that computes only the K/V tiles a plan lists.
//
// Source of the method: "Decoupling Logical Masks from GPU Execution for
// Dynamic Block-Sparse Attention" (Tessera), abstract -- compute only the
// blocks a logical mask selects, with tiles grouped per GPU task so that data
// movement overlaps computation.  Online softmax over tiles (running max and
// sum, rescaling the partial output) is the FlashAttention fusion the pages
// refer to ("Sol-Attn" summary: inline sparsification inside the online
// softmax).
//
// One CTA (384 threads) per SM, looping over plan rows (one 128-row q-tile of
// one head each) in longest-row-first order:
//   warp 0   (one thread) takes the work items, publishes them to the other
//            roles, loads each row's Q tile and the K tiles of its slots into
//            the K ring (shared-memory stages guarded by full/empty mbarriers);
//   warp 3   (one thread) loads the V tiles into the V ring.  A slot of 128
//            keys is gathered as rk boxes of ku rows (ku = 128 / rk);
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
//            64-127), which exchange their half-row maxima through shared
//            memory so both use one running max and one O accumulator.
//
// Tensor memory (512 x 32-bit columns x 128 lanes; lane = q-tile row):
//   [0,128) S buffer 0   [128,256) S buffer 1   [256,256+d) O
//   [384,448) P buffer 0 [448,512) P buffer 1   (P: bf16 pairs, keys 2c, 2c+1
//   in column c).  Slot g of the CTA uses S and P buffer g mod 2.
//
// Every wait is bounded (watchdog): on expiry the CTA records
// BSA_ERR_TIMEOUT in the plan's status word, lets its in-flight copies and
// MMAs land, frees tensor memory and exits.
#include <cstdint>
#include <cuda_bf16.h>

#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

using namespace dev;

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
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past 2^8 growth
// Work items (positions in the longest-row-first order) are taken from a
// global atomic counter by the K producer and handed to the other roles
// through a small ring in shared memory.
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 2 + 8;  // V producer, two MMA threads, one lane per softmax warp

template <int D>
struct Cfg {
  static constexpr int kTileBytes = 128 * D * 2;   // 128 rows x d bf16
  static constexpr int kChunks = D / 64;           // 64-column (128-byte) swizzle blocks
  static constexpr int kChunkBytes = 128 * 128;    // one block of 128 rows
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
  static constexpr int kOffSched = kOffMisc + 16;          // int [kSchedSlots] work items
  static constexpr int kOffX = kOffSched + 4 * kSchedSlots;  // float [2 parities][2 halves][128 rows]
  static constexpr int kSmemBytes = kOffX + 2 * 2 * 128 * 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Q buffer index and phase parity of the q_it-th non-empty row of a CTA.
template <int D>
__device__ __forceinline__ int q_buf(uint32_t q_it) { return (int)(q_it % Cfg<D>::kQBufs); }
template <int D>
__device__ __forceinline__ uint32_t q_par(uint32_t q_it) { return (q_it / Cfg<D>::kQBufs) & 1u; }

struct Item {
  int n;       // slots of the row (0 = empty or rejected)
  int s0;      // first slot index
  int bh;      // b*H + h
  int qt;      // q-tile
  int kvrow0;  // first K/V row of the head's sequence in the [B*Hkv*Nk, d] view
  bool valid;  // the schedule entry named a plan row
};

__device__ __forceinline__ void record_status(int32_t* ctl, int code, int site) {
  if (atomicCAS(ctl + kCtlStatus, 0, code) == 0)
    atomicExch(ctl + kCtlDetail, (int)((blockIdx.x << 8) | (site & 0xff)));
}

// Decode one schedule entry, rejecting out-of-range plan data (the row is then
// treated as empty and BSA_ERR_PLAN_MISMATCH is recorded).
__device__ __forceinline__ Item load_item(const FwdParams& p, int it, bool report) {
  Item m{0, 0, 0, 0, 0, false};
  const int row = __ldg(p.order + it);
  if (row < 0 || row >= p.rows) {
    if (report) record_status(p.control, -7, kSitePlanRange);
    return m;
  }
  m.valid = true;
  const int s0 = __ldg(p.row_ptr + row), s1 = __ldg(p.row_ptr + row + 1);
  m.bh = row / p.NQT;
  m.qt = row % p.NQT;
  if (s0 < 0 || s1 < s0 || (long long)s1 > p.slot_capacity) {
    if (report) record_status(p.control, -7, kSitePlanRange + 1);
    return m;
  }
  const int b = m.bh / p.H, h = m.bh % p.H;
  m.n = s1 - s0;
  m.s0 = s0;
  m.kvrow0 = (b * p.Hkv + h / p.g) * p.Nk;
  return m;
}

// Shared-memory views common to all roles.
template <int D>
struct Smem {
  using C = Cfg<D>;
  uint32_t base;
  __device__ __forceinline__ uint32_t bar(int i) const { return base + C::kOffBar + 8u * (uint32_t)i; }
  __device__ __forceinline__ uint32_t q(int qb) const { return base + C::kOffQ + qb * C::kTileBytes; }
  __device__ __forceinline__ uint32_t kst(int s) const { return base + C::kOffK + s * C::kTileBytes; }
  __device__ __forceinline__ uint32_t vst(int s) const { return base + C::kOffV + s * C::kTileBytes; }
};

// Consumer side of the work-item ring: wait for entry t, read it, release it.
// Returns the item (position in the schedule), -1 at the end, or -2 when the
// wait gave up.  `lane_arrives`: whether this thread releases the entry.
template <int D>
__device__ __forceinline__ int sched_take(const Smem<D>& sm, const uint8_t* smem, uint32_t t,
                                          bool lane_arrives, bool warp_sync, const Watchdog& wd) {
  using C = Cfg<D>;
  const int slot = (int)(t % kSchedSlots);
  bool ok = mbar_wait(sm.bar(C::kBarSchedFull + slot), (t / kSchedSlots) & 1u, wd, kSiteSched);
  if (warp_sync) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return -2;
  const int item = reinterpret_cast<const volatile int*>(smem + C::kOffSched)[slot];
  if (warp_sync) __syncwarp();
  if (lane_arrives) mbar_arrive(sm.bar(C::kBarSchedEmpty + slot));
  return item;
}

// Bounded wait used during teardown: ignores the abort flag, short limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  volatile int no_abort = 0;
  Watchdog quick{&no_abort, wd.status, wd.detail, 100000000ll};
  mbar_wait(bar, parity, quick, kSiteDrain);
}

// ------------------------------------------------------------------ producers
// K/V units of one slot as the plan lists them (rk <= 4 entries, -1 = padding).
// A producer reads them two slots ahead, so the global-load latency overlaps
// its stage waits instead of sitting between a stage freeing and its copy.
struct SlotKeys {
  int y[4];
};
__device__ __forceinline__ SlotKeys fetch_keys(const FwdParams& p, const Item& m, int j) {
  SlotKeys k;
  const int32_t* ent = p.slot_ku + (size_t)(m.s0 + j) * p.rk;
#pragma unroll
  for (int u = 0; u < 4; ++u) k.y[u] = (u < p.rk) ? __ldg(ent + u) : -1;
  return k;
}

// One ring of tile stages with a single producer and a single consumer.
struct Ring {
  uint32_t data;   // shared address of stage 0
  uint32_t full;   // barrier of stage 0 (stage s at +8 s)
  uint32_t empty;
  int stages;
};

// Gather the 128 keys of one slot into the next stage of `r`.
template <int D>
__device__ __forceinline__ bool load_tile(const FwdParams& p, const CUtensorMap* map, const Ring& r,
                                          const Item& m, const SlotKeys& keys, uint32_t& it,
                                          uint64_t pol, const Watchdog& wd) {
  using C = Cfg<D>;
  const uint32_t stage = it % (uint32_t)r.stages;
  const uint32_t ph = (it / (uint32_t)r.stages) & 1u;
  if (!mbar_wait(r.empty + 8u * stage, ph ^ 1u, wd, kSiteKvEmpty)) return false;
  const uint32_t full = r.full + 8u * stage;
  mbar_arrive_expect_tx(full, C::kTileBytes);
  int first = keys.y[0];
  if (first < 0 || first >= p.NKU) {
    record_status(p.control, -7, kSitePlanRange + 2);
    first = 0;
  }
  const uint32_t dst0 = r.data + stage * (uint32_t)C::kTileBytes;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (u >= p.rk) break;
    int y = keys.y[u];
    if (y < 0) {
      y = first;  // padding position: load real rows, the sub-mask hides them
    } else if (y >= p.NKU) {
      record_status(p.control, -7, kSitePlanRange + 3);
      y = first;
    }
    const int row = m.kvrow0 + y * p.ku;
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c)
      tma_load_2d(dst0 + c * C::kChunkBytes + u * p.ku * 128, map, c * 64, row, full, pol);
  }
  ++it;
  return true;
}

// K producer (kside): takes work items from the global counter, publishes
// them, loads each row's Q tile and the K tile of every slot.  V producer:
// reads the published items and loads the V tile of every slot.  Both load in
// slot order, which is the order the MMA thread consumes each ring in.
template <int D>
__device__ __noinline__ void producer_role(const FwdParams& p, uint8_t* smem, const Smem<D> sm,
                                           const Watchdog wd, bool kside) {
  using C = Cfg<D>;
  const CUtensorMap* map = kside ? &p.tmK : &p.tmV;
  if (kside) tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(map);
  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();
  const Ring r = kside ? Ring{sm.kst(0), sm.bar(C::kBarKFull), sm.bar(C::kBarKEmpty), C::kStagesK}
                       : Ring{sm.vst(0), sm.bar(C::kBarVFull), sm.bar(C::kBarVEmpty), C::kStagesV};
  uint32_t q_it = 0, kv_it = 0;
  bool ok = true;
  volatile int* sched = reinterpret_cast<volatile int*>(smem + C::kOffSched);
  for (uint32_t t = 0; ok; ++t) {
    int it;
    if (kside) {
      const int slot = (int)(t % kSchedSlots);
      if (!mbar_wait(sm.bar(C::kBarSchedEmpty + slot), ((t / kSchedSlots) & 1u) ^ 1u, wd,
                     kSiteSched))
        break;
      it = atomicAdd(p.control + kCtlWorkCounter, 1);
      if (it >= p.rows) it = -1;
      sched[slot] = it;
      mbar_arrive(sm.bar(C::kBarSchedFull + slot));
    } else {
      it = sched_take<D>(sm, smem, t, true, false, wd);
    }
    if (it < 0) break;
    const Item m = load_item(p, it, kside);
    if (m.n == 0) continue;
    if (kside) {
      const int qb = q_buf<D>(q_it);
      if (!mbar_wait(sm.bar(C::kBarQEmpty + qb), q_par<D>(q_it) ^ 1u, wd, kSiteQEmpty)) break;
      mbar_arrive_expect_tx(sm.bar(C::kBarQFull + qb), C::kTileBytes);
      const int qrow = m.bh * p.Nq + m.qt * 128;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_2d(sm.q(qb) + c * C::kChunkBytes, &p.tmQ, c * 64, qrow,
                    sm.bar(C::kBarQFull + qb), pol_q);
      ++q_it;
    }
    SlotKeys k0 = fetch_keys(p, m, 0), k1 = k0;
    if (m.n > 1) k1 = fetch_keys(p, m, 1);
    for (int j = 0; j < m.n && ok; ++j) {
      SlotKeys k2 = k1;
      if (j + 2 < m.n) k2 = fetch_keys(p, m, j + 2);
      ok = load_tile<D>(p, map, r, m, k0, kv_it, pol_kv, wd);
      k0 = k1;
      k1 = k2;
    }
  }
  if (*wd.abort_flag) {
    // Let copies already issued land before the CTA's shared memory goes away.
    const uint32_t nst = (uint32_t)r.stages;
    const uint32_t nk = kv_it < nst ? kv_it : nst;
    for (uint32_t t = kv_it - nk; t < kv_it; ++t)
      drain_wait(r.full + 8u * (t % nst), (t / nst) & 1u, wd);
    if (kside) {
      const uint32_t nq = q_it < (uint32_t)C::kQBufs ? q_it : (uint32_t)C::kQBufs;
      for (uint32_t t = q_it - nq; t < q_it; ++t)
        drain_wait(sm.bar(C::kBarQFull + q_buf<D>(t)), q_par<D>(t), wd);
    }
  }
}

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
// instructions), once the softmax has read that buffer's previous tile.
template <int D>
__device__ __forceinline__ bool issue_s(const Smem<D>& sm, MmaState<D>& st, uint32_t tmem, int qb,
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
// [16kk, 16kk+16) start 2048 bytes apart.
template <int D>
__device__ __forceinline__ void issue_pv(MmaState<D>& st, uint32_t tmem, uint32_t stage,
                                         bool accumulate) {
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);
  const uint32_t pcol = tmem + kColP + 64u * (st.pg & 1u);
  const uint64_t vd = st.vdesc0 + (uint64_t)stage * MmaState<D>::kStageStep;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(tmem + kColO, pcol + 8u * (uint32_t)kk, vd + (uint64_t)(kk * (2048 >> 4)), kIdescPV,
           (accumulate || kk > 0) ? 1u : 0u);
}

// S issuer: S of every slot, in slot order, as soon as its S buffer has been
// read out by the softmax (two slots back) and its K tile has landed.
template <int D>
__device__ __noinline__ void s_issuer_role(const FwdParams& p, const uint8_t* smem, const Smem<D> sm,
                                           uint32_t tmem, const Watchdog wd) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.qdesc[0] = smem_desc_sw128(sm.q(0), 16, 1024);
  st.qdesc[1] = smem_desc_sw128(sm.q(C::kQBufs - 1), 16, 1024);
  st.kdesc0 = smem_desc_sw128(sm.kst(0), 16, 1024);
  uint32_t q_it = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const int it = sched_take<D>(sm, smem, t, true, false, wd);
    if (it < 0) break;
    const Item m = load_item(p, it, false);
    if (m.n == 0) continue;
    const int qb = q_buf<D>(q_it);
    if (!mbar_wait(sm.bar(C::kBarQFull + qb), q_par<D>(q_it), wd, kSiteQFull)) break;
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
__device__ __noinline__ void pv_issuer_role(const FwdParams& p, const uint8_t* smem, const Smem<D> sm,
                                            uint32_t tmem, const Watchdog wd) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.vdesc0 = smem_desc_sw128(sm.vst(0), C::kChunkBytes, 1024);
  uint32_t rows = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const int it = sched_take<D>(sm, smem, t, true, false, wd);
    if (it < 0) break;
    const Item m = load_item(p, it, false);
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
      issue_pv<D>(st, tmem, stage, j > 0);
      mma_commit(sm.bar(C::kBarVEmpty + (int)stage));
      mma_commit(sm.bar(C::kBarPFree + b));
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
template <int D>
__device__ __forceinline__ void softmax_role(const FwdParams& p, uint8_t* smem, const Smem<D>& sm,
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
  uint32_t sg = 0, rows = 0, xc = 0;
  uint32_t bits = 0xffffffffu;  // this row's sub-mask bits for the current slot

  // One float per row with the thread of the other key half that owns the
  // same row (warp quad + 4 <-> quad + 8); double-buffered by round parity.
  auto exchange = [&](float mine, float& theirs) -> bool {
    const int par = (int)(xc & 1u);
    xbuf[(par * 2 + h) * 128 + rloc] = mine;
    __syncwarp();
    const uint32_t bar = sm.bar(C::kBarXchg + quad * 2 + par);
    if (lane == 0) mbar_arrive(bar);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, (xc >> 1) & 1u, wd, kSiteXchg));
    if (ok) theirs = xbuf[(par * 2 + (h ^ 1)) * 128 + rloc];
    ++xc;
    return ok;
  };
  // This thread's 64 scores of the slot in S buffer `sbuf` (masked -> -inf).
  auto load_s = [&](uint32_t sbuf, uint32_t (&v)[64]) {
    tmem_ld32_at<0>(sbuf + 64u * (uint32_t)h, v);
    tmem_ld32_at<32>(sbuf + 64u * (uint32_t)h + 32u, v);
    tmem_wait_ld();
    if (submask) {
      // 32-key chunk 2h + c lies in k-unit (2h + c) >> ku_shift; a warp's rows
      // share one q-unit, so the branch is warp-uniform.
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!((bits >> ((2 * h + c) >> ku_shift)) & 1u)) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[c * 32 + e] = __float_as_uint(-INFINITY);
        }
      }
    }
  };
  // p = 2^(s*scale*log2e - m), packed in place as bf16 pairs into v[0..32);
  // returns the sum of the 64 values of p.
  auto exp_pack = [&](uint32_t (&v)[64], float m) -> float {
    const float mb = (m == -INFINITY) ? 0.f : m;
    const uint64_t nmbx2 = f2_make(-mb, -mb);
    uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float x0, x1;
      f2_split(ffma2(f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2x2, nmbx2),
               x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      acc2[e & 1] = fadd2(acc2[e & 1], f2_make(p0, p1));
      v[e] = pack_bf16x2(p0, p1);
    }
    float s0, s1, s2, s3;
    f2_split(acc2[0], s0, s1);
    f2_split(acc2[1], s2, s3);
    return (s0 + s1) + (s2 + s3);
  };

  for (uint32_t t = 0;; ++t) {
    const int it = sched_take<D>(sm, smem, t, lane == 0, true, wd);
    if (it < 0) break;
    const Item m = load_item(p, it, false);
    if (!m.valid) continue;
    const size_t orow = (size_t)m.bh * p.Nq + (size_t)m.qt * 128 + rloc;
    uint4* optr = reinterpret_cast<uint4*>(p.O + orow * D + h * (D / 2));
    if (m.n == 0) {  // no selected key: O = 0, LSE = -inf
#pragma unroll
      for (int c = 0; c < D / 16; ++c) optr[c] = make_uint4(0u, 0u, 0u, 0u);
      if (h == 0) p.LSE[orow] = -INFINITY;
      continue;
    }
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < m.n; ++j) {
      const int b = (int)(sg & 1u);
      const uint32_t u = sg >> 1;
      if (submask) bits = (__ldg(p.slot_mask + m.s0 + j) >> (qi * p.rk)) & my_bits_mask;
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
      // Max of this half-row, then of the whole row with the partner's half.
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
      mx = fmaxf(mx, mo);
      // Both threads of a row see the same maximum, so they keep the same
      // reference and take the same rescale decisions.
      const float m_new = fmaxf(m_ref, mx * sl2);
      float factor = 1.f;
      if (m_ref == -INFINITY) {
        m_ref = m_new;  // nothing weighted accumulated yet
      } else if (m_new > m_ref + kRescaleThreshold) {
        factor = ex2_approx(m_ref - m_new);
        m_ref = m_new;
      }
      const float sum = exp_pack(v, m_ref);
      // P buffer b was last read by the P V of slot g - 2.
      if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + b), (u - 1) & 1u, wd, kSitePFull))) {
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, factor != 1.f)) {
        // O changes scale: the P V of slot g - 1 must have finished with it
        // (the one of slot g starts only after this slot's P is published).
        const uint32_t g1 = sg - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + (int)(g1 & 1u)), (g1 >> 1) & 1u, wd, kSitePFull))) {
          ok = false;
          break;
        }
        tc_fence_after();
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
      tmem_st32_at<0>(tmem + tl + kColP + 64u * (uint32_t)b + 32u * (uint32_t)h, v);
      tmem_wait_st();
      l_run = l_run * factor + sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(C::kBarPFull + b));  // one arrival per warp
      ++sg;
    }
    if (!ok) break;
    // ------------------------------------------------------------ epilogue
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarOFull), rows & 1u, wd, kSiteODone))) break;
    tc_fence_after();
    float l_other = 0.f;
    if (!exchange(l_run, l_other)) break;
    const float L = l_run + l_other;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
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
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        optr[c * 4 + q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
    }
    // O has been read: the next row's first P V may overwrite it.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarOFree));
    if (h == 0) p.LSE[orow] = (L > 0.f) ? (m_ref + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    ++rows;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bsa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Smem<D> sm{smem_u32(smem)};
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Watchdog wd{abort_flag, p.control + kCtlStatus, p.control + kCtlDetail, p.watchdog_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    if (sm.base & 1023u) record_failure(wd, -4, 0);  // layout assumption violated
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.bar(C::kBarQFull + i), 1);
      mbar_init(sm.bar(C::kBarQEmpty + i), 1);
      mbar_init(sm.bar(C::kBarSFull + i), 1);
      mbar_init(sm.bar(C::kBarSFree + i), 8);  // one arrival per softmax warp
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
    softmax_role<D>(p, smem, sm, tmem, wd);
  } else {
    regs_dec<kRegsControl>();
    if (lane == 0 && !*abort_flag) {
      if (warp == 0) producer_role<D>(p, smem, sm, wd, true);
      else if (warp == 1) s_issuer_role<D>(p, smem, sm, tmem, wd);
      else if (warp == 2) pv_issuer_role<D>(p, smem, sm, tmem, wd);
      else if (warp == 3) producer_role<D>(p, smem, sm, wd, false);
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

template <int D>
cudaError_t launch_d(const FwdParams& p, int grid, cudaStream_t stream) {
  const int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(bsa_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bsa_fwd_kernel<D><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int forward_smem_bytes(int d) { return d == 64 ? Cfg<64>::kSmemBytes : Cfg<128>::kSmemBytes; }

cudaError_t launch_forward(const FwdParams& p, int d, int grid, cudaStream_t stream) {
  if (d == 64) return launch_d<64>(p, grid, stream);
  return launch_d<128>(p, grid, stream);
}

cudaError_t launch_watchdog_selftest(int32_t* status, long long limit_ns, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace bsa
