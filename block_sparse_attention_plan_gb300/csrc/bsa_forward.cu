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
//   warps 0, 2  TMA producers, one per softmax group: each loads the K and V
//               tiles of its group's slots into its own ring of shared-memory
//               stages guarded by full/empty mbarriers; warp 0 also takes the
//               work items and loads each row's Q tile.  A slot of 128 keys is
//               gathered as rk boxes of ku rows (ku = 128 / rk).
//   warps 1, 3  MMA issuers (one thread each, one per softmax group):
//               tcgen05.mma S = Q K^T and O += P V, all operands in shared
//               memory, accumulators in tensor memory.
//   warp 2      also owns the tensor-memory allocation (512 columns).
//   warps 4-7   softmax warpgroup A: even slots of the row.
//   warps 8-11  softmax warpgroup B: odd slots of the row.
// Each warpgroup keeps its own running max/sum and its own O accumulator, so
// the tensor pipe works on one group's tile while the other group runs its
// softmax; the two partial results are merged in the epilogue.
//
// Tensor memory (512 fp32 columns x 128 lanes; lane = q-tile row):
//   [0,128) S_A   [128,256) S_B   [256,256+d) O_A   [384,384+d) O_B
// P (bf16) goes through shared memory, one 32 KB buffer per softmax group, so
// a group's S buffer is free as soon as its softmax has read it: the MMA
// thread computes the next S while the softmax is still computing P.
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
__device__ __forceinline__ uint32_t col_s(int w) { return (uint32_t)(w * 128); }
__device__ __forceinline__ uint32_t col_o(int w) { return (uint32_t)(256 + w * 128); }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past 2^8 growth
// Work items (positions in the longest-row-first order) are taken from a
// global atomic counter by the producer and handed to the other roles through
// a small ring in shared memory.
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 2 + 8;  // ring-B producer, two MMA threads, one lane per softmax warp

template <int D>
struct Cfg {
  static constexpr int kTileBytes = 128 * D * 2;   // 128 rows x d bf16
  static constexpr int kChunks = D / 64;           // 64-column (128-byte) swizzle blocks
  static constexpr int kChunkBytes = 128 * 128;    // one block of 128 rows
  static constexpr int kPBytes = 128 * 128 * 2;    // P: 128 rows x 128 keys bf16
  // One K/V ring per softmax group (group A takes the even slots of a row,
  // group B the odd ones); each ring is consumed in order by one MMA thread.
  static constexpr int kStagesA = (D == 128) ? 2 : 4;
  static constexpr int kStagesB = (D == 128) ? 2 : 4;
  static constexpr int kQBufs = (D == 128) ? 1 : 2;  // Q tile buffers
  static constexpr int kOffQ = 0;
  static constexpr int kOffP = kQBufs * kTileBytes;           // P of group A, then B
  static constexpr int kOffRingA = kOffP + 2 * kPBytes;
  static constexpr int kOffRingB = kOffRingA + kStagesA * kTileBytes;
  static constexpr int kOffBar = kOffRingB + kStagesB * kTileBytes;
  // barriers
  static constexpr int kBarQFull = 0, kBarQEmpty = 2;
  static constexpr int kBarKvFullA = 4;
  static constexpr int kBarKvEmptyA = kBarKvFullA + kStagesA;
  static constexpr int kBarKvFullB = kBarKvEmptyA + kStagesA;
  static constexpr int kBarKvEmptyB = kBarKvFullB + kStagesB;
  static constexpr int kBarSFull = kBarKvEmptyB + kStagesB;
  static constexpr int kBarSFree = kBarSFull + 2;
  static constexpr int kBarPFull = kBarSFree + 2;
  static constexpr int kBarPFree = kBarPFull + 2;
  static constexpr int kBarODone = kBarPFree + 2;
  static constexpr int kBarXchg = kBarODone + 2;
  static constexpr int kBarDrain = kBarXchg + 2;
  static constexpr int kBarSchedFull = kBarDrain + 1;
  static constexpr int kBarSchedEmpty = kBarSchedFull + kSchedSlots;
  static constexpr int kNumBars = kBarSchedEmpty + kSchedSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kOffSched = kOffMisc + 16;          // int [kSchedSlots] work items
  static constexpr int kOffML = kOffSched + 4 * kSchedSlots;  // float [4][128]: mA, mB, lA, lB
  static constexpr int kSmemBytes = kOffML + 4 * 128 * 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  __host__ __device__ static constexpr int stages(int w) { return w ? kStagesB : kStagesA; }
  __host__ __device__ static constexpr int bar_full(int w) { return w ? kBarKvFullB : kBarKvFullA; }
  __host__ __device__ static constexpr int bar_empty(int w) { return w ? kBarKvEmptyB : kBarKvEmptyA; }
  __host__ __device__ static constexpr int ring(int w) { return w ? kOffRingB : kOffRingA; }
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
};

__device__ __forceinline__ void record_status(int32_t* ctl, int code, int site) {
  if (atomicCAS(ctl + kCtlStatus, 0, code) == 0)
    atomicExch(ctl + kCtlDetail, (int)((blockIdx.x << 8) | (site & 0xff)));
}

// Decode one schedule entry, rejecting out-of-range plan data (the row is then
// treated as empty and BSA_ERR_PLAN_MISMATCH is recorded).
__device__ __forceinline__ Item load_item(const FwdParams& p, int it, bool report) {
  Item m{0, 0, 0, 0, 0};
  const int row = __ldg(p.order + it);
  if (row < 0 || row >= p.rows) {
    if (report) record_status(p.control, -7, kSitePlanRange);
    return m;
  }
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
  __device__ __forceinline__ uint32_t pbuf(int w) const { return base + C::kOffP + w * C::kPBytes; }
  __device__ __forceinline__ uint32_t stage(int w, int s) const {
    return base + C::ring(w) + (uint32_t)s * C::kTileBytes;
  }
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

// ------------------------------------------------------------------ producer
// K/V units of one slot as the plan lists them (rk <= 4 entries, -1 = padding).
// The producer reads them a slot ahead, so the global-load latency overlaps
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

template <int D>
__device__ __forceinline__ bool load_kv_tile(const FwdParams& p, const Smem<D>& sm,
                                             const CUtensorMap* map, const Item& m, int j,
                                             const SlotKeys& keys, uint32_t (&kv_it)[2],
                                             uint64_t pol, const Watchdog& wd) {
  using C = Cfg<D>;
  const int w = j & 1;  // ring of the softmax group that owns slot j
  const int nst = C::stages(w);
  const int stage = (int)(kv_it[w] % nst);
  const uint32_t ph = (kv_it[w] / nst) & 1u;
  if (!mbar_wait(sm.bar(C::bar_empty(w) + stage), ph ^ 1u, wd, kSiteKvEmpty)) return false;
  const uint32_t full = sm.bar(C::bar_full(w) + stage);
  mbar_arrive_expect_tx(full, C::kTileBytes);
  int first = keys.y[0];
  if (first < 0 || first >= p.NKU) {
    record_status(p.control, -7, kSitePlanRange + 2);
    first = 0;
  }
  const uint32_t dst0 = sm.stage(w, stage);
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
  ++kv_it[w];
  return true;
}

// Producer of ring w.  The ring-A producer (w = 0) also takes work items from
// the global counter, publishes them, and loads each row's Q tile; the ring-B
// producer (w = 1) reads the published items.  Each loads, in consumption
// order, the K and V tiles of its group's slots j = w, w+2, ...
template <int D>
__device__ __noinline__ void producer_role(const FwdParams& p, uint8_t* smem, const Smem<D> sm,
                                           const Watchdog wd, int w) {
  using C = Cfg<D>;
  if (w == 0) tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();
  uint32_t q_it = 0, kv_it[2] = {0u, 0u};
  bool ok = true;
  volatile int* sched = reinterpret_cast<volatile int*>(smem + C::kOffSched);
  for (uint32_t t = 0; ok; ++t) {
    int it;
    if (w == 0) {
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
    const Item m = load_item(p, it, w == 0);
    if (m.n == 0) continue;
    if (w == 0) {
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
    // Ring w in consumption order: K_w, then K_{j+2}, V_j for j = w, w+2, ...
    // (the MMA thread computes S of slot j+2 while slot j's softmax runs).
    // V_j reuses the units read for K_j; slot j+4's are read before the waits
    // of K_{j+2} and V_j.
    if (w >= m.n) continue;
    SlotKeys kc = fetch_keys(p, m, w), kn = kc;
    if (w + 2 < m.n) kn = fetch_keys(p, m, w + 2);
    ok = load_kv_tile<D>(p, sm, &p.tmK, m, w, kc, kv_it, pol_kv, wd);
    for (int j = w; j < m.n && ok; j += 2) {
      SlotKeys kn2 = kn;
      if (j + 4 < m.n) kn2 = fetch_keys(p, m, j + 4);
      if (j + 2 < m.n) ok = load_kv_tile<D>(p, sm, &p.tmK, m, j + 2, kn, kv_it, pol_kv, wd);
      if (ok) ok = load_kv_tile<D>(p, sm, &p.tmV, m, j, kc, kv_it, pol_kv, wd);
      kc = kn;
      kn = kn2;
    }
  }
  if (*wd.abort_flag) {
    // Let copies already issued land before the CTA's shared memory goes away.
    const uint32_t nst = (uint32_t)C::stages(w);
    const uint32_t nk = kv_it[w] < nst ? kv_it[w] : nst;
    for (uint32_t t = kv_it[w] - nk; t < kv_it[w]; ++t)
      drain_wait(sm.bar(C::bar_full(w) + (int)(t % nst)), (t / nst) & 1u, wd);
    if (w == 0) {
      const uint32_t nq = q_it < (uint32_t)C::kQBufs ? q_it : (uint32_t)C::kQBufs;
      for (uint32_t t = q_it - nq; t < q_it; ++t)
        drain_wait(sm.bar(C::kBarQFull + q_buf<D>(t)), q_par<D>(t), wd);
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
// Descriptors are built once; per instruction only a compile-time offset is
// added (the start-address field is the low 14 bits of the descriptor and
// shared-memory offsets here never carry out of it), so each tcgen05.mma costs
// the issuing thread a couple of instructions.
template <int D>
struct MmaDesc {
  using C = Cfg<D>;
  uint64_t q[2];   // K-major SW128 descriptor of each Q buffer
  uint64_t kv0;    // K-major SW128 descriptor of stage 0 of this thread's ring (K tiles)
  uint64_t v0;     // MN-major SW128 descriptor of the same stage (V tiles)
  static constexpr uint64_t kStageStep = (uint64_t)(C::kTileBytes >> 4);
};

// S_w = Q K^T: M=128, N=128, K=16 per instruction, d/16 instructions.
template <int D>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc) {
  using C = Cfg<D>;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4);
    mma_ss(d_tmem, adesc + off, bdesc + off, kIdescS, kk > 0 ? 1u : 0u);
  }
}

// O_w (+)= P_w V: M=128, N=d, K=16 keys per instruction, 8 instructions.
// P (shared memory, K-major 128B swizzle like Q) advances like Q does in
// mma_qk; V rows [16kk, 16kk+16) start 2048 bytes apart (MN-major: LBO = next
// 64 columns).
template <int D>
__device__ __forceinline__ void mma_pv(uint32_t o_tmem, uint64_t pdesc, uint64_t vdesc,
                                       uint32_t acc) {
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * (128 * 128) + (kk % 4) * 32) >> 4);
    mma_ss(o_tmem, pdesc + off, vdesc + (uint64_t)(kk * (2048 >> 4)), kIdescPV,
           (acc || kk > 0) ? 1u : 0u);
  }
}

// State of one MMA issuer (softmax group w).
template <int D>
struct MmaState {
  MmaDesc<D> ds;
  uint64_t pdesc;    // K-major SW128 descriptor of this group's P buffer
  uint32_t kv = 0;   // tiles consumed from ring w
  uint32_t ns = 0;   // S tiles issued (the n-th waits for s_free completion n-1)
  uint32_t pc = 0;   // P tiles consumed
};

// S_w = Q K^T into this group's S buffer, once the softmax has read the
// previous S out of it.
template <int D>
__device__ __forceinline__ bool issue_s(const Smem<D>& sm, MmaState<D>& st, uint32_t tmem, int qb,
                                        int w, const Watchdog& wd) {
  using C = Cfg<D>;
  if (st.ns > 0 &&
      !mbar_wait(sm.bar(C::kBarSFree + w), (st.ns - 1) & 1u, wd, kSiteSFull))
    return false;
  const int stage = (int)(st.kv % C::stages(w));
  if (!mbar_wait(sm.bar(C::bar_full(w) + stage), (st.kv / C::stages(w)) & 1u, wd, kSiteKvFull))
    return false;
  tc_fence_after();
  mma_qk<D>(tmem + col_s(w), st.ds.q[qb], st.ds.kv0 + (uint64_t)stage * MmaDesc<D>::kStageStep);
  mma_commit(sm.bar(C::bar_empty(w) + stage));
  mma_commit(sm.bar(C::kBarSFull + w));
  ++st.kv;
  ++st.ns;
  return true;
}

// MMA issuer of softmax group w (slots j = w, w+2, ... of each row), fed by
// ring w.  Two of these run in separate warps: tcgen05.mma issue is close to
// synchronous with execution, so while one thread is held issuing, the other
// does its barrier waits and has its next group of MMAs ready.  Within a
// group, S of slot j+2 is issued before P V of slot j, so it runs while slot
// j's softmax is still computing P.
template <int D>
__device__ __noinline__ void mma_role(const FwdParams& p, const uint8_t* smem, const Smem<D> sm,
                                      uint32_t tmem, const Watchdog wd, int w) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.ds.q[0] = smem_desc_sw128(sm.q(0), 16, 1024);
  st.ds.q[1] = smem_desc_sw128(sm.q(C::kQBufs - 1), 16, 1024);
  st.ds.kv0 = smem_desc_sw128(sm.stage(w, 0), 16, 1024);
  st.ds.v0 = smem_desc_sw128(sm.stage(w, 0), C::kChunkBytes, 1024);
  st.pdesc = smem_desc_sw128(sm.pbuf(w), 16, 1024);
  uint32_t q_it = 0;
  bool ok = true;
  for (uint32_t t = 0; ok; ++t) {
    const int it = sched_take<D>(sm, smem, t, true, false, wd);
    if (it < 0) break;
    const Item m = load_item(p, it, false);
    const int n = m.n;
    if (n == 0) continue;
    const int qb = q_buf<D>(q_it);
    const uint32_t q_empty = sm.bar(C::kBarQEmpty + qb);
    // Every MMA thread waits for the row's Q before releasing it, so neither
    // can arrive on q_empty twice within one phase.
    if (!mbar_wait(sm.bar(C::kBarQFull + qb), q_par<D>(q_it), wd, kSiteQFull)) break;
    tc_fence_after();
    if (w >= n) {
      mbar_arrive(q_empty);  // this group has no slot in the row
    } else {
      ok = issue_s<D>(sm, st, tmem, qb, w, wd);
      if (ok && w + 2 >= n) mma_commit(q_empty);
      for (int j = w; j < n && ok; j += 2) {
        if (j + 2 < n) {
          ok = issue_s<D>(sm, st, tmem, qb, w, wd);
          if (ok && j + 4 >= n) mma_commit(q_empty);
          if (!ok) break;
        }
        if (!mbar_wait(sm.bar(C::kBarPFull + w), st.pc & 1u, wd, kSitePFull)) {
          ok = false;
          break;
        }
        ++st.pc;
        tc_fence_after();
        const int stage = (int)(st.kv % C::stages(w));
        if (!mbar_wait(sm.bar(C::bar_full(w) + stage), (st.kv / C::stages(w)) & 1u, wd,
                       kSiteKvFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_pv<D>(tmem + col_o(w), st.pdesc, st.ds.v0 + (uint64_t)stage * MmaDesc<D>::kStageStep,
                  j >= 2 ? 1u : 0u);
        mma_commit(sm.bar(C::bar_empty(w) + stage));
        mma_commit(sm.bar(C::kBarPFree + w));
        ++st.kv;
        if (j + 2 >= n) mma_commit(sm.bar(C::kBarODone + w));
      }
    }
    ++q_it;
  }
  // Drain: every MMA this thread issued has completed once its commit arrives.
  mma_commit(sm.bar(C::kBarDrain));
  drain_wait(sm.bar(C::kBarDrain), 0, wd);
}

// ------------------------------------------------------------------ softmax
template <int D>
__device__ __forceinline__ void softmax_role(const FwdParams& p, uint8_t* smem, const Smem<D>& sm,
                                             uint32_t tmem, const Watchdog& wd) {
  using C = Cfg<D>;
  float* ml = reinterpret_cast<float*>(smem + C::kOffML);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int w = (warp - 4) >> 2;          // 0 = group A (even slots), 1 = group B (odd slots)
  const int quad = warp & 3;              // TMEM lane quadrant of this warp
  const int rloc = quad * 32 + lane;      // row within the q-tile
  const uint32_t tl = (uint32_t)(quad * 32) << 16;
  const uint32_t s_addr = tmem + tl + col_s(w);
  const int qi = rloc / p.qu;
  const bool submask = (p.rq * p.rk) > 1;
  const int ku_shift = p.ku == 32 ? 0 : (p.ku == 64 ? 1 : 2);  // log2(ku / 32)
  const uint32_t my_bits_mask = (1u << p.rk) - 1u;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_make(sl2, sl2);
  uint32_t bits = 0xffffffffu;  // this row's sub-mask bits for the current slot
  // S row of the current slot -> registers (masked columns -> -inf).
  auto load_s = [&](uint32_t (&v)[128]) {
    tmem_ld32_at<0>(s_addr + 0, v);
    tmem_ld32_at<32>(s_addr + 32, v);
    tmem_ld32_at<64>(s_addr + 64, v);
    tmem_ld32_at<96>(s_addr + 96, v);
    tmem_wait_ld();
    if (submask) {
      // 32-column chunk c lies in k-unit c >> ku_shift; a warp's rows share
      // one q-unit, so the branch is warp-uniform.
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (!((bits >> (c >> ku_shift)) & 1u)) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[c * 32 + e] = __float_as_uint(-INFINITY);
        }
      }
    }
  };
  // p = 2^(s*scale*log2e - m), packed in place as bf16 pairs into v[0..64);
  // returns the row sum of p; with `mx` also returns the max of the raw row.
  auto exp_pack = [&](uint32_t (&v)[128], float m, float* mx) -> float {
    const float mb = (m == -INFINITY) ? 0.f : m;
    const uint64_t nmbx2 = f2_make(-mb, -mb);
    uint64_t acc2[2] = {0ull, 0ull};
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int e = 0; e < 64; ++e) {
      const float a0 = __uint_as_float(v[2 * e]), a1 = __uint_as_float(v[2 * e + 1]);
      if (mx) mx4[e & 3] = fmax3(mx4[e & 3], a0, a1);
      float x0, x1;
      f2_split(ffma2(f2_make(a0, a1), sl2x2, nmbx2), x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      acc2[e & 1] = fadd2(acc2[e & 1], f2_make(p0, p1));
      v[e] = pack_bf16x2(p0, p1);
    }
    if (mx) *mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    float s0, s1, s2, s3;
    f2_split(acc2[0], s0, s1);
    f2_split(acc2[1], s2, s3);
    return (s0 + s1) + (s2 + s3);
  };
  uint32_t sc = 0, oc = 0, xc = 0, np = 0;
  const uint32_t p_row = sm.pbuf(w) + (uint32_t)rloc * 128;  // this row in P chunk 0
  for (uint32_t t = 0;; ++t) {
    const int it = sched_take<D>(sm, smem, t, lane == 0, true, wd);
    if (it < 0) break;
    const Item m = load_item(p, it, false);
    const int nw = (w == 0) ? (m.n + 1) >> 1 : m.n >> 1;
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int k = 0; k < nw; ++k) {
      const int slot = m.s0 + 2 * k + w;
      if (submask) bits = (__ldg(p.slot_mask + slot) >> (qi * p.rk)) & my_bits_mask;
      if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarSFull + w), sc & 1u, wd, kSiteSFull))) {
        ok = false;
        break;
      }
      ++sc;
      tc_fence_after();
      uint32_t v[128];
      load_s(v);
      // The S row is in registers: hand the S buffer back for the next S MMA.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(C::kBarSFree + w));
      // Row max, then exponentials against the reference max.
      float mx4[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) mx4[c] = fmaxf(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
#pragma unroll
      for (int e = 8; e < 128; e += 8) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          mx4[c] = fmax3(mx4[c], __uint_as_float(v[e + 2 * c]), __uint_as_float(v[e + 2 * c + 1]));
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_new = fmaxf(m_ref, mx * sl2);
      float factor = 1.f;
      if (m_ref == -INFINITY) {
        m_ref = m_new;  // nothing weighted accumulated yet: O holds zeros
      } else if (m_new > m_ref + kRescaleThreshold) {
        factor = ex2_approx(m_ref - m_new);
        m_ref = m_new;
      }
      const float sum = exp_pack(v, m_ref, nullptr);
      // The previous P V of this group must be done with the P buffer (and
      // with O) before P is overwritten or O rescaled.
      if (np > 0 && !__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarPFree + w), (np - 1) & 1u, wd,
                                                       kSitePFull))) {
        ok = false;
        break;
      }
      ++np;
      // P -> shared memory in the K-major 128B-swizzled layout the MMA reads:
      // row r, keys [64c + 8u, +8) at chunk c, 16-byte unit u ^ (r % 8).
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t addr = p_row + c * (128 * 128) + ((u ^ (rloc & 7)) << 4);
          st_shared_v4(addr, v[c * 32 + u * 4], v[c * 32 + u * 4 + 1], v[c * 32 + u * 4 + 2],
                       v[c * 32 + u * 4 + 3]);
        }
      }
      fence_proxy_async_smem();  // make the stores visible to the tensor core
      if (__any_sync(0xffffffffu, factor != 1.f)) {
        const uint32_t o_addr = tmem + tl + col_o(w);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st32(o_addr + c * 32, o);
        }
      }
      tmem_wait_st();
      l_run = l_run * factor + sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(C::kBarPFull + w));  // one arrival per warp
    }
    if (!ok) break;
    // ------------------------------------------------------------ epilogue
    if (nw > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarODone + w), oc & 1u, wd, kSiteODone)))
        break;
      ++oc;
    }
    ml[w * 128 + rloc] = m_ref;
    ml[(2 + w) * 128 + rloc] = l_run;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarXchg + 0));
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarXchg + 0), xc & 1u, wd, kSiteXchg))) break;
    tc_fence_after();
    const float mA = ml[rloc], mB = ml[128 + rloc];
    const float lA = ml[256 + rloc], lB = ml[384 + rloc];
    const int nA = (m.n + 1) >> 1, nB = m.n >> 1;
    const float M = fmaxf(mA, mB);
    const float fA = (lA > 0.f) ? ex2_approx(mA - M) : 0.f;
    const float fB = (nB > 0 && lB > 0.f) ? ex2_approx(mB - M) : 0.f;
    const float L = lA * fA + lB * fB;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    const size_t orow = (size_t)m.bh * p.Nq + (size_t)m.qt * 128 + rloc;
    uint4* optr = reinterpret_cast<uint4*>(p.O + orow * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {  // this group's half of the columns, 16 at a time
      const int col0 = w * (D / 2) + c * 16;
      uint32_t a[16], bb[16];
      if (nA > 0) tmem_ld16(tmem + tl + col_o(0) + col0, a);
      if (nB > 0) tmem_ld16(tmem + tl + col_o(1) + col0, bb);
      tmem_wait_ld();
      uint32_t pk[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float o0 = 0.f, o1 = 0.f;
        if (nA > 0) {
          o0 = __uint_as_float(a[2 * e]) * fA;
          o1 = __uint_as_float(a[2 * e + 1]) * fA;
        }
        if (nB > 0) {
          o0 = fmaf(__uint_as_float(bb[2 * e]), fB, o0);
          o1 = fmaf(__uint_as_float(bb[2 * e + 1]), fB, o1);
        }
        pk[e] = pack_bf16x2(o0 * inv, o1 * inv);
      }
      optr[col0 / 8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      optr[col0 / 8 + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    if (w == 0) p.LSE[orow] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(C::kBarXchg + 1));
    if (!__all_sync(0xffffffffu, mbar_wait(sm.bar(C::kBarXchg + 1), xc & 1u, wd, kSiteXchg))) break;
    ++xc;
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
      mbar_init(sm.bar(C::kBarQEmpty + i), 2);  // one arrival per MMA thread
      mbar_init(sm.bar(C::kBarSFull + i), 1);
      mbar_init(sm.bar(C::kBarSFree + i), 4);    // one arrival per softmax warp
      mbar_init(sm.bar(C::kBarPFull + i), 4);    // one arrival per softmax warp
      mbar_init(sm.bar(C::kBarPFree + i), 1);
      mbar_init(sm.bar(C::kBarODone + i), 1);
      mbar_init(sm.bar(C::kBarXchg + i), 8);     // one arrival per softmax warp of both groups
    }
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(sm.bar(C::kBarKvFullA + s), 1);
      mbar_init(sm.bar(C::kBarKvEmptyA + s), 1);
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(sm.bar(C::kBarKvFullB + s), 1);
      mbar_init(sm.bar(C::kBarKvEmptyB + s), 1);
    }
    mbar_init(sm.bar(C::kBarDrain), 2);
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
      if (warp == 0) producer_role<D>(p, smem, sm, wd, 0);
      else if (warp == 1) mma_role<D>(p, smem, sm, tmem, wd, 0);
      else if (warp == 2) producer_role<D>(p, smem, sm, wd, 1);
      else mma_role<D>(p, smem, sm, tmem, wd, 1);
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
