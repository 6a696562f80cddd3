// Device-side pieces shared by the forward kernels (128-row and 64-row
// q-tiles): the work items and the shared-memory ring that hands them from
// the K producer to the other roles, and the two TMA producer roles that
// gather a row's Q tile and the K/V tiles its plan lists into mbarrier
// rings.  Each kernel supplies a configuration type C with its shared-memory
// layout and barrier indices:
//   kQBytes, kQChunkBytes, kQBufs           Q tile bytes / 64-column chunk bytes / buffers
//   kTileBytes, kChunks, kChunkBytes        K/V tile (128 keys) bytes, chunks, chunk bytes
//   kStagesK, kStagesV                      ring depths
//   kKSweeps                                K tiles loaded per slot (sweeps over a row)
//   kQueueSplit                             leave rows needing split weights to the exact pass
//   kOffQ, kOffK, kOffV, kOffBar, kOffSched and the kBar* barrier indices.
#pragma once

#include <cstdint>

#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

using namespace dev;

// Work items (positions in the plan's schedule: K/V-head groups heaviest
// first, rows longest first inside a group) are taken from a global atomic
// counter by the K producer and handed to the other roles through a small
// ring in shared memory.
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 2 + 8;  // V producer, two MMA threads, one lane per softmax warp
// Rows whose K/V units hold a value of magnitude above this apply split
// weights (hi + lo).  Values of N(0,1) inputs stay below it (their largest
// magnitude over millions of draws is about 5.5), where the error of bf16
// weights stays a few thousandths of the output scale.
constexpr float kSplitV = 8.0f;
// Bounded pass: weights below 2^-126 are flushed to zero, so a row of at most
// n keys whose weights sum to at least n * 2^-102 loses under 2^-24 of its
// total weight (fp32 precision); a row below that (while it has selected
// keys) is recomputed by the exact pass.
constexpr float kFallbackPerKey = 0x1p-102f;

// Q buffer index and phase parity of the q_it-th non-empty row of a CTA.
template <class C>
__device__ __forceinline__ int q_buf(uint32_t q_it) { return (int)(q_it % C::kQBufs); }
template <class C>
__device__ __forceinline__ uint32_t q_par(uint32_t q_it) { return (q_it / C::kQBufs) & 1u; }

struct Item {
  int n;       // slots of the row (0 = empty or rejected)
  int s0;      // first slot index
  int bh;      // b*H + h
  int qx;      // first q-unit of the row's q-tile (its q-unit i is qx + i*qs)
  int qs;      // q-unit stride of the plane (1 unless the plan regrouped it)
  int kvrow0;  // first K/V row of the head's sequence in the [B*Hkv*Nk, d] view
  bool valid;  // the schedule entry named a plan row
  int row;     // plan row
  int it;      // schedule position; < 0: no more work (-2: a wait gave up)
  float kb;    // largest key norm over the row's K units
  bool split;  // apply the row's weights as hi + lo bf16 terms
};


__device__ __forceinline__ void record_status(int32_t* ctl, int code, int site) {
  if (atomicCAS(ctl + kCtlStatus, 0, code) == 0)
    atomicExch(ctl + kCtlDetail, (int)((blockIdx.x << 8) | (site & 0xff)));
}

// Decode one schedule entry, rejecting out-of-range plan data (the row is then
// treated as empty and BSA_ERR_PLAN_MISMATCH is recorded).
__device__ __forceinline__ Item load_item(const FwdParams& p, int it, bool report) {
  Item m{0, 0, 0, 0, 1, 0, false, 0, it, 0.f, false};
  const int row = __ldg(p.order + it);
  if (row < 0 || row >= p.rows) {
    if (report) record_status(p.control, -7, kSitePlanRange);
    return m;
  }
  m.valid = true;
  m.row = row;
  const int s0 = __ldg(p.row_ptr + row), s1 = __ldg(p.row_ptr + row + 1);
  m.bh = row / p.NQT;
  const int qt = row % p.NQT;
  m.qs = 1;
  m.qx = qt * p.rq;
  if (p.sigma != nullptr) {  // a plan built with regrouping
    int sig = __ldg(p.sigma + m.bh);
    if (!(sig == 1 || sig == 2 || sig == 4 || sig == 8 || sig == 16) || p.NQT % sig) {
      if (report) record_status(p.control, -7, kSitePlanRange + 5);
      sig = 1;
    }
    m.qs = sig;
    m.qx = (qt / sig) * sig * p.rq + qt % sig;
  }
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
template <class C>
struct Smem {
  uint32_t base;
  __device__ __forceinline__ uint32_t bar(int i) const { return base + C::kOffBar + 8u * (uint32_t)i; }
  __device__ __forceinline__ uint32_t q(int qb) const { return base + C::kOffQ + qb * C::kQBytes; }
  __device__ __forceinline__ uint32_t kst(int s) const { return base + C::kOffK + s * C::kTileBytes; }
  __device__ __forceinline__ uint32_t vst(int s) const { return base + C::kOffV + s * C::kTileBytes; }
};

// The work-item ring: the K producer decodes each schedule entry once (its
// global loads run ahead of everyone else) and publishes the whole item, 8
// words, so that no other role touches global memory at a row start.
template <class C>
__device__ __forceinline__ void sched_publish(uint8_t* smem, int slot, const Item& m) {
  volatile int* e = reinterpret_cast<volatile int*>(smem + C::kOffSched) + slot * 8;
  e[0] = m.it;
  e[1] = m.n;
  e[2] = m.s0;
  e[3] = m.bh;
  e[4] = (m.qx << 6) | (m.split ? 32 : 0) | m.qs;
  e[5] = m.kvrow0;
  e[6] = m.valid ? m.row : -1;
  e[7] = __float_as_int(m.kb);
}

// Consumer side: wait for entry t, read it, release it (`lane_arrives`: this
// thread releases the entry).  it = -2 when the wait gave up.
template <class C>
__device__ __forceinline__ Item sched_take(const Smem<C>& sm, const uint8_t* smem, uint32_t t,
                                           bool lane_arrives, bool warp_sync, const Watchdog& wd) {
  Item m{0, 0, 0, 0, 1, 0, false, 0, -2, 0.f, false};
  const int slot = (int)(t % kSchedSlots);
  bool ok = mbar_wait(sm.bar(C::kBarSchedFull + slot), (t / kSchedSlots) & 1u, wd, kSiteSched);
  if (warp_sync) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return m;
  const volatile int* e = reinterpret_cast<const volatile int*>(smem + C::kOffSched) + slot * 8;
  m.it = e[0];
  m.n = e[1];
  m.s0 = e[2];
  m.bh = e[3];
  m.qx = e[4] >> 6;
  m.split = (e[4] & 32) != 0;
  m.qs = e[4] & 31;
  m.kvrow0 = e[5];
  const int row = e[6];
  m.valid = row >= 0;
  m.row = m.valid ? row : 0;
  m.kb = __int_as_float(e[7]);
  if (warp_sync) __syncwarp();
  if (lane_arrives) mbar_arrive(sm.bar(C::kBarSchedEmpty + slot));
  return m;
}

// Bounded wait used during teardown: ignores the abort flag, short limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  volatile int no_abort = 0;
  Watchdog quick{&no_abort, wd.status, wd.detail, 100000000ll};
  mbar_wait(bar, parity, quick, kSiteDrain);
}

// ------------------------------------------------------------------ producers
// A TMA copy instruction does not return until the copy engine has taken it,
// about 300 cycles per box under load, so one thread issuing every box of a
// slot made small-block slots (2-4 units of 32 or 64 keys, a box per unit and
// 64-column half) wait for their K/V tiles.  For slots of several units
// (kWarp) the producers run on their whole warp and each lane issues one box
// (measured: chunked prefill +16 %, regular patterns +40 %, outputs
// bit-identical); control flow is then warp-uniform and lane 0
// alone takes the single-thread steps (work counter, publishing, barrier
// arrivals, byte counts).  Slots of one unit keep a single thread, which is
// 2 % faster there than the warp form.
constexpr unsigned kFullMask = 0xffffffffu;

// This lane's K/V unit of slot j of the row (lane u < rk: slot position u,
// -1 = padding, or for paged K/V its pool row as the row-bound pass
// resolved it; other lanes -1).  A producer reads it two slots ahead, so the
// global-load latency overlaps its stage waits instead of sitting between a
// stage freeing and its copy (a block-table lookup there, dependent on the
// plan entry, cost the paged path about 40 %).
template <bool kGeneral>
__device__ __forceinline__ int fetch_key(const FwdParams& p, const Item& m, int j, int lane) {
  const int32_t* ent = ((kGeneral && p.prow) ? p.prow : p.slot_ku) + (size_t)(m.s0 + j) * p.rk;
  return lane < p.rk ? __ldg(ent + lane) : -1;
}

// One ring of tile stages with a single producer and a single consumer.
struct Ring {
  uint32_t data;   // shared address of stage 0
  uint32_t full;   // barrier of stage 0 (stage s at +8 s)
  uint32_t empty;
  int stages;
};

// Gather the 128 keys of one slot into the next stage of `r` (called by the
// whole warp; `key` is the lane's unit from fetch_key).
// kBox3: slots of one 128-key unit at d = 128 through the 3D view (one box
// per unit), a compile-time choice so that each producer loop carries one
// form only (the 3D branch in the 2D producer's loop slowed it by 4.5 %).
template <class C, bool kGeneral, bool kBox3, bool kWarp>
__device__ __forceinline__ bool load_tile(const FwdParams& p, const CUtensorMap* map, const Ring& r,
                                          const Item& m, int key, int lane, uint32_t& it,
                                          uint64_t pol, const Watchdog& wd) {
  const uint32_t stage = it % (uint32_t)r.stages;
  const uint32_t ph = (it / (uint32_t)r.stages) & 1u;
  bool waited = mbar_wait(r.empty + 8u * stage, ph ^ 1u, wd, kSiteKvEmpty);
  if (kWarp) waited = __all_sync(kFullMask, waited);
  if (!waited) return false;
  const uint32_t full = r.full + 8u * stage;
  if (lane == 0) mbar_arrive_expect_tx(full, C::kTileBytes);
  if (kWarp) __syncwarp();
  const bool paged = kGeneral && p.prow != nullptr;  // keys are pool rows
  int first = kWarp ? __shfl_sync(kFullMask, key, 0) : key;
  if (first < 0 || (!paged && first >= p.NKU)) {
    if (lane == 0) record_status(p.control, -7, kSitePlanRange + 2);
    first = 0;
  }
  const uint32_t dst0 = r.data + stage * (uint32_t)C::kTileBytes;
  if constexpr (kBox3) {  // one 128-key unit: both halves in one box
    if (lane == 0) tma_load_3d(dst0, map, 0, paged ? first : m.kvrow0 + first * p.ku, 0, full, pol);
  } else {
    // Warp form: lane u * kChunks + c copies 64-column chunk c of unit u (one
    // box per lane); single thread: lane 0 copies every chunk of its unit.
    const int u = kWarp ? lane / C::kChunks : lane;
    int y = kWarp ? __shfl_sync(kFullMask, key, u) : key;
    if (u < p.rk) {
      if (y < 0) {
        y = first;  // padding position: load real rows, the sub-mask hides them
      } else if (!paged && y >= p.NKU) {
        record_status(p.control, -7, kSitePlanRange + 3);
        y = first;
      }
      const int row = paged ? y : m.kvrow0 + y * p.ku;
#pragma unroll
      for (int c = kWarp ? lane % C::kChunks : 0; c < C::kChunks; c += kWarp ? C::kChunks : 1)
        tma_load_2d(dst0 + c * C::kChunkBytes + u * p.ku * 128, map, c * 64, row, full, pol);
    }
  }
  ++it;
  return true;
}

// K producer (kside): takes work items from the global counter, publishes
// them, loads each row's Q tile and the K tile of every slot (of every sweep
// over the row's slots).  V producer:
// reads the published items and loads the V tile of every slot.  Both load in
// slot order, which is the order the MMA thread consumes each ring in.
// kWarp: run by the whole warp, else by lane 0 alone.
template <class C, bool kGeneral, bool kBox3, bool kWarp>
__device__ __noinline__ void producer_body(const FwdParams& p, uint8_t* smem, const Smem<C> sm,
                                           const Watchdog wd, bool kside) {
  static_assert(!(kBox3 && kWarp), "3D boxes carry one unit per slot");
  const int lane = kWarp ? (int)(threadIdx.x & 31) : 0;
  auto all = [](bool v) { return kWarp ? __all_sync(kFullMask, v) : v; };
  auto from0 = [](int v) { return kWarp ? __shfl_sync(kFullMask, v, 0) : v; };
  const CUtensorMap* map = kBox3 ? (kside ? &p.tmK3 : &p.tmV3) : (kside ? &p.tmK : &p.tmV);
  if (lane == 0) {
    if (kside) {
      tma_prefetch_desc((C::kChunks == 2 && p.q_box3) ? &p.tmQ3 : &p.tmQ);
      tma_prefetch_desc(&p.tmQu);
    }
    tma_prefetch_desc(map);
  }
  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();
  const Ring r = kside ? Ring{sm.kst(0), sm.bar(C::kBarKFull), sm.bar(C::kBarKEmpty), C::kStagesK}
                       : Ring{sm.vst(0), sm.bar(C::kBarVFull), sm.bar(C::kBarVEmpty), C::kStagesV};
  uint32_t q_it = 0, kv_it = 0;
  bool ok = true;
  const int nwork =
      p.work_count ? *reinterpret_cast<const volatile int32_t*>(p.work_count) : p.rows;
  for (uint32_t t = 0; ok; ++t) {
    Item m;
    if (kside) {
      const int slot = (int)(t % kSchedSlots);
      if (!all(mbar_wait(sm.bar(C::kBarSchedEmpty + slot), ((t / kSchedSlots) & 1u) ^ 1u, wd,
                         kSiteSched)))
        break;
      int it = 0;
      if (lane == 0) it = atomicAdd(p.work_counter, 1);
      it = from0(it);
      if (it >= nwork) it = -1;
      if (it >= 0) {
        m = load_item(p, it, lane == 0);  // the same loads on every lane
        if (m.n > 0) {
          m.kb = __ldg(p.rowk + m.row);
          m.split = p.split_all || __ldg(p.rowv + m.row) > kSplitV;
          if (C::kQueueSplit && m.split) {
            // This pass does not apply split weights: the row is left to
            // the exact pass (queued once) and handed on as skipped.
            if (lane == 0 && atomicExch(p.fb_flag + m.row, 1) == 0)
              p.fb_list[atomicAdd(p.control + kCtlFallbackCount, 1)] = m.row;
            m.n = 0;
            m.valid = false;
          }
        }
      } else {
        m = Item{0, 0, 0, 0, 1, 0, false, 0, -1, 0.f, false};
      }
      if (lane == 0) {
        sched_publish<C>(smem, slot, m);
        mbar_arrive(sm.bar(C::kBarSchedFull + slot));
      }
    } else {
      m = sched_take<C>(sm, smem, t, lane == 0, kWarp, wd);
    }
    if (m.it < 0) break;
    if (m.n == 0) continue;
    if (kside) {
      const int qb = q_buf<C>(q_it);
      if (!all(mbar_wait(sm.bar(C::kBarQEmpty + qb), q_par<C>(q_it) ^ 1u, wd, kSiteQEmpty))) break;
      if (lane == 0) mbar_arrive_expect_tx(sm.bar(C::kBarQFull + qb), C::kQBytes);
      if (kWarp) __syncwarp();
      if (m.qs == 1) {  // the tile's q-units are contiguous: one box of the tile's rows
        if (lane == 0) {
          const int qrow = m.bh * p.Nq + m.qx * p.qu;
          if (C::kChunks == 2 && p.q_box3) {
            tma_load_3d(sm.q(qb), &p.tmQ3, 0, qrow, 0, sm.bar(C::kBarQFull + qb), pol_q);
          } else {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_2d(sm.q(qb) + c * C::kQChunkBytes, &p.tmQ, c * 64, qrow,
                          sm.bar(C::kBarQFull + qb), pol_q);
          }
        }
      } else {
        // q-unit i (qu rows) into tile rows [i*qu, (i+1)*qu): lane i, or
        // every one by lane 0
        for (int i = lane; i < p.rq; i += kWarp ? 32 : 1) {
          const int qrow = m.bh * p.Nq + (m.qx + i * m.qs) * p.qu;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(sm.q(qb) + c * C::kQChunkBytes + i * p.qu * 128, &p.tmQu, c * 64, qrow,
                        sm.bar(C::kBarQFull + qb), pol_q);
        }
      }
      ++q_it;
    }
    // Tiles of this row in consumption order: the K tiles once per sweep of
    // the row's slots (C::kKSweeps), the V tiles once.
    const int nt = (kside ? C::kKSweeps : 1) * m.n;
    int k0 = fetch_key<kGeneral>(p, m, 0, lane), k1 = k0;
    if (nt > 1) k1 = fetch_key<kGeneral>(p, m, C::kKSweeps == 1 ? 1 : 1 % m.n, lane);
    for (int j = 0; j < nt && ok; ++j) {
      int k2 = k1;
      if (j + 2 < nt) k2 = fetch_key<kGeneral>(p, m, C::kKSweeps == 1 ? j + 2 : (j + 2) % m.n, lane);
      ok = load_tile<C, kGeneral, kBox3, kWarp>(p, map, r, m, k0, lane, kv_it, pol_kv, wd);
      k0 = k1;
      k1 = k2;
    }
  }
  int aborted = 0;
  if (lane == 0) aborted = *wd.abort_flag;
  if (from0(aborted) && lane == 0) {
    // Let copies already issued land before the CTA's shared memory goes away.
    const uint32_t nst = (uint32_t)r.stages;
    const uint32_t nk = kv_it < nst ? kv_it : nst;
    for (uint32_t t = kv_it - nk; t < kv_it; ++t)
      drain_wait(r.full + 8u * (t % nst), (t / nst) & 1u, wd);
    if (kside) {
      const uint32_t nq = q_it < (uint32_t)C::kQBufs ? q_it : (uint32_t)C::kQBufs;
      for (uint32_t t = q_it - nq; t < q_it; ++t)
        drain_wait(sm.bar(C::kBarQFull + q_buf<C>(t)), q_par<C>(t), wd);
    }
  }
}

// Producer of a kernel whose slots hold one unit (p.rk == 1): lane 0 alone.
template <class C, bool kGeneral>
__device__ __forceinline__ void producer_role(const FwdParams& p, uint8_t* smem, const Smem<C> sm,
                                              const Watchdog wd, bool kside) {
  if (C::kChunks == 2 && p.kv_box3) producer_body<C, kGeneral, C::kChunks == 2, false>(p, smem, sm, wd, kside);
  else producer_body<C, kGeneral, false, false>(p, smem, sm, wd, kside);
}
// Producer of a kernel whose slots hold several units (p.rk > 1): every lane
// of the warp.
template <class C, bool kGeneral>
__device__ __forceinline__ void producer_role_warp(const FwdParams& p, uint8_t* smem, const Smem<C> sm,
                                                   const Watchdog wd, bool kside) {
  producer_body<C, kGeneral, false, true>(p, smem, sm, wd, kside);
}

}  // namespace
}  // namespace bsa
