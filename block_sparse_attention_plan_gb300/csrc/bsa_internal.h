// Internal declarations shared by the host API and the kernels of libbsa.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa.h"

namespace bsa {

constexpr int kTile = 128;            // physical q-tile rows and K/V slot rows
constexpr int kMaxKeys = 12288;       // bound on (slots per row + 1) for the sort
constexpr int kMaxGroups = 8192;      // bound on K/V-head groups (B * Hkv)
constexpr int kMaxRemapTiles = 8192;  // planes with more q-tiles keep grouping stride 1
constexpr int kCtlWorkCounter = 0;    // control word indices
constexpr int kCtlStatus = 1;
constexpr int kCtlDetail = 2;
constexpr int kCtlFallbackCount = 3;  // rows queued for the exact second pass
constexpr int kCtlFallbackWork = 4;   // work counter of that pass
constexpr int kCtlKnormStatus = 5;    // status / detail of the key-norm pass (its stage may
constexpr int kCtlKnormDetail = 6;    // run beside the plan kernels; reset by that stage)

// Wait sites recorded in the status detail word (low 8 bits).
enum WaitSite : int {
  kSiteQEmpty = 1, kSiteQFull, kSiteKvEmpty, kSiteKvFull, kSiteSFull, kSitePFull,
  kSiteODone, kSiteXchg, kSiteDrain, kSiteSelftest, kSiteSched, kSitePlanRange = 0x40
};

// Device views of a plan's workspace.
struct PlanDev {
  const uint8_t* mask;
  int32_t* row_ptr;
  int32_t* slot_ku;
  uint32_t* slot_mask;
  int32_t* urow_ptr;
  int32_t* ukb;
  int32_t* order;
  long long* totals;
  int32_t* control;
  int32_t* slots;   // scratch: slots per row
  int32_t* lcnt;    // scratch: selected logical blocks owned by the row
  int32_t* ucnt;    // scratch: union entries per union row
  int32_t* gstart;  // scratch: first schedule position of each K/V-head group
  uint32_t* qbits;  // scratch: [rows][rq][W] selected k-units of each q-unit, 32 per word
  uint32_t* ubits;  // scratch: [urows][W] union k-units of each union row
  int B, H, Hkv, g, NQB, NKB;
  int qu, rq, sq, ku, rk, sk;
  int NQT, NKU, rows, urows, nkeys, groups;
  const int32_t* seg;      // affine row segments [nseg][4] = {a, b, stride, count}, or nullptr
  const int32_t* seg_ptr;  // [H + 1]: head h owns segments seg_ptr[h] .. seg_ptr[h+1]-1
  int nseg;
  int32_t* sigma;  // [B*H] q-unit grouping stride of each plane
  int remap;       // choose the strides (else all 1)
  int W;    // bitmap words per q-unit: ceil(NKU / 32)
  int vec;  // mask rows may be read 16 bytes at a time (16-byte aligned mask, NKB % 16 == 0)
};

inline uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

// Plan-construction scratch inside a plan workspace, after the plan arrays.
struct PlanScratch {
  uint64_t off_slots, off_lcnt, off_ucnt, off_gstart, off_qbits, off_ubits, end;
};
inline PlanScratch plan_scratch(const bsa_plan_layout& L) {
  const uint64_t W = ((uint64_t)L.NKU + 31) / 32;
  PlanScratch s;
  uint64_t off = L.off_scratch;
  s.off_slots = off;  off = align256(off + 4ull * (uint64_t)L.rows);
  s.off_lcnt = off;   off = align256(off + 4ull * (uint64_t)L.rows);
  s.off_ucnt = off;   off = align256(off + 4ull * ((uint64_t)L.urows + 1));
  s.off_gstart = off; off = align256(off + 4ull * (uint64_t)L.groups);
  s.off_qbits = off;  off = align256(off + 4ull * (uint64_t)L.rows * L.rq * W);
  s.off_ubits = off;  off = align256(off + 4ull * (uint64_t)L.urows * W);
  s.end = off;
  return s;
}

// Points the plan views of `d` at workspace `ws` laid out by `L`.
inline void set_plan_views(PlanDev& d, uint8_t* ws, const bsa_plan_layout& L) {
  d.row_ptr = reinterpret_cast<int32_t*>(ws + L.off_row_ptr);
  d.slot_ku = reinterpret_cast<int32_t*>(ws + L.off_slot_ku);
  d.slot_mask = reinterpret_cast<uint32_t*>(ws + L.off_slot_mask);
  d.urow_ptr = reinterpret_cast<int32_t*>(ws + L.off_urow_ptr);
  d.ukb = reinterpret_cast<int32_t*>(ws + L.off_ukb);
  d.order = reinterpret_cast<int32_t*>(ws + L.off_order);
  d.totals = reinterpret_cast<long long*>(ws + L.off_totals);
  d.control = reinterpret_cast<int32_t*>(ws + L.off_control);
  d.sigma = reinterpret_cast<int32_t*>(ws + L.off_sigma);
  const PlanScratch s = plan_scratch(L);
  d.slots = reinterpret_cast<int32_t*>(ws + s.off_slots);
  d.lcnt = reinterpret_cast<int32_t*>(ws + s.off_lcnt);
  d.ucnt = reinterpret_cast<int32_t*>(ws + s.off_ucnt);
  d.gstart = reinterpret_cast<int32_t*>(ws + s.off_gstart);
  d.qbits = reinterpret_cast<uint32_t*>(ws + s.off_qbits);
  d.ubits = reinterpret_cast<uint32_t*>(ws + s.off_ubits);
  d.W = (L.NKU + 31) / 32;
}

// Forward-pass scratch inside a plan workspace, after the plan-construction
// scratch: the largest key norm of every K unit (float[B*Hkv*NKU]), that of
// every plan row's selected units (float[rows]), a fallback flag per plan row
// and the list of rows queued for the exact pass (int32[rows] each), for
// paged K/V the pool row of every slot position (int32[slot_capacity*rk]),
// and the largest |v| element of every V unit and of every plan row's units
// (float[B*Hkv*NKU], float[rows]).
struct FwdScratch {
  uint64_t off_kmax, off_rowk, off_fb_flag, off_fb_list, off_prow, off_vmax, off_rowv, end;
};
inline FwdScratch fwd_scratch(const bsa_plan_layout& L) {
  uint64_t off = plan_scratch(L).end;
  FwdScratch f;
  f.off_kmax = off;    off = align256(off + 4ull * (uint64_t)L.B * L.Hkv * L.NKU);
  f.off_rowk = off;    off = align256(off + 4ull * (uint64_t)L.rows);
  f.off_fb_flag = off; off = align256(off + 4ull * (uint64_t)L.rows);
  f.off_fb_list = off; off = align256(off + 4ull * (uint64_t)L.rows);
  f.off_prow = off;    off = align256(off + 4ull * (uint64_t)L.slot_capacity * L.rk);
  f.off_vmax = off;    off = align256(off + 4ull * (uint64_t)L.B * L.Hkv * L.NKU);
  f.off_rowv = off;    off = align256(off + 4ull * (uint64_t)L.rows);
  f.end = off;
  return f;
}

// Kernel parameters of the forward pass (passed as a __grid_constant__).
struct FwdParams {
  CUtensorMap tmQ;   // Q viewed as [B*Hq*Nq, d], box {64, 128}, 128B swizzle
  CUtensorMap tmK;   // K viewed as [B*Hkv*Nk, d], box {64, ku}
  CUtensorMap tmV;   // V likewise
  CUtensorMap tmQu;  // Q viewed as [B*Hq*Nq, d], box {64, qu}: one q-unit (regrouped tiles)
  // d = 128: the same tensors viewed in 3D as (64 columns, rows, 2 halves of
  // a row), so that one box brings both 64-column halves of a tile, laid out
  // in shared memory half after half as the MMA reads them (two 2D boxes
  // otherwise).  Used when kv_box3 / q_box3 are set.
  CUtensorMap tmQ3;  // box {64, q-tile rows, 2}
  CUtensorMap tmK3;  // box {64, 128, 2} (slots of one 128-key unit)
  CUtensorMap tmV3;
  int q_box3;        // the contiguous Q tile is loaded through tmQ3
  int kv_box3;       // K/V slots (one unit each) are loaded through tmK3 / tmV3
  const int32_t* row_ptr;
  const int32_t* slot_ku;
  const uint32_t* slot_mask;
  const int32_t* order;
  int32_t* control;
  uint16_t* O;       // bf16 bits
  float* LSE;
  int o_v8;          // O is 32-byte aligned: rows are written with 32-byte stores
  const uint16_t* K;     // bf16 bits, [B*Hkv*Nk, d] (read by the key-norm pass)
  const uint16_t* V;     // bf16 bits, same view as K (read by the key-norm pass)
  float* kmax;           // largest key norm per K unit
  float* rowk;           // largest key norm over each plan row's K units
  float* vmax;           // largest |v| element per V unit
  float* rowv;           // largest |v| element over each plan row's V units
  int split_all;         // every row applies split (hi + lo) weights
  int32_t* fb_flag;      // per plan row: queued for the exact pass
  int32_t* fb_list;      // plan rows queued for the exact pass
  // Paged K/V (block_table == nullptr: contiguous [B*Hkv*Nk, d]).
  const int32_t* block_table;    // [B][max_pages] physical page per logical page
  int max_pages, page_size, num_pages;
  // Paged K/V: first pool row of the unit at each slot position (-1 = padding
  // or an entry out of range), written by the row-bound pass; nullptr when
  // contiguous.
  int32_t* prow;
  const int32_t* sigma;  // [B*H] q-unit grouping stride of each plane (plan array);
                         // nullptr when the plan was built without regrouping
  // Element mask inside selected blocks.
  const int32_t* kv_lens;        // [B] or nullptr
  int causal;                    // key j visible to query i iff j <= i + causal_off
  int causal_off;                // Nk - Nq
  int elem_mask;                 // causal || kv_lens
  int32_t* work_counter;         // set by launch_forward: the pass's work counter
  const int32_t* work_count;     // number of work items (nullptr: rows)
  long long slot_capacity;
  long long watchdog_ns;
  int B, H, Hkv, g, NQT, NKU, Nq, Nk, rq, rk, qu, ku, rows;
  int sms;           // multiprocessors of the device (grid of the key-norm pass)
  float scale_log2;  // scale * log2(e)
};

cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream);
// Key-norm pass, bounded-reference pass over every plan row, then the exact
// pass over the rows the first one queued (see bsa_forward.cu).
// `stages`: BSA_STAGE_* bits (the key-norm and row-bound passes, the bounded
// pass, the exact pass), launched in that order.
cudaError_t launch_forward(const FwdParams& p, int d, int grid, cudaStream_t stream,
                           int stages = BSA_STAGE_ALL);
int forward_smem_bytes(int d);
// Key-norm and row-bound passes of `stages` (BSA_STAGE_PREPARE, _KNORM,
// _ROWBOUND bits; others ignored), see bsa_prep.cu.
cudaError_t launch_prep(const FwdParams& p, int d, int stages, cudaStream_t stream);
// Bounded (exact = false) or exact pass of a plan with 64-row q-tiles
// (bsa_forward_q64.cu); launched by launch_forward for such plans.
cudaError_t launch_forward_q64(const FwdParams& p, int d, int grid, cudaStream_t stream, bool exact);
// Forward parameters and grid of one plan for the given tensors (bsa_api.cu).
bsa_status make_fwd_params(const bsa_plan_layout& L, const PlanDev& pd, uint8_t* ws, bool remapped,
                           const void* Q, const void* K, const void* V, const bsa_kv_pages* pages,
                           const int32_t* kv_lens, int flags, void* O, float* LSE, int d,
                           float scale, int dev, long long watchdog_ns, long long grid_override,
                           FwdParams* out, int* grid_out);
cudaError_t launch_watchdog_selftest(int32_t* status, long long limit_ns, cudaStream_t stream);

}  // namespace bsa
