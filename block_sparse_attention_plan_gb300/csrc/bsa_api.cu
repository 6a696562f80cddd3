// Host side of libbsa: argument validation, workspace layout, TMA tensor-map
// encoding, launches and status reporting.  See include/bsa.h for the
// contract of every entry point.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "bsa_internal.h"
#include "bsa_regime_table.h"

using namespace bsa;

namespace {

constexpr uint32_t kPlanMagic = 0xB5A9147Au;

struct PlanImpl {
  uint32_t magic;
  bsa_plan_layout L;
  uint8_t* ws;
  PlanDev dev;
  int device;
};

inline bool supported_block(int b) { return b == 32 || b == 64 || b == 128 || b == 256; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bsa_status compute_layout(int B, int H, int NQB, int NKB, int bq, int bk, int g, int flags,
                          bsa_plan_layout* L, int* nkeys_out) {
  if (!L) return BSA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || NQB < 1 || NKB < 1 || g < 1) return BSA_ERR_INVALID_ARG;
  if (!supported_block(bq) || !supported_block(bk)) return BSA_ERR_UNSUPPORTED;
  if (H % g) return BSA_ERR_INVALID_ARG;
  if (flags & ~(BSA_PLAN_NO_UNION | BSA_PLAN_REMAP | BSA_PLAN_Q64)) return BSA_ERR_INVALID_ARG;
  // Physical q-tile height: 128 rows, or 64 for blocks of at most 64 rows.
  const int qtile = (flags & BSA_PLAN_Q64) ? 64 : kTile;
  if (qtile < bq && qtile < kTile) return BSA_ERR_UNSUPPORTED;
  bsa_plan_layout l;
  std::memset(&l, 0, sizeof(l));
  l.B = B; l.H = H; l.Hkv = H / g; l.NQB = NQB; l.NKB = NKB; l.bq = bq; l.bk = bk; l.gqa_group = g;
  l.qu = bq < qtile ? bq : qtile;
  l.rq = qtile / l.qu;
  l.sq = bq / l.qu;
  l.ku = bk < kTile ? bk : kTile;
  l.rk = kTile / l.ku;
  l.sk = bk / l.ku;
  const long long NQU = (long long)NQB * l.sq;
  if (NQU % l.rq) return BSA_ERR_INVALID_ARG;  // Nq must be a multiple of the q-tile height
  const long long NQT = NQU / l.rq;
  const long long NKU = (long long)NKB * l.sk;
  const long long rows = (long long)B * H * NQT;
  const long long urows = (g > 1 && !(flags & BSA_PLAN_NO_UNION)) ? (long long)B * (H / g) * NQT : 0;
  const long long max_slots = (NKU + l.rk - 1) / l.rk;
  if (rows > (1ll << 30) || NKU > (1ll << 30)) return BSA_ERR_UNSUPPORTED;
  if (max_slots + 1 > kMaxKeys) return BSA_ERR_UNSUPPORTED;
  if ((long long)B * (H / g) > kMaxGroups) return BSA_ERR_UNSUPPORTED;
  const long long slot_cap = rows * max_slots;
  const long long union_cap = urows * NKU;
  if (slot_cap * l.rk >= (1ll << 31) || union_cap >= (1ll << 31)) return BSA_ERR_UNSUPPORTED;
  l.NQT = (int)NQT;
  l.NKU = (int)NKU;
  l.rows = (int)rows;
  l.urows = (int)urows;
  l.max_row_slots = (int)max_slots;
  l.groups = B * (H / g);
  l.slot_capacity = slot_cap;
  l.union_capacity = union_cap;
  const int nkeys = (int)max_slots + 1;
  uint64_t off = 0;
  l.off_row_ptr = off;   off = align256(off + 4ull * (rows + 1));
  l.off_slot_ku = off;   off = align256(off + 4ull * slot_cap * l.rk);
  l.off_slot_mask = off; off = align256(off + 4ull * slot_cap);
  l.off_urow_ptr = off;  off = align256(off + 4ull * (urows + 1));
  l.off_ukb = off;       off = align256(off + 4ull * union_cap);
  l.off_order = off;     off = align256(off + 4ull * rows);
  l.off_totals = off;    off = align256(off + 8ull * 4);
  l.off_control = off;   off = align256(off + 4ull * 16);
  l.off_sigma = off;     off = align256(off + 4ull * (uint64_t)B * H);
  l.off_scratch = off;
  l.workspace_bytes = fwd_scratch(l).end;  // plan scratch, then forward scratch
  *L = l;
  if (nkeys_out) *nkeys_out = nkeys;
  return BSA_OK;
}

// Device capability check, cached per device.
bsa_status check_arch(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  static std::mutex mu;
  static std::vector<int> cache;  // 0 unknown, 1 ok, 2 bad
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return BSA_ERR_CUDA;
    cache[dev] = (maj == 10 && min == 3) ? 1 : 2;
  }
  if (dev_out) *dev_out = dev;
  return cache[dev] == 1 ? BSA_OK : BSA_ERR_ARCH;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2D bf16 view [rows, d] with a box of {64, box_rows} and 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// d = 128 bf16 rows viewed as (64 columns, rows, 2 halves): strides 2 bytes,
// 256 bytes (next row), 128 bytes (second half of the row); box
// {64, box_rows, 2}.  A box lands in shared memory as box_rows rows of the
// first half, then box_rows rows of the second, each 128-byte-swizzled: the
// layout two {64, box_rows} boxes of the 2D view give.  Returns false if the
// driver does not take the view (the caller then uses the 2D one).
bool encode_map_halves(CUtensorMap* m, const void* base, uint64_t rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64u, (cuuint64_t)rows, 2u};
  cuuint64_t strides[2] = {256u, 128u};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 2u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

long long env_ll(const char* name, long long dflt) {
  const char* s = std::getenv(name);
  if (!s || !*s) return dflt;
  char* end = nullptr;
  const long long v = std::strtoll(s, &end, 10);
  return (end && *end == 0 && v > 0) ? v : dflt;
}

const PlanImpl* as_impl(const bsa_plan* p) {
  const PlanImpl* q = reinterpret_cast<const PlanImpl*>(p);
  return (q && q->magic == kPlanMagic) ? q : nullptr;
}

}  // namespace

namespace bsa {
// Forward parameters of one plan (layout L, device views pd, workspace ws)
// for the given tensors: the TMA views of Q (128-row and q-unit boxes), K and
// V (contiguous or paged pools), the plan and scratch pointers, the element
// mask and the grid (one CTA per SM, at most one per plan row; grid_override
// > 0 replaces the SM count).  Validates the pages and the view sizes.
bsa_status make_fwd_params(const bsa_plan_layout& L, const PlanDev& pd, uint8_t* ws, bool remapped,
                           const void* Q, const void* K, const void* V, const bsa_kv_pages* pages,
                           const int32_t* kv_lens, int flags, void* O, float* LSE, int d,
                           float scale, int dev, long long watchdog_ns, long long grid_override,
                           FwdParams* out, int* grid_out) {
  const long long Nq = (long long)L.NQB * L.bq, Nk = (long long)L.NKB * L.bk;
  const long long qrows = (long long)L.B * L.H * Nq;
  long long kvrows = (long long)L.B * L.Hkv * Nk;
  if (pages) {
    if (!pages->block_table || pages->max_pages < 1 || pages->page_size < 1 || pages->num_pages < 1)
      return BSA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(pages->block_table) & 3u) return BSA_ERR_INVALID_ARG;
    if (pages->page_size % L.ku) return BSA_ERR_UNSUPPORTED;
    if ((long long)pages->max_pages * pages->page_size < Nk) return BSA_ERR_INVALID_ARG;
    kvrows = (long long)pages->num_pages * L.Hkv * pages->page_size;
  }
  if (qrows >= (1ll << 31) || kvrows >= (1ll << 31)) return BSA_ERR_UNSUPPORTED;

  FwdParams& fp = *out;
  std::memset(&fp, 0, sizeof(fp));
  if (!encode_map(&fp.tmQ, Q, (uint64_t)qrows, d, L.qu * L.rq) ||
      !encode_map(&fp.tmQu, Q, (uint64_t)qrows, d, L.qu) ||
      !encode_map(&fp.tmK, K, (uint64_t)kvrows, d, L.ku) ||
      !encode_map(&fp.tmV, V, (uint64_t)kvrows, d, L.ku))
    return BSA_ERR_CUDA;
  if (d == 128) {
    fp.q_box3 = encode_map_halves(&fp.tmQ3, Q, (uint64_t)qrows, L.qu * L.rq) ? 1 : 0;
    fp.kv_box3 = (L.rk == 1 && encode_map_halves(&fp.tmK3, K, (uint64_t)kvrows, kTile) &&
                  encode_map_halves(&fp.tmV3, V, (uint64_t)kvrows, kTile)) ? 1 : 0;
  }
  fp.row_ptr = pd.row_ptr;
  fp.slot_ku = pd.slot_ku;
  fp.slot_mask = pd.slot_mask;
  fp.order = pd.order;
  fp.control = pd.control;
  fp.O = static_cast<uint16_t*>(O);
  fp.o_v8 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0 ? 1 : 0;
  fp.LSE = LSE;
  fp.K = static_cast<const uint16_t*>(K);
  fp.V = static_cast<const uint16_t*>(V);
  const FwdScratch fs = fwd_scratch(L);
  fp.kmax = reinterpret_cast<float*>(ws + fs.off_kmax);
  fp.rowk = reinterpret_cast<float*>(ws + fs.off_rowk);
  fp.vmax = reinterpret_cast<float*>(ws + fs.off_vmax);
  fp.rowv = reinterpret_cast<float*>(ws + fs.off_rowv);
  fp.split_all = (flags & BSA_FWD_SPLIT_P) ? 1 : 0;
  fp.fb_flag = reinterpret_cast<int32_t*>(ws + fs.off_fb_flag);
  fp.fb_list = reinterpret_cast<int32_t*>(ws + fs.off_fb_list);
  fp.sigma = remapped ? reinterpret_cast<const int32_t*>(ws + L.off_sigma) : nullptr;
  fp.slot_capacity = L.slot_capacity;
  fp.watchdog_ns = watchdog_ns;
  if (pages) {
    fp.block_table = pages->block_table;
    fp.max_pages = pages->max_pages;
    fp.page_size = pages->page_size;
    fp.num_pages = pages->num_pages;
    fp.prow = reinterpret_cast<int32_t*>(ws + fs.off_prow);
  }
  fp.kv_lens = kv_lens;
  fp.causal = (flags & BSA_FWD_CAUSAL) ? 1 : 0;
  fp.causal_off = (int)(Nk - Nq);
  fp.elem_mask = (fp.causal || kv_lens) ? 1 : 0;
  fp.B = L.B; fp.H = L.H; fp.Hkv = L.Hkv; fp.g = L.gqa_group; fp.NQT = L.NQT; fp.NKU = L.NKU;
  fp.Nq = (int)Nq; fp.Nk = (int)Nk; fp.rq = L.rq; fp.rk = L.rk; fp.qu = L.qu; fp.ku = L.ku;
  fp.rows = L.rows;
  const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)d);
  fp.scale_log2 = (float)(sc * 1.4426950408889634);

  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BSA_ERR_CUDA;
  fp.sms = sms;
  long long grid = grid_override > 0 ? grid_override : sms;
  if (grid > L.rows) grid = L.rows;
  if (grid < 1) grid = 1;
  *grid_out = (int)grid;
  return BSA_OK;
}
}  // namespace bsa

extern "C" {

int bsa_version(void) { return BSA_VERSION; }

const char* bsa_status_string(int s) {
  switch (s) {
    case BSA_OK: return "BSA_OK";
    case BSA_ERR_INVALID_ARG: return "BSA_ERR_INVALID_ARG";
    case BSA_ERR_UNSUPPORTED: return "BSA_ERR_UNSUPPORTED";
    case BSA_ERR_ARCH: return "BSA_ERR_ARCH";
    case BSA_ERR_CUDA: return "BSA_ERR_CUDA";
    case BSA_ERR_WORKSPACE: return "BSA_ERR_WORKSPACE";
    case BSA_ERR_TIMEOUT: return "BSA_ERR_TIMEOUT";
    case BSA_ERR_PLAN_MISMATCH: return "BSA_ERR_PLAN_MISMATCH";
    default: return "BSA_ERR_UNKNOWN";
  }
}

bsa_status bsa_plan_layout_query(int B, int H, int NQB, int NKB, int bq, int bk, int gqa_group,
                                 int flags, bsa_plan_layout* out) {
  return compute_layout(B, H, NQB, NKB, bq, bk, gqa_group, flags, out, nullptr);
}

int bsa_plan_select_flags(int B, int H, int NQB, int NKB, int bq, int bk, int gqa_group, int d) {
  bsa_plan_layout L;
  bsa_status st = compute_layout(B, H, NQB, NKB, bq, bk, gqa_group, 0, &L, nullptr);
  if (st != BSA_OK) return st;
  if (d != 64 && d != 128) return BSA_ERR_UNSUPPORTED;
  int tile = kTile;
  for (const RegimeEntry& e : kRegimeTable)
    if (e.bq == bq && e.bk == bk && e.d == d) tile = e.tile;
  int flags = 0;
  bsa_plan_layout L64;
  if (tile == 64 && compute_layout(B, H, NQB, NKB, bq, bk, gqa_group, BSA_PLAN_Q64, &L64, nullptr) == BSA_OK) {
    flags |= BSA_PLAN_Q64;
    if (L64.rq > 1 && gqa_group == 1) flags |= BSA_PLAN_REMAP;
  } else if (L.rq > 1 && gqa_group == 1) {
    flags |= BSA_PLAN_REMAP;
  }
  return flags;
}

size_t bsa_plan_workspace_bytes(int B, int H, int NQB, int NKB, int bq, int bk, int gqa_group) {
  bsa_plan_layout L;
  if (compute_layout(B, H, NQB, NKB, bq, bk, gqa_group, 0, &L, nullptr) != BSA_OK) return 0;
  return (size_t)L.workspace_bytes;
}

namespace {

// Plan of a logical mask given as mask bytes, affine row segments, or both
// (their union); see bsa_plan_create and bsa_plan_create_affine.
bsa_status create_plan(const uint8_t* mask, const int32_t* seg, const int32_t* seg_ptr, int nseg,
                       int B, int H, int NQB, int NKB, int bq, int bk, int gqa_group,
                       void* workspace, size_t workspace_bytes, int flags, void* stream,
                       bsa_plan** out) {
  if (!out) return BSA_ERR_INVALID_ARG;
  *out = nullptr;
  if ((!mask && !seg_ptr) || !workspace) return BSA_ERR_INVALID_ARG;
  if (seg_ptr && (nseg < 0 || (nseg > 0 && (!seg || !aligned16(seg))))) return BSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return BSA_ERR_INVALID_ARG;
  bsa_plan_layout L;
  int nkeys = 0;
  bsa_status st = compute_layout(B, H, NQB, NKB, bq, bk, gqa_group, flags, &L, &nkeys);
  if (st != BSA_OK) return st;
  if (workspace_bytes < L.workspace_bytes) return BSA_ERR_WORKSPACE;
  int dev = 0;
  st = check_arch(&dev);
  if (st != BSA_OK) return st;

  PlanImpl* impl = new (std::nothrow) PlanImpl;
  if (!impl) return BSA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  impl->magic = kPlanMagic;
  impl->L = L;
  impl->ws = ws;
  impl->device = dev;
  PlanDev& d = impl->dev;
  d.mask = mask;
  d.seg = seg_ptr ? seg : nullptr;
  d.seg_ptr = seg_ptr;
  d.nseg = seg_ptr ? nseg : 0;
  set_plan_views(d, ws, L);
  d.vec = (mask && aligned16(mask) && NKB % 16 == 0) ? 1 : 0;
  d.B = B; d.H = H; d.Hkv = L.Hkv; d.g = gqa_group; d.NQB = NQB; d.NKB = NKB;
  d.qu = L.qu; d.rq = L.rq; d.sq = L.sq; d.ku = L.ku; d.rk = L.rk; d.sk = L.sk;
  d.NQT = L.NQT; d.NKU = L.NKU; d.rows = L.rows; d.urows = L.urows;
  d.nkeys = nkeys; d.groups = L.groups;
  d.remap = ((flags & BSA_PLAN_REMAP) && L.rq > 1 && gqa_group == 1 && L.NQT <= kMaxRemapTiles) ? 1 : 0;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Pass counters and forward status only: a key-norm stage of this plan's
  // forward may already be running on another stream.
  if (cudaMemsetAsync(d.control, 0, 4 * (kCtlFallbackWork + 1), s) != cudaSuccess ||
      launch_plan(d, s) != cudaSuccess) {
    delete impl;
    return BSA_ERR_CUDA;
  }
  *out = reinterpret_cast<bsa_plan*>(impl);
  return BSA_OK;
}

}  // namespace

bsa_status bsa_plan_create(const uint8_t* mask, int B, int H, int NQB, int NKB, int bq, int bk,
                           int gqa_group, void* workspace, size_t workspace_bytes, int flags,
                           void* stream, bsa_plan** out) {
  if (!mask) {
    if (out) *out = nullptr;
    return BSA_ERR_INVALID_ARG;
  }
  return create_plan(mask, nullptr, nullptr, 0, B, H, NQB, NKB, bq, bk, gqa_group, workspace,
                     workspace_bytes, flags, stream, out);
}

bsa_status bsa_plan_create_affine(const uint8_t* mask, const int32_t* segments,
                                  const int32_t* seg_ptr, int nseg, int B, int H, int NQB,
                                  int NKB, int bq, int bk, int gqa_group, void* workspace,
                                  size_t workspace_bytes, int flags, void* stream,
                                  bsa_plan** out) {
  if (!seg_ptr) {
    if (out) *out = nullptr;
    return BSA_ERR_INVALID_ARG;
  }
  return create_plan(mask, segments, seg_ptr, nseg, B, H, NQB, NKB, bq, bk, gqa_group, workspace,
                     workspace_bytes, flags, stream, out);
}

bsa_status bsa_plan_get_layout(const bsa_plan* plan, bsa_plan_layout* out) {
  const PlanImpl* p = as_impl(plan);
  if (!p || !out) return BSA_ERR_INVALID_ARG;
  *out = p->L;
  return BSA_OK;
}

void* bsa_plan_workspace(const bsa_plan* plan) {
  const PlanImpl* p = as_impl(plan);
  return p ? p->ws : nullptr;
}

void bsa_plan_destroy(bsa_plan* plan) {
  PlanImpl* p = reinterpret_cast<PlanImpl*>(plan);
  if (!p || p->magic != kPlanMagic) return;
  p->magic = 0;
  delete p;
}

bsa_status bsa_forward(const bsa_plan* plan, const void* Q, const void* K, const void* V, void* O,
                       float* LSE, int d, float scale, void* stream) {
  return bsa_forward_ex(plan, Q, K, V, nullptr, nullptr, 0, O, LSE, d, scale, stream);
}

bsa_status bsa_forward_ex(const bsa_plan* plan, const void* Q, const void* K, const void* V,
                          const bsa_kv_pages* pages, const int32_t* kv_lens, int flags,
                          void* O, float* LSE, int d, float scale, void* stream) {
  return bsa_forward_stage(plan, Q, K, V, pages, kv_lens, flags, O, LSE, d, scale,
                           BSA_STAGE_ALL, stream);
}

bsa_status bsa_forward_stage(const bsa_plan* plan, const void* Q, const void* K, const void* V,
                             const bsa_kv_pages* pages, const int32_t* kv_lens, int flags,
                             void* O, float* LSE, int d, float scale, int stages, void* stream) {
  constexpr int kAllBits = BSA_STAGE_ALL | BSA_STAGE_KNORM | BSA_STAGE_ROWBOUND;
  if (stages <= 0 || (stages & ~kAllBits)) return BSA_ERR_INVALID_ARG;
  const PlanImpl* p = as_impl(plan);
  if (!plan) return BSA_ERR_INVALID_ARG;
  if (!p) return BSA_ERR_PLAN_MISMATCH;
  if (!Q || !K || !V || !O || !LSE) return BSA_ERR_INVALID_ARG;
  if (flags & ~(BSA_FWD_CAUSAL | BSA_FWD_SPLIT_P)) return BSA_ERR_INVALID_ARG;
  if (kv_lens && (reinterpret_cast<uintptr_t>(kv_lens) & 3u)) return BSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return BSA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return BSA_ERR_UNSUPPORTED;
  if (!(scale == scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
  int dev = 0;
  bsa_status st = check_arch(&dev);
  if (st != BSA_OK) return st;
  if (dev != p->device) return BSA_ERR_PLAN_MISMATCH;
  // 64-row q-tiles: contiguous K/V without an element mask only.
  if (p->L.qu * p->L.rq == 64 && (pages || kv_lens || (flags & BSA_FWD_CAUSAL)))
    return BSA_ERR_UNSUPPORTED;
  const PlanDev& pd = p->dev;
  FwdParams fp;
  int grid = 1;
  st = make_fwd_params(p->L, pd, p->ws, p->dev.remap != 0, Q, K, V, pages, kv_lens, flags, O, LSE,
                       d, scale, dev, env_ll("BSA_WATCHDOG_MS", 1000) * 1000000ll,
                       env_ll("BSA_GRID", 0), &fp, &grid);
  if (st != BSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The key-norm stage resets its own status words, the row-bound stage the
  // pass counters and the forward status (the two may run on different
  // streams, the first beside the plan kernels).
  const bool knorm = stages & (BSA_STAGE_PREPARE | BSA_STAGE_KNORM);
  const bool rowbound = stages & (BSA_STAGE_PREPARE | BSA_STAGE_ROWBOUND);
  if (knorm && rowbound) {  // one reset of both sets of words
    if (cudaMemsetAsync(pd.control, 0, 4 * (kCtlKnormDetail + 1), s) != cudaSuccess) return BSA_ERR_CUDA;
  } else if (knorm) {
    if (cudaMemsetAsync(pd.control + kCtlKnormStatus, 0, 8, s) != cudaSuccess) return BSA_ERR_CUDA;
  } else if (rowbound) {
    if (cudaMemsetAsync(pd.control, 0, 4 * (kCtlFallbackWork + 1), s) != cudaSuccess) return BSA_ERR_CUDA;
  }
  if (launch_forward(fp, d, (int)grid, s, stages) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status bsa_sync_status(const bsa_plan* plan, void* stream, int32_t* detail) {
  const PlanImpl* p = as_impl(plan);
  if (!p) return BSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSA_ERR_CUDA;
  int32_t ctl[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (cudaMemcpy(ctl, p->dev.control, sizeof(ctl), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BSA_ERR_CUDA;
  const bool knorm = ctl[kCtlStatus] == 0 && ctl[kCtlKnormStatus] != 0;
  if (detail) *detail = knorm ? ctl[kCtlKnormDetail] : ctl[kCtlDetail];
  return static_cast<bsa_status>(knorm ? ctl[kCtlKnormStatus] : ctl[kCtlStatus]);
}

bsa_status bsa_plan_check(const bsa_plan* plan, void* stream) {
  const PlanImpl* p = as_impl(plan);
  if (!p) return BSA_ERR_INVALID_ARG;
  const bsa_plan_layout& L = p->L;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSA_ERR_CUDA;
  std::vector<int32_t> rp(L.rows + 1), order(L.rows);
  if (cudaMemcpy(rp.data(), p->dev.row_ptr, 4ull * (L.rows + 1), cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(order.data(), p->dev.order, 4ull * L.rows, cudaMemcpyDeviceToHost) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (rp[0] != 0) return BSA_ERR_PLAN_MISMATCH;
  for (int r = 0; r < L.rows; ++r)
    if (rp[r + 1] < rp[r] || rp[r + 1] - rp[r] > L.max_row_slots) return BSA_ERR_PLAN_MISMATCH;
  const long long S = rp[L.rows];
  if (S > L.slot_capacity) return BSA_ERR_PLAN_MISMATCH;
  std::vector<int32_t> ku((size_t)S * L.rk);
  if (S > 0 && cudaMemcpy(ku.data(), p->dev.slot_ku, 4ull * S * L.rk, cudaMemcpyDeviceToHost) !=
                   cudaSuccess)
    return BSA_ERR_CUDA;
  for (int r = 0; r < L.rows; ++r) {
    const long long a = (long long)rp[r] * L.rk, b = (long long)rp[r + 1] * L.rk;
    int prev = -1;
    bool padded = false;
    for (long long i = a; i < b; ++i) {
      const int y = ku[i];
      if (y < 0) {
        if (y != -1 || b - i > L.rk - 1) return BSA_ERR_PLAN_MISMATCH;  // only in the last slot
        padded = true;
        continue;
      }
      if (padded || y >= L.NKU || y <= prev) return BSA_ERR_PLAN_MISMATCH;
      prev = y;
    }
    if (b > a && ku[a] < 0) return BSA_ERR_PLAN_MISMATCH;
  }
  std::vector<char> seen(L.rows, 0);
  for (int i = 0; i < L.rows; ++i) {
    const int r = order[i];
    if (r < 0 || r >= L.rows || seen[r]) return BSA_ERR_PLAN_MISMATCH;
    seen[r] = 1;
  }
  return BSA_OK;
}

bsa_status bsa_plan_export(const bsa_plan* plan, void* stream, bsa_plan_arrays* out) {
  const PlanImpl* p = as_impl(plan);
  if (!p || !out) return BSA_ERR_INVALID_ARG;
  const bsa_plan_layout& L = p->L;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSA_ERR_CUDA;
  if (cudaMemcpy(out->totals, p->dev.totals, sizeof(out->totals), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return BSA_ERR_CUDA;
  const long long S = out->totals[0], U = out->totals[2];
  if (S < 0 || S > L.slot_capacity || U < 0 || U > L.union_capacity) return BSA_ERR_PLAN_MISMATCH;
  struct Copy {
    void* dst;
    size_t cap;
    const void* src;
    size_t n;  // elements (4 bytes each)
  };
  const Copy copies[] = {
      {out->row_ptr, out->row_ptr_cap, p->dev.row_ptr, (size_t)L.rows + 1},
      {out->slot_ku, out->slot_ku_cap, p->dev.slot_ku, (size_t)S * L.rk},
      {out->slot_mask, out->slot_mask_cap, p->dev.slot_mask, (size_t)S},
      {out->urow_ptr, out->urow_ptr_cap, p->dev.urow_ptr, (size_t)L.urows + 1},
      {out->ukb, out->ukb_cap, p->dev.ukb, (size_t)U},
      {out->order, out->order_cap, p->dev.order, (size_t)L.rows},
      {out->plane_sigma, out->plane_sigma_cap, p->dev.sigma, (size_t)L.B * L.H},
  };
  for (const Copy& c : copies)
    if (c.dst && c.cap < c.n) return BSA_ERR_WORKSPACE;
  for (const Copy& c : copies) {
    if (!c.dst || c.n == 0) continue;
    if (cudaMemcpy(c.dst, c.src, 4 * c.n, cudaMemcpyDeviceToHost) != cudaSuccess) return BSA_ERR_CUDA;
  }
  return BSA_OK;
}

bsa_status bsa_watchdog_selftest(int32_t* status, int limit_us, void* stream) {
  if (!status || limit_us <= 0) return BSA_ERR_INVALID_ARG;
  bsa_status st = check_arch(nullptr);
  if (st != BSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, 16, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (launch_watchdog_selftest(status, (long long)limit_us * 1000ll, s) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSA_ERR_CUDA;
  int32_t h[4];
  if (cudaMemcpy(h, status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return BSA_ERR_CUDA;
  if (h[3] != 0) return BSA_OK;  // the wait completed: no timeout observed
  return static_cast<bsa_status>(h[kCtlStatus]);
}

}  // extern "C"
