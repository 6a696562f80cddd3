// bsa_attention_static: plan + forward in one call, for callers that cannot
// allocate device memory.
//
// Some callers are not allowed to allocate: an inference-engine plugin whose
// execute/enqueue step must not call cudaMalloc, a component that runs under
// a memory budget fixed before execution starts, or a host program that only
// ever receives device pointers for its inputs and outputs.  bsa_plan_create
// needs a caller-provided workspace; this entry point instead keeps the plan
// in a scratch area compiled into the library: a file-scope __device__ array
// of BSA_STATIC_WORKSPACE_BYTES, which every GPU that loads the library holds
// until the process exits.  The caller passes only inputs and outputs.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is looked up once per
// device with cudaGetSymbolAddress, on the first call made with that device
// current, and cached.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "bsa_internal.h"

using namespace bsa;

namespace {

constexpr int kMaxDevices = 64;

// The scratch area: plan arrays, schedule, control words.  Shared by every
// call on a device; it keeps the previous call's contents.
static __device__ __align__(256) uint8_t g_static_workspace[BSA_STATIC_WORKSPACE_BYTES];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

bsa_status static_workspace(int dev, uint8_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr)
      return BSA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_addr[dev]);
  return BSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_static() {
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

bool encode_2d(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows) {
  auto fn = encode_fn_static();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" bsa_status bsa_attention_static(const uint8_t* mask, int B, int H, int NQB, int NKB,
                                           int bq, int bk, int gqa_group, const void* Q,
                                           const void* K, const void* V, void* O, float* LSE,
                                           int d, float scale, void* stream) {
  if (!mask || !Q || !K || !V || !O || !LSE) return BSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return BSA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return BSA_ERR_UNSUPPORTED;
  if (!(scale == scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
  // The forward pass does not read the GQA union table: leave it out.
  bsa_plan_layout L;
  bsa_status st = bsa_plan_layout_query(B, H, NQB, NKB, bq, bk, gqa_group, BSA_PLAN_NO_UNION, &L);
  if (st != BSA_OK) return st;
  if (L.workspace_bytes > (uint64_t)BSA_STATIC_WORKSPACE_BYTES) return BSA_ERR_WORKSPACE;
  const long long Nq = (long long)NQB * bq, Nk = (long long)NKB * bk;
  const long long qrows = (long long)B * H * Nq, kvrows = (long long)B * L.Hkv * Nk;
  if (qrows >= (1ll << 31) || kvrows >= (1ll << 31)) return BSA_ERR_UNSUPPORTED;

  int dev = 0, maj = 0, min = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (maj != 10 || min != 3) return BSA_ERR_ARCH;
  uint8_t* ws = nullptr;
  st = static_workspace(dev, &ws);
  if (st != BSA_OK) return st;

  // Plan views into the static scratch (same layout as a caller workspace).
  PlanDev pd;
  std::memset(&pd, 0, sizeof(pd));
  pd.mask = mask;
  set_plan_views(pd, ws, L);
  pd.vec = ((reinterpret_cast<uintptr_t>(mask) & 15u) == 0 && NKB % 16 == 0) ? 1 : 0;
  pd.B = B; pd.H = H; pd.Hkv = L.Hkv; pd.g = gqa_group; pd.NQB = NQB; pd.NKB = NKB;
  pd.qu = L.qu; pd.rq = L.rq; pd.sq = L.sq; pd.ku = L.ku; pd.rk = L.rk; pd.sk = L.sk;
  pd.NQT = L.NQT; pd.NKU = L.NKU; pd.rows = L.rows; pd.urows = L.urows;
  pd.nkeys = L.max_row_slots + 1; pd.groups = L.groups;

  FwdParams fp;
  std::memset(&fp, 0, sizeof(fp));
  if (!encode_2d(&fp.tmQ, Q, (uint64_t)qrows, d, kTile) ||
      !encode_2d(&fp.tmQu, Q, (uint64_t)qrows, d, L.qu) ||
      !encode_2d(&fp.tmK, K, (uint64_t)kvrows, d, L.ku) ||
      !encode_2d(&fp.tmV, V, (uint64_t)kvrows, d, L.ku))
    return BSA_ERR_CUDA;
  fp.row_ptr = pd.row_ptr;
  fp.slot_ku = pd.slot_ku;
  fp.slot_mask = pd.slot_mask;
  fp.order = pd.order;
  fp.control = pd.control;
  fp.O = static_cast<uint16_t*>(O);
  fp.LSE = LSE;
  fp.K = static_cast<const uint16_t*>(K);
  const FwdScratch fs = fwd_scratch(L);
  fp.kmax = reinterpret_cast<float*>(ws + fs.off_kmax);
  fp.rowk = reinterpret_cast<float*>(ws + fs.off_rowk);
  fp.fb_flag = reinterpret_cast<int32_t*>(ws + fs.off_fb_flag);
  fp.fb_list = reinterpret_cast<int32_t*>(ws + fs.off_fb_list);
  fp.slot_capacity = L.slot_capacity;
  fp.watchdog_ns = 1000ll * 1000000ll;
  fp.B = B;
  fp.H = H; fp.Hkv = L.Hkv; fp.g = gqa_group; fp.NQT = L.NQT; fp.NKU = L.NKU;
  fp.Nq = (int)Nq; fp.Nk = (int)Nk; fp.rq = L.rq; fp.rk = L.rk; fp.qu = L.qu; fp.ku = L.ku;
  fp.rows = L.rows;
  const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)d);
  fp.scale_log2 = (float)(sc * 1.4426950408889634);
  fp.sms = sms;
  const int grid = sms < L.rows ? sms : L.rows;

  // The control words (work counter, status) must start at zero on every call.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(pd.control, 0, 64, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (launch_plan(pd, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (launch_forward(fp, d, grid, s) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}
