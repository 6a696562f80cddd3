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


#include "bsa_internal.h"

using namespace bsa;

namespace {

constexpr int kMaxDevices = 64;

// The scratch area: plan arrays, schedule, control words.  Shared by every
// call on a device; it keeps the previous call's contents.
static __device__ __align__(256) uint8_t g_static_workspace[BSA_STATIC_WORKSPACE_BYTES];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
// Byte offset of the control words (status, detail) inside the scratch area
// for the last call on each device (they move with the problem's layout);
// 0 before the first call.
uint64_t g_ctl_off[kMaxDevices] = {};
bool g_called[kMaxDevices] = {};

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

  int dev = 0, maj = 0, min = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
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
  int grid = 1;
  st = make_fwd_params(L, pd, ws, false, Q, K, V, nullptr, nullptr, 0, O, LSE, d, scale, dev,
                       1000ll * 1000000ll, 0, &fp, &grid);
  if (st != BSA_OK) return st;

  {
    std::lock_guard<std::mutex> lock(g_mu);
    g_ctl_off[dev] = L.off_control;
    g_called[dev] = true;
  }
  // The control words (work counter, status) must start at zero on every call.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(pd.control, 0, 64, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (launch_plan(pd, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (launch_forward(fp, d, grid, s) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

// Status the kernels of the last bsa_attention_static call on the current
// device recorded in the scratch area (see include/bsa.h).
extern "C" bsa_status bsa_attention_static_status(void* stream, int32_t* detail) {
  if (detail) *detail = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
  uint64_t off = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_called[dev]) return BSA_OK;  // nothing has run on this device
    off = g_ctl_off[dev];
  }
  uint8_t* ws = nullptr;
  bsa_status st = static_workspace(dev, &ws);
  if (st != BSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t ctl[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (cudaMemcpyAsync(ctl, ws + off, sizeof(ctl), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return BSA_ERR_CUDA;
  const bool knorm = ctl[kCtlStatus] == 0 && ctl[kCtlKnormStatus] != 0;
  if (detail) *detail = knorm ? ctl[kCtlKnormDetail] : ctl[kCtlDetail];
  return static_cast<bsa_status>(knorm ? ctl[kCtlKnormStatus] : ctl[kCtlStatus]);
}
