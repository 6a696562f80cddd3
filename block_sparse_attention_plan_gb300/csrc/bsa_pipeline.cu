// bsa_attention_host: plan + forward from host buffers, with the copies to
// and from the device overlapped with the computation.
//
// The B*Hkv (batch, K/V head) units of a problem are independent BSA problems
// (no row of one reads another's K/V), and in the [B][H..][N][d] layouts a
// contiguous range of units is a contiguous slice of every tensor: the g
// query heads of each unit in Q, O, LSE and the mask, the unit itself in K and
// V.  The units are cut into C chunks.  Chunk i goes through three streams:
// its inputs are copied host -> device on a copy-in stream, its plan and
// forward run on the caller's stream, its O and LSE are copied device -> host
// on a copy-out stream.  Two device slots alternate between chunks, so while
// chunk i computes, chunk i+1 is copied in and chunk i-1 copied out.  Events
// order each slot's reuse: chunk i+2 is copied into a slot only after chunk i
// has computed from it, and computes into it only after chunk i's output has
// been copied out.
//
// The pages describe the attention computation and its GPU execution, not
// host transfers: this entry point is plumbing around the same plan and
// forward kernels (each chunk is planned and run exactly as bsa_plan_create
// + bsa_forward would run it, so every row's result is bit-identical to a
// single device-resident call).  Plans are not regrouped (BSA_PLAN_REMAP):
// here the copies bound the time and the extra plan launch per chunk cost
// more than regrouping saved (regular workload end to end 1.26 -> 1.38 ms).
#include <cstdint>
#include <cstring>

#include "bsa_internal.h"

using namespace bsa;

namespace {

struct SlotLayout {
  uint64_t mask, q, k, v, o, lse, ws, bytes;  // offsets inside one slot, and its size
};

struct PipeGeom {
  int units, chunks, per;  // B*Hkv units, chunks, units per chunk (the last may hold fewer)
  long long Nq, Nk;
  SlotLayout slot;
  uint64_t status_off, total;
};

bsa_status geometry(int B, int H, int NQB, int NKB, int bq, int bk, int g, int d, int chunks,
                    PipeGeom* G) {
  if (B < 1 || H < 1 || g < 1 || H % g) return BSA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return BSA_ERR_UNSUPPORTED;
  if (chunks < 1) return BSA_ERR_INVALID_ARG;
  const int Hkv = H / g;
  G->units = B * Hkv;
  G->chunks = chunks < G->units ? chunks : G->units;
  G->per = (G->units + G->chunks - 1) / G->chunks;
  G->chunks = (G->units + G->per - 1) / G->per;
  G->Nq = (long long)NQB * bq;
  G->Nk = (long long)NKB * bk;
  // A chunk of `per` units is planned as one batch of per*g query heads.
  bsa_plan_layout L;
  const bsa_status st = bsa_plan_layout_query(1, G->per * g, NQB, NKB, bq, bk, g, BSA_PLAN_NO_UNION, &L);
  if (st != BSA_OK) return st;
  const uint64_t hq = (uint64_t)G->per * g;
  SlotLayout& s = G->slot;
  uint64_t off = 0;
  s.mask = off; off = align256(off + hq * NQB * NKB);
  s.q = off;    off = align256(off + hq * G->Nq * d * 2);
  s.k = off;    off = align256(off + (uint64_t)G->per * G->Nk * d * 2);
  s.v = off;    off = align256(off + (uint64_t)G->per * G->Nk * d * 2);
  s.o = off;    off = align256(off + hq * G->Nq * d * 2);
  s.lse = off;  off = align256(off + hq * G->Nq * 4);
  s.ws = off;   off = align256(off + L.workspace_bytes);
  s.bytes = off;
  const int nslots = G->chunks > 1 ? 2 : 1;
  G->status_off = s.bytes * nslots;
  G->total = G->status_off + align256(24ull * G->chunks);  // control words 1..6 of each chunk
  return BSA_OK;
}

// Streams and events of one call, released at the end (release is deferred
// by the runtime until the work enqueued on them has finished).
struct PipeObjects {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr, h2d[2] = {}, comp[2] = {}, d2h[2] = {};
  ~PipeObjects() {
    for (cudaEvent_t* e : {&start, &done, &h2d[0], &h2d[1], &comp[0], &comp[1], &d2h[0], &d2h[1]})
      if (*e) cudaEventDestroy(*e);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
  bool create() {
    if (cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) != cudaSuccess)
      return false;
    for (cudaEvent_t* e : {&start, &done, &h2d[0], &h2d[1], &comp[0], &comp[1], &d2h[0], &d2h[1]})
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
};

}  // namespace

extern "C" bsa_status bsa_attention_host_buffer_bytes(int B, int H, int NQB, int NKB, int bq, int bk,
                                                      int gqa_group, int d, int chunks,
                                                      size_t* bytes) {
  if (!bytes) return BSA_ERR_INVALID_ARG;
  PipeGeom G;
  const bsa_status st = geometry(B, H, NQB, NKB, bq, bk, gqa_group, d, chunks, &G);
  if (st != BSA_OK) return st;
  *bytes = (size_t)G.total;
  return BSA_OK;
}

extern "C" bsa_status bsa_attention_host(const uint8_t* mask, int B, int H, int NQB, int NKB,
                                         int bq, int bk, int gqa_group, const void* Q,
                                         const void* K, const void* V, void* O, float* LSE, int d,
                                         float scale, int chunks, void* buffer,
                                         size_t buffer_bytes, void* stream) {
  if (!mask || !Q || !K || !V || !O || !LSE || !buffer) return BSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(buffer) & 255u) return BSA_ERR_INVALID_ARG;
  PipeGeom G;
  bsa_status st = geometry(B, H, NQB, NKB, bq, bk, gqa_group, d, chunks, &G);
  if (st != BSA_OK) return st;
  if (buffer_bytes < G.total) return BSA_ERR_WORKSPACE;
  const int g = gqa_group;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(buffer);
  int32_t* status_d = reinterpret_cast<int32_t*>(base + G.status_off);
  const uint64_t mask_u = (uint64_t)g * NQB * NKB;      // bytes per unit
  const uint64_t q_u = (uint64_t)g * G.Nq * d * 2;
  const uint64_t kv_u = (uint64_t)G.Nk * d * 2;
  const uint64_t lse_u = (uint64_t)g * G.Nq * 4;

  PipeObjects P;
  if (!P.create()) return BSA_ERR_CUDA;
  // Both side streams start after everything already enqueued on the caller's
  // stream (the buffer may still be in use by an earlier call).
  if (cudaEventRecord(P.start, user) != cudaSuccess ||
      cudaStreamWaitEvent(P.in, P.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(P.out, P.start, 0) != cudaSuccess ||
      cudaMemsetAsync(status_d, 0, 24ull * G.chunks, user) != cudaSuccess)
    return BSA_ERR_CUDA;

  for (int i = 0; i < G.chunks; ++i) {
    const int s = i & 1;
    const int u0 = i * G.per;
    const int nu = (G.units - u0) < G.per ? (G.units - u0) : G.per;
    uint8_t* sb = base + (uint64_t)s * G.slot.bytes;
    // Inputs of chunk i into slot s, once chunk i-2 has computed from it.
    if (i >= 2 && cudaStreamWaitEvent(P.in, P.comp[s], 0) != cudaSuccess) return BSA_ERR_CUDA;
    if (cudaMemcpyAsync(sb + G.slot.mask, mask + (uint64_t)u0 * mask_u, nu * mask_u,
                        cudaMemcpyHostToDevice, P.in) != cudaSuccess ||
        cudaMemcpyAsync(sb + G.slot.q, static_cast<const uint8_t*>(Q) + (uint64_t)u0 * q_u, nu * q_u,
                        cudaMemcpyHostToDevice, P.in) != cudaSuccess ||
        cudaMemcpyAsync(sb + G.slot.k, static_cast<const uint8_t*>(K) + (uint64_t)u0 * kv_u, nu * kv_u,
                        cudaMemcpyHostToDevice, P.in) != cudaSuccess ||
        cudaMemcpyAsync(sb + G.slot.v, static_cast<const uint8_t*>(V) + (uint64_t)u0 * kv_u, nu * kv_u,
                        cudaMemcpyHostToDevice, P.in) != cudaSuccess ||
        cudaEventRecord(P.h2d[s], P.in) != cudaSuccess)
      return BSA_ERR_CUDA;
    // Plan + forward on the caller's stream, once the inputs are in and the
    // output of chunk i-2 has left the slot.
    if (cudaStreamWaitEvent(user, P.h2d[s], 0) != cudaSuccess) return BSA_ERR_CUDA;
    if (i >= 2 && cudaStreamWaitEvent(user, P.d2h[s], 0) != cudaSuccess) return BSA_ERR_CUDA;
    bsa_plan* plan = nullptr;
    st = bsa_plan_create(sb + G.slot.mask, 1, nu * g, NQB, NKB, bq, bk, g, sb + G.slot.ws,
                         (size_t)(G.slot.bytes - G.slot.ws), BSA_PLAN_NO_UNION, user, &plan);
    if (st != BSA_OK) return st;
    bsa_plan_layout L;
    bsa_plan_get_layout(plan, &L);
    st = bsa_forward(plan, sb + G.slot.q, sb + G.slot.k, sb + G.slot.v, sb + G.slot.o,
                     reinterpret_cast<float*>(sb + G.slot.lse), d, scale, user);
    bsa_plan_destroy(plan);
    if (st != BSA_OK) return st;
    // Keep the chunk's control words 1..6 -- among them the forward's and the
    // key-norm pass's status (the next chunk in this slot resets them).
    if (cudaMemcpyAsync(status_d + 6 * i, sb + G.slot.ws + L.off_control + 4 * kCtlStatus, 24,
                        cudaMemcpyDeviceToDevice, user) != cudaSuccess ||
        cudaEventRecord(P.comp[s], user) != cudaSuccess)
      return BSA_ERR_CUDA;
    // Outputs of chunk i back to the host.
    if (cudaStreamWaitEvent(P.out, P.comp[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(O) + (uint64_t)u0 * q_u, sb + G.slot.o, nu * q_u,
                        cudaMemcpyDeviceToHost, P.out) != cudaSuccess ||
        cudaMemcpyAsync(reinterpret_cast<uint8_t*>(LSE) + (uint64_t)u0 * lse_u, sb + G.slot.lse,
                        nu * lse_u, cudaMemcpyDeviceToHost, P.out) != cudaSuccess ||
        cudaEventRecord(P.d2h[s], P.out) != cudaSuccess)
      return BSA_ERR_CUDA;
  }
  if (cudaEventRecord(P.done, P.out) != cudaSuccess || cudaStreamWaitEvent(user, P.done, 0) != cudaSuccess)
    return BSA_ERR_CUDA;
  // Host outputs are complete once the caller's stream is; report the first
  // chunk whose forward recorded a failure.
  int32_t status_h[6 * 16];
  if (cudaStreamSynchronize(user) != cudaSuccess) return BSA_ERR_CUDA;
  for (int c0 = 0; c0 < G.chunks; c0 += 16) {
    const int n = (G.chunks - c0) < 16 ? (G.chunks - c0) : 16;
    if (cudaMemcpy(status_h, status_d + 6 * c0, 24ull * n, cudaMemcpyDeviceToHost) != cudaSuccess)
      return BSA_ERR_CUDA;
    for (int c = 0; c < n; ++c) {
      const int32_t fwd = status_h[6 * c], knorm = status_h[6 * c + (kCtlKnormStatus - kCtlStatus)];
      if (fwd != 0) return static_cast<bsa_status>(fwd);
      if (knorm != 0) return static_cast<bsa_status>(knorm);
    }
  }
  return BSA_OK;
}
