// sparse_attn_plan_static: the routing call with its scratch memory in a
// fixed device array instead of a caller-provided workspace.
//
// Who needs it: code that cannot hand the library device scratch memory.
// Examples are plugins loaded into a host application whose device memory is
// owned by the host's own pool allocator, with no allocation hook offered to
// plugins, and callers that must not call cudaMalloc at this point because it
// synchronises the device.  They still pass Q, K and the output buffers.
//
// The scratch (status word + block means) lives in `g_plan_scratch`, a
// file-scope device array of SA_PLAN_STATIC_SCRATCH_BYTES.  Every GPU that
// loads this library holds that array until the process exits.  All calls
// share it and it keeps the last call's contents, so calls that overlap on
// the GPU (other streams, other host threads) race; the caller serialises
// them.  The host cannot use the array's name as a device address: the first
// call on each device looks the address up with cudaGetSymbolAddress while
// that device is current, and caches it with its context (a new context, as
// after a device reset, is looked up again).  That first call should come
// before any stream capture.
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "internal.h"
#include "sparse_attn.h"

#define SA_API extern "C" __attribute__((visibility("default")))

namespace {
using namespace sa;

static __device__ __align__(256) uint8_t g_plan_scratch[SA_PLAN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;

uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// Set-up per device and context: the sm_103 check and the device address of
// g_plan_scratch, looked up with that device current.  The address is
// cached per device together with the context it was resolved in; when the
// current context is another one (say the device was reset and its primary
// context created again, which loads the module again), it is looked up
// again.  cuCtxGetCurrent is cheap and allowed during stream capture.
sa_status scratch_for_current_device(uint8_t** out) {
  static std::mutex mu;
  static uint8_t* addr[kMaxDevices] = {nullptr};
  static CUcontext ctx_of[kMaxDevices] = {nullptr};
  static signed char state[kMaxDevices] = {0};  // 0 not checked, 1 sm_103, -1 unsupported
  int dev = 0;
  if (cuda_failed(cudaGetDevice(&dev))) return SA_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_EUNSUPPORTED;
  auto get_ctx = ctx_get_current();
  if (!get_ctx) return SA_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (state[dev] == 0) {
    int major = 0, minor = 0;
    if (cuda_failed(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        cuda_failed(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)))
      return SA_ECUDA;
    state[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (state[dev] != 1) return SA_EUNSUPPORTED;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return SA_ECUDA;
  if (ctx == nullptr || ctx != ctx_of[dev] || addr[dev] == nullptr) {
    void* p = nullptr;
    if (cuda_failed(cudaGetSymbolAddress(&p, g_plan_scratch))) return SA_ECUDA;
    if (p == nullptr) return SA_ECUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return SA_ECUDA;  // the runtime may have made the context
    addr[dev] = static_cast<uint8_t*>(p);
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return SA_OK;
}

}  // namespace

SA_API sa_status sparse_attn_plan_static(const sa_params* p, const void* q, const void* k,
                                         int32_t* idx, int32_t* cnt, float* route_scores,
                                         cudaStream_t stream) {
  sa_sizes sz;
  sa_status st = sparse_attn_query(p, &sz);
  if (st != SA_OK) return st;
  if (sz.plan_ws_bytes > SA_PLAN_STATIC_SCRATCH_BYTES) return SA_EUNSUPPORTED;
  if (!q || !k || !idx || !cnt) return SA_EINVAL;
  auto misaligned = [](const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) % a) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(idx, 4) || misaligned(cnt, 4) ||
      (route_scores && misaligned(route_scores, 4)))
    return SA_EINVAL;
  uint8_t* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != SA_OK) return st;

  Geometry g;
  g.T = p->T;
  g.H = p->H;
  g.Nv = p->video_tokens;
  g.nvk = sz.nvk;
  g.tail = sz.tail;
  g.nblk = sz.nblk;
  g.nq = sz.nq;
  g.K = sz.topk;
  g.R = p->radius > sz.nvk ? sz.nvk : p->radius;
  g.pad = sz.nq > sz.nvk ? 1 : 0;
  g.nsink = sz.nsink;
  g.maxl = sz.maxl;
  g.r0 = sz.dense_row_start;

  PlanArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.qc = reinterpret_cast<float*>(scratch + kStatusBytes);
  a.kc = reinterpret_cast<float*>(scratch + kStatusBytes +
                                  align256(uint64_t(g.H) * g.nq * kHeadDim * 4));
  a.idx = idx;
  a.cnt = cnt;
  a.scores = route_scores;
  // The status area starts at zero on every call (the pooling kernel clears
  // it); the means are fully overwritten by the pooling kernel.
  a.status = reinterpret_cast<int32_t*>(scratch);
  a.g = g;
  if (cuda_failed(launch_pool(a, stream))) return SA_ECUDA;
  if (cuda_failed(launch_route_topk(a, stream))) return SA_ECUDA;
  return SA_OK;
}
