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
// that device is current, and caches it.  That first call should come before
// any stream capture.
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "sparse_attn.h"

#define SA_API extern "C" __attribute__((visibility("default")))

namespace {
using namespace sa;

static __device__ __align__(256) uint8_t g_plan_scratch[SA_PLAN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;

uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

// Per-device set-up: sm_103 check and the device address of g_plan_scratch.
sa_status scratch_for_current_device(uint8_t** out) {
  static std::mutex mu;
  static uint8_t* addr[kMaxDevices] = {nullptr};
  static signed char state[kMaxDevices] = {0};  // 0 not set up, 1 ready, -1 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (state[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SA_ECUDA;
    if (!(major == 10 && minor == 3)) {
      state[dev] = -1;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr) return SA_ECUDA;
      addr[dev] = static_cast<uint8_t*>(p);
      state[dev] = 1;
    }
  }
  if (state[dev] != 1) return SA_EUNSUPPORTED;
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
  a.g = g;
  // The status area must start at zero on every call; the means are fully
  // overwritten by the pooling kernel.
  if (cudaMemsetAsync(scratch, 0, kStatusBytes, stream) != cudaSuccess) return SA_ECUDA;
  if (launch_pool(a, stream) != cudaSuccess) return SA_ECUDA;
  if (launch_route_topk(a, stream) != cudaSuccess) return SA_ECUDA;
  return SA_OK;
}
