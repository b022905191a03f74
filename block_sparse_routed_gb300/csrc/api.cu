// Host side of the C ABI declared in include/sparse_attn.h: argument
// validation, derived sizes, workspace layout, TMA descriptors and launch
// sequencing.  Every check happens before anything is enqueued; there is no
// fallback path.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "internal.h"
#include "sparse_attn.h"

#define SA_API extern "C" __attribute__((visibility("default")))

namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
}  // namespace

bool sa::cuda_failed(cudaError_t e) {
  if (e == cudaSuccess) return false;
  g_last_cuda_error = e;
  return true;
}

namespace {
using namespace sa;

// Testing hook: launch the attention kernel's single-probe-wait build (see
// sparse_attn_set_single_probe_waits).
std::atomic<int> g_probe_once{0};

constexpr uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

sa_status derive(const sa_params* p, Geometry* g, sa_sizes* out) {
  if (p == nullptr) return SA_EINVAL;
  if (p->abi_version != SA_ABI_VERSION) return SA_EINVAL;
  if (p->B != 1 || p->D != kHeadDim) return SA_EUNSUPPORTED;
  if (p->T < 1 || p->H < 1) return SA_EINVAL;
  if (p->video_tokens < kBlock || p->video_tokens > p->T) return SA_EINVAL;
  if (!(p->topk_ratio > 0.0 && p->topk_ratio <= 1.0)) return SA_EINVAL;
  if (p->radius < 0) return SA_EINVAL;
  if (p->tail_mode != SA_TAIL_DENSE && p->tail_mode != SA_TAIL_PAD) return SA_EINVAL;
  const int64_t T = p->T, H = p->H, Nv = p->video_tokens;
  const int64_t nvk = Nv / kBlock;
  const int64_t tail = Nv - kBlock * nvk;
  const int64_t nblk = (T + kBlock - 1) / kBlock;
  const bool pad = p->tail_mode == SA_TAIL_PAD && tail > 0;
  if (pad && T < kBlock * (nvk + 1)) return SA_EINVAL;
  if (T * H * kHeadDim >= (int64_t(1) << 31)) return SA_EUNSUPPORTED;
  if (nvk > kMaxVideoBlocks) return SA_EUNSUPPORTED;
  const int64_t nq = nvk + (pad ? 1 : 0);
  // K = ceil(r * nvk) taken on the decimal value of r: a relative slack of
  // 1e-9 absorbs the binary representation error of r (0.1 * 30 -> 3).
  const double prod = p->topk_ratio * static_cast<double>(nvk);
  int64_t K = static_cast<int64_t>(std::ceil(prod - 1e-9 * prod));
  if (K < 1) K = 1;
  if (K > nvk) K = nvk;
  const int64_t R = p->radius;
  const int64_t nsink = nblk - nvk;
  const int64_t local = (2 * R + 1 + K < nvk) ? 2 * R + 1 + K : nvk;
  const int64_t maxl = local + nsink;
  if (maxl > kMaxList) return SA_EUNSUPPORTED;
  const int64_t r0 = (p->tail_mode == SA_TAIL_DENSE) ? kBlock * nvk : Nv;
  if (g) {
    g->T = static_cast<int>(T);
    g->H = static_cast<int>(H);
    g->Nv = static_cast<int>(Nv);
    g->nvk = static_cast<int>(nvk);
    g->tail = static_cast<int>(tail);
    g->nblk = static_cast<int>(nblk);
    g->nq = static_cast<int>(nq);
    g->K = static_cast<int>(K);
    g->R = static_cast<int>(R > nvk ? nvk : R);
    g->pad = pad ? 1 : 0;
    g->nsink = static_cast<int>(nsink);
    g->maxl = static_cast<int>(maxl);
    g->r0 = static_cast<int>(r0);
  }
  if (out) {
    out->nvk = static_cast<int32_t>(nvk);
    out->tail = static_cast<int32_t>(tail);
    out->nblk = static_cast<int32_t>(nblk);
    out->nq = static_cast<int32_t>(nq);
    out->topk = static_cast<int32_t>(K);
    out->nsink = static_cast<int32_t>(nsink);
    out->maxl = static_cast<int32_t>(maxl);
    out->dense_row_start = static_cast<int32_t>(r0);
    out->plan_ws_bytes = kStatusBytes + align256(uint64_t(H) * nq * kHeadDim * 4) +
                         align256(uint64_t(H) * nvk * kHeadDim * 4);
    out->fwd_ws_bytes = kStatusBytes + align256(uint64_t(T) * 4);
  }
  return SA_OK;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Per-device check that the current device is an sm_103 part (this library
// carries sm_103a code only).  Cached: one attribute query per device.
sa_status check_device() {
  static std::mutex mu;
  static signed char state[128] = {0};  // 0 unknown, 1 ok, -1 unsupported
  int dev = 0;
  if (cuda_failed(cudaGetDevice(&dev))) return SA_ECUDA;
  if (dev < 0 || dev >= 128) return SA_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (state[dev] == 0) {
    int major = 0, minor = 0;
    if (cuda_failed(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        cuda_failed(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)))
      return SA_ECUDA;
    state[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return state[dev] == 1 ? SA_OK : SA_EUNSUPPORTED;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
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

// 2-D view [rows, cols] of a row-major BF16 tensor, box of 64 columns (128
// bytes, one swizzle row) x box_rows rows, 128-byte swizzle, zero fill past
// the last row.
bool make_map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T rows, H*128 columns] view of a BF16 [T, H, 128] tensor.
bool make_map(CUtensorMap* m, const void* ptr, const Geometry& g, uint32_t box_rows) {
  return make_map_2d(m, ptr, static_cast<uint64_t>(g.T), static_cast<uint64_t>(g.H) * kHeadDim, box_rows);
}

// Workspace of the merged (Spark) forward, after the 256-byte status area.
struct SparkLayout {
  uint64_t b2, anchor, partial, ak, av, lm, lm2, vbias, total;
  int nch, nblkp, vstride;
};
SparkLayout spark_layout(const Geometry& g) {
  SparkLayout L;
  const uint64_t H = g.H, nblk = g.nblk;
  L.nch = anchor_chunks(g.Nv);
  L.nblkp = ((g.nvk + kBlock - 1) / kBlock) * kBlock;
  uint64_t off = kStatusBytes;
  L.b2 = off;      off += align256(uint64_t(g.T) * 4);
  L.anchor = off;  off += align256(H * kHeadDim * 2);
  L.partial = off; off += align256(H * L.nch * kHeadDim * 4);
  L.ak = off;      off += align256(H * nblk * kHeadDim * 2);
  L.av = off;      off += align256(H * nblk * kHeadDim * 2);
  L.lm = off;      off += align256(H * nblk * 4);
  L.lm2 = off;     off += align256(H * L.nblkp * 4);
  L.vstride = 2 * L.nblkp;  // nvc chunks x 2 row halves x 64 keys
  L.vbias = off;   off += align256(uint64_t(kMaxMergedCtas) * 2 * L.vstride * 4);
  L.total = off;
  return L;
}

}  // namespace

SA_API sa_status sparse_attn_query(const sa_params* p, sa_sizes* out) {
  if (out == nullptr) return SA_EINVAL;
  return derive(p, nullptr, out);
}

SA_API sa_status sparse_attn_plan(const sa_params* p, const void* q, const void* k, int32_t* idx,
                                  int32_t* cnt, float* route_scores, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  Geometry g;
  sa_sizes sz;
  sa_status st = derive(p, &g, &sz);
  if (st != SA_OK) return st;
  if (!q || !k || !idx || !cnt || !ws) return SA_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(idx, 4) || !aligned(cnt, 4) ||
      !aligned(ws, 256) || (route_scores && !aligned(route_scores, 4)))
    return SA_EINVAL;
  if (ws_bytes < sz.plan_ws_bytes) return SA_EINVAL;
  st = check_device();
  if (st != SA_OK) return st;

  uint8_t* w = static_cast<uint8_t*>(ws);
  PlanArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.qc = reinterpret_cast<float*>(w + kStatusBytes);
  a.kc = reinterpret_cast<float*>(w + kStatusBytes +
                                  align256(uint64_t(g.H) * g.nq * kHeadDim * 4));
  a.idx = idx;
  a.cnt = cnt;
  a.scores = route_scores;
  a.status = reinterpret_cast<int32_t*>(w);  // zeroed by the pool kernel
  a.g = g;
  if (cuda_failed(launch_pool(a, stream))) return SA_ECUDA;
  if (cuda_failed(launch_route_topk(a, stream))) return SA_ECUDA;
  return SA_OK;
}

SA_API sa_status sparse_attn_fwd(const sa_params* p, const void* q, const void* k, const void* v,
                                 const float* key_bias, const int32_t* idx, const int32_t* cnt,
                                 void* o, void* ws, size_t ws_bytes, cudaStream_t stream) {
  Geometry g;
  sa_sizes sz;
  sa_status st = derive(p, &g, &sz);
  if (st != SA_OK) return st;
  if (!q || !k || !v || !idx || !cnt || !o || !ws) return SA_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 32) ||
      !aligned(idx, 4) || !aligned(cnt, 4) || !aligned(ws, 256) ||
      (key_bias && !aligned(key_bias, 4)))
    return SA_EINVAL;
  if (ws_bytes < sz.fwd_ws_bytes) return SA_EINVAL;
  st = check_device();
  if (st != SA_OK) return st;

  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, g, 128) || !make_map(&tk, k, g, 64) || !make_map(&tv, v, g, 64))
    return SA_ECUDA;

  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  float* b2 = key_bias ? reinterpret_cast<float*>(w + kStatusBytes) : nullptr;
  if (cuda_failed(cudaMemsetAsync(ws, 0, kStatusBytes, stream))) return SA_ECUDA;
  if (key_bias && cuda_failed(launch_bias_prep(key_bias, b2, status, g, stream))) return SA_ECUDA;

  AttnArgs a;
  a.idx = idx;
  a.cnt = cnt;
  a.b2 = b2;
  a.o = static_cast<uint16_t*>(o);
  a.status = status;
  a.unit_counter = status + 1;  // inside the status area, cleared above
  a.bias_nz = status + 2;
  a.g = g;
  a.n_dense = (g.T - g.r0 + 127) / 128;
  a.n_pairs = (g.nq + 1) / 2;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
  a.merged = 0;
  a.lm2 = nullptr;
  a.nblkp = 0;
  a.vbias = nullptr;
  a.vstride = 0;
  a.fused = 0;
  a.qc = a.kc = nullptr;
  a.idx_w = a.cnt_w = nullptr;
  a.probe_once = g_probe_once.load();
  // the summary maps are unused without merging
  if (cuda_failed(launch_attention(tq, tk, tv, tk, tv, a, stream))) return SA_ECUDA;
  return SA_OK;
}

// Workspace of the fused call, after the 256-byte status area: key bias in
// log2 units [T], Qmean [H, nq, 128], Kmean [H, nvk, 128].
struct FusedLayout {
  uint64_t b2, qc, kc, total;
};
FusedLayout fused_layout(const Geometry& g) {
  FusedLayout L;
  uint64_t off = kStatusBytes;
  L.b2 = off; off += align256(uint64_t(g.T) * 4);
  L.qc = off; off += align256(uint64_t(g.H) * g.nq * kHeadDim * 4);
  L.kc = off; off += align256(uint64_t(g.H) * g.nvk * kHeadDim * 4);
  L.total = off;
  return L;
}

SA_API sa_status sparse_attn_fused_ws_bytes(const sa_params* p, uint64_t* out) {
  if (out == nullptr) return SA_EINVAL;
  Geometry g;
  const sa_status st = derive(p, &g, nullptr);
  if (st != SA_OK) return st;
  if (g.nvk > kMaxFusedVideoBlocks) return SA_EUNSUPPORTED;
  *out = fused_layout(g).total;
  return SA_OK;
}

SA_API sa_status sparse_attn_fused(const sa_params* p, const void* q, const void* k, const void* v,
                                   const float* key_bias, int32_t* idx, int32_t* cnt, void* o, void* ws,
                                   size_t ws_bytes, cudaStream_t stream) {
  Geometry g;
  sa_sizes sz;
  sa_status st = derive(p, &g, &sz);
  if (st != SA_OK) return st;
  if (g.nvk > kMaxFusedVideoBlocks) return SA_EUNSUPPORTED;
  if (!q || !k || !v || !idx || !cnt || !o || !ws) return SA_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 32) ||
      !aligned(idx, 4) || !aligned(cnt, 4) || !aligned(ws, 256) ||
      (key_bias && !aligned(key_bias, 4)))
    return SA_EINVAL;
  const FusedLayout L = fused_layout(g);
  if (ws_bytes < L.total) return SA_EINVAL;
  st = check_device();
  if (st != SA_OK) return st;

  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, g, 128) || !make_map(&tk, k, g, 64) || !make_map(&tv, v, g, 64))
    return SA_ECUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  float* b2 = key_bias ? reinterpret_cast<float*>(w + L.b2) : nullptr;
  if (cuda_failed(cudaMemsetAsync(ws, 0, kStatusBytes, stream))) return SA_ECUDA;
  // block means (the routing kernel's first half); the route runs in the
  // attention kernel's scheduler
  PlanArgs pa;
  pa.q = static_cast<const uint16_t*>(q);
  pa.k = static_cast<const uint16_t*>(k);
  pa.qc = reinterpret_cast<float*>(w + L.qc);
  pa.kc = reinterpret_cast<float*>(w + L.kc);
  pa.idx = idx;
  pa.cnt = cnt;
  pa.scores = nullptr;
  pa.status = nullptr;  // zeroed above (the attention kernel's counter too)
  pa.g = g;
  if (cuda_failed(launch_pool(pa, stream))) return SA_ECUDA;
  if (key_bias && cuda_failed(launch_bias_prep(key_bias, b2, status, g, stream))) return SA_ECUDA;

  AttnArgs a;
  a.idx = idx;
  a.cnt = cnt;
  a.b2 = b2;
  a.o = static_cast<uint16_t*>(o);
  a.status = status;
  a.unit_counter = status + 1;  // inside the status area, cleared above
  a.bias_nz = status + 2;
  a.g = g;
  a.n_dense = (g.T - g.r0 + 127) / 128;
  a.n_pairs = (g.nq + 1) / 2;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
  a.merged = 0;
  a.lm2 = nullptr;
  a.nblkp = 0;
  a.vbias = nullptr;
  a.vstride = 0;
  a.fused = 1;
  a.qc = pa.qc;
  a.kc = pa.kc;
  a.idx_w = idx;
  a.cnt_w = cnt;
  a.probe_once = g_probe_once.load();
  if (cuda_failed(launch_attention(tq, tk, tv, tk, tv, a, stream))) return SA_ECUDA;
  return SA_OK;
}

SA_API sa_status sparse_attn_spark_ws_bytes(const sa_params* p, uint64_t* out) {
  if (out == nullptr) return SA_EINVAL;
  Geometry g;
  const sa_status st = derive(p, &g, nullptr);
  if (st != SA_OK) return st;
  const uint64_t nblk = g.nblk;
  if (uint64_t(g.H) * nblk * kHeadDim >= (uint64_t(1) << 31)) return SA_EUNSUPPORTED;
  *out = spark_layout(g).total;
  return SA_OK;
}

SA_API sa_status sparse_attn_spark_fwd(const sa_params* p, const void* q, const void* k, const void* v,
                                       const float* key_bias, const int32_t* idx, const int32_t* cnt,
                                       void* o, void* ws, size_t ws_bytes, cudaStream_t stream) {
  Geometry g;
  sa_sizes sz;
  sa_status st = derive(p, &g, &sz);
  if (st != SA_OK) return st;
  if (uint64_t(g.H) * uint64_t(g.nblk) * kHeadDim >= (uint64_t(1) << 31)) return SA_EUNSUPPORTED;
  if (!q || !k || !v || !idx || !cnt || !o || !ws) return SA_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 32) ||
      !aligned(idx, 4) || !aligned(cnt, 4) || !aligned(ws, 256) ||
      (key_bias && !aligned(key_bias, 4)))
    return SA_EINVAL;
  const SparkLayout L = spark_layout(g);
  if (ws_bytes < L.total) return SA_EINVAL;
  st = check_device();
  if (st != SA_OK) return st;

  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* anchor = reinterpret_cast<uint16_t*>(w + L.anchor);
  uint16_t* ak = reinterpret_cast<uint16_t*>(w + L.ak);
  uint16_t* av = reinterpret_cast<uint16_t*>(w + L.av);
  float* lm = reinterpret_cast<float*>(w + L.lm);
  float* lm2 = reinterpret_cast<float*>(w + L.lm2);
  CUtensorMap tq, tk, tv, tak, tav;
  if (!make_map(&tq, q, g, 128) || !make_map(&tk, k, g, 64) || !make_map(&tv, v, g, 64) ||
      !make_map_2d(&tak, ak, uint64_t(g.H) * g.nblk, kHeadDim, 64) ||
      !make_map_2d(&tav, av, uint64_t(g.H) * g.nblk, kHeadDim, 64))
    return SA_ECUDA;

  int32_t* status = reinterpret_cast<int32_t*>(w);
  float* b2 = key_bias ? reinterpret_cast<float*>(w + L.b2) : nullptr;
  if (cuda_failed(cudaMemsetAsync(ws, 0, kStatusBytes, stream))) return SA_ECUDA;
  if (key_bias && cuda_failed(launch_bias_prep(key_bias, b2, status, g, stream))) return SA_ECUDA;
  // the per-head anchor, its summaries of every block, the log-mass in log2
  if (cuda_failed(launch_video_query_mean(static_cast<const uint16_t*>(q),
                                          reinterpret_cast<float*>(w + L.partial), anchor, g.H, g.Nv,
                                          stream)))
    return SA_ECUDA;
  ReweightArgs r;
  r.a = anchor;
  r.k = static_cast<const uint16_t*>(k);
  r.v = static_cast<const uint16_t*>(v);
  r.ak = ak;
  r.av = av;
  r.lm = lm;
  r.T = g.T;
  r.H = g.H;
  r.P = 1;
  r.nblk = g.nblk;
  r.lm2 = lm2;  // the log2 row for the attention kernel, written alongside lm
  r.nvk = g.nvk;
  r.nblkp = L.nblkp;
  if (cuda_failed(launch_spark_reweight(r, stream))) return SA_ECUDA;

  AttnArgs a;
  a.idx = idx;
  a.cnt = cnt;
  a.b2 = b2;
  a.o = static_cast<uint16_t*>(o);
  a.status = status;
  a.unit_counter = status + 1;  // inside the status area, cleared above
  a.bias_nz = status + 2;
  a.g = g;
  a.n_dense = (g.T - g.r0 + 127) / 128;
  a.n_pairs = (g.nq + 1) / 2;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
  a.merged = 1;
  a.lm2 = lm2;
  a.nblkp = L.nblkp;
  a.vbias = reinterpret_cast<float*>(w + L.vbias);
  a.vstride = L.vstride;
  a.fused = 0;
  a.qc = a.kc = nullptr;
  a.idx_w = a.cnt_w = nullptr;
  a.probe_once = g_probe_once.load();
  if (cuda_failed(launch_attention(tq, tk, tv, tak, tav, a, stream))) return SA_ECUDA;
  return SA_OK;
}

SA_API sa_status sparse_attn_spark_reweight(const sa_reweight_params* p, const void* a, const void* k,
                                            const void* v, void* ak, void* av, float* lm,
                                            cudaStream_t stream) {
  if (p == nullptr) return SA_EINVAL;
  if (p->abi_version != SA_ABI_VERSION) return SA_EINVAL;
  if (p->B != 1 || p->D != kHeadDim) return SA_EUNSUPPORTED;
  if (p->T < 1 || p->H < 1 || p->P < 1) return SA_EINVAL;
  const int64_t nblk = (static_cast<int64_t>(p->T) + kBlock - 1) / kBlock;
  const int64_t lim = int64_t(1) << 31;
  if (int64_t(p->T) * p->H * kHeadDim >= lim || int64_t(p->P) * p->H * nblk * kHeadDim >= lim)
    return SA_EUNSUPPORTED;
  if (!a || !k || !v || !ak || !av || !lm) return SA_EINVAL;
  if (!aligned(a, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(ak, 16) ||
      !aligned(av, 16) || !aligned(lm, 4))
    return SA_EINVAL;
  const sa_status st = check_device();
  if (st != SA_OK) return st;
  ReweightArgs r;
  r.a = static_cast<const uint16_t*>(a);
  r.k = static_cast<const uint16_t*>(k);
  r.v = static_cast<const uint16_t*>(v);
  r.ak = static_cast<uint16_t*>(ak);
  r.av = static_cast<uint16_t*>(av);
  r.lm = lm;
  r.T = p->T;
  r.H = p->H;
  r.P = p->P;
  r.nblk = static_cast<int>(nblk);
  r.lm2 = nullptr;  // summaries only
  r.nvk = r.nblkp = 0;
  if (cuda_failed(launch_spark_reweight(r, stream))) return SA_ECUDA;
  return SA_OK;
}

namespace {
sa_status check_reblock(const sa_reblock_params* p) {
  if (p == nullptr) return SA_EINVAL;
  if (p->abi_version != SA_ABI_VERSION) return SA_EINVAL;
  if (p->D != kHeadDim) return SA_EUNSUPPORTED;
  if (p->T < 1 || p->H < 1) return SA_EINVAL;
  if (p->fanout < 2 || p->fanout > kReblockMaxFanout || (p->fanout & (p->fanout - 1)) != 0) return SA_EINVAL;
  if (p->landmarks < 2 || p->landmarks > kReblockMaxLandmarks) return SA_EINVAL;
  if (p->token_stride < 0 || p->head_stride < 0 || p->token_stride % 8 != 0 || p->head_stride % 8 != 0)
    return SA_EINVAL;
  if (p->H > 65535 || int64_t(p->T) * p->H >= (int64_t(1) << 31)) return SA_EUNSUPPORTED;
  return SA_OK;
}
}  // namespace

SA_API sa_status sparse_attn_reblock_ws_bytes(const sa_reblock_params* p, uint64_t* out) {
  if (out == nullptr) return SA_EINVAL;
  const sa_status st = check_reblock(p);
  if (st != SA_OK) return st;
  *out = reblock_layout(p->T, p->H).total;
  return SA_OK;
}

SA_API sa_status sparse_attn_spark_reblock(const sa_reblock_params* p, const void* x, int32_t* perm,
                                           int32_t* inv, void* ws, size_t ws_bytes, cudaStream_t stream) {
  sa_status st = check_reblock(p);
  if (st != SA_OK) return st;
  if (!x || !perm || !inv || !ws) return SA_EINVAL;
  if (!aligned(x, 16) || !aligned(perm, 4) || !aligned(inv, 4) || !aligned(ws, 256)) return SA_EINVAL;
  if (ws_bytes < reblock_layout(p->T, p->H).total) return SA_EINVAL;
  st = check_device();
  if (st != SA_OK) return st;
  ReblockArgs r;
  r.x = static_cast<const uint16_t*>(x);
  r.token_stride = p->token_stride;
  r.head_stride = p->head_stride;
  r.T = p->T;
  r.H = p->H;
  r.fanout = p->fanout;
  r.landmarks = p->landmarks;
  r.perm = perm;
  r.inv = inv;
  r.ws = ws;
  if (cuda_failed(launch_reblock(r, stream))) return SA_ECUDA;
  return SA_OK;
}

SA_API sa_status sparse_attn_last_device_status(const void* ws, cudaStream_t stream,
                                                sa_status* out) {
  if (!ws || !out) return SA_EINVAL;
  int32_t v = 0;
  if (cuda_failed(cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, stream)))
    return SA_ECUDA;
  if (cuda_failed(cudaStreamSynchronize(stream))) return SA_ECUDA;
  *out = static_cast<sa_status>(v);
  return SA_OK;
}

SA_API int sparse_attn_set_single_probe_waits(int on) { return g_probe_once.exchange(on ? 1 : 0); }

SA_API int sparse_attn_last_cuda_error(const char** message) {
  const cudaError_t e = g_last_cuda_error;
  if (message) *message = cudaGetErrorString(e);
  return static_cast<int>(e);
}

SA_API const char* sparse_attn_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "SA_OK";
    case SA_EINVAL: return "SA_EINVAL: invalid argument";
    case SA_EUNSUPPORTED: return "SA_EUNSUPPORTED: unsupported shape or device";
    case SA_ENOSINKBIAS: return "SA_ENOSINKBIAS: key bias on a routed video key";
    case SA_ECUDA: return "SA_ECUDA: CUDA error";
    case SA_ETIMEOUT: return "SA_ETIMEOUT: on-device wait timed out";
  }
  return "unknown sa_status";
}
