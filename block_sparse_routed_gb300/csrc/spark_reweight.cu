// Spark virtual summaries (spark_reweight) for sm_103a.
//
// What is computed ("Sol-Attn and Spark for MiniMax-H3", section "Spark
// primitives"; default numerics from section "Spark inference integration"):
// for every anchor a_p (a query representative of head h) and physical
// 64-token block b of K/V, over the block's real keys u (a partial last block
// has fewer),
//     s_u = a_p . k_u / sqrt(128),  w = softmax_u(s)
//     ak  = sum_u w_u k_u,  av = sum_u w_u v_u              stored as BF16
//     lm  = logsumexp_u(s_u) - a_p . ak / sqrt(128)          FP32
// where the ak in lm is the stored BF16 one.
//
// The work is one pass over K and V (HBM-bound for a few anchors).  One warp
// takes one (block, head) pair, consecutive warps the heads of one block so
// that they read adjacent 256-byte row segments.  Lane l owns dimensions
// 4l..4l+3 of every row (8-byte loads, one 256-byte row per warp load).
//   pass 1: for each half of the block (32 keys) each lane forms its
//           4-dimension partial products; a butterfly over 5 lane distances
//           (31 shuffles) leaves lane l with the full dot product of key l of
//           that half.  Meanwhile the V rows are prefetched into L2.  Block
//           maximum and sum of 2^((d - dmax) log2(e)/sqrt(128)) by warp
//           reductions;
//   pass 2: each lane accumulates w_u k_u and w_u v_u over its 4 dimensions,
//           the weights broadcast by shuffle; the K rows come back from L2.
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

constexpr int kRwWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1/sqrt(128)

__device__ __forceinline__ void bf16x4(uint2 w, float (&f)[4]) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xFFFF0000u);
}

// Round-to-nearest-even FP32 -> BF16 pair (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  return x;
}

// One butterfly stage: 2N values per lane -> N, lanes with bit `o` set keep
// the upper half of the keys.
template <int N>
__device__ __forceinline__ void fold(float* v, int lane, int o) {
  const bool upper = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float send = upper ? v[i] : v[i + N];
    const float keep = upper ? v[i + N] : v[i];
    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
  }
}

__global__ void __launch_bounds__(32 * kRwWarps, 2) spark_reweight_kernel(const ReweightArgs r) {
  griddep_launch_dependents();  // the next kernel of the call may be launched
  griddep_wait();               // (each waits for its predecessor's writes)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kRwWarps + warp;
  if (item >= static_cast<int64_t>(r.nblk) * r.H) return;
  const int b = static_cast<int>(item / r.H), h = static_cast<int>(item % r.H);
  const int u0 = b * kBlock;
  const int n = min(kBlock, r.T - u0);
  const size_t stride = static_cast<size_t>(r.H) * (kHeadDim / 4);  // row stride in uint2
  const uint2* krow = reinterpret_cast<const uint2*>(r.k) + (static_cast<size_t>(u0) * r.H + h) * (kHeadDim / 4) + lane;
  const uint2* vrow = reinterpret_cast<const uint2*>(r.v) + (static_cast<size_t>(u0) * r.H + h) * (kHeadDim / 4) + lane;

  for (int p = 0; p < r.P; ++p) {
    float a[4];
    bf16x4(__ldg(reinterpret_cast<const uint2*>(r.a) + (static_cast<size_t>(p) * r.H + h) * (kHeadDim / 4) + lane), a);
    // pass 1: per half, partial dot products of this lane's 4 dimensions
    float dk[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      // all 32 row loads of the half are issued before any is used
      uint2 kw[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int u = 32 * hf + i;
        kw[i] = (u < n) ? __ldg(krow + u * stride) : make_uint2(0u, 0u);
      }
      if (p == 0) {
#pragma unroll 4
        for (int i = 0; i < 32; ++i)
          if (32 * hf + i < n) asm volatile("prefetch.global.L2 [%0];" ::"l"(vrow + (32 * hf + i) * stride));
      }
      float d[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float kf[4];
        bf16x4(kw[i], kf);
        d[i] = fmaf(a[3], kf[3], fmaf(a[2], kf[2], fmaf(a[1], kf[1], a[0] * kf[0])));
      }
      fold<16>(d, lane, 16);
      fold<8>(d, lane, 8);
      fold<4>(d, lane, 4);
      fold<2>(d, lane, 2);
      fold<1>(d, lane, 1);
      dk[hf] = d[0];  // key 32 hf + lane
    }
    const bool ok0 = lane < n, ok1 = 32 + lane < n;
    const float dmax = warp_max(fmaxf(ok0 ? dk[0] : -INFINITY, ok1 ? dk[1] : -INFINITY));
    const float c = kLog2e * kInvSqrtD;
    const float e0 = ok0 ? exp2f((dk[0] - dmax) * c) : 0.f;
    const float e1 = ok1 ? exp2f((dk[1] - dmax) * c) : 0.f;
    const float l = warp_sum(e0 + e1);
    // pass 2: weighted keys and values over this lane's dimensions
    float ak[4] = {0.f, 0.f, 0.f, 0.f}, av[4] = {0.f, 0.f, 0.f, 0.f};
    // 16 keys at a time: their 32 row loads are issued before any is used
#pragma unroll 1
    for (int u0 = 0; u0 < n; u0 += 16) {
      uint2 kw[16], vw[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool in = u0 + i < n;
        kw[i] = in ? __ldg(krow + (u0 + i) * stride) : make_uint2(0u, 0u);
        vw[i] = in ? __ldg(vrow + (u0 + i) * stride) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int u = u0 + i;
        // zero weight past the block end (those rows were not loaded)
        const float w = __shfl_sync(0xFFFFFFFFu, (u < 32) ? e0 : e1, u & 31);
        float kf[4], vf[4];
        bf16x4(kw[i], kf);
        bf16x4(vw[i], vf);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          ak[t] = fmaf(w, kf[t], ak[t]);
          av[t] = fmaf(w, vf[t], av[t]);
        }
      }
    }
    const float inv_l = 1.0f / l;
    uint2 ko, vo;
    ko.x = pack_bf16(ak[0] * inv_l, ak[1] * inv_l);
    ko.y = pack_bf16(ak[2] * inv_l, ak[3] * inv_l);
    vo.x = pack_bf16(av[0] * inv_l, av[1] * inv_l);
    vo.y = pack_bf16(av[2] * inv_l, av[3] * inv_l);
    const size_t orow = ((static_cast<size_t>(p) * r.H + h) * r.nblk + b);
    reinterpret_cast<uint2*>(r.ak)[orow * (kHeadDim / 4) + lane] = ko;
    reinterpret_cast<uint2*>(r.av)[orow * (kHeadDim / 4) + lane] = vo;
    // log-mass against the stored (rounded) summary key
    float kr[4];
    bf16x4(ko, kr);
    const float key = warp_sum(fmaf(a[3], kr[3], fmaf(a[2], kr[2], fmaf(a[1], kr[1], a[0] * kr[0]))));
    const float lmv = (dmax - key) * kInvSqrtD + logf(l);
    if (lane == 0) r.lm[orow] = lmv;
    if (r.lm2 != nullptr && p == 0) {
      // the log2 row the merged attention kernel reads, nblkp entries (the
      // video blocks rounded up to 64): 0 past the video keys, and over any
      // padding past the last block, which the head's last block writes
      float* row2 = r.lm2 + static_cast<size_t>(h) * r.nblkp;
      if (lane == 0 && b < r.nblkp) row2[b] = (b < r.nvk) ? lmv * kLog2e : 0.f;
      if (b == r.nblk - 1)
        for (int j = r.nblk + lane; j < r.nblkp; j += 32) row2[j] = 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_spark_reweight(const ReweightArgs& r, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(r.nblk) * r.H;
  const int64_t grid = (items + kRwWarps - 1) / kRwWarps;
  if (grid == 0) return cudaSuccess;
  return launch_dependent(spark_reweight_kernel, dim3(static_cast<unsigned>(grid)), dim3(32 * kRwWarps), 0, s, r);
}

}  // namespace sa

// ---------------------------------------------------------------- anchors
// One global representative per head: the mean of the target-video query
// rows t < Nv, stored as BF16 ("Sol-Attn and Spark for MiniMax-H3", section
// "Spark inference integration").  Deterministic two-level sum: partial sums
// over row chunks in a fixed order, then the chunks in order.
namespace sa {
namespace {

constexpr int kAnchorRows = 1024;  // rows per partial sum

// grid (chunk, head); thread (slice s = tid % 16, group r = tid / 16) sums
// dimensions 8s..8s+7 over rows r, r+16, ... of the chunk.
__global__ void __launch_bounds__(256) anchor_partial_kernel(const uint16_t* __restrict__ q, float* partial,
                                                             int H, int Nv) {
  griddep_launch_dependents();  // the next kernel of the call may be launched
  griddep_wait();               // (each waits for its predecessor's writes)
  const int c = blockIdx.x, h = blockIdx.y;
  const int s = threadIdx.x % 16, r = threadIdx.x / 16;
  const int t0 = c * kAnchorRows, t1 = min(Nv, t0 + kAnchorRows);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int t = t0 + r; t < t1; t += 16) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(q + (static_cast<size_t>(t) * H + h) * kHeadDim) + s);
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += __uint_as_float(x[i] << 16);
      acc[2 * i + 1] += __uint_as_float(x[i] & 0xFFFF0000u);
    }
  }
  __shared__ float red[16][128];
#pragma unroll
  for (int i = 0; i < 8; ++i) red[r][8 * s + i] = acc[i];
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    float sum = 0.f;
    for (int g = 0; g < 16; ++g) sum += red[g][threadIdx.x];
    partial[(static_cast<size_t>(h) * gridDim.x + c) * kHeadDim + threadIdx.x] = sum;
  }
}

__global__ void anchor_final_kernel(const float* partial, uint16_t* anchor, int nch, int Nv) {
  griddep_launch_dependents();  // the next kernel of the call may be launched
  griddep_wait();               // (each waits for its predecessor's writes)
  const int h = blockIdx.x, d = threadIdx.x;
  float sum = 0.f;
  for (int c = 0; c < nch; ++c) sum += partial[(static_cast<size_t>(h) * nch + c) * kHeadDim + d];
  const float mean = sum / static_cast<float>(Nv);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(mean));
  anchor[static_cast<size_t>(h) * kHeadDim + d] = static_cast<uint16_t>(r & 0xFFFFu);
}

}  // namespace

int anchor_chunks(int Nv) { return (Nv + kAnchorRows - 1) / kAnchorRows; }

cudaError_t launch_video_query_mean(const uint16_t* q, float* partial, uint16_t* anchor, int H, int Nv,
                                    cudaStream_t s) {
  const int nch = anchor_chunks(Nv);
  const cudaError_t e = launch_dependent(anchor_partial_kernel, dim3(nch, H), dim3(256), 0, s, q, partial, H, Nv);
  if (e != cudaSuccess) return e;
  return launch_dependent(anchor_final_kernel, dim3(H), dim3(kHeadDim), 0, s, partial, anchor, nch, Nv);
}

}  // namespace sa
