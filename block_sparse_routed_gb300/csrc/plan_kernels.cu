// Routing kernels: block mean pooling, and route scores + Top-K + block-list
// compaction.
//
// Pooling follows "Sol-Attn and Spark for MiniMax-H3", section "Spark
// inference integration" (native mean Top-K routing): the route centroid of
// a 64-token block is the mean of its rows; in pad mode the tail block's
// centroid is the mean of its real video rows (section "H3 pipeline
// integration").  Route scores are Qmean . Kmean / sqrt(128) in FP32; the
// Top-K boundary is found by an exact radix search over FP32 keys (the same
// page names "exact FP32 radix boundary selection"), ties going to the lower
// block index.  Forced local blocks (self +- radius) are not candidates and
// are added outside the budget; sink blocks are always in the list ("Add key
// bias to chunked Sol-Attn producers", "Tests and source audit").
#include <cstdint>

#include "internal.h"

namespace sa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One CTA per (block, 256-slice column chunk, tensor): blockIdx.y = 0 pools
// Q over the nq query blocks, 1 pools K over the nvk video key blocks.  Each
// thread owns one 16-byte column slice of a token row (8 dims of one head)
// and sums it down the block's rows; consecutive threads read consecutive
// 16-byte slices, so every row is read with full coalescing.  HBM-bound.
constexpr int kPoolThreads = 256;

__global__ void __launch_bounds__(kPoolThreads) pool_kernel(const PlanArgs a, int nchunks) {
  const Geometry g = a.g;
  const bool isq = blockIdx.y == 0;
  const int nblocks = isq ? g.nq : g.nvk;
  const int i = blockIdx.x / nchunks;
  const int chunk = blockIdx.x % nchunks;
  if (i >= nblocks) return;
  const int n = (i < g.nvk) ? kBlock : g.tail;  // the pad tail block owns `tail` rows
  const int vpr = g.H * (kHeadDim / 8);  // 16-byte slices per token row
  const int c = chunk * kPoolThreads + threadIdx.x;
  if (c >= vpr) return;
  const uint4* p = reinterpret_cast<const uint4*>(isq ? a.q : a.k) +
                   static_cast<size_t>(i) * kBlock * vpr + c;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 16
  for (int r = 0; r < n; ++r) {
    const uint4 v = __ldg(p + static_cast<size_t>(r) * vpr);
    acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
    acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
    acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
    acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
  }
  const float fn = static_cast<float>(n);
  const int h = c / (kHeadDim / 8);
  const int d0 = (c % (kHeadDim / 8)) * 8;
  float* dst = isq ? a.qc : a.kc;
  float4* o = reinterpret_cast<float4*>(dst + (static_cast<size_t>(h) * nblocks + i) * kHeadDim + d0);
  o[0] = make_float4(acc[0] / fn, acc[1] / fn, acc[2] / fn, acc[3] / fn);
  o[1] = make_float4(acc[4] / fn, acc[5] / fn, acc[6] / fn, acc[7] / fn);
}

// Order-preserving map of an FP32 score to an unsigned key; -0 and +0 map to
// the same key.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (f == 0.0f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kRouteThreads = 256;
constexpr int kKeyChunk = 128;           // Kmean rows staged per step
constexpr int kKcStride = kHeadDim + 1;  // padded row: conflict-free column reads

// One CTA per (QB query blocks, head).
// Phase 1: the QB x nvk score strip in shared memory.  Each thread owns QPT
// query blocks x KPT key blocks of every 128-key chunk and accumulates
// s = sum_d Qmean[d] Kmean[d] in FP32, d = 0..127 in order; the query values
// are broadcast reads, the key values come from padded rows (consecutive
// lanes take consecutive keys, so the reads are conflict-free).
// Phase 2: one warp per query block turns its scores into order-preserving
// keys (forced local blocks become key 0, below every score), finds the
// K'-th largest key exactly by a most-significant-digit-first radix select
// (four 8-bit digits, a 256-bin histogram per pass) and emits the sorted
// union of forced local blocks, selected blocks and sinks.
template <int QB, int QPT, int KPT>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(PlanArgs a) {
  constexpr int NQG = QB / QPT;              // query groups
  constexpr int NKG = kRouteThreads / NQG;   // key groups
  static_assert(NKG * KPT == kKeyChunk, "chunk mapping");
  const Geometry& g = a.g;
  extern __shared__ __align__(16) float rsm[];
  float* qcT = rsm;                              // [128][QB]
  float* kcs = qcT + kHeadDim * QB;              // [128][129]
  float* sc = kcs + kKeyChunk * kKcStride;       // [QB][nvk]
  int* hist_all = reinterpret_cast<int*>(sc + QB * g.nvk);  // [warps][256]
  const int h = blockIdx.y;
  const int i0 = blockIdx.x * QB;
  const int tid = threadIdx.x;

  for (int e = tid; e < QB * kHeadDim; e += kRouteThreads) {
    const int qi = e / kHeadDim, d = e % kHeadDim;
    const int i = i0 + qi;
    qcT[d * QB + qi] = (i < g.nq) ? a.qc[(static_cast<size_t>(h) * g.nq + i) * kHeadDim + d] : 0.f;
  }

  const int kg = tid % NKG;
  const int qg = tid / NKG;
  const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
  for (int j0 = 0; j0 < g.nvk; j0 += kKeyChunk) {
    __syncthreads();
    for (int e = tid; e < kKeyChunk * (kHeadDim / 4); e += kRouteThreads) {
      const int r = e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
      const int j = j0 + r;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < g.nvk)
        v = *reinterpret_cast<const float4*>(a.kc + (static_cast<size_t>(h) * g.nvk + j) * kHeadDim + 4 * c4);
      float* dst = kcs + r * kKcStride + 4 * c4;
      dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
    }
    __syncthreads();
    float acc[QPT][KPT];
#pragma unroll
    for (int q = 0; q < QPT; ++q)
#pragma unroll
      for (int e = 0; e < KPT; ++e) acc[q][e] = 0.f;
#pragma unroll 4
    for (int d = 0; d < kHeadDim; ++d) {
      float kv[KPT];
#pragma unroll
      for (int e = 0; e < KPT; ++e) kv[e] = kcs[(kg + NKG * e) * kKcStride + d];
      // the QPT query values are contiguous and 8/16-byte aligned: vector loads
      float qv[QPT];
      if constexpr (QPT % 4 == 0) {
#pragma unroll
        for (int q = 0; q < QPT; q += 4) {
          const float4 t = *reinterpret_cast<const float4*>(qcT + d * QB + qg * QPT + q);
          qv[q] = t.x; qv[q + 1] = t.y; qv[q + 2] = t.z; qv[q + 3] = t.w;
        }
      } else {
        static_assert(QPT == 2, "query values per thread");
        const float2 t = *reinterpret_cast<const float2*>(qcT + d * QB + qg * QPT);
        qv[0] = t.x; qv[1] = t.y;
      }
#pragma unroll
      for (int q = 0; q < QPT; ++q)
#pragma unroll
        for (int e = 0; e < KPT; ++e) acc[q][e] = fmaf(qv[q], kv[e], acc[q][e]);
    }
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const int j = j0 + kg + NKG * e;
      if (j < g.nvk) {
#pragma unroll
        for (int q = 0; q < QPT; ++q) sc[(qg * QPT + q) * g.nvk + j] = acc[q][e] * inv_sqrt_d;
      }
    }
  }
  __syncthreads();

  if (a.scores != nullptr) {
    for (int qi = 0; qi < QB; ++qi) {
      const int i = i0 + qi;
      if (i >= g.nq) break;
      float* dst = a.scores + (static_cast<size_t>(h) * g.nq + i) * g.nvk;
      for (int j = tid; j < g.nvk; j += kRouteThreads) dst[j] = sc[qi * g.nvk + j];
    }
    __syncthreads();
  }

  const int warp = tid / 32, lane = tid % 32;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int qi = warp; qi < QB; qi += kRouteThreads / 32) {
    const int i = i0 + qi;
    if (i >= g.nq) break;
    uint32_t* krow = reinterpret_cast<uint32_t*>(sc + qi * g.nvk);
    const int lo = max(0, i - g.R);
    const int hi = min(g.nvk - 1, i + g.R);
    const int nlv = max(0, hi - lo + 1);
    const int ncand = g.nvk - nlv;
    const int kp = min(g.K, ncand);
    const bool take_all = (kp == ncand);
    for (int j = lane; j < g.nvk; j += 32) {
      const float f = __uint_as_float(krow[j]);
      krow[j] = (j >= lo && j <= hi) ? 0u : order_key(f);
    }
    __syncwarp();
    uint32_t tau = 0;
    int need = 0;
    if (!take_all) {
      // Digits of the kp-th largest key, most significant first.  `need`
      // counts how many keys equal to the prefix found so far still have to
      // be taken; the keys above the prefix's bin are already counted out.
      int* hist = hist_all + warp * 256;
      uint32_t prefix = 0, pmask = 0;
      need = kp;
#pragma unroll 1
      for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
        for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0;
        __syncwarp();
        for (int j = lane; j < g.nvk; j += 32) {
          const uint32_t kk = krow[j];
          if ((kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
        }
        __syncwarp();
        // lane l owns bins 8l..8l+7; count from the top bin down
        int c[8], tot = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) { c[b] = hist[lane * 8 + b]; tot += c[b]; }
        int above = tot;  // keys in this lane's bins and every higher lane's
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_down_sync(0xFFFFFFFFu, above, o);
          if (lane + o < 32) above += v;
        }
        const int higher = above - tot;  // keys in higher lanes' bins
        // the digit's lane: higher < need <= above
        const unsigned own = __ballot_sync(0xFFFFFFFFu, higher < need && need <= above);
        const int src = __ffs(own) - 1;
        int digit = 0, rem = 0;
        if (lane == src) {
          int acc = higher;
          bool found = false;
#pragma unroll
          for (int b = 7; b >= 0; --b) {
            if (!found && acc + c[b] >= need) {
              found = true;
              digit = lane * 8 + b;
              rem = need - acc;
            }
            acc += c[b];
          }
        }
        digit = __shfl_sync(0xFFFFFFFFu, digit, src);
        need = __shfl_sync(0xFFFFFFFFu, rem, src);
        prefix |= static_cast<uint32_t>(digit) << shift;
        pmask |= 255u << shift;
        __syncwarp();
      }
      tau = prefix;
    }
    int32_t* out = a.idx + (static_cast<size_t>(h) * g.nq + i) * g.maxl;
    int pos = 0, eq_seen = 0;
    for (int j0 = 0; j0 < g.nblk; j0 += 32) {
      const int j = j0 + lane;
      bool sel = false, eq = false;
      if (j < g.nvk) {
        if (j >= lo && j <= hi) {
          sel = true;
        } else if (take_all) {
          sel = true;
        } else {
          const uint32_t kk = krow[j];
          if (kk > tau) sel = true;
          else if (kk == tau) eq = true;
        }
      } else if (j < g.nblk) {
        sel = true;  // sink block
      }
      const unsigned eqm = __ballot_sync(0xFFFFFFFFu, eq);
      if (eq) sel = (eq_seen + __popc(eqm & lt_mask)) < need;
      eq_seen += __popc(eqm);
      const unsigned sm = __ballot_sync(0xFFFFFFFFu, sel);
      if (sel) out[pos + __popc(sm & lt_mask)] = j;
      pos += __popc(sm);
    }
    for (int p = pos + lane; p < g.maxl; p += 32) out[p] = -1;
    if (lane == 0) a.cnt[static_cast<size_t>(h) * g.nq + i] = pos;
  }
}

int route_qb(const Geometry& g) {
  if (g.nvk <= 1024) return 32;
  if (g.nvk <= 2048) return 16;
  if (g.nvk <= 4096) return 8;
  return 4;
}

}  // namespace

size_t route_topk_smem_bytes(const Geometry& g) {
  const int qb = route_qb(g);
  return sizeof(float) * (static_cast<size_t>(kHeadDim) * qb + kKeyChunk * kKcStride +
                          static_cast<size_t>(qb) * g.nvk + (kRouteThreads / 32) * 256);
}

cudaError_t launch_pool(const PlanArgs& a, cudaStream_t s) {
  const int nb = a.g.nq > a.g.nvk ? a.g.nq : a.g.nvk;
  const int vpr = a.g.H * (kHeadDim / 8);
  const int nchunks = (vpr + kPoolThreads - 1) / kPoolThreads;
  pool_kernel<<<dim3(nb * nchunks, 2), kPoolThreads, 0, s>>>(a, nchunks);
  return cudaGetLastError();
}

template <int QB, int QPT, int KPT>
static cudaError_t launch_route_variant(const PlanArgs& a, size_t smem, cudaStream_t s) {
  auto* k = route_topk_kernel<QB, QPT, KPT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid((a.g.nq + QB - 1) / QB, a.g.H);
  k<<<grid, kRouteThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_route_topk(const PlanArgs& a, cudaStream_t s) {
  const size_t smem = route_topk_smem_bytes(a.g);
  switch (route_qb(a.g)) {
    case 32: return launch_route_variant<32, 8, 2>(a, smem, s);
    case 16: return launch_route_variant<16, 4, 2>(a, smem, s);
    case 8: return launch_route_variant<8, 4, 1>(a, smem, s);
    default: return launch_route_variant<4, 2, 1>(a, smem, s);
  }
}

}  // namespace sa
