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
#include "sm103_ptx.cuh"

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
  // The call's status words (the plan itself records no error) are zeroed
  // here instead of by a separate memset.
  if (a.status != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < kStatusBytes / 4)
    a.status[threadIdx.x] = 0;
  // The dependent routing grid may be launched once every pool CTA runs.
  griddep_launch_dependents();
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

// Scores of one staged key chunk (keys j0 ..): thread (qg, kg) takes query
// blocks qg*QPT .. +QPT-1 and keys kg + NKG*e, e < KPT, of the chunk, each
// s = sum_d Qmean[d] Kmean[d] in FP32, d = 0..127 in order, times 1/sqrt(128).
// The query values are broadcast reads, the key values come from padded rows
// (consecutive lanes take consecutive keys, so the reads are conflict-free).
template <int QB, int QPT, int KPT>
__device__ __forceinline__ void score_tile(const float* qcT, const float* kcs, float* sc, int nvk, int j0,
                                           int tid) {
  constexpr int NQG = QB / QPT;             // query groups
  constexpr int NKG = kRouteThreads / NQG;  // key groups
  const int kg = tid % NKG;
  const int qg = tid / NKG;
  const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
  // a thread whose first key is past the end has no key in this chunk
  if (j0 + kg >= nvk) return;
  float acc[QPT][KPT];
#pragma unroll
  for (int q = 0; q < QPT; ++q)
#pragma unroll
    for (int e = 0; e < KPT; ++e) acc[q][e] = 0.f;
#pragma unroll 8
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
    if (j < nvk) {
#pragma unroll
      for (int q = 0; q < QPT; ++q) sc[(qg * QPT + q) * nvk + j] = acc[q][e] * inv_sqrt_d;
    }
  }
}

// One CTA per (QB query blocks, head).
// Phase 1: the QB x nvk score strip in shared memory, staged 128 Kmean rows
// at a time (score_tile: QPT query blocks x KPT key blocks per thread for a
// full chunk, one key per thread for a short last chunk).
// Phase 2: one warp per query block turns its scores into order-preserving
// keys (forced local blocks become key 0, below every score), finds the
// K'-th largest key exactly by a bitwise radix search (keys held in
// registers, KPL per lane, when the row fits; else read from shared memory)
// and emits the sorted union of forced local blocks, selected blocks and
// sinks.
template <int QB, int QPT, int KPT, int KPL>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(PlanArgs a) {
  static_assert((kRouteThreads / (QB / QPT)) * KPT == kKeyChunk, "chunk mapping");
  griddep_wait();  // the block means of the pool grid
  const Geometry& g = a.g;
  extern __shared__ __align__(16) float rsm[];
  float* qcT = rsm;                              // [128][QB]
  float* kcs = qcT + kHeadDim * QB;              // [128][129]
  float* sc = kcs + kKeyChunk * kKcStride;       // [QB][nvk]
  const int h = blockIdx.y;
  const int i0 = blockIdx.x * QB;
  const int tid = threadIdx.x;

  // Qmean strip, transposed: consecutive lanes take consecutive query blocks
  // (conflict-free stores); all of a thread's loads are issued before its
  // stores.
  {
    constexpr int kTot = QB * (kHeadDim / 4);
    constexpr int kPer = (kTot + kRouteThreads - 1) / kRouteThreads;
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kRouteThreads;
      const int qi = e % QB, d4 = e / QB;
      const int i = i0 + qi;
      v[u] = (e < kTot && i < g.nq)
                 ? *reinterpret_cast<const float4*>(a.qc + (static_cast<size_t>(h) * g.nq + i) * kHeadDim + 4 * d4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kRouteThreads;
      if (e >= kTot) break;
      const int qi = e % QB, d4 = e / QB;
      qcT[(4 * d4 + 0) * QB + qi] = v[u].x;
      qcT[(4 * d4 + 1) * QB + qi] = v[u].y;
      qcT[(4 * d4 + 2) * QB + qi] = v[u].z;
      qcT[(4 * d4 + 3) * QB + qi] = v[u].w;
    }
  }

  for (int j0 = 0; j0 < g.nvk; j0 += kKeyChunk) {
    __syncthreads();
    // Kmean chunk: loads in batches of 8 per thread, then the stores.
    constexpr int kPerK = kKeyChunk * (kHeadDim / 4) / kRouteThreads;
    static_assert(kPerK % 8 == 0, "Kmean fill mapping");
#pragma unroll 1
    for (int u0 = 0; u0 < kPerK; u0 += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = tid + (u0 + u) * kRouteThreads;
        const int j = j0 + e / (kHeadDim / 4), c4 = e % (kHeadDim / 4);
        v[u] = (j < g.nvk) ? *reinterpret_cast<const float4*>(a.kc + (static_cast<size_t>(h) * g.nvk + j) * kHeadDim + 4 * c4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = tid + (u0 + u) * kRouteThreads;
        float* dst = kcs + (e / (kHeadDim / 4)) * kKcStride + 4 * (e % (kHeadDim / 4));
        dst[0] = v[u].x; dst[1] = v[u].y; dst[2] = v[u].z; dst[3] = v[u].w;
      }
    }
    __syncthreads();
    const int nk = min(kKeyChunk, g.nvk - j0);
    // A short last chunk takes one key per thread (more query blocks per
    // thread) so that every thread has work; each score is the same ordered
    // FP32 sum whichever tile computes it.
    if (nk == kKeyChunk) {
      score_tile<QB, QPT, KPT>(qcT, kcs, sc, g.nvk, j0, tid);
    } else if (QB % 2 == 0 && nk <= kRouteThreads * 2 / QB && QPT > 2) {
      score_tile<QB, 2, 1>(qcT, kcs, sc, g.nvk, j0, tid);
    } else if (QB % 4 == 0 && nk <= kRouteThreads * 4 / QB && QPT > 4) {
      score_tile<QB, (QB % 4 == 0 ? 4 : 2), 1>(qcT, kcs, sc, g.nvk, j0, tid);
    } else if (QB % 8 == 0 && nk <= kRouteThreads * 8 / QB && (QPT > 8 || KPT > 1)) {
      score_tile<QB, (QB % 8 == 0 ? 8 : 2), 1>(qcT, kcs, sc, g.nvk, j0, tid);
    } else {
      score_tile<QB, QPT, KPT>(qcT, kcs, sc, g.nvk, j0, tid);
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
  // Per query block i: forced local range [lo, hi], budget kp.
  struct Row {
    int i, lo, hi, kp;
    bool take_all;
  };
  auto row_of = [&](int qi) {
    Row r;
    r.i = i0 + qi;
    r.lo = max(0, r.i - g.R);
    r.hi = min(g.nvk - 1, r.i + g.R);
    const int ncand = g.nvk - max(0, r.hi - r.lo + 1);
    r.kp = min(g.K, ncand);
    r.take_all = (r.kp == ncand);
    return r;
  };
  // Writes row r's sorted list: `key_of(j)` gives block j's key (j < nvk).
  // Keys above tau are taken, keys equal to tau lowest index first until
  // `need` of them are, forced local blocks and sinks always.
  auto emit_row = [&](const Row& r, uint32_t tau, int need, auto key_of) {
    int32_t* out = a.idx + (static_cast<size_t>(h) * g.nq + r.i) * g.maxl;
    int pos = 0, eq_seen = 0;
    for (int j0 = 0; j0 < g.nblk; j0 += 32) {
      const int j = j0 + lane;
      bool sel = false, eq = false;
      if (j < g.nvk) {
        if ((j >= r.lo && j <= r.hi) || r.take_all) {
          sel = true;
        } else {
          const uint32_t kk = key_of(j0, j);
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
    if (lane == 0) a.cnt[static_cast<size_t>(h) * g.nq + r.i] = pos;
  };
  constexpr int kWarps = kRouteThreads / 32;
  if constexpr (KPL > 0) {
    // Keys in registers (lane owns blocks lane + 32 m).  The warp's rows
    // qi = warp + 8 r are searched RI at a time: their bitwise searches are
    // independent, so their warp reductions overlap.
    constexpr int RPW = QB / kWarps;
    constexpr int RI = (KPL <= 16) ? RPW : (RPW < 2 ? RPW : 2);
    static_assert(RPW % RI == 0, "rows per warp");
#pragma unroll 1
    for (int r0 = 0; r0 < RPW; r0 += RI) {
      Row rw[RI];
      uint32_t kr[RI][KPL];
      uint32_t tau[RI];
      int need[RI];
#pragma unroll
      for (int r = 0; r < RI; ++r) {
        const int qi = warp + kWarps * (r0 + r);
        rw[r] = row_of(qi);
        const bool live = rw[r].i < g.nq;
        if (!live) rw[r].take_all = true;  // nothing to search
        const float* srow = sc + qi * g.nvk;
#pragma unroll
        for (int m = 0; m < KPL; ++m) {
          const int j = lane + 32 * m;
          const bool cand = live && j < g.nvk && (j < rw[r].lo || j > rw[r].hi);
          kr[r][m] = cand ? order_key(srow[j]) : 0u;
        }
        tau[r] = 0;
      }
      // Largest tau with #{keys >= tau} >= kp, bit by bit.
#pragma unroll 1
      for (int bit = 31; bit >= 0; --bit) {
        unsigned c[RI];
#pragma unroll
        for (int r = 0; r < RI; ++r) {
          const uint32_t t = tau[r] | (1u << bit);
          c[r] = 0;
#pragma unroll
          for (int m = 0; m < KPL; ++m) c[r] += (kr[r][m] >= t) ? 1u : 0u;
        }
#pragma unroll
        for (int r = 0; r < RI; ++r) c[r] = __reduce_add_sync(0xFFFFFFFFu, c[r]);
#pragma unroll
        for (int r = 0; r < RI; ++r)
          if (static_cast<int>(c[r]) >= rw[r].kp) tau[r] |= (1u << bit);
      }
      {
        unsigned c[RI];
#pragma unroll
        for (int r = 0; r < RI; ++r) {
          c[r] = 0;
#pragma unroll
          for (int m = 0; m < KPL; ++m) c[r] += (kr[r][m] > tau[r]) ? 1u : 0u;
        }
#pragma unroll
        for (int r = 0; r < RI; ++r) need[r] = rw[r].kp - static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, c[r]));
      }
#pragma unroll
      for (int r = 0; r < RI; ++r) {
        if (rw[r].i >= g.nq) continue;
        const float* srow = sc + (warp + kWarps * (r0 + r)) * g.nvk;
        emit_row(rw[r], tau[r], need[r], [&](int, int j) { return order_key(srow[j]); });
      }
    }
  } else {
    // Keys in shared memory (long rows), one row at a time.
    for (int qi = warp; qi < QB; qi += kWarps) {
      const Row rw = row_of(qi);
      if (rw.i >= g.nq) break;
      uint32_t* krow = reinterpret_cast<uint32_t*>(sc + qi * g.nvk);
      for (int j = lane; j < g.nvk; j += 32) {
        const float f = __uint_as_float(krow[j]);
        krow[j] = (j >= rw.lo && j <= rw.hi) ? 0u : order_key(f);
      }
      __syncwarp();
      uint32_t tau = 0;
      int need = 0;
      if (!rw.take_all) {
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t t = tau | (1u << bit);
          unsigned c = 0;
          for (int j = lane; j < g.nvk; j += 32) c += (krow[j] >= t) ? 1u : 0u;
          if (static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, c)) >= rw.kp) tau = t;
        }
        unsigned c = 0;
        for (int j = lane; j < g.nvk; j += 32) c += (krow[j] > tau) ? 1u : 0u;
        need = rw.kp - static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, c));
      }
      emit_row(rw, tau, need, [&](int, int j) { return krow[j]; });
    }
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
                          static_cast<size_t>(qb) * g.nvk);
}

cudaError_t launch_pool(const PlanArgs& a, cudaStream_t s) {
  const int nb = a.g.nq > a.g.nvk ? a.g.nq : a.g.nvk;
  const int vpr = a.g.H * (kHeadDim / 8);
  const int nchunks = (vpr + kPoolThreads - 1) / kPoolThreads;
  pool_kernel<<<dim3(nb * nchunks, 2), kPoolThreads, 0, s>>>(a, nchunks);
  return cudaGetLastError();
}

template <int QB, int QPT, int KPT, int KPL>
static cudaError_t launch_route_variant(const PlanArgs& a, size_t smem, cudaStream_t s) {
  auto* k = route_topk_kernel<QB, QPT, KPT, KPL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // the pool grid's programmatic dependent: it starts while the pool grid
  // finishes and waits for it in the kernel
  return launch_dependent(k, dim3((a.g.nq + QB - 1) / QB, a.g.H), dim3(kRouteThreads), smem, s, a);
}

cudaError_t launch_route_topk(const PlanArgs& a, cudaStream_t s) {
  const size_t smem = route_topk_smem_bytes(a.g);
  switch (route_qb(a.g)) {
    case 32:
      if (a.g.nvk <= 128) return launch_route_variant<32, 8, 2, 4>(a, smem, s);
      if (a.g.nvk <= 160) return launch_route_variant<32, 8, 2, 5>(a, smem, s);
      if (a.g.nvk <= 256) return launch_route_variant<32, 8, 2, 8>(a, smem, s);
      if (a.g.nvk <= 512) return launch_route_variant<32, 8, 2, 16>(a, smem, s);
      return launch_route_variant<32, 8, 2, 32>(a, smem, s);
    case 16: return launch_route_variant<16, 4, 2, 0>(a, smem, s);
    case 8: return launch_route_variant<8, 4, 1, 0>(a, smem, s);
    default: return launch_route_variant<4, 2, 1, 0>(a, smem, s);
  }
}

}  // namespace sa
