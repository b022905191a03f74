// Exact attention over block lists, and dense attention over every key, for
// sm_103a: TMA loads of 64-key K/V blocks into 128-byte-swizzled shared
// memory, QK^T and PV on tcgen05 tensor cores with FP32 accumulators in
// tensor memory, and an online base-2 softmax in registers.
//
// What is computed ("Sol-Attn and Spark for MiniMax-H3", "H3 pipeline
// integration"; "Add key bias to chunked Sol-Attn producers", "Summary" and
// "Contract"): each video query row attends, with one softmax, to every key of
// the blocks in its block list; context rows (and, in dense tail mode, the
// rows of the video block cut by the boundary) attend to every key.  Logits
// are (q . k) / sqrt(128) plus an optional per-key bias that is given in
// natural-log units and converted once to log2 units, so the kernel works in
// base 2 throughout: l2 = (q . k) * log2(e) / sqrt(128) + bias * log2(e).
//
// Work units (one CTA each, two CTAs per SM):
//   * sparse: a pair of consecutive query blocks of one head (128 rows).  The
//     CTA walks the sorted union of the two lists; a key block that is in
//     only one list is masked to -inf for the other block's 64 rows.
//   * dense: 128 consecutive densely evaluated rows of one head, walking all
//     key blocks.
// Warp roles: warp 0 issues TMA loads, warp 1 owns tensor memory and issues
// the MMAs (one thread), warps 2-5 run the softmax (thread = query row =
// tensor-memory lane) and the epilogue.
//
// Tensor memory (256 columns): O accumulator in columns [0, 128); two S
// buffers of 64 FP32 columns at 128 and 192.  After the softmax has read S_j
// it writes P_j as packed BF16 pairs into the first 32 columns of the same
// buffer, and PV_j reads P_j from there (A operand in tensor memory).
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 128;  // S buffer b at kColS + 64 b

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr uint32_t kOffQ = 0;             // Q tile: 2 chunks x [128 rows x 128 B]
constexpr uint32_t kOffK = 32768;         // K stage s: 2 chunks x [64 rows x 128 B]
constexpr uint32_t kOffV = 65536;         // V stage s
constexpr uint32_t kStageBytes = 16384;   // one 64-key block of K (or V)
constexpr uint32_t kOffEnt = 98304;       // union list entries (int32)
constexpr int kMaxEnt = 2 * kMaxList;
constexpr uint32_t kOffBar = kOffEnt + 4 * kMaxEnt;
constexpr uint32_t kOffMisc = kOffBar + 256;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // alignment slack

// Merge scratch lives in the V stages, which are untouched until the list is
// ready.
constexpr uint32_t kOffListA = kOffV;
constexpr uint32_t kOffListB = kOffV + 4 * kMaxList;
constexpr uint32_t kOffMerged = kOffV + 8 * kMaxList;
static_assert(kOffMerged + 4 * kMaxEnt <= kOffEnt, "merge scratch must fit in the V stages");

// Barrier indices (8 bytes each).
enum {
  BAR_Q = 0,
  BAR_KFULL = 1,   // +s
  BAR_VFULL = 3,   // +s
  BAR_KEMPTY = 5,  // +s
  BAR_VEMPTY = 7,  // +s
  BAR_SFULL = 9,   // +b
  BAR_PFULL = 11,  // +b
  BAR_PVDONE = 13, // +b
  BAR_OFULL = 15,
  BAR_DRAIN = 16,
  NUM_BARS = 17
};

constexpr uint32_t kEntMaskShift = 30;
constexpr uint32_t kEntBlockMask = (1u << kEntMaskShift) - 1u;

__device__ __forceinline__ int lower_bound_s(const int32_t* a, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}
__device__ __forceinline__ int upper_bound_s(const int32_t* a, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Packed two-wide FP32 arithmetic and a three-input max (sm_100+ forms).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Max of 64 values: a depth-4 tree of three-input maxima.
__device__ __forceinline__ float max64(const uint32_t (&s)[64]) {
  float m[22];
#pragma unroll
  for (int i = 0; i < 21; ++i)
    m[i] = fmax3(__uint_as_float(s[3 * i]), __uint_as_float(s[3 * i + 1]), __uint_as_float(s[3 * i + 2]));
  m[21] = __uint_as_float(s[63]);
  float n[8];
#pragma unroll
  for (int i = 0; i < 7; ++i) n[i] = fmax3(m[3 * i], m[3 * i + 1], m[3 * i + 2]);
  n[7] = m[21];
  return fmaxf(fmax3(n[0], n[1], n[2]), fmax3(n[3], n[4], fmax3(n[5], n[6], n[7])));
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

__global__ void __launch_bounds__(kThreads, 2)
attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  const Geometry& g = a.g;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  int32_t* ent = reinterpret_cast<int32_t*>(base + kOffEnt);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + kOffMisc);
  volatile int32_t* s_nent = reinterpret_cast<volatile int32_t*>(base + kOffMisc + 8);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(base + kOffMisc + 16);
  volatile int32_t* s_status = reinterpret_cast<volatile int32_t*>(base + kOffMisc + 24);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * i; };

  if (threadIdx.x == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(a.status);
    *s_abort = 0;
    *s_nent = 0;
  }
  __syncthreads();
  if (*s_status != 0) return;  // an earlier step on this stream failed

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // ---- which unit
  const int units_dense = g.H * a.n_dense;
  const bool dense = static_cast<int>(blockIdx.x) < units_dense;
  int h, row0, iA = 0, iB = -1;
  if (dense) {
    h = blockIdx.x / a.n_dense;
    row0 = g.r0 + 128 * (blockIdx.x % a.n_dense);
  } else {
    const int v = blockIdx.x - units_dense;
    h = v / a.n_pairs;
    const int p = v % a.n_pairs;
    iA = 2 * p;
    iB = (2 * p + 1 < g.nq) ? 2 * p + 1 : -1;
    row0 = kBlock * iA;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(BAR_PFULL + 0), 4);
    mbar_init(bar(BAR_PFULL + 1), 4);
    if (dense) *s_nent = g.nblk;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), kTmemCols);
    tmem_relinquish();
  }

  // ---- union of the two block lists (sparse units), warps 2..5
  if (!dense && warp >= 2) {
    const int t2 = threadIdx.x - 64;
    int32_t* la = reinterpret_cast<int32_t*>(base + kOffListA);
    int32_t* lb = reinterpret_cast<int32_t*>(base + kOffListB);
    int32_t* mg = reinterpret_cast<int32_t*>(base + kOffMerged);
    const int nA = a.cnt[static_cast<size_t>(h) * g.nq + iA];
    const int nB = (iB >= 0) ? a.cnt[static_cast<size_t>(h) * g.nq + iB] : 0;
    const bool bad_cnt = nA < 1 || nA > g.maxl || nB < 0 || nB > g.maxl;
    if (!bad_cnt) {
      const int32_t* ga = a.idx + (static_cast<size_t>(h) * g.nq + iA) * g.maxl;
      for (int k = t2; k < nA; k += 128) la[k] = ga[k];
      if (iB >= 0) {
        const int32_t* gb = a.idx + (static_cast<size_t>(h) * g.nq + iB) * g.maxl;
        for (int k = t2; k < nB; k += 128) lb[k] = gb[k];
      }
    }
    named_bar_sync(1, 128);
    // validate: ascending, in range
    bool bad = bad_cnt;
    if (!bad_cnt) {
      for (int k = t2; k < nA; k += 128)
        bad |= la[k] < 0 || la[k] >= g.nblk || (k + 1 < nA && la[k] >= la[k + 1]);
      for (int k = t2; k < nB; k += 128)
        bad |= lb[k] < 0 || lb[k] >= g.nblk || (k + 1 < nB && lb[k] >= lb[k + 1]);
    }
    if (bad) *s_abort = 1;
    named_bar_sync(1, 128);
    if (*s_abort == 0) {
      // stable merge with duplicates: A before an equal B
      for (int k = t2; k < nA; k += 128)
        mg[k + lower_bound_s(lb, nB, la[k])] = la[k] | (1 << kEntMaskShift);
      for (int k = t2; k < nB; k += 128)
        mg[k + upper_bound_s(la, nA, lb[k])] = lb[k] | (2 << kEntMaskShift);
      named_bar_sync(1, 128);
      if (warp == 2) {
        const int n = nA + nB;
        int pos = 0;
        for (int m0 = 0; m0 < n; m0 += 32) {
          const int m = m0 + lane;
          bool keep = false;
          int32_t val = 0;
          if (m < n) {
            const int32_t cur = mg[m];
            const int32_t blk = cur & kEntBlockMask;
            const bool dup_of_prev = m > 0 && (mg[m - 1] & kEntBlockMask) == blk;
            const bool next_same = m + 1 < n && (mg[m + 1] & kEntBlockMask) == blk;
            keep = !dup_of_prev;
            val = next_same ? (blk | (3 << kEntMaskShift)) : cur;
          }
          const unsigned km = __ballot_sync(0xFFFFFFFFu, keep);
          if (keep) ent[pos + __popc(km & ((1u << lane) - 1u))] = val;
          pos += __popc(km);
        }
        if (lane == 0) *s_nent = pos;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (*s_abort != 0) {
    if (threadIdx.x == 0) set_status(a.status, 1 /* SA_EINVAL */);
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int n = *s_nent;
  const uint32_t sQ = sbase + kOffQ;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int xq = h * kHeadDim;
      mbar_arrive_expect_tx(bar(BAR_Q), 2 * 16384);
      tma_load_2d(sQ, &tm_q, bar(BAR_Q), xq, row0);
      tma_load_2d(sQ + 16384, &tm_q, bar(BAR_Q), xq + 64, row0);
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int s = j & 1;
        const uint32_t par = ((j >> 1) & 1) ^ 1;
        const int blk = dense ? j : (ent[j] & kEntBlockMask);
        const int y = blk * kBlock;
        if (!mbar_wait(bar(BAR_KEMPTY + s), par, kWaitLimitNs)) { ok = false; break; }
        const uint32_t sK = sbase + kOffK + s * kStageBytes;
        mbar_arrive_expect_tx(bar(BAR_KFULL + s), kStageBytes);
        tma_load_2d(sK, &tm_k, bar(BAR_KFULL + s), xq, y);
        tma_load_2d(sK + 8192, &tm_k, bar(BAR_KFULL + s), xq + 64, y);
        issued_k = j + 1;
        if (!mbar_wait(bar(BAR_VEMPTY + s), par, kWaitLimitNs)) { ok = false; break; }
        const uint32_t sV = sbase + kOffV + s * kStageBytes;
        mbar_arrive_expect_tx(bar(BAR_VFULL + s), kStageBytes);
        tma_load_2d(sV, &tm_v, bar(BAR_VFULL + s), xq, y);
        tma_load_2d(sV + 8192, &tm_v, bar(BAR_VFULL + s), xq + 64, y);
        issued_v = j + 1;
        if (*s_abort) { ok = false; break; }
      }
      if (!ok) {
        *s_abort = 1;
        set_status(a.status, 5 /* SA_ETIMEOUT */);
        // let copies in flight land before the CTA exits (bounded)
        for (int j = max(0, issued_k - 2); j < issued_k; ++j)
          mbar_wait(bar(BAR_KFULL + (j & 1)), (j >> 1) & 1, kWaitLimitNs);
        for (int j = max(0, issued_v - 2); j < issued_v; ++j)
          mbar_wait(bar(BAR_VFULL + (j & 1)), (j >> 1) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 64, false, false);   // S = Q K^T, both K-major
      const uint32_t id_o = idesc_bf16(128, 128, false, true);   // O += P V, V is MN-major
      bool ok = mbar_wait(bar(BAR_Q), 0, kWaitLimitNs);
      tc_fence_after();
      auto issue_pv = [&](int jj) -> bool {
        const int b = jj & 1;
        const uint32_t par = (jj >> 1) & 1;
        if (!mbar_wait(bar(BAR_PFULL + b), par, kWaitLimitNs)) return false;
        if (!mbar_wait(bar(BAR_VFULL + b), par, kWaitLimitNs)) return false;
        tc_fence_after();
        const uint32_t sV = sbase + kOffV + b * kStageBytes;
        const uint32_t pcol = tmem + kColS + 64u * b;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = sdesc_sw128(sV + kk * 2048, 8192, 1024);
          umma_ts(tmem + kColO, pcol + kk * 8, bd, id_o, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(BAR_VEMPTY + b));
        umma_commit(bar(BAR_PVDONE + b));
        return true;
      };
      for (int j = 0; j < n && ok; ++j) {
        const int b = j & 1;
        const uint32_t par = (j >> 1) & 1;
        if (!mbar_wait(bar(BAR_KFULL + b), par, kWaitLimitNs)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(BAR_PVDONE + b), par ^ 1, kWaitLimitNs)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sK = sbase + kOffK + b * kStageBytes;
        const uint32_t scol = tmem + kColS + 64u * b;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sK + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
          umma_ss(scol, ad, bd, id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(BAR_KEMPTY + b));
        umma_commit(bar(BAR_SFULL + b));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
        if (*s_abort) { ok = false; break; }
      }
      if (ok && n > 0) ok = issue_pv(n - 1);
      if (ok) {
        umma_commit(bar(BAR_OFULL));
      } else {
        *s_abort = 1;
        set_status(a.status, 5 /* SA_ETIMEOUT */);
        umma_commit(bar(BAR_DRAIN));
        mbar_wait(bar(BAR_DRAIN), 0, kWaitLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;             // tensor-memory lane quarter of this warp
    const int row = quad * 32 + lane;      // query row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int half = row >> 6;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      const uint32_t par = (j >> 1) & 1;
      int blk, bits;
      if (dense) { blk = j; bits = 3; }
      else { const int32_t e = ent[j]; blk = e & kEntBlockMask; bits = (e >> kEntMaskShift) & 3; }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_SFULL + b), par, kWaitLimitNs))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[64];
      {
        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
        uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
        tmem_ld32(tmem + lane_addr + kColS + 64u * b, s0);
        tmem_ld32(tmem + lane_addr + kColS + 64u * b + 32, s1);
        tmem_wait_ld();
      }
      const bool row_ok = (bits >> half) & 1;  // uniform across the warp
      const int nvalid = min(kBlock, g.T - blk * kBlock);
      const bool add_bias = (a.b2 != nullptr) && blk >= g.nvk;
      const bool fast = row_ok && nvalid == kBlock && !add_bias;
      // Logit in log2 units: l = s * log2(e)/sqrt(128) + b2 (b2 = 0 off sinks).
      // Both paths round identically where b2 = 0: the maximum of fma(s, c, 0)
      // equals c * max(s), and p = 2^fma(s, c, b2 - m).
      const float4* bb = add_bias ? reinterpret_cast<const float4*>(a.b2 + static_cast<size_t>(blk) * kBlock)
                                  : nullptr;
      float mx;
      if (fast) {
        mx = max64(s) * sl2;
      } else {
        mx = -INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 bv = add_bias ? __ldg(bb + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float bq[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 4 * q4 + e;
            const float bk = (k < nvalid) ? bq[e] : 0.f;
            const float x = fmaf(__uint_as_float(s[k]), sl2, bk);
            if (row_ok && k < nvalid) mx = fmaxf(mx, x);
          }
        }
      }
      const float m_new = fmaxf(m_run, mx);
      const bool resc = (m_run != -INFINITY) && (m_new > m_run + 8.0f);
      if (m_run == -INFINITY) m_run = m_new;
      if (__any_sync(0xFFFFFFFFu, resc)) {
        // PV_{j-1} must have finished before O is rescaled (j >= 1 here).
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_PVDONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1,
                                               kWaitLimitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = resc ? ex2_approx(m_run - m_new) : 1.0f;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_addr + kColO + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(tmem + lane_addr + kColO + c0, o);
        }
        tmem_wait_st();
        if (resc) {
          l_run *= alpha;
          m_run = m_new;
        }
      }
      const float msub = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t p[32];
      uint64_t acc[4];
      if (fast) {
        // p = 2^(s * scale - m): one packed FMA per pair, one MUFU per value
        const uint64_t sc2 = f2(sl2, sl2);
        const uint64_t nm2 = f2(-msub, -msub);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = f2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          float x0, x1;
          unf2(ffma2(f2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), sc2, nm2), x0, x1);
          const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
          acc[(k >> 1) & 3] = fadd2(acc[(k >> 1) & 3], f2(e0, e1));
          p[k / 2] = pack_bf16x2(e0, e1);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = f2(0.f, 0.f);
        float e[64];
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 bv = add_bias ? __ldg(bb + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float bq[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int k = 4 * q4 + t;
            const float bk = (k < nvalid) ? bq[t] : 0.f;
            const float x = fmaf(__uint_as_float(s[k]), sl2, bk - msub);
            e[k] = (row_ok && k < nvalid) ? ex2_approx(x) : 0.f;
          }
        }
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          acc[(k >> 1) & 3] = fadd2(acc[(k >> 1) & 3], f2(e[k], e[k + 1]));
          p[k / 2] = pack_bf16x2(e[k], e[k + 1]);
        }
      }
      {
        float a0, a1, b0, b1, c0, c1, d0, d1;
        unf2(acc[0], a0, a1);
        unf2(acc[1], b0, b1);
        unf2(acc[2], c0, c1);
        unf2(acc[3], d0, d1);
        l_run += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
      }
      tmem_st32(tmem + lane_addr + kColS + 64u * b, p);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_PFULL + b));
      if (__any_sync(0xFFFFFFFFu, *s_abort != 0)) { ok = false; break; }
    }
    if (ok && !__all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_OFULL), 0, kWaitLimitNs))) ok = false;
    if (!ok) {
      *s_abort = 1;
      set_status(a.status, 5 /* SA_ETIMEOUT */);
    } else {
      tc_fence_after();
      // ---- epilogue: O / l -> BF16
      int t;
      bool real;
      if (dense) {
        t = row0 + row;
        real = t < g.T;
      } else {
        const int ib = half ? iB : iA;
        const int r = row & 63;
        t = kBlock * ib + r;
        const int nreal = (ib < 0) ? 0 : (ib < g.nvk ? kBlock : g.tail);
        real = ib >= 0 && r < nreal;
      }
      const float inv_l = (l_run > 0.f) ? 1.0f / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(a.o + (static_cast<size_t>(t) * g.H + h) * kHeadDim);
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + kColO + c0, o);
        tmem_wait_ld();
        if (real) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l);
            dst[c0 / 8 + q4] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Key bias: log2 conversion and the sink-only rule.
__global__ void bias_prep_kernel(const float* __restrict__ bias, float* __restrict__ b2,
                                 int32_t* status, int T, int video_keys) {
  const float kLog2e = 1.4426950408889634f;
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < T; u += gridDim.x * blockDim.x) {
    const float b = bias[u];
    if (isnan(b) || b == INFINITY) {
      set_status(status, 1 /* SA_EINVAL */);
    } else if (u < video_keys && b != 0.0f) {
      set_status(status, 3 /* SA_ENOSINKBIAS */);
    }
    b2[u] = b * kLog2e;
  }
}

}  // namespace

size_t attention_smem_bytes() { return kSmemBytes; }

cudaError_t launch_bias_prep(const float* bias, float* b2, int32_t* status, const Geometry& g,
                             cudaStream_t s) {
  const int threads = 256;
  int blocks = (g.T + threads - 1) / threads;
  if (blocks > 1024) blocks = 1024;
  bias_prep_kernel<<<blocks, threads, 0, s>>>(bias, b2, status, g.T, g.nvk * kBlock);
  return cudaGetLastError();
}

cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnArgs& a, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int units = a.g.H * (a.n_dense + a.n_pairs);
  if (units == 0) return cudaSuccess;
  attention_kernel<<<units, kThreads, kSmemBytes, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace sa
