// Exact attention over block lists, and dense attention over every key, for
// sm_103a: TMA loads of K/V blocks into 128-byte-swizzled shared memory,
// QK^T and PV on tcgen05 tensor cores with FP32 accumulators in tensor
// memory, and an online base-2 softmax in registers.
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
// Work units (128 query rows each, the M of one tcgen05.mma):
//   * sparse: a pair of consecutive query blocks of one head.  The walk is
//     the sorted union of the two lists; a key block that is in only one list
//     is masked to -inf for the other block's 64 rows.
//   * dense: 128 consecutive densely evaluated rows of one head, walking all
//     key blocks.
// The walk advances 128 keys (two entries) per step; an odd last entry is
// paired with a masked copy of itself.
//
// The kernel is persistent: one CTA per SM takes units from a global counter
// (dense units first, the longest).  A scheduler warp prepares the next unit
// (list merge) while the current one runs, Q is double-buffered, and the K/V
// ring, the S buffers and every barrier phase continue across units, so the
// next unit's loads and first MMAs overlap the current unit's tail.
//
// Schedule.  Two threads issue the MMAs, one per dependency chain: warp 1
// the S MMAs (S_x = Q K_x^T, which wait for K and for a free S buffer) and
// warp 3 the PV MMAs (O += P_x V_x, which wait for P and V), each on its own
// accumulator.  (A 16-MMA phase at this shape, M = N = 128, K = 16, takes
// 1024 cycles from two threads and 1102 from one: the tensor pipe's rate of
// 64 cycles per MMA, nearly.)  Three S buffers (step x in buffer x mod 3) give the
// softmax two steps of lead: S_{x+3} is issued as soon as PV_x has completed,
// since P_x is written as packed BF16 over the first 64 columns of S_x's
// buffer.
//
// Warp roles (12 warps, three warpgroups): warpgroup 0 holds the
// single-thread roles: warp 0 issues TMA loads (Q per unit; K and V per step
// through a 4-slot ring), warp 1 owns tensor memory and issues the S MMAs,
// warp 2 schedules units and merges their block lists, warp 3 issues the PV
// MMAs.
// Warpgroups 1 (warps 4-7, softmax group 0) and 2 (warps 8-11, group 1) each
// own one query row per thread (= tensor-memory lane); group 0 takes even
// global steps and group 1 odd ones, all 128 columns each, so two steps'
// softmax run at once.  The groups share one lazily updated reference maximum
// per row, passed step to step through shared memory; each keeps a partial
// row sum; both merge and store the output in the unit's epilogue.
// Warpgroup 0 hands registers to the softmax warpgroups (setmaxnreg).
//
// Tensor memory (512 columns): O in [0, 128); S buffers at 128, 256, 384.
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;  // warps 4..11
// Register budgets after the split: warpgroup 0 (single-thread roles) gives
// registers to the two softmax warpgroups.  128 x 88 + 256 x 208 = 64512 =
// 384 x 168, the block's allocation at launch.
constexpr uint32_t kRegsControl = 88;
constexpr uint32_t kRegsSoftmax = 208;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr int kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 128;  // S buffer b at kColS + 128 b, b in {0, 1, 2}; P_x over S_x's first 64
constexpr int kSlots = 4;        // K/V ring slots
constexpr uint32_t kSlotBytes = 32768;  // K or V of 128 keys: 2 chunks x [128 rows x 128 B]
constexpr uint32_t kQBytes = 32768;     // Q tile: 2 chunks x [128 rows x 128 B]
constexpr float kRescaleLog2 = 32.0f;

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int kMaxChunks = kMaxVideoBlocks / kBlock;  // chunks of 64 summary keys
constexpr int kMaxEnt = 2 * kMaxList + kMaxChunks;
constexpr uint32_t kOffQ = 0;                                   // 2 Q buffers
constexpr uint32_t kOffRing = 2 * kQBytes;                      // kSlots x kSlotBytes
constexpr uint32_t kOffEnt = kOffRing + kSlots * kSlotBytes;    // 2 x kMaxEnt int32
constexpr uint32_t kOffScratch = kOffEnt + 2 * 4 * kMaxEnt;     // 2 x kMaxList int32 (merge)
constexpr uint32_t kOffMask = kOffScratch + 2 * 4 * kMaxList;   // 2 x [kMaxChunks][2] uint64
constexpr uint32_t kOffQrow = kOffMask + 2 * 8 * 2 * kMaxChunks; // 2 x 128 float (fused route)
constexpr uint32_t kOffXchg = kOffQrow + 2 * 4 * kHeadDim;       // [3][128] refs + [2][128] sums
constexpr uint32_t kOffUnit = kOffXchg + 4 * 5 * 128;           // 2 unit descriptors
constexpr uint32_t kOffBar = kOffUnit + 64;
constexpr uint32_t kOffMisc = kOffBar + 512;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Barrier indices (8 bytes each).
enum {
  BAR_QFULL = 0,     // +slot (2): Q tile landed
  BAR_QEMPTY = 2,    // +slot: the unit's last S MMA completed
  BAR_FULL = 4,      // +ring slot (4)
  BAR_EMPTY = 8,     // +ring slot
  BAR_SFULL = 12,    // +buffer (3)
  BAR_PFULL = 15,    // +buffer
  BAR_PVDONE = 18,   // +buffer: PV of that step completed
  BAR_MREADY = 21,   // +buffer: reference of that step published
  BAR_OFULL = 24,    // the unit's last PV completed
  BAR_OEMPTY = 25,   // the epilogue has read O
  BAR_UFULL = 26,    // +slot (2): unit descriptor ready
  BAR_UEMPTY = 28,   // +slot: every role is done with the descriptor
  BAR_DRAIN = 30,    // the S issuer's MMAs drained (abort)
  BAR_DRAIN2 = 31,   // the PV issuer's MMAs drained (abort)
  NUM_BARS = 32
};
static_assert(NUM_BARS * 8 <= 512, "barrier area");

struct UnitDesc {
  int32_t valid;  // 0 marks the end of the work
  int32_t h;
  int32_t row0;
  int32_t iA;
  int32_t iB;     // -1 when the pair has one block
  int32_t dense;
  int32_t n_ent;  // list entries (dense: all key blocks)
  int32_t pad;
};
static_assert(sizeof(UnitDesc) * 2 <= 64, "unit area");

constexpr uint32_t kEntMaskShift = 30;
constexpr uint32_t kEntVirtual = 1u << 29;          // a chunk of 64 summary keys
constexpr uint32_t kEntBlockMask = kEntVirtual - 1u;

// Order-preserving map of an FP32 score to an unsigned key; -0 and +0 map to
// the same key (the routing kernel's convention).
__device__ __forceinline__ uint32_t order_key_f(float f) {
  uint32_t u = __float_as_uint(f);
  if (f == 0.0f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

// Barrier over `n` threads that also returns the OR of `pred` across them,
// so that a failure seen by any thread is acted on by all of them together.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
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

// Work unit u: dense tiles first (they are the longest), then the sparse
// query-block pairs, head-major.
__device__ __forceinline__ void decode_unit(const AttnArgs& a, int u, UnitDesc& d) {
  const Geometry& g = a.g;
  const int units_dense = g.H * a.n_dense;
  d.valid = 1;
  d.pad = 0;
  if (u < units_dense) {
    d.dense = 1;
    d.h = u / a.n_dense;
    d.row0 = g.r0 + 128 * (u % a.n_dense);
    d.iA = 0;
    d.iB = -1;
    d.n_ent = g.nblk;
  } else {
    const int v = u - units_dense;
    d.dense = 0;
    d.h = v / a.n_pairs;
    const int p = v % a.n_pairs;
    d.iA = 2 * p;
    d.iB = (2 * p + 1 < g.nq) ? 2 * p + 1 : -1;
    d.row0 = kBlock * d.iA;
    d.n_ent = 0;
  }
}

// kMerged: Spark's merged mode (skipped video blocks enter as summary keys).
// kFused: the scheduler routes each unit itself (CTA-local Top-K from the
// block means) instead of reading the plan's lists, and exports the lists.
// Each mode is its own instantiation so that the exact path's softmax code
// stays as compact as it can be.
// kProbeOnce: every pipeline wait is a single probe (a testing build of the
// kernel that exercises the timeout path; the abort drains keep their limit).
template <bool kMerged, bool kFused, bool kProbeOnce>
__global__ void __launch_bounds__(kThreads, 1)
attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_ak,
                 const __grid_constant__ CUtensorMap tm_av, const AttnArgs a) {
  const Geometry& g = a.g;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  float* xchg = reinterpret_cast<float*>(base + kOffXchg);
  UnitDesc* udesc = reinterpret_cast<UnitDesc*>(base + kOffUnit);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + kOffMisc);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(base + kOffMisc + 16);
  volatile int32_t* s_status = reinterpret_cast<volatile int32_t*>(base + kOffMisc + 24);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * i; };
  constexpr uint64_t lim = kProbeOnce ? 0 : kWaitLimitNs;  // pipeline waits (drains: kWaitLimitNs)
  auto ent_buf = [&](int slot) { return reinterpret_cast<int32_t*>(base + kOffEnt + 4u * kMaxEnt * slot); };
  // keep-masks of the summary keys of a unit: [chunk][row half], bit u set
  // when video block 64 chunk + u is skipped by that half's list
  auto vmask = [&](int slot) { return reinterpret_cast<unsigned long long*>(base + kOffMask) + slot * 2 * kMaxChunks; };

  // The merged build is launched as a programmatic dependent: the previous
  // kernels' results are read only after this.  (In the exact build the
  // wait, with no dependency to wait for, still measured ~2 us per call.)
  if constexpr (kMerged) griddep_wait();
  if (threadIdx.x == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(a.status);
    *s_abort = 0;
  }
  __syncthreads();
  if (*s_status != 0) return;  // an earlier step on this stream failed

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int total_units = g.H * (a.n_dense + a.n_pairs);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(bar(i), 1);
    for (int b = 0; b < 3; ++b) mbar_init(bar(BAR_PFULL + b), 4);   // the owning group's 4 warps
    for (int b = 0; b < 3; ++b) mbar_init(bar(BAR_MREADY + b), 4);
    mbar_init(bar(BAR_OEMPTY), 8);                                   // all softmax warps
    for (int s = 0; s < 2; ++s) mbar_init(bar(BAR_UEMPTY + s), 11);  // producer + 2 MMA issuers + 8 softmax
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // Entry e of unit `d` (descriptor slot `slot`): block index and row-half
  // mask (bit 0: rows 0-63, bit 1: rows 64-127).  An odd count is padded with
  // a masked copy of the last entry so every step loads two real blocks.
  auto entry = [&](const UnitDesc& d, int slot, int e, int& blk, int& bits, bool& virt) {
    const bool pad = e >= d.n_ent;
    const int ee = pad ? d.n_ent - 1 : e;
    virt = false;
    if (d.dense) {
      blk = ee;
      bits = 3;
    } else {
      const uint32_t v = static_cast<uint32_t>(ent_buf(slot)[ee]);
      virt = kMerged && (v & kEntVirtual) != 0;
      blk = static_cast<int>(v & kEntBlockMask);
      bits = static_cast<int>(v >> kEntMaskShift);
    }
    if (pad) bits = 0;
  };
  // Waits for unit k's descriptor; false when waiting failed.
  auto wait_unit = [&](int k) -> bool {
    return mbar_wait(bar(BAR_UFULL + (k & 1)), (k >> 1) & 1, lim);
  };

  // Fused route of a sparse unit (scheduler warp): for query blocks iA and
  // iB, the scores s_j = Qmean . Kmean_j / sqrt(128) summed in FP32 over
  // d = 0..127 in order (as the routing kernel does), Top-K by the bitwise
  // boundary search, and the sorted union of forced local blocks, selected
  // blocks and sinks, written to la / lb and exported to idx / cnt.
  auto route_pair = [&](const UnitDesc& d, int32_t* la_, int32_t* lb_) -> int2 {
    float* qs = reinterpret_cast<float*>(base + kOffQrow);
    const int nrow = d.iB >= 0 ? 2 : 1;
    for (int e = lane; e < nrow * kHeadDim; e += 32) {
      const int i = e < kHeadDim ? d.iA : d.iB;
      qs[e] = a.qc[(static_cast<size_t>(d.h) * g.nq + i) * kHeadDim + (e % kHeadDim)];
    }
    __syncwarp();
    constexpr int kKpl = kMaxFusedVideoBlocks / 32;  // keys per lane
    uint32_t kr[2][kKpl];
    const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
    // All of a lane's keys advance together over d = 0..127 (each sum still
    // in order of d): 2 x kKpl independent FMA chains instead of two.
    float acc[2][kKpl];
#pragma unroll
    for (int m = 0; m < kKpl; ++m) acc[0][m] = acc[1][m] = 0.f;
    const float4* kbase = reinterpret_cast<const float4*>(a.kc + static_cast<size_t>(d.h) * g.nvk * kHeadDim);
#pragma unroll 1
    for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
      const float4 q0 = *reinterpret_cast<const float4*>(qs + 4 * d4);
      const float4 q1 = *reinterpret_cast<const float4*>(qs + kHeadDim + 4 * d4);
#pragma unroll
      for (int m = 0; m < kKpl; ++m) {
        const int j = lane + 32 * m;
        if (j < g.nvk) {
          const float4 kv = __ldg(kbase + static_cast<size_t>(j) * (kHeadDim / 4) + d4);
          acc[0][m] = fmaf(q0.x, kv.x, acc[0][m]);
          acc[0][m] = fmaf(q0.y, kv.y, acc[0][m]);
          acc[0][m] = fmaf(q0.z, kv.z, acc[0][m]);
          acc[0][m] = fmaf(q0.w, kv.w, acc[0][m]);
          acc[1][m] = fmaf(q1.x, kv.x, acc[1][m]);
          acc[1][m] = fmaf(q1.y, kv.y, acc[1][m]);
          acc[1][m] = fmaf(q1.z, kv.z, acc[1][m]);
          acc[1][m] = fmaf(q1.w, kv.w, acc[1][m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kKpl; ++m) {
      const int j = lane + 32 * m;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = r == 0 ? d.iA : d.iB;
        const int lo = max(0, i - g.R), hi = min(g.nvk - 1, i + g.R);
        const bool cand = j < g.nvk && (j < lo || j > hi) && (r == 0 || d.iB >= 0);
        kr[r][m] = cand ? order_key_f(acc[r][m] * inv_sqrt_d) : 0u;
      }
    }
    // largest tau with #{keys >= tau} >= kp, both rows' searches together
    int kp[2], need[2];
    bool take_all[2];
    uint32_t tau[2] = {0u, 0u};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = r == 0 ? d.iA : (d.iB >= 0 ? d.iB : d.iA);
      const int lo = max(0, i - g.R), hi = min(g.nvk - 1, i + g.R);
      const int ncand = g.nvk - max(0, hi - lo + 1);
      kp[r] = min(g.K, ncand);
      take_all[r] = kp[r] == ncand;
    }
#pragma unroll 1
    for (int bit = 31; bit >= 0; --bit) {
      unsigned c[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t t = tau[r] | (1u << bit);
        c[r] = 0;
#pragma unroll
        for (int m = 0; m < kKpl; ++m) c[r] += (kr[r][m] >= t) ? 1u : 0u;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) c[r] = __reduce_add_sync(0xFFFFFFFFu, c[r]);
#pragma unroll
      for (int r = 0; r < 2; ++r)
        if (static_cast<int>(c[r]) >= kp[r]) tau[r] |= (1u << bit);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      unsigned c = 0;
#pragma unroll
      for (int m = 0; m < kKpl; ++m) c += (kr[r][m] > tau[r]) ? 1u : 0u;
      need[r] = kp[r] - static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, c));
    }
    const unsigned lt = (1u << lane) - 1u;
    int2 cnt_ab = make_int2(0, 0);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r == 1 && d.iB < 0) break;
      const int i = r == 0 ? d.iA : d.iB;
      const int lo = max(0, i - g.R), hi = min(g.nvk - 1, i + g.R);
      int32_t* out = r == 0 ? la_ : lb_;
      int32_t* gout = a.idx_w + (static_cast<size_t>(d.h) * g.nq + i) * g.maxl;
      int pos = 0, eq_seen = 0;
      auto emit = [&](int j, bool sel, bool eq) {
        const unsigned eqm = __ballot_sync(0xFFFFFFFFu, eq);
        if (eq) sel = (eq_seen + __popc(eqm & lt)) < need[r];
        eq_seen += __popc(eqm);
        const unsigned sm = __ballot_sync(0xFFFFFFFFu, sel);
        if (sel) {
          out[pos + __popc(sm & lt)] = j;
          gout[pos + __popc(sm & lt)] = j;
        }
        pos += __popc(sm);
      };
#pragma unroll
      for (int m = 0; m < kKpl; ++m) {
        if (32 * m >= g.nblk) break;
        const int j = 32 * m + lane;
        bool sel = false, eq = false;
        if (j < g.nvk) {
          if ((j >= lo && j <= hi) || take_all[r]) sel = true;
          else if (kr[r][m] > tau[r]) sel = true;
          else if (kr[r][m] == tau[r]) eq = true;
        } else {
          sel = j < g.nblk;  // sink block
        }
        emit(j, sel, eq);
      }
      for (int j0 = 32 * kKpl; j0 < g.nblk; j0 += 32) emit(j0 + lane, j0 + lane < g.nblk, false);
      for (int q = pos + lane; q < g.maxl; q += 32) gout[q] = -1;
      if (lane == 0) a.cnt_w[static_cast<size_t>(d.h) * g.nq + i] = pos;
      (r == 0 ? cnt_ab.x : cnt_ab.y) = pos;
    }
    __syncwarp();
    return cnt_ab;
  };

  if (warp < 4) {
    setmaxnreg_dec<kRegsControl>();
  }
  if (warp == 2) {
    // ------------------------------------------------------------ scheduler
    int32_t* la = reinterpret_cast<int32_t*>(base + kOffScratch);
    int32_t* lb = la + kMaxList;
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      bool ok = true;
      if (k >= 2) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_UEMPTY + slot), ((k - 2) >> 1) & 1, lim));
      if (!ok || *s_abort) {
        *s_abort = 1;
        set_status(a.status, 5 /* SA_ETIMEOUT */);
        break;
      }
      int u = 0;
      if (lane == 0) u = atomicAdd(a.unit_counter, 1);
      u = __shfl_sync(0xFFFFFFFFu, u, 0);
      UnitDesc d;
      bool bad = false;
      if (u >= total_units) {
        d.valid = 0;
      } else {
        decode_unit(a, u, d);
        if (!d.dense) {
          int nA, nB;
          if constexpr (kFused) {
            const int2 n = route_pair(d, la, lb);  // lists straight into la / lb
            nA = n.x;
            nB = n.y;
          } else {
            nA = a.cnt[static_cast<size_t>(d.h) * g.nq + d.iA];
            nB = (d.iB >= 0) ? a.cnt[static_cast<size_t>(d.h) * g.nq + d.iB] : 0;
          }
          bad = nA < 1 || nA > g.maxl || (d.iB >= 0 && (nB < 1 || nB > g.maxl));
          if (!bad) {
            if constexpr (!kFused) {
              const int32_t* ga = a.idx + (static_cast<size_t>(d.h) * g.nq + d.iA) * g.maxl;
              for (int k2 = lane; k2 < nA; k2 += 32) la[k2] = ga[k2];
              if (d.iB >= 0) {
                const int32_t* gb = a.idx + (static_cast<size_t>(d.h) * g.nq + d.iB) * g.maxl;
                for (int k2 = lane; k2 < nB; k2 += 32) lb[k2] = gb[k2];
              }
            }
            __syncwarp();
            for (int k2 = lane; k2 < nA; k2 += 32)
              bad |= la[k2] < 0 || la[k2] >= g.nblk || (k2 + 1 < nA && la[k2] >= la[k2 + 1]);
            for (int k2 = lane; k2 < nB; k2 += 32)
              bad |= lb[k2] < 0 || lb[k2] >= g.nblk || (k2 + 1 < nB && lb[k2] >= lb[k2 + 1]);
          }
          bad = __any_sync(0xFFFFFFFFu, bad);
          if (!bad) {
            // stable merge with duplicates (A before an equal B), then drop
            // the second copy of each duplicated block and mark it for both
            int32_t* mg = ent_buf(slot);
            for (int k2 = lane; k2 < nA; k2 += 32)
              mg[k2 + lower_bound_s(lb, nB, la[k2])] = static_cast<int32_t>(la[k2] | (1u << kEntMaskShift));
            for (int k2 = lane; k2 < nB; k2 += 32)
              mg[k2 + upper_bound_s(la, nA, lb[k2])] = static_cast<int32_t>(lb[k2] | (2u << kEntMaskShift));
            __syncwarp();
            const int nm = nA + nB;
            int pos = 0;
            int32_t prev_blk = -1;  // block of the element before this chunk
            for (int m0 = 0; m0 < nm; m0 += 32) {
              const int m = m0 + lane;
              int32_t cur = 0, nxt = -1;
              if (m < nm) cur = mg[m];
              if (m + 1 < nm) nxt = static_cast<int32_t>(static_cast<uint32_t>(mg[m + 1]) & kEntBlockMask);
              const int32_t blk = (m < nm) ? static_cast<int32_t>(static_cast<uint32_t>(cur) & kEntBlockMask) : -2;
              int32_t before = __shfl_up_sync(0xFFFFFFFFu, blk, 1);
              if (lane == 0) before = prev_blk;
              const bool keep = m < nm && blk != before;
              const int32_t val = (nxt == blk) ? static_cast<int32_t>(static_cast<uint32_t>(blk) | (3u << kEntMaskShift)) : cur;
              prev_blk = __shfl_sync(0xFFFFFFFFu, blk, 31);
              const unsigned km = __ballot_sync(0xFFFFFFFFu, keep);
              __syncwarp();  // all reads of this chunk precede its writes
              if (keep) mg[pos + __popc(km & ((1u << lane) - 1u))] = val;
              pos += __popc(km);
              __syncwarp();
            }
            d.n_ent = pos;
            if (kMerged) {
              // Every video block the lists skip enters as one summary key:
              // append the chunks of 64 summary keys, masked per row half.
              const int nvc = (g.nvk + kBlock - 1) / kBlock;
              unsigned long long* vm = vmask(slot);
              for (int c = lane; c < nvc; c += 32) {
                const int nb = min(kBlock, g.nvk - kBlock * c);
                const unsigned long long all = (nb == kBlock) ? ~0ull : ((1ull << nb) - 1ull);
                vm[2 * c] = all;
                vm[2 * c + 1] = (d.iB >= 0) ? all : 0ull;
              }
              __syncwarp();
              for (int m = lane; m < pos; m += 32) {
                const uint32_t v = static_cast<uint32_t>(mg[m]);
                const int blk = static_cast<int>(v & kEntBlockMask);
                if (blk >= g.nvk) continue;
                const unsigned long long bit = 1ull << (blk % kBlock);
                if (v & (1u << kEntMaskShift)) atomicAnd(&vm[2 * (blk / kBlock)], ~bit);
                if (v & (2u << kEntMaskShift)) atomicAnd(&vm[2 * (blk / kBlock) + 1], ~bit);
              }
              __syncwarp();
              // Additive logits of the summary keys, per row half: the
              // log-mass where the half's list skips the block, -inf where
              // it lists it.  Written to this CTA's rows for the slot; the
              // unit's descriptor barrier publishes them.
              float* vb = a.vbias + (static_cast<size_t>(blockIdx.x) * 2 + slot) * a.vstride;
              const float* lmh = a.lm2 + static_cast<size_t>(d.h) * a.nblkp;
              for (int e = lane; e < nvc * 2 * kBlock; e += 32) {
                const int c = e / (2 * kBlock), hf = (e / kBlock) & 1, u = e % kBlock;
                vb[e] = ((vm[2 * c + hf] >> u) & 1ull) ? lmh[kBlock * c + u] : -INFINITY;
              }
              const uint32_t hb = (d.iB >= 0) ? 3u : 1u;
              for (int c = lane; c < nvc; c += 32)
                mg[pos + c] = static_cast<int32_t>(static_cast<uint32_t>(c) | kEntVirtual | (hb << kEntMaskShift));
              __syncwarp();
              d.n_ent = pos + nvc;
            }
          }
        }
      }
      if (bad) {
        if (lane == 0) set_status(a.status, 1 /* SA_EINVAL */);
        *s_abort = 1;
        d.valid = 0;
      }
      if (lane == 0) udesc[slot] = d;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_UFULL + slot));
      if (!d.valid) break;
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (kMerged) {
        tma_prefetch_desc(&tm_ak);
        tma_prefetch_desc(&tm_av);
      }
      int seq = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!wait_unit(k)) { ok = false; break; }
        const UnitDesc d = udesc[slot];
        if (!d.valid) break;
        const int n = (d.n_ent + 1) / 2;
        const int xq = d.h * kHeadDim;
        if (k >= 2 && !mbar_wait(bar(BAR_QEMPTY + slot), ((k - 2) >> 1) & 1, lim)) { ok = false; break; }
        const uint32_t sQ = sbase + kOffQ + slot * kQBytes;
        mbar_arrive_expect_tx(bar(BAR_QFULL + slot), kQBytes);
        tma_load_2d(sQ, &tm_q, bar(BAR_QFULL + slot), xq, d.row0);
        tma_load_2d(sQ + 16384, &tm_q, bar(BAR_QFULL + slot), xq + 64, d.row0);
        // Load order (the MMA issuers consume in the same order): K0, K1,
        // K2, then per step j: V_j, K_{j+3}.
        // kind 0: K (or summary keys), kind 1: V (or summary values)
        auto load = [&](int kind, int step) -> bool {
          const int s = seq % kSlots;
          const uint32_t par = ((seq / kSlots) & 1) ^ 1;
          if (!mbar_wait(bar(BAR_EMPTY + s), par, lim)) return false;
          const uint32_t dst = sbase + kOffRing + s * kSlotBytes;
          mbar_arrive_expect_tx(bar(BAR_FULL + s), kSlotBytes);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            int blk, bits;
            bool virt;
            entry(d, slot, 2 * step + hh, blk, bits, virt);
            if (!kMerged || !virt) {
              const CUtensorMap* map = kind == 0 ? &tm_k : &tm_v;
              tma_load_2d(dst + hh * 8192, map, bar(BAR_FULL + s), xq, blk * kBlock);
              tma_load_2d(dst + 16384 + hh * 8192, map, bar(BAR_FULL + s), xq + 64, blk * kBlock);
            } else {
              // summaries are [H * nblk rows, 128 columns]; K/V [T rows, H * 128]
              const CUtensorMap* map = kind == 0 ? &tm_ak : &tm_av;
              const int y0 = d.h * g.nblk + blk * kBlock;
              tma_load_2d(dst + hh * 8192, map, bar(BAR_FULL + s), 0, y0);
              tma_load_2d(dst + 16384 + hh * 8192, map, bar(BAR_FULL + s), 64, y0);
            }
          }
          ++seq;
          return true;
        };
        for (int j = 0; j < 3 && j < n && ok; ++j) ok = load(0, j);
        for (int j = 0; j < n && ok; ++j) {
          ok = load(1, j);
          if (ok && j + 3 < n) ok = load(0, j + 3);
          if (*s_abort) ok = false;
        }
        if (ok) mbar_arrive(bar(BAR_UEMPTY + slot));
      }
      if (!ok) {
        *s_abort = 1;
        set_status(a.status, 5 /* SA_ETIMEOUT */);
        // let copies in flight land before the CTA exits (bounded)
        for (int q = max(0, seq - kSlots); q < seq; ++q)
          mbar_wait(bar(BAR_FULL + q % kSlots), (q / kSlots) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // S_x = Q K_x^T.  Two threads issue the MMAs (this one S, warp 3's lane 0
    // PV): one thread's tcgen05.mma issue, not the tensor pipe, limits a
    // single stream.  Both walk the same ring sequence (K0, K1, K2, then
    // V_j, K_{j+3} per step) and consume their own kind of slot.
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T, both K-major
      // A descriptor's start address is its low 14 bits (16-byte units):
      // stepping through a tile is one add of a compile-time offset.
      auto kmaj_off = [](int kk) { return static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
      auto slot_addr = [&](int q) { return sbase + kOffRing + (q % kSlots) * kSlotBytes; };
      auto wait_full = [&](int q) { return mbar_wait(bar(BAR_FULL + q % kSlots), (q / kSlots) & 1, lim); };
      // S_x goes to the buffer of S_{x-3}, which holds P_{x-3} until PV_{x-3}
      // has completed.
      auto s_col = [&](int gs) { return tmem + kColS + 128u * (gs % 3); };
      auto buffer_free = [&](int x) {
        return x < 3 || mbar_wait(bar(BAR_PVDONE + x % 3), ((x - 3) / 3) & 1, lim);
      };
      auto issue_s = [&](int x, uint64_t q_base, int qk) {
        const uint64_t ks = sdesc_sw128(slot_addr(qk), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(s_col(x), q_base + kmaj_off(kk), ks + kmaj_off(kk), id_s, kk > 0 ? 1u : 0u);
        umma_commit(bar(BAR_EMPTY + qk % kSlots));
        umma_commit(bar(BAR_SFULL + x % 3));
      };
      int seq = 0, G = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!wait_unit(k)) { ok = false; break; }
        const UnitDesc d = udesc[slot];
        if (!d.valid) break;
        const int n = (d.n_ent + 1) / 2;
        if (!mbar_wait(bar(BAR_QFULL + slot), (k >> 1) & 1, lim)) { ok = false; break; }
        const uint64_t q_base = sdesc_sw128(sbase + kOffQ + slot * kQBytes, 16, 1024);
        // S_G .. S_{G+2}
        for (int j = 0; j < 3 && j < n; ++j) {
          const int qk = seq++;
          if (!buffer_free(G + j) || !wait_full(qk)) { ok = false; break; }
          tc_fence_after();
          issue_s(G + j, q_base, qk);
        }
        if (!ok) break;
        if (n <= 3) umma_commit(bar(BAR_QEMPTY + slot));  // the unit's last S MMA
        for (int j = 0; j < n && ok; ++j) {
          ++seq;  // V_j: the PV issuer's slot
          if (j + 3 >= n) continue;
          const int qk = seq++;
          if (!buffer_free(G + j + 3) || !wait_full(qk)) { ok = false; break; }
          tc_fence_after();
          issue_s(G + j + 3, q_base, qk);
          if (j + 3 == n - 1) umma_commit(bar(BAR_QEMPTY + slot));  // the unit's last S MMA
          if (*s_abort) { ok = false; break; }
        }
        if (!ok) break;
        mbar_arrive(bar(BAR_UEMPTY + slot));
        G += n;
      }
      if (!ok) {
        *s_abort = 1;
        set_status(a.status, 5 /* SA_ETIMEOUT */);
        umma_commit(bar(BAR_DRAIN));
        mbar_wait(bar(BAR_DRAIN), 0, kWaitLimitNs);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      const uint32_t id_o = idesc_bf16(128, 128, false, true);  // O += P V, V is MN-major
      auto vmaj_off = [](int kk) { return static_cast<uint64_t>((kk * 2048) >> 4); };
      auto slot_addr = [&](int q) { return sbase + kOffRing + (q % kSlots) * kSlotBytes; };
      auto wait_full = [&](int q) { return mbar_wait(bar(BAR_FULL + q % kSlots), (q / kSlots) & 1, lim); };
      auto p_col = [&](int gs) { return tmem + kColS + 128u * (gs % 3); };
      int seq = 0, G = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!wait_unit(k)) { ok = false; break; }
        const UnitDesc d = udesc[slot];
        if (!d.valid) break;
        const int n = (d.n_ent + 1) / 2;
        seq += n < 3 ? n : 3;  // K0 .. K2: the S issuer's slots
        for (int j = 0; j < n && ok; ++j) {
          const int gs = G + j;
          const int qv = seq++;
          if (j + 3 < n) ++seq;  // K_{j+3}
          if (!wait_full(qv)) { ok = false; break; }
          if (!mbar_wait(bar(BAR_PFULL + gs % 3), (gs / 3) & 1, lim)) { ok = false; break; }
          // The unit's first PV overwrites O: the previous epilogue must be done.
          if (j == 0 && k >= 1 && !mbar_wait(bar(BAR_OEMPTY), (k - 1) & 1, lim)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vs = sdesc_sw128(slot_addr(qv), 16384, 1024);
          const uint32_t pcol = p_col(gs);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + kColO, pcol + kk * 8, vs + vmaj_off(kk), id_o, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(BAR_EMPTY + qv % kSlots));
          umma_commit(bar(BAR_PVDONE + gs % 3));
          if (*s_abort) { ok = false; break; }
        }
        if (!ok) break;
        umma_commit(bar(BAR_OFULL));
        mbar_arrive(bar(BAR_UEMPTY + slot));
        G += n;
      }
      if (!ok) {
        *s_abort = 1;
        set_status(a.status, 5 /* SA_ETIMEOUT */);
        umma_commit(bar(BAR_DRAIN2));
        mbar_wait(bar(BAR_DRAIN2), 0, kWaitLimitNs);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<kRegsSoftmax>();
    const int grp = (warp - 4) / 4;        // owns global steps with parity grp
    const int quad = warp & 3;             // tensor-memory lane quarter of this warp
    const int row = quad * 32 + lane;      // query row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int half = row >> 6;
    const float sl2 = a.scale_log2;
    // An all-zero key bias takes the no-bias path, so that it gives the same
    // output bit for bit (the bias prep flags any nonzero value).
    const bool key_bias = a.b2 != nullptr && *a.bias_nz != 0;
    float* rref = xchg;                    // [3][128]: reference after step g at g % 3
    float* xl = xchg + 3 * 128;            // [2][128]: partial row sums
    int G = 0;
    // All 256 softmax threads agree on entering each unit (its descriptor
    // arrived for every warp): a warp whose wait gave up must not leave the
    // others at the group barriers.  The agreement for unit k + 1 rides on
    // the barrier that ends unit k.
    bool ok = !named_bar_or(2, kSoftmaxThreads, !__all_sync(0xFFFFFFFFu, wait_unit(0)) || *s_abort != 0);
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      const UnitDesc d = udesc[slot];
      if (!d.valid) break;
      const int n = (d.n_ent + 1) / 2;
      // Reference maximum (log2 units) that P, O and the row sums are
      // relative to.  It moves only when a step's maximum exceeds it by more
      // than 2^32 (then O is rescaled once); p <= 2^32 keeps every sum far
      // inside FP32.
      float ref = -INFINITY;     // reference after the previous step (either group)
      float my_ref = -INFINITY;  // reference this group's partial sum is kept in
      float l_run = 0.f;
      for (int j = ((G & 1) == grp) ? 0 : 1; j < n && ok; j += 2) {
        const int gs = G + j;
        const int b = gs % 3;        // reference slot
        const int sb = gs % 3;       // S buffer (P_g goes over S_g's first 64 columns)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_SFULL + sb), (gs / 3) & 1, lim));
        if (!ok) break;
        tc_fence_after();
        const uint32_t scol = tmem + lane_addr + kColS + 128u * sb;
        // The two 64-key halves come from list entries 2j and 2j+1.  Pass 1
        // takes the row maximum over both halves, pass 2 reloads each half
        // from tensor memory and turns it into P (keeps 64 values live).
        int blk[2], bits[2];
        bool virt[2];
        entry(d, slot, 2 * j, blk[0], bits[0], virt[0]);
        entry(d, slot, 2 * j + 1, blk[1], bits[1], virt[1]);
        bool row_ok[2], fast[2], add_bias[2];
        int nvalid[2];
        // Additive logits (log2 units) of a half on the general path: the
        // key bias on sinks, or (merged mode) the summary keys' log-mass,
        // -inf for the blocks this row half's list holds exactly.
        auto bias_of = [&](int hh) -> const float4* {
          if constexpr (kMerged)
            if (virt[hh])
              return reinterpret_cast<const float4*>(
                  a.vbias + (static_cast<size_t>(blockIdx.x) * 2 + slot) * a.vstride + (2 * blk[hh] + half) * kBlock);
          return reinterpret_cast<const float4*>(a.b2 + static_cast<size_t>(blk[hh]) * kBlock);
        };
        // Summary-key logits are rewritten every other unit by this CTA:
        // ordinary (coherent) loads, ordered after the descriptor barrier.
        auto bias_ld = [&](const float4* p) { return kMerged ? *p : __ldg(p); };
        float mx = -INFINITY;
        auto half_flags = [&](int hh) {
          row_ok[hh] = (bits[hh] >> half) & 1;  // uniform across the warp
          nvalid[hh] = virt[hh] ? kBlock : min(kBlock, g.T - blk[hh] * kBlock);
          add_bias[hh] = virt[hh] || (key_bias && blk[hh] >= g.nvk);
          fast[hh] = row_ok[hh] && nvalid[hh] == kBlock && !add_bias[hh];
        };
        if constexpr (kMerged) {
          half_flags(0);
          half_flags(1);
        }
        // Both passes walk the two halves taking each half's flags by scalar
        // selects, so that the loops can stay rolled without local memory:
        // the merged build rolls them (one copy of the code; the
        // tensor-memory loads order the halves anyway), measured faster
        // there and slower in the exact build.
        uint32_t ok_m = 0, fast_m = 0, bias_m = 0;
        const float4* bb0 = nullptr;
        const float4* bb1 = nullptr;
        if constexpr (kMerged) {
          ok_m = (row_ok[0] ? 1u : 0u) | (row_ok[1] ? 2u : 0u);
          fast_m = (fast[0] ? 1u : 0u) | (fast[1] ? 2u : 0u);
          bias_m = (add_bias[0] ? 1u : 0u) | (add_bias[1] ? 2u : 0u);
          bb0 = bias_of(0);
          bb1 = bias_of(1);
        }
        auto flag = [&](uint32_t m, const bool (&f)[2], int hh) -> bool {
          if constexpr (kMerged) return (m >> hh) & 1u;
          return f[hh];
        };
#pragma unroll(kMerged ? 1 : 2)
        for (int hh = 0; hh < 2; ++hh) {
          if constexpr (!kMerged) half_flags(hh);  // unrolled: constant index
          if (!flag(ok_m, row_ok, hh)) continue;
          uint32_t sh[64];
          tmem_ld32(scol + 64u * hh, *reinterpret_cast<uint32_t(*)[32]>(&sh[0]));
          tmem_ld32(scol + 64u * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&sh[32]));
          tmem_wait_ld();
          // Logit in log2 units: l = s * log2(e)/sqrt(128) + b2 (b2 = 0 off
          // sinks).  A full half without additive logits needs only its
          // maximum here (c * max(s) is the maximum of the rounded c * s);
          // pass 2 forms p = 2^fma(s, c, -ref) from the scores.
          if (flag(fast_m, fast, hh)) {
            mx = fmaxf(mx, max64(sh) * sl2);
          } else {
            // General half: the logits l = s * scale + b (-inf past the
            // sequence end) replace the scores in tensor memory, so the
            // bias is read once and pass 2 runs the packed path on them.
            const float4* bb = kMerged ? (hh ? bb1 : bb0) : bias_of(hh);
            const bool ab = flag(bias_m, add_bias, hh);
            const int nv = kMerged ? (hh ? nvalid[1] : nvalid[0]) : nvalid[hh];
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
              const float4 bv = ab ? bias_ld(bb + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
              const float bq[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int kx = 4 * q4 + e;
                const float x = (kx < nv) ? fmaf(__uint_as_float(sh[kx]), sl2, bq[e]) : -INFINITY;
                sh[kx] = __float_as_uint(x);
              }
            }
            mx = fmaxf(mx, max64(sh));  // a tree, not a chain of 64 dependent maxima
            tmem_st32(scol + 64u * hh, *reinterpret_cast<uint32_t(*)[32]>(&sh[0]));
            tmem_st32(scol + 64u * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&sh[32]));
          }
        }
        if (!fast[0] || !fast[1]) tmem_wait_st();  // pass 2 reads the logits back
        // reference after step g-1 of this unit (published by the other group)
        if (j > 0) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_MREADY + (gs - 1) % 3), ((gs - 1) / 3) & 1,
                                                 lim))) {
            ok = false;
            break;
          }
          ref = rref[((gs - 1) % 3) * 128 + row];
        }
        const float prev = ref;
        if (prev == -INFINITY || mx > prev + kRescaleLog2) ref = fmaxf(prev, mx);
        rref[b * 128 + row] = ref;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_MREADY + b));
        const bool resc = prev != -INFINITY && ref != prev;
        if (my_ref != ref) {
          if (my_ref != -INFINITY) l_run *= ex2_approx(my_ref - ref);
          my_ref = ref;
        }
        const float msub = (ref == -INFINITY) ? 0.f : ref;
        // P_g goes over S_g's first 64 columns, after both passes have read
        // them (half 0's P after half 0's reads).
        uint64_t acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = f2(0.f, 0.f);
#pragma unroll(kMerged ? 1 : 2)
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t p[32];
          if (!flag(ok_m, row_ok, hh)) {
#pragma unroll
            for (int kx = 0; kx < 32; ++kx) p[kx] = 0u;
          } else {
            uint32_t sh[64];
            tmem_ld32(scol + 64u * hh, *reinterpret_cast<uint32_t(*)[32]>(&sh[0]));
            tmem_ld32(scol + 64u * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&sh[32]));
            tmem_wait_ld();
            {
              // p = 2^(x * c - ref): one packed FMA per pair, one MUFU per
              // value; x is a score (c = scale) or, on a general half, a
              // logit from pass 1 (c = 1).
              const float c = flag(fast_m, fast, hh) ? sl2 : 1.0f;
              const uint64_t sc2 = f2(c, c);
              const uint64_t nm2 = f2(-msub, -msub);
#pragma unroll
              for (int kx = 0; kx < 64; kx += 2) {
                float x0, x1;
                unf2(ffma2(f2(__uint_as_float(sh[kx]), __uint_as_float(sh[kx + 1])), sc2, nm2), x0, x1);
                const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
                acc[(kx >> 1) & 3] = fadd2(acc[(kx >> 1) & 3], f2(e0, e1));
                p[kx / 2] = pack_bf16x2(e0, e1);
              }
            }
          }
          // P (BF16 pairs) of this half into columns [32 hh, 32 hh + 32) of
          // S_g's buffer: columns already consumed by both passes of half 0.
          tmem_st32(tmem + lane_addr + kColS + 128u * sb + 32u * hh, p);
        }
        {
          float a0, a1, b0, b1, c0, c1, d0, d1;
          unf2(acc[0], a0, a1);
          unf2(acc[1], b0, b1);
          unf2(acc[2], c0, c1);
          unf2(acc[3], d0, d1);
          l_run += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
        }
        tmem_wait_st();
        // O holds sum_{i<g} P_i V_i relative to `prev`; move it to `ref`
        // before P_g is released to the PV issuer.
        if (__any_sync(0xFFFFFFFFu, resc)) {
          // PV_{g-1} must have finished before O is rescaled (j >= 1 here).
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_PVDONE + (gs - 1) % 3), ((gs - 1) / 3) & 1,
                                                 lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = resc ? ex2_approx(prev - ref) : 1.0f;
          // (rolled in the merged build: measured faster there, slower in
          // the exact one)
#pragma unroll(kMerged ? 1 : 4)
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_addr + kColO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(tmem + lane_addr + kColO + c0, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_PFULL + sb));
        if (__any_sync(0xFFFFFFFFu, *s_abort != 0)) ok = false;
      }
      // ---- epilogue of the unit
      ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_OFULL), k & 1, lim));
      const int last = G + n - 1;
      if (ok && (last & 1) != grp)  // the other group published the last reference
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(BAR_MREADY + last % 3), (last / 3) & 1, lim));
      float fin = -INFINITY;
      if (ok) {
        tc_fence_after();
        fin = rref[(last % 3) * 128 + row];
      }
      const float l_mine = (my_ref == -INFINITY || !ok) ? 0.f : l_run * ex2_approx(my_ref - fin);
      xl[grp * 128 + row] = l_mine;
      // both groups meet here; the OR-reduction makes the outcome uniform
      ok = !named_bar_or(2, kSoftmaxThreads, !ok || *s_abort != 0);
      const float l_tot = l_mine + xl[(grp ^ 1) * 128 + row];
      if (!ok) break;
      int t;
      bool real;
      if (d.dense) {
        t = d.row0 + row;
        real = t < g.T;
      } else {
        const int ib = half ? d.iB : d.iA;
        const int r = row & 63;
        t = kBlock * ib + r;
        const int nreal = (ib < 0) ? 0 : (ib < g.nvk ? kBlock : g.tail);
        real = ib >= 0 && r < nreal;
      }
      const float inv_l = (l_tot > 0.f) ? 1.0f / l_tot : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(a.o + (static_cast<size_t>(t) * g.H + d.h) * kHeadDim + 64 * grp);
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + kColO + 64u * grp + c0, o);
        tmem_wait_ld();
        if (real) {
          // 32-byte stores (o is 32-byte aligned): whole L2 sectors, half
          // the store instructions of 16-byte ones, each of which touches
          // 32 rows.
#pragma unroll
          for (int q8 = 0; q8 < 2; ++q8) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[q8 * 16 + 2 * e]) * inv_l,
                                 __uint_as_float(o[q8 * 16 + 2 * e + 1]) * inv_l);
            st_global_v8(dst + c0 / 8 + 2 * q8, w);
          }
        }
      }
      // O has been read: the next unit's first PV may overwrite it.  The
      // second named barrier keeps the exchanged sums stable until both
      // groups have read them.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(BAR_OEMPTY));
        mbar_arrive(bar(BAR_UEMPTY + slot));
      }
      const bool got = __all_sync(0xFFFFFFFFu, wait_unit(k + 1));
      ok = !named_bar_or(2, kSoftmaxThreads, !got || *s_abort != 0);
      G += n;
    }
    if (!ok) {
      *s_abort = 1;
      set_status(a.status, 5 /* SA_ETIMEOUT */);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Key bias: log2 conversion, the sink-only rule, and the flag (status word
// 2) that some bias value is nonzero.
__global__ void bias_prep_kernel(const float* __restrict__ bias, float* __restrict__ b2,
                                 int32_t* status, int T, int video_keys) {
  griddep_launch_dependents();
  griddep_wait();  // b2 may share memory the previous kernel reads
  const float kLog2e = 1.4426950408889634f;
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < T; u += gridDim.x * blockDim.x) {
    const float b = bias[u];
    if (isnan(b) || b == INFINITY) {
      set_status(status, 1 /* SA_EINVAL */);
    } else if (u < video_keys && b != 0.0f) {
      set_status(status, 3 /* SA_ENOSINKBIAS */);
    }
    if (b != 0.0f) status[2] = 1;  // some bias is nonzero (-0 counts as zero)
    b2[u] = b * kLog2e;
  }
}

int sm_count() {
  static int cached[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

size_t attention_smem_bytes() { return kSmemBytes; }

cudaError_t launch_bias_prep(const float* bias, float* b2, int32_t* status, const Geometry& g,
                             cudaStream_t s) {
  const int threads = 256;
  int blocks = (g.T + threads - 1) / threads;
  if (blocks > 1024) blocks = 1024;
  return launch_dependent(bias_prep_kernel, dim3(blocks), dim3(threads), 0, s, bias, b2, status, g.T,
                          g.nvk * kBlock);
}

cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tak, const CUtensorMap& tav, const AttnArgs& a,
                             cudaStream_t s) {
  const bool probe = a.probe_once != 0;
  auto* kern = a.merged ? (probe ? attention_kernel<true, false, true> : attention_kernel<true, false, false>)
                        : (a.fused ? (probe ? attention_kernel<false, true, true> : attention_kernel<false, true, false>)
                                   : (probe ? attention_kernel<false, false, true> : attention_kernel<false, false, false>));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  // The register split redistributes the block's launch allocation; a build
  // that allocated fewer registers per thread would make setmaxnreg.inc wait
  // forever, so refuse to launch it.
  static int regs[6] = {-1, -1, -1, -1, -1, -1};
  int& rg = regs[(a.merged ? 1 : (a.fused ? 2 : 0)) + (probe ? 3 : 0)];
  if (rg < 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    rg = fa.numRegs;
  }
  if (rg * kThreads < static_cast<int>(128 * kRegsControl + 256 * kRegsSoftmax)) return cudaErrorInvalidConfiguration;
  const int units = a.g.H * (a.n_dense + a.n_pairs);
  if (units == 0) return cudaSuccess;
  const int grid = units < sm_count() ? units : sm_count();
  if (a.merged && grid > kMaxMergedCtas) return cudaErrorInvalidConfiguration;
  // The merged forward's attention follows its summaries kernel and is
  // launched as that grid's programmatic dependent; after a memset (the
  // exact and fused forwards) the ordinary launch measured faster.
  if (a.merged)
    return launch_dependent(kern, dim3(grid), dim3(kThreads), kSmemBytes, s, tq, tk, tv, tak, tav, a);
  kern<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, tak, tav, a);
  return cudaGetLastError();
}

}  // namespace sa
