// Spark token reblocking: the landmark tree ("Sol-Attn and Spark for
// MiniMax-H3", section "Spark primitives", spark_reblock; fanout with
// power-of-two scheduling and cosine scoring on normalized FP16 vectors from
// section "Spark inference integration").
//
// Per head, the N = 64 floor(T / 64) leading tokens are split recursively:
// a node of m > 1 blocks of 64 gets c children (the largest power of two not
// above min(fanout, m)) of floor(m / c) or ceil(m / c) blocks.  The node's L
// landmarks are the tokens at positions floor(j n / L) of its current order;
// the two farthest apart in cosine (smallest cosine, ties to the lower pair)
// are a and b, every token gets kappa = cos(t, a) - cos(t, b), and the
// tokens ranked by (kappa, position) are cut into the children, each of
// which keeps the node's order.  The remainder tokens stay last.
//
// GPU shape: one launch writes every token's FP16 unit row; three launches
// per tree level follow: the farthest landmark pair of every split node (a
// CTA per node and head; one Gram entry per thread), the keys of every token
// of the level's split nodes (a warp per 64-token block, eight tokens in
// flight, spread over the whole GPU), and per node an 8-bit radix selection
// of the child boundaries on unique 64-bit keys followed by a stable scatter;
// a last launch writes the permutation and its inverse.
// All floating-point decisions use explicit round-to-nearest FP32 operations
// in a fixed order, so the integer result does not depend on the compiler's
// contractions.

#include <cuda_fp16.h>

#include <algorithm>
#include <vector>

#include "internal.h"

namespace sa {
namespace {

constexpr int kRbThreads = 512;
constexpr int kRbWarps = kRbThreads / 32;
constexpr int kPairThreads = 256;
constexpr int kLandStride = kHeadDim + 4;  // floats per landmark row in shared memory
constexpr int kKeyTokens = 8;  // tokens in flight per warp in the keys kernel

// Sum of a 128-term product held as four terms per lane: the lane's terms
// left to right, then a butterfly over lane offsets 16, 8, 4, 2, 1 (every
// lane ends with the same value).
__device__ __forceinline__ float fold128(float p0, float p1, float p2, float p3) {
  float s = __fadd_rn(__fadd_rn(__fadd_rn(p0, p1), p2), p3);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, off));
  return s;
}

__device__ __forceinline__ float dot128(const float a[4], const float b[4]) {
  return fold128(__fmul_rn(a[0], b[0]), __fmul_rn(a[1], b[1]), __fmul_rn(a[2], b[2]), __fmul_rn(a[3], b[3]));
}

// Order-preserving 32-bit image of a finite float; -0 and +0 are one value.
__device__ __forceinline__ uint32_t order_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ int pow2_children(int m, int fanout) {
  const int lim = m < fanout ? m : fanout;
  int c = 1;
  while (c * 2 <= lim) c *= 2;
  return c;
}

// Node of tree depth `level` that holds block x (blocks of 64 tokens,
// numbered in the final order's span): its first block and block count, or
// the leaf (one block) that holds x when the tree ends above that depth.
__device__ __forceinline__ void find_node(int x, int m_root, int fanout, int level, int& start, int& m,
                                          bool& leaf) {
  start = 0;
  m = m_root;
  leaf = false;
  for (int d = 0; d < level; ++d) {
    if (m == 1) {
      leaf = true;
      return;
    }
    const int c = pow2_children(m, fanout);
    const int base = m / c, extra = m % c;
    const int off = x - start;
    const int i = off < extra * (base + 1) ? off / (base + 1) : extra + (off - extra * (base + 1)) / base;
    start += i * base + (i < extra ? i : extra);
    m = base + (i < extra ? 1 : 0);
  }
  leaf = m == 1;
}

// The same 128-term sum as fold128, by one thread over values in shared
// memory: 32 partial sums of four products left to right, then the
// butterfly's pairings (at offset o, partial l takes partial l + o), which
// reproduce lane 0's operand order exactly.
__device__ __forceinline__ float dot128_serial(const float* a, const float* b) {
  float s[32];
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const float4 x = *reinterpret_cast<const float4*>(a + 4 * l);
    const float4 y = *reinterpret_cast<const float4*>(b + 4 * l);
    s[l] = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(x.x, y.x), __fmul_rn(x.y, y.y)), __fmul_rn(x.z, y.z)),
                     __fmul_rn(x.w, y.w));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
    for (int l = 0; l < o; ++l) s[l] = __fadd_rn(s[l], s[l + o]);
  return s[0];
}

struct Samples {
  const uint16_t* x;  // BF16
  int64_t ts, hs;     // token and head strides (elements)
  __device__ __forceinline__ uint2 raw(int t, int h, int lane) const {
    return *reinterpret_cast<const uint2*>(x + t * ts + h * hs + 4 * lane);
  }
};

// This lane's four values of the FP16 unit row of a BF16 row (held as four
// per lane): ss = sum of squares (exact squares), r = sqrt(ss) and x / r
// rounded to nearest FP32, then to FP16; a zero row stays zero.
__device__ __forceinline__ void unit4(uint2 raw, float u[4]) {
  float v[4];
  v[0] = __uint_as_float(raw.x << 16);
  v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  v[2] = __uint_as_float(raw.y << 16);
  v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  const float r = __fsqrt_rn(dot128(v, v));
#pragma unroll
  for (int e = 0; e < 4; ++e) u[e] = __half2float(__float2half_rn(r > 0.f ? __fdiv_rn(v[e], r) : 0.f));
}

__device__ __forceinline__ void load_half4(const __half* p, float v[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x);
  const __half2 hi = *reinterpret_cast<const __half2*>(&raw.y);
  v[0] = __low2float(lo);
  v[1] = __high2float(lo);
  v[2] = __low2float(hi);
  v[3] = __high2float(hi);
}

// FP16 unit rows of every token t < N of every head, [H, N, 128]: a warp per
// eight tokens of one head, all eight rows in flight.
__global__ void __launch_bounds__(256) reblock_unit_kernel(Samples xs, int N, int H, __half* __restrict__ xh) {
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int groups = (N + kKeyTokens - 1) / kKeyTokens;
  if (w >= static_cast<int64_t>(groups) * H) return;
  const int h = static_cast<int>(w % H), t0 = static_cast<int>(w / H) * kKeyTokens;
  uint2 raw[kKeyTokens];
#pragma unroll
  for (int u = 0; u < kKeyTokens; ++u) raw[u] = xs.raw(min(t0 + u, N - 1), h, lane);
#pragma unroll
  for (int u = 0; u < kKeyTokens; ++u) {
    if (t0 + u >= N) break;
    float v[4];
    unit4(raw[u], v);
    __half2 out[2];
    out[0] = __floats2half2_rn(v[0], v[1]);  // exact: the values are FP16 already
    out[1] = __floats2half2_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(xh + (static_cast<size_t>(h) * N + t0 + u) * kHeadDim + 4 * lane) =
        *reinterpret_cast<const uint2*>(out);
  }
}

// Token at position i of the level's order (the root keeps the flat order).
__device__ __forceinline__ int token_at(const int32_t* ord, size_t hb, int i, int level, int N) {
  return level == 0 ? i : min(max(ord[hb + i], 0), N - 1);  // ids are < N; the clamp only bounds a bad order
}

// Split nodes of one tree level (their first blocks), passed by value.
struct LevelNodes {
  int count;
  int start[kReblockMaxLevelNodes];
};

// The node of depth `level` that starts at block x (a split node).
__device__ __forceinline__ int node_blocks(int x, int m_root, int fanout, int level) {
  int start, m;
  bool leaf;
  find_node(x, m_root, fanout, level, start, m, leaf);
  return m;
}

// Farthest landmark pair of every split node of the level: CTA (k, h).  The
// landmarks' unit rows go to shared memory; each thread takes Gram entries
// in increasing pair number (pairs numbered in (j, j') order) and keeps the
// smallest cosine with a strict <, so ties go to the lower pair.
__global__ void __launch_bounds__(kPairThreads) reblock_pair_kernel(const __half* __restrict__ xh,
                                                                   const int32_t* __restrict__ ord,
                                                                   int2* __restrict__ pairs, int N, int fanout,
                                                                   int L, int level,
                                                                   const __grid_constant__ LevelNodes nodes) {
  constexpr int kWarps = kPairThreads / 32;
  // [L][132]: 16-byte rows for vector loads; 132 = 4 mod 32 words keeps the
  // eight rows a quarter-warp reads in distinct banks
  extern __shared__ __align__(16) float land_raw[];
  auto land = [&](int j) { return land_raw + j * kLandStride; };
  __shared__ int ltok[kReblockMaxLandmarks];
  __shared__ float bc_s[kPairThreads];
  __shared__ int bp_s[kPairThreads];
  const int x = nodes.start[blockIdx.x], h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int m_root = N / kBlock;
  const int n = kBlock * node_blocks(x, m_root, fanout, level);
  const size_t hb = static_cast<size_t>(h) * N;
  const size_t nb0 = hb + static_cast<size_t>(kBlock) * x;  // the node's first position
  const int nl = L < n ? L : n;
  for (int j = warp; j < nl; j += kWarps) {
    const int pos = static_cast<int>((static_cast<int64_t>(j) * n) / nl);
    const int t = level == 0 ? kBlock * x + pos : token_at(ord, nb0, pos, 1, N);
    float u[4];
    load_half4(xh + (hb + t) * kHeadDim + 4 * lane, u);
#pragma unroll
    for (int e = 0; e < 4; ++e) land(j)[4 * lane + e] = u[e];
    if (lane == 0) ltok[j] = t;
  }
  __syncthreads();
  const int P = nl * (nl - 1) / 2;
  float bc = 0.f;
  int bp = -1;
  for (int p = tid; p < P; p += kPairThreads) {
    int j = 0, q = p;
    while (q >= nl - 1 - j) {
      q -= nl - 1 - j;
      ++j;
    }
    const float cs = dot128_serial(land(j), land(j + 1 + q));
    if (bp < 0 || cs < bc) {
      bc = cs;
      bp = p;
    }
  }
  bc_s[tid] = bc;
  bp_s[tid] = bp;
  __syncthreads();
  for (int w = kPairThreads / 2; w > 0; w >>= 1) {
    if (tid < w) {
      const int q = bp_s[tid + w];
      if (q >= 0 && (bp_s[tid] < 0 || bc_s[tid + w] < bc_s[tid] || (bc_s[tid + w] == bc_s[tid] && q < bp_s[tid]))) {
        bc_s[tid] = bc_s[tid + w];
        bp_s[tid] = q;
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    int j = 0, q = bp_s[0];
    while (q >= nl - 1 - j) {
      q -= nl - 1 - j;
      ++j;
    }
    pairs[static_cast<size_t>(h) * m_root + x] = make_int2(ltok[j], ltok[j + 1 + q]);
  }
}

// Keys of every token in a split node of the level: warp per 64-token block
// (16 blocks per CTA), eight tokens in flight per warp.  key = (order bits
// of kappa) << 32 | position in the node, kappa = cos(t, a) - cos(t, b).
__global__ void __launch_bounds__(kRbThreads) reblock_keys_kernel(const __half* __restrict__ xh,
                                                                 const int32_t* __restrict__ ord,
                                                                 const int2* __restrict__ pairs,
                                                                 uint64_t* __restrict__ keys, int N, int fanout,
                                                                 int level) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int x = blockIdx.x * kRbWarps + warp, h = blockIdx.y;
  const int m_root = N / kBlock;
  if (x >= m_root) return;
  int start, m;
  bool leaf;
  find_node(x, m_root, fanout, level, start, m, leaf);
  if (leaf) return;
  const size_t hb = static_cast<size_t>(h) * N;
  const int2 pr = pairs[static_cast<size_t>(h) * m_root + start];
  float a[4], b[4];
  load_half4(xh + (hb + min(max(pr.x, 0), N - 1)) * kHeadDim + 4 * lane, a);
  load_half4(xh + (hb + min(max(pr.y, 0), N - 1)) * kHeadDim + 4 * lane, b);
  const int p0 = kBlock * x;  // first position of the block in the head's order
  const int t_lo = token_at(ord, hb, p0 + lane, level, N);
  const int t_hi = token_at(ord, hb, p0 + 32 + lane, level, N);
  const uint32_t pos0 = static_cast<uint32_t>(kBlock * (x - start));
  for (int r0 = 0; r0 < kBlock; r0 += kKeyTokens) {
    float v[kKeyTokens][4];
#pragma unroll
    for (int u = 0; u < kKeyTokens; ++u) {
      const int r = r0 + u;
      const int t = __shfl_sync(0xFFFFFFFFu, r < 32 ? t_lo : t_hi, r & 31);
      load_half4(xh + (hb + t) * kHeadDim + 4 * lane, v[u]);
    }
    uint64_t mine = 0;
#pragma unroll
    for (int u = 0; u < kKeyTokens; ++u) {
      const float kap = __fsub_rn(dot128(v[u], a), dot128(v[u], b));
      if (lane == u) mine = (static_cast<uint64_t>(order_bits(kap)) << 32) | (pos0 + r0 + u);
    }
    if (lane < kKeyTokens) keys[hb + p0 + r0 + lane] = mine;
  }
}

// Child boundaries and the stable scatter of every split node of the level:
// CTA (k, h).  The keys of ranks cstart[1..c-1] are found by a radix
// selection, 8 bits a pass from the top; boundaries whose prefixes agree
// share a histogram (a key matches at most one prefix), increments are
// aggregated per warp, and the passes stop once every boundary's bin holds
// one key.
template <int kT>
__global__ void __launch_bounds__(kT) reblock_split_kernel(const int32_t* __restrict__ ord_in,
                                                          int32_t* __restrict__ ord_out,
                                                          const uint64_t* __restrict__ keys, int N, int fanout,
                                                          int level, const __grid_constant__ LevelNodes nodes) {
  constexpr int kNb = kReblockMaxFanout - 1;
  constexpr int kW = kT / 32;
  __shared__ uint32_t hist[kNb * 256];
  __shared__ uint64_t prefix[kNb], gprefix[kNb], bound[kNb];
  __shared__ uint32_t rank[kNb], bincnt[kNb];
  __shared__ int bgroup[kNb];
  __shared__ int ngroup, all_single;
  __shared__ int wcnt[kW][kReblockMaxFanout];
  __shared__ int running[kReblockMaxFanout], cstart[kReblockMaxFanout];

  const int x = nodes.start[blockIdx.x], h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int m = node_blocks(x, N / kBlock, fanout, level);
  const int n = kBlock * m;
  const size_t off = static_cast<size_t>(h) * N + static_cast<size_t>(kBlock) * x;
  int32_t* dst = ord_out + off;
  const uint64_t* key = keys + off;
  const int c = pow2_children(m, fanout);
  const int nb = c - 1;
  if (tid < c) {
    const int base = m / c, extra = m % c;
    cstart[tid] = kBlock * (tid * base + (tid < extra ? tid : extra));
    running[tid] = 0;
  }
  __syncthreads();
  if (tid < nb) {
    prefix[tid] = 0;
    rank[tid] = static_cast<uint32_t>(cstart[tid + 1]);  // rank of child tid+1's first token
  }
  int pass = 0;
  for (;; ++pass) {
    const int shift = 56 - 8 * pass;
    if (tid == 0) {
      int ng = 0;
      for (int b = 0; b < nb; ++b) {
        int g = 0;
        while (g < ng && gprefix[g] != prefix[b]) ++g;
        if (g == ng) gprefix[ng++] = prefix[b];
        bgroup[b] = g;
      }
      ngroup = ng;
    }
    __syncthreads();
    const int ng = ngroup;
    for (int e = tid; e < ng * 256; e += kT) hist[e] = 0u;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kT) {
      const int i = i0 + tid;
      int g = -1;
      uint32_t dig = 0;
      if (i < n) {
        const uint64_t k = key[i];
        dig = static_cast<uint32_t>(k >> shift) & 255u;
        if (pass == 0) {
          g = 0;
        } else {
          for (int q = 0; q < ng; ++q)
            if (((k ^ gprefix[q]) >> (shift + 8)) == 0) {
              g = q;
              break;
            }
        }
      }
      const uint32_t tag = g >= 0 ? (static_cast<uint32_t>(g) << 8) | dig : 0x10000u | static_cast<uint32_t>(lane);
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, tag);
      if (g >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[g * 256 + dig], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    // boundary b's bin: a warp scans the 256 counts, eight per lane
    for (int b = warp; b < nb; b += kW) {
      const uint32_t* hg = hist + bgroup[b] * 256 + 8 * lane;
      uint32_t c8[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c8[q] = hg[q];
        sum += c8[q];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum, r = rank[b];
      // the lane whose eight bins hold rank r (counts sum to more than r)
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, r >= excl && r < incl);
      if (lane == __ffs(hit) - 1) {
        uint32_t cum = excl, cnt = 0;
        int sel = -1;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (sel < 0 && (q == 7 || r < cum + c8[q])) {
            sel = q;
            cnt = c8[q];
          } else if (sel < 0) {
            cum += c8[q];
          }
        }
        prefix[b] |= static_cast<uint64_t>(8 * lane + sel) << shift;
        rank[b] = r - cum;
        bincnt[b] = cnt;
      }
    }
    __syncthreads();
    if (tid == 0) {
      int one = 1;
      for (int b = 0; b < nb; ++b) one &= bincnt[b] == 1u ? 1 : 0;
      all_single = one;
    }
    __syncthreads();
    if (all_single || pass == 7) break;
  }
  // The single key of each boundary's bin is the boundary key.
  {
    const int shift = 56 - 8 * pass;
    for (int i = tid; i < n; i += kT) {
      const uint64_t k = key[i];
      for (int b = 0; b < nb; ++b)
        if ((k >> shift) == (prefix[b] >> shift)) bound[b] = k;
    }
  }
  __syncthreads();

  // Stable scatter: child = number of boundary keys <= the token's key;
  // inside a child, tokens keep the node's order.
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += kT) {
    const int i = c0 + tid;
    const bool in = i < n;
    int ch = 0, t = 0;
    if (in) {
      const uint64_t k = key[i];
      for (int b = 0; b < nb; ++b) ch += k >= bound[b] ? 1 : 0;
      t = level == 0 ? kBlock * x + i : ord_in[off + i];
    }
    int my = 0;
    for (int b = 0; b < c; ++b) {
      const unsigned msk = __ballot_sync(0xFFFFFFFFu, in && ch == b);
      if (in && ch == b) my = __popc(msk & lt);
      if (lane == 0) wcnt[warp][b] = __popc(msk);
    }
    __syncthreads();
    if (tid < c) {
      int run = running[tid];
      for (int w = 0; w < kW; ++w) {
        const int v = wcnt[w][tid];
        wcnt[w][tid] = run;
        run += v;
      }
      running[tid] = run;
    }
    __syncthreads();
    const int d = cstart[ch] + wcnt[warp][ch] + my;
    if (in && d < n) dst[d] = t;  // d < n always; the test only keeps a bad split in bounds
    __syncthreads();
  }
}

// perm[h, i] = token at new position i (the remainder keeps its place at the
// end); inv[h, perm[h, i]] = i.  A block's final order sits in the buffer its
// leaf was written to: the one of the parity of the leaf's depth (depth 0,
// a root of one block, is the flat order).
__global__ void reblock_finish_kernel(const int32_t* __restrict__ ord0, const int32_t* __restrict__ ord1, int N,
                                      int T, int H, int fanout, int32_t* __restrict__ perm,
                                      int32_t* __restrict__ inv) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(T) * H) return;
  const int h = static_cast<int>(e / T), i = static_cast<int>(e % T);
  int t = i;
  if (i < N) {
    const int x = i / kBlock, m_root = N / kBlock;
    int start = 0, m = m_root, d = 0;
    while (m > 1) {
      const int c = pow2_children(m, fanout);
      const int base = m / c, extra = m % c;
      const int o = x - start;
      const int j = o < extra * (base + 1) ? o / (base + 1) : extra + (o - extra * (base + 1)) / base;
      start += j * base + (j < extra ? j : extra);
      m = base + (j < extra ? 1 : 0);
      ++d;
    }
    if (d > 0) t = ((d & 1) ? ord1 : ord0)[static_cast<size_t>(h) * N + i];  // a root leaf keeps the flat order
  }
  perm[e] = t;
  if (t >= 0 && t < T) inv[static_cast<size_t>(h) * T + t] = i;
}

}  // namespace

// Levels below a node of m blocks.  Not monotone in m (fanout 8: a node of
// 8 blocks is one level deep, one of 7 two), so both child sizes count.
int reblock_depth(int m, int fanout) {
  if (m <= 1) return 0;
  const int c = pow2_children(m, fanout);
  const int lo = reblock_depth(m / c, fanout);
  const int hi = m % c ? reblock_depth(m / c + 1, fanout) : lo;
  return 1 + (lo > hi ? lo : hi);
}

ReblockLayout reblock_layout(int T, int H) {
  ReblockLayout l;
  const size_t N = static_cast<size_t>(kBlock) * (T / kBlock);
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  size_t off = 0;
  l.xh = off;
  off += up(N * H * kHeadDim * 2);
  l.keys = off;
  off += up(N * H * 8);
  l.ord0 = off;
  off += up(N * H * 4);
  l.ord1 = off;
  off += up(N * H * 4);
  l.pairs = off;
  off += up((N / kBlock) * H * 8);
  l.total = off;
  return l;
}

namespace {
// First blocks of the split nodes of depth `level` (host copy of the walk).
std::vector<int> level_nodes(int m_root, int fanout, int level, int* max_m = nullptr) {
  std::vector<int> out;
  if (max_m) *max_m = 0;
  for (int x = 0; x < m_root; ++x) {
    int start = 0, m = m_root;
    bool leaf = false;
    for (int d = 0; d < level && !leaf; ++d) {
      if (m == 1) {
        leaf = true;
        break;
      }
      const int c = pow2_children(m, fanout);
      const int base = m / c, extra = m % c;
      const int o = x - start;
      const int i = o < extra * (base + 1) ? o / (base + 1) : extra + (o - extra * (base + 1)) / base;
      start += i * base + (i < extra ? i : extra);
      m = base + (i < extra ? 1 : 0);
    }
    if (!leaf && m > 1 && start == x) {
      out.push_back(x);
      if (max_m && m > *max_m) *max_m = m;
    }
  }
  return out;
}
}  // namespace

cudaError_t launch_reblock(const ReblockArgs& r, cudaStream_t stream) {
  const int N = kBlock * (r.T / kBlock);
  const int m_root = N / kBlock;
  const ReblockLayout l = reblock_layout(r.T, r.H);
  char* ws = static_cast<char*>(r.ws);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + l.keys);
  int32_t* ord[2] = {reinterpret_cast<int32_t*>(ws + l.ord0), reinterpret_cast<int32_t*>(ws + l.ord1)};
  int2* pairs = reinterpret_cast<int2*>(ws + l.pairs);
  __half* xh = reinterpret_cast<__half*>(ws + l.xh);
  const Samples xs{r.x, r.token_stride, r.head_stride};
  cudaError_t e;
  const int depth = N > 0 ? reblock_depth(m_root, r.fanout) : 0;
  if (depth > 0) {
    const int64_t warps = static_cast<int64_t>((N + kKeyTokens - 1) / kKeyTokens) * r.H;
    reblock_unit_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(xs, N, r.H, xh);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  for (int lv = 0; lv < depth; ++lv) {
    int max_m = 0;
    const std::vector<int> all = level_nodes(m_root, r.fanout, lv, &max_m);
    const int threads = kBlock * max_m <= 1024 ? 128 : (kBlock * max_m <= 4096 ? 512 : 1024);
    for (int pass = 0; pass < 3; ++pass) {
      if (pass == 1) {
        reblock_keys_kernel<<<dim3((m_root + kRbWarps - 1) / kRbWarps, r.H), kRbThreads, 0, stream>>>(
            xh, ord[lv & 1], pairs, keys, N, r.fanout, lv);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        continue;
      }
      for (size_t k0 = 0; k0 < all.size(); k0 += kReblockMaxLevelNodes) {
        LevelNodes nodes;
        nodes.count = static_cast<int>(std::min<size_t>(kReblockMaxLevelNodes, all.size() - k0));
        for (int k = 0; k < nodes.count; ++k) nodes.start[k] = all[k0 + k];
        const dim3 grid(nodes.count, r.H);
        if (pass == 0)
          reblock_pair_kernel<<<grid, kPairThreads, r.landmarks * kLandStride * sizeof(float), stream>>>(
              xh, ord[lv & 1], pairs, N, r.fanout, r.landmarks, lv, nodes);
        else if (threads == 128)  // CTA size follows the level's node size
          reblock_split_kernel<128><<<grid, 128, 0, stream>>>(ord[lv & 1], ord[(lv + 1) & 1], keys, N, r.fanout,
                                                             lv, nodes);
        else if (threads == 512)
          reblock_split_kernel<512><<<grid, 512, 0, stream>>>(ord[lv & 1], ord[(lv + 1) & 1], keys, N, r.fanout,
                                                             lv, nodes);
        else
          reblock_split_kernel<1024><<<grid, 1024, 0, stream>>>(ord[lv & 1], ord[(lv + 1) & 1], keys, N, r.fanout,
                                                               lv, nodes);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
    }
  }
  const int64_t total = static_cast<int64_t>(r.T) * r.H;
  reblock_finish_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, stream>>>(ord[0], ord[1], N, r.T, r.H,
                                                                                       r.fanout, r.perm, r.inv);
  return cudaGetLastError();
}

}  // namespace sa
