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
// GPU shape: one launch normalises every token to an FP16 unit row; one
// launch per tree level splits every node of that level for every head (a
// CTA per node and head: landmark pair, keys, an 8-pass radix selection of
// the child boundaries on unique 64-bit keys, then a stable scatter); a last
// launch writes the permutation and its inverse.  All floating-point
// decisions use explicit round-to-nearest FP32 operations in a fixed order,
// so the integer result does not depend on the compiler's contractions.

#include <cuda_fp16.h>

#include "internal.h"

namespace sa {
namespace {

constexpr int kRbThreads = 512;
constexpr int kRbWarps = kRbThreads / 32;
constexpr int kUnitWarps = 8;

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

__device__ __forceinline__ void load_half4(const __half* p, float v[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x);
  const __half2 hi = *reinterpret_cast<const __half2*>(&raw.y);
  v[0] = __low2float(lo);
  v[1] = __high2float(lo);
  v[2] = __low2float(hi);
  v[3] = __high2float(hi);
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
// numbered in the final order's span): its first block and block count.
// `leaf` when the walk met a finished leaf before that depth.
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

// Warp per (token t < N, head h): the FP16 unit row of x[t, h] and the
// identity order.  ss = sum of squares (exact squares of BF16 values), r =
// sqrt(ss) and x / r rounded to nearest; a zero row stays zero.
__global__ void __launch_bounds__(kUnitWarps * 32) reblock_unit_kernel(const uint16_t* __restrict__ x, int64_t ts,
                                                                      int64_t hs, int N, int H,
                                                                      __half* __restrict__ xh,
                                                                      int32_t* __restrict__ ord) {
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kUnitWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (w >= static_cast<int64_t>(N) * H) return;
  const int t = static_cast<int>(w / H), h = static_cast<int>(w % H);
  const uint2 raw = *reinterpret_cast<const uint2*>(x + t * ts + h * hs + 4 * lane);
  float v[4];
  v[0] = __uint_as_float(raw.x << 16);
  v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  v[2] = __uint_as_float(raw.y << 16);
  v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  const float ss = dot128(v, v);
  const float r = __fsqrt_rn(ss);
  __half2 out[2];
  float y[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) y[e] = r > 0.f ? __fdiv_rn(v[e], r) : 0.f;
  out[0] = __halves2half2(__float2half_rn(y[0]), __float2half_rn(y[1]));
  out[1] = __halves2half2(__float2half_rn(y[2]), __float2half_rn(y[3]));
  const size_t row = static_cast<size_t>(h) * N + t;
  *reinterpret_cast<uint2*>(xh + row * kHeadDim + 4 * lane) = *reinterpret_cast<const uint2*>(out);
  if (lane == 0) ord[row] = t;
}

// One tree level: CTA (x, h) splits the node of this depth whose first
// block is x (or copies a finished leaf); other CTAs return at once.
__global__ void __launch_bounds__(kRbThreads) reblock_level_kernel(const __half* __restrict__ xh,
                                                                  const int32_t* __restrict__ ord_in,
                                                                  int32_t* __restrict__ ord_out,
                                                                  uint64_t* __restrict__ keys, int N, int fanout,
                                                                  int L, int level) {
  __shared__ __align__(16) __half land[kReblockMaxLandmarks][kHeadDim];
  __shared__ float ua[kHeadDim], ub[kHeadDim];
  __shared__ float wbest_c[kRbWarps];
  __shared__ int wbest_p[kRbWarps];
  __shared__ uint32_t hist[(kReblockMaxFanout - 1) * 256];
  __shared__ uint64_t prefix[kReblockMaxFanout - 1];
  __shared__ uint32_t rank[kReblockMaxFanout - 1];
  __shared__ int wcnt[kRbWarps][kReblockMaxFanout];
  __shared__ int running[kReblockMaxFanout], cstart[kReblockMaxFanout];
  __shared__ int pair[2];

  const int x = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int start, m;
  bool leaf;
  find_node(x, N / kBlock, fanout, level, start, m, leaf);
  if (start != x) return;
  const size_t hb = static_cast<size_t>(h) * N;
  const int n = kBlock * m;
  const int32_t* src = ord_in + hb + static_cast<size_t>(kBlock) * start;
  int32_t* dst = ord_out + hb + static_cast<size_t>(kBlock) * start;
  uint64_t* key = keys + hb + static_cast<size_t>(kBlock) * start;
  if (leaf) {
    for (int i = tid; i < n; i += kRbThreads) dst[i] = src[i];
    return;
  }
  const int c = pow2_children(m, fanout);
  const int nb = c - 1;
  const int nl = L < n ? L : n;

  // Landmark rows.
  for (int j = warp; j < nl; j += kRbWarps) {
    const int pos = static_cast<int>((static_cast<int64_t>(j) * n) / nl);
    const int t = min(max(src[pos], 0), N - 1);  // token ids are < N; the clamp only bounds a bad order
    *reinterpret_cast<uint2*>(&land[j][4 * lane]) =
        *reinterpret_cast<const uint2*>(xh + (hb + t) * kHeadDim + 4 * lane);
  }
  if (tid < c) {
    const int base = m / c, extra = m % c;
    cstart[tid] = kBlock * (tid * base + (tid < extra ? tid : extra));
    running[tid] = 0;
  }
  __syncthreads();

  // Farthest landmark pair: the smallest cosine, ties to the lower pair in
  // (j, j') order (pairs are numbered in that order; each warp walks its
  // share in increasing number, so a strict < keeps the lowest).
  {
    float bc = 0.f;
    int bp = -1;
    int p = 0;
    for (int j = 0; j < nl; ++j) {
      float a[4];
      a[0] = __half2float(land[j][4 * lane]);
      a[1] = __half2float(land[j][4 * lane + 1]);
      a[2] = __half2float(land[j][4 * lane + 2]);
      a[3] = __half2float(land[j][4 * lane + 3]);
      for (int jj = j + 1; jj < nl; ++jj, ++p) {
        if (p % kRbWarps != warp) continue;
        float b[4];
        b[0] = __half2float(land[jj][4 * lane]);
        b[1] = __half2float(land[jj][4 * lane + 1]);
        b[2] = __half2float(land[jj][4 * lane + 2]);
        b[3] = __half2float(land[jj][4 * lane + 3]);
        const float cs = dot128(a, b);
        if (bp < 0 || cs < bc) {
          bc = cs;
          bp = p;
        }
      }
    }
    if (lane == 0) {
      wbest_c[warp] = bc;
      wbest_p[warp] = bp;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float bc = 0.f;
    int bp = -1;
    for (int w = 0; w < kRbWarps; ++w) {
      const int p = wbest_p[w];
      if (p < 0) continue;
      if (bp < 0 || wbest_c[w] < bc || (wbest_c[w] == bc && p < bp)) {
        bc = wbest_c[w];
        bp = p;
      }
    }
    int j = 0;
    while (bp >= nl - 1 - j) {
      bp -= nl - 1 - j;
      ++j;
    }
    pair[0] = j;
    pair[1] = j + 1 + bp;
  }
  __syncthreads();
  if (tid < kHeadDim) {
    ua[tid] = __half2float(land[pair[0]][tid]);
    ub[tid] = __half2float(land[pair[1]][tid]);
  }
  __syncthreads();

  // Keys: (order bits of kappa) << 32 | position, unique within the node.
  {
    float a[4], b[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a[e] = ua[4 * lane + e];
      b[e] = ub[4 * lane + e];
    }
    for (int i = warp; i < n; i += kRbWarps) {
      const int t = min(max(src[i], 0), N - 1);
      float v[4];
      load_half4(xh + (hb + t) * kHeadDim + 4 * lane, v);
      const float kap = __fsub_rn(dot128(v, a), dot128(v, b));
      if (lane == 0) key[i] = (static_cast<uint64_t>(order_bits(kap)) << 32) | static_cast<uint32_t>(i);
    }
  }
  if (tid < nb) {
    prefix[tid] = 0;
    rank[tid] = static_cast<uint32_t>(cstart[tid + 1]);  // rank of child tid+1's first token
  }
  __syncthreads();

  // Radix selection of the keys of ranks cstart[1..c-1], 8 bits per pass.
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int e = tid; e < nb * 256; e += kRbThreads) hist[e] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kRbThreads) {
      const uint64_t k = key[i];
      const uint32_t dig = static_cast<uint32_t>(k >> shift) & 255u;
      for (int b = 0; b < nb; ++b)
        if (pass == 0 || ((k ^ prefix[b]) >> (shift + 8)) == 0) atomicAdd(&hist[b * 256 + dig], 1u);
    }
    __syncthreads();
    if (tid < nb) {
      const uint32_t r = rank[tid];
      uint32_t cum = 0;
      int d = 0;
      for (; d < 255; ++d) {
        const uint32_t hc = hist[tid * 256 + d];
        if (r < cum + hc) break;
        cum += hc;
      }
      prefix[tid] |= static_cast<uint64_t>(d) << shift;
      rank[tid] = r - cum;
    }
    __syncthreads();
  }

  // Stable scatter: child = number of boundary keys <= the token's key;
  // inside a child, tokens keep the node's order.
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += kRbThreads) {
    const int i = c0 + tid;
    const bool in = i < n;
    int ch = 0, t = 0;
    if (in) {
      const uint64_t k = key[i];
      for (int b = 0; b < nb; ++b) ch += k >= prefix[b] ? 1 : 0;
      t = src[i];
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
      for (int w = 0; w < kRbWarps; ++w) {
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
// end); inv[h, perm[h, i]] = i.
__global__ void reblock_finish_kernel(const int32_t* __restrict__ ord, int N, int T, int H,
                                      int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(T) * H) return;
  const int h = static_cast<int>(e / T), i = static_cast<int>(e % T);
  const int t = i < N ? ord[static_cast<size_t>(h) * N + i] : i;
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
  l.total = off;
  return l;
}

cudaError_t launch_reblock(const ReblockArgs& r, cudaStream_t stream) {
  const int N = kBlock * (r.T / kBlock);
  const ReblockLayout l = reblock_layout(r.T, r.H);
  char* ws = static_cast<char*>(r.ws);
  __half* xh = reinterpret_cast<__half*>(ws + l.xh);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + l.keys);
  int32_t* ord[2] = {reinterpret_cast<int32_t*>(ws + l.ord0), reinterpret_cast<int32_t*>(ws + l.ord1)};
  int depth = 0;
  if (N > 0) {
    const int64_t warps = static_cast<int64_t>(N) * r.H;
    reblock_unit_kernel<<<static_cast<unsigned>((warps + kUnitWarps - 1) / kUnitWarps), kUnitWarps * 32, 0, stream>>>(
        r.x, r.token_stride, r.head_stride, N, r.H, xh, ord[0]);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    depth = reblock_depth(N / kBlock, r.fanout);
    for (int lv = 0; lv < depth; ++lv) {
      reblock_level_kernel<<<dim3(N / kBlock, r.H), kRbThreads, 0, stream>>>(xh, ord[lv & 1], ord[(lv + 1) & 1], keys,
                                                                             N, r.fanout, r.landmarks, lv);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  const int64_t total = static_cast<int64_t>(r.T) * r.H;
  reblock_finish_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, stream>>>(ord[depth & 1], N, r.T, r.H,
                                                                                       r.perm, r.inv);
  return cudaGetLastError();
}

int reblock_launches(int T, int fanout) {
  const int N = kBlock * (T / kBlock);
  return N > 0 ? 2 + reblock_depth(N / kBlock, fanout) : 1;
}

}  // namespace sa
