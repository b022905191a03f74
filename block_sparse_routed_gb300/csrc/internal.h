// Definitions shared by the host side of the C ABI and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sa {

constexpr int kBlock = 64;         // tokens per physical block
constexpr int kHeadDim = 128;      // head dimension
constexpr int kStatusBytes = 256;  // device status area at the start of a workspace
constexpr int kMaxList = 1024;     // largest supported block-list width (maxl)
constexpr int kMaxVideoBlocks = 8192;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded on-device waits: 1 s

// Block bookkeeping derived from sa_params (see sparse_attn.h).
struct Geometry {
  int T, H, Nv;
  int nvk;    // full video blocks
  int tail;   // Nv - 64 nvk
  int nblk;   // ceil(T / 64)
  int nq;     // sparse query blocks
  int K;      // Top-K budget
  int R;      // forced local radius
  int pad;    // 1 when the video tail block is routed (pad mode with tail > 0)
  int nsink;  // nblk - nvk
  int maxl;   // block-list width
  int r0;     // first dense query row
};

struct PlanArgs {
  const uint16_t* q;  // BF16 bits [T, H, 128]
  const uint16_t* k;
  float* qc;          // [H, nq, 128]
  float* kc;          // [H, nvk, 128]
  int32_t* idx;       // [H, nq, maxl]
  int32_t* cnt;       // [H, nq]
  float* scores;      // [H, nq, nvk] or null
  int32_t* status;    // the call's status words, zeroed by the pool kernel (or null)
  Geometry g;
};

struct AttnArgs {
  const int32_t* idx;
  const int32_t* cnt;
  const float* b2;     // key bias in log2 units [T], or null
  uint16_t* o;         // BF16 bits [T, H, 128]
  int32_t* status;     // device status word
  int32_t* unit_counter;  // next work unit (zeroed before the launch)
  const int32_t* bias_nz; // 1 when some key bias is nonzero (set by the bias prep)
  Geometry g;
  int n_dense;         // dense 128-row tiles per head
  int n_pairs;         // sparse query-block pairs per head
  float scale_log2;    // log2(e) / sqrt(128)
  // merged (Spark) mode: skipped video blocks enter as summary keys
  int merged;
  const float* lm2;    // log-mass in log2 units [H, nblkp]
  int nblkp;           // row stride of lm2 (a multiple of 64)
  float* vbias;        // per CTA and descriptor slot: summary-key logits [nvc][2][64]
  int vstride;         // floats per (CTA, slot): nvc * 2 * 64
  // fused mode: the kernel routes each unit from the block means and
  // exports the lists to idx_w / cnt_w (then read back as idx / cnt)
  int fused;
  const float* qc;     // [H, nq, 128]
  const float* kc;     // [H, nvk, 128]
  int32_t* idx_w;
  int32_t* cnt_w;
  int probe_once;      // testing build: every pipeline wait is a single probe
};

constexpr int kMaxFusedVideoBlocks = 256;  // video key blocks a fused route supports

constexpr int kMaxMergedCtas = 256;  // CTAs a merged launch may use (summary-key logit rows)

struct ReweightArgs {
  const uint16_t* a;   // BF16 anchors [P, H, 128]
  const uint16_t* k;   // BF16 [T, H, 128]
  const uint16_t* v;
  uint16_t* ak;        // BF16 [P, H, nblk, 128]
  uint16_t* av;
  float* lm;           // [P, H, nblk]
  int T, H, P, nblk;
  // Optional (merged forward, P = 1): lm in log2 units for the attention
  // kernel, [H, nblkp], 0 for blocks >= nvk and the padding.
  float* lm2;
  int nvk, nblkp;
};

// Launches `kern` with programmatic stream serialization: it may start while
// the stream's previous kernel finishes, and waits for that kernel on the
// device (griddep_wait) before touching what it wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Records a failed CUDA call for sparse_attn_last_cuda_error (thread-local,
// defined in api.cu); returns true when `e` is an error.
bool cuda_failed(cudaError_t e);

// Launchers (defined in the kernel translation units).
cudaError_t launch_pool(const PlanArgs& a, cudaStream_t s);
cudaError_t launch_route_topk(const PlanArgs& a, cudaStream_t s);
cudaError_t launch_bias_prep(const float* bias, float* b2, int32_t* status, const Geometry& g,
                             cudaStream_t s);
cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tak, const CUtensorMap& tav, const AttnArgs& a,
                             cudaStream_t s);
cudaError_t launch_spark_reweight(const ReweightArgs& r, cudaStream_t s);

// Spark token reblocking (landmark tree).
constexpr int kReblockMaxLandmarks = 64;
constexpr int kReblockMaxFanout = 16;
constexpr int kReblockMaxLevelNodes = 2000;  // split nodes per launch (the list is a kernel parameter)

struct ReblockArgs {
  const uint16_t* x;     // BF16 samples: row (t, h) at x + t * token_stride + h * head_stride
  int64_t token_stride;  // elements
  int64_t head_stride;   // elements
  int T, H, fanout, landmarks;
  int32_t* perm;         // [H, T]
  int32_t* inv;          // [H, T]
  void* ws;              // reblock_layout(T, H).total bytes, 256-byte aligned
};

struct ReblockLayout {
  size_t xh, keys, ord0, ord1, pairs, total;  // byte offsets: FP16 unit rows [H, N, 128], keys [H, N],
                                              // orders [H, N], landmark pairs int2 [H, N / 64]
};

ReblockLayout reblock_layout(int T, int H);
int reblock_depth(int m, int fanout);
cudaError_t launch_reblock(const ReblockArgs& r, cudaStream_t s);
int anchor_chunks(int Nv);
cudaError_t launch_video_query_mean(const uint16_t* q, float* partial, uint16_t* anchor, int H, int Nv,
                                    cudaStream_t s);
size_t route_topk_smem_bytes(const Geometry& g);
size_t attention_smem_bytes();

}  // namespace sa
