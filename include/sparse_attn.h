/*
 * sparse_attn.h -- C ABI of the GB300 (sm_103a) Top-K block-sparse routed
 * attention library (forward pass, one GPU, one process).
 *
 * The method (sources are web pages, cited by title and section):
 *
 *   Q, K, V are contiguous BF16 [B=1, T, H, 128] ("Sol-Attn and Spark for
 *   MiniMax-H3", section "Install").  T is a target-video prefix of
 *   `video_tokens` tokens followed by a context suffix (same page, "H3
 *   pipeline integration").  Blocks are 64 tokens.  Let
 *     nvk  = floor(video_tokens / 64)      full video blocks (routed keys)
 *     nblk = ceil(T / 64)                  physical key blocks
 *     sinks = blocks nvk .. nblk-1         context sink blocks (always exact)
 *     K    = min(nvk, ceil(topk_ratio * nvk))
 *   sparse_attn_plan mean-pools Q and K per block, scores every video query
 *   block against every video key block, s = Qmean . Kmean / sqrt(128)
 *   ("Spark inference integration": native mean Top-K routing, packed route
 *   exported once), keeps the K best blocks by FP32 score (ties to the lower
 *   index) among the non-local video blocks, and adds the self block, its
 *   +-radius neighbours and every sink block outside the budget ("H3
 *   pipeline integration", sol_exact_block_radius; "Add key bias to chunked
 *   Sol-Attn producers", "Tests and source audit": sinks go straight into the
 *   exact list).
 *   sparse_attn_fwd runs exact softmax attention of each video query block
 *   over the union of its list, and dense attention over every key for the
 *   context rows and, with tail_mode = SA_TAIL_DENSE, for the rows of a video
 *   block cut by the boundary ("H3 pipeline integration").  With
 *   SA_TAIL_PAD that block is routed and attends sparsely; its centroid is
 *   the mean of its real video rows.  An optional key bias in natural-log
 *   units is added to the logits of sink keys only ("Add key bias to chunked
 *   Sol-Attn producers", "Summary" and "Contract").
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller, 16-byte aligned and contiguous; the output `o` of
 *     the attention calls is 32-byte aligned (its rows are written by
 *     32-byte stores).  No entry point
 *     allocates device memory (the one fixed scratch array of
 *     sparse_attn_plan_static is part of the loaded library).
 *   - All GPU work is enqueued on `stream`; plan and fwd never synchronise
 *     the host.  Argument errors are returned before anything is enqueued.
 *   - A workspace `ws` of the size reported by sparse_attn_query belongs to
 *     one stream at a time; its first 256 bytes hold a device status word.
 *   - No fallback: when the GPU path cannot run, the call fails.
 */
#ifndef SPARSE_ATTN_H_
#define SPARSE_ATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SA_ABI_VERSION 1u

typedef enum sa_status {
  SA_OK = 0,
  SA_EINVAL = 1,        /* bad argument, shape, pointer, size or key-bias value  */
  SA_EUNSUPPORTED = 2,  /* outside what this build supports (B != 1, D != 128,
                           a device that is not sm_103, sizes past the limits) */
  SA_ENOSINKBIAS = 3,   /* nonzero key bias on a routed video key (u < 64 nvk)  */
  SA_ECUDA = 4,         /* a CUDA runtime call or a kernel launch failed        */
  SA_ETIMEOUT = 5       /* a bounded on-device wait gave up; outputs invalid    */
} sa_status;

typedef enum sa_tail_mode { SA_TAIL_DENSE = 0, SA_TAIL_PAD = 1 } sa_tail_mode;

/* Problem description, passed by pointer to every call. */
typedef struct sa_params {
  uint32_t abi_version; /* must be SA_ABI_VERSION                               */
  int32_t B;            /* batch, must be 1 (packed batch size one)             */
  int32_t T;            /* packed tokens, >= 1                                  */
  int32_t H;            /* heads, >= 1                                          */
  int32_t D;            /* head dimension, must be 128                          */
  int32_t video_tokens; /* target-video prefix length Nv, 64 <= Nv <= T         */
  int32_t radius;       /* forced local radius R >= 0                           */
  int32_t tail_mode;    /* sa_tail_mode                                         */
  double topk_ratio;    /* Top-K ratio in (0, 1]; K = min(nvk, ceil(r * nvk)),
                           the product rounded as a decimal: a relative slack
                           of 1e-9 absorbs the binary representation of r     */
} sa_params;

/* Derived sizes and workspace requirements. */
typedef struct sa_sizes {
  int32_t nvk;             /* full video blocks                               */
  int32_t tail;            /* video_tokens - 64 nvk                           */
  int32_t nblk;            /* ceil(T / 64)                                    */
  int32_t nq;              /* sparse query blocks: nvk, +1 for a pad tail     */
  int32_t topk;            /* K                                               */
  int32_t nsink;           /* nblk - nvk                                      */
  int32_t maxl;            /* list width: min(nvk, 2R + 1 + K) + nsink        */
  int32_t dense_row_start; /* first densely evaluated query row               */
  uint64_t plan_ws_bytes;  /* workspace bytes for sparse_attn_plan            */
  uint64_t fwd_ws_bytes;   /* workspace bytes for sparse_attn_fwd             */
} sa_sizes;

/*
 * Validates `p` and fills `out`.  Host only: touches no device.
 * Errors: SA_EINVAL (null pointer, abi_version mismatch, T < 1, H < 1,
 * video_tokens outside [64, T], topk_ratio outside (0, 1], radius < 0,
 * unknown tail_mode, pad mode with T < 64 (nvk + 1) when the video tail is
 * nonempty); SA_EUNSUPPORTED (B != 1, D != 128, nvk > 8192, maxl > 1024,
 * T * H * 128 beyond 2^31 elements).
 */
sa_status sparse_attn_query(const sa_params* p, sa_sizes* out);

/*
 * Routing: pool + route scores + Top-K + block lists.
 *   q, k          BF16 [1, T, H, 128]
 *   idx           int32 [1, H, nq, maxl]: row (h, i) holds the sorted block
 *                 list of query block i in head h, padded with -1
 *   cnt           int32 [1, H, nq]: list lengths
 *   route_scores  optional (may be NULL) float32 [H, nq, nvk]: the scores
 *                 the selection compared (Qmean . Kmean / sqrt(128))
 *   ws, ws_bytes  workspace of at least plan_ws_bytes.  Layout after the
 *                 256-byte status area: Qmean float32 [H, nq, 128], then
 *                 Kmean float32 [H, nvk, 128], each 256-byte aligned.
 * Errors before launch: as sparse_attn_query, plus SA_EINVAL for a null or
 * misaligned required pointer or a short workspace.  SA_ECUDA if a launch
 * fails.
 */
sa_status sparse_attn_plan(const sa_params* p, const void* q, const void* k, int32_t* idx,
                           int32_t* cnt, float* route_scores, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/*
 * Attention: sparse video blocks over their lists, dense rows over all keys.
 *   q, k, v   BF16 [1, T, H, 128]
 *   key_bias  optional (may be NULL) float32 [B * T] in natural-log units.
 *             Converted once to log2 units.  Must be 0 on every key
 *             u < 64 nvk (else SA_ENOSINKBIAS); NaN or +inf anywhere gives
 *             SA_EINVAL; -inf removes the key.  Both are device-detected:
 *             read them with sparse_attn_last_device_status.
 *   idx, cnt  block lists from sparse_attn_plan (same params).  Lists are
 *             checked on the device before any of their blocks is loaded:
 *             1 <= cnt <= maxl, entries in [0, nblk) and strictly increasing,
 *             else SA_EINVAL (device-detected)
 *   o         BF16 [1, T, H, 128], 32-byte aligned; every row is written
 *             when the device status is SA_OK
 *   ws        workspace of at least fwd_ws_bytes (may alias none of the
 *             tensors above)
 * Errors before launch: as sparse_attn_plan.  Device-detected conditions
 * leave `o` unspecified and are reported by sparse_attn_last_device_status.
 */
sa_status sparse_attn_fwd(const sa_params* p, const void* q, const void* k, const void* v,
                          const float* key_bias, const int32_t* idx, const int32_t* cnt, void* o,
                          void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Routing without a caller workspace: the same computation and outputs as
 * sparse_attn_plan, with its scratch (status word and block means) kept in a
 * file-scope device array of SA_PLAN_STATIC_SCRATCH_BYTES instead of `ws`.
 * The source pages have no counterpart to this entry point.  It is for
 * callers that cannot give the library device scratch memory: plugins in a
 * host application whose device memory belongs to the host's own pool
 * allocator with no allocation hook for plugins, and code that must not call
 * cudaMalloc because it synchronises the device.  It allocates nothing.
 *   - Every GPU that loads the library holds the array until process exit.
 *   - Problems whose plan workspace (sparse_attn_query's plan_ws_bytes)
 *     exceeds SA_PLAN_STATIC_SCRATCH_BYTES return SA_EUNSUPPORTED before any
 *     launch.  The five reference workloads need at most 25.2 MiB.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents: calls
 *     that overlap on the GPU (several streams or host threads) race, and the
 *     caller must serialise them.  The status area is cleared on each call.
 * Errors: as sparse_attn_plan (no workspace arguments).
 */
#define SA_PLAN_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
sa_status sparse_attn_plan_static(const sa_params* p, const void* q, const void* k, int32_t* idx,
                                  int32_t* cnt, float* route_scores, cudaStream_t stream);

/*
 * Spark virtual summaries ("Sol-Attn and Spark for MiniMax-H3", section
 * "Spark primitives", spark_reweight; default numerics from section "Spark
 * inference integration").  For every anchor p, head h and physical 64-token
 * block b of K/V (a partial last block uses only its T - 64 b real keys):
 *     s_u = a[p, h] . k[u, h] / sqrt(128),   w = softmax over the block's u
 *     ak[p, h, b] = sum_u w_u k[u, h]        BF16 (round to nearest even)
 *     av[p, h, b] = sum_u w_u v[u, h]        BF16
 *     lm[p, h, b] = logsumexp_u(s_u) - a[p, h] . ak[p, h, b] / sqrt(128)
 * where the ak in lm is the stored BF16 value.  Scores, weights and sums are
 * FP32.  It does not choose anchors, routes or merge outputs.
 *   a        BF16 [1, P, H, 128] anchors (query representatives)
 *   k, v     BF16 [1, T, H, 128]
 *   ak, av   BF16 [1, P, H, nblk, 128], nblk = ceil(T / 64)
 *   lm       float32 [1, P, H, nblk]
 * Errors before launch: SA_EINVAL (null params or tensor pointer,
 * abi_version mismatch, T < 1, H < 1, P < 1, a tensor pointer not 16-byte
 * aligned, lm not 4-byte aligned); SA_EUNSUPPORTED (B != 1, D != 128,
 * T * H * 128 or P * H * nblk * 128 beyond 2^31 elements, a device that is
 * not sm_103).  SA_ECUDA if the launch fails.  Nothing is device-detected.
 */
typedef struct sa_reweight_params {
  uint32_t abi_version; /* must be SA_ABI_VERSION                               */
  int32_t B;            /* batch, must be 1                                     */
  int32_t T;            /* tokens of K and V, >= 1                              */
  int32_t H;            /* heads, >= 1                                          */
  int32_t D;            /* head dimension, must be 128                          */
  int32_t P;            /* anchors per head, >= 1                               */
} sa_reweight_params;

sa_status sparse_attn_spark_reweight(const sa_reweight_params* p, const void* a, const void* k,
                                     const void* v, void* ak, void* av, float* lm,
                                     cudaStream_t stream);

/*
 * Spark's merged attention ("Sol-Attn and Spark for MiniMax-H3", section
 * "Spark inference integration": one global representative per head formed
 * by averaging all target-video queries, stored as BF16; global-anchor K/V
 * and log-mass summaries merged with exact attention).  Same arguments,
 * lists and exact part as sparse_attn_fwd; in addition, per head, the
 * anchor a = BF16(mean of q rows t < video_tokens) is formed, its summaries
 * of every key block are computed as by sparse_attn_spark_reweight (P = 1),
 * and every video key block j < nvk that a sparse query block's list skips
 * enters that block's softmax as one extra key: ak[h, j] with logit
 * q . ak[h, j] / sqrt(128) + lm[h, j] and value av[h, j].  Dense rows are
 * exact over all keys as in sparse_attn_fwd.  The source pages have no
 * separate name for this call.
 *   ws  workspace of at least sparse_attn_spark_ws_bytes(p) bytes, 256-byte
 *       aligned.  Layout after the 256-byte status area (each part 256-byte
 *       aligned): key bias in log2 units float32 [T]; anchors BF16 [H, 128];
 *       anchor partial sums float32 [H, ceil(video_tokens / 1024), 128];
 *       ak, av BF16 [H, nblk, 128]; lm float32 [H, nblk]; lm in log2 units
 *       float32 [H, 64 ceil(nvk / 64)]; summary-key logits of each
 *       attention CTA float32 [256][2][ceil(nvk / 64)][2][64].
 * Errors: as sparse_attn_fwd (with this workspace size); SA_EUNSUPPORTED
 * also when H * nblk * 128 reaches 2^31.
 */
sa_status sparse_attn_spark_ws_bytes(const sa_params* p, uint64_t* out);
sa_status sparse_attn_spark_fwd(const sa_params* p, const void* q, const void* k, const void* v,
                                const float* key_bias, const int32_t* idx, const int32_t* cnt,
                                void* o, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Routing and attention in one call, with the Top-K taken inside the
 * attention kernel ("Sol-Attn and Spark for MiniMax-H3", section "Spark
 * inference integration": CTA-local fused Top-K routing, which removes the
 * external route pass).  Computes exactly what sparse_attn_plan followed by
 * sparse_attn_fwd computes, with the same FP32 scores and selection rule:
 * block means first, then each attention work unit scores its query blocks
 * against every video key block's mean, selects, and walks the lists it
 * made.  The lists are exported to idx / cnt (the layout of
 * sparse_attn_plan's outputs; here outputs of this call).
 *   ws  workspace of at least sparse_attn_fused_ws_bytes(p) bytes, 256-byte
 *       aligned: 256-byte status area, key bias in log2 units float32 [T],
 *       Qmean float32 [H, nq, 128], Kmean float32 [H, nvk, 128] (each part
 *       256-byte aligned).
 * Errors: as sparse_attn_fwd (with this workspace size); SA_EUNSUPPORTED
 * also when nvk > 256 (rows of at most 256 video blocks are routed in one
 * warp's registers).
 */
sa_status sparse_attn_fused_ws_bytes(const sa_params* p, uint64_t* out);
sa_status sparse_attn_fused(const sa_params* p, const void* q, const void* k, const void* v,
                            const float* key_bias, int32_t* idx, int32_t* cnt, void* o, void* ws,
                            size_t ws_bytes, cudaStream_t stream);

/*
 * Spark token reblocking ("Sol-Attn and Spark for MiniMax-H3", section
 * "Spark primitives", spark_reblock: a permutation of each head's tokens
 * into 64-token blocks by a landmark tree, with its inverse; fanout with
 * power-of-two scheduling and cosine scoring on normalized FP16 vectors from
 * section "Spark inference integration").  The pages name the ingredients,
 * not the steps; this call computes, per head h independently:
 *   N = 64 floor(T / 64); tokens t >= N (the flat order's remainder) keep
 *   their place at the end.  Each token is scored as its FP16 unit vector
 *   (FP32 norm, zero rows stay zero).  The root node is [0, N) in flat
 *   order; a node of m > 1 blocks splits into c children, c the largest
 *   power of two <= min(fanout, m), child i taking floor(m / c) + [i < m % c]
 *   blocks.  Its landmarks are the tokens at positions floor(j n / L),
 *   j < L = min(landmarks, n), of its current order (n tokens); the pair
 *   with the smallest cosine (ties to the lower (j, j')) gives a and b;
 *   tokens ranked by (cos(t, a) - cos(t, b), position) fill child 0, 1, ...
 *   in turn, and each child keeps the node's order.  Leaves are the blocks.
 *   Cosines are FP32 sums of exact FP16 products in a fixed order (per
 *   lane four consecutive terms left to right, then a butterfly over 32
 *   lanes), so the integer result is reproducible bit for bit.
 *   x      BF16 samples, row (t, h) at x + t * token_stride + h * head_stride
 *          (elements; [1, T, H, 128] has token_stride = 128 H, head_stride =
 *          128); 16-byte aligned, strides multiples of 8.  Read only.
 *   perm   int32 [H, T]: perm[h, i] = original token at new position i;
 *          the blocks are perm[h, 64 b : 64 b + 64], the excluded remainder
 *          perm[h, N:].
 *   inv    int32 [H, T]: inv[h, perm[h, i]] = i.
 *   ws     workspace of sparse_attn_reblock_ws_bytes(p) bytes, 256-byte
 *          aligned: FP16 unit rows [H, N, 128], keys uint64 [H, N], two
 *          orders int32 [H, N], landmark pairs int32 [H, N / 64, 2] (each
 *          256-byte aligned).  Owned by the caller.
 * Errors before launch: SA_EINVAL (null params or pointer, abi_version
 * mismatch, T < 1, H < 1, fanout not a power of two in [2, 16], landmarks
 * outside [2, 64], a negative stride or one not a multiple of 8, x not
 * 16-byte aligned, perm or inv not 4-byte aligned, ws not 256-byte aligned or
 * short); SA_EUNSUPPORTED (D != 128, H > 65535, T * H >= 2^31, a device that
 * is not sm_103).  SA_ECUDA if a launch fails.  Nothing is device-detected.
 */
typedef struct sa_reblock_params {
  uint32_t abi_version; /* must be SA_ABI_VERSION                               */
  int32_t T;            /* tokens, >= 1                                         */
  int32_t H;            /* heads (independent sample matrices), >= 1            */
  int32_t D;            /* feature dimension, must be 128                       */
  int32_t fanout;       /* children per split at most: 2, 4, 8 or 16            */
  int32_t landmarks;    /* landmarks per split, [2, 64] (32 by default)         */
  int64_t token_stride; /* elements between tokens t and t + 1 of one head      */
  int64_t head_stride;  /* elements between heads h and h + 1 of one token      */
} sa_reblock_params;

sa_status sparse_attn_reblock_ws_bytes(const sa_reblock_params* p, uint64_t* out);
sa_status sparse_attn_spark_reblock(const sa_reblock_params* p, const void* x, int32_t* perm,
                                    int32_t* inv, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Reads the device status word of `ws` (written by the last plan or fwd
 * enqueued with it).  Synchronises `stream`.  SA_ECUDA if the copy fails.
 */
sa_status sparse_attn_last_device_status(const void* ws, cudaStream_t stream, sa_status* out);

/*
 * Testing hook (the source pages have no counterpart).  Every on-device
 * pipeline wait of the attention kernels gives up after 1 s: the kernel then
 * records SA_ETIMEOUT in the workspace status word, lets its own copies and
 * MMAs in flight finish (those waits keep the 1 s limit), frees its tensor
 * memory and returns; the outputs of that call are invalid.  With `on`
 * nonzero, later launches by sparse_attn_fwd, sparse_attn_spark_fwd and
 * sparse_attn_fused use a build of the kernel in which every pipeline wait
 * is a single probe, so that a call almost surely times out: it exists to
 * test that path.  Process-wide; returns the previous setting (0 or 1).
 * Host only: touches no device.
 */
int sparse_attn_set_single_probe_waits(int on);

/*
 * The last CUDA runtime error that made an entry point return SA_ECUDA on
 * the calling host thread (0 = none since the thread started), and its
 * message when `message` is not NULL.  Host only.
 */
int sparse_attn_last_cuda_error(const char** message);

/* Static, human-readable name of a status code. */
const char* sparse_attn_status_string(sa_status s);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H_ */
