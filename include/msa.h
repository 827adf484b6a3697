/*
 * msa.h -- C ABI of the GB300 (sm_103a) MiniMax Sparse Attention (MSA)
 * training hot path on one GQA layer.
 *
 * The method (itinai.ru "How to solve the memory problem with MiniMax Sparse
 * Attention", sections "Two-stage process", "How the indexer works" and
 * "Training sparse attention"; dothoosh.com "how Flash-MSA cuts
 * million-token training cost", sections "Block-sparsity mechanism",
 * "Kernel design and execution" and "Fixing the KL-divergence bottleneck"):
 *
 *   1. msa_index_topk  -- index branch: every causally visible token is scored
 *      with the group's index query against the shared index key, scores are
 *      max-pooled over Bk-token KV blocks, and each (group, query) keeps k
 *      blocks: its own block plus the best k-1 earlier ones.
 *   2. msa_sparse_fwd  -- main branch: exact causal softmax attention over the
 *      selected blocks only; writes O and the log-sum-exp kept for the backward.
 *   3. msa_bwd         -- fused backward: dQ, dK, dV of the main branch and the
 *      KL-alignment gradient of the index branch, whose score gradient is
 *      p_px - p_main (index softmax over the selected tokens minus the
 *      head-averaged, detached main softmax), giving dq_idx and dk_idx.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller; the library
 *   never allocates device memory. Scratch comes from the caller's workspace,
 *   sized by msa_workspace_size() (256-byte aligned base required).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream). Host-side argument checks run before anything is enqueued; on a
 *   non-OK status nothing was launched and msa_last_error() describes why.
 * - bf16 tensors are passed as `void*` holding IEEE bfloat16 values; the
 *   backward's gradients are fp32 (`float*`), accumulated and written in fp32.
 * - Layouts (row-major, innermost last):
 *     Q, O, dO            [B, T, Hq, d]      bf16      dQ      fp32
 *     K, V                [B, T, G, d]       bf16      dK, dV  fp32 (one KV head per group)
 *     q_idx               [B, T, G, d_idx]   bf16      dq_idx  fp32
 *     k_idx               [B, T, d_idx]      bf16      dk_idx  fp32 (shared by all groups)
 *     block_idx           [B, G, T, k]       int32  (ascending ids, -1 padded)
 *     LSE                 [B, T, Hq]         fp32   (natural log, scaled scores)
 *     KL                  [B, G, T]          fp32   (one KL term per query)
 *   Head h belongs to group h / (Hq / G).
 * - Supported shapes (MSA_ERR_UNSUPPORTED otherwise): d = 128, d_idx = 64,
 *   Bk = 128, Hq / G in {1, 2, 4, 8} with Hq % G == 0, T % 128 == 0,
 *   1 <= T <= 2^20, 1 <= k <= 128, B >= 1, scale and scale_idx > 0 after
 *   defaulting; the index top-k (msa_index_topk, msa_index_topk_fp8,
 *   msa_index_topk_noalloc, and the MSA_WS_TOPK / MSA_WS_TOPK_FP8 workspace
 *   sizes) keeps at most k = 64 blocks per row. Kernels need an sm_100-family
 *   GPU (built for sm_103a).
 * - Device-side checks (bounded waits, block ids out of range) write an error
 *   word in the workspace; msa_check_device_status() reads it.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define MSA_API __attribute__((visibility("default")))
#else
#define MSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *msa_stream_t;

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad enum       */
  MSA_ERR_UNSUPPORTED = 2, /* shape outside the supported set above, or no GPU */
  MSA_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small      */
  MSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (see msa_last_error) */
  MSA_ERR_DEVICE = 5       /* a kernel reported a timeout or a bad block id   */
} msa_status;

typedef struct msa_shape {
  int32_t B;       /* batch                                                 */
  int32_t T;       /* sequence length                                       */
  int32_t Hq;      /* query heads                                           */
  int32_t G;       /* GQA groups = KV heads = index queries per position    */
  int32_t d;       /* head dim of Q/K/V                                     */
  int32_t d_idx;   /* index dim of q_idx/k_idx                              */
  int32_t Bk;      /* tokens per KV block                                   */
  int32_t k;       /* blocks kept per (group, query), own block included    */
  float scale;     /* main softmax scale; <= 0 selects 1/sqrt(d)            */
  float scale_idx; /* index score scale; <= 0 selects 1/sqrt(d_idx)         */
} msa_shape;

/* Which entry point a workspace is sized for. */
enum { MSA_WS_TOPK = 0, MSA_WS_FWD = 1, MSA_WS_BWD = 2, MSA_WS_TOPK_FP8 = 3, MSA_WS_DENSE = 4 };

/* Bytes of device workspace the entry point `which` needs for `shape`
 * (0 if the shape is invalid or unsupported). A workspace sized for
 * MSA_WS_BWD also serves MSA_WS_TOPK and MSA_WS_FWD; MSA_WS_TOPK_FP8 is
 * sized on its own (its E4M3 copies start right after the header). */
MSA_API size_t msa_workspace_size(const msa_shape *shape, int which);

/*
 * Index branch (itinai.ru "How the indexer works"; dothoosh.com Flash-MSA,
 * "Block-sparsity mechanism" and "Kernel design and execution": the proxy
 * pass accumulates no output, only scores and the running top-k).
 *
 * For every (b, g, t) with own block c_t = t / Bk:
 *   s[j]  = <q_idx[b,t,g,:], k_idx[b,j,:]>            for j <= t (fp32 sums of
 *           exact bf16 products; the positive scale_idx does not change order)
 *   pool[c] = max_{j in block c} s[j]                  for c < c_t
 *   block_idx[b,g,t,:] = {c_t} U top-(k-1) of pool under (score descending,
 *           block id ascending), written in ascending order, then -1 padding.
 * No T x T (or T x n_blocks) tensor is materialised.
 *
 * q_idx: [B,T,G,d_idx] bf16, k_idx: [B,T,d_idx] bf16 (both 16-byte aligned).
 * block_idx: [B,G,T,k] int32, fully written.
 */
MSA_API msa_status msa_index_topk(const msa_shape *shape, const void *q_idx, const void *k_idx, int32_t *block_idx,
                          void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* msa_index_topk with a low-precision indexer (dothoosh.com "how Flash-MSA
 * cuts million-token training cost", "Current limits and future scaling":
 * training the indexer in low precision, as at inference). The index scores
 * are computed from E4M3 copies of q_idx and k_idx made inside the call: one
 * scale per q_idx row (b, t, g) and one per 128-key block of k_idx (b, c);
 * each value is multiplied by 448 / amax in fp32 and rounded to the nearest
 * E4M3 value (ties to even, saturating at +-448); the scale is amax / 448
 * (1 when amax = 0). Pooling and selection are those of msa_index_topk on
 * the scores (q8 * sq) . (k8 * sk) * scale_idx, so block_idx can differ from
 * msa_index_topk's where quantization reorders blocks. `workspace` is sized
 * with MSA_WS_TOPK_FP8 (it holds the E4M3 copies: B*T*(G+1)*d_idx bytes plus
 * one float per key block); same arguments and errors as msa_index_topk. */
MSA_API msa_status msa_index_topk_fp8(const msa_shape *shape, const void *q_idx, const void *k_idx,
                                      int32_t *block_idx, void *workspace, size_t workspace_bytes,
                                      msa_stream_t stream);

/*
 * Main branch forward (itinai.ru "Two-stage process": exact softmax over the
 * selected tokens only; dothoosh.com Flash-MSA, "Kernel design and
 * execution": keep the LSE for the backward; dothoosh.com "how FlashAttention
 * cuts GPU memory traffic", "Online-softmax trick": the (m, l, a) merge).
 *
 * For head h in group g and query t, over S(g,t) = { j <= t : j / Bk listed in
 * block_idx[b,g,t,:] }:
 *   s_j = scale * <Q[b,t,h,:], K[b,j,g,:]>,  LSE = ln sum_j exp(s_j),
 *   O[b,t,h,:] = sum_j exp(s_j - LSE) V[b,j,g,:].
 * block_idx may come from msa_index_topk or from anywhere else, but every row
 * must hold distinct ids in [0, t / Bk] in ascending order followed by -1s
 * and must include t / Bk (violations set the device error word and the
 * offending row's outputs are unspecified).
 *
 * O: [B,T,Hq,d] bf16, LSE: [B,T,Hq] fp32, both fully written.
 */
MSA_API msa_status msa_sparse_fwd(const msa_shape *shape, const void *Q, const void *K, const void *V,
                          const int32_t *block_idx, void *O, float *LSE, void *workspace,
                          size_t workspace_bytes, msa_stream_t stream);

/*
 * Fused backward (dothoosh.com Flash-MSA, "Kernel design and execution": one
 * backward over proxy and main branch, scheduled through the inverted
 * block -> query map; "Fixing the KL-divergence bottleneck": d KL / d s_px =
 * p_px - p_main; itinai.ru "Training sparse attention": KL alignment to the
 * head-averaged main softmax, gradient detached from the backbone;
 * dothoosh.com FlashAttention page, "Training and the backward pass").
 *
 * Main branch, with P = exp(s - LSE) rebuilt from the saved LSE:
 *   D = rowsum(dO * O), dP = dO V^T, dS = P (dP - D),
 *   dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
 * Index branch, per (b, g, t) over S(g,t):
 *   p_main_j = mean over the group's heads of P_h,j (detached),
 *   p_px_j   = softmax_j(scale_idx <q_idx[b,t,g,:], k_idx[b,j,:]>),
 *   KL[b,g,t] = sum_j p_main_j (ln p_main_j - ln p_px_j),
 *   gs_j = kl_weight (p_px_j - p_main_j),
 *   dq_idx[b,t,g,:] = scale_idx sum_j gs_j k_idx[b,j,:],
 *   dk_idx[b,j,:]  += scale_idx sum_{g,t} gs_j q_idx[b,t,g,:].
 * The loss is kl_weight * sum over rows of KL (pass 1/(B*G*T) for a mean).
 * No KL gradient reaches Q, K, V and no dO gradient reaches q_idx, k_idx.
 *
 * Inputs as in msa_sparse_fwd; O and LSE are the forward's outputs for the
 * same block_idx. Outputs dQ, dK, dV, dq_idx, dk_idx and KL (all fp32) are
 * fully written: every key block is selected at least by its own queries, so
 * every dK/dV/dk_idx row receives its sum (rows of a block whose queries all
 * had invalid block_idx rows are unspecified, as is everything else when the
 * device error word is set). Every sum runs in a fixed order (per-slot and
 * per-group partials, merged in order; no floating-point atomics), so the
 * outputs, like those of msa_index_topk and msa_sparse_fwd, are the same bits
 * in every run on the same inputs.
 */
MSA_API msa_status msa_bwd(const msa_shape *shape, const void *Q, const void *K, const void *V, const void *O,
                   const void *dO, const float *LSE, const void *q_idx, const void *k_idx,
                   const int32_t *block_idx, float kl_weight, float *dQ, float *dK, float *dV, float *dq_idx,
                   float *dk_idx, float *KL, void *workspace, size_t workspace_bytes, msa_stream_t stream);

/*
 * Index top-k for callers that cannot allocate device memory. The method's
 * description has no counterpart to this call; it computes exactly what
 * msa_index_topk does.
 *
 * Some callers cannot call cudaMalloc: a plugin inside a host application
 * that owns every byte of device memory and hands the plugin no allocator,
 * or code on a latency-critical path where cudaMalloc's implicit device-wide
 * synchronisation is not acceptable. This variant needs no workspace: its
 * scratch (the kernel's error word and work counter, 256 bytes) lives in a
 * static device array of MSA_NOALLOC_SCRATCH_BYTES bytes inside the library,
 * which every GPU that loads the library holds until the process exits.
 *
 * - Each GPU has its own copy of the array. The first call on a device looks
 *   up the address of that device's copy (once per device, with the device
 *   current) and the library keeps it; make that first call before any stream
 *   capture. The address belongs to the device's primary context: after
 *   cudaDeviceReset() on that device, reload the library before calling
 *   this function again.
 * - Every call clears the scratch it relies on (asynchronously, on `stream`)
 *   and then reuses it: calls that overlap on the same GPU (for example on
 *   two streams of one device) race on it. Serialise them; calls on
 *   different GPUs use different copies and do not race.
 * - A shape whose scratch would exceed MSA_NOALLOC_SCRATCH_BYTES is rejected
 *   with MSA_ERR_UNSUPPORTED.
 * - check != 0 synchronises `stream` and returns MSA_ERR_DEVICE if the kernel
 *   reported a timeout; check == 0 returns without waiting (device-side
 *   errors then go unreported).
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define MSA_NOALLOC_SCRATCH_BYTES 4096
MSA_API msa_status msa_index_topk_noalloc(const msa_shape *shape, const void *q_idx, const void *k_idx,
                                          int32_t *block_idx, int32_t check, msa_stream_t stream);

/* IndexShare: one selection shared by several layers (dothoosh.com "how
 * Flash-MSA cuts million-token training cost", "Current limits and future
 * scaling": sharing the proxy (index) heads across layers, so later layers
 * reuse an earlier layer's block indices). msa_block_map
 * builds the inverted block -> query map of `block_idx` once, into a
 * MSA_WS_BWD-sized `workspace`, with the work items of both the forward and
 * the backward; msa_sparse_fwd_mapped and msa_bwd_mapped then run on that map
 * instead of building their own (same arguments, results and errors as
 * msa_sparse_fwd and msa_bwd). The map stays valid for as long as `block_idx`
 * and the workspace's map region are unchanged: msa_index_topk,
 * msa_sparse_fwd and msa_bwd on the same workspace overwrite it, the mapped
 * calls do not. The caller guarantees that the `block_idx` passed to the
 * mapped calls is the one the map was built from; rows that fail validation
 * are reported by msa_block_map (device error word). */
MSA_API msa_status msa_block_map(const msa_shape *shape, const int32_t *block_idx, void *workspace,
                                 size_t workspace_bytes, msa_stream_t stream);
MSA_API msa_status msa_sparse_fwd_mapped(const msa_shape *shape, const void *Q, const void *K, const void *V,
                                         const int32_t *block_idx, void *O, float *LSE, void *workspace,
                                         size_t workspace_bytes, msa_stream_t stream);
MSA_API msa_status msa_bwd_mapped(const msa_shape *shape, const void *Q, const void *K, const void *V,
                                  const void *O, const void *dO, const float *LSE, const void *q_idx,
                                  const void *k_idx, const int32_t *block_idx, float kl_weight, float *dQ, float *dK,
                                  float *dV, float *dq_idx, float *dk_idx, float *KL, void *workspace,
                                  size_t workspace_bytes, msa_stream_t stream);

/* Indexer warmup (itinai.ru "How to solve the memory problem with MiniMax
 * Sparse Attention", "Training sparse attention": the first iterations run
 * full attention so that the indexer learns before it routes). Writes into
 * `block_idx` [B,G,T,k] int32 (device, caller-owned) the selection of full
 * causal attention: row (b, g, t) holds the blocks 0 .. t / Bk ascending,
 * then -1. Given it, msa_sparse_fwd computes dense causal attention and
 * msa_bwd the KL of the index branch against the dense teacher (the head mean
 * of the full attention weights) over every visible token, with its gradients
 * to q_idx and k_idx. No index scores are computed and no workspace is used.
 * MSA_ERR_UNSUPPORTED unless k >= T / Bk (so at most T = 128 * Bk). */
MSA_API msa_status msa_warmup_block_idx(const msa_shape *shape, int32_t *block_idx, msa_stream_t stream);

/*
 * Full attention at any T: the forward and backward that msa_sparse_fwd and
 * msa_bwd compute for the selection msa_warmup_block_idx writes (every
 * visible block), without a block list and without per-(query, block)
 * scratch, so that the indexer warmup (itinai.ru "How to solve the memory
 * problem with MiniMax Sparse Attention", "Training sparse attention": the
 * first iterations run full attention) reaches the sequence lengths of the
 * sparse path. For head h in group g and query t, over every j <= t:
 *   O, LSE as msa_sparse_fwd with S(g,t) = { 0 .. t };
 *   dQ, dK, dV, dq_idx, dk_idx, KL as msa_bwd over the same set (the KL of
 *   the index softmax over every visible token against the head mean of the
 *   full attention weights).
 * Same tensors, layouts and scales as msa_sparse_fwd / msa_bwd; no block_idx.
 * shape->k is not used (any value is accepted). Supported: Hq / G in {4, 8}
 * (MSA_ERR_UNSUPPORTED otherwise: 1 or 2 heads per group take
 * msa_warmup_block_idx with the sparse calls, T <= 128 * Bk), and the other
 * limits of the common conventions. Workspace: MSA_WS_DENSE (msa_dense_fwd
 * needs only its 256-byte header).
 *
 * msa_dense_fwd is query-outer (the running maximum, sum and O of each row
 * stay on chip) and writes O and LSE once; deterministic.
 * msa_dense_bwd overwrites its six outputs with sums accumulated by fp32
 * atomic and TMA reduce-add operations from concurrent CTAs: the summation
 * order, hence the last bits, varies from run to run. O and LSE must be
 * msa_dense_fwd's outputs (or the sparse forward's under the full selection).
 */
MSA_API msa_status msa_dense_fwd(const msa_shape *shape, const void *Q, const void *K, const void *V, void *O,
                                 float *LSE, void *workspace, size_t workspace_bytes, msa_stream_t stream);
MSA_API msa_status msa_dense_bwd(const msa_shape *shape, const void *Q, const void *K, const void *V, const void *O,
                                 const void *dO, const float *LSE, const void *q_idx, const void *k_idx,
                                 float kl_weight, float *dQ, float *dK, float *dV, float *dq_idx, float *dk_idx,
                                 float *KL, void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* Message describing the last non-OK status returned on this thread. */
MSA_API const char *msa_last_error(void);

/* Synchronises `stream`, then reads and clears the device error word of
 * `workspace` (the one the last call on it used). MSA_ERR_DEVICE if a kernel
 * gave up on a wait or met a block id out of range; msa_last_error() says
 * which kernel and where. */
MSA_API msa_status msa_check_device_status(const void *workspace, msa_stream_t stream);

/* Failure-detection self-test: launches one block whose wait on an mbarrier
 * that nothing ever arrives at is bounded by `limit_us` microseconds
 * (1..1000000). The wait runs out, the kernel records a timeout in the error
 * word of `workspace` (>= 256 bytes, device memory) and returns; a following
 * msa_check_device_status() reports MSA_ERR_DEVICE. Exercises the same bounded
 * wait every kernel uses, without faulting or hanging the GPU. */
MSA_API msa_status msa_selftest_wait_timeout(void *workspace, int32_t limit_us, msa_stream_t stream);

/* Kernel timing for benchmarks. The main kernel of one stage: */
enum {
  MSA_TIME_INDEX_TOPK = 0, /* index_topk_kernel (msa_index_topk, msa_index_topk_fp8, the no-workspace call) */
  MSA_TIME_SPARSE_FWD = 1, /* sparse_fwd_kernel (msa_sparse_fwd, msa_sparse_fwd_mapped), not the map or merge */
  MSA_TIME_BWD = 2,        /* the fused backward kernel (msa_bwd, msa_bwd_mapped), not the pre-passes or merges */
  MSA_TIME_DENSE_FWD = 3,  /* dense_fwd_kernel (msa_dense_fwd) */
  MSA_TIME_DENSE_BWD = 4   /* the backward kernel of msa_dense_bwd, not D or the index LSE */
};

/* While set, every launch of kernel `which` is bracketed by
 * cudaEventRecord(start_event) and cudaEventRecord(stop_event) on the call's
 * stream, so that the caller can read the kernel's own duration with
 * cudaEventElapsedTime. The events are the caller's cudaEvent_t handles (created
 * with timing enabled, on this device) and stay the caller's; each launch
 * re-records them. Both NULL stops the recording. The setting is process-wide
 * and not synchronised between threads. MSA_ERR_INVALID_ARG for an unknown
 * `which` or for exactly one NULL event. */
MSA_API msa_status msa_set_timing_events(int32_t which, void *start_event, void *stop_event);

/* Number of kernels this library has launched in the calling process since it
 * was loaded (monotonic; for accounting in benchmarks and tests). */
MSA_API int64_t msa_kernel_launches(void);

/* ABI version: (major << 16) | minor. */
MSA_API int32_t msa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
