// Host-side internals shared by the MSA entry points and kernel launchers:
// validated problem description, workspace layout, tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/msa.h"

namespace msa {

// Validated, defaulted shape.
struct Prob {
  int B, T, Hq, G, d, E, Bk, k;  // E = d_idx
  int hg;                        // heads per group
  int n;                         // KV blocks = T / Bk
  float scale, scale_idx;
  long long BT() const { return (long long)B * T; }
};

// Workspace regions (byte offsets from the workspace base, 256-aligned).
struct WsLayout {
  size_t err = 0;           // int32 error word
  size_t counters = 64;     // int32 work counters [16]
  size_t list_count = 0;    // int32 [B*G*n]   selections per KV block
  size_t list_off = 0;      // int32 [B*G*n+1] exclusive prefix of list_count
  size_t chunk_off = 0;     // int32 [B*G, n(n+1)/2] per (list, query block): position of its first entry
  size_t list_poff = 0;     // int32 [B*G*n+1] prefix of list lengths padded to whole tiles
  size_t rev = 0;           // int32 [B*G*T*k] padded entry index of (b, g, t, slot)
  size_t entries = 0;       // int32 [B*G*T*k] (t << 8 | slot), grouped by list
  size_t items = 0;         // int4  [max_items] work items (list, tile range)
  size_t items2 = 0;        // int4  [max_items] the backward's items of a shared map (msa_block_map)
  size_t n_items = 0;       // int32 [4]       number of work items per kernel
  size_t o_part = 0;        // bf16  [padded entries, hg, d] forward partial outputs (normalised), tile order
  size_t lse_part = 0;      // fp32  [padded entries, hg]    forward partial log-sum-exp
  size_t drow = 0;          // fp32  [B,T,Hq]       rowsum(dO * O)
  size_t px_part = 0;       // fp32  [B,T,G,k]      index-branch partial LSE per slot
  size_t lse_px = 0;        // fp32  [B,T,G]        index-branch LSE over S(g,t)
  size_t dq_part = 0;       // bf16  [padded entries, hg, d] dQ partials, tile order
  size_t dqi_part = 0;      // bf16  [padded entries, E]     dq_idx partials, tile order
  size_t kl_part = 0;       // fp32  [B,T,G,k,4]    KL partials per slot and key quarter
  size_t dki_part = 0;      // fp32  [B,G,T,E]      dk_idx per group
  size_t q8 = 0;            // e4m3  [B,T,G,E]      FP8 index queries (MSA_WS_TOPK_FP8)
  size_t k8 = 0;            // e4m3  [B,T,E]        FP8 index keys
  size_t k_scale = 0;       // fp32  [B,n]          dequantization scale per key block
  size_t total = 256;
  int max_items = 0;
  long long max_padded = 0;  // capacity in padded entries (queries x slots, tile-padded per list)
};

WsLayout ws_layout(const Prob& p, int which);

// Maximum work-item count of the sparse kernels for a problem.
int max_work_items(const Prob& p, int tiles_per_item, int rows_per_tile);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
bool encode_tmap(CUtensorMap* map, void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                 const uint32_t* box, CUtensorMapSwizzle swz,
                 CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

int num_sms();

// Current device id, clamped to [0, kMaxDevices): index of per-device state
// such as kernel attributes, which belong to each device's context.
constexpr int kMaxDevices = 64;
int device_slot();

// Count of kernels launched by the library (msa_kernel_launches).
void count_launches(int n);

// Caller-owned events recorded around a main kernel (msa_set_timing_events):
// which = one of the MSA_TIME_* kernels.
void timing_begin(int which, cudaStream_t st);
void timing_end(int which, cudaStream_t st);

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_index_topk(const Prob& p, const void* q_idx, const void* k_idx, int32_t* block_idx, void* ws,
                              const WsLayout& L, cudaStream_t st);
cudaError_t launch_index_topk_fp8(const Prob& p, const void* q_idx, const void* k_idx, int32_t* block_idx, void* ws,
                                  const WsLayout& L, cudaStream_t st);

// Full causal selection (every visible block) for the indexer warmup.
cudaError_t launch_warmup_block_idx(const Prob& p, int32_t* block_idx, cudaStream_t st);

// Inverted block -> query lists and work items (rows_per_tile * tiles_per_item
// entries per item).
cudaError_t build_block_map(const Prob& p, const int32_t* block_idx, uint8_t* ws, const WsLayout& L,
                            int rows_per_tile, int tiles_per_item, cudaStream_t st);

// The same map with lists padded to pad_rows entries and two item lists: the
// forward's in `items` (n_items[0]) and, when two_lists, the backward's in
// `items2` (n_items[1]), so both kernels can run on it without rebuilding it.
cudaError_t build_block_map2(const Prob& p, const int32_t* block_idx, uint8_t* ws, const WsLayout& L, int pad_rows,
                             long long per_item_a, long long per_item_b, bool two_lists, cudaStream_t st);

// Queries per forward tile / per backward tile, and the forward's tiles per item.
inline int fwd_tile_queries(const Prob& p) { return 128 / p.hg; }
inline int bwd_tile_queries(const Prob& p) { return (p.hg >= 4 ? 128 : 64) / p.hg; }
constexpr int kFwdTilesPerItem = 32;

// mapped: use the map (and the forward's items) that build_block_map2 left
// in the workspace instead of building one.
cudaError_t launch_sparse_fwd(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* block_idx,
                              void* O, float* LSE, uint8_t* ws, const WsLayout& L, cudaStream_t st,
                              bool mapped = false);

// mapped: use the map and the backward's items (items2) left by build_block_map2.
cudaError_t launch_bwd(const Prob& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                       const float* LSE, const void* q_idx, const void* k_idx, const int32_t* block_idx,
                       float kl_weight, void* dQ, void* dK, void* dV, void* dq_idx, void* dk_idx, float* KL,
                       uint8_t* ws, const WsLayout& L, cudaStream_t st, bool mapped = false);

// Full attention (indexer warmup at any T; heads per group 4 or 8).
// The backward's work items: every (KV block c, query t >= 128 c) pair, cut
// into segments of `seg` queries (dense_schedule; items <= INT_MAX checked).
struct DenseSchedule {
  int seg;     // queries per segment (multiple of 128)
  int per_b;   // work items per batch entry
  int items;   // all work items
};
bool dense_schedule(const Prob& p, DenseSchedule* ds);
cudaError_t launch_dense_fwd(const Prob& p, const void* Q, const void* K, const void* V, void* O, float* LSE,
                             uint8_t* ws, const WsLayout& L, cudaStream_t st);
cudaError_t launch_dense_px(const Prob& p, const void* q_idx, const void* k_idx, float* lse_px, uint8_t* ws,
                            const WsLayout& L, cudaStream_t st);
cudaError_t launch_bwd_dense(const Prob& p, const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, const void* q_idx, const void* k_idx, float kl_weight,
                             float* dQ, float* dK, float* dV, float* dq_idx, float* dk_idx, float* KL, uint8_t* ws,
                             const WsLayout& L, const DenseSchedule& ds, cudaStream_t st);

cudaError_t launch_selftest_wait_timeout(int* err, long long limit_ns, cudaStream_t st);

}  // namespace msa
