// C ABI of the MSA hot path: argument validation, workspace carving and
// kernel launch order. See include/msa.h for the contract of each call.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {

static thread_local char g_err[512];

static msa_status fail(msa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

static std::atomic<long long> g_launches{0};

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int device_slot() {
  int dev = 0;
  cudaGetDevice(&dev);
  return (dev < 0 || dev >= kMaxDevices) ? 0 : dev;
}

int num_sms() {
  static int cached[kMaxDevices] = {0};
  const int dev = device_slot();
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

bool encode_tmap(CUtensorMap* map, void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                 const uint32_t* box, CUtensorMapSwizzle swz, CUtensorMapDataType dtype) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = reinterpret_cast<EncodeFn>(p);
  }
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return fn(map, dtype, rank, base, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int max_work_items(const Prob& p, int tiles_per_item, int rows_per_tile) {
  // each list of length L gives ceil(ceil(L / rows) / tiles) items; the sum is
  // bounded by total_tiles / tiles + lists, total_tiles <= entries / rows + lists
  const long long lists = (long long)p.B * p.G * p.n;
  const long long entries = (long long)p.B * p.G * p.T * p.k;
  const long long tiles = entries / rows_per_tile + lists;
  return (int)(tiles / tiles_per_item + lists + 1);
}

bool dense_schedule(const Prob& p, DenseSchedule* ds) {
  // segments of 4096 queries: the dQ rows the CTAs add into at the same time (a segment of every group:
  // 4096 x Hq x d fp32, 64 MB at Hq = 32) stay in L2
  const long long seg = std::min<long long>(4096, p.T);
  const long long nseg = (p.T + seg - 1) / seg;
  long long per_b = 0;
  for (long long s = 0; s < nseg; ++s) per_b += (long long)p.G * std::min<long long>((s + 1) * seg / 128, p.n);
  const long long items = per_b * p.B;
  if (items > 0x7fffffffLL) return false;
  ds->seg = (int)seg;
  ds->per_b = (int)per_b;
  ds->items = (int)items;
  return true;
}

WsLayout ws_layout(const Prob& p, int which) {
  WsLayout L;
  size_t off = 256;  // header: error word + counters
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t lists = (size_t)p.B * p.G * p.n;
  const size_t rows = (size_t)p.B * p.T;
  if (which == MSA_WS_DENSE) {
    L.drow = take(rows * p.Hq * 4);
    L.lse_px = take(rows * p.G * 4);
    L.total = off;
    return L;
  }
  if (which == MSA_WS_TOPK_FP8) {
    L.q8 = take(rows * p.G * p.E);
    L.k8 = take(rows * p.E);
    L.k_scale = take((size_t)p.B * p.n * 4);
    L.total = off;
    return L;
  }
  if (which == MSA_WS_FWD || which == MSA_WS_BWD) {
    L.list_count = take(lists * 4);
    L.list_off = take((lists + 1) * 4);
    L.chunk_off = take((size_t)p.B * p.G * ((size_t)p.n * (p.n + 1) / 2) * 4);
    L.list_poff = take((lists + 1) * 4);
    L.entries = take(rows * p.G * p.k * 4);
    L.rev = take(rows * p.G * p.k * 4);
    // lists are padded to whole tiles of at most 128 queries
    L.max_padded = (long long)(rows * p.G * p.k) + (long long)lists * 128;
    L.max_items = max_work_items(p, 1, 16);
    L.items = take((size_t)L.max_items * 16);
    L.n_items = take(16);
    if (which == MSA_WS_BWD) L.items2 = take((size_t)L.max_items * 16);
  }
  if (which == MSA_WS_FWD) {
    L.o_part = take((size_t)L.max_padded * p.hg * p.d * 2);
    L.lse_part = take((size_t)L.max_padded * p.hg * 4);
  }
  if (which == MSA_WS_BWD) {
    // the forward's partial buffers alias the backward's larger ones
    L.drow = take(rows * p.Hq * 4);
    L.px_part = take(rows * p.G * p.k * 4);
    L.lse_px = take(rows * p.G * 4);
    L.dq_part = take((size_t)L.max_padded * p.hg * p.d * 2);
    L.dqi_part = take((size_t)L.max_padded * p.E * 2);
    L.kl_part = take(rows * p.G * p.k * 16);
    L.dki_part = take((size_t)p.B * p.G * p.T * p.E * 4);
    L.o_part = L.dq_part;
    L.lse_part = take((size_t)L.max_padded * p.hg * 4);
  }
  L.total = off;
  return L;
}

static msa_status validate(const msa_shape* s, Prob* p) {
  if (!s) return fail(MSA_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->T < 1 || s->Hq < 1 || s->G < 1 || s->d < 1 || s->d_idx < 1 || s->Bk < 1 || s->k < 1)
    return fail(MSA_ERR_INVALID_ARG, "shape fields must be positive (B=%d T=%d Hq=%d G=%d d=%d d_idx=%d Bk=%d k=%d)",
                s->B, s->T, s->Hq, s->G, s->d, s->d_idx, s->Bk, s->k);
  if (s->Hq % s->G) return fail(MSA_ERR_INVALID_ARG, "Hq=%d is not a multiple of G=%d", s->Hq, s->G);
  const int hg = s->Hq / s->G;
  if (s->d != 128) return fail(MSA_ERR_UNSUPPORTED, "d=%d: only head dim 128 is supported", s->d);
  if (s->d_idx != 64) return fail(MSA_ERR_UNSUPPORTED, "d_idx=%d: only index dim 64 is supported", s->d_idx);
  if (s->Bk != 128) return fail(MSA_ERR_UNSUPPORTED, "Bk=%d: only 128-token blocks are supported", s->Bk);
  if (!(hg == 1 || hg == 2 || hg == 4 || hg == 8))
    return fail(MSA_ERR_UNSUPPORTED, "Hq/G=%d: heads per group must be 1, 2, 4 or 8", hg);
  if (s->T % 128) return fail(MSA_ERR_UNSUPPORTED, "T=%d is not a multiple of 128", s->T);
  if (s->T > (1 << 20)) return fail(MSA_ERR_UNSUPPORTED, "T=%d exceeds 2^20", s->T);
  if (s->k > 128) return fail(MSA_ERR_UNSUPPORTED, "k=%d exceeds 128", s->k);
  if ((long long)s->B * s->T > (1LL << 30)) return fail(MSA_ERR_UNSUPPORTED, "B*T too large");
  const float sc = s->scale > 0 ? s->scale : 1.0f / sqrtf((float)s->d);
  const float sci = s->scale_idx > 0 ? s->scale_idx : 1.0f / sqrtf((float)s->d_idx);
  if (!(sc > 0) || !isfinite(sc) || !(sci > 0) || !isfinite(sci))
    return fail(MSA_ERR_INVALID_ARG, "scales must be finite");
  p->B = s->B;
  p->T = s->T;
  p->Hq = s->Hq;
  p->G = s->G;
  p->d = s->d;
  p->E = s->d_idx;
  p->Bk = s->Bk;
  p->k = s->k;
  p->hg = hg;
  p->n = s->T / s->Bk;
  p->scale = sc;
  p->scale_idx = sci;
  return MSA_OK;
}

// The full-attention calls take no block list (shape->k is not used) and run
// the 128-row-tile kernels: 4 or 8 heads per group.
static msa_status validate_dense(const msa_shape* s, Prob* p) {
  if (!s) return fail(MSA_ERR_INVALID_ARG, "shape is NULL");
  msa_shape c = *s;
  c.k = 1;
  msa_status st;
  if ((st = validate(&c, p)) != MSA_OK) return st;
  if (p->hg != 4 && p->hg != 8)
    return fail(MSA_ERR_UNSUPPORTED,
                "Hq/G=%d: full attention needs 4 or 8 heads per group (with 1 or 2, use msa_warmup_block_idx "
                "with the sparse calls up to T = 128 * Bk)",
                p->hg);
  return MSA_OK;
}

// The index top-k keeps its list in registers: at most 64 blocks per row.
static msa_status check_topk_k(const Prob& p) {
  if (p.k > 64) return fail(MSA_ERR_UNSUPPORTED, "index top-k keeps at most 64 blocks (k=%d)", p.k);
  return MSA_OK;
}

static msa_status check_ptr(const void* ptr, const char* name, size_t align) {
  if (!ptr) return fail(MSA_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(ptr) % align)
    return fail(MSA_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
  return MSA_OK;
}

static msa_status check_ws(const Prob& p, int which, void* ws, size_t bytes, WsLayout* L) {
  *L = ws_layout(p, which);
  if (!ws) return fail(MSA_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(MSA_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (bytes < L->total)
    return fail(MSA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", bytes, L->total);
  return MSA_OK;
}

static msa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MSA_ERR_UNSUPPORTED, "no CUDA device");
  int major = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (major != 10) return fail(MSA_ERR_UNSUPPORTED, "device %d has compute capability %d.x, sm_10x needed", dev, major);
  return MSA_OK;
}

static msa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MSA_OK;
  cudaGetLastError();
  return fail(MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

cudaEvent_t g_timing[5][2] = {};  // caller's events per timed kernel (msa_set_timing_events)

void timing_begin(int which, cudaStream_t st) {
  if (g_timing[which][0]) cudaEventRecord(g_timing[which][0], st);
}
void timing_end(int which, cudaStream_t st) {
  if (g_timing[which][1]) cudaEventRecord(g_timing[which][1], st);
}

}  // namespace msa

using namespace msa;

extern "C" {

int32_t msa_version(void) { return (1 << 16) | 4; }

int64_t msa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* msa_last_error(void) { return g_err; }

size_t msa_workspace_size(const msa_shape* shape, int which) {
  Prob p{};
  if (which < MSA_WS_TOPK || which > MSA_WS_DENSE) return 0;
  if (which == MSA_WS_DENSE) {
    if (validate_dense(shape, &p) != MSA_OK) return 0;
    return ws_layout(p, which).total;
  }
  if (validate(shape, &p) != MSA_OK) return 0;
  if ((which == MSA_WS_TOPK || which == MSA_WS_TOPK_FP8) && p.k > 64) return 0;
  return ws_layout(p, which).total;
}

msa_status msa_index_topk(const msa_shape* shape, const void* q_idx, const void* k_idx, int32_t* block_idx,
                          void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  if ((s = check_topk_k(p)) != MSA_OK) return s;
  if ((s = check_ptr(q_idx, "q_idx", 16)) != MSA_OK) return s;
  if ((s = check_ptr(k_idx, "k_idx", 16)) != MSA_OK) return s;
  if ((s = check_ptr(block_idx, "block_idx", 16)) != MSA_OK) return s;
  if ((s = check_ws(p, MSA_WS_TOPK, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_index_topk(p, q_idx, k_idx, block_idx, workspace, L, st), "index top-k launch");
}

msa_status msa_index_topk_fp8(const msa_shape* shape, const void* q_idx, const void* k_idx, int32_t* block_idx,
                              void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  if ((s = check_topk_k(p)) != MSA_OK) return s;
  if ((s = check_ptr(q_idx, "q_idx", 16)) != MSA_OK) return s;
  if ((s = check_ptr(k_idx, "k_idx", 16)) != MSA_OK) return s;
  if ((s = check_ptr(block_idx, "block_idx", 16)) != MSA_OK) return s;
  if ((s = check_ws(p, MSA_WS_TOPK_FP8, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_index_topk_fp8(p, q_idx, k_idx, block_idx, workspace, L, st), "FP8 index top-k launch");
}

static msa_status sparse_fwd_impl(const msa_shape* shape, const void* Q, const void* K, const void* V,
                                  const int32_t* block_idx, void* O, float* LSE, void* workspace,
                                  size_t workspace_bytes, msa_stream_t stream, bool mapped) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  if ((s = check_ptr(Q, "Q", 16)) != MSA_OK) return s;
  if ((s = check_ptr(K, "K", 16)) != MSA_OK) return s;
  if ((s = check_ptr(V, "V", 16)) != MSA_OK) return s;
  if ((s = check_ptr(block_idx, "block_idx", 4)) != MSA_OK) return s;
  if ((s = check_ptr(O, "O", 16)) != MSA_OK) return s;
  if ((s = check_ptr(LSE, "LSE", 4)) != MSA_OK) return s;
  // a shared map lives in a backward-sized workspace (it holds both item lists)
  if ((s = check_ws(p, mapped ? MSA_WS_BWD : MSA_WS_FWD, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_sparse_fwd(p, Q, K, V, block_idx, O, LSE, w, L, st, mapped), "sparse forward launch");
}

msa_status msa_sparse_fwd(const msa_shape* shape, const void* Q, const void* K, const void* V,
                          const int32_t* block_idx, void* O, float* LSE, void* workspace, size_t workspace_bytes,
                          msa_stream_t stream) {
  return sparse_fwd_impl(shape, Q, K, V, block_idx, O, LSE, workspace, workspace_bytes, stream, false);
}

msa_status msa_sparse_fwd_mapped(const msa_shape* shape, const void* Q, const void* K, const void* V,
                                 const int32_t* block_idx, void* O, float* LSE, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream) {
  return sparse_fwd_impl(shape, Q, K, V, block_idx, O, LSE, workspace, workspace_bytes, stream, true);
}

static msa_status bwd_impl(const msa_shape* shape, const void* Q, const void* K, const void* V, const void* O,
                           const void* dO, const float* LSE, const void* q_idx, const void* k_idx,
                           const int32_t* block_idx, float kl_weight, float* dQ, float* dK, float* dV, float* dq_idx,
                           float* dk_idx, float* KL, void* workspace, size_t workspace_bytes, msa_stream_t stream,
                           bool mapped) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  const void* in16[] = {Q, K, V, O, dO, q_idx, k_idx, dQ, dK, dV, dq_idx, dk_idx};
  const char* names16[] = {"Q", "K", "V", "O", "dO", "q_idx", "k_idx", "dQ", "dK", "dV", "dq_idx", "dk_idx"};
  for (int i = 0; i < 12; ++i)
    if ((s = check_ptr(in16[i], names16[i], 16)) != MSA_OK) return s;
  if ((s = check_ptr(LSE, "LSE", 4)) != MSA_OK) return s;
  if ((s = check_ptr(block_idx, "block_idx", 4)) != MSA_OK) return s;
  if ((s = check_ptr(KL, "KL", 4)) != MSA_OK) return s;
  if (!isfinite(kl_weight)) return fail(MSA_ERR_INVALID_ARG, "kl_weight must be finite");
  if ((s = check_ws(p, MSA_WS_BWD, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_bwd(p, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight, dQ, dK, dV, dq_idx,
                                dk_idx, KL, w, L, st, mapped),
                     "backward launch");
}

msa_status msa_bwd(const msa_shape* shape, const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, const void* q_idx, const void* k_idx, const int32_t* block_idx,
                   float kl_weight, float* dQ, float* dK, float* dV, float* dq_idx, float* dk_idx, float* KL,
                   void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return bwd_impl(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight, dQ, dK, dV, dq_idx, dk_idx, KL,
                  workspace, workspace_bytes, stream, false);
}

msa_status msa_bwd_mapped(const msa_shape* shape, const void* Q, const void* K, const void* V, const void* O,
                          const void* dO, const float* LSE, const void* q_idx, const void* k_idx,
                          const int32_t* block_idx, float kl_weight, float* dQ, float* dK, float* dV, float* dq_idx,
                          float* dk_idx, float* KL, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return bwd_impl(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight, dQ, dK, dV, dq_idx, dk_idx, KL,
                  workspace, workspace_bytes, stream, true);
}

msa_status msa_block_map(const msa_shape* shape, const int32_t* block_idx, void* workspace, size_t workspace_bytes,
                         msa_stream_t stream) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  if ((s = check_ptr(block_idx, "block_idx", 4)) != MSA_OK) return s;
  if ((s = check_ws(p, MSA_WS_BWD, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  // lists padded to whole forward tiles (a multiple of the backward tile)
  const int fq = fwd_tile_queries(p);
  return cuda_status(build_block_map2(p, block_idx, w, L, fq, (long long)fq * kFwdTilesPerItem, 1LL << 30, true, st),
                     "block map launch");
}

msa_status msa_warmup_block_idx(const msa_shape* shape, int32_t* block_idx, msa_stream_t stream) {
  Prob p{};
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  if (p.k < p.n)
    return fail(MSA_ERR_UNSUPPORTED, "full attention needs k >= T / Bk = %d blocks (k=%d)", p.n, p.k);
  if ((s = check_ptr(block_idx, "block_idx", 4)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  return cuda_status(launch_warmup_block_idx(p, block_idx, reinterpret_cast<cudaStream_t>(stream)),
                     "warmup block_idx launch");
}

msa_status msa_dense_fwd(const msa_shape* shape, const void* Q, const void* K, const void* V, void* O, float* LSE,
                         void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate_dense(shape, &p)) != MSA_OK) return s;
  if ((s = check_ptr(Q, "Q", 16)) != MSA_OK) return s;
  if ((s = check_ptr(K, "K", 16)) != MSA_OK) return s;
  if ((s = check_ptr(V, "V", 16)) != MSA_OK) return s;
  if ((s = check_ptr(O, "O", 16)) != MSA_OK) return s;
  if ((s = check_ptr(LSE, "LSE", 4)) != MSA_OK) return s;
  if ((s = check_ws(p, MSA_WS_DENSE, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_dense_fwd(p, Q, K, V, O, LSE, w, L, st), "dense forward launch");
}

msa_status msa_dense_bwd(const msa_shape* shape, const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, const void* q_idx, const void* k_idx, float kl_weight,
                         float* dQ, float* dK, float* dV, float* dq_idx, float* dk_idx, float* KL, void* workspace,
                         size_t workspace_bytes, msa_stream_t stream) {
  Prob p{};
  WsLayout L;
  msa_status s;
  if ((s = validate_dense(shape, &p)) != MSA_OK) return s;
  const void* in16[] = {Q, K, V, O, dO, q_idx, k_idx, dQ, dK, dV, dq_idx, dk_idx};
  const char* names16[] = {"Q", "K", "V", "O", "dO", "q_idx", "k_idx", "dQ", "dK", "dV", "dq_idx", "dk_idx"};
  for (int i = 0; i < 12; ++i)
    if ((s = check_ptr(in16[i], names16[i], 16)) != MSA_OK) return s;
  if ((s = check_ptr(LSE, "LSE", 4)) != MSA_OK) return s;
  if ((s = check_ptr(KL, "KL", 4)) != MSA_OK) return s;
  if (!isfinite(kl_weight)) return fail(MSA_ERR_INVALID_ARG, "kl_weight must be finite");
  DenseSchedule ds;
  if (!dense_schedule(p, &ds)) return fail(MSA_ERR_UNSUPPORTED, "B*T too large for the full-attention schedule");
  if ((s = check_ws(p, MSA_WS_DENSE, workspace, workspace_bytes, &L)) != MSA_OK) return s;
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if ((s = cuda_status(cudaMemsetAsync(w, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_bwd_dense(p, Q, K, V, O, dO, LSE, q_idx, k_idx, kl_weight, dQ, dK, dV, dq_idx, dk_idx,
                                      KL, w, L, ds, st),
                     "dense backward launch");
}

msa_status msa_set_timing_events(int32_t which, void* start_event, void* stop_event) {
  if (which < MSA_TIME_INDEX_TOPK || which > MSA_TIME_DENSE_BWD)
    return fail(MSA_ERR_INVALID_ARG, "which=%d is not a timed kernel", which);
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(MSA_ERR_INVALID_ARG, "give both events or neither");
  g_timing[which][0] = static_cast<cudaEvent_t>(start_event);
  g_timing[which][1] = static_cast<cudaEvent_t>(stop_event);
  return MSA_OK;
}

msa_status msa_selftest_wait_timeout(void* workspace, int32_t limit_us, msa_stream_t stream) {
  msa_status s;
  if ((s = check_ptr(workspace, "workspace", 256)) != MSA_OK) return s;
  if (limit_us < 1 || limit_us > 1000000) return fail(MSA_ERR_INVALID_ARG, "limit_us=%d outside [1, 1e6]", limit_us);
  if ((s = check_device()) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = cuda_status(cudaMemsetAsync(workspace, 0, 256, st), "clearing workspace header")) != MSA_OK) return s;
  return cuda_status(launch_selftest_wait_timeout(static_cast<int*>(workspace), (long long)limit_us * 1000, st),
                     "self-test launch");
}

msa_status msa_check_device_status(const void* workspace, msa_stream_t stream) {
  if (!workspace) return fail(MSA_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  msa_status s;
  if ((s = cuda_status(cudaStreamSynchronize(st), "stream synchronize")) != MSA_OK) return s;
  int word = 0;
  if ((s = cuda_status(cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost), "reading error word")) !=
      MSA_OK)
    return s;
  if (word == 0) return MSA_OK;
  cudaMemset(const_cast<void*>(workspace), 0, sizeof word);
  const int code = word / 65536, where = word % 65536;
  return fail(MSA_ERR_DEVICE, "device error %s at site %d",
              code == kDevTimeout ? "timeout (a bounded wait ran out)"
                                  : (code == kDevBadIndex ? "block id out of range" : "unknown"),
              where);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Index top-k without a caller workspace: scratch in a static device array.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MSA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
msa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(MSA_ERR_UNSUPPORTED, "no usable current CUDA device");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return fail(MSA_ERR_CUDA, "looking up the static scratch on device %d: %s", dev, cudaGetErrorString(e));
    }
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return MSA_OK;
}
}  // namespace

extern "C" msa_status msa_index_topk_noalloc(const msa_shape* shape, const void* q_idx, const void* k_idx,
                                             int32_t* block_idx, int32_t check, msa_stream_t stream) {
  Prob p{};
  msa_status s;
  if ((s = validate(shape, &p)) != MSA_OK) return s;
  if ((s = check_topk_k(p)) != MSA_OK) return s;
  if ((s = check_ptr(q_idx, "q_idx", 16)) != MSA_OK) return s;
  if ((s = check_ptr(k_idx, "k_idx", 16)) != MSA_OK) return s;
  if ((s = check_ptr(block_idx, "block_idx", 16)) != MSA_OK) return s;
  const WsLayout L = ws_layout(p, MSA_WS_TOPK);
  if (L.total > (size_t)MSA_NOALLOC_SCRATCH_BYTES)
    return fail(MSA_ERR_UNSUPPORTED, "this shape needs %zu bytes of scratch; the static scratch holds %d", L.total,
                MSA_NOALLOC_SCRATCH_BYTES);
  if ((s = check_device()) != MSA_OK) return s;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // error word and work counter must start at zero; the rest is not read
  if ((s = cuda_status(cudaMemsetAsync(scratch, 0, 256, st), "clearing static scratch")) != MSA_OK) return s;
  if ((s = cuda_status(launch_index_topk(p, q_idx, k_idx, block_idx, scratch, L, st), "index top-k launch")) !=
      MSA_OK)
    return s;
  if (!check) return MSA_OK;
  int word = 0;
  if ((s = cuda_status(cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, st),
                       "reading the error word")) != MSA_OK)
    return s;
  if ((s = cuda_status(cudaStreamSynchronize(st), "stream synchronize")) != MSA_OK) return s;
  if (word != 0)
    return fail(MSA_ERR_DEVICE, "device error %s at site %d",
                word / 65536 == kDevTimeout ? "timeout (a bounded wait ran out)" : "unknown", word % 65536);
  return MSA_OK;
}
