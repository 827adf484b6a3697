// Index branch of MiniMax Sparse Attention: scores, block max-pool and top-k.
//
// itinai.ru "How to solve the memory problem with MiniMax Sparse Attention",
// section "How the indexer works": score every visible token with the
// group's index query against the shared index key, max-pool per block, keep
// the top-k blocks with the query's own block always included; section
// "Kernel optimisations": selection runs on the raw scores (softmax keeps the
// order, so no exp or sum is needed). dothoosh.com "how Flash-MSA cuts
// million-token training cost", "Kernel design and execution": the proxy pass
// accumulates no output, only scores and the running top-k.
//
// GB300 design. One work item = 128 consecutive queries (one query block qb)
// of one (b, g). Its 128 index-query rows (128 x 64 bf16) are the UMMA A
// operand; every earlier KV block c < qb of k_idx (128 x 64) is a B operand.
// Because Bk = 128 = UMMA N, the 128 fp32 columns of one accumulator are
// exactly one block, so each epilogue thread (one TMEM lane = one query) takes
// its block max (from TMEM loads that reduce as they read) and inserts
// (max, c) into a register top-(k-1).
// The own block needs no score: it is always kept.
//
// Warp roles (192 threads, 2 CTAs per SM, persistent over work items handed
// out largest-qb-first by an atomic counter):
//   warp 0      TMA producer: q tile per item, k_idx tiles into a 4-stage ring
//   warp 1      TMEM owner and UMMA issuer (one thread), 2 accumulators
//   warps 2..5  epilogue: tcgen05.ld.red (scores and their max), running top-k, output
#include <cuda_fp8.h>

#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 4;
constexpr int kTileBytes = 128 * 128;  // 128 rows x 64 bf16 (the FP8 path uses half of each tile)
constexpr int kSmemBytes = (2 + kStages) * kTileBytes + 1024;
constexpr int kSmem8 = (2 + kStages) * (kTileBytes / 2) + 1024;  // FP8: 8 KB tiles
// CTAs per SM (each with two TMEM accumulators of 128 columns).
constexpr int kCtasPerSm = 2;

struct TopkArgs {
  int B, T, G, n, k;
  int num_items;
  int32_t* block_idx;
  int* counter;
  int* err;
  const float* k_scale;  // FP8 path: dequantization scale of each (b, key block)
};

struct TopkShared {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t it_full[2], it_empty[2];
  int item[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void decode_item(int item, int B, int G, int n, int& b, int& g, int& qb) {
  const int BG = B * G;
  qb = n - 1 - item / BG;
  const int bg = item % BG;
  b = bg / G;
  g = bg % G;
}

// Insert (v, c) into a list sorted by (value desc, id asc). Ids arrive in
// increasing order, so (v, c) goes after every entry >= v: slot i takes
// (v, c) if v beats entry i but not entry i-1, entry i-1 if v beats both, and
// keeps its own entry otherwise. Every slot is decided from the old list at
// once (no chain through the slots), and the entries below the insertion point
// move down one slot in order, so among equal values the lower ids stay first
// and the last one falls off.
template <int CAP>
__device__ __forceinline__ void topk_insert(float (&val)[CAP], int (&idx)[CAP], float v, int c) {
  if (!(v > val[CAP - 1])) return;
  bool gt[CAP];
#pragma unroll
  for (int i = 0; i < CAP; ++i) gt[i] = v > val[i];
#pragma unroll
  for (int i = CAP - 1; i > 0; --i) {
    val[i] = gt[i] ? (gt[i - 1] ? val[i - 1] : v) : val[i];
    idx[i] = gt[i] ? (gt[i - 1] ? idx[i - 1] : c) : idx[i];
  }
  val[0] = gt[0] ? v : val[0];
  idx[0] = gt[0] ? c : idx[0];
}

// FP8: q and k tiles are E4M3 (128 rows x 64 bytes, 64-byte swizzle), the
// MMAs are kind::f8f6f4 (K = 32 per instruction), and each block's max is
// multiplied by its key-block scale before it enters the top-k (the query
// row's own scale is positive and common to all its blocks: it cannot change
// the selection).
template <int CAP, bool FP8>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    index_topk_kernel(TopkArgs a, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k) {
  constexpr int kLoadBytes = FP8 ? kTileBytes / 2 : kTileBytes;  // bytes a q or k tile load brings
  constexpr int kTB = kLoadBytes;                                 // stage spacing in shared memory
  constexpr int NACC = 2;                                         // TMEM accumulators (128 columns each)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;           // 2 q tiles
  uint8_t* sK = smem + 2 * kTB;  // kStages k tiles
  __shared__ TopkShared sh;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.q_full[i], 1);
      mbar_init(&sh.q_empty[i], 1);
      mbar_init(&sh.acc_full[i], 1);
      mbar_init(&sh.acc_empty[i], 4);
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], 5);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
    }
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, NACC * 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      uint32_t kc = 0;
      for (int it = 0;; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 101)) { *abort_flag = 1; break; }
        int item = atomicAdd(a.counter, 1);
        if (item >= a.num_items || *abort_flag) item = -1;
        sh.item[s] = item;
        mbar_arrive(&sh.it_full[s]);
        if (item < 0) break;
        int b, g, qb;
        decode_item(item, a.B, a.G, a.n, b, g, qb);
        if (!mbar_wait(&sh.q_empty[s], ph ^ 1, a.err, 102)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&sh.q_full[s], kLoadBytes);
        tma_load_3d(sQ + s * kTB, &map_q, &sh.q_full[s], 0, g, b * a.T + qb * 128);
        bool ok = true;
        for (int c = 0; c < qb; ++c, ++kc) {
          const int st = kc % kStages;
          if (!mbar_wait(&sh.k_empty[st], ((kc / kStages) & 1) ^ 1, a.err, 103)) { ok = false; break; }
          mbar_arrive_expect_tx(&sh.k_full[st], kLoadBytes);
          tma_load_2d(sK + st * kTB, &map_k, &sh.k_full[st], 0, b * a.T + c * 128);
        }
        if (!ok) { *abort_flag = 1; break; }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = FP8 ? make_idesc_e4m3(128, 128) : make_idesc_bf16(128, 128, false, false);
      uint32_t kc = 0, ac = 0;
      for (int it = 0;; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 111)) { *abort_flag = 1; break; }
        const int item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item < 0) break;
        int b, g, qb;
        decode_item(item, a.B, a.G, a.n, b, g, qb);
        if (!mbar_wait(&sh.q_full[s], ph, a.err, 112)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t qaddr = smem_u32(sQ + s * kTB);
        bool ok = true;
        for (int c = 0; c < qb; ++c, ++kc, ++ac) {
          const int st = kc % kStages;
          const int ab = ac % NACC;
          if (!mbar_wait(&sh.k_full[st], (kc / kStages) & 1, a.err, 113)) { ok = false; break; }
          if (!mbar_wait(&sh.acc_empty[ab], ((ac / NACC) & 1) ^ 1, a.err, 114)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = smem_u32(sK + st * kTB);
          if constexpr (FP8) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {  // K = 64 bytes = 2 x 32 E4M3 values
              const uint64_t ad = make_sdesc(qaddr + ks * 32, 16, 512, kSw64);
              const uint64_t bd = make_sdesc(kaddr + ks * 32, 16, 512, kSw64);
              umma_e4m3_ss(tmem + ab * 128, ad, bd, idesc, ks > 0);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t ad = make_sdesc(qaddr + ks * 32, 16, 1024, kSw128);
              const uint64_t bd = make_sdesc(kaddr + ks * 32, 16, 1024, kSw128);
              umma_bf16_ss(tmem + ab * 128, ad, bd, idesc, ks > 0);
            }
          }
          umma_commit(&sh.k_empty[st]);
          umma_commit(&sh.acc_full[ab]);
        }
        umma_commit(&sh.q_empty[s]);
        if (!ok) { *abort_flag = 1; break; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t ac = 0;
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 121)) { *abort_flag = 1; break; }
      const int item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item < 0) break;
      int b, g, qb;
      decode_item(item, a.B, a.G, a.n, b, g, qb);
      float val[CAP];
      int idx[CAP];
#pragma unroll
      for (int i = 0; i < CAP; ++i) {
        val[i] = -INFINITY;
        idx[i] = -1;
      }
      bool ok = true;
#pragma unroll 1
      for (int c = 0; c < qb; ++c, ++ac) {
        const int ab = ac % NACC;
        if (!mbar_wait(&sh.acc_full[ab], (ac / NACC) & 1, a.err, 122)) { ok = false; break; }
        tc_fence_after();
        // the block max comes from the loads themselves (the scores are not otherwise needed)
        float mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[32];
          tmem_ld32_max(lane_addr + ab * 128 + q * 32, v, mq[q]);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.acc_empty[ab]);
        float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        if constexpr (FP8) mx *= a.k_scale[(size_t)b * a.n + c];
        topk_insert<CAP>(val, idx, mx, c);
      }
      if (!ok) { *abort_flag = 1; break; }
      // keep the best k-1, order them by block id, append the own block
      const int nsel = min(a.k - 1, qb);
#pragma unroll
      for (int i = 0; i < CAP; ++i)
        if (i >= nsel) idx[i] = 0x7fffffff;
#pragma unroll
      for (int pass = 0; pass < CAP; ++pass) {
#pragma unroll
        for (int i = pass & 1; i + 1 < CAP; i += 2) {
          const int lo = min(idx[i], idx[i + 1]), hi = max(idx[i], idx[i + 1]);
          idx[i] = lo;
          idx[i + 1] = hi;
        }
      }
      const int t = qb * 128 + row;
      int32_t* dst = a.block_idx + (((size_t)b * a.G + g) * a.T + t) * a.k;
#pragma unroll
      for (int i = 0; i <= CAP; ++i) {
        if (i < a.k) {
          const int v = i < nsel ? idx[i < CAP ? i : 0] : (i == nsel ? qb : -1);
          dst[i] = v;
        }
      }
      for (int i = CAP + 1; i < a.k; ++i) dst[i] = -1;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, NACC * 128);
}

template <int CAP, bool FP8>
cudaError_t launch_cap(const Prob& p, const TopkArgs& args, const CUtensorMap& mq, const CUtensorMap& mk,
                       cudaStream_t st) {
  auto kern = index_topk_kernel<CAP, FP8>;
  constexpr int smem_bytes = FP8 ? kSmem8 : kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  const int grid = min(args.num_items, kCtasPerSm * num_sms());
  timing_begin(MSA_TIME_INDEX_TOPK, st);
  kern<<<grid, kThreads, smem_bytes, st>>>(args, mq, mk);
  timing_end(MSA_TIME_INDEX_TOPK, st);
  count_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- FP8 index inputs
// E4M3 copies of the index queries (one scale per (b, t, g) row) and keys
// (one scale per (b, 128-key block)): x * (448 / amax) rounded to nearest
// (ties to even) with saturation; the dequantization scale is amax / 448.
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// One warp per q_idx row of 64 values.
__global__ void quant_q_kernel(const __nv_bfloat16* __restrict__ q, uint16_t* __restrict__ q8, long long rows) {
  const int lane = threadIdx.x & 31;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((long long)gridDim.x * blockDim.x) >> 5) {
    const float2 v = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(q + r * 64)[lane]);
    float amax = fmaxf(fabsf(v.x), fabsf(v.y));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float mul = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    q8[r * 32 + lane] = to_e4m3x2(__fmul_rn(v.x, mul), __fmul_rn(v.y, mul));
  }
}

// One 256-thread CTA per (b, key block): 128 rows x 64 values.
__global__ void __launch_bounds__(256) quant_k_kernel(const __nv_bfloat16* __restrict__ k, uint16_t* __restrict__ k8,
                                                      float* __restrict__ k_scale, int T, int n) {
  __shared__ float wmax[8];
  const int bc = blockIdx.x, b = bc / n, c = bc % n;
  const size_t base = ((size_t)b * T + (size_t)c * 128) * 64;  // 128 x 64 bf16 = 4096 pairs
  const __nv_bfloat162* src = reinterpret_cast<const __nv_bfloat162*>(k + base);
  float2 v[16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = __bfloat1622float2(src[threadIdx.x + 256 * i]);
    amax = fmaxf(amax, fmaxf(fabsf(v[i].x), fabsf(v[i].y)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, wmax[i]);
  const float mul = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
  if (threadIdx.x == 0) k_scale[bc] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint16_t* dst = k8 + base / 2;
#pragma unroll
  for (int i = 0; i < 16; ++i) dst[threadIdx.x + 256 * i] = to_e4m3x2(__fmul_rn(v[i].x, mul), __fmul_rn(v[i].y, mul));
}

}  // namespace

cudaError_t launch_index_topk(const Prob& p, const void* q_idx, const void* k_idx, int32_t* block_idx, void* ws,
                              const WsLayout& L, cudaStream_t st) {
  CUtensorMap mq, mk;
  {
    const uint64_t dims[3] = {(uint64_t)p.E, (uint64_t)p.G, (uint64_t)p.BT()};
    const uint64_t strides[2] = {(uint64_t)p.E * 2, (uint64_t)p.G * p.E * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap(&mq, const_cast<void*>(q_idx), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)p.E, (uint64_t)p.BT()};
    const uint64_t strides[1] = {(uint64_t)p.E * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap(&mk, const_cast<void*>(k_idx), 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  TopkArgs args;
  args.B = p.B;
  args.T = p.T;
  args.G = p.G;
  args.n = p.n;
  args.k = p.k;
  args.num_items = p.B * p.G * p.n;
  args.block_idx = block_idx;
  args.counter = reinterpret_cast<int*>(w + L.counters);
  args.err = reinterpret_cast<int*>(w + L.err);
  cudaError_t e = cudaMemsetAsync(args.counter, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  args.k_scale = nullptr;
  const int need = p.k - 1;
  if (need <= 4) return launch_cap<4, false>(p, args, mq, mk, st);
  if (need <= 16) return launch_cap<16, false>(p, args, mq, mk, st);
  if (need <= 32) return launch_cap<32, false>(p, args, mq, mk, st);
  return launch_cap<64, false>(p, args, mq, mk, st);
}

cudaError_t launch_index_topk_fp8(const Prob& p, const void* q_idx, const void* k_idx, int32_t* block_idx, void* ws,
                                  const WsLayout& L, cudaStream_t st) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* q8 = reinterpret_cast<uint16_t*>(w + L.q8);
  uint16_t* k8 = reinterpret_cast<uint16_t*>(w + L.k8);
  float* ks = reinterpret_cast<float*>(w + L.k_scale);
  const long long qrows = (long long)p.B * p.T * p.G;
  quant_q_kernel<<<(int)std::min<long long>((qrows * 32 + 255) / 256, 16LL * num_sms()), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q_idx), q8, qrows);
  quant_k_kernel<<<p.B * p.n, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(k_idx), k8, ks, p.T, p.n);
  count_launches(2);
  CUtensorMap mq, mk;
  {
    const uint64_t dims[3] = {64, (uint64_t)p.G, (uint64_t)p.BT()};
    const uint64_t strides[2] = {64, (uint64_t)p.G * 64};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap(&mq, q8, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {64, (uint64_t)p.BT()};
    const uint64_t strides[1] = {64};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap(&mk, k8, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return cudaErrorInvalidValue;
  }
  TopkArgs args;
  args.B = p.B;
  args.T = p.T;
  args.G = p.G;
  args.n = p.n;
  args.k = p.k;
  args.num_items = p.B * p.G * p.n;
  args.block_idx = block_idx;
  args.counter = reinterpret_cast<int*>(w + L.counters);
  args.err = reinterpret_cast<int*>(w + L.err);
  args.k_scale = ks;
  cudaError_t e = cudaMemsetAsync(args.counter, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  const int need = p.k - 1;
  if (need <= 4) return launch_cap<4, true>(p, args, mq, mk, st);
  if (need <= 16) return launch_cap<16, true>(p, args, mq, mk, st);
  if (need <= 32) return launch_cap<32, true>(p, args, mq, mk, st);
  return launch_cap<64, true>(p, args, mq, mk, st);
}

}  // namespace msa
