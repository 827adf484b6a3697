// Fused backward of MiniMax Sparse Attention: main-branch dQ/dK/dV and the
// KL-alignment gradient of the index branch in one pass over the selected
// blocks.
//
// dothoosh.com "how Flash-MSA cuts million-token training cost", "Kernel
// design and execution": the backward fuses proxy and main attention because
// the proxy's training signal needs both distributions at once, and inverting
// the block-index map schedules the query chunks of each sparse KV block so
// the block is reused from shared memory; "Fixing the KL-divergence
// bottleneck": d KL / d s_px = p_px - p_main, so no full KL distribution is
// materialised. itinai.ru "How to solve the memory problem with MiniMax
// Sparse Attention", "Training sparse attention": the teacher is the main
// softmax averaged over the group's heads, detached from the backbone.
// dothoosh.com "how FlashAttention cuts GPU memory traffic", "Training and the
// backward pass": P is rebuilt from the saved LSE; dV += P^T dO, dP = dO V^T.
//
// Kernels, in launch order:
//   drow_kernel       D[b,t,h] = rowsum(dO * O)
//   px_stats_kernel   index-branch log-sum-exp over S(g,t), per (query, slot):
//                     tcgen05 S_px = q_idx rows x k_idx block^T, one query
//                     per TMEM lane, 128 queries per tile
//   px_merge_kernel   lse_px[b,t,g] from the k partials
//   bwd_kernel        per KV block c of (b, g), over the tiles of queries that
//                     selected it (keys on TMEM lanes, 64 (query, head) rows
//                     per tile):
//                       S^T = K_c Q^T, dP^T = V_c dO^T, X^T = KI_c QI^T
//                       P = exp(s - LSE), dS = P (dP - D), p_main = head mean,
//                       p_px = exp(x - lse_px), gs = w (p_px - p_main), KL terms
//                       dV += P^T dO, dK += dS^T Q, dk_idx += gs^T QI (TMEM,
//                       across all tiles of the block), dQ^T = K_c^T dS^T and
//                       dq_idx^T = KI_c^T gs^T (per tile, to slot partials)
//   bwd_merge_kernel  dQ, dq_idx, KL = sums of the slot partials; dk_idx = sum
//                     over groups of the per-group dk_idx rows
#include "bwd_common.cuh"

namespace msa {
namespace {

using bwdc::decode_list;
using bwdc::fast_exp2;
using bwdc::LanesSum;
using bwdc::lanes_sum;
using bwdc::pack_bf16;
constexpr float kLog2e = kBwdLog2e;
constexpr float kLn2 = kBwdLn2;

// ============================================================================ D
__global__ void drow_kernel(const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
                            float* __restrict__ drow, long long rows) {
  const int lane = threadIdx.x & 31;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((long long)gridDim.x * blockDim.x) >> 5) {
    const uint2 a = *reinterpret_cast<const uint2*>(O + r * 128 + lane * 4);
    const uint2 b = *reinterpret_cast<const uint2*>(dO + r * 128 + lane * 4);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
    const float2 a0 = __bfloat1622float2(pa[0]), a1 = __bfloat1622float2(pa[1]);
    const float2 b0 = __bfloat1622float2(pb[0]), b1 = __bfloat1622float2(pb[1]);
    float s = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) drow[r] = s;
  }
}

// ============================================================================ px stats
// One CTA per SM, persistent over whole lists. 128 queries per tile, gathered
// by four producer warps (32 rows each: warp 0, which also fetches the items
// and the k_idx block, and warps 6-8) into three stages; warp 1 issues the
// UMMAs, warps 2-5 reduce the 128 scores of their row.
constexpr int kPxThreads = 288;
constexpr int kPxTile = 16384;  // 128 rows x 64 bf16
constexpr int kPxStages = 3;
constexpr int kPxSmem = (1 + kPxStages) * kPxTile + 1024;

struct PxArgs {
  const __nv_bfloat16* q_idx;
  const int32_t* entries;
  const int4* items;
  const int* n_items;
  int* counter;
  int* err;
  float* px_part;  // [B,T,G,k]
  int B, T, G, n, k;
  float scale_log2;
};

struct PxShared {
  uint64_t it_full[2], it_empty[2];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[kPxStages], q_empty[kPxStages];
  uint64_t s_full[2], s_empty[2];
  int4 item[2];
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kPxThreads, 1)
    px_stats_kernel(PxArgs a, const __grid_constant__ CUtensorMap map_ki) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKI = smem;
  uint8_t* sQ = smem + kPxTile;  // kPxStages tiles
  __shared__ PxShared sh;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], 3 + 1 + 4);  // other producers, UMMA, reduction warps
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.s_empty[i], 4);
    }
    for (int i = 0; i < kPxStages; ++i) {
      mbar_init(&sh.q_full[i], 128);  // every producer lane, after its copies
      mbar_init(&sh.q_empty[i], 1);
    }
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort;
  const int n_items = *a.n_items;

  const int pxp = warp == 0 ? 0 : (warp >= 6 ? warp - 5 : -1);  // producer index: rows [32 pxp, 32 pxp + 32)
  if (pxp >= 0) {
    uint32_t tj = 0;
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      int4 item = make_int4(-1, 0, 0, 0);
      if (pxp == 0) {
        if (lane == 0) {
          if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 401)) *abort_flag = 1;
          const int id = atomicAdd(a.counter, 1);
          if (id < n_items && !*abort_flag) item = a.items[id];
          sh.item[s] = item;
          mbar_arrive(&sh.it_full[s]);
        }
        item.x = __shfl_sync(0xffffffffu, item.x, 0);
        item.y = __shfl_sync(0xffffffffu, item.y, 0);
        item.z = __shfl_sync(0xffffffffu, item.z, 0);
      } else {
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 404)) { *abort_flag = 1; break; }
        item = sh.item[s];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      }
      if (item.x < 0) break;
      int b, g, c;
      decode_list(item.x, a.n, a.G, b, g, c);
      if (pxp == 0) {
        if (lane == 0) {
          if (mbar_wait(&sh.kv_empty, (it & 1) ^ 1, a.err, 402)) {
            mbar_arrive_expect_tx(&sh.kv_full, kPxTile);
            tma_load_2d(sKI, &map_ki, &sh.kv_full, 0, b * a.T + c * 128);
          } else {
            *abort_flag = 1;
          }
        }
        __syncwarp();
        if (*abort_flag) break;
      }
      const int ntiles = (item.z + 127) / 128;
      // lane = row 32 pxp + lane: its query, one tile ahead
      auto row_t = [&](int j) -> int {
        const int idx = j * 128 + 32 * pxp + lane;
        return idx < item.z ? (a.entries[item.y + idx] >> 8) : -1;
      };
      int t_own = row_t(0);
      bool ok = true;
      for (int j = 0; j < ntiles; ++j, ++tj) {
        const int qs = tj % kPxStages;
        if (!mbar_wait(&sh.q_empty[qs], ((tj / kPxStages) & 1) ^ 1, a.err, 403)) { ok = false; break; }
        const uint32_t dst0 = smem_u32(sQ + qs * kPxTile);
        // 32 rows x 8 chunks: lane -> (row 4 i + lane / 8, chunk lane % 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rl = 4 * i + (lane >> 3), chunk = lane & 7;
          const int tq = __shfl_sync(0xffffffffu, t_own, rl);
          const bool valid = tq >= 0;
          const __nv_bfloat16* src = a.q_idx + ((((size_t)b * a.T + (valid ? tq : 0)) * a.G + g) * 64 + chunk * 8);
          cp_async_16_zfill(dst0 + sw128_off(32 * pxp + rl, chunk), src, valid);
        }
        cp_async_commit();
        if (j + 1 < ntiles) t_own = row_t(j + 1);
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(&sh.q_full[qs]);
        __syncwarp();
      }
      if (!ok) { *abort_flag = 1; break; }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(128, 128, false, false);
      const uint32_t k0 = smem_u32(sKI);
      uint32_t tj = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 411)) { ok = false; break; }
        const int4 item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item.x < 0) break;
        const int ntiles = (item.z + 127) / 128;
        if (!mbar_wait(&sh.kv_full, it & 1, a.err, 412)) { ok = false; break; }
        for (int j = 0; j < ntiles; ++j, ++tj) {
          const int sb = tj & 1, qs = tj % kPxStages;
          if (!mbar_wait(&sh.q_full[qs], (tj / kPxStages) & 1, a.err, 413)) { ok = false; break; }
          if (!mbar_wait(&sh.s_empty[sb], ((tj >> 1) & 1) ^ 1, a.err, 414)) { ok = false; break; }
          tc_fence_after();
          const uint32_t q0 = smem_u32(sQ + qs * kPxTile);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16_ss(tmem + sb * 128, make_sdesc(q0 + ks * 32, 16, 1024, kSw128),
                         make_sdesc(k0 + ks * 32, 16, 1024, kSw128), idesc, ks > 0);
          umma_commit(&sh.s_full[sb]);
          umma_commit(&sh.q_empty[qs]);
        }
        umma_commit(&sh.kv_empty);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t tj = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 421)) { ok = false; break; }
      const int4 item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item.x < 0) break;
      int b, g, c;
      decode_list(item.x, a.n, a.G, b, g, c);
      const int ntiles = (item.z + 127) / 128;
      for (int j = 0; j < ntiles; ++j, ++tj) {
        const int sb = tj & 1;
        const int idx = j * 128 + row;
        const int entry = idx < item.z ? a.entries[item.y + idx] : -1;
        const int lim = entry >= 0 ? (entry >> 8) - c * 128 : -1;
        if (!mbar_wait(&sh.s_full[sb], (tj >> 1) & 1, a.err, 422)) { ok = false; break; }
        tc_fence_after();
        float x[128], mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32_max(tmem + lane_off + sb * 128 + q * 32, *reinterpret_cast<float(*)[32]>(x + q * 32), mq[q]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.s_empty[sb]);
        float mm, l = 0.f;
        if (lim >= 127) {  // every key visible: the loads' own maximum (scale > 0 keeps it the maximum)
          mm = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.scale_log2;
#pragma unroll
          for (int i = 0; i < 128; ++i) l += fast_exp2(fmaf(x[i], a.scale_log2, -mm));
        } else {
          float m = -INFINITY;
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            x[i] = (i <= lim) ? x[i] * a.scale_log2 : -INFINITY;
            m = fmaxf(m, x[i]);
          }
          mm = (m == -INFINITY) ? 0.f : m;
#pragma unroll
          for (int i = 0; i < 128; ++i) l += fast_exp2(x[i] - mm);
        }
        if (entry >= 0) {
          const int t = entry >> 8, slot = entry & 255;
          a.px_part[(((size_t)b * a.T + t) * a.G + g) * a.k + slot] = (mm + __log2f(l)) * kLn2;
        }
      }
    }
    if (!ok) *abort_flag = 1;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// lse_px[b,t,g] = ln sum_s exp(px_part[b,t,g,s]) over the valid slots.
__global__ void px_merge_kernel(const int32_t* __restrict__ block_idx, const float* __restrict__ px_part,
                                float* __restrict__ lse_px, int B, int T, int G, int k) {
  const long long rows = (long long)B * T * G;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(r % G);
    const long long bt = r / G;
    const int t = (int)(bt % T), b = (int)(bt / T);
    const int32_t* sel = block_idx + (((size_t)b * G + g) * T + t) * k;
    float mx = -INFINITY;
    for (int s = 0; s < k; ++s)
      if (sel[s] >= 0) mx = fmaxf(mx, px_part[r * k + s]);
    float z = 0.f;
    for (int s = 0; s < k; ++s)
      if (sel[s] >= 0) z += expf(px_part[r * k + s] - mx);
    lse_px[r] = mx + logf(z);
  }
}

// ============================================================================ fused backward
constexpr int kBwdThreads = 512;  // 7 producer warps, 1 UMMA warp, 8 epilogue warps (two column halves)
constexpr int kProd = 7;          // producer warps: 0, 6, 11..15
constexpr int kRows = 64;                // (query, head) rows per tile
constexpr int kKV = 32768;               // 128 keys x 128 d
constexpr int kKIb = 16384;              // 128 keys x 64
constexpr int kRowTile = kRows * 256;    // 64 rows x 128 d  (16 KB)
constexpr int kRowChunk = kRows * 128;   // one 64-column chunk of it (8 KB)
constexpr int kKeyRows = 128 * 128;      // 128 keys x 64 bf16 (16 KB)
// smem map (the dynamic base is 1024-aligned; checked at entry): K, V, k_idx
// of the block, then the per-HG part (BwdLayout)
constexpr int oK = 0, oV = kKV, oKI = 2 * kKV;
// TMEM columns. A tile's 64 columns at cR[tile parity] hold S^T, then dP^T
// (once the epilogue has loaded S), then dQ^T (once it has loaded dP): the
// next tile's S^T goes to the other region while this tile finishes. cX holds
// the index scores X^T, then dq_idx^T. cP holds P^T as packed bf16 pairs,
// the A operand of dV += P^T dO, when cX leaves room for it (hg >= 2).
constexpr uint32_t cR0 = 0, cX = 128, cP = 160, cDV = 192, cDK = 320, cKI = 448;

// Per (query, head) row of a tile, structure of arrays so that a 16-byte
// shared load serves four columns. Padding rows hold +inf log-sum-exps, which
// make their probabilities exactly zero without a mask.
struct __align__(16) RowMeta {
  float lse2[kRows];  // LSE * log2 e
  float dsc[kRows];   // D * scale
  float lpx2[kRows];  // lse_px * log2 e
  int ent[kRows];     // entry bits t << 8 | slot, -1 for padding
  int diag[8];        // per producer: some row sees only part of the block (causal mask needed)
};

struct BwdShared {
  uint64_t it_full[2], it_empty[2];
  uint64_t kv_full, kv_empty;
  uint64_t g_full[3], g_empty[3];
  uint64_t s_full, s_read, dp_full, x_full;  // S^T computed / loaded by the epilogue, dP^T and X^T computed
  uint64_t p_ready, ds_ready, gs_ready, ph2_full;
  uint64_t r_free[2], x_free;  // a tile's dQ^T / dq_idx^T read out of TMEM (by tile parity / every tile)
  uint64_t pv_free;            // dV += P^T dO of a tile complete: P^T may be overwritten
  uint64_t acc_free;
  RowMeta meta[3];  // one per gather buffer
  int4 item[2];
  uint32_t tmem_base;
  int abort;
};
// Shared-memory layout for HG heads per group. A tile's gather buffer holds
// its Q and dO rows and its q_idx rows (one per query, NX of them). Three
// buffers when P^T lives in TMEM (its shared image is not needed), else two.
template <int HG>
struct BwdLayout {
  static constexpr int kNpos = kRows / HG;                    // queries per tile
  static constexpr int kNX = kNpos < 16 ? 16 : kNpos;         // index-score columns (MMA N >= 16)
  static constexpr bool kPTmem = kNX <= 32;                   // P^T fits in TMEM beside X^T
  static constexpr int kQI = kNX * 128;                       // q_idx rows of a tile
  static constexpr int kGather = 2 * kRowTile + kQI;          // Q, dO, q_idx
  static constexpr int kNG = kPTmem ? 3 : 2;                  // gather buffers
  static constexpr int oG = 2 * kKV + kKIb;
  static constexpr int oPT = oG + kNG * kGather;              // P^T image (only without TMEM room)
  static constexpr int oDST = oPT + (kPTmem ? 0 : kKeyRows);  // dS^T
  static constexpr int oGST = oDST + kKeyRows;                // gs^T
  static constexpr int oSh = oGST + kKeyRows;                 // BwdShared
  static constexpr int kSmem = oSh + (int)sizeof(BwdShared);
  static_assert(kGather % 1024 == 0, "gather buffers keep the 1024-byte swizzle alignment");
  static_assert(kSmem <= 232448, "backward kernel exceeds 227 KB of shared memory");
};

template <int HG>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(BwdArgs a, const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
               const __grid_constant__ CUtensorMap map_ki, const __grid_constant__ CUtensorMap map_dq,
               const __grid_constant__ CUtensorMap map_dqi, const __grid_constant__ CUtensorMap map_q,
               const __grid_constant__ CUtensorMap map_do, const __grid_constant__ CUtensorMap map_qi) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // uniform for the block: nothing started yet
    if (threadIdx.x == 0) dev_fail(a.err, kDevSmemAlign, 500);
    return;
  }
  using L = BwdLayout<HG>;
  constexpr int oG = L::oG, kGather = L::kGather, kNG = L::kNG;
  constexpr int oPT = L::oPT, oDST = L::oDST, oGST = L::oGST;
  BwdShared& sh = *reinterpret_cast<BwdShared*>(smem + L::oSh);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) sh.meta[0].diag[i] = sh.meta[1].diag[i] = sh.meta[2].diag[i] = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], kProd - 1 + 1 + 8);  // other producers, UMMA, epilogue warps
    }
    for (int i = 0; i < kNG; ++i) {
      mbar_init(&sh.g_full[i], kProd);   // every producer warp (with its TMA bytes)
      mbar_init(&sh.g_empty[i], 1 + 8);  // MMA commit + epilogue warps (meta, store staging)
    }
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.s_read, 8);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.x_full, 1);
    mbar_init(&sh.p_ready, 8);
    mbar_init(&sh.ds_ready, 8);
    mbar_init(&sh.gs_ready, 8);
    mbar_init(&sh.ph2_full, 1);
    mbar_init(&sh.r_free[0], 8);
    mbar_init(&sh.r_free[1], 8);
    mbar_init(&sh.x_free, 8);
    mbar_init(&sh.pv_free, 1);
    mbar_init(&sh.acc_free, 8);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  // q_idx rows and gs^T columns past the queries of a tile (hg = 8 pads the
  // index MMAs to N = 16) are never written by the pipeline: zero them once
  for (int i = threadIdx.x; i < kNG * (L::kQI / 16); i += kBwdThreads)
    reinterpret_cast<uint4*>(smem + oG + (i / (L::kQI / 16)) * kGather + 2 * kRowTile)[i % (L::kQI / 16)] =
        make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < kKeyRows / 16; i += kBwdThreads)
    reinterpret_cast<uint4*>(smem + oGST)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort;
  const int n_items = *a.n_items;
  constexpr int hg = HG;          // heads per group (compile time: static register indexing)
  constexpr int npos = L::kNpos;   // queries per tile
  constexpr int NX = L::kNX;        // index-score columns (one per query; MMA N >= 16)
  constexpr int kQ = 32 / hg;       // queries in the 32 rows of a producer warp / epilogue column half
  constexpr bool kPTmem = L::kPTmem;

  // Producer warps (kProd of them): producer p owns the queries p, p + kProd,
  // ... of every tile, i.e. their metadata rows and their TMA boxes, so the
  // producers never wait on one another. Lane l < (its queries) x hg holds
  // the row of query p + kProd (l / hg), head l % hg. The next tile's entry
  // and metadata are loaded into registers right after the current tile is
  // published, so their memory latency overlaps the wait for the next buffer.
  auto load_entry = [&](const int4& item, int j, int q) -> int {
    const int idx = j * npos + q;
    return idx < item.z ? a.entries[item.y + idx] : -1;
  };
  auto load_rec = [&](int b, int g, int e, int h) -> float4 {
    if (e < 0) return make_float4(INFINITY, 0.f, INFINITY, __int_as_float(e));
    const int t = e >> 8;
    const size_t hr = ((size_t)b * a.T + t) * a.Hq + g * hg + h;
    const float l = a.LSE[hr], d = a.drow[hr];
    const float x = a.lse_px[((size_t)b * a.T + t) * a.G + g];
    return make_float4(l * kLog2e, d * a.scale, x * kLog2e, __int_as_float(e));
  };
  // Writes this producer's metadata rows of buffer gb and gathers its queries
  // with TMA: per query, its hg consecutive head rows of Q and dO (one box per
  // 64-column chunk) and its q_idx row (row = query index in the tile). TMA
  // swizzles by the shared address, so a box landing at row r0 matches the
  // tile's 128-byte swizzle; padding queries load an out-of-range box, which
  // is zero-filled. key_last is the last key of the block: rows with an
  // earlier query need the causal mask.
  auto fill_part = [&](int p, int nq, int b, int g, int key_last, int gb, const float4& rec) {
    uint8_t* buf = smem + oG + gb * kGather;
    RowMeta& m = sh.meta[gb];
    const bool mine = lane < nq * hg;
    const int e_own = __float_as_int(rec.w);
    if (mine) {
      const int r = (p + kProd * (lane / hg)) * hg + lane % hg;
      m.lse2[r] = rec.x;
      m.dsc[r] = rec.y;
      m.lpx2[r] = rec.z;
      m.ent[r] = e_own;
    }
    const unsigned dg = __ballot_sync(0xffffffffu, mine && e_own >= 0 && (e_own >> 8) < key_last);
    if (lane == 0) {
      m.diag[p] = dg != 0u;
      mbar_arrive_expect_tx(&sh.g_full[gb], nq * (2 * hg * 256 + 128));
    }
    __syncwarp();
    const int BT = a.B * a.T;
#pragma unroll 1
    for (int o = lane; o < nq * 5; o += 32) {  // per query: Q and dO chunk boxes, then the q_idx row
      const int i = o / 5, op = o - i * 5;
      const int q = p + kProd * i;
      const int r0 = q * hg;
      const int e = m.ent[r0];
      const int bt = e >= 0 ? b * a.T + (e >> 8) : BT;  // BT: out of range, zero fill
      if (op < 4) {
        const int which = op >> 1, chunk = op & 1;
        tma_load_3d(buf + which * kRowTile + chunk * kRowChunk + r0 * 128, which ? &map_do : &map_q,
                    &sh.g_full[gb], chunk * 64, g * hg, bt);
      } else {
        tma_load_2d(buf + 2 * kRowTile + q * 128, &map_qi, &sh.g_full[gb], 0, bt * a.G + g);
      }
    }
    __syncwarp();
  };
  // All tiles of one item for producer p.
  auto fill_item = [&](int p, const int4& item, int b, int g, int c, uint32_t& tj) -> bool {
    const int ntiles = (item.z + npos - 1) / npos;
    const int nq = (npos - p + kProd - 1) / kProd;  // queries of this producer in a tile
    const int q = p + kProd * (lane / hg), h = lane % hg;
    const bool mine = lane < nq * hg;
    int e_next = mine ? load_entry(item, 0, q) : -1;
    float4 rec = load_rec(b, g, e_next, h);
    e_next = (mine && ntiles > 1) ? load_entry(item, 1, q) : -1;
    for (int j = 0; j < ntiles; ++j, ++tj) {
      const int gb = tj % kNG;
      if (!mbar_wait(&sh.g_empty[gb], ((tj / kNG) & 1) ^ 1, a.err, 503 + p)) return false;
      fill_part(p, nq, b, g, c * 128 + 127, gb, rec);
      if (j + 1 < ntiles) {
        rec = load_rec(b, g, e_next, h);
        e_next = (mine && j + 2 < ntiles) ? load_entry(item, j + 2, q) : -1;
      }
    }
    return true;
  };

  const int prod = warp == 0 ? 0 : warp == 6 ? 1 : warp >= 11 ? warp - 9 : -1;
  if (prod >= 0) {
    // ------------------------------------------------------------ producers; producer 0 also
    // fetches the work items and loads each item's K, V and k_idx block
    uint32_t tj = 0;
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      int4 item = make_int4(-1, 0, 0, 0);
      if (prod == 0) {
        if (lane == 0) {
          if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 501)) *abort_flag = 1;
          const int id = atomicAdd(a.counter, 1);
          if (id < n_items && !*abort_flag) item = a.items[id];
          sh.item[s] = item;
          mbar_arrive(&sh.it_full[s]);
        }
        item.x = __shfl_sync(0xffffffffu, item.x, 0);
        item.y = __shfl_sync(0xffffffffu, item.y, 0);
        item.z = __shfl_sync(0xffffffffu, item.z, 0);
        item.w = __shfl_sync(0xffffffffu, item.w, 0);
      } else {
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 531)) { *abort_flag = 1; break; }
        item = sh.item[s];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      }
      if (item.x < 0) break;
      int b, g, c;
      decode_list(item.x, a.n, a.G, b, g, c);
      if (prod == 0) {
        if (lane == 0) {
          if (mbar_wait(&sh.kv_empty, (it & 1) ^ 1, a.err, 502)) {
            mbar_arrive_expect_tx(&sh.kv_full, 2 * kKV + kKIb);
            const int row0 = b * a.T + c * 128;
            tma_load_3d(smem + oK, &map_k, &sh.kv_full, 0, g, row0);
            tma_load_3d(smem + oK + kKV / 2, &map_k, &sh.kv_full, 64, g, row0);
            tma_load_3d(smem + oV, &map_v, &sh.kv_full, 0, g, row0);
            tma_load_3d(smem + oV + kKV / 2, &map_v, &sh.kv_full, 64, g, row0);
            tma_load_2d(smem + oKI, &map_ki, &sh.kv_full, 0, row0);
          } else {
            *abort_flag = 1;
          }
        }
        __syncwarp();
        if (*abort_flag) break;
      }
      if (!fill_item(prod, item, b, g, c, tj)) { *abort_flag = 1; break; }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sT = make_idesc_bf16(128, 64, false, false);   // K-major x K-major, N=64
      constexpr uint32_t id_acc = make_idesc_bf16(128, 128, false, true);  // K-major A, MN-major B, N=128
      constexpr uint32_t id_tr = make_idesc_bf16(128, 64, true, true);     // MN-major A and B, N=64
      constexpr uint32_t id_ki = make_idesc_bf16(128, 64, false, true);    // K-major A, MN-major B, N=64
      constexpr uint32_t id_x = make_idesc_bf16(128, NX, false, false);    // K-major x K-major, N=NX
      constexpr uint32_t id_trx = make_idesc_bf16(128, NX, true, true);    // MN-major A and B, N=NX
      // Shared-memory descriptors, built once: a k-step or the other gather
      // buffer moves only the start-address field, so every UMMA below adds a
      // constant to one of these bases.
      const uint64_t dK = make_sdesc(smem_u32(smem + oK), 16, 1024, kSw128);        // K, K-major
      const uint64_t dKt = make_sdesc(smem_u32(smem + oK), kKV / 2, 1024, kSw128);   // K as MN-major A
      const uint64_t dV = make_sdesc(smem_u32(smem + oV), 16, 1024, kSw128);
      const uint64_t dKI = make_sdesc(smem_u32(smem + oKI), 16, 1024, kSw128);
      const uint64_t dKIt = make_sdesc(smem_u32(smem + oKI), kKIb, 1024, kSw128);
      const uint64_t dPT = make_sdesc(smem_u32(smem + oPT), 16, 1024, kSw128);
      const uint64_t dDS = make_sdesc(smem_u32(smem + oDST), 16, 1024, kSw128);
      const uint64_t dGS = make_sdesc(smem_u32(smem + oGST), 16, 1024, kSw128);
      const uint64_t dG = make_sdesc(smem_u32(smem + oG), 16, 1024, kSw128);
      const uint64_t dGt = make_sdesc(smem_u32(smem + oG), kRowChunk, 1024, kSw128);  // rows as MN-major B
      auto at = [](uint64_t d, uint32_t off) -> uint64_t { return d + (uint64_t)(off >> 4); };
      uint32_t tj = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 511)) { ok = false; break; }
        const int4 item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item.x < 0) break;
        const int ntiles = (item.z + npos - 1) / npos;
        if (!mbar_wait(&sh.kv_full, it & 1, a.err, 512)) { ok = false; break; }
        // S^T of a tile, into region cR[tile & 1], once its gather buffer is
        // full and the readout of tile - 2 has freed that region
        auto issue_s = [&](uint32_t u) -> bool {
          const int ub = u % kNG;
          if (!mbar_wait(&sh.g_full[ub], (u / kNG) & 1, a.err, 513)) return false;
          if (!mbar_wait(&sh.r_free[u & 1], ((u >> 1) & 1) ^ 1, a.err, 514)) return false;
          tc_fence_after();
          const uint64_t bq = at(dG, ub * kGather);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ao = (ks >> 2) * (kKV / 2) + (ks & 3) * 32;
            const uint32_t bo = (ks >> 2) * kRowChunk + (ks & 3) * 32;
            umma_bf16_ss(tmem + cR0 + 64 * (u & 1), at(dK, ao), at(bq, bo), id_sT, ks > 0);
          }
          umma_commit(&sh.s_full);
          return true;
        };
        // Per tile, in the order the epilogue releases its operands; the next
        // tile's S^T goes out once this tile's dK / dQ^T are queued, so that it
        // is computed while the epilogue works on this tile's index branch.
        bool s_issued = false;  // this tile's S^T went out during the previous tile
        for (int j = 0; j < ntiles; ++j, ++tj) {
          const int gb = tj % kNG;
          if (!s_issued && !issue_s(tj)) { ok = false; break; }
          s_issued = false;
          const uint32_t tR = tmem + cR0 + 64 * (tj & 1);
          const uint32_t goff = gb * kGather;
          const uint64_t bO = at(dG, goff + kRowTile), bQI = at(dG, goff + 2 * kRowTile);
          const uint64_t bQt = at(dGt, goff), bOt = at(dGt, goff + kRowTile);
          // dP^T = V dO^T into S^T's columns, once every epilogue warp has loaded S^T
          if (!mbar_wait(&sh.s_read, tj & 1, a.err, 520)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ao = (ks >> 2) * (kKV / 2) + (ks & 3) * 32;
            const uint32_t bo = (ks >> 2) * kRowChunk + (ks & 3) * 32;
            umma_bf16_ss(tR, at(dV, ao), at(bO, bo), id_sT, ks > 0);
          }
          umma_commit(&sh.dp_full);
          // dV += P^T dO   (K = 64 rows, 16 per step)
          if (!mbar_wait(&sh.p_ready, tj & 1, a.err, 515)) { ok = false; break; }
          if (j == 0 && !mbar_wait(&sh.acc_free, (it & 1) ^ 1, a.err, 516)) { ok = false; break; }
          tc_fence_after();
          const uint32_t acc = (j > 0) ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            if constexpr (kPTmem)
              umma_bf16_ts(tmem + cDV, tmem + cP + ks * 8, at(bOt, ks * 2048), id_acc, acc | (ks > 0));
            else
              umma_bf16_ss(tmem + cDV, at(dPT, ks * 32), at(bOt, ks * 2048), id_acc, acc | (ks > 0));
          }
          umma_commit(&sh.pv_free);
          // X^T = KI QI^T, once the previous tile's dq_idx^T has been read
          if (!mbar_wait(&sh.x_free, (tj & 1) ^ 1, a.err, 519)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) umma_bf16_ss(tmem + cX, at(dKI, ks * 32), at(bQI, ks * 32), id_x, ks > 0);
          umma_commit(&sh.x_full);
          if (!mbar_wait(&sh.ds_ready, tj & 1, a.err, 517)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // dK += dS^T Q
            umma_bf16_ss(tmem + cDK, at(dDS, ks * 32), at(bQt, ks * 2048), id_acc, acc | (ks > 0));
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // dQ^T = K^T dS^T into cR (dP^T has been loaded)   (K = 128 keys)
            umma_bf16_ss(tR, at(dKt, ks * 2048), at(dDS, ks * 2048), id_tr, ks > 0);
          if (j + 1 < ntiles) {
            if (!issue_s(tj + 1)) { ok = false; break; }
            s_issued = true;
          }
          if (!mbar_wait(&sh.gs_ready, tj & 1, a.err, 518)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < NX / 16; ++ks)  // dk_idx += gs^T QI   (K = NX queries)
            umma_bf16_ss(tmem + cKI, at(dGS, ks * 32), at(bQI, ks * 2048), id_ki, acc | (ks > 0));
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // dq_idx^T = KI^T gs^T
            umma_bf16_ss(tmem + cX, at(dKIt, ks * 2048), at(dGS, ks * 2048), id_trx, ks > 0);
          umma_commit(&sh.ph2_full);
          umma_commit(&sh.g_empty[gb]);
        }
        umma_commit(&sh.kv_empty);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue (thread = key / d lane)
    // Warps 2-5 and 7-10: two warps per TMEM lane quarter, warpgroup hf owns
    // the tile columns (rows of the tile) [32 hf, 32 hf + 32).
    const int quarter = warp & 3;
    const int hf = warp < 6 ? 0 : 1;
    const int col0 = 32 * hf;
    const int kk = quarter * 32 + lane;  // TMEM lane: key in block c (phase 1), d (dQ^T), e (dq_idx^T)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t tj = 0;
    bool ok = true;
    // Tile whose phase-2 results (dQ^T, dq_idx^T) are still in TMEM: they are
    // read out after the next tile's stage A, so the tensor core computes that
    // tile's dP^T while this readout runs.
    bool pend = false;
    uint32_t p_tj = 0;
    int p_pos0 = 0;
    // Gather buffer whose staged partials are being stored: it goes back to
    // the producers once the stores have read it, checked one stage later so
    // the wait stays off the epilogue's path.
    int rel_gb = -1;
    auto release = [&]() {
      if (rel_gb >= 0) {
        if (lane == 0) {
          bulk_wait_read_all();
          mbar_arrive(&sh.g_empty[rel_gb]);
        }
        __syncwarp();
        rel_gb = -1;
      }
    };
    // ---- phase-2 readout: dQ^T (lane = d), dq_idx^T (lane = e < 64)
    // Partials are in tile order: a tile's 64 (query, head) rows are
    // consecutive. Each warp stages its 32 x 32 slice row-major in the tile's
    // own gather buffer (free once the phase-2 MMAs are complete) and writes
    // it with one TMA store; the buffer goes back to the producers when the
    // stores have read it.
    auto epi2 = [&]() -> bool {
      const int pgb = p_tj % kNG;
      if (!mbar_wait(&sh.ph2_full, p_tj & 1, a.err, 524)) return false;
      tc_fence_after();
      {
        uint8_t* gbuf = smem + oG + pgb * kGather;
        const int prow0 = p_pos0 * hg;  // first dQ partial row of the tile
        __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(gbuf + (hf * 4 + quarter) * 2048);
        __nv_bfloat16* stq = reinterpret_cast<__nv_bfloat16*>(gbuf + kRowTile + (hf * 2 + (quarter & 1)) * 4096);
        float dq[32];
        tmem_ld32(tmem + lane_off + cR0 + 64 * (p_tj & 1) + col0, dq);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[i * 32 + lane] = __float2bfloat16_rn(dq[i]);
        if (quarter < 2) {
          float dqi[kQ];
          tmem_ld_cols<kQ>(tmem + lane_off + cX + hf * kQ, dqi);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kQ; ++i) stq[i * 32 + lane] = __float2bfloat16_rn(dqi[i]);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh.r_free[p_tj & 1]);  // TMEM read: cR may take tile p_tj + 2's S^T,
          mbar_arrive(&sh.x_free);            // cX the next tile's X^T
          tma_store_2d(&map_dq, stg, quarter * 32, prow0 + col0);
          if (quarter < 2) tma_store_2d(&map_dqi, stq, quarter * 32, p_pos0 + hf * kQ);
          bulk_commit();
        }
      }
      rel_gb = pgb;
      return true;
    };
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 521)) { ok = false; break; }
      const int4 item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item.x < 0) break;
      int b, g, c;
      decode_list(item.x, a.n, a.G, b, g, c);
      const int key = c * 128 + kk;
      const int ntiles = (item.z + npos - 1) / npos;
      for (int j = 0; j < ntiles; ++j, ++tj) {
        const int gb = tj % kNG;
        const RowMeta& m = sh.meta[gb];
        if (!mbar_wait(&sh.g_full[gb], (tj / kNG) & 1, a.err, 522)) { ok = false; break; }
        if (!mbar_wait(&sh.s_full, tj & 1, a.err, 523)) { ok = false; break; }
        tc_fence_after();
        const uint32_t cR = cR0 + 64 * (tj & 1);
        const int4 dg0 = *reinterpret_cast<const int4*>(m.diag);
        const int4 dg1 = *reinterpret_cast<const int4*>(m.diag + 4);
        const bool masked = (dg0.x | dg0.y | dg0.z | dg0.w | dg1.x | dg1.y | dg1.z | dg1.w) != 0;
        // ---- phase-1 epilogue in three stages, each handing work to the
        // UMMA warp as soon as its operand is in shared memory
        float pv[32];
        {  // stage A: P = exp(s - LSE) (zero on masked keys and padding rows); P^T as bf16, into TMEM or an image
          float sv[32];
          tmem_ld32(tmem + lane_off + cR + col0, sv);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.s_read);  // the UMMA warp may overwrite S^T with dP^T
          const float4* l4 = reinterpret_cast<const float4*>(m.lse2 + col0);
          if (!masked) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 l = l4[i];
              pv[4 * i + 0] = fast_exp2(fmaf(sv[4 * i + 0], a.scale_log2, -l.x));
              pv[4 * i + 1] = fast_exp2(fmaf(sv[4 * i + 1], a.scale_log2, -l.y));
              pv[4 * i + 2] = fast_exp2(fmaf(sv[4 * i + 2], a.scale_log2, -l.z));
              pv[4 * i + 3] = fast_exp2(fmaf(sv[4 * i + 3], a.scale_log2, -l.w));
            }
          } else {
            const int4* e4 = reinterpret_cast<const int4*>(m.ent + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 l = l4[i];
              const int4 e = e4[i];
              pv[4 * i + 0] = key <= (e.x >> 8) ? fast_exp2(fmaf(sv[4 * i + 0], a.scale_log2, -l.x)) : 0.f;
              pv[4 * i + 1] = key <= (e.y >> 8) ? fast_exp2(fmaf(sv[4 * i + 1], a.scale_log2, -l.y)) : 0.f;
              pv[4 * i + 2] = key <= (e.z >> 8) ? fast_exp2(fmaf(sv[4 * i + 2], a.scale_log2, -l.z)) : 0.f;
              pv[4 * i + 3] = key <= (e.w >> 8) ? fast_exp2(fmaf(sv[4 * i + 3], a.scale_log2, -l.w)) : 0.f;
            }
          }
          // the previous tile's dV MMA has read P^T
          if (!mbar_wait(&sh.pv_free, (tj & 1) ^ 1, a.err, 529)) { ok = false; break; }
          tc_fence_after();
          if constexpr (kPTmem) {
            uint32_t pk[16];  // P^T row of this key, bf16 pairs (low half = even row)
#pragma unroll
            for (int z = 0; z < 16; ++z) pk[z] = pack_bf16(pv[2 * z], pv[2 * z + 1]);
            tmem_st16(tmem + lane_off + cP + 16 * hf, pk);
            tmem_wait_st();
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(smem + oPT + sw128_off(kk, 4 * hf + cc)) =
                  make_uint4(pack_bf16(pv[8 * cc + 0], pv[8 * cc + 1]), pack_bf16(pv[8 * cc + 2], pv[8 * cc + 3]),
                             pack_bf16(pv[8 * cc + 4], pv[8 * cc + 5]), pack_bf16(pv[8 * cc + 6], pv[8 * cc + 7]));
          }
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.p_ready);
        }
        if (pend) {  // the previous tile's phase-2 readout
          if (!epi2()) { ok = false; break; }
          pend = false;
        }
        {  // stage B: dS = P (dP - D) * scale
          float dp[32];
          if (!mbar_wait(&sh.dp_full, tj & 1, a.err, 527)) { ok = false; break; }
          tc_fence_after();
          tmem_ld32(tmem + lane_off + cR + col0, dp);
          tmem_wait_ld();
          const float4* d4 = reinterpret_cast<const float4*>(m.dsc + col0);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const float4 da = d4[2 * cc], db = d4[2 * cc + 1];
            const float dv[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
            float d8[8];
#pragma unroll
            for (int z = 0; z < 8; ++z) d8[z] = pv[8 * cc + z] * fmaf(dp[8 * cc + z], a.scale, -dv[z]);
            *reinterpret_cast<uint4*>(smem + oDST + sw128_off(kk, 4 * hf + cc)) =
                make_uint4(pack_bf16(d8[0], d8[1]), pack_bf16(d8[2], d8[3]), pack_bf16(d8[4], d8[5]),
                           pack_bf16(d8[6], d8[7]));
          }
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.ds_ready);
        }
        release();  // the previous tile's gather buffer
        {  // stage C: index branch; X^T and gs^T have one column per query
          float xv[kQ];
          float term[kQ];
          uint32_t gp[kQ / 2];  // this key's gs^T entries for the half's queries, bf16 pairs
#pragma unroll
          for (int z = 0; z < kQ / 2; ++z) gp[z] = 0u;
          if (!mbar_wait(&sh.x_full, tj & 1, a.err, 528)) { ok = false; break; }
          tc_fence_after();
          tmem_ld_cols<kQ>(tmem + lane_off + cX + hf * kQ, xv);
          tmem_wait_ld();
#pragma unroll
          for (int qq = 0; qq < kQ; ++qq) {
            const int r = qq * hg;  // local column of the query's first head row
            float pm = 0.f;
#pragma unroll
            for (int h = 0; h < hg; ++h) pm += pv[r + h];
            pm *= 1.f / (float)hg;
            const float lpx2 = fmaf(xv[qq], a.scale_idx_log2, -m.lpx2[col0 + r]);  // log2 p_px
            float ppx = fast_exp2(lpx2);
            if (masked && key > (m.ent[col0 + r] >> 8)) ppx = 0.f;
            const float gsv = a.kl_weight * (ppx - pm) * a.scale_idx;
            const uint32_t bits = pack_bf16(gsv, 0.f) & 0xffffu;
            gp[qq >> 1] |= (qq & 1) ? (bits << 16) : bits;
            term[qq] = pm > 0.f ? pm * (__log2f(pm) - lpx2) * kLn2 : 0.f;
          }
          // columns [hf kQ, hf kQ + kQ) of the gs^T row
          if constexpr (kQ >= 8) {
#pragma unroll
            for (int cc = 0; cc < kQ / 8; ++cc)
              *reinterpret_cast<uint4*>(smem + oGST + sw128_off(kk, hf * (kQ / 8) + cc)) =
                  make_uint4(gp[4 * cc], gp[4 * cc + 1], gp[4 * cc + 2], gp[4 * cc + 3]);
          } else {
            *reinterpret_cast<uint2*>(smem + oGST + sw128_off(kk, 0) + 8 * hf) = make_uint2(gp[0], gp[1]);
          }
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.gs_ready);
          // KL terms summed over this warp's 32 keys (a butterfly over the lanes); each key quarter
          // writes its own sums, which the merge adds in order (the same bits in every run)
          const int base = lanes_sum<kQ>(term, lane);
          if ((lane & (LanesSum<kQ>::kDup - 1)) == 0) {
#pragma unroll
            for (int i = 0; i < LanesSum<kQ>::kKeep; ++i) {
              const int e = m.ent[col0 + (base + i) * hg];
              if (e >= 0)
                a.kl_part[((((size_t)b * a.T + (e >> 8)) * a.G + g) * a.k + (e & 255)) * 4 + quarter] = term[i];
            }
          }
        }
        pend = true;  // this tile's dQ^T / dq_idx^T are read out after the next tile's stage A
        p_tj = tj;
        p_pos0 = item.w + j * npos;
      }
      if (!ok) break;
      if (pend) {
        if (!epi2()) { ok = false; break; }
        pend = false;
      }
      release();
      // ---- list end: dV, dK, dk_idx accumulators (lane = key); warpgroup hf
      // takes dV/dK columns [64 hf, 64 hf + 64) and dk_idx columns [32 hf, 32 hf + 32)
      {
        const size_t orow = ((size_t)b * a.T + key) * a.G + g;
        float v[32];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int d0 = 64 * hf + 32 * q;
          tmem_ld32(tmem + lane_off + cDV + d0, v);
          tmem_wait_ld();
          float4* dst = reinterpret_cast<float4*>(a.dV + orow * 128 + d0);
#pragma unroll
          for (int z = 0; z < 8; ++z) dst[z] = make_float4(v[4 * z], v[4 * z + 1], v[4 * z + 2], v[4 * z + 3]);
          tmem_ld32(tmem + lane_off + cDK + d0, v);
          tmem_wait_ld();
          dst = reinterpret_cast<float4*>(a.dK + orow * 128 + d0);
#pragma unroll
          for (int z = 0; z < 8; ++z) dst[z] = make_float4(v[4 * z], v[4 * z + 1], v[4 * z + 2], v[4 * z + 3]);
        }
        float* dki = a.dki_part + (((size_t)b * a.G + g) * a.T + key) * 64 + 32 * hf;
        tmem_ld32(tmem + lane_off + cKI + 32 * hf, v);
        tmem_wait_ld();
#pragma unroll
        for (int z = 0; z < 8; ++z)
          reinterpret_cast<float4*>(dki)[z] = make_float4(v[4 * z], v[4 * z + 1], v[4 * z + 2], v[4 * z + 3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.acc_free);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (!ok) *abort_flag = 1;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// One warp per (b, t, g): dQ rows of its heads, dq_idx and KL from the slots.
// Loads n consecutive bf16 values (n = 4 or a multiple of 8) as fp32.
template <int N>
__device__ __forceinline__ void load_bf16_row(const __nv_bfloat16* src, float (&out)[N]) {
  if constexpr (N % 8 == 0) {
#pragma unroll
    for (int q = 0; q < N / 8; ++q) {
      const uint4 raw = reinterpret_cast<const uint4*>(src)[q];
      const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const float2 f = __bfloat1622float2(v[z]);
        out[q * 8 + 2 * z] = f.x;
        out[q * 8 + 2 * z + 1] = f.y;
      }
    }
  } else {
    static_assert(N == 4, "4 or a multiple of 8 values");
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const float2 f0 = __bfloat1622float2(v[0]), f1 = __bfloat1622float2(v[1]);
    out[0] = f0.x;
    out[1] = f0.y;
    out[2] = f1.x;
    out[3] = f1.y;
  }
}

// The partials of (b, g, t, slot) sit at padded entry rev[(b*G + g)*T + t][slot]
// (dQ: HG contiguous rows entry*HG + h; dq_idx: row entry); KL partials at
// (b, t, g, slot). One warp per (b, t, g); every lane owns 4 * HG consecutive
// dQ values and 2 dq_idx values. The warp of group 0 also writes dk_idx[b, t]
// as the sum over groups of the backward kernel's per-group rows.
template <int HG, int NSL>  // NSL slots per lane: k <= 32 NSL
__global__ void bwd_merge_kernel(const int32_t* __restrict__ block_idx, const int32_t* __restrict__ rev,
                                 const __nv_bfloat16* __restrict__ dq_part, const __nv_bfloat16* __restrict__ dqi_part,
                                 const float* __restrict__ kl_part, const float* __restrict__ dki_part,
                                 float* __restrict__ dQ, float* __restrict__ dq_idx, float* __restrict__ KL,
                                 float* __restrict__ dk_idx, int B, int T, int Hq, int G, int k,
                                 long long max_padded) {
  constexpr int kPer = 4 * HG;
  const long long rows = (long long)B * T * G;
  const int lane = threadIdx.x & 31;
  for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; w < rows;
       w += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int g = (int)(w % G);
    const long long bt = w / G;
    const int t = (int)(bt % T), b = (int)(bt / T);
    const size_t sel_row = (((size_t)b * G + g) * T + t) * k;
    int rv_own[NSL];
    float kl_own = 0.f;
#pragma unroll
    for (int u = 0; u < NSL; ++u) {
      const int sidx = lane + 32 * u;
      int r = -1;
      if (sidx < k && block_idx[sel_row + sidx] >= 0) {
        r = rev[sel_row + sidx];
        if (r >= 0 && (long long)r >= max_padded) r = -1;
      }
      rv_own[u] = r;
      if (r >= 0) {  // the slot's four key-quarter sums, in order
        const float4 q4 = reinterpret_cast<const float4*>(kl_part)[(size_t)w * k + sidx];
        kl_own += ((q4.x + q4.y) + q4.z) + q4.w;
      }
    }
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int u = 0; u < NSL; ++u) {
      for (int src = 0; src < 32 && 32 * u + src < k; ++src) {
        const int r = __shfl_sync(0xffffffffu, rv_own[u], src);
        if (r < 0) continue;
        float v[kPer];
        load_bf16_row<kPer>(dq_part + (size_t)r * HG * 128 + lane * kPer, v);
#pragma unroll
        for (int i = 0; i < kPer; ++i) acc[i] += v[i];
        const float2 vi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dqi_part + (size_t)r * 64 + lane * 2));
        a0 += vi.x;
        a1 += vi.y;
      }
    }
    float4* dst = reinterpret_cast<float4*>(dQ + (((size_t)b * T + t) * Hq + g * HG) * 128) + lane * (kPer / 4);
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    *reinterpret_cast<float2*>(dq_idx + (size_t)w * 64 + lane * 2) = make_float2(a0, a1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kl_own += __shfl_xor_sync(0xffffffffu, kl_own, o);
    if (lane == 0) KL[((size_t)b * G + g) * T + t] = kl_own;
    if (g == 0) {  // dk_idx[b,t,:] = sum_g dki_part[b,g,t,:], groups in ascending order
      float s0 = 0.f, s1 = 0.f;
      for (int gg = 0; gg < G; ++gg) {
        const float2 v = *reinterpret_cast<const float2*>(dki_part + (((size_t)b * G + gg) * T + t) * 64 + lane * 2);
        s0 += v.x;
        s1 += v.y;
      }
      *reinterpret_cast<float2*>(dk_idx + bt * 64 + lane * 2) = make_float2(s0, s1);
    }
  }
}

// Two slots per lane up to k = 64, four up to k = 128.
template <int HG>
void bwd_merge(const Prob& p, const int32_t* block_idx, const int32_t* rev, const BwdArgs& ba, float* dQ,
               float* dq_idx, float* KL, float* dk_idx, long long max_padded, int grid, cudaStream_t st) {
  if (p.k <= 64)
    bwd_merge_kernel<HG, 2><<<grid, 256, 0, st>>>(block_idx, rev, ba.dq_part, ba.dqi_part, ba.kl_part, ba.dki_part,
                                                   dQ, dq_idx, KL, dk_idx, p.B, p.T, p.Hq, p.G, p.k, max_padded);
  else
    bwd_merge_kernel<HG, 4><<<grid, 256, 0, st>>>(block_idx, rev, ba.dq_part, ba.dqi_part, ba.kl_part, ba.dki_part,
                                                   dQ, dq_idx, KL, dk_idx, p.B, p.T, p.Hq, p.G, p.k, max_padded);
}

}  // namespace

// Tensor maps of the backward's inputs: K, V (box 64 d x 1 x 128 keys), k_idx
// (64 x 128), and the gathered rows of one query: Q, dO (64 d x hg heads x 1
// token), q_idx (64 x 1).
struct BwdMaps {
  CUtensorMap mk, mv, mki, mq, mdo, mqi;
};

static bool make_bwd_maps(const Prob& p, const void* Q, const void* K, const void* V, const void* dO,
                          const void* q_idx, const void* k_idx, BwdMaps* m) {
  {
    const uint64_t dims[2] = {64, (uint64_t)p.BT()};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap(&m->mki, const_cast<void*>(k_idx), 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  {
    const uint64_t dims[3] = {128, (uint64_t)p.G, (uint64_t)p.BT()};
    const uint64_t strides[2] = {256, (uint64_t)p.G * 256};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap(&m->mk, const_cast<void*>(K), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&m->mv, const_cast<void*>(V), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  {
    const uint64_t dims[3] = {128, (uint64_t)p.Hq, (uint64_t)p.BT()};
    const uint64_t strides[2] = {256, (uint64_t)p.Hq * 256};
    const uint32_t box[3] = {64, (uint32_t)p.hg, 1};
    if (!encode_tmap(&m->mq, const_cast<void*>(Q), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&m->mdo, const_cast<void*>(dO), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    const uint64_t dims2[2] = {64, (uint64_t)p.BT() * p.G};
    const uint64_t strides2[1] = {128};
    const uint32_t box2[2] = {64, 1};
    if (!encode_tmap(&m->mqi, const_cast<void*>(q_idx), 2, dims2, strides2, box2, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  return true;
}

cudaError_t launch_bwd(const Prob& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                       const float* LSE, const void* q_idx, const void* k_idx, const int32_t* block_idx,
                       float kl_weight, void* dQ, void* dK, void* dV, void* dq_idx, void* dk_idx, float* KL,
                       uint8_t* ws, const WsLayout& L, cudaStream_t st, bool mapped) {
  const int npos = bwd_tile_queries(p);  // queries per backward tile (64 (query, head) rows)
  cudaError_t e;
  if (!mapped && (e = build_block_map(p, block_idx, ws, L, npos, (1 << 30) / npos, st)) != cudaSuccess) return e;
  int* err = reinterpret_cast<int*>(ws + L.err);
  int* counters = reinterpret_cast<int*>(ws + L.counters);
  float* drow = reinterpret_cast<float*>(ws + L.drow);
  float* px_part = reinterpret_cast<float*>(ws + L.px_part);
  float* lse_px = reinterpret_cast<float*>(ws + L.lse_px);
  const long long hrows = (long long)p.B * p.T * p.Hq;
  const long long grows = (long long)p.B * p.T * p.G;
  const int sms = num_sms();
  drow_kernel<<<(int)std::min<long long>((hrows * 32 + 255) / 256, 16LL * sms), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), drow, hrows);
  if ((e = cudaMemsetAsync(counters + 2, 0, 2 * sizeof(int), st)) != cudaSuccess) return e;

  BwdMaps mp;
  if (!make_bwd_maps(p, Q, K, V, dO, q_idx, k_idx, &mp)) return cudaErrorInvalidValue;
  // 64-row tiles (1 or 2 heads per group) store 32 rows per epilogue warp,
  // 128-row tiles (4 or 8) 64 rows
  const bool wide = p.hg >= 4;
  const uint32_t rows_per_warp = wide ? 64 : 32;
  CUtensorMap mdq, mdqi;
  {
    const uint64_t dims[2] = {128, (uint64_t)L.max_padded * p.hg};
    const uint64_t strides[1] = {256};
    const uint32_t box[2] = {32, rows_per_warp};  // 32 d x the warp's rows
    if (!encode_tmap(&mdq, ws + L.dq_part, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    const uint64_t dims2[2] = {64, (uint64_t)L.max_padded};
    const uint64_t strides2[1] = {128};
    const uint32_t box2[2] = {32, rows_per_warp / (uint32_t)p.hg};  // 32 e x the queries of those rows
    if (!encode_tmap(&mdqi, ws + L.dqi_part, 2, dims2, strides2, box2, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  static bool attr[kMaxDevices] = {};  // kernel attributes are per device context
  const int dslot = device_slot();
  if (!attr[dslot]) {
    if ((e = cudaFuncSetAttribute(px_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPxSmem)) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(bwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  BwdLayout<1>::kSmem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  BwdLayout<2>::kSmem)) != cudaSuccess)
      return e;
    attr[dslot] = true;
  }
  PxArgs pa;
  pa.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  pa.entries = reinterpret_cast<const int32_t*>(ws + L.entries);
  // a shared map keeps the backward's items (whole lists) in items2 / n_items[1]
  pa.items = reinterpret_cast<const int4*>(ws + (mapped ? L.items2 : L.items));
  pa.n_items = reinterpret_cast<const int*>(ws + L.n_items) + (mapped ? 1 : 0);
  pa.counter = counters + 2;
  pa.err = err;
  pa.px_part = px_part;
  pa.B = p.B;
  pa.T = p.T;
  pa.G = p.G;
  pa.n = p.n;
  pa.k = p.k;
  pa.scale_log2 = p.scale_idx * kLog2e;
  px_stats_kernel<<<sms, kPxThreads, kPxSmem, st>>>(pa, mp.mki);
  px_merge_kernel<<<(int)std::min<long long>((grows + 255) / 256, 16LL * sms), 256, 0, st>>>(
      block_idx, px_part, lse_px, p.B, p.T, p.G, p.k);

  BwdArgs ba;
  ba.Q = static_cast<const __nv_bfloat16*>(Q);
  ba.dO = static_cast<const __nv_bfloat16*>(dO);
  ba.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  ba.LSE = LSE;
  ba.drow = drow;
  ba.lse_px = lse_px;
  ba.entries = pa.entries;
  ba.items = pa.items;
  ba.n_items = pa.n_items;
  ba.counter = counters + 3;
  ba.err = err;
  ba.dK = static_cast<float*>(dK);
  ba.dV = static_cast<float*>(dV);
  ba.dq_part = reinterpret_cast<__nv_bfloat16*>(ws + L.dq_part);
  ba.dqi_part = reinterpret_cast<__nv_bfloat16*>(ws + L.dqi_part);
  ba.kl_part = reinterpret_cast<float*>(ws + L.kl_part);
  ba.dki_part = reinterpret_cast<float*>(ws + L.dki_part);
  ba.B = p.B;
  ba.T = p.T;
  ba.Hq = p.Hq;
  ba.G = p.G;
  ba.hg = p.hg;
  ba.n = p.n;
  ba.k = p.k;
  ba.scale_log2 = p.scale * kLog2e;
  ba.scale = p.scale;
  ba.scale_idx_log2 = p.scale_idx * kLog2e;
  ba.scale_idx = p.scale_idx;
  ba.kl_weight = kl_weight;
  timing_begin(MSA_TIME_BWD, st);
  if (wide) {
    if ((e = launch_bwd_wide(ba, mp.mk, mp.mv, mp.mki, mdq, mdqi, mp.mq, mp.mdo, mp.mqi, st)) != cudaSuccess)
      return e;
  } else if (p.hg == 1) {
    bwd_kernel<1><<<sms, kBwdThreads, BwdLayout<1>::kSmem, st>>>(ba, mp.mk, mp.mv, mp.mki, mdq, mdqi, mp.mq, mp.mdo,
                                                                 mp.mqi);
  } else {
    bwd_kernel<2><<<sms, kBwdThreads, BwdLayout<2>::kSmem, st>>>(ba, mp.mk, mp.mv, mp.mki, mdq, mdqi, mp.mq, mp.mdo,
                                                                 mp.mqi);
  }
  timing_end(MSA_TIME_BWD, st);
  count_launches(5);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    const int grid = (int)std::min<long long>((grows * 32 + 255) / 256, 16LL * sms);
    const int32_t* rev = reinterpret_cast<const int32_t*>(ws + L.rev);
    float* dQf = static_cast<float*>(dQ);
    float* dqif = static_cast<float*>(dq_idx);
    float* dkif = static_cast<float*>(dk_idx);
    switch (p.hg) {
      case 1: bwd_merge<1>(p, block_idx, rev, ba, dQf, dqif, KL, dkif, L.max_padded, grid, st); break;
      case 2: bwd_merge<2>(p, block_idx, rev, ba, dQf, dqif, KL, dkif, L.max_padded, grid, st); break;
      case 4: bwd_merge<4>(p, block_idx, rev, ba, dQf, dqif, KL, dkif, L.max_padded, grid, st); break;
      default: bwd_merge<8>(p, block_idx, rev, ba, dQf, dqif, KL, dkif, L.max_padded, grid, st); break;
    }
  }
  return cudaGetLastError();
}

// Full attention (the indexer warmup at any T): D, the index LSE over every
// visible token, then the 128-row-tile backward over every (block, query >=
// block) pair, adding into the zeroed outputs.
cudaError_t launch_bwd_dense(const Prob& p, const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, const void* q_idx, const void* k_idx, float kl_weight,
                             float* dQ, float* dK, float* dV, float* dq_idx, float* dk_idx, float* KL, uint8_t* ws,
                             const WsLayout& L, const DenseSchedule& ds, cudaStream_t st) {
  cudaError_t e;
  const size_t rows = (size_t)p.BT();
  const struct {
    void* ptr;
    size_t bytes;
  } zero[] = {{dQ, rows * p.Hq * p.d * 4}, {dK, rows * p.G * p.d * 4}, {dV, rows * p.G * p.d * 4},
              {dq_idx, rows * p.G * p.E * 4}, {dk_idx, rows * p.E * 4}, {KL, rows * p.G * 4}};
  for (const auto& z : zero)
    if ((e = cudaMemsetAsync(z.ptr, 0, z.bytes, st)) != cudaSuccess) return e;
  int* err = reinterpret_cast<int*>(ws + L.err);
  int* counters = reinterpret_cast<int*>(ws + L.counters);
  float* drow = reinterpret_cast<float*>(ws + L.drow);
  float* lse_px = reinterpret_cast<float*>(ws + L.lse_px);
  const long long hrows = (long long)p.B * p.T * p.Hq;
  const int sms = num_sms();
  drow_kernel<<<(int)std::min<long long>((hrows * 32 + 255) / 256, 16LL * sms), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), drow, hrows);
  count_launches(1);
  if ((e = launch_dense_px(p, q_idx, k_idx, lse_px, ws, L, st)) != cudaSuccess) return e;
  BwdMaps mp;
  if (!make_bwd_maps(p, Q, K, V, dO, q_idx, k_idx, &mp)) return cudaErrorInvalidValue;
  {
    // a tile's queries are consecutive tokens: whole-tile boxes (128 / hg tokens) for Q, dO and q_idx
    const uint32_t npos = 128 / p.hg;
    const uint64_t dims[3] = {128, (uint64_t)p.Hq, (uint64_t)p.BT()};
    const uint64_t strides[2] = {256, (uint64_t)p.Hq * 256};
    const uint32_t box[3] = {64, (uint32_t)p.hg, npos};
    if (!encode_tmap(&mp.mq, const_cast<void*>(Q), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&mp.mdo, const_cast<void*>(dO), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const uint64_t dims2[3] = {64, (uint64_t)p.G, (uint64_t)p.BT()};
    const uint64_t strides2[2] = {128, (uint64_t)p.G * 128};
    const uint32_t box2[3] = {64, 1, npos};
    if (!encode_tmap(&mp.mqi, const_cast<void*>(q_idx), 3, dims2, strides2, box2, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  CUtensorMap mdq;
  {
    // the caller's fp32 dQ, added into per half tile: 32 d x hg heads x (64 / hg) queries
    const uint64_t dims[3] = {128, (uint64_t)p.Hq, (uint64_t)p.BT()};
    const uint64_t strides[2] = {512, (uint64_t)p.Hq * 512};
    const uint32_t box[3] = {32, (uint32_t)p.hg, (uint32_t)(64 / p.hg)};
    if (!encode_tmap(&mdq, dQ, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return cudaErrorInvalidValue;
  }
  BwdArgs ba = {};
  ba.Q = static_cast<const __nv_bfloat16*>(Q);
  ba.dO = static_cast<const __nv_bfloat16*>(dO);
  ba.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  ba.LSE = LSE;
  ba.drow = drow;
  ba.lse_px = lse_px;
  ba.counter = counters + 6;
  ba.err = err;
  ba.dK = dK;
  ba.dV = dV;
  ba.dq_idx = dq_idx;
  ba.dk_idx = dk_idx;
  ba.KL = KL;
  ba.dense_seg = ds.seg;
  ba.dense_per_b = ds.per_b;
  ba.dense_items = ds.items;
  ba.B = p.B;
  ba.T = p.T;
  ba.Hq = p.Hq;
  ba.G = p.G;
  ba.hg = p.hg;
  ba.n = p.n;
  ba.k = p.k;
  ba.scale_log2 = p.scale * kLog2e;
  ba.scale = p.scale;
  ba.scale_idx_log2 = p.scale_idx * kLog2e;
  ba.scale_idx = p.scale_idx;
  ba.kl_weight = kl_weight;
  if ((e = cudaMemsetAsync(ba.counter, 0, sizeof(int), st)) != cudaSuccess) return e;
  timing_begin(MSA_TIME_DENSE_BWD, st);
  e = launch_bwd_wide_dense(ba, mp.mk, mp.mv, mp.mki, mdq, mp.mq, mp.mdo, mp.mqi, st);
  timing_end(MSA_TIME_DENSE_BWD, st);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
