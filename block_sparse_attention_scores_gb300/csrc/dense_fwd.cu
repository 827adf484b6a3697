// Full causal attention for the indexer warmup: the main-branch forward over
// every visible token, and the index branch's log-sum-exp over the same set.
//
// itinai.ru "How to solve the memory problem with MiniMax Sparse Attention",
// "Training sparse attention": the first iterations attend to every visible
// token, so that the indexer learns from the full attention before it routes.
// dothoosh.com "how FlashAttention cuts GPU memory traffic", "Online-softmax
// trick": a running maximum and sum per row, with the accumulated output
// rescaled when the maximum moves; "Exactness vs approximation": the result
// is the exact softmax attention.
//
// GB300 design (query-outer, nothing per (query, block) leaves the SM).
// dense_fwd_kernel: a work item is one 128-query block qb of one (b, g) and
// two heads of the group, which share every K/V block. Per KV block c <= qb:
//   S_t = Q_t K_c^T (tcgen05, TMEM)      for both heads t = 0, 1
//   P_t = exp2(S_t * scale * log2 e - m) (bf16, written back over S_t's columns)
//   O_t += P_t V_c                       (tcgen05 with P_t from TMEM, O_t in TMEM)
// The running maximum m of a row moves only when a block raises it by more
// than 2^8: until then P <= 256 and O_t, l keep their scale, so the O
// rescale (a TMEM load and store of the row) is rare. The two heads ping-pong:
// the tensor core computes one head's PV and next S while the softmax warps
// of the other head work. O = O_t / l (bf16) and LSE = (m + log2 l) ln 2 leave
// once per item.
//
// dense_px_kernel: the index branch's LSE over every visible token, per
// (b, g, query): X = q_idx k_idx_c^T per 128-query block and KV block
// (tcgen05), reduced by the epilogue with the same lazy running maximum.
#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Log2 headroom of the lazy rescale: P = exp2(s - m) stays <= 2^kHeadroom.
constexpr float kHeadroom = 8.f;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ============================================================================ forward
constexpr int kFThreads = 320;  // warp 0 TMA, warp 1 UMMA + TMEM, warps 2-5 and 6-9 softmax of heads 0 and 1
constexpr int kTile = 32768;    // 128 rows x 128 bf16, two 64-column SW128 chunks
constexpr int kChunk = 16384;
constexpr int kStages = 2;      // K/V ring
constexpr int oQ = 0, oK = 2 * kTile, oV = oK + kStages * kTile;
constexpr int kFSmem = oV + kStages * kTile + 1024;  // + 1024-byte alignment slack

struct DenseFwdArgs {
  int B, T, Hq, G, hg, n;
  int num_items;
  int* counter;
  int* err;
  __nv_bfloat16* O;
  float* LSE;
  float scale_log2;
};

struct DenseFwdShared {
  uint64_t it_full[2], it_empty[2];
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
  int item[2];
  uint32_t tmem_base;
  int abort;
};

// Items: 128-query block qb (largest first, the longest rows), then (b, g, head pair).
__device__ __forceinline__ void decode_fwd_item(int id, const DenseFwdArgs& a, int& b, int& g, int& qb, int& h0) {
  const int pairs = a.hg / 2;
  const int per_qb = a.B * a.G * pairs;
  qb = a.n - 1 - id / per_qb;
  int r = id % per_qb;
  const int pr = r % pairs;
  r /= pairs;
  g = r % a.G;
  b = r / a.G;
  h0 = g * a.hg + 2 * pr;
}

__global__ void __launch_bounds__(kFThreads, 1)
    dense_fwd_kernel(DenseFwdArgs a, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DenseFwdShared sh;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], 1 + 8);  // UMMA thread, softmax warps
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], 4);
      mbar_init(&sh.o_full[i], 1);
      mbar_init(&sh.o_free[i], 4);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;  // S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512)
  volatile int* abort_flag = &sh.abort;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      uint32_t kc = 0;
      for (int it = 0;; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 1001)) { *abort_flag = 1; break; }
        int item = atomicAdd(a.counter, 1);
        if (item >= a.num_items || *abort_flag) item = -1;
        sh.item[s] = item;
        mbar_arrive(&sh.it_full[s]);
        if (item < 0) break;
        int b, g, qb, h0;
        decode_fwd_item(item, a, b, g, qb, h0);
        const int row0 = b * a.T + qb * 128;
        if (!mbar_wait(&sh.q_empty, (it & 1) ^ 1, a.err, 1002)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&sh.q_full, 2 * kTile);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          tma_load_3d(smem + oQ + t * kTile, &map_q, &sh.q_full, 0, h0 + t, row0);
          tma_load_3d(smem + oQ + t * kTile + kChunk, &map_q, &sh.q_full, 64, h0 + t, row0);
        }
        bool ok = true;
        for (int c = 0; c <= qb; ++c, ++kc) {
          const int st = kc % kStages;
          const uint32_t par = ((kc / kStages) & 1) ^ 1;
          const int krow = b * a.T + c * 128;
          if (!mbar_wait(&sh.k_empty[st], par, a.err, 1003)) { ok = false; break; }
          mbar_arrive_expect_tx(&sh.k_full[st], kTile);
          tma_load_3d(smem + oK + st * kTile, &map_k, &sh.k_full[st], 0, g, krow);
          tma_load_3d(smem + oK + st * kTile + kChunk, &map_k, &sh.k_full[st], 64, g, krow);
          if (!mbar_wait(&sh.v_empty[st], par, a.err, 1004)) { ok = false; break; }
          mbar_arrive_expect_tx(&sh.v_full[st], kTile);
          tma_load_3d(smem + oV + st * kTile, &map_v, &sh.v_full[st], 0, g, krow);
          tma_load_3d(smem + oV + st * kTile + kChunk, &map_v, &sh.v_full[st], 64, g, krow);
        }
        if (!ok) { *abort_flag = 1; break; }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = make_idesc_bf16(128, 128, false, false);  // Q, K both K-major
      constexpr uint32_t id_o = make_idesc_bf16(128, 128, false, true);   // P from TMEM, V MN-major
      const uint32_t q0 = smem_u32(smem + oQ);
      uint32_t kc = 0;
      bool ok = true;
      // S_t = Q_t K^T for the block in stage st
      auto issue_s = [&](int t, int st) {
        const uint32_t qa = q0 + t * kTile, ka = smem_u32(smem + oK + st * kTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * kChunk + (ks & 3) * 32;
          umma_bf16_ss(tmem + t * 128, make_sdesc(qa + off, 16, 1024, kSw128), make_sdesc(ka + off, 16, 1024, kSw128),
                       id_s, ks > 0);
        }
        umma_commit(&sh.s_full[t]);
      };
      // O_t (+)= P_t V for the block in stage st, P_t packed in S_t's first 64 columns
      auto issue_o = [&](int t, int st, bool acc) {
        const uint32_t va = smem_u32(smem + oV + st * kTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16_ts(tmem + 256 + t * 128, tmem + t * 128 + ks * 8, make_sdesc(va + ks * 2048, kChunk, 1024, kSw128),
                       id_o, acc || ks > 0);
      };
      for (int it = 0; ok; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 1011)) { ok = false; break; }
        const int item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item < 0) break;
        int b, g, qb, h0;
        decode_fwd_item(item, a, b, g, qb, h0);
        if (!mbar_wait(&sh.q_full, it & 1, a.err, 1012)) { ok = false; break; }
        {
          const int st = kc % kStages;
          if (!mbar_wait(&sh.k_full[st], (kc / kStages) & 1, a.err, 1013)) { ok = false; break; }
          tc_fence_after();
          issue_s(0, st);
          issue_s(1, st);
          umma_commit(&sh.k_empty[st]);
          if (qb == 0) umma_commit(&sh.q_empty);
        }
        for (int c = 0; c <= qb; ++c, ++kc) {
          const int st = kc % kStages, st1 = (kc + 1) % kStages;
          const uint32_t par = (kc / kStages) & 1, par1 = ((kc + 1) / kStages) & 1;
          const bool last = c == qb;
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            // P_t of this block written (and O_t rescaled if its row maximum moved)
            if (!mbar_wait(&sh.p_full[t], kc & 1, a.err, 1014 + t)) { ok = false; break; }
            if (c == 0 && !mbar_wait(&sh.o_free[t], (it & 1) ^ 1, a.err, 1016 + t)) { ok = false; break; }
            if (t == 0 && !mbar_wait(&sh.v_full[st], par, a.err, 1018)) { ok = false; break; }
            tc_fence_after();
            issue_o(t, st, c > 0);
            if (t == 1) umma_commit(&sh.v_empty[st]);
            if (!last) {
              // the next block's S_t: after this PV_t in issue order, so it overwrites P_t only once read
              if (t == 0 && !mbar_wait(&sh.k_full[st1], par1, a.err, 1019)) { ok = false; break; }
              tc_fence_after();
              issue_s(t, st1);
              if (t == 1) {
                umma_commit(&sh.k_empty[st1]);
                if (c + 1 == qb) umma_commit(&sh.q_empty);
              }
            } else {
              umma_commit(&sh.o_full[t]);
            }
          }
          if (!ok) break;
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ---------------------------------------------------------------- softmax (thread = query row)
    const int t = (warp - 2) >> 2;  // head of the pair
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_col = t * 128, o_col = 256 + t * 128;
    uint32_t kc = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 1021)) { ok = false; break; }
      const int item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item < 0) break;
      int b, g, qb, h0;
      decode_fwd_item(item, a, b, g, qb, h0);
      float m_run = -INFINITY, l_run = 0.f;
      for (int c = 0; c <= qb; ++c, ++kc) {
        if (!mbar_wait(&sh.s_full[t], kc & 1, a.err, 1022 + t)) { ok = false; break; }
        tc_fence_after();
        float sv[128], mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32_max(tmem + lane_off + s_col + q * 32, *reinterpret_cast<float(*)[32]>(sv + 32 * q), mq[q]);
        tmem_wait_ld();
        float m_raw = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));  // the loads' own maximum
        if (c == qb) {  // the query's own block: keys after it are masked, and the maximum is taken again
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int j = 0; j < 128; ++j) {
            if (j > row) sv[j] = -INFINITY;
            m4[j & 3] = fmaxf(m4[j & 3], sv[j]);
          }
          m_raw = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        const float m_blk = m_raw * a.scale_log2;
        const bool need = m_blk > m_run + kHeadroom;
        if (__any_sync(0xffffffffu, need)) {
          // rescale l and (past the first block) O_t to the new maximum; PV_t of the previous block is done
          // (it was issued before this block's S_t)
          const float alpha = need ? fast_exp2(m_run - m_blk) : 1.f;
          if (need) m_run = m_blk;
          l_run *= alpha;
          if (c > 0) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
              float o[32];
              tmem_ld32(tmem + lane_off + o_col + q * 32, o);
              tmem_wait_ld();
              uint32_t ob[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) ob[i] = __float_as_uint(o[i] * alpha);
              tmem_st32(tmem + lane_off + o_col + q * 32, ob);
            }
            tmem_wait_st();
          }
        }
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int z = 0; z < 32; ++z) {
            const float p0 = fast_exp2(fmaf(sv[64 * h + 2 * z], a.scale_log2, -m_run));
            const float p1 = fast_exp2(fmaf(sv[64 * h + 2 * z + 1], a.scale_log2, -m_run));
            l4[(2 * z) & 3] += p0;
            l4[(2 * z + 1) & 3] += p1;
            pk[z] = pack_bf16(p0, p1);
          }
          tmem_st32(tmem + lane_off + s_col + 32 * h, pk);
        }
        tmem_wait_st();
        l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_full[t]);
      }
      if (!ok) break;
      // ---- item end: O = O_t / l (bf16) and the LSE of the row
      if (!mbar_wait(&sh.o_full[t], it & 1, a.err, 1024 + t)) { ok = false; break; }
      tc_fence_after();
      const int h = h0 + t;
      const size_t orow = ((size_t)b * a.T + qb * 128 + row) * a.Hq + h;
      const float inv = 1.f / l_run;
      uint4* dst = reinterpret_cast<uint4*>(a.O + orow * 128);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[32];
        tmem_ld32(tmem + lane_off + o_col + q * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int z = 0; z < 4; ++z)
          dst[4 * q + z] = make_uint4(pack_bf16(o[8 * z] * inv, o[8 * z + 1] * inv),
                                      pack_bf16(o[8 * z + 2] * inv, o[8 * z + 3] * inv),
                                      pack_bf16(o[8 * z + 4] * inv, o[8 * z + 5] * inv),
                                      pack_bf16(o[8 * z + 6] * inv, o[8 * z + 7] * inv));
      }
      a.LSE[orow] = (m_run + __log2f(l_run)) * kLn2;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.o_free[t]);
    }
    if (!ok) *abort_flag = 1;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ============================================================================ index LSE
constexpr int kPThreads = 192;  // warp 0 TMA, warp 1 UMMA + TMEM, warps 2-5 epilogue
constexpr int kPStages = 4;
constexpr int kPTile = 16384;    // 128 rows x 64 bf16
constexpr int kPSmem = (2 + kPStages) * kPTile + 1024;

struct DensePxArgs {
  int B, T, G, n;
  int* counter;
  int* err;
  float* lse_px;  // [B,T,G]
  float scale_log2;
};

struct DensePxShared {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kPStages], k_empty[kPStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t it_full[2], it_empty[2];
  int item[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void decode_px_item(int item, int B, int G, int n, int& b, int& g, int& qb) {
  const int BG = B * G;
  qb = n - 1 - item / BG;
  const int bg = item % BG;
  b = bg / G;
  g = bg % G;
}

__global__ void __launch_bounds__(kPThreads, 2)
    dense_px_kernel(DensePxArgs a, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + 2 * kPTile;
  __shared__ DensePxShared sh;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int num_items = a.B * a.G * a.n;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.q_full[i], 1);
      mbar_init(&sh.q_empty[i], 1);
      mbar_init(&sh.acc_full[i], 1);
      mbar_init(&sh.acc_empty[i], 4);
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], 5);
    }
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
    }
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

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      uint32_t kc = 0;
      for (int it = 0;; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 1101)) { *abort_flag = 1; break; }
        int item = atomicAdd(a.counter, 1);
        if (item >= num_items || *abort_flag) item = -1;
        sh.item[s] = item;
        mbar_arrive(&sh.it_full[s]);
        if (item < 0) break;
        int b, g, qb;
        decode_px_item(item, a.B, a.G, a.n, b, g, qb);
        if (!mbar_wait(&sh.q_empty[s], ph ^ 1, a.err, 1102)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&sh.q_full[s], kPTile);
        tma_load_3d(sQ + s * kPTile, &map_q, &sh.q_full[s], 0, g, b * a.T + qb * 128);
        bool ok = true;
        for (int c = 0; c <= qb; ++c, ++kc) {
          const int st = kc % kPStages;
          if (!mbar_wait(&sh.k_empty[st], ((kc / kPStages) & 1) ^ 1, a.err, 1103)) { ok = false; break; }
          mbar_arrive_expect_tx(&sh.k_full[st], kPTile);
          tma_load_2d(sK + st * kPTile, &map_k, &sh.k_full[st], 0, b * a.T + c * 128);
        }
        if (!ok) { *abort_flag = 1; break; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(128, 128, false, false);
      uint32_t kc = 0, ac = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 1111)) { ok = false; break; }
        const int item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item < 0) break;
        int b, g, qb;
        decode_px_item(item, a.B, a.G, a.n, b, g, qb);
        if (!mbar_wait(&sh.q_full[s], ph, a.err, 1112)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qaddr = smem_u32(sQ + s * kPTile);
        for (int c = 0; c <= qb; ++c, ++kc, ++ac) {
          const int st = kc % kPStages;
          const int ab = ac & 1;
          if (!mbar_wait(&sh.k_full[st], (kc / kPStages) & 1, a.err, 1113)) { ok = false; break; }
          if (!mbar_wait(&sh.acc_empty[ab], ((ac >> 1) & 1) ^ 1, a.err, 1114)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = smem_u32(sK + st * kPTile);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16_ss(tmem + ab * 128, make_sdesc(qaddr + ks * 32, 16, 1024, kSw128),
                         make_sdesc(kaddr + ks * 32, 16, 1024, kSw128), idesc, ks > 0);
          umma_commit(&sh.k_empty[st]);
          umma_commit(&sh.acc_full[ab]);
        }
        umma_commit(&sh.q_empty[s]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ---------------------------------------------------------------- epilogue (thread = query)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t ac = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 1121)) { ok = false; break; }
      const int item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item < 0) break;
      int b, g, qb;
      decode_px_item(item, a.B, a.G, a.n, b, g, qb);
      float m_run = -INFINITY, l_run = 0.f;
      for (int c = 0; c <= qb; ++c, ++ac) {
        const int ab = ac & 1;
        if (!mbar_wait(&sh.acc_full[ab], (ac >> 1) & 1, a.err, 1122)) { ok = false; break; }
        tc_fence_after();
        float xv[128], mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32_max(lane_addr + ab * 128 + q * 32, *reinterpret_cast<float(*)[32]>(xv + 32 * q), mq[q]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.acc_empty[ab]);
        float m_raw = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));  // the loads' own maximum
        if (c == qb) {  // the own block: keys after the query are masked, the maximum taken again
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int j = 0; j < 128; ++j) {
            if (j > row) xv[j] = -INFINITY;
            m4[j & 3] = fmaxf(m4[j & 3], xv[j]);
          }
          m_raw = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        const float m_blk = m_raw * a.scale_log2;
        if (m_blk > m_run + kHeadroom) {
          l_run *= fast_exp2(m_run - m_blk);
          m_run = m_blk;
        }
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 128; ++j) l4[j & 3] += fast_exp2(fmaf(xv[j], a.scale_log2, -m_run));
        l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      }
      if (!ok) break;
      const int t = qb * 128 + row;
      a.lse_px[((size_t)b * a.T + t) * a.G + g] = (m_run + __log2f(l_run)) * kLn2;
    }
    if (!ok) *abort_flag = 1;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_dense_fwd(const Prob& p, const void* Q, const void* K, const void* V, void* O, float* LSE,
                             uint8_t* ws, const WsLayout& L, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  {
    // one head's 128 query rows: box {64 d, 1 head, 128 tokens}
    const uint64_t dims[3] = {128, (uint64_t)p.Hq, (uint64_t)p.BT()};
    const uint64_t strides[2] = {256, (uint64_t)p.Hq * 256};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap(&mq, const_cast<void*>(Q), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {128, (uint64_t)p.G, (uint64_t)p.BT()};
    const uint64_t strides[2] = {256, (uint64_t)p.G * 256};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap(&mk, const_cast<void*>(K), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&mv, const_cast<void*>(V), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  DenseFwdArgs a;
  a.B = p.B;
  a.T = p.T;
  a.Hq = p.Hq;
  a.G = p.G;
  a.hg = p.hg;
  a.n = p.n;
  a.num_items = p.B * p.G * p.n * (p.hg / 2);
  a.counter = reinterpret_cast<int*>(ws + L.counters) + 4;
  a.err = reinterpret_cast<int*>(ws + L.err);
  a.O = static_cast<__nv_bfloat16*>(O);
  a.LSE = LSE;
  a.scale_log2 = p.scale * kLog2e;
  cudaError_t e;
  if ((e = cudaMemsetAsync(a.counter, 0, sizeof(int), st)) != cudaSuccess) return e;
  static bool attr[kMaxDevices] = {};  // kernel attributes are per device context
  const int dslot = device_slot();
  if (!attr[dslot]) {
    if ((e = cudaFuncSetAttribute(dense_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem)) !=
        cudaSuccess)
      return e;
    attr[dslot] = true;
  }
  const int grid = std::min(a.num_items, num_sms());
  timing_begin(MSA_TIME_DENSE_FWD, st);
  dense_fwd_kernel<<<grid, kFThreads, kFSmem, st>>>(a, mq, mk, mv);
  timing_end(MSA_TIME_DENSE_FWD, st);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dense_px(const Prob& p, const void* q_idx, const void* k_idx, float* lse_px, uint8_t* ws,
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
  DensePxArgs a;
  a.B = p.B;
  a.T = p.T;
  a.G = p.G;
  a.n = p.n;
  a.counter = reinterpret_cast<int*>(ws + L.counters) + 5;
  a.err = reinterpret_cast<int*>(ws + L.err);
  a.lse_px = lse_px;
  a.scale_log2 = p.scale_idx * kLog2e;
  cudaError_t e;
  if ((e = cudaMemsetAsync(a.counter, 0, sizeof(int), st)) != cudaSuccess) return e;
  static bool attr[kMaxDevices] = {};
  const int dslot = device_slot();
  if (!attr[dslot]) {
    if ((e = cudaFuncSetAttribute(dense_px_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem)) !=
        cudaSuccess)
      return e;
    attr[dslot] = true;
  }
  const int grid = std::min(p.B * p.G * p.n, 2 * num_sms());
  dense_px_kernel<<<grid, kPThreads, kPSmem, st>>>(a, mq, mk);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
