// Main-branch forward of MiniMax Sparse Attention: exact causal softmax
// attention over the selected KV blocks, with the LSE kept for the backward.
//
// itinai.ru "How to solve the memory problem with MiniMax Sparse Attention",
// "Two-stage process": ordinary scaled dot-product softmax, but only over the
// selected tokens; "Kernel optimisations": iterate over KV blocks (KV-outer)
// and pack ceil(128 / heads-per-group) query positions x heads-per-group
// heads into one 128 x 128 MMA. dothoosh.com "how FlashAttention cuts GPU
// memory traffic", "Online-softmax trick": partial results (m, l, a) of
// different KV blocks merge exactly.
//
// GB300 design. A work item is a run of up to 32 tiles from the inverted list
// of one (b, g, KV block c). K_c and V_c (128 x 128 bf16 each) are staged once
// per item by TMA; each tile gathers the Q rows of 128 / hg selecting queries
// with TMA, one box per query and 64-column chunk holding its hg head rows,
// into a 128 x 128 K-major SW128 tile (TMA swizzles by the shared address, so
// a box landing at row q * hg matches the tile's swizzle). Per tile, tcgen05 computes S = Q K_c^T into TMEM; the softmax
// warps (one TMEM lane = one (query, head) row) mask keys past the query,
// exponentiate, write P (bf16) to shared memory; tcgen05 computes O = P V_c
// into TMEM; the same warps write the normalised partial O and its partial
// LSE for (query, slot), in tile order (one TMA store per warp and 64-column
// chunk). Two S and two O accumulators (512 TMEM columns) let
// the tensor core work on one tile while the softmax warps work on the other.
// A second kernel merges the k partials of every (query, head):
// LSE = ln sum_s exp(lse_s), O = sum_s exp(lse_s - LSE) O_s.
//
// Warp roles (384 threads, one CTA per SM, persistent):
//   warp 0      item fetch, K/V TMA, and producer 0
//   warps 10-11 producers 1 and 2; producer p gathers the queries p, p + 3, ...
//               of every tile into one of three Q stages, with the next tile's
//               entries prefetched into registers
//   warp 1      TMEM owner, UMMA issuer (one thread)
//   warps 2..9  softmax + partial-output epilogue, two warpgroups that take
//               even and odd tiles (ping-pong over the two S/O/P buffers)
#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {
namespace {

constexpr int kThreads = 384;  // 3 producer warps, 1 UMMA warp, 2 x 4 softmax/epilogue warps
constexpr int kFProd = 3;      // producer warps 0, 10, 11
constexpr int kQStages = 3;
constexpr int kTile = 32768;  // 128 rows x 128 bf16, as two 64-column SW128 chunks
constexpr int kChunk = 16384;
constexpr int kSmemBytes = (2 + kQStages + 2) * kTile + 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct FwdArgs {
  const __nv_bfloat16* Q;
  const int32_t* entries;
  const int4* items;
  const int* n_items;
  int* counter;
  int* err;
  __nv_bfloat16* o_part;
  float* lse_part;
  int B, T, Hq, G, hg, n, k;
  int pos_per_tile;
  float scale_log2;  // softmax scale * log2(e)
};

struct FwdShared {
  uint64_t it_full[2], it_empty[2];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_free[2];
  uint64_t o_full[2], o_empty[2];
  int4 item[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int HG>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_fwd_kernel(FwdArgs a, const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_o, const __grid_constant__ CUtensorMap map_q) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTile;
  uint8_t* sQ = smem + 2 * kTile;                // kQStages tiles
  uint8_t* sP = smem + (2 + kQStages) * kTile;   // 2 tiles
  __shared__ FwdShared sh;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], kFProd - 1 + 1 + 8);  // other producers, UMMA, softmax warps
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.s_empty[i], 4);
      mbar_init(&sh.p_full[i], 4);
      mbar_init(&sh.p_free[i], 1);
      mbar_init(&sh.o_full[i], 1);
      mbar_init(&sh.o_empty[i], 4);
    }
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&sh.q_full[i], kFProd);  // every producer (with its TMA bytes)
      mbar_init(&sh.q_empty[i], 1);
    }
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
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
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort;
  constexpr int P = 128 / HG;  // query positions per tile
  const int n_items = *a.n_items;

  // Producer p owns the queries p, p + kFProd, ... of every tile: per query,
  // two TMA boxes (one per 64-column chunk) of its hg head rows, landing at
  // rows q * hg. Padding queries load an out-of-range box (zero fill). Lane u
  // issues requests lane + 32 u; their token rows come from the entries,
  // prefetched one tile ahead.
  constexpr int kMaxQ = (P + kFProd - 1) / kFProd;    // queries of producer 0 per tile
  constexpr int kRPL = (2 * kMaxQ + 31) / 32;         // requests per lane
  auto load_rows = [&](int p, int b, const int4& item, int j, int (&bt)[kRPL]) {
    const int nq = (P - p + kFProd - 1) / kFProd;
    const int BT = a.B * a.T;
#pragma unroll
    for (int u = 0; u < kRPL; ++u) {
      const int o = lane + 32 * u;
      int v = BT;
      if (o < 2 * nq) {
        const int idx = j * P + p + kFProd * (o >> 1);
        if (idx < item.z) v = b * a.T + (a.entries[item.y + idx] >> 8);
      }
      bt[u] = v;
    }
  };
  auto issue_rows = [&](int p, int g, int qs, const int (&bt)[kRPL]) {
    const int nq = (P - p + kFProd - 1) / kFProd;
    if (lane == 0) mbar_arrive_expect_tx(&sh.q_full[qs], nq * HG * 256);
    __syncwarp();
    uint8_t* dst = sQ + qs * kTile;
#pragma unroll
    for (int u = 0; u < kRPL; ++u) {
      const int o = lane + 32 * u;
      if (o < 2 * nq) {
        const int q = p + kFProd * (o >> 1), chunk = o & 1;
        tma_load_3d(dst + chunk * kChunk + q * HG * 128, &map_q, &sh.q_full[qs], chunk * 64, g * HG, bt[u]);
      }
    }
    __syncwarp();
  };
  auto produce_item = [&](int p, const int4& item, int b, int g, uint32_t& tj) -> bool {
    const int ntiles = (item.z + P - 1) / P;
    int bt[kRPL];
    load_rows(p, b, item, 0, bt);
    for (int j = 0; j < ntiles; ++j, ++tj) {
      const int qs = tj % kQStages;
      if (!mbar_wait(&sh.q_empty[qs], ((tj / kQStages) & 1) ^ 1, a.err, 303 + 30 * p)) return false;
      issue_rows(p, g, qs, bt);
      if (j + 1 < ntiles) load_rows(p, b, item, j + 1, bt);
    }
    return true;
  };

  const int prod = warp == 0 ? 0 : warp >= 10 ? warp - 9 : -1;
  if (prod > 0) {
    // ------------------------------------------------------------ producers 1, 2
    if (lane == 0) tma_prefetch_desc(&map_q);
    uint32_t tj = 0;
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 331)) { *abort_flag = 1; break; }
      const int4 item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item.x < 0) break;
      const int bg = item.x / a.n;
      const int b = bg / a.G, g = bg % a.G;
      if (!produce_item(prod, item, b, g, tj)) { *abort_flag = 1; break; }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ items, K/V, producer 0
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_q);
    }
    uint32_t tj = 0;
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      int4 item = make_int4(-1, 0, 0, 0);
      if (lane == 0) {
        if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 301)) *abort_flag = 1;
        int id = atomicAdd(a.counter, 1);
        if (id < n_items && !*abort_flag) item = a.items[id];
        sh.item[s] = item;
        mbar_arrive(&sh.it_full[s]);
      }
      item.x = __shfl_sync(0xffffffffu, item.x, 0);
      item.y = __shfl_sync(0xffffffffu, item.y, 0);
      item.z = __shfl_sync(0xffffffffu, item.z, 0);
      if (item.x < 0) break;
      const int bg = item.x / a.n, c = item.x % a.n;
      const int b = bg / a.G, g = bg % a.G;
      if (lane == 0) {
        bool ok = mbar_wait(&sh.kv_empty, (it & 1) ^ 1, a.err, 302);
        if (ok) {
          mbar_arrive_expect_tx(&sh.kv_full, 2 * kTile);
          const int row0 = b * a.T + c * 128;
          tma_load_3d(sK, &map_k, &sh.kv_full, 0, g, row0);
          tma_load_3d(sK + kChunk, &map_k, &sh.kv_full, 64, g, row0);
          tma_load_3d(sV, &map_v, &sh.kv_full, 0, g, row0);
          tma_load_3d(sV + kChunk, &map_v, &sh.kv_full, 64, g, row0);
        } else {
          *abort_flag = 1;
        }
      }
      __syncwarp();
      if (*abort_flag) break;
      if (!produce_item(0, item, b, g, tj)) { *abort_flag = 1; break; }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(128, 128, false, true);
      const uint32_t k0 = smem_u32(sK), v0 = smem_u32(sV);
      uint32_t tj = 0;
      bool ok = true;
      auto issue_o = [&](uint32_t u) -> bool {
        const int sb = u & 1;
        if (!mbar_wait(&sh.p_full[sb], (u >> 1) & 1, a.err, 311)) return false;
        if (!mbar_wait(&sh.o_empty[sb], ((u >> 1) & 1) ^ 1, a.err, 312)) return false;
        tc_fence_after();
        const uint32_t p0 = smem_u32(sP + sb * kTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ad = make_sdesc(p0 + (ks >> 2) * kChunk + (ks & 3) * 32, 16, 1024, kSw128);
          const uint64_t bd = make_sdesc(v0 + ks * 2048, kChunk, 1024, kSw128);
          umma_bf16_ss(tmem + 256 + sb * 128, ad, bd, idesc_o, ks > 0);
        }
        umma_commit(&sh.o_full[sb]);
        umma_commit(&sh.p_free[sb]);
        return true;
      };
      for (int it = 0; ok; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 313)) { ok = false; break; }
        const int4 item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item.x < 0) break;
        const int ntiles = (item.z + P - 1) / P;
        if (!mbar_wait(&sh.kv_full, it & 1, a.err, 314)) { ok = false; break; }
        for (int j = 0; j < ntiles && ok; ++j, ++tj) {
          const int sb = tj & 1, qs = tj % kQStages;
          if (!mbar_wait(&sh.q_full[qs], (tj / kQStages) & 1, a.err, 315)) { ok = false; break; }
          if (!mbar_wait(&sh.s_empty[sb], ((tj >> 1) & 1) ^ 1, a.err, 316)) { ok = false; break; }
          tc_fence_after();
          const uint32_t q0 = smem_u32(sQ + qs * kTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kChunk + (ks & 3) * 32;
            umma_bf16_ss(tmem + sb * 128, make_sdesc(q0 + off, 16, 1024, kSw128),
                         make_sdesc(k0 + off, 16, 1024, kSw128), idesc_s, ks > 0);
          }
          umma_commit(&sh.s_full[sb]);
          umma_commit(&sh.q_empty[qs]);
          if (j > 0 && !issue_o(tj - 1)) { ok = false; break; }
        }
        if (ok && ntiles > 0 && !issue_o(tj - 1)) ok = false;
        umma_commit(&sh.kv_empty);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Two warpgroups ping-pong: warpgroup wg owns the tiles tj with
    // (tj & 1) == wg, hence S/O TMEM buffer wg and P buffer wg.
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int p_in_tile = row / HG;
    const uint32_t s_col = wg * 128, o_col = 256 + wg * 128;
    uint8_t* pbuf = sP + wg * kTile;
    uint32_t tj = 0;
    bool ok = true;
    // pending tile of this warpgroup (softmax done, output not yet written)
    bool pending = false;
    uint32_t pu = 0;
    float pm = 0.f, pl = 0.f;
    int pentry = -1;
    int prow0 = 0;
    // Partial outputs live in tile order: the tile's rows are consecutive, so
    // each warp stages its 32 normalised rows (bf16, SW128 image) in the P
    // buffer the O MMA has finished with and writes them with one TMA store
    // per 64-column chunk.
    auto epilogue = [&]() -> bool {
      if (!mbar_wait(&sh.o_full[wg], (pu >> 1) & 1, a.err, 321)) return false;
      tc_fence_after();
      const float inv = pentry >= 0 ? 1.f / pl : 0.f;
      // each 64-column chunk leaves by its own TMA store (one bulk group
      // each) as soon as it is staged; pass 2 of the next tile waits for
      // each chunk's store separately
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[32];
        tmem_ld32(tmem + lane_off + o_col + q * 32, o);
        tmem_wait_ld();
        if (q == 3) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.o_empty[wg]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int c16 = q * 4 + c;
          *reinterpret_cast<uint4*>(pbuf + (c16 >> 3) * kChunk + sw128_off(row, c16 & 7)) = make_uint4(
              pack_bf16(o[8 * c + 0] * inv, o[8 * c + 1] * inv), pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
              pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv), pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
        }
        if (q & 1) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_o, pbuf + (q >> 1) * kChunk + quarter * 4096, (q >> 1) * 64, prow0 + quarter * 32);
            bulk_commit();
          }
        }
      }
      if (pentry >= 0) a.lse_part[(size_t)prow0 + row] = (pm + __log2f(pl)) * kLn2;
      return true;
    };
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 322)) { ok = false; break; }
      const int4 item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item.x < 0) break;
      const int c = item.x % a.n;
      const int ntiles = (item.z + P - 1) / P;
      for (int j = 0; j < ntiles; ++j, ++tj) {
        if ((int)(tj & 1) != wg) continue;
        const int idx = j * P + p_in_tile;
        const int entry = idx < item.z ? a.entries[item.y + idx] : -1;
        const int lim = entry >= 0 ? (entry >> 8) - c * 128 : -1;  // last visible key column
        if (!mbar_wait(&sh.s_full[wg], (tj >> 1) & 1, a.err, 323)) { ok = false; break; }
        tc_fence_after();
        // pass 1: row max over the visible keys (four independent chains;
        // a warp whose rows all see the whole block skips the mask)
        const bool full = __all_sync(0xffffffffu, lim >= 127);
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[32];
          if (full) {  // the loads' own maximum (tcgen05.ld.red)
            tmem_ld32_max(tmem + lane_off + s_col + q * 32, x, m4[q]);
            tmem_wait_ld();
          } else {
            tmem_ld32(tmem + lane_off + s_col + q * 32, x);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (q * 32 + i <= lim) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
          }
        }
        const float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float mm = (m == -INFINITY) ? 0.f : m * a.scale_log2;
        // Tile tj-2 (same warpgroup, same P buffer) is finished first: its O
        // is staged through P buffer wg, so it must leave before P(tj) goes in.
        if (pending && !epilogue()) { ok = false; break; }
        pending = false;
        // P buffer wg is free once the O MMA of tile tj-2 has read it; each
        // chunk of it once this warp's store of tile tj-2's rows has read it
        if (!mbar_wait(&sh.p_free[wg], ((tj >> 1) & 1) ^ 1, a.err, 324)) { ok = false; break; }
        // pass 2: P = exp2(s * scale * log2 e - max), row sum, bf16 image.
        // S is released to the tensor core right after its last TMEM load.
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[32];
          tmem_ld32(tmem + lane_off + s_col + q * 32, x);
          tmem_wait_ld();
          if (q == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.s_empty[wg]);
          }
          if (q == 0 || q == 2) {  // chunk q / 2 of the P buffer: its staged O rows have left
            if (lane == 0) {
              if (q == 0) bulk_wait_read_but_one();
              else bulk_wait_read_all();
            }
            __syncwarp();
          }
          if (full) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = fast_exp2(fmaf(x[i], a.scale_log2, -mm));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              x[i] = (q * 32 + i <= lim) ? fast_exp2(fmaf(x[i], a.scale_log2, -mm)) : 0.f;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) l4[i & 3] += x[i];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c16 = q * 4 + cc;
            *reinterpret_cast<uint4*>(pbuf + (c16 >> 3) * kChunk + sw128_off(row, c16 & 7)) =
                make_uint4(pack_bf16(x[8 * cc + 0], x[8 * cc + 1]), pack_bf16(x[8 * cc + 2], x[8 * cc + 3]),
                           pack_bf16(x[8 * cc + 4], x[8 * cc + 5]), pack_bf16(x[8 * cc + 6], x[8 * cc + 7]));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_full[wg]);
        pending = true;
        pu = tj;
        pm = mm;
        pl = (l4[0] + l4[1]) + (l4[2] + l4[3]);
        pentry = entry;
        prow0 = (item.w + j * P) * HG;
      }
    }
    if (ok && pending) ok = epilogue();
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (!ok) *abort_flag = 1;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

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

// One warp per (b, t, g): merge the k partials of each of the HG heads. The
// partial of (b, g, t, slot) sits at padded entry rev[(b*G + g)*T + t][slot];
// its HG head rows are one contiguous HG * 256-byte run. Lane s owns slots s
// and s + 32: it reads their partial LSEs, and once the row's LSEs are known
// it writes their partial rows and merge weights e^{lse_s - LSE} to shared
// memory; every lane then owns 4 * HG consecutive output values (head
// lane / (32 / HG)) and sums the partial rows with one shared load per slot.
constexpr int kMergeThreads = 256;
template <int HG, int NSL>  // NSL slots per lane: k <= 32 NSL
__global__ void __launch_bounds__(kMergeThreads)
    fwd_merge_kernel(const int32_t* __restrict__ block_idx, const int32_t* __restrict__ rev,
                     const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ lse_part,
                     __nv_bfloat16* __restrict__ O, float* __restrict__ LSE, int B, int T, int Hq, int G, int k,
                     long long max_padded) {
  constexpr int kPer = 4 * HG;  // output values per lane
  constexpr int kLanesPerHead = 32 / HG;
  __shared__ int s_row[kMergeThreads / 32][32 * NSL];
  __shared__ float s_wgt[kMergeThreads / 32][32 * NSL][HG];
  const long long rows = (long long)B * T * G;
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int my_head = lane / kLanesPerHead;
  for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; w < rows;
       w += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int g = (int)(w % G);
    const long long bt = w / G;
    const int t = (int)(bt % T), b = (int)(bt / T);
    const size_t sel_row = (((size_t)b * G + g) * T + t) * k;
    // a slot counts only if the map placed it (rows that failed validation
    // keep -1 and are left unspecified, with the error word set)
    float l_own[NSL][HG];
    int rv_own[NSL];
#pragma unroll
    for (int u = 0; u < NSL; ++u) {
      const int sidx = lane + 32 * u;
      int r = -1;
      if (sidx < k && block_idx[sel_row + sidx] >= 0) {
        r = rev[sel_row + sidx];
        if (r >= 0 && (long long)r >= max_padded) r = -1;
      }
      rv_own[u] = r;
#pragma unroll
      for (int h = 0; h < HG; ++h) l_own[u][h] = r >= 0 ? lse_part[(size_t)r * HG + h] : -INFINITY;
    }
    float lse[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float mx = l_own[0][h];
#pragma unroll
      for (int u = 1; u < NSL; ++u) mx = fmaxf(mx, l_own[u][h]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float z = 0.f;
#pragma unroll
      for (int u = 0; u < NSL; ++u) z += l_own[u][h] > -INFINITY ? expf(l_own[u][h] - mx) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      lse[h] = mx + logf(z);
    }
#pragma unroll
    for (int u = 0; u < NSL; ++u) {
      const int sidx = lane + 32 * u;
      if (sidx < k) {
        s_row[wib][sidx] = rv_own[u];
#pragma unroll
        for (int h = 0; h < HG; ++h) s_wgt[wib][sidx][h] = rv_own[u] >= 0 ? expf(l_own[u][h] - lse[h]) : 0.f;
      }
    }
    __syncwarp();
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    // slots in ascending order, two rows' loads in flight before they are added
    for (int s0 = 0; s0 < k; s0 += 2) {
      int r[2];
      uint4 raw[2][kPer / 8 > 0 ? kPer / 8 : 1];
      uint2 raw4[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        r[j] = s0 + j < k ? s_row[wib][s0 + j] : -1;
        if (r[j] >= 0) {
          const __nv_bfloat16* row = o_part + (size_t)r[j] * HG * 128 + lane * kPer;
          if constexpr (kPer % 8 == 0) {
#pragma unroll
            for (int q = 0; q < kPer / 8; ++q) raw[j][q] = reinterpret_cast<const uint4*>(row)[q];
          } else {
            raw4[j] = *reinterpret_cast<const uint2*>(row);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (r[j] < 0) continue;
        const float wgt = s_wgt[wib][s0 + j][my_head];
        if constexpr (kPer % 8 == 0) {
#pragma unroll
          for (int q = 0; q < kPer / 8; ++q) {
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[j][q]);
#pragma unroll
            for (int z = 0; z < 4; ++z) {
              const float2 f = __bfloat1622float2(h2[z]);
              acc[q * 8 + 2 * z] = fmaf(wgt, f.x, acc[q * 8 + 2 * z]);
              acc[q * 8 + 2 * z + 1] = fmaf(wgt, f.y, acc[q * 8 + 2 * z + 1]);
            }
          }
        } else {
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw4[j]);
          const float2 f0 = __bfloat1622float2(h2[0]), f1 = __bfloat1622float2(h2[1]);
          acc[0] = fmaf(wgt, f0.x, acc[0]);
          acc[1] = fmaf(wgt, f0.y, acc[1]);
          acc[2] = fmaf(wgt, f1.x, acc[2]);
          acc[3] = fmaf(wgt, f1.y, acc[3]);
        }
      }
    }
    __syncwarp();  // the next row rewrites this warp's slot table
    const size_t orow0 = ((size_t)b * T + t) * Hq + g * HG;
    uint2* dst = reinterpret_cast<uint2*>(O + orow0 * 128 + lane * kPer);
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q)
      dst[q] = make_uint2(pack_bf16(acc[q * 4 + 0], acc[q * 4 + 1]), pack_bf16(acc[q * 4 + 2], acc[q * 4 + 3]));
    if (lane < HG) {
      float v = lse[0];
#pragma unroll
      for (int h = 1; h < HG; ++h)
        if (lane == h) v = lse[h];
      LSE[orow0 + lane] = v;
    }
  }
}

// Two slots per lane up to k = 64, four up to k = 128.
template <int HG>
void fwd_merge(const Prob& p, const int32_t* block_idx, const int32_t* rev, const __nv_bfloat16* o_part,
               const float* lse_part, __nv_bfloat16* O, float* LSE, long long max_padded, int grid, cudaStream_t st) {
  if (p.k <= 64)
    fwd_merge_kernel<HG, 2><<<grid, kMergeThreads, 0, st>>>(block_idx, rev, o_part, lse_part, O, LSE, p.B, p.T, p.Hq,
                                                             p.G, p.k, max_padded);
  else
    fwd_merge_kernel<HG, 4><<<grid, kMergeThreads, 0, st>>>(block_idx, rev, o_part, lse_part, O, LSE, p.B, p.T, p.Hq,
                                                             p.G, p.k, max_padded);
}

}  // namespace

cudaError_t launch_sparse_fwd(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* block_idx,
                              void* O, float* LSE, uint8_t* ws, const WsLayout& L, cudaStream_t st, bool mapped) {
  const int pos_per_tile = fwd_tile_queries(p);
  cudaError_t e;
  if (!mapped && (e = build_block_map(p, block_idx, ws, L, pos_per_tile, kFwdTilesPerItem, st)) != cudaSuccess)
    return e;
  CUtensorMap mk, mv;
  const uint64_t dims[3] = {(uint64_t)p.d, (uint64_t)p.G, (uint64_t)p.BT()};
  const uint64_t strides[2] = {(uint64_t)p.d * 2, (uint64_t)p.G * p.d * 2};
  const uint32_t box[3] = {64, 1, 128};
  if (!encode_tmap(&mk, const_cast<void*>(K), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tmap(&mv, const_cast<void*>(V), 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  CUtensorMap mo, mq;
  {
    // one query's head rows of its group: box {64 d, hg heads, 1 token}
    const uint64_t qdims[3] = {128, (uint64_t)p.Hq, (uint64_t)p.BT()};
    const uint64_t qstr[2] = {256, (uint64_t)p.Hq * 256};
    const uint32_t qbox[3] = {64, (uint32_t)p.hg, 1};
    if (!encode_tmap(&mq, const_cast<void*>(Q), 3, qdims, qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t odims[2] = {128, (uint64_t)L.max_padded * p.hg};
    const uint64_t ostr[1] = {256};
    const uint32_t obox[2] = {64, 32};
    if (!encode_tmap(&mo, ws + L.o_part, 2, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  FwdArgs a;
  a.Q = static_cast<const __nv_bfloat16*>(Q);
  a.entries = reinterpret_cast<const int32_t*>(ws + L.entries);
  a.items = reinterpret_cast<const int4*>(ws + L.items);
  a.n_items = reinterpret_cast<const int*>(ws + L.n_items);
  a.counter = reinterpret_cast<int*>(ws + L.counters) + 1;
  a.err = reinterpret_cast<int*>(ws + L.err);
  a.o_part = reinterpret_cast<__nv_bfloat16*>(ws + L.o_part);
  a.lse_part = reinterpret_cast<float*>(ws + L.lse_part);
  a.B = p.B;
  a.T = p.T;
  a.Hq = p.Hq;
  a.G = p.G;
  a.hg = p.hg;
  a.n = p.n;
  a.k = p.k;
  a.pos_per_tile = pos_per_tile;
  a.scale_log2 = p.scale * kLog2e;
  if ((e = cudaMemsetAsync(a.counter, 0, sizeof(int), st)) != cudaSuccess) return e;
  static bool attr[kMaxDevices] = {};  // kernel attributes are per device context
  const int dslot = device_slot();
  if (!attr[dslot]) {
    for (auto f : {sparse_fwd_kernel<1>, sparse_fwd_kernel<2>, sparse_fwd_kernel<4>, sparse_fwd_kernel<8>})
      if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) != cudaSuccess)
        return e;
    attr[dslot] = true;
  }
  timing_begin(MSA_TIME_SPARSE_FWD, st);
  switch (p.hg) {
    case 1: sparse_fwd_kernel<1><<<num_sms(), kThreads, kSmemBytes, st>>>(a, mk, mv, mo, mq); break;
    case 2: sparse_fwd_kernel<2><<<num_sms(), kThreads, kSmemBytes, st>>>(a, mk, mv, mo, mq); break;
    case 4: sparse_fwd_kernel<4><<<num_sms(), kThreads, kSmemBytes, st>>>(a, mk, mv, mo, mq); break;
    default: sparse_fwd_kernel<8><<<num_sms(), kThreads, kSmemBytes, st>>>(a, mk, mv, mo, mq); break;
  }
  timing_end(MSA_TIME_SPARSE_FWD, st);
  count_launches(2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.T * p.G;
  const int grid = (int)std::min<long long>((rows * 32 + 255) / 256, 16LL * num_sms());
  const int32_t* rev = reinterpret_cast<const int32_t*>(ws + L.rev);
  __nv_bfloat16* Ob = static_cast<__nv_bfloat16*>(O);
  switch (p.hg) {
    case 1: fwd_merge<1>(p, block_idx, rev, a.o_part, a.lse_part, Ob, LSE, L.max_padded, grid, st); break;
    case 2: fwd_merge<2>(p, block_idx, rev, a.o_part, a.lse_part, Ob, LSE, L.max_padded, grid, st); break;
    case 4: fwd_merge<4>(p, block_idx, rev, a.o_part, a.lse_part, Ob, LSE, L.max_padded, grid, st); break;
    default: fwd_merge<8>(p, block_idx, rev, a.o_part, a.lse_part, Ob, LSE, L.max_padded, grid, st); break;
  }
  return cudaGetLastError();
}

}  // namespace msa
