// Fused backward of MiniMax Sparse Attention on 128-row tiles, for 4 or 8
// query heads per GQA group: main-branch dQ/dK/dV and the KL-alignment
// gradient of the index branch in one pass over the selected blocks.
//
// dothoosh.com "how Flash-MSA cuts million-token training cost", "Kernel
// design and execution": one fused backward over proxy and main branch,
// scheduled through the inverted block -> query map so that each KV block is
// staged once for all query chunks that chose it; "Fixing the KL-divergence
// bottleneck": d KL / d s_px = p_px - p_main. itinai.ru "How to solve the
// memory problem with MiniMax Sparse Attention", "Training sparse attention":
// the teacher is the head-averaged main softmax, detached. dothoosh.com "how
// FlashAttention cuts GPU memory traffic", "Training and the backward pass":
// P is rebuilt from the saved LSE; dV += P^T dO, dP = dO V^T.
//
// Per KV block c of (b, g) (one work item = one inverted list), keys on TMEM
// lanes, tiles of 128 (query, head) rows = 128 / hg queries x hg heads:
//   S^T  = K_c Q^T     (N = 128)      X^T = KI_c QI^T   (N = queries)
//   P    = exp(s - LSE), p_main = head mean, p_px = exp(x - lse_px)
//   dP^T = V_c dO^T    (N = 128)      dS = P (dP - D)
//   dV  += P^T dO      (P^T from TMEM) dK += dS^T Q      (TMEM, whole list)
//   dQ^T = K_c^T dS^T  (N = 128)       -> bf16 slot partial, TMA store
//   gs   = w (p_px - p_main)           dk_idx += gs^T QI (TMEM, whole list)
//   dq_idx^T = KI_c^T gs^T             -> bf16 slot partial, TMA store
//   KL terms summed over each warp's 32 keys -> fp32 partial per (slot, key quarter)
// Every MMA of a tile has N = 128 except the index ones, so the tensor pipe
// runs near its per-instruction rate instead of at the N = 64 floor of a
// 64-row tile. The merge adds slot partials (and a slot's four key-quarter KL
// sums) in a fixed order, so every output is the same in every run.
//
// TMEM (512 columns): R [0, 128) holds S^T, then dP^T (once the epilogue has
// loaded S^T), then dQ^T; P [128, 192) holds X^T, then P^T as packed bf16
// pairs (once every epilogue warp has loaded X^T), then dq_idx^T (once dV has
// read P^T); dV [192, 320), dK [320, 448), dk_idx [448, 512) accumulate over
// the list.
//
// Shared memory: K, V, k_idx of the block (80 KB), two gather buffers of
// 68 KB (Q, dO: 128 rows x 256 B each; q_idx: one 128-byte row per query) and
// the tile's gs^T image (8 KB). Inside a tile's buffer, dS^T goes where dO was
// (once dV has read it), and the dQ partials (where dS^T was) and dq_idx
// partials (where Q was) are staged for their TMA stores. A buffer goes back
// to the producers once the next tile's X^T is complete.
//
// Full attention (DENSE): the lists are every query from the block on, built
// from the item number in segments of 4096 queries; a tile's queries are
// consecutive tokens, gathered with five whole-tile boxes; dQ is added into
// the caller's fp32 dQ by TMA reduce-add, dq_idx, KL, dK, dV and dk_idx by
// atomic adds.
//
// Warp roles (512 threads, one CTA per SM, persistent; registers split 64 /
// 192 between the first two warpgroups and the last two):
//   warp 0       TMEM owner, UMMA issuer (one thread)
//   warps 1-7    producers 0-6: producer p gathers the queries p, p + 7, ...
//                of every tile (TMA boxes of their hg head rows of Q and dO,
//                and their q_idx row) and writes their row metadata;
//                producer 0 also fetches the work items and loads K, V, k_idx
//   warps 8-15   epilogue: TMEM lane quarter = warp % 4, warpgroup hf owns
//                the tile rows [64 hf, 64 hf + 64)
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

constexpr int kThreads = 512;
constexpr int kProd = 7;                  // producer warps 1..7
constexpr int kRows = 128;                // (query, head) rows per tile
constexpr int kKV = 32768;                // 128 keys x 128 d bf16
constexpr int kChunk = 16384;             // 128 rows x 64 bf16 (one SW128 column chunk)
constexpr int kKIb = 16384;               // 128 keys x 64 bf16
// smem map: K, V, k_idx, then two gather buffers, then the shared state
constexpr int oK = 0, oV = kKV, oKI = 2 * kKV, oG = 2 * kKV + kKIb;
constexpr int oQ = 0, oDO = 2 * kChunk, oQI = 4 * kChunk;  // inside a gather buffer
constexpr int kQIb = 4096;                                  // up to 32 q_idx rows
constexpr int kGather = oQI + kQIb;
// gs^T of the current tile: 128 keys x (queries per tile) bf16, 64-byte rows with 64-byte swizzle
// (4 heads per group, 32 queries) or 32-byte rows with 32-byte swizzle (8 heads, 16 queries)
constexpr int oGS = oG + 2 * kGather;
constexpr int kGSb = 8192;
constexpr int oSh = oGS + kGSb;
// TMEM columns
constexpr uint32_t cR = 0, cP = 128, cDV = 192, cDK = 320, cKI = 448;

struct __align__(16) RowMeta {
  float lse2[kRows];  // per (query, head) row: LSE * log2 e (+inf for padding rows: P = 0 there)
  float dsc[kRows];   // per row: D * scale
  float lpx2[32];     // per query: lse_px * log2 e (+inf for padding queries)
  int ent[32];        // per query: entry bits t << 8 | slot, -1 for padding
  int diag[8];        // per producer: some row sees only part of the block (causal mask needed)
};

struct Shared {
  uint64_t it_full[2], it_empty[2];
  uint64_t kv_full, kv_empty;
  uint64_t g_full[2], g_empty[2];
  uint64_t s_full, x_full, s_read, x_read, dp_full, dp_read, p_ready, pv_done, ds_tmem, ds_smem, dk_done;
  uint64_t gs_ready, dq_full, ph2_full;
  uint64_t r_free, x_free, acc_free;
  RowMeta meta[2];
  int4 item[2];
  uint32_t tmem_base;
  int abort;
};
constexpr int kSmem = oSh + (int)sizeof(Shared);
static_assert(kGather % 1024 == 0, "gather buffers keep the 1024-byte swizzle alignment");
static_assert(kSmem <= 232448, "backward kernel exceeds 227 KB of shared memory");

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The value unchanged, through an instruction the compiler cannot see through.
__device__ __forceinline__ uint32_t opaque_u32(uint32_t x) {
  asm volatile("mov.b32 %0, %0;" : "+r"(x));
  return x;
}

__device__ __forceinline__ void regs_dealloc64() { asm volatile("setmaxnreg.dec.sync.aligned.u32 64;\n" ::: "memory"); }
__device__ __forceinline__ void regs_alloc192() { asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory"); }

// Full attention: work item id -> {list (b, g, c), first query, number of queries, 0}. Items run over the
// batch entries, then segments of dense_seg queries, then blocks c ascending (longest first) and groups,
// so that the CTAs running at the same time add into the dQ rows of one segment, which stay in L2.
__device__ __forceinline__ int4 dense_item(int id, const BwdArgs& a) {
  const int b = id / a.dense_per_b;
  int r = id - b * a.dense_per_b;
  const int bps = a.dense_seg / 128;  // blocks per segment
  const int nseg = (a.T + a.dense_seg - 1) / a.dense_seg;
  int s = 0;
  for (; s < nseg - 1; ++s) {
    const int cnt = a.G * min((s + 1) * bps, a.n);
    if (r < cnt) break;
    r -= cnt;
  }
  const int c = r / a.G, g = r - c * a.G;
  const int t0 = max(c * 128, s * a.dense_seg);
  const int t1 = min((s + 1) * a.dense_seg, a.T);
  return make_int4((b * a.G + g) * a.n + c, t0, t1 - t0, 0);
}

// DENSE: full attention. The lists are every query from the block on, cut into segments (dense_item);
// dQ leaves by TMA reduce-add into the caller's fp32 dQ, dq_idx, KL, dK, dV and dk_idx by atomic adds.
template <int HG, bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_wide_kernel(BwdArgs a, const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                    const __grid_constant__ CUtensorMap map_ki, const __grid_constant__ CUtensorMap map_dq,
                    const __grid_constant__ CUtensorMap map_dqi, const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_do, const __grid_constant__ CUtensorMap map_qi) {
  static_assert(HG == 4 || HG == 8, "128-row tiles for 4 or 8 heads per group");
  constexpr int hg = HG;
  constexpr int npos = kRows / HG;  // queries per tile (32 or 16)
  constexpr int kHQ = npos / 2;     // queries of one epilogue half
  constexpr uint32_t kGsRow = npos * 2;       // bytes of one key's gs^T row
  constexpr uint32_t kGsAtom = 8 * kGsRow;    // 8-row swizzle atom
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // uniform for the block: nothing started yet
    if (threadIdx.x == 0) dev_fail(a.err, kDevSmemAlign, 600);
    return;
  }
  Shared& sh = *reinterpret_cast<Shared*>(smem + oSh);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) sh.meta[0].diag[i] = sh.meta[1].diag[i] = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.it_full[i], 1);
      mbar_init(&sh.it_empty[i], kProd - 1 + 1 + 8);  // other producers, UMMA, epilogue warps
      mbar_init(&sh.g_full[i], kProd);                // every producer warp (with its TMA bytes)
      mbar_init(&sh.g_empty[i], 8);                   // epilogue warps, once their stores have read the buffer
    }
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.x_full, 1);
    mbar_init(&sh.s_read, 8);
    mbar_init(&sh.x_read, 8);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.dp_read, 8);
    mbar_init(&sh.p_ready, 8);
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.ds_tmem, 8);
    mbar_init(&sh.ds_smem, 8);
    mbar_init(&sh.dk_done, 1);
    mbar_init(&sh.gs_ready, 8);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.ph2_full, 1);
    mbar_init(&sh.r_free, 8);
    mbar_init(&sh.x_free, 4);  // the warps of TMEM lanes 0..63, which hold dq_idx^T
    mbar_init(&sh.acc_free, 8);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort;
  const int n_items = DENSE ? a.dense_items : *a.n_items;

  // The register split is set where it dominates each role's code, so that
  // the compiler gives the epilogue its 192 registers.
  if (warp < 8) {
  regs_dealloc64();
  if (warp >= 1) {
    // ------------------------------------------------------------ producers
    const int p = warp - 1;
    const int nq = (npos - p + kProd - 1) / kProd;  // queries of this producer in a tile
    const int qmine = p + kProd * (lane / hg), hmine = lane % hg;
    const bool mine = lane < nq * hg;  // lane's (query, head) row
    auto load_entry = [&](const int4& item, int j) -> int {
      const int idx = j * npos + qmine;
      if constexpr (DENSE) return (mine && idx < item.z) ? (item.y + idx) << 8 : -1;
      else return (mine && idx < item.z) ? a.entries[item.y + idx] : -1;
    };
    auto load_rec = [&](int b, int g, int e) -> float4 {
      if (e < 0) return make_float4(INFINITY, 0.f, INFINITY, __int_as_float(e));
      const int t = e >> 8;
      const size_t hr = ((size_t)b * a.T + t) * a.Hq + g * hg + hmine;
      const float l = a.LSE[hr], d = a.drow[hr];
      const float x = a.lse_px[((size_t)b * a.T + t) * a.G + g];
      return make_float4(l * kLog2e, d * a.scale, x * kLog2e, __int_as_float(e));
    };
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_do);
      tma_prefetch_desc(&map_qi);
      if (p == 0) {
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
        tma_prefetch_desc(&map_ki);
      }
    }
    uint32_t tj = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      int4 item = make_int4(-1, 0, 0, 0);
      if (p == 0) {
        if (lane == 0) {
          if (!mbar_wait(&sh.it_empty[s], ph ^ 1, a.err, 601)) *abort_flag = 1;
          const int id = atomicAdd(a.counter, 1);
          if (id < n_items && !*abort_flag) {
            if constexpr (DENSE) item = dense_item(id, a);
            else item = a.items[id];
          }
          sh.item[s] = item;
          mbar_arrive(&sh.it_full[s]);
        }
        item.x = __shfl_sync(0xffffffffu, item.x, 0);
        item.y = __shfl_sync(0xffffffffu, item.y, 0);
        item.z = __shfl_sync(0xffffffffu, item.z, 0);
        item.w = __shfl_sync(0xffffffffu, item.w, 0);
      } else {
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 602)) { ok = false; break; }
        item = sh.item[s];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      }
      if (item.x < 0) break;
      int b, g, c;
      decode_list(item.x, a.n, a.G, b, g, c);
      if (p == 0) {
        if (lane == 0) {
          if (mbar_wait(&sh.kv_empty, (it & 1) ^ 1, a.err, 603)) {
            mbar_arrive_expect_tx(&sh.kv_full, 2 * kKV + kKIb);
            const int row0 = b * a.T + c * 128;
            tma_load_3d(smem + oK, &map_k, &sh.kv_full, 0, g, row0);
            tma_load_3d(smem + oK + kChunk, &map_k, &sh.kv_full, 64, g, row0);
            tma_load_3d(smem + oV, &map_v, &sh.kv_full, 0, g, row0);
            tma_load_3d(smem + oV + kChunk, &map_v, &sh.kv_full, 64, g, row0);
            tma_load_2d(smem + oKI, &map_ki, &sh.kv_full, 0, row0);
          } else {
            *abort_flag = 1;
          }
        }
        __syncwarp();
        if (*abort_flag) break;
      }
      const int ntiles = (item.z + npos - 1) / npos;
      const int key_last = c * 128 + 127;
      const int BT = a.B * a.T;
      int e_next = load_entry(item, 0);
      float4 rec = load_rec(b, g, e_next);
      e_next = ntiles > 1 ? load_entry(item, 1) : -1;
      for (int j = 0; j < ntiles; ++j, ++tj) {
        const int gb = tj & 1;
        if (!mbar_wait(&sh.g_empty[gb], ((tj >> 1) & 1) ^ 1, a.err, 604 + p)) { ok = false; break; }
        uint8_t* buf = smem + oG + gb * kGather;
        RowMeta& m = sh.meta[gb];
        const int e_own = __float_as_int(rec.w);
        if (mine) {
          const int r = qmine * hg + hmine;
          m.lse2[r] = rec.x;
          m.dsc[r] = rec.y;
          if (hmine == 0) {
            m.lpx2[qmine] = rec.z;
            m.ent[qmine] = e_own;
          }
        }
        const unsigned dg = __ballot_sync(0xffffffffu, mine && e_own >= 0 && (e_own >> 8) < key_last);
        if constexpr (DENSE) {
          // consecutive queries: producer 0 loads the whole tile with five boxes (Q and dO per 64-column
          // chunk: 128 / hg tokens x hg heads, landing at row q * hg as the one-query boxes would; q_idx:
          // one row per token); the other producers only write their rows' metadata
          if (lane == 0) {
            m.diag[p] = dg != 0u;
            if (p == 0) {
              mbar_arrive_expect_tx(&sh.g_full[gb], npos * (2 * hg * 256 + 128));
              const int bt0 = b * a.T + item.y + j * npos;
              tma_load_3d(buf + oQ, &map_q, &sh.g_full[gb], 0, g * hg, bt0);
              tma_load_3d(buf + oQ + kChunk, &map_q, &sh.g_full[gb], 64, g * hg, bt0);
              tma_load_3d(buf + oDO, &map_do, &sh.g_full[gb], 0, g * hg, bt0);
              tma_load_3d(buf + oDO + kChunk, &map_do, &sh.g_full[gb], 64, g * hg, bt0);
              tma_load_3d(buf + oQI, &map_qi, &sh.g_full[gb], 0, g, bt0);
            } else {
              mbar_arrive(&sh.g_full[gb]);
            }
          }
          __syncwarp();
        } else {
        if (lane == 0) {
          m.diag[p] = dg != 0u;
          mbar_arrive_expect_tx(&sh.g_full[gb], nq * (2 * hg * 256 + 128));
        }
        __syncwarp();
        // per query: Q and dO boxes of its hg head rows (one per 64-column
        // chunk) at row q * hg, then its q_idx row at row q; padding queries
        // load an out-of-range box (zero fill, bytes still counted)
#pragma unroll 1
        for (int o = lane; o < nq * 5; o += 32) {
          const int i = o / 5, op = o - i * 5;
          const int q = p + kProd * i;
          const int e = m.ent[q];
          const int bt = e >= 0 ? b * a.T + (e >> 8) : BT;
          if (op < 4) {
            const int which = op >> 1, chunk = op & 1;
            tma_load_3d(buf + (which ? oDO : oQ) + chunk * kChunk + q * hg * 128, which ? &map_do : &map_q,
                        &sh.g_full[gb], chunk * 64, g * hg, bt);
          } else {
            tma_load_2d(buf + oQI + q * 128, &map_qi, &sh.g_full[gb], 0, bt * a.G + g);
          }
        }
        __syncwarp();
        }
        if (j + 1 < ntiles) {
          rec = load_rec(b, g, e_next);
          e_next = j + 2 < ntiles ? load_entry(item, j + 2) : -1;
        }
      }
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = make_idesc_bf16(128, 128, false, false);   // K-major x K-major, N = 128
      constexpr uint32_t id_acc = make_idesc_bf16(128, 128, false, true);  // K-major A, MN-major B
      constexpr uint32_t id_dq = make_idesc_bf16(128, 128, true, true);    // MN-major A and B
      constexpr uint32_t id_x = make_idesc_bf16(128, npos, false, false);
      constexpr uint32_t id_ki = make_idesc_bf16(128, 64, false, true);
      constexpr uint32_t id_dqi = make_idesc_bf16(128, npos, true, true);
      // Descriptors as 32-bit low words sharing one high word (SBO 1024, 128-byte swizzle): every
      // MMA below is one or two immediate adds and the issue, so that this thread, which shares its
      // scheduler with two epilogue warps, keeps the tensor pipe fed at its N = 128 rate.
      constexpr uint32_t hi = sdesc_hi_sw128_sbo1024();
      const uint32_t kA0 = sdesc_lo(smem_u32(smem + oK), 16);        // K, K-major
      const uint32_t kT0 = sdesc_lo(smem_u32(smem + oK), kChunk);    // K as MN-major A (M = d)
      const uint32_t vA0 = sdesc_lo(smem_u32(smem + oV), 16);
      const uint32_t iA0 = sdesc_lo(smem_u32(smem + oKI), 16);
      const uint32_t iT0 = sdesc_lo(smem_u32(smem + oKI), kChunk);
      const uint32_t gA0 = sdesc_lo(smem_u32(smem + oG), 16);       // gather-buffer operands, K-major
      const uint32_t gT0 = sdesc_lo(smem_u32(smem + oG), kChunk);   // and MN-major
      // gs^T: rows of npos bf16 (64 or 32 bytes), atoms of 8 rows; K-major A of dk_idx and MN-major B
      // of dq_idx^T (one atom wide) from the same image
      constexpr uint32_t hiGS = sdesc_hi(kGsAtom, npos == 32 ? kSw64 : kSw32);
      const uint32_t gsA = sdesc_lo(smem_u32(smem + oGS), 16);
      const uint32_t gsB = sdesc_lo(smem_u32(smem + oGS), kGSb);
      uint32_t tj = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&sh.it_full[s], ph, a.err, 611)) { ok = false; break; }
        const int4 item = sh.item[s];
        mbar_arrive(&sh.it_empty[s]);
        if (item.x < 0) break;
        const int ntiles = (item.z + npos - 1) / npos;
        if (!mbar_wait(&sh.kv_full, it & 1, a.err, 612)) { ok = false; break; }
        bool s_issued = false;  // this tile's S^T went out during the previous tile
        for (int j = 0; j < ntiles; ++j, ++tj) {
          const uint32_t par = tj & 1;
          const uint32_t gA = gA0 + ((tj & 1) * kGather >> 4), gT = gT0 + ((tj & 1) * kGather >> 4);
          // per-tile copies the compiler cannot hoist: otherwise it keeps every base + k-step sum of
          // the tile loop live in registers across it
          const uint32_t kA = opaque_u32(kA0), kT = opaque_u32(kT0), vA = opaque_u32(vA0);
          const uint32_t iA = opaque_u32(iA0), iT = opaque_u32(iT0);
          // a K-major k-step inside a tile of two 64-column chunks, in descriptor units
#define KSTEP(ks) ((uint32_t)((((ks) >> 2) * kChunk + ((ks) & 3) * 32) >> 4))
          // S^T = K Q^T into R, once the tile is gathered and the last dQ^T has been read out (issued
          // during the previous tile, right after its dQ^T, unless this is the list's first tile)
          auto issue_s = [&](uint32_t u) -> bool {
            if (!mbar_wait(&sh.g_full[u & 1], (u >> 1) & 1, a.err, 613)) return false;
            if (!mbar_wait(&sh.r_free, (u & 1) ^ 1, a.err, 614)) return false;
            tc_fence_after();
            const uint32_t gAu = gA0 + ((u & 1) * kGather >> 4);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_bf16_ss_w(tmem + cR, kA + KSTEP(ks), gAu + (oQ >> 4) + KSTEP(ks), hi, id_s, ks > 0);
            umma_commit(&sh.s_full);
            return true;
          };
          if (!s_issued && !issue_s(tj)) { ok = false; break; }
          s_issued = false;
          // X^T = KI QI^T into P, once the last dq_idx^T has been read out
          if (!mbar_wait(&sh.x_free, par ^ 1, a.err, 615)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16_ss_w(tmem + cP, iA + 2 * ks, gA + (oQI >> 4) + 2 * ks, hi, id_x, ks > 0);
          umma_commit(&sh.x_full);
          // dP^T = V dO^T into R, once every epilogue warp has loaded S^T
          if (!mbar_wait(&sh.s_read, par, a.err, 616)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ss_w(tmem + cR, vA + KSTEP(ks), gA + (oDO >> 4) + KSTEP(ks), hi, id_s, ks > 0);
          umma_commit(&sh.dp_full);
          // dV += P^T dO with P^T from TMEM (K = 128 rows, 16 per step; an MN-major step is 2048 bytes)
          if (!mbar_wait(&sh.p_ready, par, a.err, 617)) { ok = false; break; }
          if (j == 0 && !mbar_wait(&sh.acc_free, (it & 1) ^ 1, a.err, 618)) { ok = false; break; }
          tc_fence_after();
          const uint32_t acc = j > 0 ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ts_w(tmem + cDV, tmem + cP + ks * 8, gT + (oDO >> 4) + 128 * ks, hi, id_acc, acc | (ks > 0));
          umma_commit(&sh.pv_done);
          // dK += dS^T Q with dS^T from TMEM (packed bf16 in R's first 64 columns, K = 128 rows)
          if (!mbar_wait(&sh.ds_tmem, par, a.err, 619)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ts_w(tmem + cDK, tmem + cR + ks * 8, gT + (oQ >> 4) + 128 * ks, hi, id_acc, acc | (ks > 0));
          umma_commit(&sh.dk_done);
          // dQ^T = K^T dS^T into R, with dS^T's shared-memory copy (where dO was): it is the B operand
          if (!mbar_wait(&sh.ds_smem, par, a.err, 632)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ss_w(tmem + cR, kT + 128 * ks, gT + (oDO >> 4) + 128 * ks, hi, id_dq, ks > 0);
          umma_commit(&sh.dq_full);
          // index branch (gs^T, stored by the epilogue at the end of its stage C1, while dQ^T runs):
          // dk_idx += gs^T QI, dq_idx^T = KI^T gs^T into P, after dV has read P^T (same issuing thread: in
          // order). It goes before the next tile's S^T, which has slack, so that the warps reading dq_idx^T
          // find it done
          if (!mbar_wait(&sh.gs_ready, par, a.err, 620)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < npos / 16; ++ks)
            umma_bf16_ss_w2(tmem + cKI, gsA + 2 * ks, hiGS, gT + (oQI >> 4) + 128 * ks, hi, id_ki, acc | (ks > 0));
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ss_w2(tmem + cP, iT + 128 * ks, hi, gsB + ks * (2 * kGsAtom >> 4), hiGS, id_dqi, ks > 0);
#undef KSTEP
          umma_commit(&sh.ph2_full);
          if (j + 1 < ntiles) {  // the next tile's S^T, once this dQ^T has left R
            if (!issue_s(tj + 1)) { ok = false; break; }
            s_issued = true;
          }
        }
        umma_commit(&sh.kv_empty);
      }
      if (!ok) *abort_flag = 1;
    }
  }
  } else {
    regs_alloc192();
    // ------------------------------------------------------------ epilogue (thread = TMEM lane)
    const int quarter = warp & 3;
    const int hf = (warp >> 2) & 1;
    const int col0 = 64 * hf;                // this half's tile rows
    const int kk = quarter * 32 + lane;      // TMEM lane: key (S, dP, P, X), d (dQ^T), e (dq_idx^T)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t tj = 0;
    bool ok = true;
    int rel_gb = -1;  // gather buffer whose partial stores must finish reading before it is handed back
    for (int it = 0; ok; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!mbar_wait(&sh.it_full[s], ph, a.err, 621)) { ok = false; break; }
      const int4 item = sh.item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.it_empty[s]);
      if (item.x < 0) break;
      int b, g, c;
      decode_list(item.x, a.n, a.G, b, g, c);
      const int key = c * 128 + kk;
      const int ntiles = (item.z + npos - 1) / npos;
      for (int j = 0; j < ntiles; ++j, ++tj) {
        const int gb = tj & 1;
        const uint32_t par = tj & 1;
        uint8_t* buf = smem + oG + gb * kGather;
        const RowMeta& m = sh.meta[gb];
        if (!mbar_wait(&sh.g_full[gb], (tj >> 1) & 1, a.err, 622)) { ok = false; break; }
        if (!mbar_wait(&sh.s_full, par, a.err, 623)) { ok = false; break; }
        tc_fence_after();
        const int4 dg0 = *reinterpret_cast<const int4*>(m.diag);
        const int4 dg1 = *reinterpret_cast<const int4*>(m.diag + 4);
        const bool masked = (dg0.x | dg0.y | dg0.z | dg0.w | dg1.x | dg1.y | dg1.z | dg1.w) != 0;
        // ---- stage A: P = exp(s - LSE), zero on masked keys and padding rows; P^T into TMEM.
        // S^T goes back to the tensor core (for dP^T) as soon as it is in registers.
        float pv[64];
        tmem_ld32(tmem + lane_off + cR + col0, *reinterpret_cast<float(*)[32]>(pv));
        tmem_ld32(tmem + lane_off + cR + col0 + 32, *reinterpret_cast<float(*)[32]>(pv + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.s_read);  // R may take dP^T
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float4* l4 = reinterpret_cast<const float4*>(m.lse2 + col0 + 32 * h2);
          float* sv = pv + 32 * h2;
          if (!masked) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 l = l4[i];
              sv[4 * i + 0] = fast_exp2(fmaf(sv[4 * i + 0], a.scale_log2, -l.x));
              sv[4 * i + 1] = fast_exp2(fmaf(sv[4 * i + 1], a.scale_log2, -l.y));
              sv[4 * i + 2] = fast_exp2(fmaf(sv[4 * i + 2], a.scale_log2, -l.z));
              sv[4 * i + 3] = fast_exp2(fmaf(sv[4 * i + 3], a.scale_log2, -l.w));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 l = l4[i];
              const bool vis = key <= (m.ent[(col0 + 32 * h2 + 4 * i) / hg] >> 8);  // 4 rows: one query
              sv[4 * i + 0] = vis ? fast_exp2(fmaf(sv[4 * i + 0], a.scale_log2, -l.x)) : 0.f;
              sv[4 * i + 1] = vis ? fast_exp2(fmaf(sv[4 * i + 1], a.scale_log2, -l.y)) : 0.f;
              sv[4 * i + 2] = vis ? fast_exp2(fmaf(sv[4 * i + 2], a.scale_log2, -l.z)) : 0.f;
              sv[4 * i + 3] = vis ? fast_exp2(fmaf(sv[4 * i + 3], a.scale_log2, -l.w)) : 0.f;
            }
          }
        }
        // X^T is complete (and, since it was issued after them, every MMA of the previous tile,
        // the readers of the previous gs^T included)
        if (!mbar_wait(&sh.x_full, par, a.err, 633)) { ok = false; break; }
        tc_fence_after();
        // the previous tile's gather buffer goes back to the producers as early as it can: every MMA on it
        // is done (X^T of this tile was issued after them) and its partial stores, issued a stage ago, have
        // read their staging; the next tile's gather is what the tensor core waits for
        if (rel_gb >= 0) {
          if (lane == 0) {
            bulk_wait_read_all();
            mbar_arrive(&sh.g_empty[rel_gb]);
          }
          __syncwarp();
          rel_gb = -1;
        }
        float xv[kHQ];
        tmem_ld_cols<kHQ>(tmem + lane_off + cP + hf * kHQ, xv);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.x_read);  // X^T leaves the P columns once every warp has it
        if (!mbar_wait(&sh.x_read, par, a.err, 624)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t pk[32];  // this key's P^T row over the half's 64 rows, bf16 pairs (low half = even row)
#pragma unroll
          for (int z = 0; z < 32; ++z) pk[z] = pack_bf16(pv[2 * z], pv[2 * z + 1]);
          tmem_st32(tmem + lane_off + cP + 32 * hf, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_ready);
        // ---- stage B: dS = P (dP - D) * scale, bf16. Packed into R's first 64 columns (the
        // TMEM A operand of dK) once every warp has loaded dP^T, and copied into the dO area
        // (the B operand of dQ^T) once dV has read dO
        {
          uint32_t dsk[32];
          if (!mbar_wait(&sh.dp_full, par, a.err, 625)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float dp[32];
            tmem_ld32(tmem + lane_off + cR + col0 + 32 * h2, dp);
            tmem_wait_ld();
            const float4* d4 = reinterpret_cast<const float4*>(m.dsc + col0 + 32 * h2);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 dv = d4[i];
              const int r = 32 * h2 + 4 * i;
              dsk[16 * h2 + 2 * i] = pack_bf16(pv[r] * fmaf(dp[4 * i], a.scale, -dv.x),
                                               pv[r + 1] * fmaf(dp[4 * i + 1], a.scale, -dv.y));
              dsk[16 * h2 + 2 * i + 1] = pack_bf16(pv[r + 2] * fmaf(dp[4 * i + 2], a.scale, -dv.z),
                                                   pv[r + 3] * fmaf(dp[4 * i + 3], a.scale, -dv.w));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.dp_read);
          if (!mbar_wait(&sh.dp_read, par, a.err, 634)) { ok = false; break; }
          tc_fence_after();
          tmem_st32(tmem + lane_off + cR + 32 * hf, dsk);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.ds_tmem);
          if (!mbar_wait(&sh.pv_done, par, a.err, 626)) { ok = false; break; }
          uint8_t* dst = buf + oDO + hf * kChunk;  // dS^T rows [64 hf, 64 hf + 64) of key kk
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4*>(dst + sw128_off(kk, cc)) =
                make_uint4(dsk[4 * cc], dsk[4 * cc + 1], dsk[4 * cc + 2], dsk[4 * cc + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.ds_smem);
        }
        // ---- stage C1: index branch in registers (p_main, p_px, gs, KL terms), while dQ^T is computed
        float term[kHQ];
        uint32_t gp[kHQ / 2];  // this key's gs^T entries for the half's queries, bf16 pairs (low half = even query)
        {
          const float ws = a.kl_weight * a.scale_idx;
#pragma unroll
          for (int q2 = 0; q2 < kHQ / 2; ++q2) {
            float gsv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int qq = 2 * q2 + u;
              const int r = qq * hg;          // the query's first head row in this half
              const int q = col0 / hg + qq;   // the query in the tile
              float pm = 0.f;
#pragma unroll
              for (int h = 0; h < hg; ++h) pm += pv[r + h];
              pm *= 1.f / (float)hg;
              const float lpx2 = fmaf(xv[qq], a.scale_idx_log2, -m.lpx2[q]);  // log2 p_px
              float ppx = fast_exp2(lpx2);
              if (masked && key > (m.ent[q] >> 8)) ppx = 0.f;
              gsv[u] = ws * (ppx - pm);
              // p_main ln(p_main / p_px); p_main below the smallest normal float adds nothing visible
              term[qq] = pm >= 1.17549435e-38f ? pm * (fast_log2(pm) - lpx2) * kLn2 : 0.f;
            }
            gp[q2] = pack_bf16(gsv[0], gsv[1]);
          }
          // gs^T into shared memory for the index MMAs, issued right after dQ^T (the previous tile's, the
          // last readers of this image, were done before this tile's X^T)
          // gs^T row kk: 16-byte chunks of 8 queries, swizzled like the TMA image of the same width
          if constexpr (npos == 32) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
              *reinterpret_cast<uint4*>(smem + oGS + kk * 64 + (((2 * hf + cc) ^ ((kk >> 1) & 3)) << 4)) =
                  make_uint4(gp[4 * cc], gp[4 * cc + 1], gp[4 * cc + 2], gp[4 * cc + 3]);
          } else {
            *reinterpret_cast<uint4*>(smem + oGS + kk * 32 + ((hf ^ ((kk >> 2) & 1)) << 4)) =
                make_uint4(gp[0], gp[1], gp[2], gp[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.gs_ready);
        }
        // ---- stage D1: read out dQ^T (lane = d) as bf16 slot partials, staged where dS^T was
        // (dQ^T is its last reader); R goes back to the tensor core for the next tile's S^T
        const int pos0 = item.w + j * npos;  // padded entry of the tile's first query
        const int tq0 = item.y + j * npos;   // DENSE: the tile's first query
        if constexpr (DENSE) {
          // dQ^T (lane = d) added into dQ: fp32 rows staged where Q and dO were (dK and dQ^T, their last
          // readers, are done), one TMA reduce per warp (32 d x the half's 64 (query, head) rows)
          if (!mbar_wait(&sh.dq_full, par, a.err, 629)) { ok = false; break; }
          tc_fence_after();
          float* stg = reinterpret_cast<float*>(buf + oQ + (hf * 4 + quarter) * 8192);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float dq[32];
            tmem_ld32(tmem + lane_off + cR + col0 + 32 * h2, dq);
            tmem_wait_ld();
            if (h2 == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh.r_free);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) stg[(32 * h2 + i) * 32 + lane] = dq[i];
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&map_dq, stg, quarter * 32, g * hg, b * a.T + tq0 + hf * kHQ);
            bulk_commit();
          }
        } else {
          if (!mbar_wait(&sh.dq_full, par, a.err, 629)) { ok = false; break; }
          tc_fence_after();
          __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(buf + oDO + (hf * 4 + quarter) * 4096);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float dq[32];
            tmem_ld32(tmem + lane_off + cR + col0 + 32 * h2, dq);
            tmem_wait_ld();
            if (h2 == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh.r_free);  // R may take the next tile's S^T
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) stg[(32 * h2 + i) * 32 + lane] = __float2bfloat16_rn(dq[i]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_dq, stg, quarter * 32, pos0 * hg + col0);
            bulk_commit();
          }
        }
        // ---- stage C2: the KL terms summed over this warp's 32 keys (a butterfly over the lanes); each key
        // quarter writes its own sums, which the merge adds in order (the same bits in every run)
        {
          const int base = lanes_sum<kHQ>(term, lane);
          if ((lane & (LanesSum<kHQ>::kDup - 1)) == 0) {
#pragma unroll
            for (int i = 0; i < LanesSum<kHQ>::kKeep; ++i) {
              const int e = m.ent[hf * kHQ + base + i];
              if (e < 0) continue;
              if constexpr (DENSE)
                atomicAdd(a.KL + ((size_t)b * a.G + g) * a.T + (e >> 8), term[i]);
              else
                a.kl_part[((((size_t)b * a.T + (e >> 8)) * a.G + g) * a.k + (e & 255)) * 4 + quarter] = term[i];
            }
          }
        }
        // ---- stage D2: dq_idx^T (TMEM lanes 0..63) as bf16 slot partials, staged where Q was (dK,
        // its last reader, is done)
        {
          if (quarter < 2) {
            if (!mbar_wait(&sh.ph2_full, par, a.err, 630)) { ok = false; break; }
            tc_fence_after();
            float dqi[kHQ];
            tmem_ld_cols<kHQ>(tmem + lane_off + cP + hf * kHQ, dqi);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.x_free);  // P may take the next tile's X^T
            if constexpr (DENSE) {
              float* dst = a.dq_idx + (((size_t)b * a.T + tq0 + hf * kHQ) * a.G + g) * 64 + kk;
#pragma unroll
              for (int i = 0; i < kHQ; ++i) atomicAdd(dst + (size_t)i * a.G * 64, dqi[i]);
            } else {
            __nv_bfloat16* stq = reinterpret_cast<__nv_bfloat16*>(buf + oQ + (hf * 2 + quarter) * (kHQ * 64));
#pragma unroll
            for (int i = 0; i < kHQ; ++i) stq[i * 32 + lane] = __float2bfloat16_rn(dqi[i]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&map_dqi, stq, quarter * 32, pos0 + hf * kHQ);
              bulk_commit();
            }
            }
          }
          rel_gb = gb;
        }
      }
      if (!ok) break;
      // ---- list end: dV, dK (columns [64 hf, 64 hf + 64)) and dk_idx ([32 hf, 32 hf + 32)), lane = key.
      // dV and dK were final when this warp saw pv_done and dq_full of the last tile; dk_idx is final once
      // that tile's index MMAs are (only the warps of lanes 0..63 waited for them, for dq_idx^T)
      if (!mbar_wait(&sh.ph2_full, (tj - 1) & 1, a.err, 635)) { ok = false; break; }
      tc_fence_after();
      {
        const size_t orow = ((size_t)b * a.T + key) * a.G + g;
        // a dense item covers one segment of the block's queries: its sums are added
        auto put4 = [&](float* p, const float (&v)[32]) {
          float4* dst = reinterpret_cast<float4*>(p);
#pragma unroll
          for (int z = 0; z < 8; ++z) {
            const float4 x = make_float4(v[4 * z], v[4 * z + 1], v[4 * z + 2], v[4 * z + 3]);
            if constexpr (DENSE) atomicAdd(dst + z, x);
            else dst[z] = x;
          }
        };
        float v[32];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int d0 = 64 * hf + 32 * q;
          tmem_ld32(tmem + lane_off + cDV + d0, v);
          tmem_wait_ld();
          put4(a.dV + orow * 128 + d0, v);
          tmem_ld32(tmem + lane_off + cDK + d0, v);
          tmem_wait_ld();
          put4(a.dK + orow * 128 + d0, v);
        }
        tmem_ld32(tmem + lane_off + cKI + 32 * hf, v);
        tmem_wait_ld();
        if constexpr (DENSE) put4(a.dk_idx + ((size_t)b * a.T + key) * 64 + 32 * hf, v);  // summed over groups too
        else put4(a.dki_part + (((size_t)b * a.G + g) * a.T + key) * 64 + 32 * hf, v);
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
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

static cudaError_t set_wide_attributes() {
  static bool attr[kMaxDevices] = {};  // kernel attributes are per device context
  const int dslot = device_slot();
  cudaError_t e;
  if (!attr[dslot]) {
    for (auto f : {bwd_wide_kernel<4, false>, bwd_wide_kernel<8, false>, bwd_wide_kernel<4, true>,
                   bwd_wide_kernel<8, true>}) {
      if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess) return e;
      // the 64 / 192 register split redistributes exactly the 128 x 512 registers the block is launched
      // with; any other launch count would leave the epilogue's increase waiting for registers
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, f)) != cudaSuccess) return e;
      if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
    }
    attr[dslot] = true;
  }
  return cudaSuccess;
}

cudaError_t launch_bwd_wide(const BwdArgs& a, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mki,
                            const CUtensorMap& mdq, const CUtensorMap& mdqi, const CUtensorMap& mq,
                            const CUtensorMap& mdo, const CUtensorMap& mqi, cudaStream_t st) {
  cudaError_t e;
  if ((e = set_wide_attributes()) != cudaSuccess) return e;
  if (a.hg == 4)
    bwd_wide_kernel<4, false><<<num_sms(), kThreads, kSmem, st>>>(a, mk, mv, mki, mdq, mdqi, mq, mdo, mqi);
  else
    bwd_wide_kernel<8, false><<<num_sms(), kThreads, kSmem, st>>>(a, mk, mv, mki, mdq, mdqi, mq, mdo, mqi);
  return cudaGetLastError();
}

cudaError_t launch_bwd_wide_dense(const BwdArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                                  const CUtensorMap& mki, const CUtensorMap& mdq, const CUtensorMap& mq,
                                  const CUtensorMap& mdo, const CUtensorMap& mqi, cudaStream_t st) {
  cudaError_t e;
  if ((e = set_wide_attributes()) != cudaSuccess) return e;
  const int grid = std::min(a.dense_items, num_sms());
  if (a.hg == 4)
    bwd_wide_kernel<4, true><<<grid, kThreads, kSmem, st>>>(a, mk, mv, mki, mdq, mdq, mq, mdo, mqi);
  else
    bwd_wide_kernel<8, true><<<grid, kThreads, kSmem, st>>>(a, mk, mv, mki, mdq, mdq, mq, mdo, mqi);
  return cudaGetLastError();
}

}  // namespace msa
