// Pieces shared by the two fused-backward kernels (64-row tiles for 1 or 2
// heads per group, 128-row tiles for 4 or 8): the argument block, and the
// small device helpers of their epilogues.
#pragma once

#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {

constexpr float kBwdLog2e = 1.4426950408889634f;
constexpr float kBwdLn2 = 0.6931471805599453f;

struct BwdArgs {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* dO;
  const __nv_bfloat16* q_idx;
  const float* LSE;
  const float* drow;
  const float* lse_px;
  const int32_t* entries;
  const int4* items;
  const int* n_items;
  int* counter;
  int* err;
  float* dK;
  float* dV;
  __nv_bfloat16* dq_part;  // [padded entries, hg, d], tile order
  __nv_bfloat16* dqi_part; // [padded entries, E], tile order
  float* kl_part;          // [B,T,G,k,4]: per slot, the four key quarters' KL sums
  float* dki_part;         // [B,G,T,E]
  // Full attention (every query t >= 128 c sees block c): the lists are not
  // stored but cut into segments of dense_seg queries; the outputs are the
  // caller's, zeroed, and receive fp32 sums (dQ through the dq tensor map).
  float* dq_idx;           // [B,T,G,E]
  float* dk_idx;           // [B,T,E]
  float* KL;               // [B,G,T]
  int dense_seg;           // queries per segment, a multiple of 128
  int dense_per_b;         // work items per batch entry
  int dense_items;         // all work items
  int B, T, Hq, G, hg, n, k;
  float scale_log2, scale, scale_idx_log2, scale_idx, kl_weight;
};

// The 128-row-tile backward (heads per group 4 or 8). Tensor maps: K, V
// (box 64 x 1 x 128), k_idx (64 x 128), dQ partial store (32 x 64), dq_idx
// partial store (32 x queries per half tile), Q and dO (64 x hg x 1), q_idx (64 x 1).
cudaError_t launch_bwd_wide(const BwdArgs& a, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mki,
                            const CUtensorMap& mdq, const CUtensorMap& mdqi, const CUtensorMap& mq,
                            const CUtensorMap& mdo, const CUtensorMap& mqi, cudaStream_t st);

// The same kernel under full attention: mdq is an fp32 map of the caller's dQ
// ([B*T, Hq, d], box 32 x hg x queries per half tile) that the kernel adds into.
cudaError_t launch_bwd_wide_dense(const BwdArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                                  const CUtensorMap& mki, const CUtensorMap& mdq, const CUtensorMap& mq,
                                  const CUtensorMap& mdo, const CUtensorMap& mqi, cudaStream_t st);

namespace bwdc {

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void decode_list(int l, int n, int G, int& b, int& g, int& c) {
  const int bg = l / n;
  c = l - bg * n;
  b = bg / G;
  g = bg - b * G;
}

// Sum over the 32 lanes of NV per-lane values, with a butterfly that halves
// the values a lane keeps at each step (NV - 1 shuffles instead of 5 NV). On
// return the lanes with lane % kDup == 0 hold in v[0 .. kKeep) the sums of the
// values [base, base + kKeep); the function returns base.
template <int NV>
struct LanesSum {
  static constexpr int kKeep = NV >= 32 ? NV / 32 : 1;
  static constexpr int kDup = NV >= 32 ? 1 : 32 / NV;  // lanes holding the same sums
};
template <int NV>
__device__ __forceinline__ int lanes_sum(float (&v)[NV], int lane) {
  int base = 0;
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int off = 16 >> s;
    constexpr int kNV = NV;
    const int n = kNV >> s;
    if (n >= 2) {
      const int half = n >> 1;
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < (kNV >> (s + 1)); ++i) {
        const float send = up ? v[i] : v[i + half];
        const float keep = up ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
      if (up) base += half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  return base;
}

}  // namespace bwdc
}  // namespace msa
