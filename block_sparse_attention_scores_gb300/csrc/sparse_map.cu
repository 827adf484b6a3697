// Inverted block -> query map of the selected blocks (CSR per (b, g, block)).
//
// dothoosh.com "how Flash-MSA cuts million-token training cost", "Kernel
// design and execution": inverting the block-index map lets the kernels
// schedule, for each sparse KV block, the query chunks that selected it, so
// the block is staged in shared memory once and reused by all of them.
//
// Lists are keyed by l = (b * G + g) * n + c. Entry = (t << 8) | slot, where
// slot is the position of c in block_idx[b, g, t, :]. Build:
//   1. count   -- validate every row, count selections per list (atomics)
//   2. scan    -- exclusive prefix over lists; emit work items in descending
//                 list-length order (block id ascending first, which is the
//                 order of decreasing expected length)
//   3. scatter -- place entries with per-list cursors (atomics)
//   4. sort    -- sort each list by t (deterministic order; lists longer than
//                 the shared-memory buffer keep scatter order, which changes
//                 only the fp32 summation order downstream), and record the
//                 reverse map (b, g, t, slot) -> padded entry index, so the
//                 kernels can write per-(query, slot) partials in tile order
//                 (whole tiles, one TMA store each) and the merges find them
#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {
namespace {

// Checks one block_idx row: ascending distinct ids in [0, own], own present,
// -1 padding only at the end. Returns the number of valid ids or -1.
__device__ __forceinline__ int check_row(const int32_t* row, int k, int own) {
  int nvalid = 0, prev = -1;
  bool pad = false, ok = true, has_own = false;
  for (int i = 0; i < k; ++i) {
    const int c = row[i];
    if (c < 0) {
      pad = true;
      ok &= (c == -1);
      continue;
    }
    ok &= !pad && c > prev && c <= own;
    has_own |= (c == own);
    prev = c;
    ++nvalid;
  }
  return (ok && has_own) ? nvalid : -1;
}

__global__ void map_count_kernel(const int32_t* __restrict__ block_idx, int B, int G, int T, int n, int k,
                                 int* __restrict__ count, int* err) {
  const long long rows = (long long)B * G * T;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(r % T);
    const long long bg = r / T;
    const int32_t* row = block_idx + r * k;
    if (check_row(row, k, t / 128) < 0) {
      dev_fail(err, kDevBadIndex, 201);
      continue;
    }
    for (int i = 0; i < k; ++i) {
      const int c = row[i];
      if (c >= 0) atomicAdd(&count[bg * n + c], 1);
    }
  }
}

// Exclusive scan of one value per thread across a 1024-thread block, chained
// through `carry` (block-uniform running total).
__device__ __forceinline__ int block_scan_excl(int v, int* warp_sums, int* carry) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int excl = *carry + (wid ? warp_sums[wid - 1] : 0) + x - v;
  __syncthreads();
  if (tid == 1023) *carry = excl + v;
  __syncthreads();
  return excl;
}

// Single CTA. Exclusive scans of list lengths (entry offsets) and of list
// lengths padded to whole tiles (partial-output row offsets), both in list
// order; then of work items in block-id-major order, and the items:
// int4 {list, first entry, entries, padded offset of the first entry}.
__global__ void __launch_bounds__(1024) map_scan_kernel(const int* __restrict__ count, int L, int BG, int n,
                                                        int rows_per_tile, int tiles_per_item,
                                                        int* __restrict__ off, int* __restrict__ poff,
                                                        int4* __restrict__ items, int max_items,
                                                        int* __restrict__ n_items, int* err) {
  __shared__ int warp_sums[32];
  __shared__ int carry, pcarry;
  const int tid = threadIdx.x;
  const long long per_item_ll = (long long)rows_per_tile * tiles_per_item;
  const int per_item = per_item_ll > (1 << 30) ? (1 << 30) : (int)per_item_ll;
  if (tid == 0) carry = pcarry = 0;
  __syncthreads();
  for (int base = 0; base < L; base += 1024) {
    const int i = base + tid;
    const int v = i < L ? count[i] : 0;
    const int pv = (v + rows_per_tile - 1) / rows_per_tile * rows_per_tile;
    const int e = block_scan_excl(v, warp_sums, &carry);
    const int pe = block_scan_excl(pv, warp_sums, &pcarry);
    if (i < L) {
      off[i] = e;
      poff[i] = pe;
    }
  }
  if (tid == 0) {
    off[L] = carry;
    poff[L] = pcarry;
    carry = 0;
  }
  __syncthreads();
  for (int base = 0; base < L; base += 1024) {
    const int j = base + tid;  // block-id-major index
    int v = 0, lid = 0;
    if (j < L) {
      const int c = j / BG, bg = j % BG;
      lid = bg * n + c;
      v = (count[lid] + per_item - 1) / per_item;
    }
    const int first = block_scan_excl(v, warp_sums, &carry);
    if (j < L) {
      const int len = count[lid], start = off[lid], pstart = poff[lid];
      for (int q = 0; q < v; ++q) {
        const int it = first + q;
        if (it < max_items) {
          const int e0 = q * per_item;
          items[it] = make_int4(lid, start + e0, min(per_item, len - e0), pstart + e0);
        } else {
          dev_fail(err, kDevBadIndex, 202);
        }
      }
    }
  }
  if (tid == 0) *n_items = min(carry, max_items);
}

__global__ void map_scatter_kernel(const int32_t* __restrict__ block_idx, int B, int G, int T, int n, int k,
                                   const int* __restrict__ off, int* __restrict__ cursor,
                                   int32_t* __restrict__ entries) {
  const long long rows = (long long)B * G * T;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(r % T);
    const long long bg = r / T;
    const int32_t* row = block_idx + r * k;
    if (check_row(row, k, t / 128) < 0) continue;
    for (int i = 0; i < k; ++i) {
      const int c = row[i];
      if (c < 0) continue;
      const long long l = bg * n + c;
      const int pos = atomicAdd(&cursor[l], 1);
      entries[off[l] + pos] = (t << 8) | i;
    }
  }
}

constexpr int kSortCap = 16384;

// Sorts each list by query (lists up to kSortCap entries; longer ones keep
// scatter order), then records for every (b, g, t, slot) the padded
// partial-output index of its entry: rev[(bg * T + t) * k + slot].
__global__ void __launch_bounds__(1024) map_sort_kernel(const int* __restrict__ off, const int* __restrict__ poff,
                                                        int L, int n, int T, int k, int32_t* __restrict__ entries,
                                                        int32_t* __restrict__ rev) {
  extern __shared__ int32_t keys[];
  for (int l = blockIdx.x; l < L; l += gridDim.x) {
    const int start = off[l], len = off[l + 1] - start;
    if (len > 1 && len <= kSortCap) {
      int np = 1;
      while (np < len) np <<= 1;
      for (int i = threadIdx.x; i < np; i += blockDim.x) keys[i] = i < len ? entries[start + i] : 0x7fffffff;
      __syncthreads();
      for (int size = 2; size <= np; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int i = threadIdx.x; i < np / 2; i += blockDim.x) {
            const int lo = 2 * i - (i & (stride - 1));
            const int hi = lo + stride;
            const bool up = ((lo & size) == 0);
            const int a = keys[lo], b = keys[hi];
            if ((a > b) == up) {
              keys[lo] = b;
              keys[hi] = a;
            }
          }
          __syncthreads();
        }
      }
      for (int i = threadIdx.x; i < len; i += blockDim.x) entries[start + i] = keys[i];
      __syncthreads();
    }
    const long long bg = l / n;
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
      const int e = entries[start + i];
      rev[(bg * T + (e >> 8)) * k + (e & 255)] = poff[l] + i;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t build_block_map(const Prob& p, const int32_t* block_idx, uint8_t* ws, const WsLayout& L,
                            int rows_per_tile, int tiles_per_item, cudaStream_t st) {
  const int lists = p.B * p.G * p.n;
  int* count = reinterpret_cast<int*>(ws + L.list_count);
  int* off = reinterpret_cast<int*>(ws + L.list_off);
  int* cursor = reinterpret_cast<int*>(ws + L.list_cursor);
  int* poff = reinterpret_cast<int*>(ws + L.list_poff);
  int32_t* rev = reinterpret_cast<int32_t*>(ws + L.rev);
  int32_t* entries = reinterpret_cast<int32_t*>(ws + L.entries);
  int4* items = reinterpret_cast<int4*>(ws + L.items);
  int* n_items = reinterpret_cast<int*>(ws + L.n_items);
  int* err = reinterpret_cast<int*>(ws + L.err);
  cudaError_t e;
  if ((e = cudaMemsetAsync(count, 0, (size_t)lists * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(cursor, 0, (size_t)lists * 4, st)) != cudaSuccess) return e;
  // rows that fail validation never get an entry: their reverse-map slots stay -1
  if ((e = cudaMemsetAsync(rev, 0xff, (size_t)p.B * p.G * p.T * p.k * 4, st)) != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.G * p.T;
  const int grid = (int)std::min<long long>((rows + 255) / 256, 8LL * num_sms());
  map_count_kernel<<<grid, 256, 0, st>>>(block_idx, p.B, p.G, p.T, p.n, p.k, count, err);
  map_scan_kernel<<<1, 1024, 0, st>>>(count, lists, p.B * p.G, p.n, rows_per_tile, tiles_per_item, off, poff,
                                      items, L.max_items, n_items, err);
  map_scatter_kernel<<<grid, 256, 0, st>>>(block_idx, p.B, p.G, p.T, p.n, p.k, off, cursor, entries);
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(map_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSortCap * 4)) !=
        cudaSuccess)
      return e;
    attr_set = true;
  }
  map_sort_kernel<<<std::min(lists, 4 * num_sms()), 1024, kSortCap * 4, st>>>(off, poff, lists, p.n, p.T, p.k,
                                                                              entries, rev);
  count_launches(4);
  return cudaGetLastError();
}

}  // namespace msa
