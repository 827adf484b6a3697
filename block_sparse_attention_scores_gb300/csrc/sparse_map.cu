// Inverted block -> query map of the selected blocks (CSR per (b, g, block)).
//
// dothoosh.com "how Flash-MSA cuts million-token training cost", "Kernel
// design and execution": inverting the block-index map lets the kernels
// schedule, for each sparse KV block, the query chunks that selected it, so
// the block is staged in shared memory once and reused by all of them.
//
// Lists are keyed by l = (b * G + g) * n + c. Entry = (t << 8) | slot, where
// slot is the position of c in block_idx[b, g, t, :]. Every list comes out
// sorted by t, with no atomics on global counters and no sort pass: the
// queries are cut into chunks of 128 (one query block qb), and a chunk only
// selects blocks c <= qb. Build:
//   1. chunk count -- one CTA per (b, g, qb): validate its 128 rows, mark in
//                     shared bitmaps which rows select each block c, write the
//                     popcounts to chunk_off[(b, g), c, qb] (upper triangle)
//   2. chunk scan  -- per list: exclusive prefix over qb (the chunk's first
//                     position in the list) and the list length
//   3. list scan   -- exclusive prefix over lists (and over lists padded to
//                     whole tiles); work items (b, g)-major, block id ascending
//                     within a (b, g): the order of decreasing expected list
//                     length
//   4. scatter     -- one CTA per chunk again: an entry's position is its
//                     chunk's offset plus the rows before it in the bitmap;
//                     also the reverse map (b, g, t, slot) -> padded entry
//                     index, so the kernels write per-(query, slot) partials in
//                     tile order and the merges find them
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

// Position of (block c, query block qb), 0 <= c <= qb < n, in one (b, g)'s
// upper triangle, stored list-major: the chunks of list c are contiguous.
__device__ __forceinline__ long long tri_index(int c, int qb, int n) {
  return (long long)c * n - (long long)c * (c - 1) / 2 + (qb - c);
}

// Shared bitmaps of one chunk: bit (row) of mask[4 c .. 4 c + 3] is set when
// that row of the chunk selects block c. Returns false for an invalid row.
__device__ __forceinline__ bool chunk_masks(const int32_t* __restrict__ block_idx, long long bg, int qb, int T,
                                            int k, uint32_t* mask, int* err, int where) {
  const int tl = threadIdx.x;
  for (int i = tl; i < (qb + 1) * 4; i += 128) mask[i] = 0u;
  __syncthreads();
  const int32_t* row = block_idx + ((size_t)bg * T + (size_t)qb * 128 + tl) * k;
  const bool valid = check_row(row, k, qb) >= 0;
  if (!valid) {
    dev_fail(err, kDevBadIndex, where);
  } else {
    for (int i = 0; i < k; ++i) {
      const int c = row[i];
      if (c >= 0) atomicOr(&mask[c * 4 + (tl >> 5)], 1u << (tl & 31));
    }
  }
  __syncthreads();
  return valid;
}

// One CTA (128 threads = rows) per (b, g, qb).
__global__ void __launch_bounds__(128) map_chunk_count_kernel(const int32_t* __restrict__ block_idx, int T, int n,
                                                              int k, int* __restrict__ chunk_off, int* err) {
  extern __shared__ uint32_t mask[];
  const int qb = blockIdx.x % n;
  const long long bg = blockIdx.x / n;
  chunk_masks(block_idx, bg, qb, T, k, mask, err, 201);
  int* tri = chunk_off + bg * ((long long)n * (n + 1) / 2);
  for (int c = threadIdx.x; c <= qb; c += 128)
    tri[tri_index(c, qb, n)] =
        __popc(mask[4 * c]) + __popc(mask[4 * c + 1]) + __popc(mask[4 * c + 2]) + __popc(mask[4 * c + 3]);
}

// One warp per list (bg, c): exclusive prefix of its chunk counts over qb, in
// place, and the list length.
__global__ void map_chunk_scan_kernel(int L, int n, int* __restrict__ chunk_off, int* __restrict__ count) {
  const int lane = threadIdx.x & 31;
  for (long long l = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; l < L;
       l += ((long long)gridDim.x * blockDim.x) >> 5) {
    const long long bg = l / n;
    const int c = (int)(l - bg * n);
    int* run = chunk_off + bg * ((long long)n * (n + 1) / 2) + tri_index(c, c, n);
    const int len = n - c;
    int carry = 0;
    for (int base = 0; base < len; base += 32) {
      const int i = base + lane;
      const int v = i < len ? run[i] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (i < len) run[i] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) count[l] = carry;
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

// Work items of one kernel, (b, g)-major and block id ascending within a
// (b, g) (the order of decreasing expected list length): int4 {list, first
// entry, entries, padded offset of the first entry}, at most per_item entries
// each. The CTAs running together then gather the query rows of one (b, g),
// which L2 holds far better than the rows of every group. Called by one CTA
// of 1024 threads; `carry` is block-uniform scratch.
__device__ void emit_items(const int* __restrict__ count, const int* __restrict__ off,
                           const int* __restrict__ poff, int L, int BG, int n, int per_item,
                           int4* __restrict__ items, int max_items, int* __restrict__ n_items, int* err,
                           int* warp_sums, int* carry) {
  const int tid = threadIdx.x;
  if (tid == 0) *carry = 0;
  __syncthreads();
  for (int base = 0; base < L; base += 1024) {
    const int j = base + tid;  // (b, g)-major index: list id
    int v = 0, lid = 0;
    if (j < L) {
      lid = j;
      v = (count[lid] + per_item - 1) / per_item;
    }
    const int first = block_scan_excl(v, warp_sums, carry);
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
  if (tid == 0) *n_items = min(*carry, max_items);
  __syncthreads();
}

// Single CTA. Exclusive scans of list lengths (entry offsets) and of list
// lengths padded to whole tiles of pad_rows entries (partial-output row
// offsets), both in list order; then the work items of one kernel, and of a
// second one when items_b is given (a map shared by the forward and the
// backward).
__global__ void __launch_bounds__(1024) map_scan_kernel(const int* __restrict__ count, int L, int BG, int n,
                                                        int pad_rows, int per_item_a, int per_item_b,
                                                        int* __restrict__ off, int* __restrict__ poff,
                                                        int4* __restrict__ items_a, int4* __restrict__ items_b,
                                                        int max_items, int* __restrict__ n_items, int* err) {
  __shared__ int warp_sums[32];
  __shared__ int carry, pcarry;
  const int tid = threadIdx.x;
  if (tid == 0) carry = pcarry = 0;
  __syncthreads();
  for (int base = 0; base < L; base += 1024) {
    const int i = base + tid;
    const int v = i < L ? count[i] : 0;
    const int pv = (v + pad_rows - 1) / pad_rows * pad_rows;
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
  }
  __syncthreads();
  emit_items(count, off, poff, L, BG, n, per_item_a, items_a, max_items, n_items, err, warp_sums, &carry);
  if (items_b) emit_items(count, off, poff, L, BG, n, per_item_b, items_b, max_items, n_items + 1, err, warp_sums,
                          &carry);
}

// One CTA (128 threads = rows) per (b, g, qb): entries in query order and
// the reverse map.
__global__ void __launch_bounds__(128) map_chunk_scatter_kernel(const int32_t* __restrict__ block_idx, int T, int n,
                                                                int k, const int* __restrict__ chunk_off,
                                                                const int* __restrict__ off,
                                                                const int* __restrict__ poff,
                                                                int32_t* __restrict__ entries,
                                                                int32_t* __restrict__ rev, int* err) {
  extern __shared__ uint32_t mask[];
  const int qb = blockIdx.x % n;
  const long long bg = blockIdx.x / n;
  if (!chunk_masks(block_idx, bg, qb, T, k, mask, err, 203)) return;  // after the last barrier
  const int tl = threadIdx.x, t = qb * 128 + tl;
  const int w = tl >> 5;
  const uint32_t below = (1u << (tl & 31)) - 1u;
  const int* tri = chunk_off + bg * ((long long)n * (n + 1) / 2);
  const size_t rrow = ((size_t)bg * T + t) * k;
  for (int i = 0; i < k; ++i) {
    const int c = block_idx[rrow + i];
    if (c < 0) continue;
    const uint32_t* mk = mask + 4 * c;
    int rank = __popc(mk[w] & below);
    for (int u = 0; u < w; ++u) rank += __popc(mk[u]);
    const long long l = bg * n + c;
    const int pos = tri[tri_index(c, qb, n)] + rank;  // position within the list
    entries[off[l] + pos] = (t << 8) | i;
    rev[rrow + i] = poff[l] + pos;
  }
}

// Selection of full causal attention: row (b, g, t) lists the blocks
// 0 .. t / Bk ascending, then -1 (k >= number of blocks, checked by the caller).
__global__ void warmup_block_idx_kernel(int32_t* __restrict__ block_idx, long long rows, int T, int Bk, int k) {
  const long long total = rows * k;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / k;
    const int slot = (int)(i - row * k);
    const int own = (int)(row % T) / Bk;
    block_idx[i] = slot <= own ? slot : -1;
  }
}

}  // namespace

cudaError_t build_block_map(const Prob& p, const int32_t* block_idx, uint8_t* ws, const WsLayout& L,
                            int rows_per_tile, int tiles_per_item, cudaStream_t st) {
  return build_block_map2(p, block_idx, ws, L, rows_per_tile, rows_per_tile * tiles_per_item, 0, false, st);
}

cudaError_t build_block_map2(const Prob& p, const int32_t* block_idx, uint8_t* ws, const WsLayout& L, int pad_rows,
                             long long per_item_a, long long per_item_b, bool two_lists, cudaStream_t st) {
  const int lists = p.B * p.G * p.n;
  int* count = reinterpret_cast<int*>(ws + L.list_count);
  int* off = reinterpret_cast<int*>(ws + L.list_off);
  int* chunk = reinterpret_cast<int*>(ws + L.chunk_off);
  int* poff = reinterpret_cast<int*>(ws + L.list_poff);
  int32_t* rev = reinterpret_cast<int32_t*>(ws + L.rev);
  int32_t* entries = reinterpret_cast<int32_t*>(ws + L.entries);
  int4* items = reinterpret_cast<int4*>(ws + L.items);
  int* n_items = reinterpret_cast<int*>(ws + L.n_items);
  int* err = reinterpret_cast<int*>(ws + L.err);
  cudaError_t e;
  // rows that fail validation never get an entry: their reverse-map slots stay -1
  if ((e = cudaMemsetAsync(rev, 0xff, (size_t)p.B * p.G * p.T * p.k * 4, st)) != cudaSuccess) return e;
  const int chunks = p.B * p.G * p.n;  // one per (b, g, query block)
  const int mask_bytes = p.n * 16;     // bitmaps of blocks 0..qb, 128 rows each
  static int attr_bytes[kMaxDevices] = {};  // kernel attributes are per device context
  const int dslot = device_slot();
  if (mask_bytes > 48 * 1024 && mask_bytes > attr_bytes[dslot]) {
    if ((e = cudaFuncSetAttribute(map_chunk_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  mask_bytes)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(map_chunk_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  mask_bytes)) != cudaSuccess)
      return e;
    attr_bytes[dslot] = mask_bytes;
  }
  map_chunk_count_kernel<<<chunks, 128, mask_bytes, st>>>(block_idx, p.T, p.n, p.k, chunk, err);
  map_chunk_scan_kernel<<<(int)std::min<long long>(((long long)lists * 32 + 255) / 256, 16LL * num_sms()), 256, 0,
                          st>>>(lists, p.n, chunk, count);
  auto clamp = [](long long v) { return v > (1 << 30) ? (1 << 30) : (int)v; };
  int4* items_b = two_lists ? reinterpret_cast<int4*>(ws + L.items2) : nullptr;
  map_scan_kernel<<<1, 1024, 0, st>>>(count, lists, p.B * p.G, p.n, pad_rows, clamp(per_item_a), clamp(per_item_b),
                                      off, poff, items, items_b, L.max_items, n_items, err);
  map_chunk_scatter_kernel<<<chunks, 128, mask_bytes, st>>>(block_idx, p.T, p.n, p.k, chunk, off, poff, entries,
                                                             rev, err);
  count_launches(4);
  return cudaGetLastError();
}

cudaError_t launch_warmup_block_idx(const Prob& p, int32_t* block_idx, cudaStream_t st) {
  const long long rows = (long long)p.B * p.G * p.T;
  const int grid = (int)std::min<long long>((rows * p.k + 255) / 256, 8LL * num_sms());
  warmup_block_idx_kernel<<<grid, 256, 0, st>>>(block_idx, rows, p.T, p.Bk, p.k);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
