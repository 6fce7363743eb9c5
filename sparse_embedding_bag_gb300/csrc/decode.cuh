// Per-tile decoding of lookups: which bag (and so which table) each lookup of
// a contiguous tile of `indices` belongs to, from the CSR offsets.
//
// The CSR layout is the one of "fbgemm_gpu/codegen/embedding_backward_split_template.cu"
// (offsets[t*B + b] .. offsets[t*B + b + 1] are the lookups of bag b of table t,
// tables major), expanded per lookup as in "tt_embeddings_cuda.cu",
// compute_rowidx_kernel. Here a block finds the bags that overlap its tile with
// a 256-way parallel search, then its warps expand those bags into a per-lookup
// bag id in shared memory (one warp per bag, 32 lookups per step).
#pragma once

#include "internal.cuh"

namespace embbwd {

// Largest j in [0, BT-1] with offsets[j] <= x, for x0 and x1 at once. Every
// thread of the block calls it and gets the same answers. Malformed (decreasing)
// offsets give some j in range; they are reported elsewhere.
__device__ __forceinline__ void block_bag_search2(const int64_t* __restrict__ off, uint32_t BT,
                                                  int64_t x0, int64_t x1, uint32_t* r0,
                                                  uint32_t* r1) {
  uint32_t lo0 = 0, hi0 = BT, lo1 = 0, hi1 = BT;
  while (hi0 - lo0 > 1 || hi1 - lo1 > 1) {
    const uint32_t n0 = hi0 - lo0, n1 = hi1 - lo1;
    const uint32_t st0 = (n0 + kThreads - 1) / kThreads, st1 = (n1 + kThreads - 1) / kThreads;
    const uint32_t j0 = lo0 + threadIdx.x * st0, j1 = lo1 + threadIdx.x * st1;
    const bool v0 = n0 > 1 && j0 < hi0 && off[j0] <= x0;
    const bool v1 = n1 > 1 && j1 < hi1 && off[j1] <= x1;
    int c0 = __syncthreads_count(v0);
    int c1 = __syncthreads_count(v1);
    if (n0 > 1) {
      if (c0 < 1) c0 = 1;
      const uint32_t b = lo0;
      lo0 = b + (uint32_t)(c0 - 1) * st0;
      hi0 = min(b + (uint32_t)c0 * st0, hi0);
    }
    if (n1 > 1) {
      if (c1 < 1) c1 = 1;
      const uint32_t b = lo1;
      lo1 = b + (uint32_t)(c1 - 1) * st1;
      hi1 = min(b + (uint32_t)c1 * st1, hi1);
    }
  }
  *r0 = lo0;
  *r1 = lo1;
}

// Fills s_bag[i - i0] with the bag id of every lookup i in [i0, i1) from the
// bags [bt_lo, bt_hi] that overlap the tile and, when s_len is not null,
// s_len[i - i0] with that bag's length. Ends with a barrier.
// The offsets of the overlapping bags are first staged in shared memory
// (s_off, room for off_cap entries) with one parallel load, so that the per-bag
// loop does not wait on a global load per bag; a window that does not fit is
// read from global memory directly.
__device__ __forceinline__ void expand_bag_range(const DecodeArgs& d, int64_t i0, int64_t i1,
                                                 uint32_t bt_lo, uint32_t bt_hi, uint32_t* s_bag,
                                                 uint32_t* s_len, int64_t* s_off, uint32_t off_cap) {
  if (bt_hi >= d.BT) bt_hi = d.BT - 1;
  if (bt_lo > bt_hi) bt_lo = bt_hi;
  const uint32_t span = bt_hi - bt_lo + 1;
  const bool staged = span + 1 <= off_cap;
  if (staged) {
    for (uint32_t k = threadIdx.x; k <= span; k += kThreads) s_off[k] = d.offsets[bt_lo + k];
    __syncthreads();
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint32_t bt = bt_lo + warp; bt <= bt_hi; bt += kWarps) {
    const int64_t a = staged ? s_off[bt - bt_lo] : d.offsets[bt];
    const int64_t e = staged ? s_off[bt - bt_lo + 1] : d.offsets[bt + 1];
    const int64_t lo = a > i0 ? a : i0;
    const int64_t hi = e < i1 ? e : i1;
    const uint32_t L = (uint32_t)(e - a);
    for (int64_t i = lo + lane; i < hi; i += 32) {
      s_bag[i - i0] = bt;
      if (s_len) s_len[i - i0] = L;
    }
  }
  __syncthreads();
}

// Same, finding the overlapping bags first. Contains barriers; returns the range.
__device__ __forceinline__ void expand_tile_bags(const DecodeArgs& d, int64_t i0, int64_t i1,
                                                 uint32_t* s_bag, uint32_t* s_len, int64_t* s_off,
                                                 uint32_t off_cap, uint32_t* lo_out = nullptr,
                                                 uint32_t* hi_out = nullptr) {
  uint32_t bt_lo, bt_hi;
  block_bag_search2(d.offsets, d.BT, i0, i1 - 1, &bt_lo, &bt_hi);
  if (bt_hi < bt_lo) bt_hi = bt_lo;
  if (lo_out) *lo_out = bt_lo;
  if (hi_out) *hi_out = bt_hi;
  expand_bag_range(d, i0, i1, bt_lo, bt_hi, s_bag, s_len, s_off, off_cap);
}

// Linear index (32-bit) of lookup `pos` whose bag is `bt`; sets *bad when the
// index falls outside its table. The table is clamped into range so that every
// later address stays in bounds even for malformed input.
__device__ __forceinline__ uint32_t linear_key(const DecodeArgs& d, const uint32_t* s_hsc,
                                               int64_t pos, uint32_t bt, uint32_t* t_out,
                                               bool* bad) {
  uint32_t t = div_by_B(bt, d.B, d.invB);
  if (t >= d.T) t = d.T - 1;
  const int64_t idx = d.indices[pos];
  const uint32_t base = s_hsc[t];
  const int64_t rows = (int64_t)(s_hsc[t + 1] - base);
  *bad = idx < 0 || idx >= rows;
  *t_out = t;
  return base + (uint32_t)idx;
}

}  // namespace embbwd
