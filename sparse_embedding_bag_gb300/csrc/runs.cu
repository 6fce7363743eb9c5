// Run-length encoding of the sorted linear indices and the long-run partition.
//
// k_rle: the unique sorted linear indices, the start of every run (the
//   exclusive scan of the run lengths) and the number of runs -- the outputs
//   "fbgemm_gpu/codegen/embedding_backward_split_template.cu" takes from its
//   transpose step (sorted_linear_indices_run, ..._cumulative_run_lengths,
//   ..._num_runs). One pass: each block flags run heads in its tile, counts them
//   and gets the count of all earlier tiles by decoupled look-back.
// k_long: the set of runs with at least max_segment_length_per_warp lookups
//   (that page's *_find_long_segments), produced as an ordered compaction
//   instead of an atomic append, together with the block work items for them:
//   a run is cut into parts of `part` lookups, and runs with more than one part
//   get a slot per part for fp32 partial sums that the last part to finish
//   combines in part order.
#include "internal.cuh"

namespace embbwd {

namespace {

__global__ void __launch_bounds__(kThreads) k_rle(RleArgs a) {
  __shared__ uint32_t s_tile;
  __shared__ uint32_t s_scan[kWarps];
  __shared__ uint32_t s_base;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) s_tile = atomicAdd(&a.ctl->tile_ctr[TC_RLE], 1u);
  __syncthreads();
  const uint32_t tile = s_tile;
  const int64_t i0 = (int64_t)tile * kRleTile;
  const int64_t p0 = i0 + (int64_t)threadIdx.x * kRleItems;

  uint32_t key[kRleItems];
  if (p0 + kRleItems <= a.N) {
    const uint4 u0 = *reinterpret_cast<const uint4*>(a.keys + p0);
    const uint4 u1 = *reinterpret_cast<const uint4*>(a.keys + p0 + 4);
    key[0] = u0.x; key[1] = u0.y; key[2] = u0.z; key[3] = u0.w;
    key[4] = u1.x; key[5] = u1.y; key[6] = u1.z; key[7] = u1.w;
  } else {
#pragma unroll
    for (int k = 0; k < kRleItems; ++k) key[k] = p0 + k < a.N ? a.keys[p0 + k] : 0u;
  }
  uint32_t prev = 0;
  if (p0 > 0 && p0 <= a.N) prev = a.keys[p0 - 1];
  uint32_t heads = 0;  // bit k: position p0+k starts a run
#pragma unroll
  for (int k = 0; k < kRleItems; ++k) {
    const int64_t p = p0 + k;
    const uint32_t before = k == 0 ? prev : key[k - 1];
    if (p < a.N && (p == 0 || key[k] != before)) heads |= 1u << k;
  }
  uint32_t total;
  const uint32_t excl_thread = block_excl_scan(__popc(heads), s_scan, &total);
  if (threadIdx.x < 32) {
    const uint32_t b = lookback_warp(a.lb, tile, 1, 0, total, a.ctl, a.sticky);
    if (threadIdx.x == 0) s_base = b;
  }
  __syncthreads();
  const uint32_t base = s_base;
  uint32_t r = base + excl_thread;
#pragma unroll
  for (int k = 0; k < kRleItems; ++k) {
    if (heads & (1u << k)) {
      if (r < (uint64_t)a.N) {
        a.run_key[r] = key[k];
        a.run_start[r] = (uint32_t)(p0 + k);
      }
      ++r;
    }
  }
  if (i0 + kRleTile >= a.N && threadIdx.x == 0) {
    const uint32_t U = base + total;
    if (U <= (uint64_t)a.N) {
      a.ctl->num_runs = U;
      a.run_start[U] = (uint32_t)a.N;
    } else {
      raise_error(a.ctl, a.sticky, kErrCapacity);
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_long(LongArgs a) {
  __shared__ uint32_t s_tile;
  __shared__ uint32_t s_scan[kWarps];
  __shared__ uint32_t s_base[3];
  pdl_wait();
  pdl_trigger();
  const uint32_t U = *(volatile uint32_t*)&a.ctl->num_runs;
  for (;;) {
    if (threadIdx.x == 0) s_tile = atomicAdd(&a.ctl->tile_ctr[TC_LONG], 1u);
    __syncthreads();
    const uint32_t tile = s_tile;
    const uint64_t r0 = (uint64_t)tile * kLongTile;
    if (r0 >= U) break;
    const uint64_t rt = r0 + (uint64_t)threadIdx.x * kLongItems;
    uint32_t n_long = 0, n_items = 0, n_slots = 0;
    uint32_t parts[kLongItems];
#pragma unroll
    for (int k = 0; k < kLongItems; ++k) {
      parts[k] = 0;
      const uint64_t r = rt + k;
      if (r < U) {
        const uint32_t SL = a.run_start[r + 1] - a.run_start[r];
        if (SL >= a.thr) {
          parts[k] = (SL + a.part - 1) / a.part;
          n_long += 1;
          n_items += parts[k];
          if (parts[k] > 1) n_slots += parts[k];
        }
      }
    }
    uint32_t t_long, t_items, t_slots;
    const uint32_t e_long = block_excl_scan(n_long, s_scan, &t_long);
    const uint32_t e_items = block_excl_scan(n_items, s_scan, &t_items);
    const uint32_t e_slots = block_excl_scan(n_slots, s_scan, &t_slots);
    const uint32_t warp = threadIdx.x >> 5;
    if (warp < 3) {  // one warp per channel
      const uint32_t agg = warp == 0 ? t_long : (warp == 1 ? t_items : t_slots);
      const uint32_t b = lookback_warp(a.lb, tile, 3, warp, agg, a.ctl, a.sticky);
      if ((threadIdx.x & 31) == 0) s_base[warp] = b;
    }
    __syncthreads();
    uint32_t kl = s_base[0] + e_long, ki = s_base[1] + e_items, ks = s_base[2] + e_slots;
    bool overflow = false;
#pragma unroll
    for (int k = 0; k < kLongItems; ++k) {
      if (parts[k]) {
        if (kl < a.cap_long && ki + parts[k] <= a.cap_items &&
            (parts[k] == 1 || ks + parts[k] <= a.cap_slots)) {
          a.long_ids[kl] = (uint32_t)(rt + k);
          a.item_base[kl] = ki;
          a.slot_base[kl] = ks;
          for (uint32_t p = 0; p < parts[k]; ++p) a.item_long[ki + p] = kl;
        } else {
          overflow = true;
        }
        kl += 1;
        ki += parts[k];
        if (parts[k] > 1) ks += parts[k];
      }
    }
    if (overflow) raise_error(a.ctl, a.sticky, kErrCapacity);
    if (r0 + kLongTile >= U && threadIdx.x == 0) {
      a.ctl->num_long = s_base[0] + t_long;
      a.ctl->num_items = s_base[1] + t_items;
      a.ctl->num_slots = s_base[2] + t_slots;
    }
    __syncthreads();  // s_tile / s_base are rewritten by the next tile
  }
}

}  // namespace

cudaError_t launch_rle(const RleArgs& a, cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)((a.N + kRleTile - 1) / kRleTile);
  RleArgs arg = a;
  void* args[] = {&arg};
  return launch_kernel(reinterpret_cast<const void*>(&k_rle), dim3(grid), dim3(kThreads), 0, s, args, pdl);
}

cudaError_t launch_long(const LongArgs& a, int grid, cudaStream_t s, bool pdl) {
  LongArgs arg = a;
  void* args[] = {&arg};
  return launch_kernel(reinterpret_cast<const void*>(&k_long), dim3(grid), dim3(kThreads), 0, s, args, pdl);
}

}  // namespace embbwd
