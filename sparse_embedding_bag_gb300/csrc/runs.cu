// Run-length encoding of the sorted linear indices fused with the long-run
// partition, in one pass over the sorted keys.
//
// Outputs, as in "fbgemm_gpu/codegen/embedding_backward_split_template.cu":
//   * the unique sorted linear indices, the start of every run (the exclusive
//     scan of the run lengths, last entry N) and the number of runs (that
//     page's sorted_linear_indices_run / _cumulative_run_lengths / _num_runs);
//   * the runs with at least max_segment_length_per_warp lookups (that page's
//     *_find_long_segments), as an ordered compaction instead of an atomic
//     append, each with its place in the concatenation of all long runs (the
//     prefix sum of their lengths), which the reduce cuts into equal slices.
//
// Each block owns a tile of 256 * ITEMS sorted keys and the runs whose first
// lookup lies in it. A run that continues past the tile end has its end found
// by a 32-lane parallel upper-bound search (a few rounds of one load per lane),
// so every run's length is known inside the block that owns it. When the tables
// form several segments (groups of consecutive tables the reduce treats alike),
// a run whose key is the first of its segment (or follows empty segments)
// records, for each segment it opens, that segment's first run. The three
// counts (runs, long runs, lookups in long runs) of earlier tiles come from one
// decoupled look-back per count, each walked 32 tiles at a time by a warp.
#include "internal.cuh"

namespace embbwd {

namespace {

// First position >= b whose key differs from k (or N), given that position b-1
// holds k. Called by all lanes of one warp; every lane gets the answer.
__device__ __forceinline__ uint32_t run_end_search(const uint32_t* __restrict__ keys, uint32_t N,
                                                   uint32_t b, uint32_t k) {
  const uint32_t lane = threadIdx.x & 31;
  if (b >= N) return N;
  // exponential probe: lane l tests b - 1 + 2^l
  const uint64_t q = (uint64_t)b - 1 + ((uint64_t)1 << lane);
  const bool in = lane < 31 && q < N && keys[q] == k;
  const uint32_t m = __popc(__ballot_sync(0xffffffffu, in));  // lanes 0..m-1 are inside the run
  if (m == 0) return b;
  uint64_t lo = (uint64_t)b + ((uint64_t)1 << (m - 1));               // b-1+2^(m-1) is inside
  const uint64_t cap = (uint64_t)b - 1 + ((uint64_t)1 << m);
  uint64_t hi = cap < (uint64_t)N ? cap : (uint64_t)N;  // outside, or N
  while (hi > lo) {  // invariant: positions < lo are inside, position hi is outside (or N)
    const uint64_t step = (hi - lo + 31) / 32;
    const uint64_t p = lo + lane * step;
    const bool inside = p < hi && keys[p] == k;
    const uint32_t c = __popc(__ballot_sync(0xffffffffu, inside));
    if (c == 0) break;  // position lo itself is outside
    const uint64_t nlo = lo + (uint64_t)(c - 1) * step + 1;
    const uint64_t nhi = lo + (uint64_t)c * step;
    hi = nhi < hi ? nhi : hi;
    lo = nlo;
  }
  return (uint32_t)lo;
}

// Predecessor tiles a look-back warp reads per poll and count. Every poll's
// loads are L2 traffic shared with the other tiles in flight: measured on GB300,
// the large skewed workload's run-length kernel takes 615 us reading 32, 561 at
// 16, 547 at 8, 563 at 4 (and 1370 at 128); the mixed-tables and DLRM-like ones
// do not change between 8 and 32.
constexpr int kRunsLookback = 8;

// Dynamic shared memory: run-head positions [TILE+1], first keys of segments [S+1].
template <int ITEMS>
size_t runs_smem(uint32_t S) {
  return ((size_t)kThreads * ITEMS + 1 + S + 1) * sizeof(uint32_t);
}

// MULTI: the tables form several segments whose first runs are recorded.
template <bool MULTI, int ITEMS>
__global__ void __launch_bounds__(kThreads) k_runs(RunsArgs a) {
  constexpr uint32_t TILE = kThreads * ITEMS;
  __shared__ uint32_t s_tile;
  __shared__ uint32_t s_scan[3 * kWarps];
  __shared__ uint32_t s_base[3];
  __shared__ uint32_t s_last_key;
  __shared__ uint32_t s_end_key;  // key at position N-1 (last tile only)
  extern __shared__ __align__(16) uint32_t s_dyn[];
  uint32_t* s_head_pos = s_dyn;            // [TILE+1]
  uint32_t* s_bkey = s_head_pos + TILE + 1;  // [S+1]
  if constexpr (MULTI)
    for (uint32_t i = threadIdx.x; i <= a.S; i += kThreads) s_bkey[i] = a.seg_keys[i];
  pdl_wait();
  pdl_trigger();
  // tiles in look-back order (see k_sort_pass)
  if (!a.ordered && threadIdx.x == 0) s_tile = atomicAdd(&a.ctl->tile_ctr[TC_RLE], 1u);
  __syncthreads();
  const uint32_t tile = a.ordered ? blockIdx.x : s_tile;
  if (tile >= gridDim.x) {  // only if the control block was not zero: never index past the grid
    if (threadIdx.x == 0) raise_error(a.ctl, a.sticky, kErrTimeout);
    return;
  }
  const uint32_t N = (uint32_t)a.N;
  const uint32_t i0 = tile * TILE;
  const uint32_t p0 = i0 + threadIdx.x * ITEMS;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint32_t key[ITEMS];
  if (p0 + ITEMS <= N) {
#pragma unroll
    for (int k = 0; k < ITEMS; k += 4) {
      const uint4 u = *reinterpret_cast<const uint4*>(a.keys + p0 + k);
      key[k] = u.x; key[k + 1] = u.y; key[k + 2] = u.z; key[k + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) key[k] = p0 + k < N ? a.keys[p0 + k] : 0u;
  }
  const uint32_t prev = (p0 > 0 && p0 <= N) ? a.keys[p0 - 1] : 0u;
  uint32_t heads = 0;  // bit k: position p0+k starts a run
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const uint32_t before = k == 0 ? prev : key[k - 1];
    if (p0 + k < N && (p0 + k == 0 || key[k] != before)) heads |= 1u << k;
    if (p0 + k == N - 1) s_end_key = key[k];
  }
  uint32_t n_heads;
  const uint32_t h0 = block_excl_scan(__popc(heads), s_scan, &n_heads);
  {
    uint32_t h = h0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      if (heads & (1u << k)) {
        s_head_pos[h] = p0 + k;
        if (h == n_heads - 1) s_last_key = key[k];
        ++h;
      }
    }
  }
  __syncthreads();
  // end of the tile's last run (it may continue into later tiles)
  if (warp == 0 && n_heads > 0) {
    const uint32_t tile_end = min(i0 + TILE, N);
    const uint32_t e = run_end_search(a.keys, N, tile_end, s_last_key);
    if (lane == 0) s_head_pos[n_heads] = e;
  }
  __syncthreads();

  // lengths, long runs and their lookups of this thread's runs
  uint32_t n_long = 0, n_llook = 0;
  {
    uint32_t h = h0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      if (heads & (1u << k)) {
        const uint32_t SL = s_head_pos[h + 1] - s_head_pos[h];
        if (SL >= a.thr) {
          n_long += 1;
          n_llook += SL;
        }
        ++h;
      }
    }
  }
  uint32_t e_long, e_llook, t_long, t_llook;
  block_excl_scan2(n_long, n_llook, s_scan, &e_long, &e_llook, &t_long, &t_llook);
  if (warp < 3) {  // one warp per count
    const uint32_t agg = warp == 0 ? n_heads : warp == 1 ? t_long : t_llook;
    const uint32_t b = lookback_warp<kRunsLookback>(a.lb, tile, 3, warp, agg, a.ctl, a.sticky);
    if (lane == 0) s_base[warp] = b;
  }
  __syncthreads();

  uint32_t r = s_base[0] + h0;
  uint32_t kl = s_base[1] + e_long, lp = s_base[2] + e_llook;
  bool overflow = false;
  uint32_t h = h0;
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    if (heads & (1u << k)) {
      const uint32_t start = s_head_pos[h], end = s_head_pos[h + 1];
      if (r < N) {
        a.run_key[r] = key[k];
        a.run_start[r] = start;
        if constexpr (MULTI) {  // first run of this key's segment (and of empty segments before it)
          const uint32_t sg = table_of(s_bkey, a.S, key[k]);
          const uint32_t before = k == 0 ? prev : key[k - 1];
          if (start == 0 || before < s_bkey[sg]) {
            const uint32_t s0 = start == 0 ? 0u : table_of(s_bkey, a.S, before) + 1;
            for (uint32_t q = s0; q <= sg; ++q) a.seg_runs[q] = r;
          }
        }
      } else {
        overflow = true;
      }
      const uint32_t SL = end - start;
      if (SL >= a.thr) {
        if (kl < a.cap_long) {
          a.long_ids[kl] = r;
          a.longs[kl] = LongRun{start, SL, key[k], lp};
        } else {
          overflow = true;
        }
        kl += 1;
        lp += SL;
      }
      ++r;
      ++h;
    }
  }
  if (overflow) raise_error(a.ctl, a.sticky, kErrCapacity);
  if (i0 + TILE >= N && threadIdx.x == 0) {  // the last tile knows every total
    const uint32_t U = s_base[0] + n_heads;
    if (U <= N) {
      a.ctl->num_runs = U;
      a.run_start[U] = N;
      // segments after the last key's segment are empty
      if constexpr (MULTI)
        for (uint32_t q = table_of(s_bkey, a.S, s_end_key) + 1; q <= a.S; ++q) a.seg_runs[q] = U;
    }
    a.ctl->num_long = s_base[1] + t_long;
    a.ctl->long_lookups = s_base[2] + t_llook;
  }
}

const void* runs_fn(bool multi, int items) {
  if (items == 16)
    return multi ? reinterpret_cast<const void*>(&k_runs<true, 16>) : reinterpret_cast<const void*>(&k_runs<false, 16>);
  return multi ? reinterpret_cast<const void*>(&k_runs<true, 8>) : reinterpret_cast<const void*>(&k_runs<false, 8>);
}

size_t runs_smem_bytes(int items, uint32_t S) { return items == 16 ? runs_smem<16>(S) : runs_smem<8>(S); }

}  // namespace

// Sorted keys per thread: 8 (2048-key tiles) up to 2^21 lookups, 16 above
// (half as many tiles, so half as many look-back steps and run-end searches).
int runs_items_for(int64_t N) { return N <= (int64_t)(1 << 21) ? 8 : 16; }

cudaError_t runs_configure() {
  cudaError_t e = cudaSuccess;
  for (int multi = 0; multi < 2 && e == cudaSuccess; ++multi)
    for (int items : {8, 16})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(runs_fn(multi != 0, items), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)runs_smem_bytes(items, kMaxT));
  return e;
}

int runs_capacity(int S, int items, int sms) {
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, runs_fn(S > 1, items), kThreads,
                                                    runs_smem_bytes(items, (uint32_t)S)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return blocks * sms;
}

cudaError_t launch_runs(const RunsArgs& a, int items, cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)((a.N + (int64_t)kThreads * items - 1) / ((int64_t)kThreads * items));
  RunsArgs arg = a;
  void* args[] = {&arg};
  return launch_kernel(runs_fn(a.S > 1, items), dim3(grid), dim3(kThreads), runs_smem_bytes(items, a.S), s, args,
                       pdl);
}

}  // namespace embbwd
