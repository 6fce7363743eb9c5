// Device radix sort of (linear index, payload) pairs: the sort step of
// "fbgemm_gpu/codegen/embedding_backward_split_template.cu" (its host function
// sorts linear_indices with their infos on bits [0, total_hash_size_bits)),
// written as a one-sweep LSD radix sort for sm_103a:
//   k_hist       one read of the indices: linearise each lookup to its 32-bit
//                key hash_size_cumsum[t] + idx, range-check it, validate the
//                CSR offsets, build the digit histograms of every pass, and
//                write the (key, payload) pairs the passes sort;
//   k_sort_pass  per pass: load a tile, rank it with warp match-based
//                multisplit, publish/look back per-digit tile counts (decoupled
//                look-back, bounded waits), scatter through shared memory so
//                that global writes are runs of consecutive addresses.
// The sort is stable: equal keys keep lookup order.
#include "decode.cuh"

namespace embbwd {

namespace {

constexpr uint32_t kFull = 0xffffffffu;

// FIRST: the ValueKind of the payload to build, or -1 to only check (no pairs,
// no histogram: the atomic path).
template <int ITEMS, int FIRST>
__global__ void __launch_bounds__(kThreads) k_hist(HistArgs a) {
  constexpr int TILE = kThreads * ITEMS;
  using V = typename std::conditional<FIRST == VK_BAG_SCALED, uint64_t, uint32_t>::type;
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int HW = kMaxPasses * kRadix;                          // one warp's histograms
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem);           // [8 warps][passes][256]
  uint32_t* s_bag = s_hist + kWarps * HW;                          // [TILE]
  uint32_t* s_len = s_bag + TILE;                                  // [TILE]
  uint32_t* s_hsc = s_len + TILE;                                  // [T+1]
  const DecodeArgs& d = a.d;
  pdl_wait();
  pdl_trigger();
  // s_hist first holds the staged bag offsets; it is zeroed after the expansion.
  for (uint32_t i = threadIdx.x; i <= d.T; i += kThreads) s_hsc[i] = d.hsc[i];

  // CSR validation: non-decreasing offsets from 0 to N.
  for (uint32_t bt = blockIdx.x * kThreads + threadIdx.x; bt < d.BT; bt += gridDim.x * kThreads) {
    if (d.offsets[bt + 1] < d.offsets[bt]) raise_error(a.ctl, a.sticky, kErrOffsets);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (d.offsets[0] != 0 || d.offsets[d.BT] != d.N) raise_error(a.ctl, a.sticky, kErrOffsets);
  }

  const int64_t i0 = (int64_t)blockIdx.x * TILE;
  const int64_t i1 = min(i0 + TILE, d.N);
  // the tile's indices (and per-sample weights) are independent of the bag search: load first
  int64_t idx[ITEMS];
  float psw[ITEMS];
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int64_t pos = i0 + k * kThreads + threadIdx.x;
    idx[k] = pos < i1 ? d.indices[pos] : 0;
    if constexpr (FIRST == VK_BAG_SCALED) psw[k] = (pos < i1 && d.psw) ? d.psw[pos] : 1.0f;
  }
  __syncthreads();
  expand_tile_bags(d, i0, i1, s_bag, (FIRST == VK_BAG_SCALED && d.mean) ? s_len : nullptr,
                   reinterpret_cast<int64_t*>(s_hist), kWarps * HW / 2);
  for (int i = threadIdx.x; i < kWarps * HW; i += kThreads) s_hist[i] = 0;
  __syncthreads();

  // Per-warp private histograms in shared memory: plain shared atomics, no
  // contention between warps; colliding lanes of one warp are serialised.
  uint32_t* wh = s_hist + (threadIdx.x >> 5) * HW;
  V* vals_out = reinterpret_cast<V*>(a.vals_out);
  bool any_bad = false;
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int64_t pos = i0 + k * kThreads + threadIdx.x;
    if (pos < i1) {
      const uint32_t bt = s_bag[pos - i0];
      uint32_t t = div_by_B(bt, d.B, d.invB);
      if (t >= d.T) t = d.T - 1;
      const uint32_t base = s_hsc[t];
      any_bad |= idx[k] < 0 || idx[k] >= (int64_t)(s_hsc[t + 1] - base);
      const uint32_t key = base + (uint32_t)idx[k];
      if constexpr (FIRST >= 0) {
        for (int p = 0; p < a.passes; ++p) atomicAdd(&wh[p * kRadix + ((key >> (p * kRadixBits)) & (kRadix - 1))], 1u);
        a.keys_out[pos] = key;
        if constexpr (FIRST == VK_BAG) {
          vals_out[pos] = bt;
        } else if constexpr (FIRST == VK_NOBAG) {
          vals_out[pos] = (uint32_t)pos;
        } else {
          float s = psw[k];
          if (d.mean) s = __fdiv_rn(s, (float)s_len[pos - i0]);
          vals_out[pos] = (uint64_t)bt | ((uint64_t)__float_as_uint(s) << 32);
        }
      }
    }
  }
  if (__syncthreads_or(any_bad) && threadIdx.x == 0) raise_error(a.ctl, a.sticky, kErrIndex);
  if constexpr (FIRST >= 0) {
    for (int i = threadIdx.x; i < a.passes * kRadix; i += kThreads) {
      uint32_t c = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) c += s_hist[w * HW + i];
      if (c) atomicAdd(&a.ctl->hist[0][0] + i, c);
    }
  }
}

// Lookups per thread of the large-batch tiles. Measured on GB300: 16 with two
// resident blocks per SM (128 registers) beats 8 or 12 lookups per thread at
// higher occupancy, and one block per SM with more registers.
constexpr int kBigItems = 16;

template <int ITEMS, typename V>
__global__ void __launch_bounds__(kThreads, ITEMS == kBigItems ? 2 : 3) k_sort_pass(PassArgs a) {
  constexpr int TILE = kThreads * ITEMS;
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* s_whist = reinterpret_cast<uint32_t*>(smem);  // [8][256]
  uint32_t* s_dstart = s_whist + kWarps * kRadix;         // [256]
  uint32_t* s_gbase = s_dstart + kRadix;                  // [256]
  uint32_t* s_misc = s_gbase + kRadix;                    // [32]
  uint32_t* s_keys = s_misc + 32;                         // [TILE]
  V* s_vals = reinterpret_cast<V*>(s_keys + TILE);        // [TILE]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t N = a.N;
  pdl_wait();
  pdl_trigger();

  // Tiles in look-back order: the block index when every block of the grid can be
  // resident at once (no block waits on one that cannot start), else a counter.
  if (!a.ordered && threadIdx.x == 0) s_misc[0] = atomicAdd(&a.ctl->tile_ctr[a.pass], 1u);
  const uint32_t ghist = a.ctl->hist[a.pass][threadIdx.x];  // global count of digit threadIdx.x
  for (int i = threadIdx.x; i < kWarps * kRadix; i += kThreads) s_whist[i] = 0;
  __syncthreads();
  const uint32_t tile = a.ordered ? blockIdx.x : s_misc[0];
  if (tile >= gridDim.x) {  // only if the control block was not zero: never index past the grid
    if (threadIdx.x == 0) raise_error(a.ctl, a.sticky, kErrTimeout);
    return;
  }
  const int64_t i0 = (int64_t)tile * TILE;
  const int64_t i1 = min(i0 + TILE, N);

  uint32_t keys[ITEMS];
  V vals[ITEMS];
  uint32_t ranks[ITEMS];
  const int64_t wbase = i0 + (int64_t)warp * 32 * ITEMS;
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int64_t pos = wbase + k * 32 + lane;
    keys[k] = pos < i1 ? a.keys_in[pos] : 0u;
    vals[k] = pos < i1 ? reinterpret_cast<const V*>(a.vals_in)[pos] : (V)0;
  }

  // Warp-level multisplit ranking: stable within the warp's slice of the tile.
  const uint32_t lt = lanemask_lt();
  uint32_t* wh = s_whist + warp * kRadix;
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int64_t pos = wbase + k * 32 + lane;
    const bool valid = pos < i1;
    const uint32_t digit = valid ? ((keys[k] >> a.shift) & (kRadix - 1)) : kRadix;
    const uint32_t peers = __match_any_sync(kFull, digit);
    const int leader = __ffs(peers) - 1;
    uint32_t pre = 0;
    if (lane == leader && valid) {
      pre = wh[digit];
      wh[digit] = pre + __popc(peers);
    }
    pre = __shfl_sync(kFull, pre, leader);
    ranks[k] = pre + __popc(peers & lt);
    __syncwarp();
  }
  __syncthreads();

  // Per digit (one per thread): warp offsets, tile counts, tile and global bases.
  const uint32_t dg = threadIdx.x;
  uint32_t count = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t c = s_whist[w * kRadix + dg];
    s_whist[w * kRadix + dg] = count;
    count += c;
  }
  uint32_t dstart, gdig, tot0, tot1;
  block_excl_scan2(count, ghist, s_misc + 16, &dstart, &gdig, &tot0, &tot1);
  const uint32_t excl = lookback_channel(a.lb, tile, kRadix, dg, count, a.ctl, a.sticky);
  s_dstart[dg] = dstart;
  s_gbase[dg] = gdig + excl - dstart;
  __syncthreads();

#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int64_t pos = wbase + k * 32 + lane;
    if (pos < i1) {
      const uint32_t digit = (keys[k] >> a.shift) & (kRadix - 1);
      const uint32_t q = s_dstart[digit] + s_whist[warp * kRadix + digit] + ranks[k];
      s_keys[q] = keys[k];
      s_vals[q] = vals[k];
    }
  }
  __syncthreads();
  const uint32_t n = (uint32_t)(i1 - i0);
  V* vout = reinterpret_cast<V*>(a.vals_out);
  for (uint32_t q = threadIdx.x; q < n; q += kThreads) {
    const uint32_t key = s_keys[q];
    const uint32_t digit = (key >> a.shift) & (kRadix - 1);
    const uint32_t out = s_gbase[digit] + q;
    if (out < (uint64_t)N) {  // always true unless a look-back timed out
      a.keys_out[out] = key;
      vout[out] = s_vals[q];
    }
  }
}

template <int ITEMS>
size_t hist_smem(int T) {
  return (kWarps * kMaxPasses * kRadix + 2 * kThreads * ITEMS + T + 1) * sizeof(uint32_t);
}

template <int ITEMS, typename V>
size_t pass_smem() {
  return (kWarps * kRadix + 2 * kRadix + 32) * sizeof(uint32_t) +
         (size_t)kThreads * ITEMS * (sizeof(uint32_t) + sizeof(V));
}

template <int ITEMS, int FIRST>
cudaError_t set_hist_attr() {
  return cudaFuncSetAttribute(k_hist<ITEMS, FIRST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)hist_smem<ITEMS>(kMaxT));
}

template <int ITEMS>
cudaError_t configure_items() {
  cudaError_t e = set_hist_attr<ITEMS, -1>();
  if (e == cudaSuccess) e = set_hist_attr<ITEMS, VK_BAG>();
  if (e == cudaSuccess) e = set_hist_attr<ITEMS, VK_BAG_SCALED>();
  if (e == cudaSuccess) e = set_hist_attr<ITEMS, VK_NOBAG>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_sort_pass<ITEMS, uint32_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pass_smem<ITEMS, uint32_t>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_sort_pass<ITEMS, uint64_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pass_smem<ITEMS, uint64_t>());
  return e;
}

template <int ITEMS>
const void* hist_fn(int first_kind) {
  switch (first_kind) {
    case VK_BAG: return reinterpret_cast<const void*>(&k_hist<ITEMS, VK_BAG>);
    case VK_BAG_SCALED: return reinterpret_cast<const void*>(&k_hist<ITEMS, VK_BAG_SCALED>);
    case VK_NOBAG: return reinterpret_cast<const void*>(&k_hist<ITEMS, VK_NOBAG>);
    default: return reinterpret_cast<const void*>(&k_hist<ITEMS, -1>);
  }
}

}  // namespace

// Lookups per block: small tiles keep all SMs busy on small batches, large
// tiles cut look-back traffic on large ones.
size_t sort_tile_for(int64_t N) { return N <= (int64_t)(1 << 21) ? kThreads * 4 : kThreads * kBigItems; }

// Lookups per block of the radix passes. Measured on GB300 (whole-tile
// comparisons): between 2^17 and 2^21 lookups the passes run faster on
// 2048-lookup tiles (DLRM-like batch: 27.6 against 29.3 us for three passes)
// while the histogram kernel stays faster on 1024; below, 1024 wins.
size_t pass_tile_for(int64_t N) {
  if (N <= (int64_t)(1 << 17)) return kThreads * 4;
  return N <= (int64_t)(1 << 21) ? kThreads * 8 : kThreads * kBigItems;
}

cudaError_t sort_configure(const DevProps& p) {
  (void)p;
  cudaError_t e = configure_items<4>();
  if (e == cudaSuccess) e = configure_items<8>();
  if (e == cudaSuccess) e = configure_items<kBigItems>();
  return e;
}

cudaError_t launch_hist(const HistArgs& a, int first_kind, int T, cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)((a.d.N + a.tile - 1) / a.tile);
  HistArgs arg = a;
  void* args[] = {&arg};
  if (a.tile == kThreads * 4)
    return launch_kernel(hist_fn<4>(first_kind), dim3(grid), dim3(kThreads), hist_smem<4>(T), s, args, pdl);
  return launch_kernel(hist_fn<kBigItems>(first_kind), dim3(grid), dim3(kThreads), hist_smem<kBigItems>(T), s,
                       args, pdl);
}

namespace {

const void* pass_fn(bool wide_vals, int tile, size_t* sm) {
  if (tile == kThreads * 8) {
    *sm = wide_vals ? pass_smem<8, uint64_t>() : pass_smem<8, uint32_t>();
    return wide_vals ? reinterpret_cast<const void*>(&k_sort_pass<8, uint64_t>)
                     : reinterpret_cast<const void*>(&k_sort_pass<8, uint32_t>);
  }
  if (tile == kThreads * 4) {
    *sm = wide_vals ? pass_smem<4, uint64_t>() : pass_smem<4, uint32_t>();
    return wide_vals ? reinterpret_cast<const void*>(&k_sort_pass<4, uint64_t>)
                     : reinterpret_cast<const void*>(&k_sort_pass<4, uint32_t>);
  }
  *sm = wide_vals ? pass_smem<kBigItems, uint64_t>() : pass_smem<kBigItems, uint32_t>();
  return wide_vals ? reinterpret_cast<const void*>(&k_sort_pass<kBigItems, uint64_t>)
                   : reinterpret_cast<const void*>(&k_sort_pass<kBigItems, uint32_t>);
}

}  // namespace

cudaError_t launch_sort_pass(const PassArgs& a, bool wide_vals, int tile, cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)((a.N + tile - 1) / tile);
  PassArgs arg = a;
  void* args[] = {&arg};
  size_t sm;
  const void* fn = pass_fn(wide_vals, tile, &sm);
  return launch_kernel(fn, dim3(grid), dim3(kThreads), sm, s, args, pdl);
}

int pass_tile_class(int tile) { return tile == kThreads * 4 ? 0 : (tile == kThreads * 8 ? 1 : 2); }

int sort_pass_capacity(bool wide_vals, int tile, int sms) {
  size_t sm;
  const void* fn = pass_fn(wide_vals, tile, &sm);
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kThreads, sm) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return blocks * sms;
}

}  // namespace embbwd
