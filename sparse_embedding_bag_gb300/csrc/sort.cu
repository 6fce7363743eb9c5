// Device radix sort of (linear index, payload) pairs: the sort step of
// "fbgemm_gpu/codegen/embedding_backward_split_template.cu" (its host function
// sorts linear_indices with their infos by linear index), written as a
// one-sweep LSD radix sort for sm_103a that sorts each table's segment on its
// own:
//   the lookups arrive table-major (the CSR offsets list table 0's bags first),
//   so the lookups of table t already form one contiguous segment
//   [offsets[t*B], offsets[(t+1)*B]) holding exactly the linear indices of
//   that table, [hash_size_cumsum[t], hash_size_cumsum[t+1]). Sorting every
//   segment by its row index (the linear index minus hash_size_cumsum[t])
//   therefore sorts the whole array by linear index, and the row index has
//   ceil(log2(largest table)) bits instead of ceil(log2(all rows)): one pass
//   fewer for the large workloads of many similar tables.
//   k_hist       one read of the indices: linearise each lookup to its 32-bit
//                key hash_size_cumsum[t] + idx, range-check it, validate the
//                CSR offsets, count every pass's digit of the row index per
//                table, and write the (key, payload) pairs the passes sort;
//                block 0 also lays the passes' tiles out on the segments (a
//                tile never crosses a table boundary).
//   k_sort_pass  per pass: load a tile, rank it with warp match-based
//                multisplit, publish/look back per-digit tile counts among the
//                tiles of its table (decoupled look-back, bounded waits),
//                scatter through shared memory so that global writes are runs
//                of consecutive addresses.
// Digits have 1..9 bits (the passes split the row bits evenly); the kernels
// come in 128-, 256- and 512-bucket builds. The sort is stable: equal keys
// keep lookup order.
#include "decode.cuh"

namespace embbwd {

namespace {

constexpr uint32_t kFull = 0xffffffffu;

// Histogram words per warp: passes x buckets (at most 3 passes of 128 or 512
// buckets, 4 passes of 256).
template <int RADIX>
struct HistWords {
  static constexpr int value = (RADIX == 256 ? 4 : 3) * RADIX;
};

// Lays the passes' tiles out on the tables' segments: table t's segment
// [offsets[t*B], offsets[(t+1)*B]) (clamped into [0, N]) gets ceil(len / ptile)
// tiles. Called by every thread of block 0; uses `scratch` (kWarps words).
__device__ __forceinline__ void build_tile_map(const HistArgs& a, uint32_t* scratch) {
  const DecodeArgs& d = a.d;
  const uint32_t T = d.T, pt = (uint32_t)a.ptile;
  auto seg = [&](uint32_t t) -> uint32_t {  // start of table t's segment, clamped
    const int64_t o = t >= T ? d.N : d.offsets[(size_t)t * d.B];
    return (uint32_t)(o < 0 ? 0 : (o > d.N ? d.N : o));
  };
  auto ntiles = [&](uint32_t s0, uint32_t s1) { return s1 > s0 ? (s1 - s0 + pt - 1) / pt : 0u; };
  const uint32_t per = (T + kThreads - 1) / kThreads;  // tables per thread
  const uint32_t t0 = threadIdx.x * per, t1 = min(t0 + per, T);
  uint32_t mine = 0;
  for (uint32_t t = t0; t < t1; ++t) mine += ntiles(seg(t), seg(t + 1));
  uint32_t total;
  uint32_t base = block_excl_scan(mine, scratch, &total);
  for (uint32_t t = t0; t < t1; ++t) {
    const uint32_t s0 = seg(t), s1 = seg(t + 1), n = ntiles(s0, s1);
    for (uint32_t k = 0; k < n && base + k < a.tile_cap; ++k)
      a.tile_map[base + k] = PassTile{t, s0 + k * pt, min(s0 + (k + 1) * pt, s1), base, s0, d.hsc[t]};
    base += n;
  }
  // valid offsets never reach the cap; malformed ones (whose passes do nothing) are cut at it
  if (threadIdx.x == 0) a.ctl->pass_tiles = min(total, a.tile_cap);
}

// FIRST: the ValueKind of the payload to build, or -1 to only check (no pairs,
// no histogram: the atomic path). RADIX: buckets of the histograms.
template <int ITEMS, int FIRST, int RADIX>
__global__ void __launch_bounds__(kThreads) k_hist(HistArgs a) {
  constexpr int TILE = kThreads * ITEMS;
  using V = typename std::conditional<FIRST == VK_BAG_SCALED, uint64_t, uint32_t>::type;
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int HW = HistWords<RADIX>::value;                          // one warp's histograms
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem);           // [8 warps][passes][RADIX]
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
  const int hw = a.passes * RADIX;  // histogram words in use per warp
  for (int i = threadIdx.x; i < kWarps * hw; i += kThreads) s_hist[i] = 0;
  // the table of the tile's first lookup keeps its counts in shared memory; lookups
  // of further tables (a tile that crosses table boundaries) count in global memory
  uint32_t tmain = 0;
  if (i1 > i0) {
    tmain = div_by_B(s_bag[0], d.B, d.invB);
    if (tmain >= d.T) tmain = d.T - 1;
  }
  __syncthreads();

  // Per-warp private histograms in shared memory: plain shared atomics, no
  // contention between warps; colliding lanes of one warp are serialised.
  uint32_t* wh = s_hist + (threadIdx.x >> 5) * hw;
  V* vals_out = reinterpret_cast<V*>(a.vals_out);
  const uint32_t dmask = (1u << a.rbits) - 1u;
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
      const uint32_t row = (uint32_t)idx[k];
      const uint32_t key = base + row;
      if constexpr (FIRST >= 0) {
        if (t == tmain) {
          for (int p = 0; p < a.passes; ++p) atomicAdd(&wh[p * RADIX + ((row >> (p * a.rbits)) & dmask)], 1u);
        } else {
          uint32_t* g = a.thist + (size_t)t * a.passes * RADIX;
          for (int p = 0; p < a.passes; ++p) atomicAdd(&g[p * RADIX + ((row >> (p * a.rbits)) & dmask)], 1u);
        }
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
    uint32_t* g = a.thist + (size_t)tmain * a.passes * RADIX;
    for (int i = threadIdx.x; i < hw; i += kThreads) {
      uint32_t c = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) c += s_hist[w * hw + i];
      if (c) atomicAdd(&g[i], c);
    }
    if (blockIdx.x == 0) {
      __syncthreads();
      build_tile_map(a, s_bag);  // s_bag is free here
    }
  }
}

// Lookups per thread of the large-batch tiles. Measured on GB300: 16 with two
// resident blocks per SM (128 registers) beats 8 or 12 lookups per thread at
// higher occupancy, and one block per SM with more registers. With 32-bit
// payloads three blocks per SM (80 registers, some spilled) do better still (the
// large skewed workload's three passes 3.27 -> 3.19 ms); 64-bit payloads spill
// more and stay at two (the mixed-tables passes 206 us, 223 at three).
constexpr int kBigItems = 16;
constexpr int kRankGrp = 4;  // items of a thread whose warp peer masks are found together

// Predecessor tiles a pass's look-back reads per poll and channel. Every poll of
// a tile reads window x buckets status words, and with hundreds of tiles of one
// table in flight that traffic, not the walk's length, sets the pace. Measured on
// GB300 (three passes of the large skewed workload; mixed tables; DLRM-like):
// windows of 64, 32, 16, 8, 4, 2, 1 gave 6.00, 3.58, 3.08, 2.58, 2.61, 2.45,
// 2.70 ms; 321, 230, 193, 190, 189, 191, 195 us; DLRM-like 20.0-20.4 us for 1-8.
template <int ITEMS>
struct LookbackWin {
  static constexpr int value = ITEMS >= kBigItems ? 2 : 4;
};

template <int ITEMS, typename V>
struct PassBlocks {
  static constexpr int value = ITEMS == kBigItems && sizeof(V) == 8 ? 2 : 3;
};

template <int ITEMS, typename V, int RADIX>
__global__ void __launch_bounds__(kThreads, PassBlocks<ITEMS, V>::value) k_sort_pass(PassArgs a) {
  constexpr int TILE = kThreads * ITEMS;
  constexpr int DPT = RADIX > kThreads ? RADIX / kThreads : 1;  // digits per thread
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* s_whist = reinterpret_cast<uint32_t*>(smem);  // [8][RADIX]
  uint32_t* s_dstart = s_whist + kWarps * RADIX;          // [RADIX]
  uint32_t* s_gbase = s_dstart + RADIX;                   // [RADIX]
  uint32_t* s_misc = s_gbase + RADIX;                     // [32]
  uint32_t* s_keys = s_misc + 32;                         // [TILE]
  V* s_vals = reinterpret_cast<V*>(s_keys + TILE);        // [TILE]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t N = a.N;
  pdl_wait();
  pdl_trigger();
  // Tiles in look-back order: the block index when every block of the grid can be
  // resident at once (no block waits on one that cannot start), else a counter.
  if (!a.ordered && threadIdx.x == 0) s_misc[0] = atomicAdd(&a.ctl->tile_ctr[a.pass], 1u);
  for (int i = threadIdx.x; i < kWarps * RADIX; i += kThreads) s_whist[i] = 0;
  __syncthreads();
  const uint32_t tile = a.ordered ? blockIdx.x : s_misc[0];  // < the grid <= the tile map's entries
  // one round trip: the error word, the number of tiles and this tile's entry
  const uint32_t err = ld_relaxed_u32(&a.ctl->err);
  const uint32_t ntiles = ld_relaxed_u32(&a.ctl->pass_tiles);
  const PassTile tm = a.tile_map[tile];
  // malformed offsets: the segments are not trustworthy, every block leaves (none waits);
  // the grid is an upper bound on the tiles
  if ((err & kErrOffsets) || tile >= ntiles) return;
  const uint32_t t = tm.t;
  const int64_t i0 = tm.i0, i1 = min((int64_t)tm.i1, N);
  const uint32_t seg0 = tm.seg0;    // first lookup of the table
  const uint32_t kbase = tm.kbase;  // hash_size_cumsum[t]
  const uint32_t shift = (uint32_t)(a.pass * a.rbits), dmask = (1u << a.rbits) - 1u;
  const uint32_t channels = dmask + 1u;
  // this table's count of each of the thread's digits (digits tid*DPT .. tid*DPT+DPT-1)
  const uint32_t* H = a.thist + ((size_t)t * a.passes + a.pass) * RADIX;
  uint32_t gh[DPT];
#pragma unroll
  for (int q = 0; q < DPT; ++q) {
    const uint32_t dg = threadIdx.x * DPT + q;
    gh[q] = dg < channels ? H[dg] : 0u;
  }

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
  uint32_t* wh = s_whist + warp * RADIX;
  // kRankGrp items at a time: their peer masks are found before the counts are
  // updated (the updates form one chain through the warp's histogram)
#pragma unroll
  for (int k0 = 0; k0 < ITEMS; k0 += kRankGrp) {
    uint32_t dg[kRankGrp], pm[kRankGrp];
#pragma unroll
    for (int u = 0; u < kRankGrp; ++u) {
      const int64_t pos = wbase + (k0 + u) * 32 + lane;
      dg[u] = pos < i1 ? (((keys[k0 + u] - kbase) >> shift) & dmask) : (uint32_t)RADIX;
    }
#pragma unroll
    for (int u = 0; u < kRankGrp; ++u) pm[u] = __match_any_sync(kFull, dg[u]);
#pragma unroll
    for (int u = 0; u < kRankGrp; ++u) {
      const bool valid = dg[u] < (uint32_t)RADIX;
      const int leader = __ffs(pm[u]) - 1;
      uint32_t pre = 0;
      if (lane == leader && valid) {
        pre = wh[dg[u]];
        wh[dg[u]] = pre + __popc(pm[u]);
      }
      pre = __shfl_sync(kFull, pre, leader);
      ranks[k0 + u] = pre + __popc(pm[u] & lt);
      __syncwarp();
    }
  }
  __syncthreads();

  // Per digit: warp offsets, tile counts, tile and global bases.
  uint32_t cnt[DPT], dch[DPT], cs = 0, gs = 0;
#pragma unroll
  for (int q = 0; q < DPT; ++q) {
    const uint32_t dg = threadIdx.x * DPT + q;
    dch[q] = dg;
    uint32_t count = 0;
    if (dg < (uint32_t)RADIX) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = s_whist[w * RADIX + dg];
        s_whist[w * RADIX + dg] = count;
        count += c;
      }
    }
    cnt[q] = count;
    cs += count;
    gs += gh[q];
  }
  uint32_t ec, eg, tc, tg;
  block_excl_scan2(cs, gs, s_misc + 16, &ec, &eg, &tc, &tg);
  uint32_t excl[DPT];
  lookback_channels<DPT, LookbackWin<ITEMS>::value>(a.lb, tile, tm.first, channels, dch, cnt, excl, a.ctl,
                                                     a.sticky);
#pragma unroll
  for (int q = 0; q < DPT; ++q) {
    const uint32_t dg = dch[q];
    if (dg < (uint32_t)RADIX) {
      s_dstart[dg] = ec;
      s_gbase[dg] = seg0 + eg + excl[q] - ec;
    }
    ec += cnt[q];
    eg += gh[q];
  }
  __syncthreads();

#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int64_t pos = wbase + k * 32 + lane;
    if (pos < i1) {
      const uint32_t digit = ((keys[k] - kbase) >> shift) & dmask;
      const uint32_t q = s_dstart[digit] + s_whist[warp * RADIX + digit] + ranks[k];
      s_keys[q] = keys[k];
      s_vals[q] = vals[k];
    }
  }
  __syncthreads();
  const uint32_t n = i1 > i0 ? (uint32_t)(i1 - i0) : 0u;
  V* vout = reinterpret_cast<V*>(a.vals_out);
  for (uint32_t q = threadIdx.x; q < n; q += kThreads) {
    const uint32_t key = s_keys[q];
    const uint32_t digit = ((key - kbase) >> shift) & dmask;
    const uint32_t out = s_gbase[digit] + q;
    if (out < (uint64_t)N) {  // always true unless a look-back timed out
      a.keys_out[out] = key;
      vout[out] = s_vals[q];
    }
  }
}

template <int ITEMS, int RADIX>
size_t hist_smem(int T) {
  return (kWarps * HistWords<RADIX>::value + 2 * kThreads * ITEMS + T + 1) * sizeof(uint32_t);
}

template <int ITEMS, typename V, int RADIX>
size_t pass_smem() {
  return (kWarps * RADIX + 2 * RADIX + 32) * sizeof(uint32_t) + (size_t)kThreads * ITEMS * (sizeof(uint32_t) + sizeof(V));
}

template <int ITEMS, int FIRST, int RADIX>
cudaError_t set_hist_attr() {
  return cudaFuncSetAttribute(k_hist<ITEMS, FIRST, RADIX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)hist_smem<ITEMS, RADIX>(kMaxT));
}

template <int ITEMS, int RADIX>
cudaError_t configure_hist() {
  cudaError_t e = set_hist_attr<ITEMS, VK_BAG, RADIX>();
  if (e == cudaSuccess) e = set_hist_attr<ITEMS, VK_BAG_SCALED, RADIX>();
  if (e == cudaSuccess) e = set_hist_attr<ITEMS, VK_NOBAG, RADIX>();
  return e;
}

template <int ITEMS, int RADIX>
cudaError_t configure_pass() {
  cudaError_t e = cudaFuncSetAttribute(k_sort_pass<ITEMS, uint32_t, RADIX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pass_smem<ITEMS, uint32_t, RADIX>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_sort_pass<ITEMS, uint64_t, RADIX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pass_smem<ITEMS, uint64_t, RADIX>());
  return e;
}

template <int ITEMS, int RADIX>
const void* hist_fn_r(int first_kind) {
  switch (first_kind) {
    case VK_BAG: return reinterpret_cast<const void*>(&k_hist<ITEMS, VK_BAG, RADIX>);
    case VK_BAG_SCALED: return reinterpret_cast<const void*>(&k_hist<ITEMS, VK_BAG_SCALED, RADIX>);
    case VK_NOBAG: return reinterpret_cast<const void*>(&k_hist<ITEMS, VK_NOBAG, RADIX>);
    default: return reinterpret_cast<const void*>(&k_hist<ITEMS, -1, 128>);
  }
}

template <int ITEMS>
const void* hist_fn(int first_kind, int radix, size_t* sm, int T) {
  if (first_kind < 0 || radix == 128) {
    *sm = hist_smem<ITEMS, 128>(T);
    return hist_fn_r<ITEMS, 128>(first_kind);
  }
  if (radix == 256) {
    *sm = hist_smem<ITEMS, 256>(T);
    return hist_fn_r<ITEMS, 256>(first_kind);
  }
  *sm = hist_smem<ITEMS, 512>(T);
  return hist_fn_r<ITEMS, 512>(first_kind);
}

template <int ITEMS, int RADIX>
const void* pass_fn_r(bool wide_vals, size_t* sm) {
  *sm = wide_vals ? pass_smem<ITEMS, uint64_t, RADIX>() : pass_smem<ITEMS, uint32_t, RADIX>();
  return wide_vals ? reinterpret_cast<const void*>(&k_sort_pass<ITEMS, uint64_t, RADIX>)
                   : reinterpret_cast<const void*>(&k_sort_pass<ITEMS, uint32_t, RADIX>);
}

template <int ITEMS>
const void* pass_fn_i(bool wide_vals, int radix, size_t* sm) {
  if (radix == 128) return pass_fn_r<ITEMS, 128>(wide_vals, sm);
  if (radix == 256) return pass_fn_r<ITEMS, 256>(wide_vals, sm);
  return pass_fn_r<ITEMS, 512>(wide_vals, sm);
}

const void* pass_fn(bool wide_vals, int tile, int radix, size_t* sm) {
  if (tile == kThreads * 4) return pass_fn_i<4>(wide_vals, radix, sm);
  if (tile == kThreads * 8) return pass_fn_i<8>(wide_vals, radix, sm);
  return pass_fn_i<kBigItems>(wide_vals, radix, sm);
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

// Fewest passes of at most kMaxRadixBits bits, the bits split evenly among them
// (row indices of 17 bits: two passes of 9; 21 bits: three of 7).
void radix_plan(int row_bits, int* passes, int* rbits) {
  const int b = row_bits < 1 ? 1 : row_bits;
  int p = (b + kMaxRadixBits - 1) / kMaxRadixBits;
  if (p > kMaxPasses) p = kMaxPasses;
  *passes = p;
  *rbits = (b + p - 1) / p;
}

int radix_buckets(int rbits) { return rbits <= 7 ? 128 : (rbits == 8 ? 256 : 512); }

cudaError_t sort_configure(const DevProps& p) {
  (void)p;
  cudaError_t e = cudaFuncSetAttribute(k_hist<4, -1, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)hist_smem<4, 128>(kMaxT));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_hist<kBigItems, -1, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)hist_smem<kBigItems, 128>(kMaxT));
  if (e == cudaSuccess) e = configure_hist<4, 128>();
  if (e == cudaSuccess) e = configure_hist<4, 256>();
  if (e == cudaSuccess) e = configure_hist<4, 512>();
  if (e == cudaSuccess) e = configure_hist<kBigItems, 128>();
  if (e == cudaSuccess) e = configure_hist<kBigItems, 256>();
  if (e == cudaSuccess) e = configure_hist<kBigItems, 512>();
  if (e == cudaSuccess) e = configure_pass<4, 128>();
  if (e == cudaSuccess) e = configure_pass<4, 256>();
  if (e == cudaSuccess) e = configure_pass<4, 512>();
  if (e == cudaSuccess) e = configure_pass<8, 128>();
  if (e == cudaSuccess) e = configure_pass<8, 256>();
  if (e == cudaSuccess) e = configure_pass<8, 512>();
  if (e == cudaSuccess) e = configure_pass<kBigItems, 128>();
  if (e == cudaSuccess) e = configure_pass<kBigItems, 256>();
  if (e == cudaSuccess) e = configure_pass<kBigItems, 512>();
  return e;
}

cudaError_t launch_hist(const HistArgs& a, int first_kind, int T, cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)((a.d.N + a.tile - 1) / a.tile);
  HistArgs arg = a;
  void* args[] = {&arg};
  const int radix = first_kind < 0 ? 128 : radix_buckets(a.rbits);
  size_t sm = 0;
  const void* fn = a.tile == kThreads * 4 ? hist_fn<4>(first_kind, radix, &sm, T)
                                          : hist_fn<kBigItems>(first_kind, radix, &sm, T);
  return launch_kernel(fn, dim3(grid), dim3(kThreads), sm, s, args, pdl);
}

cudaError_t launch_sort_pass(const PassArgs& a, bool wide_vals, int tile, unsigned grid, cudaStream_t s, bool pdl) {
  PassArgs arg = a;
  void* args[] = {&arg};
  size_t sm;
  const void* fn = pass_fn(wide_vals, tile, radix_buckets(a.rbits), &sm);
  return launch_kernel(fn, dim3(grid), dim3(kThreads), sm, s, args, pdl);
}

int pass_tile_class(int tile) { return tile == kThreads * 4 ? 0 : (tile == kThreads * 8 ? 1 : 2); }

int sort_pass_capacity(bool wide_vals, int tile, int rbits, int sms) {
  size_t sm;
  const void* fn = pass_fn(wide_vals, tile, radix_buckets(rbits), &sm);
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kThreads, sm) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return blocks * sms;
}

}  // namespace embbwd
