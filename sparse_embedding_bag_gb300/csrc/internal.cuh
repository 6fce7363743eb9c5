// Internal declarations shared by the CUDA translation units of libembbwd.
//
// Pipeline of one sorted call (all stream-ordered, no host synchronisation):
//   memset(ctl) -> k_hist -> k_sort_pass x passes -> k_runs -> k_reduce
// or, for batches small enough that every CTA of a per-table cluster holds its
// slice in shared memory (cfront.cu):
//   memset(ctl) -> k_cfront -> k_reduce
//   k_hist      linearises every lookup (hash_size_cumsum[t] + idx), checks it
//               against its table, validates the CSR offsets and builds, per
//               table, the digit histograms of all radix passes over the row
//               index in one read of the indices; its block 0 lays out the
//               passes' tiles on the tables' segments.
//   k_sort_pass one LSD radix pass over the row index (5..9-bit digits) with
//               decoupled look-back, each table's segment sorted on its own
//               (lookups arrive table-major, so the segments are already in key
//               order and only the row bits need sorting).
//   k_runs      run-length encode of the sorted keys (unique keys, run starts,
//               number of runs) fused with the ordered compaction of runs with
//               >= max_segment_length_per_warp lookups (with the prefix sum of
//               their lengths); one pass, decoupled look-back.
//   k_reduce    persistent: every warp first reduces an equal slice of the
//               concatenated long runs (runs cut by slice ends are combined from
//               fp32 partials in a fixed order), then strides over the short
//               runs in lane teams; fp32 accumulation of the scaled gradient rows
//               and the optimizer update fused in the same kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <type_traits>

namespace embbwd {

constexpr int kThreads = 256;  // every kernel uses 8 warps per block
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRadixBits = 9;  // digits of 1..9 bits: 2..512 buckets per pass
constexpr int kMaxPasses = 4;     // 32-bit row indices
constexpr int kRleItems = 8;   // sorted keys per thread of k_runs (16 for large batches)
constexpr int kRleTile = kThreads * kRleItems;  // smallest k_runs tile
constexpr int kMaxT = 4096;

// Device-side error bits (per call in Ctl::err, accumulated in the plan's sticky word).
constexpr uint32_t kErrIndex = 1u;
constexpr uint32_t kErrOffsets = 2u;
constexpr uint32_t kErrTimeout = 4u;
constexpr uint32_t kErrCapacity = 8u;

// Dynamic tile counters, one per kernel of a call.
enum TileCounter { TC_PASS0 = 0, TC_RLE = kMaxPasses, TC_COUNT = 8 };

// Per-call control block, zeroed by one memset at the start of every call.
struct Ctl {
  uint32_t err;
  uint32_t tile_ctr[TC_COUNT];
  uint32_t num_runs;
  uint32_t num_long;
  uint32_t long_lookups;  // lookups in long runs
  uint32_t pass_tiles;    // tiles of every radix pass (the tiles of all tables' segments)
  uint32_t pad[3];
  // Reduce: long-run slices handed out dynamically, one counter per warp index
  // of a block (each in its own 128-byte line).
  uint32_t slice_ctr[kWarps][32];
  // Reduce: short-run rounds claimed dynamically, the same way.
  uint32_t round_ctr[kWarps][32];
};
// The reduce's work counters are cleared together between its two launches of a
// row-wise update of wide rows: one range.
static_assert(offsetof(Ctl, round_ctr) == offsetof(Ctl, slice_ctr) + sizeof(Ctl::slice_ctr),
              "the reduce's work counters must be adjacent");

// Sort-value kinds: what travels with each key through the radix passes.
enum ValueKind {
  VK_BAG = 0,         // uint32 bag id t*B+b
  VK_BAG_SCALED = 1,  // uint64: bag id | float bits of (per-sample weight / L) << 32
  VK_NOBAG = 2,       // uint32 lookup position l (= gradient row)
};

// Decoupled look-back status words: [epoch:32 | flag:2 | count:30].
constexpr uint64_t kFlagAgg = 1ull << 30;
constexpr uint64_t kFlagInc = 2ull << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1;

struct LookbackCfg {
  uint64_t* status;     // [tiles][channels]
  uint32_t epoch;
  uint32_t spin_limit;
  uint32_t force_timeout;  // test flag: give up at once
};

// What every kernel needs to decode lookups of a tile.
struct DecodeArgs {
  const int64_t* indices;
  const int64_t* offsets;       // [BT+1]
  const float* psw;             // nullable
  const uint32_t* hsc;          // [T+1] (device copy of hash_size_cumsum)
  int64_t N;
  uint32_t B, T, BT;
  float invB;
  int mean;
};

// A tile of a radix pass: sorted positions [i0, i1) of table t, whose segment's
// first tile is `first`; seg0 is the first position of the table's segment and
// kbase = hash_size_cumsum[t] (kept here so a pass reads one entry, not three).
struct PassTile {
  uint32_t t, i0, i1, first, seg0, kbase;
};

struct HistArgs {
  DecodeArgs d;
  Ctl* ctl;
  uint32_t* sticky;
  int passes;
  int tile;              // lookups per block
  uint32_t* keys_out;    // linear keys in lookup order (not written when only checking)
  void* vals_out;        // payloads in lookup order
  uint32_t* thist;       // [T][passes][radix] digit counts of the row index, per table (zeroed)
  PassTile* tile_map;    // written by block 0: the passes' tiles, table by table
  int rbits;             // digit bits of a pass (radix = 1 << rbits, <= the kernel's bucket count)
  int ptile;             // lookups per tile of the passes
  uint32_t tile_cap;     // entries of tile_map (malformed offsets can ask for more; they are cut)
};

struct PassArgs {
  int64_t N;
  Ctl* ctl;
  uint32_t* sticky;
  LookbackCfg lb;
  const uint32_t* keys_in;
  const void* vals_in;
  uint32_t* keys_out;
  void* vals_out;
  const uint32_t* thist;      // [T][passes][radix]
  const PassTile* tile_map;   // [ctl->pass_tiles]
  int pass;
  int passes;
  int rbits;                  // the digit of pass p is bits [p*rbits, (p+1)*rbits) of the row index
  int ordered;  // 1: tile = blockIdx.x (the whole grid fits on the GPU at once)
};

// A long run: sorted lookups [start, start + len) of linear index `key`;
// lpos = lookups in the long runs before it (its place in the concatenation of
// all long runs, which the reduce cuts into equal slices).
struct __align__(16) LongRun {
  uint32_t start, len, key, lpos;
};

struct RunsArgs {
  const uint32_t* keys;  // sorted
  int64_t N;
  Ctl* ctl;
  uint32_t* sticky;
  LookbackCfg lb;
  uint32_t* run_key;
  uint32_t* run_start;   // [U+1]
  uint32_t thr;
  int ordered;  // 1: tile = blockIdx.x (the whole grid fits on the GPU at once)
  uint32_t* long_ids;
  LongRun* longs;
  uint32_t cap_long;
  // Segments of consecutive tables (see ReduceArgs::segs): with S > 1, the first
  // run of each segment is recorded (seg_runs[S] = number of runs).
  const uint32_t* seg_keys;  // [S+1]: first linear index of each segment, then the total rows
  uint32_t S;
  uint32_t* seg_runs;        // [S+1]
};

// Small-batch front (cfront.cu): one cluster of CTAs per table sorts and
// run-length encodes the table's segment; outputs as k_sort_pass + k_runs.
struct CfrontArgs {
  DecodeArgs d;
  Ctl* ctl;
  uint32_t* sticky;
  LookbackCfg lb;            // per-table look-back: 3 status words per table
  uint32_t* keys[2];         // pass p writes keys[p & 1] (the last pass: the sorted keys)
  void* vals[2];
  int passes, rbits;         // the digit of pass p is bits [p*rbits, (p+1)*rbits) of the row index
  uint32_t cap;              // lookups of one CTA's slice that its shared memory holds
  uint32_t* run_key;
  uint32_t* run_start;       // [U+1]
  uint32_t thr;
  uint32_t* long_ids;
  LongRun* longs;
  uint32_t cap_long;
  const uint32_t* segs;      // [S+1]: first table of each segment of tables with one team shape
  uint32_t S;
  uint32_t* seg_runs;        // [S+1] (written when S > 1)
};

struct ReduceArgs {
  Ctl* ctl;
  const uint32_t* vals;     // sorted values (uint32 or uint64, per value kind)
  const uint32_t* run_key;
  const uint32_t* run_start;
  const uint32_t* seg_runs;    // [S+1]: first run of each segment (S > 1 only)
  const uint32_t* segs;        // [S+1]: first table of each segment of tables with one team shape; segs[S] = T
  uint32_t S;
  const LongRun* longs;
  float4* partials;         // [2 * slices][KV*32]: head and tail piece of every slice
  uint32_t* done;           // [2 * slices]: arrived pieces of a group, at its first piece's slot
  uint32_t* done_run;       // [2 * slices]: arrived groups of a run, at its first piece's slot
  const void* grad;
  void* weights;
  float* momentum;
  const uint32_t* hsc;
  const int32_t* D_offsets;
  const int64_t* weights_offsets;
  const int64_t* momentum_offsets;
  uint32_t T, B;
  int64_t grad_stride;      // elements per gradient row (sum of D, or D unpooled)
  float lr, eps;
  void* grad_out;           // dense-gradient mode: weights-layout buffer that receives G
  int dense;                // 1: store G (SGD kernels) instead of updating the weights
  int sr;                   // 1: stochastic rounding of fp16 / bf16 weight stores
  uint32_t seed_lo, seed_hi, call_lo, call_hi;  // its random words: Philox key and call
  uint32_t thr, C;
  uint32_t min_slice;       // fewest long-run lookups per warp slice
  // Row-wise Adagrad of rows wider than one chunk (C > 1) takes two launches of
  // the reduce. rw_pass 1: every chunk of a run stores its sum of squares of G in
  // rw_ss[run * C + chunk]; the last chunk of the run to arrive (rw_cnt, reset to
  // 0 by it) adds them in chunk order, stores the new state to momentum and to
  // rw_m[run]. rw_pass 2: every chunk recomputes its G (the same summation order,
  // so the same bits) and applies w -= lr * G / (sqrt(rw_m[run]) + eps).
  // rw_pass 0: one launch (whole rows in one chunk).
  int rw_pass;
  float* rw_ss;             // [max_N * C]
  uint32_t* rw_cnt;         // [max_N], zero between calls
  float* rw_m;              // [max_N]
  const uint32_t* long_ids; // run index of every long run
};

struct FwdArgs {
  const void* weights;
  const int64_t* indices;
  const int64_t* offsets;          // [B*T+1]
  const float* psw;                // nullable
  void* out;                       // [B, out_stride]
  uint32_t* sticky;                // error bits
  const uint32_t* hsc;             // [T+1]
  const int32_t* D_offsets;        // [T+1]
  const int64_t* weights_offsets;  // [T]
  const uint32_t* segs;            // [S+1] segments of tables with one team shape
  uint32_t S, T, B;
  int64_t N;
  int64_t out_stride;              // D_offsets[T]
  int mean;
};

struct AtomicArgs {
  DecodeArgs d;
  Ctl* ctl;
  uint32_t* sticky;
  const void* grad;
  float* weights;
  const int64_t* weights_offsets;
  uint32_t D;
  float lr;
};

// ---------------------------------------------------------------------------
// Small device helpers.

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Programmatic dependent launch: every kernel of a call is launched so that
// it may start while its predecessor drains. pdl_wait() blocks until the
// predecessor grid has completed and its writes are visible (a no-op when the
// kernel was launched without the attribute); pdl_trigger() lets the next
// kernel start launching once every block of this grid has reached it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void raise_error(Ctl* ctl, uint32_t* sticky, uint32_t bits) {
  atomicOr(&ctl->err, bits);
  atomicOr(sticky, bits);
}

// Exclusive scan of one value per thread over a kThreads block. Returns the
// exclusive prefix; *total gets the block sum. `scratch` holds kWarps words.
// Contains __syncthreads(); every thread of the block must call it.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();  // scratch may still be read by a previous scan
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  uint32_t wbase = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = scratch[w];
    if (w < warp) wbase += s;
    tot += s;
  }
  *total = tot;
  return wbase + x - v;
}

// Exclusive scans of two values per thread at once (same barriers as one scan).
// `scratch` holds 2 * kWarps words. Every thread of the block must call it.
__device__ __forceinline__ void block_excl_scan2(uint32_t v0, uint32_t v1, uint32_t* scratch,
                                                 uint32_t* e0, uint32_t* e1, uint32_t* t0,
                                                 uint32_t* t1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x0 = v0, x1 = v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y0 = __shfl_up_sync(0xffffffffu, x0, o);
    const uint32_t y1 = __shfl_up_sync(0xffffffffu, x1, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
    }
  }
  __syncthreads();  // scratch may still be read by a previous scan
  if (lane == 31) {
    scratch[warp] = x0;
    scratch[kWarps + warp] = x1;
  }
  __syncthreads();
  uint32_t b0 = 0, b1 = 0, s0 = 0, s1 = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t a0 = scratch[w], a1 = scratch[kWarps + w];
    if (w < warp) {
      b0 += a0;
      b1 += a1;
    }
    s0 += a0;
    s1 += a1;
  }
  *e0 = b0 + x0 - v0;
  *e1 = b1 + x1 - v1;
  *t0 = s0;
  *t1 = s1;
}

// Decoupled look-back over DPT channels at once (the DPT digits a thread owns):
// publishes this tile's aggregates, walks back over the predecessors down to
// tile `first` (the first tile of the segment: nothing before it counts) until
// an inclusive prefix is found, publishes its own inclusive prefixes and returns
// the exclusive ones in excl. Channels c >= channels are skipped. Every wait is
// bounded: after spin_limit polls the tile raises kErrTimeout and carries on with
// what it has (its successors never wait forever, and nothing is updated in that
// call).
template <int DPT, int kWin>
__device__ __forceinline__ void lookback_channels(const LookbackCfg& lb, uint32_t tile, uint32_t first,
                                                  uint32_t channels, const uint32_t (&c)[DPT],
                                                  const uint32_t (&agg)[DPT], uint32_t (&excl)[DPT], Ctl* ctl,
                                                  uint32_t* sticky) {
  const uint64_t tag = (uint64_t)lb.epoch << 32;
  bool live[DPT];
#pragma unroll
  for (int q = 0; q < DPT; ++q) {
    live[q] = c[q] < channels;
    excl[q] = 0;
    if (live[q])
      st_relaxed_u64(lb.status + (size_t)tile * channels + c[q],
                     tag | (tile == first ? kFlagInc : kFlagAgg) | agg[q]);
  }
  if (tile == first) return;
  // Windowed walk: kWin predecessors are read per poll (independent loads in
  // flight), so a chain of tiles that published only aggregates is crossed kWin
  // tiles per memory round trip; every poll reads kWin words per channel, so
  // wide windows cost L2 traffic (see the callers for the measured choice).
  bool failed = lb.force_timeout != 0;
  int64_t j[DPT];
  bool done[DPT];
#pragma unroll
  for (int q = 0; q < DPT; ++q) {
    j[q] = (int64_t)tile - 1;
    done[q] = !live[q];
  }
  uint32_t polls = 0;
  while (!failed) {
    bool all = true, progress = true;
#pragma unroll
    for (int q = 0; q < DPT; ++q) {
      if (done[q]) continue;
      uint64_t w[kWin];
#pragma unroll
      for (int k = 0; k < kWin; ++k)
        w[k] = j[q] - k >= (int64_t)first ? ld_relaxed_u64(lb.status + (size_t)(j[q] - k) * channels + c[q])
                                          : (tag | kFlagInc);
      int m = 0;
      bool inc = false;
#pragma unroll
      for (int k = 0; k < kWin; ++k) {
        if (m != k) continue;  // an earlier word was not ready
        const uint64_t x = w[k];
        if ((uint32_t)(x >> 32) != lb.epoch || !(x & (kFlagAgg | kFlagInc))) continue;
        excl[q] += (uint32_t)x & kCountMask;
        if (x & kFlagInc) {
          inc = true;
          m = kWin + 1;
        } else {
          m = k + 1;
        }
      }
      if (inc) {
        done[q] = true;
        continue;
      }
      j[q] -= m;  // first tile not yet published (or the next window)
      all = false;
      if (m < kWin) progress = false;
    }
    if (all) break;
    if (!progress) {
      if (++polls > lb.spin_limit) {
        failed = true;
        break;
      }
      if (polls > 8) __nanosleep(polls > 128 ? 256 : 32);
    }
  }
  if (failed) raise_error(ctl, sticky, kErrTimeout);
#pragma unroll
  for (int q = 0; q < DPT; ++q)
    if (live[q])
      st_relaxed_u64(lb.status + (size_t)tile * channels + c[q], tag | kFlagInc | ((excl[q] + agg[q]) & kCountMask));
}

// Warp-wide decoupled look-back for one channel: all 32 lanes of a warp call
// it; lane k < WIN reads predecessor (j - k), so each round crosses up to WIN
// tiles that have published only aggregates. Same publication protocol and
// bounded waits as lookback_channels. Returns the exclusive prefix in every lane.
template <int WIN>
__device__ __forceinline__ uint32_t lookback_warp(const LookbackCfg& lb, uint32_t tile,
                                                  uint32_t channels, uint32_t c, uint32_t agg,
                                                  Ctl* ctl, uint32_t* sticky) {
  const uint32_t lane = threadIdx.x & 31;
  uint64_t* st = lb.status + (size_t)tile * channels + c;
  const uint64_t tag = (uint64_t)lb.epoch << 32;
  if (tile == 0) {
    if (lane == 0) st_relaxed_u64(st, tag | kFlagInc | agg);
    return 0;
  }
  if (lane == 0) st_relaxed_u64(st, tag | kFlagAgg | agg);
  uint32_t excl = 0;
  bool failed = lb.force_timeout != 0;
  int64_t j = (int64_t)tile - 1;
  uint32_t polls = 0;
  while (!failed) {
    const int64_t idx = j - (int64_t)lane;
    const uint64_t w = lane >= (uint32_t)WIN ? 0ull  // past the window: not ready, the walk stops there
                       : idx >= 0 ? ld_relaxed_u64(lb.status + (size_t)idx * channels + c)
                                  : (tag | kFlagInc);
    const bool ready = (uint32_t)(w >> 32) == lb.epoch && (w & (kFlagAgg | kFlagInc));
    const uint32_t nr = __ballot_sync(0xffffffffu, !ready);
    const uint32_t inc = __ballot_sync(0xffffffffu, ready && (w & kFlagInc));
    const uint32_t stop_nr = nr ? __ffs(nr) - 1 : 32u;
    const uint32_t stop_inc = inc ? __ffs(inc) - 1 : 32u;
    const bool found = stop_inc < stop_nr;
    const uint32_t take = found ? stop_inc + 1 : stop_nr;  // lanes [0, take) are summed
    uint32_t v = lane < take ? ((uint32_t)w & kCountMask) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    excl += v;
    if (found) break;
    j -= take;
    if (take < (uint32_t)WIN) {
      if (++polls > lb.spin_limit) failed = true;
      else if (polls > 8) __nanosleep(polls > 128 ? 256 : 32);
    }
  }
  if (failed && lane == 0) raise_error(ctl, sticky, kErrTimeout);
  if (lane == 0) st_relaxed_u64(st, tag | kFlagInc | ((excl + agg) & kCountMask));
  return excl;
}

// Table of a linear index: the last t with hash_size_cumsum[t] <= key (binary
// search over a shared-memory copy of the T+1 entries).
__device__ __forceinline__ uint32_t table_of(const uint32_t* s_hsc, uint32_t T, uint32_t key) {
  uint32_t lo = 0, hi = T - 1;
  while (lo < hi) {
    const uint32_t mid = (lo + hi + 1) >> 1;
    if (s_hsc[mid] <= key) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// t = bt / B without an integer divide: a float estimate corrected by one step
// each way (the estimate is off by at most one for bt < 2^31, T < 2^22).
__device__ __forceinline__ uint32_t div_by_B(uint32_t bt, uint32_t B, float invB) {
  uint32_t q = __float2uint_rz((float)bt * invB);
  if ((uint64_t)q * B > bt) --q;
  if ((uint64_t)(q + 1) * B <= bt) ++q;
  return q;
}

// ---- stochastic rounding of fp16 / bf16 stores.
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC 2011): ten rounds of two 32x32->64 multiplies by M0, M1 on a
// 4-word counter, the 2-word key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t p0 = (uint64_t)M0 * c.x, p1 = (uint64_t)M1 * c.z;  // one wide multiply each
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
                   (uint32_t)p0);
  }
  return c;
}

// fp32 x to bf16 bits, rounding away from zero with probability equal to the
// dropped fraction: 16 random bits added to the dropped half, then truncation.
__device__ __forceinline__ uint16_t sr_bf16(float x, uint32_t r) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  return (uint16_t)((u + (r & 0xFFFFu)) >> 16);
}

// fp32 x to fp16 bits: the neighbour toward zero, moved one ulp away from zero
// with probability (|x| - |lo|) / ulp, compared on 24 random bits. Both steps
// are exact in fp32: |x| - |lo| by Sterbenz (|lo| <= |x| < |lo| + ulp <= 2|lo|,
// or lo = 0), and the division by ulp = 2^(max(e,1) - 25) (e the exponent field
// of lo) is a multiplication by its exact power-of-two reciprocal. Beyond the
// largest finite value (hi would be inf) the result stays at the largest finite.
__device__ __forceinline__ uint16_t sr_half(float x, uint32_t r) {
  const __half h = __float2half_rz(x);
  const uint16_t lo = *reinterpret_cast<const uint16_t*>(&h);
  if ((lo & 0x7C00u) == 0x7C00u || (lo & 0x7FFFu) == 0x7BFFu) return lo;  // inf / nan / saturated
  const uint32_t e = max((uint32_t)(lo >> 10) & 0x1Fu, 1u);
  const float inv_ulp = __uint_as_float((127u + 25u - e) << 23);
  const float frac = (fabsf(x) - fabsf(__half2float(h))) * inv_ulp;
  return (r >> 8) < (uint32_t)(frac * 16777216.0f) ? (uint16_t)(lo + 1) : lo;
}

// ---- 4-element vector loads/stores of the storage types, as fp32.

template <typename T>
struct Vec4;

// Raw<T>: the loaded bits of 4 elements (16 bytes for fp32, 8 for 16-bit types),
// kept as loaded while a gather has loads in flight and widened to fp32 on use.
template <>
struct Vec4<float> {
  using Raw = float4;
  __device__ __forceinline__ static Raw load_raw(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
  __device__ __forceinline__ static Raw zero_raw() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ static float4 widen(Raw r) { return r; }
  __device__ __forceinline__ static float4 load(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
  __device__ __forceinline__ static float4 load_plain(const float* p) { return *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ static void store(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
  __device__ __forceinline__ static void store_sr(float* p, float4 v, uint4) { store(p, v); }
};

template <>
struct Vec4<__half> {
  using Raw = uint2;
  __device__ __forceinline__ static Raw load_raw(const __half* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
  __device__ __forceinline__ static Raw zero_raw() { return make_uint2(0u, 0u); }
  __device__ __forceinline__ static float4 widen(Raw r) { return cvt(r); }
  __device__ __forceinline__ static float4 cvt(uint2 u) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ __forceinline__ static float4 load(const __half* p) { return cvt(__ldg(reinterpret_cast<const uint2*>(p))); }
  __device__ __forceinline__ static float4 load_plain(const __half* p) { return cvt(*reinterpret_cast<const uint2*>(p)); }
  __device__ __forceinline__ static void store(__half* p, float4 v) {
    const __half2 a = __floats2half2_rn(v.x, v.y);
    const __half2 b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
  __device__ __forceinline__ static void store_sr(__half* p, float4 v, uint4 r) {
    uint2 u;
    u.x = (uint32_t)sr_half(v.x, r.x) | ((uint32_t)sr_half(v.y, r.y) << 16);
    u.y = (uint32_t)sr_half(v.z, r.z) | ((uint32_t)sr_half(v.w, r.w) << 16);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

template <>
struct Vec4<__nv_bfloat16> {
  using Raw = uint2;
  __device__ __forceinline__ static Raw load_raw(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
  __device__ __forceinline__ static Raw zero_raw() { return make_uint2(0u, 0u); }
  __device__ __forceinline__ static float4 widen(Raw r) { return cvt(r); }
  __device__ __forceinline__ static float4 cvt(uint2 u) {
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  }
  __device__ __forceinline__ static float4 load(const __nv_bfloat16* p) { return cvt(__ldg(reinterpret_cast<const uint2*>(p))); }
  __device__ __forceinline__ static float4 load_plain(const __nv_bfloat16* p) { return cvt(*reinterpret_cast<const uint2*>(p)); }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
  __device__ __forceinline__ static void store_sr(__nv_bfloat16* p, float4 v, uint4 r) {
    uint2 u;
    u.x = (uint32_t)sr_bf16(v.x, r.x) | ((uint32_t)sr_bf16(v.y, r.y) << 16);
    u.y = (uint32_t)sr_bf16(v.z, r.z) | ((uint32_t)sr_bf16(v.w, r.w) << 16);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the .cu files).

struct DevProps {
  int sms;
  int smem_optin;
};

// Launches fn(*args[0]) on `s`; with pdl set, as a programmatic dependent of
// the previous kernel on the stream (see pdl_wait / pdl_trigger).
inline cudaError_t launch_kernel(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 void** args, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// sort.cu
size_t sort_tile_for(int64_t N);  // lookups per block of the histogram kernel
size_t pass_tile_for(int64_t N);  // lookups per block of the radix passes: 1024, 2048 or 4096
int pass_tile_class(int tile);    // 0, 1, 2 for those
// Radix passes over row indices of `row_bits` bits: passes and digit bits.
void radix_plan(int row_bits, int* passes, int* rbits);
// Buckets of the kernels that serve digits of rbits bits (128, 256 or 512).
int radix_buckets(int rbits);
// first_kind: the ValueKind of the pairs to write, or -1 to only check indices and offsets.
cudaError_t launch_hist(const HistArgs& a, int first_kind, int T, cudaStream_t s, bool pdl);
// grid: tiles of the pass (an upper bound: blocks past ctl->pass_tiles exit).
cudaError_t launch_sort_pass(const PassArgs& a, bool wide_vals, int tile, unsigned grid, cudaStream_t s, bool pdl);
// Blocks of the pass kernel (and of k_runs) that fit on the GPU at once.
int sort_pass_capacity(bool wide_vals, int tile, int rbits, int sms);
int runs_capacity(int S, int items, int sms);
cudaError_t sort_configure(const DevProps& p);

// runs.cu: items = sorted keys per thread (8 or 16, runs_items_for(N)).
int runs_items_for(int64_t N);
cudaError_t launch_runs(const RunsArgs& a, int items, cudaStream_t s, bool pdl);
cudaError_t runs_configure();

// cfront.cu: the small-batch front. Shared memory of one CTA holding `cap`
// lookups; most clusters of cl CTAs resident at once (0 if none fit); launch of
// `clusters` clusters (one table each at a time, tables in order).
size_t cfront_smem(int vk, int radix, bool mean, uint32_t cap);
cudaError_t cfront_configure(int smem_optin);
int cfront_max_clusters(int vk, int radix, int cl, size_t smem);
cudaError_t launch_cfront(const CfrontArgs& a, int vk, int radix, int cl, int clusters, size_t smem,
                          cudaStream_t s, bool pdl);

// forward.cu: forward pooled lookup kernel of (weight type, output type, kv), or nullptr.
const void* fwd_kernel(int weight_dtype, int out_dtype, int kv);
size_t fwd_smem_bytes(int T, int S);

// reduce_<weight>_<grad>.cu: one entry per (weight type, gradient type) pair.
struct ReduceKey {
  int grad_dtype;   // 0 f32, 1 f16, 2 bf16
  int optimizer;    // 0 SGD (or dense gradient), 1 row-wise Adagrad, 2 elementwise Adagrad
  int value_kind;   // ValueKind
  int kv;           // 1, 2, 4, 8 vectors of 4 per lane
  bool multi;       // tables of several team shapes
};
// Kernel entry of the requested variant, or nullptr if the combination does not exist.
#define EMB_REDUCE_ENTRY(w, g) const void* reduce_kernel_##w##_##g(const ReduceKey& k);
EMB_REDUCE_ENTRY(f32, f32)
EMB_REDUCE_ENTRY(f32, f16)
EMB_REDUCE_ENTRY(f32, bf16)
EMB_REDUCE_ENTRY(f16, f32)
EMB_REDUCE_ENTRY(f16, f16)
EMB_REDUCE_ENTRY(f16, bf16)
EMB_REDUCE_ENTRY(bf16, f32)
EMB_REDUCE_ENTRY(bf16, f16)
EMB_REDUCE_ENTRY(bf16, bf16)
#undef EMB_REDUCE_ENTRY
inline size_t reduce_smem_bytes(int T) { return 4 * (size_t)(T + 1) * sizeof(uint32_t); }  // hsc, D, segments

// atomic.cu (the index / offsets check reuses launch_hist with passes = 0)
cudaError_t launch_nobag_atomic(const AtomicArgs& a, int grad_dtype, int T, cudaStream_t s, bool pdl);
cudaError_t atomic_configure();

}  // namespace embbwd
