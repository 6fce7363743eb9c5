// Row-wise sharding over W ranks: the exchange step of a deployment in which
// every rank trains on its own batch and owns a contiguous row range of every
// table (the vocabulary sharding of "Function _embedding_bwd_kernel": a device
// owns one slice of the rows and lookups outside it add nothing there), or, in
// the cyclic map, the rows congruent to its rank modulo W (local row = row / W),
// which spreads a skewed id distribution over all ranks.
//
//   bucketize (on every source rank): each lookup of the rank's batch goes to the
//     owner of its row; per owner, bag by bag in lookup order, the row relative to
//     the owner's range and the lookup's scale (per-sample weight, divided by the
//     length of its whole bag under mean pooling). Three kernels: per-(owner, bag)
//     counts, an exclusive scan of the counts (owner-major), a stable scatter.
//   (the caller exchanges the parts with an all-to-all and gathers grad_output)
//   merge (on every owner): the parts received from the W sources laid out as one
//     batch of W*B bags per table, table-major, bag s*B + b of table t holding
//     source s's bag (t, b): the layout whose gradient rows are the gathered
//     grad_output rows, so the owner's backward is the ordinary weighted-sum call.
//
// No kernel here waits on another block: scans are three-phase (block sums, one
// block over the sums, block rescans), so nothing can stall.
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <vector>

#include "embbwd.h"
#include "internal.cuh"

namespace embbwd {
namespace {

constexpr int kMaxW = 256;        // ranks of a shard map (per-warp counters in shared memory)
constexpr int kScanItems = 16;    // counts per thread of a scan block
constexpr uint32_t kScanChunk = kThreads * kScanItems;

struct BucketArgs {
  const int64_t* indices;
  const int64_t* offsets;   // [T*B+1]
  const float* psw;         // nullable
  const int64_t* bounds;    // [T][W+1] (cyclic: only [t][W], the rows of table t)
  int64_t N;
  uint32_t T, B, W;
  int mean;
  int cyclic;
  uint32_t* cnt;            // [W][T*B]: lookups of bag bt owned by r
  const int64_t* pos;       // [W*T*B+1]: exclusive scan of cnt
  int64_t* send_offsets;    // [W][T*B+1]
  int64_t* send_indices;    // [N]
  float* send_scales;       // [N] or null
  int64_t* counts;          // [W]: lookups per owner
  uint32_t* err;
};

struct ScanArgs {
  const uint32_t* in;
  int64_t* out;      // [n+1]
  int64_t* totals;   // [blocks]
  uint64_t n;
};

struct MergeArgs {
  const int64_t* recv_offsets;  // [W][T*B+1]
  const int64_t* recv_indices;
  const float* recv_scales;     // nullable
  int64_t n_recv;
  uint32_t T, B, W;
  int64_t* bases;               // [T*W]: first merged lookup of (table, source); then [W+1] source starts
  int64_t* merged_offsets;      // [T*W*B+1]
  int64_t* merged_indices;
  float* merged_scales;         // nullable
  uint32_t* err;
};

__device__ __forceinline__ uint32_t lanemask_lt_() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Owner of `row` (0 <= row < rb[W]): the r with rb[r] <= row < rb[r+1]. Binary
// search with the invariant rb[lo] <= row < rb[hi]; empty ranges never match.
__device__ __forceinline__ uint32_t owner_of(const int64_t* rb, uint32_t W, int64_t row) {
  uint32_t lo = 0, hi = W;
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (__ldg(&rb[mid]) <= row) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Owner of `row` (0 <= row < rows of its table) and the row's index on it.
__device__ __forceinline__ uint32_t route_row(const BucketArgs& a, const int64_t* rb, int64_t row,
                                              int64_t* local) {
  if (a.cyclic) {
    const int64_t q = row / a.W;
    *local = q;
    return (uint32_t)(row - q * a.W);
  }
  const uint32_t r = owner_of(rb, a.W, row);
  *local = row - __ldg(&rb[r]);
  return r;
}

// Exclusive scan of one int64 per thread over the block; *total gets the sum.
__device__ __forceinline__ int64_t block_excl_scan_i64(int64_t v, int64_t* scratch, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  int64_t wbase = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int64_t s = scratch[w];
    if (w < warp) wbase += s;
    tot += s;
  }
  *total = tot;
  return wbase + x - v;
}

// Bag bt's lookup range, or an empty one (and *bad) if the offsets are malformed.
__device__ __forceinline__ void bag_range(const BucketArgs& a, uint64_t bt, int64_t* s, int64_t* e,
                                          bool* bad) {
  *s = a.offsets[bt];
  *e = a.offsets[bt + 1];
  if (*s < 0 || *e < *s || *e > a.N) {
    *bad = true;
    *s = *e = 0;
  }
}

// Counts per (owner, bag): one warp per bag, shared-memory counters per warp.
__global__ void __launch_bounds__(kThreads) k_bucket_count(BucketArgs a) {
  __shared__ uint32_t s_cnt[kWarps][kMaxW];
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint32_t r = lane; r < a.W; r += 32) s_cnt[warp][r] = 0;
  __syncwarp();
  const uint64_t BT = (uint64_t)a.T * a.B;
  if (blockIdx.x == 0 && threadIdx.x == 0 && (a.offsets[0] != 0 || a.offsets[BT] != a.N))
    atomicOr(a.err, kErrOffsets);
  bool bad_index = false, bad_offsets = false;
  for (uint64_t bt = (uint64_t)blockIdx.x * kWarps + warp; bt < BT; bt += (uint64_t)gridDim.x * kWarps) {
    const uint32_t t = (uint32_t)(bt / a.B);
    const int64_t* rb = a.bounds + (uint64_t)t * (a.W + 1);
    const int64_t rows = __ldg(&rb[a.W]);
    int64_t s, e;
    bag_range(a, bt, &s, &e, &bad_offsets);
    for (int64_t i = s + lane; i < e; i += 32) {
      const int64_t row = a.indices[i];
      if (row < 0 || row >= rows) {
        bad_index = true;
        continue;
      }
      int64_t local;
      atomicAdd(&s_cnt[warp][route_row(a, rb, row, &local)], 1u);
    }
    __syncwarp();
    for (uint32_t r = lane; r < a.W; r += 32) {
      a.cnt[(uint64_t)r * BT + bt] = s_cnt[warp][r];
      s_cnt[warp][r] = 0;
    }
    __syncwarp();
  }
  if (bad_index) atomicOr(a.err, kErrIndex);
  if (bad_offsets) atomicOr(a.err, kErrOffsets);
}

// Counts of one scan chunk staged in shared memory (coalesced load), padded so
// that a thread's kScanItems consecutive counts fall in distinct banks.
__device__ __forceinline__ uint32_t pad_ix(uint32_t i) { return i + (i >> 5); }

__device__ __forceinline__ uint32_t stage_chunk(const ScanArgs& a, uint32_t* s_v) {
  const uint64_t base = (uint64_t)blockIdx.x * kScanChunk;
  for (uint32_t k = threadIdx.x; k < kScanChunk; k += kThreads) {
    const uint64_t i = base + k;
    s_v[pad_ix(k)] = i < a.n ? a.in[i] : 0u;
  }
  __syncthreads();
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) sum += s_v[pad_ix(threadIdx.x * kScanItems + k)];
  return sum;  // counts sum to at most N < 2^31
}

// Scan phase 1: the sum of every chunk.
__global__ void __launch_bounds__(kThreads) k_scan_sums(ScanArgs a) {
  __shared__ uint32_t s_v[kScanChunk + kScanChunk / 32];
  __shared__ uint32_t s_scr[kWarps];
  const uint32_t v = stage_chunk(a, s_v);
  uint32_t tot;
  block_excl_scan(v, s_scr, &tot);
  if (threadIdx.x == 0) a.totals[blockIdx.x] = tot;
}

// Scan phase 2 (one block): exclusive scan of the chunk sums in place; out[n] = total.
__global__ void __launch_bounds__(kThreads) k_scan_totals(ScanArgs a, uint32_t blocks) {
  __shared__ int64_t s_scr[kWarps];
  int64_t carry = 0;
  for (uint32_t c = 0; c < blocks; c += kThreads) {
    const uint32_t i = c + threadIdx.x;
    const int64_t v = i < blocks ? a.totals[i] : 0;
    int64_t tot;
    const int64_t ex = block_excl_scan_i64(v, s_scr, &tot);
    if (i < blocks) a.totals[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) a.out[a.n] = carry;
}

// Scan phase 3: every chunk rescanned with its block prefix.
__global__ void __launch_bounds__(kThreads) k_scan_out(ScanArgs a) {
  __shared__ uint32_t s_v[kScanChunk + kScanChunk / 32];
  __shared__ uint32_t s_scr[kWarps];
  const uint32_t v = stage_chunk(a, s_v);
  uint32_t tot;
  int64_t run = a.totals[blockIdx.x] + block_excl_scan(v, s_scr, &tot);
  const uint64_t base = (uint64_t)blockIdx.x * kScanChunk + (uint64_t)threadIdx.x * kScanItems;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < a.n) a.out[base + k] = run;
    run += s_v[pad_ix(threadIdx.x * kScanItems + k)];
  }
}

// Stable scatter of every lookup to its owner's part (one warp per bag; the
// lookups of one owner keep their order within the bag), then every owner's bag
// offsets counted from its first lookup, and the lookups per owner.
__global__ void __launch_bounds__(kThreads) k_bucket_scatter(BucketArgs a) {
  __shared__ uint32_t s_cnt[kWarps][kMaxW];
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint32_t r = lane; r < a.W; r += 32) s_cnt[warp][r] = 0;
  __syncwarp();
  const uint64_t BT = (uint64_t)a.T * a.B;
  bool overflow = false, bad_offsets = false;
  for (uint64_t bt = (uint64_t)blockIdx.x * kWarps + warp; bt < BT; bt += (uint64_t)gridDim.x * kWarps) {
    const uint32_t t = (uint32_t)(bt / a.B);
    const int64_t* rb = a.bounds + (uint64_t)t * (a.W + 1);
    const int64_t rows = __ldg(&rb[a.W]);
    int64_t s, e;
    bag_range(a, bt, &s, &e, &bad_offsets);
    const float L = (float)(e - s);  // the whole bag's length
    for (int64_t i0 = s; i0 < e; i0 += 32) {
      const int64_t i = i0 + lane;
      int32_t r = -1;
      int64_t local = 0;
      if (i < e) {
        const int64_t row = a.indices[i];
        if (row >= 0 && row < rows) r = (int32_t)route_row(a, rb, row, &local);
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, r);
      const uint32_t before = __popc(peers & lanemask_lt_());
      if (r >= 0) {
        const int64_t p = a.pos[(uint64_t)r * BT + bt] + s_cnt[warp][r] + before;
        if (p < 0 || p >= a.N) {
          overflow = true;
        } else {
          a.send_indices[p] = local;
          if (a.send_scales) {
            float sc = a.psw ? a.psw[i] : 1.0f;
            if (a.mean) sc = __fdiv_rn(sc, L);
            a.send_scales[p] = sc;
          }
        }
      }
      __syncwarp();
      if (r >= 0 && before == 0) s_cnt[warp][r] += __popc(peers);
      __syncwarp();
    }
    for (uint32_t r = lane; r < a.W; r += 32) s_cnt[warp][r] = 0;
    __syncwarp();
  }
  // owner r's offsets: pos[r*BT + j] - pos[r*BT], j = 0..BT (pos has W*BT+1 entries)
  const uint64_t n_off = (uint64_t)a.W * (BT + 1);
  for (uint64_t k = (uint64_t)blockIdx.x * kThreads + threadIdx.x; k < n_off; k += (uint64_t)gridDim.x * kThreads) {
    const uint64_t r = k / (BT + 1), j = k - r * (BT + 1);
    a.send_offsets[k] = a.pos[r * BT + j] - a.pos[r * BT];
  }
  if (blockIdx.x == 0)
    for (uint32_t r = threadIdx.x; r < a.W; r += kThreads) a.counts[r] = a.pos[(uint64_t)(r + 1) * BT] - a.pos[(uint64_t)r * BT];
  if (overflow) atomicOr(a.err, kErrCapacity);
  if (bad_offsets) atomicOr(a.err, kErrOffsets);
}

// Merge phase 1 (one block): first lookup of every source in the received
// buffers, and first merged lookup of every (table, source) block in
// table-major, then source order.
__global__ void __launch_bounds__(kThreads) k_merge_bases(MergeArgs a) {
  __shared__ int64_t s_scr[kWarps];
  const uint64_t BT = (uint64_t)a.T * a.B;
  int64_t* first = a.bases + (uint64_t)a.T * a.W;  // [W+1]
  int64_t carry = 0;
  for (uint32_t c = 0; c < a.W; c += kThreads) {
    const uint32_t s = c + threadIdx.x;
    const int64_t v = s < a.W ? a.recv_offsets[(uint64_t)s * (BT + 1) + BT] : 0;
    int64_t tot;
    const int64_t ex = block_excl_scan_i64(v, s_scr, &tot);
    if (s < a.W) first[s] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    first[a.W] = carry;
    if (carry != a.n_recv) atomicOr(a.err, kErrOffsets);
  }
  const uint64_t TW = (uint64_t)a.T * a.W;
  carry = 0;
  for (uint64_t c = 0; c < TW; c += kThreads) {
    const uint64_t q = c + threadIdx.x;  // q = t*W + s
    int64_t v = 0;
    if (q < TW) {
      const uint64_t t = q / a.W, s = q - t * a.W;
      const int64_t* ro = a.recv_offsets + s * (BT + 1);
      v = ro[(t + 1) * a.B] - ro[t * a.B];
    }
    int64_t tot;
    const int64_t ex = block_excl_scan_i64(v, s_scr, &tot);
    if (q < TW) a.bases[q] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) a.merged_offsets[(uint64_t)a.T * a.W * a.B] = carry;
}

// Merge phase 2. Offsets: merged bag q = (t*W + s)*B + b starts at the first
// merged lookup of block (t, s) plus bag b's place in source s's table-t part.
// Lookups: every (t, s) block is contiguous on both sides (source s's table-t
// lookups, in the received buffer and in the merged one), so each merged
// position j copies from its block's source start plus its offset in the block,
// the block found by a search of the block starts (staged in shared memory
// when they fit): coalesced reads and writes. Received offsets are checked
// against the received lookups; what does not fit is skipped and reported.
constexpr uint32_t kMergeStage = 2048;

__global__ void __launch_bounds__(kThreads) k_merge_copy(MergeArgs a) {
  __shared__ int64_t s_base[kMergeStage];
  const uint64_t BT = (uint64_t)a.T * a.B, WB = (uint64_t)a.W * a.B, Q = (uint64_t)a.T * WB;
  const uint64_t TW = (uint64_t)a.T * a.W;
  const int64_t* first = a.bases + TW;
  const bool staged = TW <= kMergeStage;
  if (staged) {
    for (uint32_t k = threadIdx.x; k < TW; k += kThreads) s_base[k] = a.bases[k];
    __syncthreads();
  }
  bool bad = false;
  const uint64_t stride = (uint64_t)gridDim.x * kThreads;
  for (uint64_t q = (uint64_t)blockIdx.x * kThreads + threadIdx.x; q < Q; q += stride) {
    const uint64_t t = q / WB, rem = q - t * WB, s = rem / a.B, b = rem - s * a.B;
    const int64_t* ro = a.recv_offsets + s * (BT + 1);
    const int64_t t0 = ro[t * a.B], lo = ro[t * a.B + b], hi = ro[t * a.B + b + 1];
    const int64_t base = staged ? s_base[t * a.W + s] : a.bases[t * a.W + s];
    // every term is checked against n_recv < 2^31 before it is added
    const bool ok = 0 <= t0 && t0 <= lo && lo <= hi && hi <= a.n_recv && 0 <= base &&
                    base <= a.n_recv && base + (lo - t0) <= a.n_recv;
    a.merged_offsets[q] = ok ? base + (lo - t0) : 0;
    bad |= !ok;
  }
  const int64_t total = min(first[a.W], a.n_recv);
  for (uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x; j < (uint64_t)max(total, (int64_t)0); j += stride) {
    // the block (t, s): the largest k with base[k] <= j (empty blocks never match)
    uint32_t lo = 0, hi = (uint32_t)TW;
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if ((staged ? s_base[mid] : a.bases[mid]) <= (int64_t)j) lo = mid;
      else hi = mid;
    }
    const uint32_t t = lo / a.W, s = lo - t * a.W;
    const int64_t base = staged ? s_base[lo] : a.bases[lo];
    const int64_t f = first[s], t0 = a.recv_offsets[(uint64_t)s * (BT + 1) + (uint64_t)t * a.B];
    const bool ok = 0 <= f && f <= a.n_recv && 0 <= t0 && t0 <= a.n_recv && base <= (int64_t)j &&
                    f + t0 + ((int64_t)j - base) < a.n_recv;
    if (!ok) {
      bad = true;
      continue;
    }
    const int64_t src = f + t0 + ((int64_t)j - base);
    a.merged_indices[j] = a.recv_indices[src];
    if (a.merged_scales) a.merged_scales[j] = a.recv_scales[src];
  }
  if (bad) atomicOr(a.err, kErrOffsets);
}

int warp_grid(uint64_t items, int sms) {
  const uint64_t blocks = (items + kWarps - 1) / kWarps;
  return (int)std::max<uint64_t>(1, std::min<uint64_t>(blocks, (uint64_t)sms * 8));
}

struct Guard {
  int prev = -1;
  bool ok = false;
  explicit Guard(int dev) {
    ok = cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess;
  }
  ~Guard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

emb_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return EMB_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? EMB_ERR_OOM : EMB_ERR_CUDA;
}

emb_status status_of_bits(uint32_t bits) {
  if (bits & kErrOffsets) return EMB_ERR_INVALID_ARG;
  if (bits & kErrIndex) return EMB_ERR_INDEX_OUT_OF_RANGE;
  if (bits & kErrCapacity) return EMB_ERR_INVALID_ARG;
  return EMB_OK;
}

}  // namespace
}  // namespace embbwd

using namespace embbwd;

struct emb_shard {
  int device = 0;
  int32_t T = 0, W = 0, max_B = 0;
  int cyclic = 0;
  int sms = 1;
  int64_t* d_bounds = nullptr;  // [T][W+1]
  uint32_t* cnt = nullptr;      // [W][T*max_B]
  int64_t* pos = nullptr;       // [W*T*max_B + 1]
  int64_t* totals = nullptr;    // scan chunk sums
  int64_t* counts = nullptr;    // [W]
  int64_t* bases = nullptr;     // [T*W + W + 1]
  uint32_t* err = nullptr;      // sticky error bits
  int64_t* h_counts = nullptr;  // pinned [W], then the error word
  cudaStream_t last_stream = nullptr;
};

namespace {

void free_shard(emb_shard* sh) {
  if (!sh) return;
  cudaFree(sh->d_bounds);
  cudaFree(sh->cnt);
  cudaFree(sh->pos);
  cudaFree(sh->totals);
  cudaFree(sh->counts);
  cudaFree(sh->bases);
  cudaFree(sh->err);
  cudaFreeHost(sh->h_counts);
  delete sh;
}

bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// Reads the sticky error word (after the stream has drained) and clears it.
emb_status take_errors(emb_shard* sh) {
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, sh->err, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(sh->err, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    return EMB_ERR_CUDA;
  }
  return status_of_bits(bits);
}

}  // namespace

namespace {

// row_bounds: [T][W+1] ranges, or (cyclic) only [t][W] = rows of table t is used.
emb_status create_shard(emb_shard** out, int device, int32_t T, int32_t W,
                        const int64_t* row_bounds, int32_t max_B, int cyclic) {
  if (!out) return EMB_ERR_INVALID_ARG;
  *out = nullptr;
  if (T <= 0 || T > kMaxT || W <= 0 || W > kMaxW || max_B <= 0 || !row_bounds) return EMB_ERR_INVALID_ARG;
  const uint64_t BT = (uint64_t)T * (uint64_t)max_B;
  if ((uint64_t)W * BT >= (1ull << 31)) return EMB_ERR_INVALID_ARG;
  for (int32_t t = 0; t < T; ++t) {
    const int64_t* rb = row_bounds + (int64_t)t * (W + 1);
    if (rb[W] <= 0) return EMB_ERR_INVALID_ARG;
    if (cyclic) continue;
    if (rb[0] != 0) return EMB_ERR_INVALID_ARG;
    for (int32_t r = 0; r < W; ++r)
      if (rb[r + 1] < rb[r]) return EMB_ERR_INVALID_ARG;
  }
  Guard g(device);
  if (!g.ok) return EMB_ERR_CUDA;
  emb_shard* sh = new emb_shard;
  sh->device = device;
  sh->T = T;
  sh->W = W;
  sh->max_B = max_B;
  sh->cyclic = cyclic;
  int sms = 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess) sh->sms = sms;
  const uint64_t n = (uint64_t)W * BT;
  const uint64_t chunks = (n + kScanChunk - 1) / kScanChunk;
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void** p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(p, bytes);
  };
  alloc(reinterpret_cast<void**>(&sh->d_bounds), sizeof(int64_t) * (size_t)T * (W + 1));
  alloc(reinterpret_cast<void**>(&sh->cnt), sizeof(uint32_t) * n);
  alloc(reinterpret_cast<void**>(&sh->pos), sizeof(int64_t) * (n + 1));
  alloc(reinterpret_cast<void**>(&sh->totals), sizeof(int64_t) * std::max<uint64_t>(chunks, 1));
  alloc(reinterpret_cast<void**>(&sh->counts), sizeof(int64_t) * W);
  alloc(reinterpret_cast<void**>(&sh->bases), sizeof(int64_t) * ((size_t)T * W + W + 1));
  alloc(reinterpret_cast<void**>(&sh->err), sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMallocHost(reinterpret_cast<void**>(&sh->h_counts), sizeof(int64_t) * W);
  if (e == cudaSuccess)
    e = cudaMemcpy(sh->d_bounds, row_bounds, sizeof(int64_t) * (size_t)T * (W + 1), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(sh->err, 0, sizeof(uint32_t));
  if (e != cudaSuccess) {
    const emb_status st = status_of(e);
    free_shard(sh);
    return st;
  }
  *out = sh;
  return EMB_OK;
}

}  // namespace

extern "C" {

emb_status emb_shard_create(emb_shard** out, int device, int32_t T, int32_t W,
                            const int64_t* row_bounds, int32_t max_B) {
  return create_shard(out, device, T, W, row_bounds, max_B, 0);
}

emb_status emb_shard_create_cyclic(emb_shard** out, int device, int32_t T, int32_t W,
                                   const int64_t* rows, int32_t max_B) {
  if (!rows || T <= 0 || T > kMaxT || W <= 0 || W > kMaxW) return EMB_ERR_INVALID_ARG;
  std::vector<int64_t> rb((size_t)T * (W + 1), 0);
  for (int32_t t = 0; t < T; ++t) rb[(size_t)t * (W + 1) + W] = rows[t];
  return create_shard(out, device, T, W, rb.data(), max_B, 1);
}

emb_status emb_shard_destroy(emb_shard* sh) {
  if (!sh) return EMB_OK;
  Guard g(sh->device);
  cudaDeviceSynchronize();
  free_shard(sh);
  return EMB_OK;
}

emb_status emb_shard_bucketize(emb_shard* sh, const int64_t* indices, const int64_t* offsets,
                               int64_t N, int32_t B, const float* per_sample_weights,
                               emb_pooling mode, int64_t* send_offsets, int64_t* send_indices,
                               float* send_scales, int64_t* send_counts, void* stream) {
  nvtxRangePushA("emb_shard_bucketize");
  struct Pop { ~Pop() { nvtxRangePop(); } } pop;
  if (!sh || !offsets || !send_offsets || !send_counts) return EMB_ERR_INVALID_ARG;
  if (B <= 0 || B > sh->max_B || N < 0 || N >= (1ll << 31)) return EMB_ERR_INVALID_ARG;
  if (mode != EMB_POOL_SUM && mode != EMB_POOL_MEAN) return EMB_ERR_INVALID_ARG;
  if (N > 0 && (!indices || !send_indices)) return EMB_ERR_INVALID_ARG;
  if (!aligned8(offsets) || !aligned8(send_offsets) || (indices && !aligned8(indices)) ||
      (send_indices && !aligned8(send_indices)))
    return EMB_ERR_INVALID_ARG;
  Guard g(sh->device);
  if (!g.ok) return EMB_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  sh->last_stream = s;
  const uint64_t BT = (uint64_t)sh->T * (uint64_t)B;
  const uint64_t n = (uint64_t)sh->W * BT;
  BucketArgs a;
  a.indices = indices;
  a.offsets = offsets;
  a.psw = per_sample_weights;
  a.bounds = sh->d_bounds;
  a.N = N;
  a.T = (uint32_t)sh->T;
  a.B = (uint32_t)B;
  a.W = (uint32_t)sh->W;
  a.mean = mode == EMB_POOL_MEAN;
  a.cyclic = sh->cyclic;
  a.cnt = sh->cnt;
  a.pos = sh->pos;
  a.send_offsets = send_offsets;
  a.send_indices = send_indices;
  a.send_scales = send_scales;
  a.counts = sh->counts;
  a.err = sh->err;
  ScanArgs sc{sh->cnt, sh->pos, sh->totals, n};
  const uint32_t chunks = (uint32_t)((n + kScanChunk - 1) / kScanChunk);
  const int grid = warp_grid(BT, sh->sms);
  {
    void* args[] = {&a};
    if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_bucket_count), dim3(grid),
                                      dim3(kThreads), 0, s, args, false))
      return status_of(e);
  }
  {
    void* args[] = {&sc};
    if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_scan_sums), dim3(chunks),
                                      dim3(kThreads), 0, s, args, false))
      return status_of(e);
    uint32_t blocks = chunks;
    void* args2[] = {&sc, &blocks};
    if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_scan_totals), dim3(1),
                                      dim3(kThreads), 0, s, args2, false))
      return status_of(e);
    if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_scan_out), dim3(chunks),
                                      dim3(kThreads), 0, s, args, false))
      return status_of(e);
  }
  {
    void* args[] = {&a};
    if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_bucket_scatter), dim3(grid),
                                      dim3(kThreads), 0, s, args, false))
      return status_of(e);
  }
  // the exchange needs the per-owner sizes on the host
  if (cudaError_t e = cudaMemcpyAsync(sh->h_counts, sh->counts, sizeof(int64_t) * sh->W,
                                      cudaMemcpyDeviceToHost, s))
    return status_of(e);
  if (cudaError_t e = cudaStreamSynchronize(s)) return status_of(e);
  const emb_status st = take_errors(sh);
  if (st != EMB_OK) return st;
  std::copy(sh->h_counts, sh->h_counts + sh->W, send_counts);
  return EMB_OK;
}

emb_status emb_shard_merge(emb_shard* sh, const int64_t* recv_offsets, const int64_t* recv_indices,
                           const float* recv_scales, int64_t n_recv, int32_t B,
                           int64_t* merged_offsets, int64_t* merged_indices, float* merged_scales,
                           void* stream) {
  nvtxRangePushA("emb_shard_merge");
  struct Pop { ~Pop() { nvtxRangePop(); } } pop;
  if (!sh || !recv_offsets || !merged_offsets) return EMB_ERR_INVALID_ARG;
  if (B <= 0 || B > sh->max_B || n_recv < 0 || n_recv >= (1ll << 31)) return EMB_ERR_INVALID_ARG;
  if (n_recv > 0 && (!recv_indices || !merged_indices)) return EMB_ERR_INVALID_ARG;
  if ((recv_scales == nullptr) != (merged_scales == nullptr)) return EMB_ERR_INVALID_ARG;
  if (!aligned8(recv_offsets) || !aligned8(merged_offsets) ||
      (recv_indices && !aligned8(recv_indices)) || (merged_indices && !aligned8(merged_indices)))
    return EMB_ERR_INVALID_ARG;
  Guard g(sh->device);
  if (!g.ok) return EMB_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  sh->last_stream = s;
  MergeArgs m;
  m.recv_offsets = recv_offsets;
  m.recv_indices = recv_indices;
  m.recv_scales = recv_scales;
  m.n_recv = n_recv;
  m.T = (uint32_t)sh->T;
  m.B = (uint32_t)B;
  m.W = (uint32_t)sh->W;
  m.bases = sh->bases;
  m.merged_offsets = merged_offsets;
  m.merged_indices = merged_indices;
  m.merged_scales = merged_scales;
  m.err = sh->err;
  void* args[] = {&m};
  if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_merge_bases), dim3(1),
                                    dim3(kThreads), 0, s, args, false))
    return status_of(e);
  const uint64_t items = std::max<uint64_t>((uint64_t)sh->T * sh->W * (uint64_t)B, (uint64_t)n_recv);
  const uint64_t blocks = std::min<uint64_t>((items + kThreads - 1) / kThreads, (uint64_t)sh->sms * 8);
  if (cudaError_t e = launch_kernel(reinterpret_cast<const void*>(&k_merge_copy),
                                    dim3((unsigned)std::max<uint64_t>(blocks, 1)), dim3(kThreads), 0, s,
                                    args, false))
    return status_of(e);
  return EMB_OK;
}

emb_status emb_shard_status(emb_shard* sh) {
  if (!sh) return EMB_ERR_INVALID_ARG;
  Guard g(sh->device);
  if (!g.ok) return EMB_ERR_CUDA;
  if (cudaStreamSynchronize(sh->last_stream) != cudaSuccess) {
    cudaGetLastError();
    return EMB_ERR_CUDA;
  }
  return take_errors(sh);
}

}  // extern "C"
