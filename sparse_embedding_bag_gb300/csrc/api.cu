// C ABI of libembbwd: argument validation, plan (scratch) management and the
// per-call launch sequence. Host code only; the kernels live in the other
// translation units. The host layer mirrors the checks of the exact_cuda host
// function of "fbgemm_gpu/codegen/embedding_backward_split_template.cu"
// (T > 0, B > 0, the embedding-dimension limit, the empty-indices
// short-circuit) and adds the alignment and capacity checks the vectorised
// kernels need.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/embbwd.h"
#include "internal.cuh"

using namespace embbwd;

namespace {

// An NVTX range over one entry point's host work: a timeline tool shows the
// launches of the call under it. A no-op when no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr uint32_t kSpinLimit = 1u << 22;  // polls before a look-back wait gives up (~1 s)
constexpr uint32_t kMinSlice = 8;          // fewest long-run lookups a reduce warp slice can have
// Fewest long-run lookups per warp slice when there is little long-run work (one
// slice per warp at most): below it, fewer warps take the long runs and the rest
// start on the short runs at once. Measured on GB300 (DLRM-like batch, 45 long-run
// lookups per warp): reduce 26.7 us with a floor of 64, 27.3 at 128, 36.0 at 256.
constexpr uint32_t kStaticMinSlice = 64;
constexpr int kStages = 5;
// Largest batch the small-batch front takes. Its CTAs hold their slices of a
// table in shared memory (ceil(N / CTAs per cluster) lookups each), which allows
// up to about 2^18 lookups; measured on GB300 (CUDA graph, PDL, L2 flushed) it
// runs the tiny batch in 24.5 instead of 29.1 us per step and the LM one (32k
// lookups, one table) in 129.7 instead of 130.0 us, but the DLRM-like one (172k
// lookups over 8 tables) in 61.3 instead of 61.0 us, so it stops at 2^16.
constexpr int64_t kCfMaxN = (int64_t)1 << 16;
// CTAs per cluster, in order of preference: the largest size of which one
// cluster per table fits on the GPU at once. Measured on GB300 at one CTA per
// SM (shared memory above half an SM): 7 clusters of 16 CTAs, 8 of 12, 15 of 8.
constexpr int kCfSizes[4] = {16, 12, 8, 4};

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

uint32_t pow2floor(uint64_t x) {
  uint32_t r = 1;
  while ((uint64_t)r * 2 <= x && r < (1u << 30)) r *= 2;
  return r;
}

}  // namespace

struct emb_plan {
  int device = 0;
  int32_t T = 0;
  emb_dtype wdt = EMB_F32, gdt = EMB_F32;
  int64_t max_N = 0;
  int32_t max_B = 0;
  uint32_t thr = 32;
  uint32_t flags = 0;
  uint64_t sr_seed = 0, sr_call = 0;  // stochastic rounding: Philox key, next call number
  int max_D = 0;
  bool uniform_D = true;
  // How the reduce splits rows: 0 pooled SGD (and the other per-element updates),
  // 1 row-wise Adagrad, 2 unpooled lookups (see split_index).
  struct RowSplit {
    int kv = 1;                     // 16-byte vectors per lane
    uint32_t C = 1;                 // chunks of kv*32 vectors per row
    // Segments of consecutive tables whose rows give the reduce the same team
    // shape (chunks per row, lanes per lookup): first table of each, then T.
    std::vector<uint32_t> segs;
    uint32_t* d_segs = nullptr;
    uint32_t* d_segkeys = nullptr;  // hash_size_cumsum of each segment's first table, then the total
  } split[3];
  int key_bits = 1;
  int passes = 1, rbits = 1;      // radix passes over row indices and their digit bits
  int radix = 128;                // buckets of the sort kernels for rbits
  uint32_t max_pass_tiles = 0;    // upper bound on the tiles of a pass (all call sizes)
  std::vector<uint32_t> hsc;
  std::vector<int32_t> Do;
  DevProps props{};

  void* arena = nullptr;
  Ctl* ctl = nullptr;
  uint32_t* thist = nullptr;     // [T][passes][radix] digit counts per table, cleared with ctl
  size_t clear_bytes = 0;        // bytes from ctl to the end of thist
  PassTile* tile_map = nullptr;  // [max_pass_tiles]
  uint32_t* sticky = nullptr;
  uint32_t* d_hsc = nullptr;
  int32_t* d_Do = nullptr;
  int64_t* d_wo = nullptr;
  int64_t* d_mo = nullptr;
  uint32_t* keys[2] = {nullptr, nullptr};
  void* vals[2] = {nullptr, nullptr};
  uint64_t* status = nullptr;
  uint32_t* run_key = nullptr;
  uint32_t* run_start = nullptr;
  uint32_t* seg_runs = nullptr;  // [T+1]: first run of each segment of the call's split
  uint32_t* long_ids = nullptr;
  LongRun* longs = nullptr;
  float4* partials = nullptr;
  uint32_t* done = nullptr;
  // row-wise Adagrad of rows of several chunks (split[1].C > 1): per-run sums of
  // squares of each chunk, arrival counters (zero between calls), new states
  float* rw_ss = nullptr;
  uint32_t* rw_cnt = nullptr;
  float* rw_m = nullptr;
  uint32_t cap_long = 0, cap_slices = 0;

  uint32_t seq = 0;
  int reduce_grid[3][3] = {{0, 0, 0}, {0, 0, 0}, {0, 0, 0}};  // [optimizer][value kind]
  int64_t w_extent = 0;  // elements of the weights layout: max over t of offset + rows * D
  // Blocks that fit on the GPU at once: sort pass [tile class][wide payload], k_runs
  // [split][8 or 16 keys per thread].
  int pass_cap[3][2] = {{0, 0}, {0, 0}, {0, 0}};  // [pass tile class][wide values]
  int runs_cap[3][2] = {{0, 0}, {0, 0}, {0, 0}};
  int fwd_grid[3] = {0, 0, 0};  // forward kernel grid per output type (0: not set up yet)
  // Small-batch front: clusters of each size in kCfSizes that can be resident
  // at once, per value kind (0: that cluster size does not fit), for calls of
  // at most cf_max_N lookups.
  int cf_clusters[3][4] = {};  // [value kind][kCfSizes index]
  int64_t cf_max_N = 0;
  cudaStream_t last_stream = nullptr;
  int last_kind = 0;  // 0 none / empty, 1 sorted, 2 atomic
  int64_t last_N = 0;

  bool profiling = false;
  bool events_ready = false;
  cudaEvent_t ev[kStages + 1] = {};
  int last_profiled = 0;  // 0 none, 1 sorted, 2 atomic
};

namespace {

// Row split of a call: row-wise Adagrad keeps whole rows in one warp; unpooled
// lookups (whole-warp rows of one table width, no bag to share) and pooled
// per-element updates split rows differently (see the plan).
int split_index(int opt, int vk) { return opt == 1 ? 1 : (vk == VK_NOBAG ? 2 : 0); }

const void* reduce_fn(const emb_plan* p, int opt, int vk) {
  const emb_plan::RowSplit& sp = p->split[split_index(opt, vk)];
  const ReduceKey k{static_cast<int>(p->gdt), opt, vk, sp.kv, sp.segs.size() > 2};
  static const void* (*const entry[3][3])(const ReduceKey&) = {
      {reduce_kernel_f32_f32, reduce_kernel_f32_f16, reduce_kernel_f32_bf16},
      {reduce_kernel_f16_f32, reduce_kernel_f16_f16, reduce_kernel_f16_bf16},
      {reduce_kernel_bf16_f32, reduce_kernel_bf16_f16, reduce_kernel_bf16_bf16}};
  return entry[static_cast<int>(p->wdt)][static_cast<int>(p->gdt)](k);
}

emb_status record(emb_plan* p, int i, cudaStream_t s) {
  if (!p->profiling) return EMB_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return EMB_ERR_CUDA;
  const cudaError_t e = cs == cudaStreamCaptureStatusActive
                            ? cudaEventRecordWithFlags(p->ev[i], s, cudaEventRecordExternal)
                            : cudaEventRecord(p->ev[i], s);
  return e == cudaSuccess ? EMB_OK : EMB_ERR_CUDA;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

size_t dtype_size(emb_dtype d) { return d == EMB_F32 ? 4 : 2; }

emb_status check_common(const emb_plan* p, const void* weights, const int64_t* indices,
                        const int64_t* offsets, int64_t N, int32_t B, const void* grad) {
  if (!p) return EMB_ERR_INVALID_ARG;
  if (N < 0 || N > p->max_N || B <= 0 || B > p->max_B) return EMB_ERR_INVALID_ARG;
  if (N == 0) return EMB_OK;
  if (!weights || !indices || !offsets || !grad) return EMB_ERR_INVALID_ARG;
  if (!aligned(weights, 4 * dtype_size(p->wdt)) || !aligned(grad, 4 * dtype_size(p->gdt)) ||
      !aligned(indices, 8) || !aligned(offsets, 8))
    return EMB_ERR_INVALID_ARG;
  return EMB_OK;
}

DecodeArgs decode_args(const emb_plan* p, const int64_t* indices, const int64_t* offsets,
                       const float* psw, int64_t N, int32_t B, int mean) {
  DecodeArgs d;
  d.indices = indices;
  d.offsets = offsets;
  d.psw = psw;
  d.hsc = p->d_hsc;
  d.N = N;
  d.B = (uint32_t)B;
  d.T = (uint32_t)p->T;
  d.BT = (uint32_t)B * (uint32_t)p->T;
  d.invB = 1.0f / (float)B;
  d.mean = mean;
  return d;
}

emb_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return EMB_OK;
  cudaGetLastError();  // clear a sticky launch error
  return e == cudaErrorMemoryAllocation ? EMB_ERR_OOM : EMB_ERR_CUDA;
}

#define EMB_TRY(expr)                     \
  do {                                    \
    const emb_status _st = (expr);        \
    if (_st != EMB_OK) return _st;        \
  } while (0)
#define EMB_CUDA(expr) EMB_TRY(cuda_status(expr))

// Sorted path: linearise + sort + run-length + long partition + fused reduce/update.
// opt: 0 SGD (or, with dense, the gradient stored to grad_out), 1 row-wise Adagrad,
// 2 elementwise Adagrad.
emb_status run_sorted(emb_plan* p, int opt, int vk, void* weights, float* momentum,
                      const int64_t* indices, const int64_t* offsets, int64_t N, int32_t B,
                      const float* psw, const void* grad, int mean, float lr, float eps,
                      void* grad_out, int dense, cudaStream_t s) {
  const int si = split_index(opt, vk);
  const uint32_t epoch = ++p->seq * 8u;
  if (p->seq >= (1u << 28)) p->seq = 0;  // epochs stay distinct from the zero-initialised words
  const DecodeArgs d = decode_args(p, indices, offsets, psw, N, B, mean);
  const int tile = (int)sort_tile_for(N), ptile = (int)pass_tile_for(N);
  const int passes = p->passes;
  const bool wide = vk == VK_BAG_SCALED;
  const LookbackCfg lb0{p->status, epoch, kSpinLimit, (p->flags & EMB_FLAG_DEBUG_FORCE_TIMEOUT) ? 1u : 0u};
  const bool pdl = !(p->flags & EMB_FLAG_NO_PDL);

  EMB_TRY(record(p, 0, s));
  // the small-batch front: one cluster per table, all resident at once
  int cl = 0;
  size_t cf_sm = 0;
  const uint32_t* d_segs = p->split[si].d_segs;
  const uint32_t S = (uint32_t)p->split[si].segs.size() - 1;
  const int fin = (passes - 1) & 1;  // the buffers the last pass writes (both fronts)
  if (N <= p->cf_max_N) {
    for (int i = 0; i < 4 && !cl; ++i) {
      if (p->T > p->cf_clusters[vk][i]) continue;
      cf_sm = cfront_smem(vk, p->radix, mean != 0, (uint32_t)((N + kCfSizes[i] - 1) / kCfSizes[i]));
      if (cf_sm <= (size_t)p->props.smem_optin) cl = kCfSizes[i];
    }
  }
  if (cl) {
    EMB_CUDA(cudaMemsetAsync(p->ctl, 0, sizeof(Ctl), s));  // control block only
    CfrontArgs ca;
    ca.d = d;
    ca.ctl = p->ctl;
    ca.sticky = p->sticky;
    ca.lb = lb0;
    ca.lb.epoch = epoch + 6;
    ca.keys[0] = p->keys[0];
    ca.keys[1] = p->keys[1];
    ca.vals[0] = p->vals[0];
    ca.vals[1] = p->vals[1];
    ca.passes = passes;
    ca.rbits = p->rbits;
    ca.cap = (uint32_t)((N + cl - 1) / cl);
    ca.run_key = p->run_key;
    ca.run_start = p->run_start;
    ca.thr = p->thr;
    ca.long_ids = p->long_ids;
    ca.longs = p->longs;
    ca.cap_long = p->cap_long;
    ca.segs = d_segs;
    ca.S = S;
    ca.seg_runs = p->seg_runs;
    EMB_CUDA(launch_cfront(ca, vk, p->radix, cl, p->T, cf_sm, s, pdl));
    EMB_TRY(record(p, 1, s));  // one kernel: the sort and run-length stages are empty
    EMB_TRY(record(p, 2, s));
    EMB_TRY(record(p, 3, s));
  } else {
  EMB_CUDA(cudaMemsetAsync(p->ctl, 0, p->clear_bytes, s));  // control block and per-table histograms
  // the linearised pairs go to buffer 1, which the first pass reads
  HistArgs ha{d,           p->ctl,       p->sticky, passes, tile, p->keys[1], p->vals[1],
              p->thist,    p->tile_map,  p->rbits,  ptile,  p->max_pass_tiles};
  EMB_CUDA(launch_hist(ha, vk, p->T, s, pdl));
  EMB_TRY(record(p, 1, s));
  // tiles of a pass: at most one partial tile per table on top of N / ptile
  const unsigned pgrid = (unsigned)((N + ptile - 1) / ptile + p->T);
  for (int pass = 0; pass < passes; ++pass) {
    PassArgs pa;
    pa.N = N;
    pa.ctl = p->ctl;
    pa.sticky = p->sticky;
    pa.lb = lb0;
    pa.lb.epoch = epoch + (uint32_t)pass;
    const int in = (pass + 1) & 1, out = pass & 1;
    pa.keys_in = p->keys[in];
    pa.vals_in = p->vals[in];
    pa.keys_out = p->keys[out];
    pa.vals_out = p->vals[out];
    pa.thist = p->thist;
    pa.tile_map = p->tile_map;
    pa.pass = pass;
    pa.passes = passes;
    pa.rbits = p->rbits;
    pa.ordered = (int)pgrid <= p->pass_cap[pass_tile_class(ptile)][wide ? 1 : 0];
    EMB_CUDA(launch_sort_pass(pa, wide, ptile, pgrid, s, pdl));
  }
  EMB_TRY(record(p, 2, s));
  RunsArgs ra;
  ra.keys = p->keys[fin];
  ra.N = N;
  ra.ctl = p->ctl;
  ra.sticky = p->sticky;
  ra.lb = lb0;
  ra.lb.epoch = epoch + 5;
  ra.run_key = p->run_key;
  ra.run_start = p->run_start;
  ra.thr = p->thr;
  const int items = runs_items_for(N);
  ra.ordered = (N + (int64_t)kThreads * items - 1) / ((int64_t)kThreads * items) <= p->runs_cap[si][items == 16];
  ra.long_ids = p->long_ids;
  ra.longs = p->longs;
  ra.cap_long = p->cap_long;
  ra.seg_keys = p->split[si].d_segkeys;
  ra.S = S;
  ra.seg_runs = p->seg_runs;
  EMB_CUDA(launch_runs(ra, items, s, pdl));
  EMB_TRY(record(p, 3, s));  // run-length and long-run partition are one kernel (no event 4)
  }

  ReduceArgs r;
  r.ctl = p->ctl;
  r.vals = static_cast<const uint32_t*>(p->vals[fin]);
  r.run_key = p->run_key;
  r.run_start = p->run_start;
  r.seg_runs = p->seg_runs;
  r.segs = d_segs;
  r.S = S;
  r.longs = p->longs;
  r.partials = p->partials;
  r.done = p->done;
  r.done_run = p->done + 2 * (size_t)p->cap_slices;
  r.grad = grad;
  r.weights = weights;
  r.momentum = momentum;
  r.hsc = p->d_hsc;
  r.D_offsets = p->d_Do;
  r.weights_offsets = p->d_wo;
  r.momentum_offsets = p->d_mo;
  r.T = (uint32_t)p->T;
  r.B = (uint32_t)B;
  r.grad_stride = vk == VK_NOBAG ? (int64_t)p->max_D : (int64_t)p->Do[p->T];
  r.lr = lr;
  r.eps = eps;
  r.thr = p->thr;
  r.min_slice = kStaticMinSlice;
  r.C = p->split[si].C;
  r.grad_out = grad_out;
  r.dense = dense;
  r.sr = (p->flags & EMB_FLAG_STOCHASTIC_ROUNDING) && !dense && p->wdt != EMB_F32;
  if (r.sr) {
    const uint64_t call = p->sr_call++;
    r.seed_lo = (uint32_t)p->sr_seed;
    r.seed_hi = (uint32_t)(p->sr_seed >> 32);
    r.call_lo = (uint32_t)call;
    r.call_hi = (uint32_t)(call >> 32);
  }
  r.rw_pass = 0;
  r.rw_ss = p->rw_ss;
  r.rw_cnt = p->rw_cnt;
  r.rw_m = p->rw_m;
  r.long_ids = p->long_ids;
  const void* fn = reduce_fn(p, opt, vk);
  if (!fn) return EMB_ERR_UNSUPPORTED;
  void* args[] = {&r};
  if (opt == 1 && r.C > 1) {
    // Row-wise Adagrad of rows of several chunks: the first launch finds every
    // row's new state from its chunks' sums of squares, the second updates the
    // weights; the reduce's work counters start again from zero in between.
    r.rw_pass = 1;
    EMB_CUDA(launch_kernel(fn, dim3(p->reduce_grid[opt][vk]), dim3(kThreads),
                           reduce_smem_bytes(p->T), s, args, pdl));
    EMB_CUDA(cudaMemsetAsync(&p->ctl->slice_ctr[0][0], 0, sizeof(p->ctl->slice_ctr) + sizeof(p->ctl->round_ctr), s));
    r.rw_pass = 2;
  }
  EMB_CUDA(launch_kernel(fn, dim3(p->reduce_grid[opt][vk]), dim3(kThreads),
                         reduce_smem_bytes(p->T), s, args, pdl));
  EMB_TRY(record(p, 5, s));
  p->last_kind = 1;
  p->last_N = N;
  p->last_stream = s;
  if (p->profiling) p->last_profiled = 1;
  return EMB_OK;
}

}  // namespace

extern "C" {

const char* emb_status_string(emb_status st) {
  switch (st) {
    case EMB_OK: return "ok";
    case EMB_ERR_INVALID_ARG: return "invalid argument";
    case EMB_ERR_UNSUPPORTED: return "unsupported";
    case EMB_ERR_INDEX_OUT_OF_RANGE: return "index out of range";
    case EMB_ERR_OOM: return "out of device memory";
    case EMB_ERR_CUDA: return "CUDA runtime error";
    case EMB_ERR_TIMEOUT: return "bounded wait timed out";
  }
  return "unknown status";
}

emb_status emb_bwd_plan(emb_plan** out, int device, int32_t T, const int64_t* hash_size_cumsum,
                        const int32_t* D_offsets, const int64_t* weights_offsets,
                        const int64_t* momentum_offsets, emb_dtype weight_dtype,
                        emb_dtype grad_dtype, int64_t max_N, int32_t max_B,
                        int32_t max_segment_length_per_warp, uint32_t flags) {
  NvtxRange nvtx("emb_bwd_plan");
  if (!out) return EMB_ERR_INVALID_ARG;
  *out = nullptr;
  // ---- host-side validation (no CUDA call before this point)
  if (T <= 0 || T > kMaxT || !hash_size_cumsum || !D_offsets || !weights_offsets)
    return EMB_ERR_INVALID_ARG;
  if (weight_dtype < EMB_F32 || weight_dtype > EMB_BF16 || grad_dtype < EMB_F32 || grad_dtype > EMB_BF16)
    return EMB_ERR_INVALID_ARG;
  if (max_N < 0 || max_N >= (int64_t)(1 << 30) || max_B <= 0 || (int64_t)max_B * T >= (int64_t)1 << 31)
    return EMB_ERR_INVALID_ARG;
  if (hash_size_cumsum[0] != 0 || D_offsets[0] != 0) return EMB_ERR_INVALID_ARG;
  int max_D = 0;
  bool uniform = true;
  for (int32_t t = 0; t < T; ++t) {
    if (hash_size_cumsum[t + 1] <= hash_size_cumsum[t]) return EMB_ERR_INVALID_ARG;
    const int32_t D = D_offsets[t + 1] - D_offsets[t];
    if (D <= 0 || D % 4 != 0 || D > 4096) return EMB_ERR_INVALID_ARG;
    if (weights_offsets[t] < 0 || weights_offsets[t] % 4 != 0) return EMB_ERR_INVALID_ARG;
    if (momentum_offsets && momentum_offsets[t] < 0) return EMB_ERR_INVALID_ARG;
    if (D != D_offsets[1] - D_offsets[0]) uniform = false;
    max_D = std::max(max_D, D);
  }
  if (hash_size_cumsum[T] > (int64_t)0xffffffffLL) return EMB_ERR_INVALID_ARG;

  emb_plan* p = new (std::nothrow) emb_plan;
  if (!p) return EMB_ERR_OOM;
  p->device = device;
  p->T = T;
  p->wdt = weight_dtype;
  p->gdt = grad_dtype;
  p->max_N = max_N;
  p->max_B = max_B;
  p->thr = max_segment_length_per_warp > 0 ? (uint32_t)max_segment_length_per_warp : 32u;
  p->flags = flags;
  p->max_D = max_D;
  p->uniform_D = uniform;
  const int nvec = max_D / 4;
  for (int si = 0; si < 3; ++si) {
    emb_plan::RowSplit& sp = p->split[si];
    // 16-byte vectors each lane holds of a row (rows wider than kv*32 vectors are
    // cut into chunks). Narrow rows take more than they need, so that a row spans
    // only a few lanes and a warp works on several short runs at once (the short
    // runs of skewed batches are mostly single lookups), and each lane has more
    // loads in flight. Measured on GB300: rows of 9-32 vectors run fastest at
    // kv = 4 (the large skewed workload's reduce: 8.6 ms at kv = 1, 7.4 at 2, 6.1
    // at 4; the DLRM-like one 30.9 us at 2, 29.2 at 4); kv = 8 costs too much
    // occupancy, so rows of 33-64 vectors stay at kv = 2. Wider rows: pooled
    // per-element updates cut them into chunks of 128 vectors (kv = 4; pooled SGD,
    // 4 x 200k rows, B = 4096, L = 20: D = 512 fp16 146.6 us per step at kv = 4,
    // 160.9 at kv = 8), unpooled lookups into chunks of 256 (kv = 8; the LM
    // workload's 1024-vector rows: reduce 114.7 us in chunks of 64, 110.6 in
    // chunks of 128, 101.6 in chunks of 256). Row-wise Adagrad needs the whole row
    // in one warp for its norm, so it widens kv instead.
    if (nvec <= 64) sp.kv = nvec <= 8 ? 1 : nvec <= 32 ? 4 : 2;
    else sp.kv = si == 0 ? 4 : (si == 2 || nvec > 128) ? 8 : 4;
    sp.C = (uint32_t)((nvec + sp.kv * 32 - 1) / (sp.kv * 32));
    auto shape = [&](int32_t t) {  // (chunks per row, lanes per lookup) of table t
      const int nv = (D_offsets[t + 1] - D_offsets[t]) / 4;
      const int chunks = (nv + sp.kv * 32 - 1) / (sp.kv * 32);
      const int per_lane = (std::min(nv, sp.kv * 32) + sp.kv - 1) / sp.kv;
      int lanes = 1;
      while (lanes < per_lane) lanes *= 2;
      return std::make_pair(chunks, lanes);
    };
    sp.segs.clear();
    for (int32_t t = 0; t < T; ++t)
      if (t == 0 || shape(t) != shape(t - 1)) sp.segs.push_back((uint32_t)t);
    sp.segs.push_back((uint32_t)T);
  }
  // the reduce counts (run x row chunk) tasks in 32 bits, with headroom
  if ((uint64_t)std::max<int64_t>(max_N, 1) * std::max({p->split[0].C, p->split[1].C, p->split[2].C}) >= (1ull << 31)) {
    delete p;
    return EMB_ERR_INVALID_ARG;
  }
  const uint64_t total_rows = (uint64_t)hash_size_cumsum[T];
  p->key_bits = 1;
  while (p->key_bits < 32 && ((uint64_t)1 << p->key_bits) < total_rows) ++p->key_bits;
  {  // the passes sort row indices within tables: bits of the largest table's rows
    int64_t max_rows = 1;
    for (int32_t t = 0; t < T; ++t) max_rows = std::max<int64_t>(max_rows, hash_size_cumsum[t + 1] - hash_size_cumsum[t]);
    int row_bits = 1;
    while (row_bits < 32 && ((int64_t)1 << row_bits) < max_rows) ++row_bits;
    radix_plan(row_bits, &p->passes, &p->rbits);
    p->radix = radix_buckets(p->rbits);
  }
  p->hsc.resize(T + 1);
  p->Do.assign(D_offsets, D_offsets + T + 1);
  for (int32_t t = 0; t <= T; ++t) p->hsc[t] = (uint32_t)hash_size_cumsum[t];
  for (int32_t t = 0; t < T; ++t)
    p->w_extent = std::max<int64_t>(p->w_extent, weights_offsets[t] + (hash_size_cumsum[t + 1] - hash_size_cumsum[t]) *
                                                                      (int64_t)(D_offsets[t + 1] - D_offsets[t]));

  DeviceGuard g(device);
  if (!g.ok) {
    delete p;
    return EMB_ERR_INVALID_ARG;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
    delete p;
    return EMB_ERR_CUDA;
  }
  p->props.sms = prop.multiProcessorCount;
  p->props.smem_optin = (int)prop.sharedMemPerBlockOptin;

  // Reduce kernels of this plan's types: shared-memory limit and persistent grid.
  int max_grid = 1;
  {
    cudaError_t e = cudaSuccess;
    for (int opt = 0; opt < 3 && e == cudaSuccess; ++opt) {
      for (int vk = 0; vk < 3 && e == cudaSuccess; ++vk) {
        const void* fn = reduce_fn(p, opt, vk);
        if (!fn) continue;
        const size_t sm = reduce_smem_bytes(T);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        int blocks = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kThreads, sm);
        p->reduce_grid[opt][vk] = std::max(blocks, 1) * p->props.sms;
        max_grid = std::max(max_grid, p->reduce_grid[opt][vk]);
      }
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return EMB_ERR_CUDA;
    }
  }

  // ---- scratch sizes
  const uint64_t N = (uint64_t)std::max<int64_t>(max_N, 1);
  {  // the most tiles any call up to max_N gives a pass (each tile class up to its largest N)
    uint64_t tiles = 0;
    for (int64_t n : {std::min<int64_t>((int64_t)N, (int64_t)1 << 17), std::min<int64_t>((int64_t)N, (int64_t)1 << 21),
                      (int64_t)N}) {
      const uint64_t pt = pass_tile_for(n);
      tiles = std::max<uint64_t>(tiles, ((uint64_t)n + pt - 1) / pt);
    }
    p->max_pass_tiles = (uint32_t)(tiles + (uint64_t)T + 1);
  }
  const uint64_t status_words =
      std::max<uint64_t>({(uint64_t)p->max_pass_tiles << p->rbits, (N + kRleTile - 1) / kRleTile * 4, 3 * (uint64_t)T});
  p->cap_long = (uint32_t)(N / p->thr + 1);
  // Slices (row chunk x slice) the reduce cuts the long runs into: at most
  // warps + C with one slice per warp; with more (slices of at least
  // pow2ceil(lookups per warp / 32), the last quarter of the lookups in slices 4x
  // smaller), at most 56 * warps + 5 * C, and at most C * (N / kMinSlice + 2).
  // Each has a head and a tail partial row of kv*32 vectors.
  {
    const uint64_t warps = (uint64_t)max_grid * kWarps;
    const uint64_t C = std::max({p->split[0].C, p->split[1].C, p->split[2].C});
    p->cap_slices = (uint32_t)(warps + 5 * C + std::min<uint64_t>(64 * warps, C * (N / kMinSlice + 2)));
  }
  const size_t part_row = (size_t)std::max({p->split[0].kv, p->split[1].kv, p->split[2].kv}) * 32 * sizeof(float4);
  struct Seg {
    void** ptr;
    size_t bytes;
  };
  void* tmp_ctl = nullptr;
  void* tmp_sticky = nullptr;
  Seg segs[] = {
      {&tmp_ctl, sizeof(Ctl)},
      {reinterpret_cast<void**>(&p->thist), (size_t)T * p->passes * p->radix * sizeof(uint32_t)},
      {&tmp_sticky, sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->tile_map), (size_t)p->max_pass_tiles * sizeof(PassTile)},
      {reinterpret_cast<void**>(&p->d_hsc), (T + 1) * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->d_Do), (T + 1) * sizeof(int32_t)},
      {reinterpret_cast<void**>(&p->d_wo), T * sizeof(int64_t)},
      {reinterpret_cast<void**>(&p->d_mo), T * sizeof(int64_t)},
      {reinterpret_cast<void**>(&p->keys[0]), N * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->keys[1]), N * sizeof(uint32_t)},
      {&p->vals[0], N * sizeof(uint64_t)},
      {&p->vals[1], N * sizeof(uint64_t)},
      {reinterpret_cast<void**>(&p->status), status_words * sizeof(uint64_t)},

      {reinterpret_cast<void**>(&p->run_key), N * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->run_start), (N + 1) * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->seg_runs), (T + 1) * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->split[0].d_segkeys), p->split[0].segs.size() * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->split[1].d_segkeys), p->split[1].segs.size() * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->split[0].d_segs), p->split[0].segs.size() * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->split[1].d_segs), p->split[1].segs.size() * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->split[2].d_segkeys), p->split[2].segs.size() * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->split[2].d_segs), p->split[2].segs.size() * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->long_ids), p->cap_long * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->longs), p->cap_long * sizeof(LongRun)},
      {reinterpret_cast<void**>(&p->partials), 2 * (size_t)p->cap_slices * part_row},
      {reinterpret_cast<void**>(&p->done), 4 * (size_t)p->cap_slices * sizeof(uint32_t)},
      {reinterpret_cast<void**>(&p->rw_ss), p->split[1].C > 1 ? N * p->split[1].C * sizeof(float) : 0},
      {reinterpret_cast<void**>(&p->rw_cnt), p->split[1].C > 1 ? N * sizeof(uint32_t) : 0},
      {reinterpret_cast<void**>(&p->rw_m), p->split[1].C > 1 ? N * sizeof(float) : 0},
  };
  size_t total = 0;
  for (const Seg& sg : segs) total = align_up(total, 256) + sg.bytes;
  if (cudaMalloc(&p->arena, total) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return EMB_ERR_OOM;
  }
  size_t off = 0;
  for (const Seg& sg : segs) {
    off = align_up(off, 256);
    *sg.ptr = static_cast<char*>(p->arena) + off;
    off += sg.bytes;
  }
  p->ctl = static_cast<Ctl*>(tmp_ctl);
  p->sticky = static_cast<uint32_t*>(tmp_sticky);
  p->clear_bytes = (size_t)(reinterpret_cast<char*>(p->thist) - reinterpret_cast<char*>(p->ctl)) +
                   (size_t)T * p->passes * p->radix * sizeof(uint32_t);

  std::vector<int64_t> mo(T);
  for (int32_t t = 0; t < T; ++t) mo[t] = momentum_offsets ? momentum_offsets[t] : hash_size_cumsum[t];
  cudaError_t e = cudaMemset(p->arena, 0, total);
  if (e == cudaSuccess) e = cudaMemcpy(p->d_hsc, p->hsc.data(), (T + 1) * sizeof(uint32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p->d_Do, D_offsets, (T + 1) * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p->d_wo, weights_offsets, T * sizeof(int64_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p->d_mo, mo.data(), T * sizeof(int64_t), cudaMemcpyHostToDevice);
  for (const emb_plan::RowSplit& sp : p->split) {
    std::vector<uint32_t> keys;
    for (uint32_t t : sp.segs) keys.push_back(p->hsc[t]);
    if (e == cudaSuccess)
      e = cudaMemcpy(sp.d_segs, sp.segs.data(), sp.segs.size() * sizeof(uint32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(sp.d_segkeys, keys.data(), keys.size() * sizeof(uint32_t), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = sort_configure(p->props);
  if (e == cudaSuccess) e = runs_configure();
  if (e == cudaSuccess) e = cfront_configure(p->props.smem_optin);
  if (e == cudaSuccess && !(flags & EMB_FLAG_NO_CLUSTER_FRONT)) {
    p->cf_max_N = std::min<int64_t>(max_N, kCfMaxN);
    for (int vk = 0; vk < 3; ++vk)
      for (int i = 0; i < 4; ++i) {
        // shared memory of the largest eligible call (mean pooling's bag lengths
        // included where they fit; a call that needs more takes the other front)
        const uint32_t cap = (uint32_t)((std::max<int64_t>(p->cf_max_N, 1) + kCfSizes[i] - 1) / kCfSizes[i]);
        size_t sm = cfront_smem(vk, p->radix, true, cap);
        if (sm > (size_t)p->props.smem_optin) sm = cfront_smem(vk, p->radix, false, cap);
        if (sm <= (size_t)p->props.smem_optin)
          p->cf_clusters[vk][i] = cfront_max_clusters(vk, p->radix, kCfSizes[i], sm);
      }
  }
  if (e == cudaSuccess) {
    const int tiles[3] = {kThreads * 4, kThreads * 8, kThreads * 16};
    for (int c = 0; c < 3; ++c)
      for (int wide = 0; wide < 2; ++wide)
        p->pass_cap[c][wide] = sort_pass_capacity(wide != 0, tiles[c], p->rbits, p->props.sms);
    for (int si = 0; si < 3; ++si)
      for (int it = 0; it < 2; ++it)
        p->runs_cap[si][it] = runs_capacity((int)p->split[si].segs.size() - 1, it ? 16 : 8, p->props.sms);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p->arena);
    delete p;
    return EMB_ERR_CUDA;
  }
  *out = p;
  return EMB_OK;
}

emb_status emb_plan_destroy(emb_plan* p) {
  if (!p) return EMB_OK;
  DeviceGuard g(p->device);
  cudaDeviceSynchronize();
  if (p->events_ready)
    for (cudaEvent_t ev : p->ev) cudaEventDestroy(ev);
  const cudaError_t e = cudaFree(p->arena);
  delete p;
  return e == cudaSuccess ? EMB_OK : EMB_ERR_CUDA;
}

emb_status emb_bag_bwd_sgd(emb_plan* p, void* weights, const int64_t* indices,
                           const int64_t* offsets, int64_t N, int32_t B,
                           const float* per_sample_weights, const void* grad_output,
                           emb_pooling mode, float lr, void* stream) {
  NvtxRange nvtx("emb_bag_bwd_sgd");
  EMB_TRY(check_common(p, weights, indices, offsets, N, B, grad_output));
  if (mode != EMB_POOL_SUM && mode != EMB_POOL_MEAN) return EMB_ERR_INVALID_ARG;
  if (per_sample_weights && !aligned(per_sample_weights, 4)) return EMB_ERR_INVALID_ARG;
  if (N == 0) {
    p->last_kind = 0;
    return EMB_OK;
  }
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  const int vk = (per_sample_weights || mode == EMB_POOL_MEAN) ? VK_BAG_SCALED : VK_BAG;
  return run_sorted(p, 0, vk, weights, nullptr, indices, offsets, N, B, per_sample_weights,
                    grad_output, mode == EMB_POOL_MEAN, lr, 0.0f, nullptr, 0,
                    static_cast<cudaStream_t>(stream));
}

emb_status emb_bag_bwd_rowwise_adagrad(emb_plan* p, void* weights, float* momentum,
                                       const int64_t* indices, const int64_t* offsets,
                                       int64_t N, int32_t B, const float* per_sample_weights,
                                       const void* grad_output, emb_pooling mode, float lr,
                                       float eps, void* stream) {
  NvtxRange nvtx("emb_bag_bwd_rowwise_adagrad");
  EMB_TRY(check_common(p, weights, indices, offsets, N, B, grad_output));
  if (mode != EMB_POOL_SUM && mode != EMB_POOL_MEAN) return EMB_ERR_INVALID_ARG;
  if (per_sample_weights && !aligned(per_sample_weights, 4)) return EMB_ERR_INVALID_ARG;
  if (N == 0) {
    p->last_kind = 0;
    return EMB_OK;
  }
  if (!momentum || !aligned(momentum, 4)) return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  const int vk = (per_sample_weights || mode == EMB_POOL_MEAN) ? VK_BAG_SCALED : VK_BAG;
  return run_sorted(p, 1, vk, weights, momentum, indices, offsets, N, B, per_sample_weights,
                    grad_output, mode == EMB_POOL_MEAN, lr, eps, nullptr, 0,
                    static_cast<cudaStream_t>(stream));
}

emb_status emb_bag_bwd_adagrad(emb_plan* p, void* weights, float* momentum, const int64_t* indices,
                               const int64_t* offsets, int64_t N, int32_t B,
                               const float* per_sample_weights, const void* grad_output,
                               emb_pooling mode, float lr, float eps, void* stream) {
  NvtxRange nvtx("emb_bag_bwd_adagrad");
  EMB_TRY(check_common(p, weights, indices, offsets, N, B, grad_output));
  if (mode != EMB_POOL_SUM && mode != EMB_POOL_MEAN) return EMB_ERR_INVALID_ARG;
  if (per_sample_weights && !aligned(per_sample_weights, 4)) return EMB_ERR_INVALID_ARG;
  if (N == 0) {
    p->last_kind = 0;
    return EMB_OK;
  }
  if (!momentum || !aligned(momentum, 16)) return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  const int vk = (per_sample_weights || mode == EMB_POOL_MEAN) ? VK_BAG_SCALED : VK_BAG;
  return run_sorted(p, 2, vk, weights, momentum, indices, offsets, N, B, per_sample_weights,
                    grad_output, mode == EMB_POOL_MEAN, lr, eps, nullptr, 0,
                    static_cast<cudaStream_t>(stream));
}

// Dense-gradient mode for pooled (vk from the pooling) or unpooled lookups.
static emb_status dense_grad(emb_plan* p, void* grad_weights, const int64_t* indices,
                      const int64_t* offsets, int64_t N, int32_t B, const float* psw,
                      const void* grad_output, int vk, int mean, void* stream) {
  if (!p || !grad_weights || !aligned(grad_weights, 4 * dtype_size(p->wdt))) return EMB_ERR_INVALID_ARG;
  EMB_TRY(check_common(p, grad_weights, indices, offsets, N, B, grad_output));
  if (psw && !aligned(psw, 4)) return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EMB_CUDA(cudaMemsetAsync(grad_weights, 0, (size_t)p->w_extent * dtype_size(p->wdt), s));
  if (N == 0) {
    p->last_kind = 0;
    p->last_stream = s;
    return EMB_OK;
  }
  return run_sorted(p, 0, vk, grad_weights, nullptr, indices, offsets, N, B, psw, grad_output, mean,
                    0.0f, 0.0f, grad_weights, 1, s);
}

emb_status emb_bag_bwd_dense_grad(emb_plan* p, void* grad_weights, const int64_t* indices,
                                  const int64_t* offsets, int64_t N, int32_t B,
                                  const float* per_sample_weights, const void* grad_output,
                                  emb_pooling mode, void* stream) {
  NvtxRange nvtx("emb_bag_bwd_dense_grad");
  if (mode != EMB_POOL_SUM && mode != EMB_POOL_MEAN) return EMB_ERR_INVALID_ARG;
  const int vk = (per_sample_weights || mode == EMB_POOL_MEAN) ? VK_BAG_SCALED : VK_BAG;
  return dense_grad(p, grad_weights, indices, offsets, N, B, per_sample_weights, grad_output, vk,
                    mode == EMB_POOL_MEAN, stream);
}

emb_status emb_nobag_bwd_dense_grad(emb_plan* p, void* grad_weights, const int64_t* indices,
                                    const int64_t* offsets, int64_t N, int32_t B,
                                    const void* grad_output, void* stream) {
  NvtxRange nvtx("emb_nobag_bwd_dense_grad");
  if (p && !p->uniform_D) return EMB_ERR_INVALID_ARG;
  return dense_grad(p, grad_weights, indices, offsets, N, B, nullptr, grad_output, VK_NOBAG, 0, stream);
}

emb_status emb_bag_fwd(emb_plan* p, const void* weights, const int64_t* indices,
                       const int64_t* offsets, int64_t N, int32_t B,
                       const float* per_sample_weights, emb_pooling mode, void* output,
                       emb_dtype output_dtype, void* stream) {
  NvtxRange nvtx("emb_bag_fwd");
  if (!p) return EMB_ERR_INVALID_ARG;
  if (N < 0 || N > p->max_N || B <= 0 || B > p->max_B) return EMB_ERR_INVALID_ARG;
  if (mode != EMB_POOL_SUM && mode != EMB_POOL_MEAN) return EMB_ERR_INVALID_ARG;
  if (output_dtype != EMB_F32 && output_dtype != EMB_F16 && output_dtype != EMB_BF16)
    return EMB_ERR_INVALID_ARG;
  if (!weights || !offsets || !output || (N > 0 && !indices)) return EMB_ERR_INVALID_ARG;
  if (!aligned(weights, 4 * dtype_size(p->wdt)) || !aligned(output, 4 * dtype_size(output_dtype)) ||
      !aligned(offsets, 8) || (indices && !aligned(indices, 8)) ||
      (per_sample_weights && !aligned(per_sample_weights, 4)))
    return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  const emb_plan::RowSplit& sp = p->split[0];
  const void* fn = fwd_kernel(static_cast<int>(p->wdt), static_cast<int>(output_dtype), sp.kv);
  if (!fn) return EMB_ERR_UNSUPPORTED;
  const uint32_t S = (uint32_t)sp.segs.size() - 1;
  const size_t sm = fwd_smem_bytes(p->T, (int)S);
  int& grid = p->fwd_grid[output_dtype];
  if (grid == 0) {  // first forward call with this output type: persistent grid
    int blocks = 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kThreads, sm) != cudaSuccess) {
      cudaGetLastError();
      return EMB_ERR_CUDA;
    }
    grid = std::max(blocks, 1) * p->props.sms;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FwdArgs a;
  a.weights = weights;
  a.indices = indices;
  a.offsets = offsets;
  a.psw = per_sample_weights;
  a.out = output;
  a.sticky = p->sticky;
  a.hsc = p->d_hsc;
  a.D_offsets = p->d_Do;
  a.weights_offsets = p->d_wo;
  a.segs = sp.d_segs;
  a.S = S;
  a.T = (uint32_t)p->T;
  a.B = (uint32_t)B;
  a.N = N;
  a.out_stride = p->Do[p->T];
  a.mean = mode == EMB_POOL_MEAN;
  void* args[] = {&a};
  EMB_CUDA(launch_kernel(fn, dim3(grid), dim3(kThreads), sm, s, args, !(p->flags & EMB_FLAG_NO_PDL)));
  p->last_stream = s;  // emb_plan_status waits for it
  return EMB_OK;
}

emb_status emb_nobag_bwd_sgd(emb_plan* p, void* weights, const int64_t* indices,
                             const int64_t* offsets, int64_t N, int32_t B,
                             const void* grad_output, float lr, emb_nobag_path path,
                             void* stream) {
  NvtxRange nvtx("emb_nobag_bwd_sgd");
  EMB_TRY(check_common(p, weights, indices, offsets, N, B, grad_output));
  if (!p->uniform_D) return EMB_ERR_INVALID_ARG;
  if (path < EMB_NOBAG_AUTO || path > EMB_NOBAG_ATOMIC) return EMB_ERR_INVALID_ARG;
  if (path == EMB_NOBAG_ATOMIC && p->wdt != EMB_F32) return EMB_ERR_UNSUPPORTED;
  if (N == 0) {
    p->last_kind = 0;
    return EMB_OK;
  }
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == EMB_NOBAG_ATOMIC) {
    const bool pdl = !(p->flags & EMB_FLAG_NO_PDL);
    const DecodeArgs d = decode_args(p, indices, offsets, nullptr, N, B, 0);
    EMB_TRY(record(p, 0, s));
    EMB_CUDA(cudaMemsetAsync(p->ctl, 0, sizeof(Ctl), s));
    HistArgs ha{d, p->ctl, p->sticky, 0, (int)sort_tile_for(N), nullptr, nullptr};
    EMB_CUDA(launch_hist(ha, -1, p->T, s, pdl));
    EMB_TRY(record(p, 1, s));
    AtomicArgs aa{d, p->ctl, p->sticky, grad_output, static_cast<float*>(weights), p->d_wo,
                  (uint32_t)p->max_D, lr};
    EMB_CUDA(launch_nobag_atomic(aa, (int)p->gdt, p->T, s, pdl));
    EMB_TRY(record(p, 5, s));
    p->last_kind = 2;
    p->last_N = N;
    p->last_stream = s;
    if (p->profiling) p->last_profiled = 2;
    return EMB_OK;
  }
  return run_sorted(p, 0, VK_NOBAG, weights, nullptr, indices, offsets, N, B, nullptr,
                    grad_output, 0, lr, 0.0f, nullptr, 0, s);
}

emb_status emb_plan_set_rounding(emb_plan* p, uint64_t seed, uint64_t next_call) {
  if (!p) return EMB_ERR_INVALID_ARG;
  p->sr_seed = seed;
  p->sr_call = next_call;
  return EMB_OK;
}

emb_status emb_plan_get_rounding(const emb_plan* p, uint64_t* seed, uint64_t* next_call) {
  if (!p) return EMB_ERR_INVALID_ARG;
  if (seed) *seed = p->sr_seed;
  if (next_call) *next_call = p->sr_call;
  return EMB_OK;
}

emb_status emb_plan_status(emb_plan* p) {
  if (!p) return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return EMB_ERR_CUDA;
  if (cudaStreamSynchronize(p->last_stream) != cudaSuccess) {
    cudaGetLastError();
    return EMB_ERR_CUDA;
  }
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, p->sticky, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(p->sticky, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    return EMB_ERR_CUDA;
  }
  if (bits & kErrOffsets) return EMB_ERR_INVALID_ARG;  // bag ids (and so tables) are meaningless
  if (bits & kErrIndex) return EMB_ERR_INDEX_OUT_OF_RANGE;
  if (bits & kErrTimeout) return EMB_ERR_TIMEOUT;
  if (bits & kErrCapacity) return EMB_ERR_OOM;
  return EMB_OK;
}

emb_status emb_plan_debug_runs(emb_plan* p, int64_t capacity, int64_t* run_keys, int32_t* run_len,
                               int32_t* cum, int32_t* num_runs, int32_t* long_ids,
                               int32_t* num_long) {
  if (!p || capacity < 0) return EMB_ERR_INVALID_ARG;
  if (p->last_kind == 0) {
    if (num_runs) *num_runs = 0;
    if (num_long) *num_long = 0;
    if (cum && capacity >= 0) cum[0] = 0;
    return EMB_OK;
  }
  if (p->last_kind != 1) return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok || cudaStreamSynchronize(p->last_stream) != cudaSuccess) return EMB_ERR_CUDA;
  Ctl c;
  if (cudaMemcpy(&c, p->ctl, sizeof(Ctl), cudaMemcpyDeviceToHost) != cudaSuccess) return EMB_ERR_CUDA;
  if ((int64_t)c.num_runs > capacity || (int64_t)c.num_long > capacity) return EMB_ERR_INVALID_ARG;
  const uint32_t U = c.num_runs;
  std::vector<uint32_t> keys(U), starts(U + 1), lids(c.num_long);
  if (cudaMemcpy(keys.data(), p->run_key, U * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(starts.data(), p->run_start, (U + 1) * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(lids.data(), p->long_ids, c.num_long * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return EMB_ERR_CUDA;
  for (uint32_t r = 0; r < U; ++r) {
    if (run_keys) run_keys[r] = keys[r];
    if (run_len) run_len[r] = (int32_t)(starts[r + 1] - starts[r]);
    if (cum) cum[r] = (int32_t)starts[r];
  }
  if (cum) cum[U] = (int32_t)starts[U];
  if (long_ids)
    for (uint32_t k = 0; k < c.num_long; ++k) long_ids[k] = (int32_t)lids[k];
  if (num_runs) *num_runs = (int32_t)U;
  if (num_long) *num_long = (int32_t)c.num_long;
  return EMB_OK;
}

emb_status emb_plan_set_profiling(emb_plan* p, int enable) {
  if (!p) return EMB_ERR_INVALID_ARG;
  if (enable && !p->events_ready) {
    DeviceGuard g(p->device);
    for (cudaEvent_t& ev : p->ev)
      if (cudaEventCreate(&ev) != cudaSuccess) return EMB_ERR_CUDA;
    p->events_ready = true;
  }
  p->profiling = enable != 0;
  return EMB_OK;
}

emb_status emb_plan_stage_ms(emb_plan* p, float* ms, int32_t n) {
  if (!p || !ms || n < 0) return EMB_ERR_INVALID_ARG;
  if (!p->events_ready || p->last_profiled == 0) return EMB_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (cudaEventSynchronize(p->ev[kStages]) != cudaSuccess) return EMB_ERR_CUDA;
  // stage i runs from event from[i] to event to[i] (-1: stage not separate)
  static const int kFromSorted[kStages] = {0, 1, 2, -1, 3}, kToSorted[kStages] = {1, 2, 3, -1, 5};
  static const int kFromAtomic[kStages] = {0, -1, -1, -1, 1}, kToAtomic[kStages] = {1, -1, -1, -1, 5};
  const int* from = p->last_profiled == 1 ? kFromSorted : kFromAtomic;
  const int* to = p->last_profiled == 1 ? kToSorted : kToAtomic;
  for (int i = 0; i < kStages && i < n; ++i) {
    float v = 0.f;
    if (from[i] >= 0 && cudaEventElapsedTime(&v, p->ev[from[i]], p->ev[to[i]]) != cudaSuccess)
      return EMB_ERR_CUDA;
    ms[i] = v;
  }
  return EMB_OK;
}

}  // extern "C"
