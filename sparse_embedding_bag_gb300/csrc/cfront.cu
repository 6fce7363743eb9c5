// Small-batch front of the sorted path: one thread-block cluster per table
// linearises, radix-sorts and run-length encodes that table's segment of the
// lookups, all in one launch.
//
// It computes what k_hist, k_sort_pass and k_runs compute (the transpose/sort
// step, the run-length encode and *_find_long_segments of the host function in
// "fbgemm_gpu/codegen/embedding_backward_split_template.cu"), with the same
// outputs bit for bit: the stable sort of each table's segment on its row
// index, the unique keys with their run starts, the number of runs, and the
// ordered compaction of the long runs with the prefix sum of their lengths.
// What changes is where the work waits. On a small batch the multi-block front
// is a chain of dependent global round trips: four launches, each with its
// decoupled look-back. Here:
//   * the lookups of table t form one contiguous segment (the offsets are
//     table-major), so the table needs nothing from other tables but the
//     number of runs before it;
//   * the segment is split evenly over the CTAs of one cluster; each CTA keeps
//     its slice in shared memory, ranks it per warp (match-based multisplit),
//     and the per-digit counts of all CTAs are exchanged through distributed
//     shared memory between two hardware cluster barriers, in place of the
//     global histogram and the look-back;
//   * elements move between passes through global memory (L2): each pass
//     scatters its slice to the final positions of the pass and, after the
//     cluster barrier, every CTA reloads its slice of the result;
//   * the run counts before the table come from a decoupled look-back over the
//     tables (one status word per table and count, 32 tables per poll).
// Shared memory holds ceil(N / CTAs per cluster) lookups per CTA, which bounds
// the batches this front can take (the host checks it, and takes the front only
// up to 2^16 lookups, where it measured faster); each table is at most the whole
// batch, so every slice fits.
#include <cooperative_groups.h>

#include "decode.cuh"

namespace embbwd {

namespace {

namespace cg = cooperative_groups;

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxCluster = 16;  // CTAs of a cluster (the non-portable limit)
// s_misc words: [0, 16) block-scan scratch; run counts of this CTA (read by the
// cluster); counts of the cluster's CTAs before this one; cluster totals; the
// look-back result (counts of the tables before this one).
constexpr int kMiscMine = 16, kMiscBelow = 20, kMiscTotal = 24, kMiscTable = 28, kMiscWords = 32;

// Byte offsets of the dynamic shared memory of one CTA (cap lookups).
struct CfLayout {
  size_t whist, cnt, gbase, misc, val, key, aux, len, total;
};

__host__ __device__ inline size_t cf_align(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline CfLayout cf_layout(int radix, size_t vbytes, bool mean, uint32_t cap) {
  CfLayout L;
  size_t o = 0;
  L.whist = o;  // [kWarps][radix] per-warp digit counts; the bag offsets staging before the first pass
  o = cf_align(o + (size_t)kWarps * radix * 4);
  L.cnt = o;    // [radix] this CTA's digit counts (read by the cluster)
  o = cf_align(o + (size_t)radix * 4);
  L.gbase = o;  // [radix] first output position of each digit of this CTA
  o = cf_align(o + (size_t)radix * 4);
  L.misc = o;
  o = cf_align(o + kMiscWords * 4);
  L.val = o;    // [cap] payloads of the slice
  o = cf_align(o + (size_t)cap * vbytes);
  L.key = o;    // [cap] keys of the slice
  o = cf_align(o + (size_t)cap * 4);
  L.aux = o;    // [cap + 1] bag ids, then ranks, then run-head positions
  o = cf_align(o + ((size_t)cap + 1) * 4);
  L.len = o;    // [cap] bag lengths (mean pooling only)
  o = cf_align(o + (mean ? (size_t)cap * 4 : 0));
  L.total = o;
  return L;
}

// First position in [b, end) whose key differs from k (or end), given that
// position b-1 holds k: an exponential probe, then a 32-way search. Called by
// all lanes of one warp; reads through L2 (the keys were written by other CTAs
// of the cluster in this launch).
__device__ __forceinline__ uint32_t run_end_in(const uint32_t* keys, uint32_t end, uint32_t b, uint32_t k) {
  const uint32_t lane = threadIdx.x & 31;
  if (b >= end) return end;
  const uint64_t q = (uint64_t)b - 1 + ((uint64_t)1 << lane);
  const bool in = lane < 31 && q < end && __ldcg(keys + q) == k;
  const uint32_t m = __popc(__ballot_sync(kFull, in));  // lanes 0..m-1 are inside the run
  if (m == 0) return b;
  uint64_t lo = (uint64_t)b + ((uint64_t)1 << (m - 1));
  const uint64_t cap = (uint64_t)b - 1 + ((uint64_t)1 << m);
  uint64_t hi = cap < (uint64_t)end ? cap : (uint64_t)end;
  while (hi > lo) {  // positions < lo are inside, position hi is outside (or end)
    const uint64_t step = (hi - lo + 31) / 32;
    const uint64_t p = lo + lane * step;
    const bool inside = p < hi && __ldcg(keys + p) == k;
    const uint32_t c = __popc(__ballot_sync(kFull, inside));
    if (c == 0) break;
    const uint64_t nlo = lo + (uint64_t)(c - 1) * step + 1;
    const uint64_t nhi = lo + (uint64_t)c * step;
    hi = nhi < hi ? nhi : hi;
    lo = nlo;
  }
  return (uint32_t)lo;
}

// Runs (channel 0), long runs (1) and their lookups (2) of the tables before
// table t: a warp-wide decoupled look-back over per-table status words, 32
// tables per poll. publish: this warp also writes table t's aggregate before
// the walk and its inclusive count after it (one CTA of the cluster does).
// Every wait is bounded; on expiry kErrTimeout is raised and the walk stops.
// Table 0 has nothing before it.
__device__ __forceinline__ uint32_t table_lookback(const LookbackCfg& lb, uint32_t t, uint32_t ch, uint32_t agg,
                                                   bool publish, Ctl* ctl, uint32_t* sticky) {
  const uint32_t lane = threadIdx.x & 31;
  uint64_t* st = lb.status + (size_t)t * 3 + ch;
  const uint64_t tag = (uint64_t)lb.epoch << 32;
  if (publish && lane == 0) st_relaxed_u64(st, tag | (t == 0 ? kFlagInc : kFlagAgg) | (agg & kCountMask));
  uint32_t excl = 0;
  bool failed = lb.force_timeout != 0;  // test flag: give up at once (table 0 included)
  int64_t j = (int64_t)t - 1;
  uint32_t polls = 0;
  while (!failed && j >= 0) {
    const int64_t idx = j - (int64_t)lane;
    const uint64_t w = idx >= 0 ? ld_relaxed_u64(lb.status + (size_t)idx * 3 + ch) : (tag | kFlagInc);
    const bool ready = (uint32_t)(w >> 32) == lb.epoch && (w & (kFlagAgg | kFlagInc));
    const uint32_t nr = __ballot_sync(kFull, !ready);
    const uint32_t inc = __ballot_sync(kFull, ready && (w & kFlagInc));
    const uint32_t stop_nr = nr ? __ffs(nr) - 1 : 32u;
    const uint32_t stop_inc = inc ? __ffs(inc) - 1 : 32u;
    const bool found = stop_inc < stop_nr;
    const uint32_t take = found ? stop_inc + 1 : stop_nr;  // lanes [0, take) are summed
    uint32_t v = lane < take ? ((uint32_t)w & kCountMask) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    excl += v;
    if (found) break;
    j -= take;
    if (take < 32) {
      if (++polls > lb.spin_limit) failed = true;
      else if (polls > 8) __nanosleep(polls > 128 ? 256 : 32);
    }
  }
  if (failed && lane == 0) raise_error(ctl, sticky, kErrTimeout);
  if (publish && lane == 0) st_relaxed_u64(st, tag | kFlagInc | ((excl + agg) & kCountMask));
  return excl;
}

// Lookups whose indices (and per-sample weights) a thread loads before the bag
// expansion, so that their latency overlaps it.
constexpr int kPre = 8;
// Steps of 32 slice positions a warp ranks or scatters side by side.
constexpr int kGrp = 8;

// The cluster barrier in two halves: arrive (no memory ordering) and wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

template <int VK, int RADIX>
__global__ void __launch_bounds__(kThreads) k_cfront(CfrontArgs a) {
  using V = typename std::conditional<VK == VK_BAG_SCALED, uint64_t, uint32_t>::type;
  constexpr int DPT = RADIX > kThreads ? RADIX / kThreads : 1;  // digits per thread
  extern __shared__ __align__(16) unsigned char smem[];
  const DecodeArgs& d = a.d;
  const bool mean = VK == VK_BAG_SCALED && d.mean;
  const CfLayout L = cf_layout(RADIX, sizeof(V), mean, a.cap);
  uint32_t* s_whist = reinterpret_cast<uint32_t*>(smem + L.whist);
  uint32_t* s_cnt = reinterpret_cast<uint32_t*>(smem + L.cnt);
  uint32_t* s_gbase = reinterpret_cast<uint32_t*>(smem + L.gbase);
  uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + L.misc);
  V* s_val = reinterpret_cast<V*>(smem + L.val);
  uint32_t* s_key = reinterpret_cast<uint32_t*>(smem + L.key);
  uint32_t* s_aux = reinterpret_cast<uint32_t*>(smem + L.aux);
  uint32_t* s_len = mean ? reinterpret_cast<uint32_t*>(smem + L.len) : nullptr;

  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t CL = cluster.num_blocks();
  const uint32_t crank = cluster.block_rank();
  const uint32_t G = gridDim.x / CL;  // clusters of the grid
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  const uint32_t N = (uint32_t)d.N;
  const uint32_t dmask = (1u << a.rbits) - 1u;
  pdl_wait();
  pdl_trigger();

  // Tables in look-back order: every cluster of the grid is resident at once
  // (the host sizes the grid so), and table t only waits on tables before it.
  for (uint32_t t = blockIdx.x / CL; t < d.T; t += G) {
    const uint32_t kbase = d.hsc[t];
    const uint32_t rows = d.hsc[t + 1] - kbase;
    const int64_t* toff = d.offsets + (size_t)t * d.B;  // the table's B+1 bag offsets
    const int64_t o0 = toff[0], o1 = toff[d.B];
    // the segment, clamped into [0, N] (malformed offsets are reported, never followed out of bounds)
    const uint32_t s0 = (uint32_t)(o0 < 0 ? 0 : (o0 > (int64_t)N ? (int64_t)N : o0));
    const uint32_t s1 = (uint32_t)(o1 < (int64_t)s0 ? (int64_t)s0 : (o1 > (int64_t)N ? (int64_t)N : o1));
    const uint32_t nseg = s1 - s0;
    const uint32_t per = (nseg + CL - 1) / CL;
    const uint32_t i0 = min(crank * per, nseg);
    uint32_t n = min(i0 + per, nseg) - i0;  // lookups of this CTA's slice
    if (n > a.cap) {  // only with a capacity the host did not size: never for a valid call
      if (threadIdx.x == 0) raise_error(a.ctl, a.sticky, kErrCapacity);
      n = a.cap;
    }
    const uint32_t g0 = s0 + i0;  // first lookup of the slice

    if (crank == 0 && threadIdx.x == 0) {
      if ((t == 0 && o0 != 0) || (t == d.T - 1 && o1 != d.N)) raise_error(a.ctl, a.sticky, kErrOffsets);
    }

    // ---- linearise the slice: key = hash_size_cumsum[t] + idx, payload
    int64_t pre_idx[kPre];
    float pre_psw[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const uint32_t j = threadIdx.x + k * kThreads;
      pre_idx[k] = j < n ? d.indices[g0 + j] : 0;
      if constexpr (VK == VK_BAG_SCALED) pre_psw[k] = (j < n && d.psw) ? d.psw[g0 + j] : 1.0f;
    }
    // Bag of every lookup of the slice, relative to the table's first bag, and
    // the CSR validation of this CTA's share of the table's bags. When the
    // table's B+1 offsets fit in the payload buffer (free until the payloads are
    // written), they are staged there with one load and searched in shared
    // memory; otherwise the bags overlapping the slice are found in global memory.
    if constexpr (VK != VK_NOBAG) {
      const uint32_t B = d.B;
      if ((size_t)(B + 1) * sizeof(uint32_t) <= (size_t)a.cap * sizeof(V)) {
        // as 32-bit positions clamped into [0, N]; this CTA's share of the bags
        // is checked on the values as given
        uint32_t* s_toff = reinterpret_cast<uint32_t*>(s_val);
        const uint32_t kc0 = min(crank * ((B + CL - 1) / CL), B), kc1 = min(kc0 + (B + CL - 1) / CL, B);
#pragma unroll 4
        for (uint32_t k = threadIdx.x; k <= B; k += kThreads) {
          const int64_t o = toff[k];
          if (k > kc0 && k <= kc1 && o < toff[k - 1]) raise_error(a.ctl, a.sticky, kErrOffsets);
          s_toff[k] = (uint32_t)(o < 0 ? 0 : (o > (int64_t)N ? (int64_t)N : o));
        }
        __syncthreads();
        // bag of lookup x: the last j in [0, B-1] with offsets[j] <= x, by a
        // binary search of fixed steps, kPre lookups of a thread side by side
        const uint32_t top = 1u << (31 - __clz(B));
        auto put_bag = [&](uint32_t j, uint32_t bt) {
          s_aux[j] = bt;
          if (mean) s_len[j] = s_toff[bt + 1] - s_toff[bt];
        };
        uint32_t lo[kPre];
#pragma unroll
        for (int k = 0; k < kPre; ++k) lo[k] = 0;
        for (uint32_t st = top; st > 0; st >>= 1) {
#pragma unroll
          for (int k = 0; k < kPre; ++k) {
            const uint32_t c = lo[k] + st;
            if (c < B && s_toff[c] <= g0 + threadIdx.x + k * kThreads) lo[k] = c;
          }
        }
#pragma unroll
        for (int k = 0; k < kPre; ++k)
          if (threadIdx.x + k * kThreads < n) put_bag(threadIdx.x + k * kThreads, lo[k]);
        for (uint32_t j = threadIdx.x + kPre * kThreads; j < n; j += kThreads) {
          uint32_t l = 0;
          for (uint32_t st = top; st > 0; st >>= 1)
            if (l + st < B && s_toff[l + st] <= g0 + j) l += st;
          put_bag(j, l);
        }
        __syncthreads();  // the offsets are read before the payloads overwrite them
      } else {
        for (uint32_t k = crank * kThreads + threadIdx.x; k < B; k += CL * kThreads)
          if (toff[k + 1] < toff[k]) raise_error(a.ctl, a.sticky, kErrOffsets);
        if (n > 0) {  // block-uniform branch
          DecodeArgs dt = d;
          dt.offsets = toff;
          dt.BT = B;
          expand_tile_bags(dt, g0, g0 + n, s_aux, s_len, reinterpret_cast<int64_t*>(s_whist), kWarps * RADIX / 2);
        }
      }
    } else {
      for (uint32_t k = crank * kThreads + threadIdx.x; k < d.B; k += CL * kThreads)
        if (toff[k + 1] < toff[k]) raise_error(a.ctl, a.sticky, kErrOffsets);
    }
    bool any_bad = false;
    auto put = [&](uint32_t j, int64_t idx, float psw) {
      any_bad |= idx < 0 || idx >= (int64_t)rows;
      s_key[j] = kbase + (uint32_t)idx;
      if constexpr (VK == VK_BAG) {
        s_val[j] = t * d.B + s_aux[j];
      } else if constexpr (VK == VK_NOBAG) {
        s_val[j] = g0 + j;
      } else {
        float s = psw;
        if (mean) s = __fdiv_rn(s, (float)s_len[j]);
        s_val[j] = (uint64_t)(t * d.B + s_aux[j]) | ((uint64_t)__float_as_uint(s) << 32);
      }
    };
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const uint32_t j = threadIdx.x + k * kThreads;
      if (j < n) put(j, pre_idx[k], VK == VK_BAG_SCALED ? pre_psw[k] : 1.0f);
    }
    for (uint32_t j = threadIdx.x + kPre * kThreads; j < n; j += kThreads)
      put(j, d.indices[g0 + j], (VK == VK_BAG_SCALED && d.psw) ? d.psw[g0 + j] : 1.0f);
    if (__syncthreads_or(any_bad) && threadIdx.x == 0) raise_error(a.ctl, a.sticky, kErrIndex);

    // ---- radix passes over the row index; warp w ranks slice positions [jb, je)
    const uint32_t Sw = (n + kWarps - 1) / kWarps;
    const uint32_t jb = min(warp * Sw, n), je = min(jb + Sw, n);
    for (int p = 0; p < a.passes; ++p) {
      if (p > 0) {  // this CTA's slice of the previous pass's output
        const uint32_t* kin = a.keys[(p + 1) & 1];
        const V* vin = reinterpret_cast<const V*>(a.vals[(p + 1) & 1]);
#pragma unroll 8
        for (uint32_t j = threadIdx.x; j < n; j += kThreads) {
          s_key[j] = __ldcg(kin + g0 + j);
          s_val[j] = __ldcg(vin + g0 + j);
        }
      }
      for (uint32_t i = threadIdx.x; i < (uint32_t)(kWarps * RADIX); i += kThreads) s_whist[i] = 0;
      __syncthreads();
      const uint32_t shift = (uint32_t)p * (uint32_t)a.rbits;
      uint32_t* wh = s_whist + warp * RADIX;
      // stable: positions in order within the warp's range, kGrp steps of 32 at a
      // time (their keys and peer masks are found before the counts are updated)
      for (uint32_t j0 = jb; j0 < je; j0 += 32 * kGrp) {
        uint32_t dg[kGrp], peers[kGrp];
#pragma unroll
        for (int u = 0; u < kGrp; ++u) {
          const uint32_t j = j0 + u * 32 + lane;
          dg[u] = j < je ? ((s_key[j] - kbase) >> shift) & dmask : (uint32_t)RADIX;
        }
#pragma unroll
        for (int u = 0; u < kGrp; ++u) peers[u] = __match_any_sync(kFull, dg[u]);
#pragma unroll
        for (int u = 0; u < kGrp; ++u) {
          const uint32_t j = j0 + u * 32 + lane;
          const bool valid = j < je;
          const int leader = __ffs(peers[u]) - 1;
          uint32_t pre = 0;
          if (lane == (uint32_t)leader && valid) {
            pre = wh[dg[u]];
            wh[dg[u]] = pre + __popc(peers[u]);
          }
          pre = __shfl_sync(kFull, pre, leader);
          if (valid) s_aux[j] = pre + __popc(peers[u] & lt);
          __syncwarp();
        }
      }
      __syncthreads();
      // per digit: the warps' exclusive offsets, and this CTA's count
#pragma unroll
      for (int qd = 0; qd < DPT; ++qd) {
        const uint32_t dg = threadIdx.x * DPT + qd;
        if (dg < (uint32_t)RADIX) {
          uint32_t count = 0;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            const uint32_t c = s_whist[w * RADIX + dg];
            s_whist[w * RADIX + dg] = count;
            count += c;
          }
          s_cnt[dg] = count;
        }
      }
      cluster.sync();  // every CTA's digit counts are published
      // per digit: counts of the cluster's CTAs before this one, and the table's total
      // (all remote loads are issued before the first is used)
      uint32_t below[DPT], tot[DPT], tsum = 0;
      uint32_t rc[DPT][kMaxCluster];
#pragma unroll
      for (int qd = 0; qd < DPT; ++qd) {
        const uint32_t dg = threadIdx.x * DPT + qd;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
          rc[qd][c] = dg < (uint32_t)RADIX && (uint32_t)c < CL ? cluster.map_shared_rank(s_cnt, c)[dg] : 0u;
      }
#pragma unroll
      for (int qd = 0; qd < DPT; ++qd) {
        below[qd] = 0;
        tot[qd] = 0;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
          if ((uint32_t)c < crank) below[qd] += rc[qd][c];
          tot[qd] += rc[qd][c];
        }
        tsum += tot[qd];
      }
      uint32_t all;
      uint32_t ex = block_excl_scan(tsum, s_misc, &all);
#pragma unroll
      for (int qd = 0; qd < DPT; ++qd) {
        const uint32_t dg = threadIdx.x * DPT + qd;
        if (dg < (uint32_t)RADIX) s_gbase[dg] = s0 + ex + below[qd];
        ex += tot[qd];
      }
      __syncthreads();
      uint32_t* kout = a.keys[p & 1];
      V* vout = reinterpret_cast<V*>(a.vals[p & 1]);
      bool over = false;
      for (uint32_t j0 = jb; j0 < je; j0 += 32 * kGrp) {
#pragma unroll
        for (int u = 0; u < kGrp; ++u) {
          const uint32_t j = j0 + u * 32 + lane;
          if (j < je) {
            const uint32_t key = s_key[j];
            const uint32_t digit = ((key - kbase) >> shift) & dmask;
            const uint32_t dst = s_gbase[digit] + wh[digit] + s_aux[j];
            if (dst < s1) {  // always true: the slices' counts add up to the segment
              kout[dst] = key;
              vout[dst] = s_val[j];
            } else {
              over = true;
            }
          }
        }
      }
      if (over) raise_error(a.ctl, a.sticky, kErrCapacity);
      cluster.sync();  // the pass's output is complete (and s_cnt may be reused)
    }

    // ---- run-length encode and long-run partition of the sorted segment
    const uint32_t* fk = a.keys[(a.passes - 1) & 1];
#pragma unroll 8
    for (uint32_t j = threadIdx.x; j < n; j += kThreads) s_key[j] = __ldcg(fk + g0 + j);
    const uint32_t prev_key = i0 > 0 ? __ldcg(fk + g0 - 1) : 0u;
    __syncthreads();
    // each thread takes m consecutive positions
    const uint32_t m = (n + kThreads - 1) / kThreads;
    const uint32_t hb = min(threadIdx.x * m, n), he = min(hb + m, n);
    auto is_head = [&](uint32_t j) {
      if (i0 + j == 0) return true;  // the table's first lookup
      return s_key[j] != (j == 0 ? prev_key : s_key[j - 1]);
    };
    uint32_t nh = 0;
    for (uint32_t j = hb; j < he; ++j) nh += is_head(j) ? 1u : 0u;
    uint32_t n_heads;
    const uint32_t h0 = block_excl_scan(nh, s_misc, &n_heads);
    {
      uint32_t h = h0;
      for (uint32_t j = hb; j < he; ++j)
        if (is_head(j)) s_aux[h++] = j;
    }
    __syncthreads();
    if (warp == 0 && n_heads > 0) {  // end of the slice's last run (it may continue into later slices)
      const uint32_t e = run_end_in(fk, s1, g0 + n, s_key[s_aux[n_heads - 1]]);
      if (lane == 0) s_aux[n_heads] = e - g0;
    }
    __syncthreads();
    uint32_t n_long = 0, n_llook = 0;
    for (uint32_t h = h0; h < h0 + nh; ++h) {
      const uint32_t SL = s_aux[h + 1] - s_aux[h];
      if (SL >= a.thr) {
        n_long += 1;
        n_llook += SL;
      }
    }
    uint32_t e_long, e_llook, t_long, t_llook;
    block_excl_scan2(n_long, n_llook, s_misc, &e_long, &e_llook, &t_long, &t_llook);
    if (threadIdx.x == 0) {
      s_misc[kMiscMine + 0] = n_heads;
      s_misc[kMiscMine + 1] = t_long;
      s_misc[kMiscMine + 2] = t_llook;
    }
    cluster.sync();  // every CTA's run counts are published
    if (threadIdx.x < 3) {
      uint32_t rv[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c)
        rv[c] = (uint32_t)c < CL ? cluster.map_shared_rank(s_misc, c)[kMiscMine + threadIdx.x] : 0u;
      uint32_t below = 0, tot = 0;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        if ((uint32_t)c < crank) below += rv[c];
        tot += rv[c];
      }
      s_misc[kMiscBelow + threadIdx.x] = below;
      s_misc[kMiscTotal + threadIdx.x] = tot;
    }
    __syncthreads();
    cluster_arrive_relaxed();  // this CTA's reads of the cluster's counts are done
    if (warp < 3) {
      const uint32_t ex = table_lookback(a.lb, t, warp, s_misc[kMiscTotal + warp], crank == 0, a.ctl, a.sticky);
      if (lane == 0) s_misc[kMiscTable + warp] = ex;
    }
    __syncthreads();
    const uint32_t R = s_misc[kMiscTable + 0] + s_misc[kMiscBelow + 0];  // first run of the slice
    uint32_t kl = s_misc[kMiscTable + 1] + s_misc[kMiscBelow + 1] + e_long;
    uint32_t lp = s_misc[kMiscTable + 2] + s_misc[kMiscBelow + 2] + e_llook;
    bool overflow = false;
    for (uint32_t h = h0; h < h0 + nh; ++h) {
      const uint32_t r = R + h;
      const uint32_t j = s_aux[h];
      const uint32_t start = g0 + j, SL = s_aux[h + 1] - j;
      const uint32_t key = s_key[j];
      if (r < N) {
        a.run_key[r] = key;
        a.run_start[r] = start;
      } else {
        overflow = true;
      }
      if (SL >= a.thr) {
        if (kl < a.cap_long) {
          a.long_ids[kl] = r;
          a.longs[kl] = LongRun{start, SL, key, lp};
        } else {
          overflow = true;
        }
        kl += 1;
        lp += SL;
      }
    }
    if (overflow) raise_error(a.ctl, a.sticky, kErrCapacity);
    if (crank == 0 && threadIdx.x == 0) {
      const uint32_t Rt = s_misc[kMiscTable + 0];  // runs of the tables before t
      const uint32_t U = Rt + s_misc[kMiscTotal + 0];
      if (a.S > 1) {  // first run of each segment of tables that starts at table t
        for (uint32_t sg = 0; sg < a.S; ++sg)
          if (a.segs[sg] == t) a.seg_runs[sg] = Rt;
        if (t == d.T - 1) a.seg_runs[a.S] = U;
      }
      if (t == d.T - 1) {  // the last table knows every total
        if (U <= N) {
          a.ctl->num_runs = U;
          a.run_start[U] = N;
        } else {
          raise_error(a.ctl, a.sticky, kErrCapacity);
        }
        a.ctl->num_long = s_misc[kMiscTable + 1] + s_misc[kMiscTotal + 1];
        a.ctl->long_lookups = s_misc[kMiscTable + 2] + s_misc[kMiscTotal + 2];
      }
    }
    cluster_wait();  // every CTA has read the counts: s_misc may be reused, the CTA may exit
  }
}

template <int VK>
const void* cfront_fn_r(int radix) {
  if (radix == 128) return reinterpret_cast<const void*>(&k_cfront<VK, 128>);
  if (radix == 256) return reinterpret_cast<const void*>(&k_cfront<VK, 256>);
  return reinterpret_cast<const void*>(&k_cfront<VK, 512>);
}

const void* cfront_fn(int vk, int radix) {
  if (vk == VK_BAG) return cfront_fn_r<VK_BAG>(radix);
  if (vk == VK_NOBAG) return cfront_fn_r<VK_NOBAG>(radix);
  return cfront_fn_r<VK_BAG_SCALED>(radix);
}

cudaLaunchConfig_t cfront_config(int cl, int clusters, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr,
                                 bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * cl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

}  // namespace

size_t cfront_smem(int vk, int radix, bool mean, uint32_t cap) {
  return cf_layout(radix, vk == VK_BAG_SCALED ? 8 : 4, vk == VK_BAG_SCALED && mean, cap).total;
}

cudaError_t cfront_configure(int smem_optin) {
  cudaError_t e = cudaSuccess;
  for (int vk : {VK_BAG, VK_BAG_SCALED, VK_NOBAG})
    for (int radix : {128, 256, 512}) {
      const void* fn = cfront_fn(vk, radix);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
  return e;
}

int cfront_max_clusters(int vk, int radix, int cl, size_t smem) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cfront_config(cl, 1, smem, nullptr, attr, false);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, cfront_fn(vk, radix), &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_cfront(const CfrontArgs& a, int vk, int radix, int cl, int clusters, size_t smem,
                          cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cfront_config(cl, clusters, smem, s, attr, pdl);
  CfrontArgs arg = a;
  void* args[] = {&arg};
  return cudaLaunchKernelExC(&cfg, cfront_fn(vk, radix), args);
}

}  // namespace embbwd
