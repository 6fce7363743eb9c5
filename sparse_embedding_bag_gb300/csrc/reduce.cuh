// Segment reduce + fused optimizer: for every unique touched row, the sum of
// the scaled gradient rows of its lookups, accumulated in fp32 registers, then
// the SGD or row-wise Adagrad update applied once to the row (and its state).
//
// Follows the two per-row kernels of
// "fbgemm_gpu/codegen/embedding_backward_split_template.cu"
// (*_kernel_warp_per_row_1 for ordinary rows, *_kernel_cta_per_row_1 for rows
// found by *_find_long_segments) with these changes for sm_103a:
//   * one persistent kernel instead of two launches: blocks first take block
//     work items of long runs from a global counter (dynamic, so hot rows are
//     balanced), then every warp strides over the short runs;
//   * a very long run is cut into parts of `part` lookups taken by different
//     blocks; each part writes an fp32 partial row and the last part to arrive
//     (an atomic counter, no waiting) sums the partials in part order and
//     applies the optimizer, so the result does not depend on scheduling;
//   * lanes are grouped by the row width: a row of cvec 16-byte vectors uses
//     Lg = pow2ceil(cvec) lanes, and 32/Lg lookups are gathered at once;
//   * the per-lookup scale (per-sample weight / L) travels with the sort
//     payload, so no gradient copy is made for mean pooling (that page's
//     grad_mean_kernel writes a scaled copy of grad_output);
//   * the weight row and its state are read and written exactly once.
// Optimizer formulas: SGD w -= lr*G; row-wise Adagrad m += sum(G^2)/D,
// w -= lr*G/(sqrt(m)+eps) ("tt_embeddings_cuda.cu",
// cache_backward_rowwise_adagrad_approx_kernel), computed in fp32 and rounded
// once to the weight's storage type.
#pragma once

#include "internal.cuh"

namespace embbwd {

template <int VK>
struct ValT {
  using type = uint32_t;
};
template <>
struct ValT<VK_BAG_SCALED> {
  using type = uint64_t;
};

__device__ __forceinline__ uint32_t log2_pow2ceil32(uint32_t n) {
  // smallest l with 2^l >= n, capped at 5 (a warp)
  if (n >= 32) return 5;
  return n <= 1 ? 0u : 32u - __clz(n - 1);
}

__device__ __forceinline__ float4 f4_fma(float s, float4 x, float4 acc) {
  return make_float4(fmaf(s, x.x, acc.x), fmaf(s, x.y, acc.y), fmaf(s, x.z, acc.z), fmaf(s, x.w, acc.w));
}
__device__ __forceinline__ float4 f4_add(float4 x, float4 acc) {
  return make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
}

// Shape of one row task: a chunk of up to KV*32 16-byte vectors of a row.
struct RowShape {
  uint32_t t;
  int64_t idx;
  uint32_t D;
  uint32_t cvec_off;  // first vector of the chunk
  uint32_t cvec;      // vectors in the chunk
  uint32_t lg;        // log2 of lanes per lookup
  int64_t goff;       // column offset of the table in a gradient row
  uint32_t run;       // index of the row's run (set where the two-launch row-wise update needs it)
};

// Lookups gathered per lane group and step, unrolled for memory-level parallelism.
// Measured on GB300: 4 vectors per lane take 3 lookups per step (the large skewed
// workload's reduce 5.67 -> 5.56 ms against 2), 8 vectors per lane 2 (the LM
// reduce 101.7 us, 108.0 at 3), 2 vectors per lane 4 (the mixed-tables reduce
// 517 us, 531 at 2).
template <int KV, typename grad_t>
struct Unroll {
  static constexpr int value = KV == 4 ? 3 : (KV > 4 ? 2 : 4);
};

// Long-run lookups per warp up to which the reduce cuts one slice per warp and
// assigns it statically; above it, slices of at least kMinDynSlice lookups
// (about 16 per warp) are handed out dynamically.
constexpr uint32_t kStaticSlice = 256;
constexpr uint32_t kMinDynSlice = 64;

// Whether the gather loads the next step's sorted values while the current
// step's gradient rows are in flight (one dependent load less per step, for a
// few more registers). Measured on GB300: pays for unweighted pooled lookups of
// one team shape (DLRM-like reduce 33.5 -> 32.0 us, the large skewed one 7.19 ->
// 6.36 ms); with several team shapes, or 64-bit (weighted) values, it spills,
// and unpooled rows (whole-warp lookups of chunked wide rows) lost 12 %.
template <int VK, bool MULTI>
struct PrefetchVals {
  static constexpr bool value = !MULTI && VK == VK_BAG;
};

// Minimum resident blocks per SM, by vectors per lane (register budget).
// Measured on GB300: 2 vectors per lane run best at 3 blocks (80 registers)
// with the prefetch above, and at 4 blocks (64 registers) otherwise, also with
// several team shapes, where a few registers spill (the mixed-tables reduce
// 538 us at 3 blocks, 517 at 4, 750 at 2). 8 vectors per lane run better at 2 blocks
// (128 registers, a few spilled) than at 1 (223 registers) with one team shape:
// the LM reduce 101.6 us; row-wise Adagrad on 4 x 200k rows, B = 4096, L = 20,
// D = 1024 fp32 236.7 against 281.7 us per step, D = 768 fp16 234.6 against 302.2.
template <int KV, bool MULTI, int VK>
struct MinBlocks {
  static constexpr int value =
      KV == 1 ? 4 : (KV == 2 ? (PrefetchVals<VK, MULTI>::value ? 3 : 4) : (KV == 4 || !MULTI ? 2 : 1));
};

// Sum over sorted positions [jb, je) of one run into acc by a team of lanes.
// Within the team, lanes form groups of Lg = 2^rs.lg (one group per lookup,
// li = lane in group covering vectors li, li+Lg, ...), P groups gather P
// lookups per step, UNR steps are issued before any result is consumed.
// `steps` is warp-uniform (teams of one warp may hold runs of different length).
// PF: the sorted values of step s+1 are loaded right after the rows of step s.
template <int VK, typename grad_t, int KV, bool PF>
__device__ __forceinline__ void team_gather(const ReduceArgs& a, const RowShape& rs, uint32_t jb,
                                            uint32_t je, uint32_t steps, uint32_t P, uint32_t g,
                                            uint32_t li, float4 (&acc)[KV]) {
  using V = typename ValT<VK>::type;
  constexpr int UNR = Unroll<KV, grad_t>::value;
  const V* vals = reinterpret_cast<const V*>(a.vals);
  // Byte address of gradient row 0 of this run's table chunk; a lookup adds
  // (bag or lookup id) * stride with one 32x32->64 multiply. For pooled rows the
  // bag id's table part t*B is folded into the base (kept as an integer).
  const uint64_t stride = (uint64_t)a.grad_stride * sizeof(grad_t);
  // (unpooled gradient rows are [N, D]: no table column offset)
  const uint64_t goff = VK == VK_NOBAG ? 0ull : (uint64_t)rs.goff;
  uint64_t base = reinterpret_cast<uint64_t>(a.grad) + (goff + rs.cvec_off * 4ull) * sizeof(grad_t);
  if constexpr (VK != VK_NOBAG) base -= (uint64_t)(rs.t * a.B) * stride;
  // per-lane columns and masks of the chunk, the same for every lookup
  uint32_t col[KV];
  bool on[KV];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const uint32_t q = li + (k << rs.lg);
    on[k] = q < rs.cvec;
    col[k] = q * 4 * (uint32_t)sizeof(grad_t);
  }
#pragma unroll
  for (int k = 0; k < KV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  V vn[UNR];
  if constexpr (PF) {
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const uint32_t j = jb + u * P + g;
      vn[u] = (steps > 0 && j < je) ? vals[j] : (V)0;
    }
  }
  for (uint32_t s = 0; s < steps; ++s) {
    V v[UNR];
    bool ok[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const uint32_t j = jb + (s * UNR + u) * P + g;
      ok[u] = j < je;
      if constexpr (PF) v[u] = vn[u];
      else v[u] = ok[u] ? vals[j] : (V)0;
    }
    typename Vec4<grad_t>::Raw x[UNR][KV];  // loaded bits, widened when added
    float scale[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const uint64_t row = base + (uint64_t)(uint32_t)v[u] * stride;
      scale[u] = 1.0f;
      if constexpr (VK == VK_BAG_SCALED) scale[u] = __uint_as_float((uint32_t)(v[u] >> 32));
#pragma unroll
      for (int k = 0; k < KV; ++k)
        x[u][k] = (ok[u] && on[k]) ? Vec4<grad_t>::load_raw(reinterpret_cast<const grad_t*>(row + col[k]))
                                   : Vec4<grad_t>::zero_raw();
    }
    if constexpr (PF) {
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const uint32_t j = jb + ((s + 1) * UNR + u) * P + g;
        vn[u] = (s + 1 < steps && j < je) ? vals[j] : (V)0;
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const float4 f = Vec4<grad_t>::widen(x[u][k]);
        if constexpr (VK == VK_BAG_SCALED) acc[k] = f4_fma(scale[u], f, acc[k]);
        else acc[k] = f4_add(f, acc[k]);
      }
    }
  }
}

// Adds up the groups of a team (xor over lane offsets Lg .. Lt/2): afterwards
// every group of the team holds the run's totals. Shuffles are warp-uniform:
// they start at lane offset Lg0, the smallest group width of the warp's teams
// (teams whose groups are wider skip the offsets below their width).
template <int KV>
__device__ __forceinline__ void team_fold(float4 (&acc)[KV], uint32_t Lg, uint32_t Lt, uint32_t Lg0) {
  for (uint32_t off = Lg0; off < Lt; off <<= 1) {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      float4 y;
      y.x = __shfl_xor_sync(0xffffffffu, acc[k].x, off);
      y.y = __shfl_xor_sync(0xffffffffu, acc[k].y, off);
      y.z = __shfl_xor_sync(0xffffffffu, acc[k].z, off);
      y.w = __shfl_xor_sync(0xffffffffu, acc[k].w, off);
      if (off >= Lg) acc[k] = f4_add(y, acc[k]);
    }
  }
}

// The old weights of a row chunk (lane group 0 only; not read in dense-gradient mode).
template <typename emb_t, int OPT, int KV>
__device__ __forceinline__ void load_row(const ReduceArgs& a, const RowShape& rs, bool active,
                                         uint32_t g, uint32_t li, float4 (&w)[KV]) {
  if constexpr (OPT == 0) active = active && !a.dense;
  // rows of several chunks (8 vectors per lane only): the first of two launches updates no weights
  if constexpr (OPT == 1 && KV == 8) active = active && a.rw_pass != 1;
  const emb_t* row = static_cast<const emb_t*>(a.weights) +
                     (active ? __ldg(&a.weights_offsets[rs.t]) + rs.idx * rs.D : 0);
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const uint32_t q = li + (k << rs.lg);
    if (active && g == 0 && q < rs.cvec) w[k] = Vec4<emb_t>::load_plain(row + (int64_t)(rs.cvec_off + q) * 4);
    else w[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Store of updated weights: vector v (row-relative) of the row of rs. fp16 / bf16
// rows take stochastic rounding when the call asks for it; the four random
// words of the vector are Philox4x32-10 of the counter (linear row index, v,
// call number) under the key (seed), one word per element.
template <typename emb_t>
__device__ __forceinline__ void store_weights(const ReduceArgs& a, const RowShape& rs, emb_t* p,
                                              uint32_t v, float4 n) {
  if constexpr (sizeof(emb_t) == 2) {
    if (a.sr) {
      const uint32_t key = __ldg(&a.hsc[rs.t]) + (uint32_t)rs.idx;
      Vec4<emb_t>::store_sr(p, n, philox4x32_10(make_uint4(key, v, a.call_lo, a.call_hi), a.seed_lo, a.seed_hi));
      return;
    }
  }
  Vec4<emb_t>::store(p, n);
}

// Optimizer update of the chunk held by lane group 0 of a team of Lt lanes
// (acc = G, w = old weights, tl = lane in team). Warp-uniform shuffles.
//   OPT 0: SGD w -= lr * G, or in dense-gradient mode G stored to grad_out;
//   OPT 1: row-wise Adagrad (state per row);
//   OPT 2: elementwise Adagrad (state per element, laid out like the weights):
//          m += G^2, w -= lr * G / (sqrt(m) + eps).
template <typename emb_t, int OPT, int KV>
__device__ __forceinline__ void update_row(const ReduceArgs& a, const RowShape& rs, bool active,
                                           uint32_t g, uint32_t li, uint32_t tl, uint32_t Lt,
                                           const float4 (&acc)[KV], const float4 (&w)[KV],
                                           float m_old) {
  float mult = a.lr;
  if constexpr (OPT == 1) {
    float ss = 0.f;
    if (active && g == 0) {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const uint32_t q = li + (k << rs.lg);
        if (q < rs.cvec) ss += acc[k].x * acc[k].x + acc[k].y * acc[k].y + acc[k].z * acc[k].z + acc[k].w * acc[k].w;
      }
    }
    for (uint32_t off = 1; off < Lt; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    // Rows of several chunks take 8 vectors per lane (a row of more than 1024
    // elements); the narrower kernels carry only the one-launch update.
    const int rw_pass = KV == 8 ? a.rw_pass : 0;
    if (rw_pass == 1) {  // rows of several chunks, first launch: the row's state only
      if (active && tl == 0) {
        const uint32_t crow = ((rs.D >> 2) + KV * 32 - 1) / (KV * 32);  // chunks of this row
        float* slot = a.rw_ss + (size_t)rs.run * a.C;
        slot[rs.cvec_off / (KV * 32)] = ss;
        __threadfence();
        if (atomicAdd(&a.rw_cnt[rs.run], 1u) == crow - 1) {  // the last chunk to arrive
          __threadfence();
          float tot = 0.f;
          for (uint32_t k = 0; k < crow; ++k) tot += __ldcg(slot + k);
          const float m_new = m_old + __fdiv_rn(tot, (float)rs.D);
          a.momentum[__ldg(&a.momentum_offsets[rs.t]) + rs.idx] = m_new;
          a.rw_m[rs.run] = m_new;
          a.rw_cnt[rs.run] = 0;
        }
      }
      return;
    }
    if (rw_pass == 2) {  // second launch: the state the first one stored
      const float m_new = active ? a.rw_m[rs.run] : 0.f;
      mult = __fdiv_rn(a.lr, __fsqrt_rn(m_new) + a.eps);
    } else {
      const float m_new = m_old + __fdiv_rn(ss, (float)rs.D);
      mult = __fdiv_rn(a.lr, __fsqrt_rn(m_new) + a.eps);
      if (active && tl == 0) a.momentum[__ldg(&a.momentum_offsets[rs.t]) + rs.idx] = m_new;
    }
  }
  if (!active || g != 0) return;
  if constexpr (OPT == 0) {
    if (a.dense) {  // the gradient itself, in the weights' type and layout
      emb_t* grow = static_cast<emb_t*>(a.grad_out) + __ldg(&a.weights_offsets[rs.t]) + rs.idx * rs.D;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const uint32_t q = li + (k << rs.lg);
        if (q < rs.cvec) Vec4<emb_t>::store(grow + (int64_t)(rs.cvec_off + q) * 4, acc[k]);
      }
      return;
    }
  }
  emb_t* row = static_cast<emb_t*>(a.weights) + __ldg(&a.weights_offsets[rs.t]) + rs.idx * rs.D;
  if constexpr (OPT == 2) {
    float* mrow = a.momentum + __ldg(&a.weights_offsets[rs.t]) + rs.idx * rs.D;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const uint32_t q = li + (k << rs.lg);
      if (q < rs.cvec) {
        float4* mp = reinterpret_cast<float4*>(mrow + (int64_t)(rs.cvec_off + q) * 4);
        float4 m = *mp;
        m = make_float4(fmaf(acc[k].x, acc[k].x, m.x), fmaf(acc[k].y, acc[k].y, m.y),
                        fmaf(acc[k].z, acc[k].z, m.z), fmaf(acc[k].w, acc[k].w, m.w));
        *mp = m;
        const float4 n = make_float4(fmaf(-__fdiv_rn(a.lr, __fsqrt_rn(m.x) + a.eps), acc[k].x, w[k].x),
                                     fmaf(-__fdiv_rn(a.lr, __fsqrt_rn(m.y) + a.eps), acc[k].y, w[k].y),
                                     fmaf(-__fdiv_rn(a.lr, __fsqrt_rn(m.z) + a.eps), acc[k].z, w[k].z),
                                     fmaf(-__fdiv_rn(a.lr, __fsqrt_rn(m.w) + a.eps), acc[k].w, w[k].w));
        store_weights<emb_t>(a, rs, row + (int64_t)(rs.cvec_off + q) * 4, rs.cvec_off + q, n);
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const uint32_t q = li + (k << rs.lg);
    if (q < rs.cvec) {
      const float4 n = make_float4(fmaf(-mult, acc[k].x, w[k].x), fmaf(-mult, acc[k].y, w[k].y),
                                   fmaf(-mult, acc[k].z, w[k].z), fmaf(-mult, acc[k].w, w[k].w));
      store_weights<emb_t>(a, rs, row + (int64_t)(rs.cvec_off + q) * 4, rs.cvec_off + q, n);
    }
  }
}

// Shape of chunk c of the row with linear index `key` in table t; false if the
// chunk lies past the row's end.
template <int KV>
__device__ __forceinline__ bool shape_in(const uint32_t* s_hsc, const int32_t* s_Do, uint32_t t,
                                         uint32_t key, uint32_t c, RowShape* rs) {
  rs->t = t;
  rs->idx = (int64_t)(key - s_hsc[rs->t]);
  const int32_t d0 = s_Do[rs->t], d1 = s_Do[rs->t + 1];
  rs->D = (uint32_t)(d1 - d0);
  rs->goff = d0;
  const uint32_t nvec = rs->D >> 2;
  rs->cvec_off = c * (KV * 32);
  rs->cvec = rs->cvec_off < nvec ? min((uint32_t)(KV * 32), nvec - rs->cvec_off) : 0u;
  // lanes per lookup: the row's vectors spread so that each lane holds KV of them
  const uint32_t per_lane = (rs->cvec + KV - 1) / KV;
  rs->lg = log2_pow2ceil32(per_lane);
  return rs->cvec != 0;
}

template <int KV>
__device__ __forceinline__ bool make_shape(const ReduceArgs& a, const uint32_t* s_hsc,
                                           const int32_t* s_Do, uint32_t key, uint32_t c,
                                           RowShape* rs) {
  return shape_in<KV>(s_hsc, s_Do, table_of(s_hsc, a.T, key), key, c, rs);
}

// Index of the last long run whose place in the concatenation of long runs is
// <= x (runs are in key order, places strictly increasing, the first is 0).
// Warp-wide 32-way search: one load per lane and round.
__device__ __forceinline__ uint32_t find_long(const LongRun* longs, uint32_t n, uint32_t x) {
  const uint32_t lane = threadIdx.x & 31;
  uint32_t lo = 0, hi = n;  // the answer is in [lo, hi); longs[lo].lpos <= x
  while (hi - lo > 1) {
    const uint32_t step = (hi - lo + 31) >> 5;
    const uint32_t i = lo + lane * step;
    const bool le = i < hi && longs[i].lpos <= x;
    const uint32_t m = __popc(__ballot_sync(0xffffffffu, le));  // >= 1: lane 0 reads lo
    lo += (m - 1) * step;
    hi = min(lo + step, hi);
  }
  return lo;
}

// Pieces of a run cut by slice ends: the run covers slices sa .. sb of a row
// chunk whose slices start at index `base`; the piece in slice q has partial row
// slot 2*(base+q)+1 if it starts the run (q == sa), else 2*(base+q). Pieces are
// combined in groups of kGroup slices: the last piece of a group to finish sums
// the group into the slot of its first piece, and the last group to finish sums
// the groups; all sums run in slice order, so the result does not depend on
// scheduling.
constexpr uint32_t kGroup = 16;

// Cut of the concatenated long runs of one row chunk (positions [0, Ltot)) into
// slices: nA slices of SLA lookups over [0, LA), then slices of SLB over the rest.
struct Slicing {
  uint32_t SLA, SLB, LA, nA, S1;
  __device__ __forceinline__ uint32_t of(uint32_t p) const { return p < LA ? p / SLA : nA + (p - LA) / SLB; }
  __device__ __forceinline__ uint32_t start(uint32_t s) const { return s < nA ? s * SLA : LA + (s - nA) * SLB; }
};

__device__ __forceinline__ size_t piece_slot(uint32_t base, uint32_t sa, uint32_t q) {
  return 2 * (size_t)(base + q) + (q == sa ? 1u : 0u);
}

// Sum of the partial rows of n pieces q_0 = q0, q_k = (q0 / step + k) * step, by
// the lane groups of a warp (group g adds q_g, q_{g+Pg}, ... in order, then the
// groups are folded). Every lane group ends with the total.
template <int KV>
__device__ __forceinline__ void sum_pieces(const ReduceArgs& a, const RowShape& rs, uint32_t g, uint32_t li,
                                           uint32_t base, uint32_t sa, uint32_t q0, uint32_t n,
                                           uint32_t step, float4 (&acc)[KV]) {
  constexpr int kAhead = 4;  // pieces loaded before any is added
  const uint32_t Pg = 32u >> rs.lg;
#pragma unroll
  for (int k = 0; k < KV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (uint32_t k0 = g; k0 < n; k0 += kAhead * Pg) {
    float4 x[kAhead][KV];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const uint32_t k = k0 + u * Pg;
      const uint32_t q = k == 0 ? q0 : (q0 / step + k) * step;
      const float4* pp = a.partials + piece_slot(base, sa, q) * (KV * 32);
#pragma unroll
      for (int kv = 0; kv < KV; ++kv) {
        const uint32_t v = li + (kv << rs.lg);
        x[u][kv] = (k < n && v < rs.cvec) ? __ldcg(pp + v) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u)
#pragma unroll
      for (int kv = 0; kv < KV; ++kv) acc[kv] = f4_add(x[u][kv], acc[kv]);
  }
  team_fold<KV>(acc, 1u << rs.lg, 32, 1u << rs.lg);
}

// Arrival of one piece (acc: its sum in every lane group). Returns true in the
// warp that completes the run, with the run's total in acc; false otherwise.
template <int KV>
__device__ __forceinline__ bool piece_arrive(const ReduceArgs& a, const RowShape& rs, uint32_t g, uint32_t li,
                                             uint32_t base, uint32_t sa, uint32_t sb, uint32_t s,
                                             float4 (&acc)[KV]) {
  const uint32_t lane = threadIdx.x & 31;
  auto store = [&](size_t slot) {
    if (g == 0) {
      float4* part = a.partials + slot * (KV * 32);
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const uint32_t v = li + (k << rs.lg);
        if (v < rs.cvec) part[v] = acc[k];
      }
    }
    __threadfence();
    __syncwarp();
  };
  auto arrive = [&](uint32_t* ctr, uint32_t expect) {  // true in the last of `expect` arrivals
    uint32_t prev = 0;
    if (lane == 0) prev = atomicAdd(ctr, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev != expect - 1) return false;
    __threadfence();
    if (lane == 0) *ctr = 0;  // ready for the next call
    return true;
  };
  store(piece_slot(base, sa, s));
  // this piece's group of slices: pieces fs .. ls
  const uint32_t fs = max(sa, s / kGroup * kGroup), ls = min(sb, s / kGroup * kGroup + kGroup - 1);
  const size_t gslot = piece_slot(base, sa, fs);
  if (!arrive(a.done + gslot, ls - fs + 1)) return false;
  sum_pieces<KV>(a, rs, g, li, base, sa, fs, ls - fs + 1, 1, acc);
  const uint32_t ga = sa / kGroup, gb = sb / kGroup;
  if (ga == gb) return true;
  store(gslot);  // the group's sum replaces its first piece
  if (!arrive(a.done_run + piece_slot(base, sa, sa), gb - ga + 1)) return false;
  sum_pieces<KV>(a, rs, g, li, base, sa, sa, gb - ga + 1, kGroup, acc);
  return true;
}

// MULTI: the tables form several segments of different team shapes (see
// phase 2); without it, one shape serves every table and phase 2 is one sweep.
template <typename emb_t, typename grad_t, int OPT, int VK, int KV, bool MULTI>
__global__ void __launch_bounds__(kThreads, MinBlocks<KV, MULTI, VK>::value) k_reduce(ReduceArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* s_hsc = reinterpret_cast<uint32_t*>(smem);  // [T+1]
  int32_t* s_Do = reinterpret_cast<int32_t*>(s_hsc + a.T + 1);  // [T+1]
  uint32_t* s_seg = reinterpret_cast<uint32_t*>(s_Do + a.T + 1);  // [S+1] first table of each segment
  uint32_t* s_segrun = s_seg + a.S + 1;                             // [S+1] first run of each segment
  constexpr int UNR = Unroll<KV, grad_t>::value;

  pdl_wait();
  pdl_trigger();
  // one round trip: the error word, the counts of the front, the table metadata
  const uint32_t err = ld_relaxed_u32(&a.ctl->err);
  const uint32_t NL = ld_relaxed_u32(&a.ctl->num_long);
  const uint32_t Ltot = ld_relaxed_u32(&a.ctl->long_lookups);
  const uint32_t U = ld_relaxed_u32(&a.ctl->num_runs);
  for (uint32_t i = threadIdx.x; i <= a.T; i += kThreads) {
    s_hsc[i] = a.hsc[i];
    s_Do[i] = a.D_offsets[i];
  }
  if constexpr (MULTI) {
    for (uint32_t i = threadIdx.x; i <= a.S; i += kThreads) {
      s_seg[i] = a.segs[i];
      s_segrun[i] = a.seg_runs[i];
    }
  }
  if (err) return;  // a check failed earlier in this call (the same word for every thread)
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t C = a.C;
  const uint32_t W = gridDim.x * kWarps, gw = blockIdx.x * kWarps + warp;

  // ---- phase 1: the long runs, concatenated and cut into S1 slices per row
  // chunk; one warp reduces one slice at a time. A run inside one
  // slice is updated at once; a run cut by slice ends leaves one fp32 partial per
  // piece, combined by the pieces that finish last (atomic counts, no waiting;
  // see piece_arrive) in slice order before the row is updated. Little long-run
  // work: one slice per warp, of at least min_slice lookups, assigned statically
  // (with less work than that per warp, fewer warps take the long runs and the
  // others start on the short runs at once). Much: about 32 slices per warp,
  // handed out through one counter per warp index of a block (slice g belongs to
  // counter g % kWarps), the next one requested while the current one is reduced.
  // Slices are handed out in key order, so their size sets how many tables'
  // gradient slabs are live at once: measured on the large skewed workload,
  // about 16 slices per warp (six tables' slabs, more than L2 holds) gave
  // 6.16 ms and 15.1 GB of DRAM traffic, about 32 gave 5.89 ms, about 64 gave
  // 5.93 ms and 10.0 GB.
  if (Ltot > 0) {
    const uint64_t per_warp = ((uint64_t)Ltot * C + W - 1) / W;
    const bool dynamic = per_warp > kStaticSlice;
    Slicing sl;
    if (!dynamic) {
      sl.SLA = sl.SLB = max((uint32_t)per_warp, a.min_slice);
      sl.nA = (Ltot + sl.SLA - 1) / sl.SLA;
      sl.LA = Ltot;
    } else {
      // about 32 slices per warp; with large slices, the last quarter of the
      // lookups in slices 4x smaller, so that the warps that take the last
      // slices finish together
      sl.SLA = max(kMinDynSlice, 1u << (32 - __clz((uint32_t)((per_warp + 31) / 32) - 1)));  // pow2ceil(per_warp / 32)
      sl.SLB = sl.SLA >= 256 ? sl.SLA / 4 : sl.SLA;
      sl.nA = (uint32_t)((uint64_t)Ltot * 3 / 4 / sl.SLA);
      sl.LA = sl.nA * sl.SLA;
    }
    sl.S1 = sl.nA + (Ltot - sl.LA + sl.SLB - 1) / sl.SLB;  // slices per row chunk
    const uint32_t S1 = sl.S1;
    const uint32_t NS = S1 * C;
    uint32_t j = blockIdx.x;  // this warp's slice is j * kWarps + warp
    for (;;) {
      const uint32_t gs = j * kWarps + warp;
      if (gs >= NS) break;
      uint32_t nj = j + gridDim.x;
      if (dynamic) {
        if (lane == 0) nj = gridDim.x + atomicAdd(&a.ctl->slice_ctr[warp][0], 1u);
        nj = __shfl_sync(0xffffffffu, nj, 0);
      }
      const uint32_t c = gs / S1, s = gs - c * S1;
      const uint32_t a0 = sl.start(s), b0 = min(sl.start(s + 1), Ltot);
      for (uint32_t kl = find_long(a.longs, NL, a0); kl < NL; ++kl) {
        const LongRun lr = a.longs[kl];
        if (lr.lpos >= b0) break;
        RowShape rs;
        if (!make_shape<KV>(a, s_hsc, s_Do, lr.key, c, &rs)) continue;  // chunk past this row's end
        if constexpr (OPT == 1 && KV == 8) rs.run = a.rw_pass ? __ldg(&a.long_ids[kl]) : 0u;
        const uint32_t p0 = lr.lpos, p1 = lr.lpos + lr.len;
        const bool whole = p0 >= a0 && p1 <= b0;
        const uint32_t Pg = 32u >> rs.lg;
        const uint32_t g = lane >> rs.lg, li = lane & ((1u << rs.lg) - 1);
        float4 wv[KV];
        float m_old = 0.f;
        const uint32_t jb = lr.start + (max(a0, p0) - p0), je = lr.start + (min(b0, p1) - p0);
        const uint32_t steps = (je - jb + Pg * UNR - 1) / (Pg * UNR);
        float4 acc[KV];
        team_gather<VK, grad_t, KV, PrefetchVals<VK, MULTI>::value>(a, rs, jb, je, steps, Pg, g, li, acc);
        team_fold<KV>(acc, 1u << rs.lg, 32, 1u << rs.lg);
        if (whole) {  // long runs: the row is read after the gather (registers)
          load_row<emb_t, OPT, KV>(a, rs, true, g, li, wv);
          if constexpr (OPT == 1) m_old = a.momentum[__ldg(&a.momentum_offsets[rs.t]) + rs.idx];
          update_row<emb_t, OPT, KV>(a, rs, true, g, li, lane, 32, acc, wv, m_old);
          continue;
        }
        // a piece of a run cut by slice ends
        if (!piece_arrive<KV>(a, rs, g, li, c * S1, sl.of(p0), sl.of(p1 - 1), s, acc)) continue;
        load_row<emb_t, OPT, KV>(a, rs, true, g, li, wv);
        if constexpr (OPT == 1) m_old = a.momentum[__ldg(&a.momentum_offsets[rs.t]) + rs.idx];
        update_row<emb_t, OPT, KV>(a, rs, true, g, li, lane, 32, acc, wv, m_old);
      }
      j = nj;
    }
  }

  // ---- phase 2: short runs, by segments of consecutive tables whose rows give
  // the same team shape (runs are in table order). In a segment a warp holds 32/Lt
  // teams of Lt lanes (Lt from the row width), one run (x chunk) each per round;
  // the rounds of all segments, in order, go round-robin to the warps. All warps
  // thus sweep the keys together (rows updated at the same time lie close in
  // memory), and narrow tables pack several runs per warp.
  // One round of a team: run bounds [start, end) and key, table t (kAnyTable:
  // found from the key), chunk c.
  constexpr uint32_t kAnyTable = 0xffffffffu;
  auto round = [&](bool active, uint32_t start, uint32_t end, uint32_t key, uint32_t t, uint32_t c,
                   uint32_t Lt, uint32_t tl, uint32_t run) {
    RowShape rs{0u, 0, 4u, 0u, 0u, 0u, 0, 0u};  // inactive teams: a harmless, in-range shape
    active = active && end - start < a.thr;
    if (active) {
      if (t == kAnyTable) t = a.T == 1 ? 0u : table_of(s_hsc, a.T, key);
      active = shape_in<KV>(s_hsc, s_Do, t, key, c, &rs);
      rs.run = run;
    }
    if (!__any_sync(0xffffffffu, active)) return;
    if (!active) {
      rs = RowShape{0u, 0, 4u, 0u, 0u, 0u, 0, 0u};
      start = end = 0;
    }
    const uint32_t Pt = Lt >> rs.lg;
    const uint32_t g = tl >> rs.lg, li = tl & ((1u << rs.lg) - 1);
    float4 wv[KV];
    load_row<emb_t, OPT, KV>(a, rs, active, g, li, wv);
    float m_old = 0.f;
    if constexpr (OPT == 1) {
      if (active) m_old = a.momentum[__ldg(&a.momentum_offsets[rs.t]) + rs.idx];
    }
    const uint32_t my_steps = (end - start + Pt * UNR - 1) / (Pt * UNR);
    const uint32_t steps = __reduce_max_sync(0xffffffffu, my_steps);
    float4 acc[KV];
    team_gather<VK, grad_t, KV, PrefetchVals<VK, MULTI>::value>(a, rs, start, end, steps, Pt, g, li, acc);
    const uint32_t lg0 = __reduce_min_sync(0xffffffffu, active ? rs.lg : 5u);
    team_fold<KV>(acc, 1u << rs.lg, Lt, 1u << lg0);
    update_row<emb_t, OPT, KV>(a, rs, active, g, li, tl, Lt, acc, wv, m_old);
  };
  if constexpr (!MULTI) {  // one team shape for all tables: one sweep over all runs
    const uint32_t nvec = (uint32_t)(s_Do[1] - s_Do[0]) >> 2;
    const uint32_t lgt = log2_pow2ceil32((min(nvec, (uint32_t)KV * 32) + KV - 1) / KV);
    const uint32_t Lt = 1u << lgt, NT = 32u >> lgt;
    const uint32_t team = lane >> lgt, tl = lane & (Lt - 1);
    const uint32_t tasks = U * C;  // < 2^31 (checked when the plan is made)
    const uint32_t rounds = (tasks + NT - 1) / NT;
    // Rounds are claimed in key order, one at a time: round k * kWarps + c from
    // counter c (the warp's index in its block), so that warps that spent longer
    // on the long runs take fewer of them; the next round is claimed, and its
    // run's bounds and key loaded, before this round's rows.
    uint32_t* ctr = &a.ctl->round_ctr[warp][0];
    auto claim = [&]() {
      uint32_t k = 0;
      if (lane == 0) k = atomicAdd(ctr, 1u);
      return __shfl_sync(0xffffffffu, k, 0) * (uint32_t)kWarps + warp;
    };
    auto meta = [&](uint32_t q, uint32_t& start, uint32_t& end, uint32_t& key) {
      const uint32_t task = q * NT + team;
      if (q < rounds && task < tasks) {
        const uint32_t r = C == 1 ? task : task / C;
        start = a.run_start[r];
        end = a.run_start[r + 1];
        key = a.run_key[r];
      }
    };
    uint32_t q = claim();
    uint32_t n_start = 0, n_end = 0, n_key = 0;
    meta(q, n_start, n_end, n_key);
    while (q < rounds) {
      const uint32_t task = q * NT + team;
      const uint32_t start = n_start, end = n_end, key = n_key;
      q = claim();
      meta(q, n_start, n_end, n_key);
      const uint32_t r = C == 1 ? task : task / C;
      round(task < tasks, start, end, key, kAnyTable, task - r * C, Lt, tl, r);
    }
  } else {
  uint32_t P = 0;  // rounds of the segments before
  for (uint32_t sg = 0; sg < a.S; ++sg) {
    const uint32_t t0 = s_seg[sg], t1 = s_seg[sg + 1];
    const uint32_t R0 = s_segrun[sg], nr = s_segrun[sg + 1] - R0;
    if (nr == 0) continue;
    const uint32_t nvec = (uint32_t)(s_Do[t0 + 1] - s_Do[t0]) >> 2;
    const uint32_t Ct = (nvec + KV * 32 - 1) / (KV * 32);  // chunks of a row
    const uint32_t lgt = log2_pow2ceil32((min(nvec, (uint32_t)KV * 32) + KV - 1) / KV);
    const uint32_t Lt = 1u << lgt, NT = 32u >> lgt;
    const uint32_t team = lane >> lgt, tl = lane & (Lt - 1);
    const uint32_t tasks = nr * Ct;
    const uint32_t rounds = (tasks + NT - 1) / NT;
    uint32_t q = (gw + W - P % W) % W;  // this warp's first round of the segment
    P += rounds;
    for (; q < rounds; q += W) {
      const uint32_t task = q * NT + team;
      uint32_t start = 0, end = 0, key = 0, t = t0, r = 0;
      if (task < tasks) {
        r = R0 + (Ct == 1 ? task : task / Ct);
        start = a.run_start[r];
        end = a.run_start[r + 1];
        key = a.run_key[r];
        if (t1 - t0 > 1) t = t0 + table_of(s_hsc + t0, t1 - t0, key);
      }
      round(task < tasks, start, end, key, t, Ct == 1 ? 0u : task % Ct, Lt, tl, r);
    }
  }
  }
}

template <typename emb_t, typename grad_t, int OPT, int VK, bool MULTI>
const void* pick_kv(int kv) {
  switch (kv) {
    case 1: return reinterpret_cast<const void*>(&k_reduce<emb_t, grad_t, OPT, VK, 1, MULTI>);
    case 2: return reinterpret_cast<const void*>(&k_reduce<emb_t, grad_t, OPT, VK, 2, MULTI>);
    case 4: return reinterpret_cast<const void*>(&k_reduce<emb_t, grad_t, OPT, VK, 4, MULTI>);
    case 8: return reinterpret_cast<const void*>(&k_reduce<emb_t, grad_t, OPT, VK, 8, MULTI>);
    default: return nullptr;
  }
}

template <typename emb_t, typename grad_t, bool MULTI>
const void* pick_vk(int opt, int vk, int kv) {
  if (opt == 0) {
    if (vk == VK_BAG) return pick_kv<emb_t, grad_t, 0, VK_BAG, MULTI>(kv);
    if (vk == VK_BAG_SCALED) return pick_kv<emb_t, grad_t, 0, VK_BAG_SCALED, MULTI>(kv);
    if (vk == VK_NOBAG) return pick_kv<emb_t, grad_t, 0, VK_NOBAG, MULTI>(kv);
  } else if (opt == 1) {
    if (vk == VK_BAG) return pick_kv<emb_t, grad_t, 1, VK_BAG, MULTI>(kv);
    if (vk == VK_BAG_SCALED) return pick_kv<emb_t, grad_t, 1, VK_BAG_SCALED, MULTI>(kv);
  } else if (opt == 2) {
    if (vk == VK_BAG) return pick_kv<emb_t, grad_t, 2, VK_BAG, MULTI>(kv);
    if (vk == VK_BAG_SCALED) return pick_kv<emb_t, grad_t, 2, VK_BAG_SCALED, MULTI>(kv);
    if (vk == VK_NOBAG) return pick_kv<emb_t, grad_t, 2, VK_NOBAG, MULTI>(kv);
  }
  return nullptr;
}

// Kernel entry of the requested variant for one (weight, gradient) type pair.
template <typename emb_t, typename grad_t>
const void* pick_reduce(const ReduceKey& k) {
  return k.multi ? pick_vk<emb_t, grad_t, true>(k.optimizer, k.value_kind, k.kv)
                 : pick_vk<emb_t, grad_t, false>(k.optimizer, k.value_kind, k.kv);
}

}  // namespace embbwd
