// Forward pooled lookup (EmbeddingBag forward): for bag b of table t,
//   out[b, D_offsets[t] + d] = sum over lookups i of the bag of s_i * W_t[indices[i], d],
// s_i = per_sample_weight_i (if given) times 1/L (mean pooling), the scale the
// backward applies to the same lookup, so the two are adjoint. A bag's output
// row is the sum of the rows it indexes as in "tt_embeddings_cuda.cu",
// cache_forward_kernel and reduce_output_kernel (fp32 accumulation of 4-wide
// vectors); here one persistent kernel for all tables: the bags of a segment of
// tables with one row width go round-robin to lane teams sized to that width
// (several bags per warp for narrow rows), rows wider than one team's chunk are
// split into chunks, gathers are unrolled 16-byte (or 8-byte for 16-bit types)
// loads, and the output is written once, rounded to its type. No sort, no
// scratch. Index and offset errors are latched in the plan's sticky word; the
// offending lookup is skipped (an offset pair out of order reads as an empty bag).
#include "internal.cuh"

namespace embbwd {

namespace {

__device__ __forceinline__ uint32_t fwd_log2_pow2ceil32(uint32_t n) {
  if (n >= 32) return 5;
  return n <= 1 ? 0u : 32u - __clz(n - 1);
}

// Lookups gathered per lane group and step. A 16-bit row vector in flight holds
// half the registers of an fp32 one, so with 4+ vectors per lane twice as many
// lookups fit (with fewer, the in-flight indices would spill).
template <int KV, typename emb_t>
struct FwdUnroll {
  static constexpr int value = KV >= 4 ? (sizeof(emb_t) == 2 ? 4 : 2) : 4;
};

template <typename emb_t, typename out_t, int KV>
__global__ void __launch_bounds__(kThreads, KV <= 2 ? 3 : (KV == 4 ? 2 : 1)) k_bag_fwd(FwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  int64_t* s_wo = reinterpret_cast<int64_t*>(smem);                // [T]
  uint32_t* s_hsc = reinterpret_cast<uint32_t*>(s_wo + a.T);       // [T+1]
  int32_t* s_Do = reinterpret_cast<int32_t*>(s_hsc + a.T + 1);     // [T+1]
  uint32_t* s_seg = reinterpret_cast<uint32_t*>(s_Do + a.T + 1);   // [S+1]
  constexpr int UNR = FwdUnroll<KV, emb_t>::value;
  pdl_wait();
  pdl_trigger();
  for (uint32_t i = threadIdx.x; i <= a.T; i += kThreads) {
    if (i < a.T) s_wo[i] = a.weights_offsets[i];
    s_hsc[i] = a.hsc[i];
    s_Do[i] = a.D_offsets[i];
  }
  for (uint32_t i = threadIdx.x; i <= a.S; i += kThreads) s_seg[i] = a.segs[i];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (a.offsets[0] != 0 || a.offsets[(int64_t)a.T * a.B] != a.N) atomicOr(a.sticky, kErrOffsets);
  }
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t W = gridDim.x * kWarps, gw = blockIdx.x * kWarps + warp;
  const emb_t* weights = static_cast<const emb_t*>(a.weights);
  bool bad_index = false, bad_offsets = false;

  uint32_t P = 0;  // rounds of the segments before
  for (uint32_t sg = 0; sg < a.S; ++sg) {
    const uint32_t t0 = s_seg[sg], t1 = s_seg[sg + 1];
    const uint32_t nvec0 = (uint32_t)(s_Do[t0 + 1] - s_Do[t0]) >> 2;
    const uint32_t Ct = (nvec0 + KV * 32 - 1) / (KV * 32);  // chunks of a row
    const uint32_t lgt = fwd_log2_pow2ceil32((min(nvec0, (uint32_t)KV * 32) + KV - 1) / KV);
    const uint32_t Lt = 1u << lgt, NT = 32u >> lgt;
    const uint32_t team = lane >> lgt, tl = lane & (Lt - 1);
    const uint32_t tasks = (t1 - t0) * a.B * Ct;  // (bag, chunk) pairs of the segment
    const uint32_t rounds = (tasks + NT - 1) / NT;
    uint32_t q = (gw + W - P % W) % W;  // this warp's first round of the segment
    P += rounds;
    for (; q < rounds; q += W) {
      const uint32_t task = q * NT + team;
      const bool valid = task < tasks;
      const uint32_t bti = valid ? (Ct == 1 ? task : task / Ct) : 0u;
      const uint32_t c = valid ? task - bti * Ct : 0u;
      const uint32_t bt = t0 * a.B + bti;
      const uint32_t t = bt / a.B, b = bt - t * a.B;
      int64_t start = 0, end = 0;
      if (valid) {
        start = a.offsets[bt];
        end = a.offsets[bt + 1];
        if (start < 0 || end < start || end > a.N) {
          bad_offsets = true;
          start = end = 0;
        }
      }
      // row shape of table t, chunk c
      const uint32_t D = (uint32_t)(s_Do[t + 1] - s_Do[t]);
      const uint32_t nvec = D >> 2;
      const uint32_t cvec_off = c * (KV * 32);
      const uint32_t cvec = valid && cvec_off < nvec ? min((uint32_t)(KV * 32), nvec - cvec_off) : 0u;
      const uint32_t lg = fwd_log2_pow2ceil32((cvec + KV - 1) / KV);
      const uint32_t Pt = Lt >> lg;
      const uint32_t g = tl >> lg, li = tl & ((1u << lg) - 1);
      const int64_t rows = (int64_t)(s_hsc[t + 1] - s_hsc[t]);
      const emb_t* tbase = weights + s_wo[t] + (int64_t)cvec_off * 4;
      const uint32_t L = (uint32_t)(end - start);
      const uint32_t my_steps = cvec ? (L + Pt * UNR - 1) / (Pt * UNR) : 0u;
      const uint32_t steps = __reduce_max_sync(0xffffffffu, my_steps);
      float4 acc[KV];
#pragma unroll
      for (int k = 0; k < KV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t st = 0; st < steps; ++st) {
        int64_t idx[UNR];
        float s[UNR];
        bool ok[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int64_t j = start + (int64_t)((st * UNR + u) * Pt + g);
          ok[u] = cvec != 0 && j < end;
          idx[u] = ok[u] ? a.indices[j] : 0;
          s[u] = 1.0f;
          if (ok[u] && a.psw) s[u] = a.psw[j];
        }
        typename Vec4<emb_t>::Raw x[UNR][KV];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          if (ok[u] && (idx[u] < 0 || idx[u] >= rows)) {
            bad_index = true;
            ok[u] = false;
          }
          if (a.mean && ok[u]) s[u] = __fdiv_rn(s[u], (float)L);
          const emb_t* row = tbase + (ok[u] ? idx[u] * (int64_t)D : 0);
#pragma unroll
          for (int k = 0; k < KV; ++k) {
            const uint32_t v = li + (k << lg);
            x[u][k] = (ok[u] && v < cvec) ? Vec4<emb_t>::load_raw(row + (int64_t)v * 4)
                                          : Vec4<emb_t>::zero_raw();
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u)
#pragma unroll
          for (int k = 0; k < KV; ++k) {
            const float4 f = Vec4<emb_t>::widen(x[u][k]);
            acc[k].x = fmaf(s[u], f.x, acc[k].x);
            acc[k].y = fmaf(s[u], f.y, acc[k].y);
            acc[k].z = fmaf(s[u], f.z, acc[k].z);
            acc[k].w = fmaf(s[u], f.w, acc[k].w);
          }
      }
      // fold the lane groups of the team (xor over lane offsets 2^lg .. Lt/2)
      for (uint32_t off = 1; off < Lt; off <<= 1) {
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          float4 y;
          y.x = __shfl_xor_sync(0xffffffffu, acc[k].x, off);
          y.y = __shfl_xor_sync(0xffffffffu, acc[k].y, off);
          y.z = __shfl_xor_sync(0xffffffffu, acc[k].z, off);
          y.w = __shfl_xor_sync(0xffffffffu, acc[k].w, off);
          if (off >= (1u << lg)) {
            acc[k].x += y.x;
            acc[k].y += y.y;
            acc[k].z += y.z;
            acc[k].w += y.w;
          }
        }
      }
      if (g == 0 && cvec) {
        out_t* orow = static_cast<out_t*>(a.out) + (int64_t)b * a.out_stride + s_Do[t] + (int64_t)cvec_off * 4;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          const uint32_t v = li + (k << lg);
          if (v < cvec) Vec4<out_t>::store(orow + (int64_t)v * 4, acc[k]);
        }
      }
    }
  }
  if (bad_index) atomicOr(a.sticky, kErrIndex);
  if (bad_offsets) atomicOr(a.sticky, kErrOffsets);
}

template <typename emb_t, typename out_t>
const void* fwd_kv(int kv) {
  switch (kv) {
    case 1: return reinterpret_cast<const void*>(&k_bag_fwd<emb_t, out_t, 1>);
    case 2: return reinterpret_cast<const void*>(&k_bag_fwd<emb_t, out_t, 2>);
    case 4: return reinterpret_cast<const void*>(&k_bag_fwd<emb_t, out_t, 4>);
    case 8: return reinterpret_cast<const void*>(&k_bag_fwd<emb_t, out_t, 8>);
    default: return nullptr;
  }
}

template <typename emb_t>
const void* fwd_out(int out_dtype, int kv) {
  switch (out_dtype) {
    case 0: return fwd_kv<emb_t, float>(kv);
    case 1: return fwd_kv<emb_t, __half>(kv);
    case 2: return fwd_kv<emb_t, __nv_bfloat16>(kv);
    default: return nullptr;
  }
}

}  // namespace

const void* fwd_kernel(int weight_dtype, int out_dtype, int kv) {
  switch (weight_dtype) {
    case 0: return fwd_out<float>(out_dtype, kv);
    case 1: return fwd_out<__half>(out_dtype, kv);
    case 2: return fwd_out<__nv_bfloat16>(out_dtype, kv);
    default: return nullptr;
  }
}

size_t fwd_smem_bytes(int T, int S) {
  return (size_t)T * sizeof(int64_t) + 2 * (size_t)(T + 1) * sizeof(uint32_t) + (size_t)(S + 1) * sizeof(uint32_t);
}

}  // namespace embbwd
