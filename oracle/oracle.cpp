// CPU oracle for the embedding backward pass with a fused row optimizer.
//
// TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
// cpu_baseline / reference leg of bench.py may load this library. The product
// path (the CUDA library under sparse_embedding_bag_gb300/) never calls it and
// shares no code, header, table or helper with it.
//
// Plain, slow, single-threaded C++ that follows the definition of the
// operation step by step:
//   1. linearise every lookup i of bag (t, b) to hash_size_cumsum[t] + indices[i]
//      ("fbgemm_gpu/codegen/embedding_backward_split_template.cu",
//       kernels *_kernel_cta_per_row_1 / *_kernel_warp_per_row_1: the linear
//       index and the hash_size_cumsum subtraction; "tt_embeddings_cuda.cu",
//       compute_rowidx_kernel: the CSR bag expansion, table-major);
//   2. sort the (linear index, lookup id) pairs with std::sort;
//   3. run-length encode the sorted keys, exclusive scan of run lengths, and
//      the set of runs at least max_segment_length_per_warp long
//      ("embedding_backward_split_template.cu", *_find_long_segments);
//   4. accumulate, in double, for every unique row the sum of the scaled
//      gradient rows of its lookups: scale = per_sample_weight (if weighted)
//      times 1/L (if mean pooling) ("embedding_backward_split_template.cu",
//      grad_mean_kernel and the weighted fma in the per-row kernels);
//   5. apply the optimizer once per unique row, in double:
//        SGD:              w <- w - lr * G
//          ("tt_embeddings_cuda.cu", update_tt_cores_sgd_kernel,
//           cache_backward_sgd_kernel)
//        row-wise Adagrad: m <- m + sum_d(G_d^2) / D ; w <- w - lr * G / (sqrt(m) + eps)
//          ("tt_embeddings_cuda.cu", cache_backward_rowwise_adagrad_approx_kernel:
//           mean of squares over D, state updated before use, eps outside the
//           square root), applied to the de-duplicated row gradient;
//   6. round w to its storage type (round to nearest, ties to even) and m to fp32.
//
// The forward pooled lookup (oracle_forward) is the adjoint of steps 1-4.
// Row-wise sharding (oracle_bucketize, oracle_merge) is the exchange step of a
// deployment over several ranks: each lookup moved to the rank owning its row.
//
// Every function here is pinned by tests/test_oracle_*.py against brute force
// (a dense one-hot matrix product), closed forms and invariants.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };
enum { OK = 0, ERR_INVALID_ARG = 1, ERR_UNSUPPORTED = 2, ERR_INDEX_OUT_OF_RANGE = 3 };

// ---- storage-type conversions, written from the IEEE 754 binary16 and the
// ---- bfloat16 (binary32 with the low 16 mantissa bits dropped) formats.

double half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);  // subnormal: m * 2^-24
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(1024 + m), e - 25);  // (1 + m/1024) * 2^(e-15)
  }
  return sign ? -v : v;
}

// Direct double -> binary16 with round-to-nearest-even (no intermediate fp32,
// so there is no double rounding).
uint16_t double_to_half(double x) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  if (std::isnan(x)) return sign | 0x7E00;
  if (std::isinf(x)) return sign | 0x7C00;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (a < std::ldexp(1.0, -14)) {
    // subnormal grid: multiples of 2^-24. rint rounds half to even.
    const double q = std::rint(std::ldexp(a, 24));
    return sign | static_cast<uint16_t>(q);  // q == 1024 encodes the smallest normal
  }
  int e2;
  std::frexp(a, &e2);  // a = f * 2^e2, f in [0.5, 1)
  int E = e2 - 1;      // a in [2^E, 2^(E+1))
  double r = std::rint(std::ldexp(a, 10 - E));  // in [1024, 2048]
  if (r == 2048.0) {
    r = 1024.0;
    E += 1;
  }
  if (E > 15) return sign | 0x7C00;  // overflow to infinity
  return sign | static_cast<uint16_t>(((E + 15) << 10) | (static_cast<int>(r) - 1024));
}

double bf16_to_double(uint16_t h) {
  const uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return static_cast<double>(f);
}

uint16_t double_to_bf16(double x) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  if (std::isnan(x)) return sign | 0x7FC0;
  if (std::isinf(x)) return sign | 0x7F80;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (a < std::ldexp(1.0, -126)) {
    const double q = std::rint(std::ldexp(a, 133));  // multiples of 2^-133
    return sign | static_cast<uint16_t>(q);
  }
  int e2;
  std::frexp(a, &e2);
  int E = e2 - 1;
  double r = std::rint(std::ldexp(a, 7 - E));  // in [128, 256]
  if (r == 256.0) {
    r = 128.0;
    E += 1;
  }
  if (E > 127) return sign | 0x7F80;
  return sign | static_cast<uint16_t>(((E + 127) << 7) | (static_cast<int>(r) - 128));
}

// ---- stochastic rounding of fp16 / bf16 stores.
// Random words: Philox4x32-10, written from its published definition (Salmon,
// Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
// ten rounds of two 32x32->64 multiplies by M0, M1 on a 4-word counter, with the
// 2-word key bumped by the Weyl constants W0, W1 between rounds.
void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k[2] = {key_in[0], key_in[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += W0;
      k[1] += W1;
    }
    const uint64_t p0 = M0 * c[0], p1 = M1 * c[2];
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    const uint32_t n[4] = {hi1 ^ c[1] ^ k[0], lo1, hi0 ^ c[3] ^ k[1], lo0};
    for (int j = 0; j < 4; ++j) c[j] = n[j];
  }
  for (int j = 0; j < 4; ++j) out[j] = c[j];
}

// fp32 x to bf16 with probability of rounding away from zero equal to the
// dropped fraction: add 16 random bits to the dropped low half, truncate.
uint16_t sr_bf16(float x, uint32_t r) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  return static_cast<uint16_t>((u + (r & 0xFFFFu)) >> 16);
}

// fp32 x to fp16: the neighbour toward zero, moved one ulp away from zero with
// probability (|x| - |lo|) / ulp, compared on 24 random bits (both exact in fp32).
uint16_t sr_half(float x, uint32_t r) {
  uint16_t lo = double_to_half(static_cast<double>(x));  // nearest; step toward zero if past x
  if (std::fabs(half_to_double(lo)) > std::fabs(static_cast<double>(x))) lo = static_cast<uint16_t>(lo - 1);
  if ((lo & 0x7C00) == 0x7C00) return lo;  // inf / nan
  const uint16_t hi = static_cast<uint16_t>(lo + 1);
  const float a = std::fabs(static_cast<float>(half_to_double(lo)));
  const float b = std::fabs(static_cast<float>(half_to_double(hi)));
  const float frac = (std::fabs(x) - a) / (b - a);
  const uint32_t thresh = static_cast<uint32_t>(frac * 16777216.0f);
  return (r >> 8) < thresh ? hi : lo;
}

double load_elem(const void* base, int dtype, int64_t i) {
  switch (dtype) {
    case DT_F32: return static_cast<double>(static_cast<const float*>(base)[i]);
    case DT_F16: return half_to_double(static_cast<const uint16_t*>(base)[i]);
    default: return bf16_to_double(static_cast<const uint16_t*>(base)[i]);
  }
}

void store_elem(void* base, int dtype, int64_t i, double v) {
  switch (dtype) {
    case DT_F32: static_cast<float*>(base)[i] = static_cast<float>(v); break;  // C cast: RNE
    case DT_F16: static_cast<uint16_t*>(base)[i] = double_to_half(v); break;
    default: static_cast<uint16_t*>(base)[i] = double_to_bf16(v); break;
  }
}

// A 16-bit store with stochastic rounding of v rounded first to fp32 (the type
// the update is computed in on the device); fp32 stores are plain.
void store_elem_sr(void* base, int dtype, int64_t i, double v, uint32_t r) {
  const float f = static_cast<float>(v);
  switch (dtype) {
    case DT_F32: static_cast<float*>(base)[i] = f; break;
    case DT_F16: static_cast<uint16_t*>(base)[i] = sr_half(f, r); break;
    default: static_cast<uint16_t*>(base)[i] = sr_bf16(f, r); break;
  }
}

// Random word of element d of the row with linear index `key` in update call
// `call`: word d % 4 of Philox4x32-10 at counter (key, d / 4, call_lo, call_hi)
// under the 64-bit seed.
uint32_t sr_word(uint64_t seed, uint64_t call, int64_t key, int32_t d) {
  const uint32_t ctr[4] = {static_cast<uint32_t>(key), static_cast<uint32_t>(d / 4),
                           static_cast<uint32_t>(call), static_cast<uint32_t>(call >> 32)};
  const uint32_t k[2] = {static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, k, out);
  return out[d % 4];
}

// Stochastic rounding of the weight stores of one call (or off).
struct Rounding {
  int on = 0;
  uint64_t seed = 0, call = 0;
  int64_t key = 0;  // linear index of the row being stored
};

struct Pair {
  int64_t key;  // linear index
  int64_t id;   // lookup id (position in indices)
};

// Steps 1-2. Also records the bag of every lookup. Returns a status code.
int linearise_and_sort(int32_t T, int32_t B, const int64_t* hsc, const int64_t* indices,
                       const int64_t* offsets, int64_t N, std::vector<Pair>* pairs,
                       std::vector<int64_t>* bag_of) {
  if (T <= 0 || B <= 0 || N < 0) return ERR_INVALID_ARG;
  if (offsets[0] != 0 || offsets[static_cast<int64_t>(B) * T] != N) return ERR_INVALID_ARG;
  pairs->clear();
  pairs->reserve(static_cast<size_t>(N));
  bag_of->assign(static_cast<size_t>(N), -1);
  for (int64_t bt = 0; bt < static_cast<int64_t>(B) * T; ++bt) {
    if (offsets[bt + 1] < offsets[bt]) return ERR_INVALID_ARG;
    const int64_t t = bt / B;
    const int64_t rows = hsc[t + 1] - hsc[t];
    for (int64_t i = offsets[bt]; i < offsets[bt + 1]; ++i) {
      if (indices[i] < 0 || indices[i] >= rows) return ERR_INDEX_OUT_OF_RANGE;
      pairs->push_back(Pair{hsc[t] + indices[i], i});
      (*bag_of)[i] = bt;
    }
  }
  std::sort(pairs->begin(), pairs->end(), [](const Pair& a, const Pair& b) {
    return a.key != b.key ? a.key < b.key : a.id < b.id;
  });
  return OK;
}

int32_t table_of_key(int32_t T, const int64_t* hsc, int64_t key) {
  int32_t t = 0;
  while (t + 1 < T && hsc[t + 1] <= key) ++t;
  return t;
}

struct Runs {
  std::vector<int64_t> keys;
  std::vector<int64_t> start;  // start[r] = first position of run r; start[U] = N
};

Runs encode_runs(const std::vector<Pair>& pairs) {
  Runs R;
  for (size_t i = 0; i < pairs.size(); ++i) {
    if (i == 0 || pairs[i].key != pairs[i - 1].key) {
      R.keys.push_back(pairs[i].key);
      R.start.push_back(static_cast<int64_t>(i));
    }
  }
  R.start.push_back(static_cast<int64_t>(pairs.size()));
  return R;
}

bool valid_tables(int32_t T, const int64_t* hsc, const int32_t* D_offsets) {
  if (hsc[0] != 0) return false;
  for (int32_t t = 0; t < T; ++t) {
    if (hsc[t + 1] <= hsc[t]) return false;  // disjoint, non-empty tables
    if (D_offsets && D_offsets[t + 1] <= D_offsets[t]) return false;
  }
  return true;
}

}  // namespace

extern "C" {

// Linearise + sort: sorted (key, lookup id) pairs. keys/ids have capacity N.
int oracle_sorted_pairs(int32_t T, int32_t B, const int64_t* hsc, const int64_t* indices,
                        const int64_t* offsets, int64_t N, int64_t* keys, int64_t* ids) {
  std::vector<Pair> pairs;
  std::vector<int64_t> bag_of;
  const int st = linearise_and_sort(T, B, hsc, indices, offsets, N, &pairs, &bag_of);
  if (st != OK) return st;
  for (int64_t i = 0; i < N; ++i) {
    keys[i] = pairs[i].key;
    ids[i] = pairs[i].id;
  }
  return OK;
}

// Integer outputs of the sort / run-length / long-segment steps.
//   run_keys[U]  ascending unique linear indices
//   run_len[U]   lookups per unique index
//   cum[U+1]     exclusive scan of run_len (cum[0] = 0, cum[U] = N)
//   long_ids[..] run ids with run_len >= max_segment_length_per_warp, ascending
// Output arrays have capacity N (cum: N + 1).
int oracle_runs(int32_t T, int32_t B, const int64_t* hsc, const int64_t* indices,
                const int64_t* offsets, int64_t N, int32_t max_segment_length_per_warp,
                int64_t* run_keys, int32_t* run_len, int32_t* cum, int64_t* num_runs,
                int32_t* long_ids, int64_t* num_long) {
  std::vector<Pair> pairs;
  std::vector<int64_t> bag_of;
  const int st = linearise_and_sort(T, B, hsc, indices, offsets, N, &pairs, &bag_of);
  if (st != OK) return st;
  const Runs R = encode_runs(pairs);
  const int64_t U = static_cast<int64_t>(R.keys.size());
  int64_t nl = 0;
  for (int64_t r = 0; r < U; ++r) {
    run_keys[r] = R.keys[r];
    run_len[r] = static_cast<int32_t>(R.start[r + 1] - R.start[r]);
    cum[r] = static_cast<int32_t>(R.start[r]);
    if (run_len[r] >= max_segment_length_per_warp) long_ids[nl++] = static_cast<int32_t>(r);
  }
  cum[U] = static_cast<int32_t>(N);
  *num_runs = U;
  *num_long = nl;
  return OK;
}

// Step 4: de-duplicated row gradients, in double.
//   nobag == 0: grad_output is [B, D_offsets[T]] and lookup i of bag (t, b)
//               contributes scale_i * grad_output[b, D_offsets[t] : D_offsets[t+1]].
//   nobag != 0: grad_output is [N, D] (all tables share D) and lookup l
//               contributes grad_output[l, :].
// Outputs: keys_out[U] and G[U * Dmax] (row r at G + r*Dmax, zero padded).
int oracle_row_grads(int32_t T, int32_t B, const int64_t* hsc, const int32_t* D_offsets,
                     const int64_t* indices, const int64_t* offsets, int64_t N,
                     const float* per_sample_weights, int32_t mean_pooling, int32_t nobag,
                     int32_t grad_dtype, const void* grad_output, int32_t Dmax,
                     int64_t* keys_out, double* G, int64_t* num_rows) {
  if (!valid_tables(T, hsc, D_offsets)) return ERR_INVALID_ARG;
  if (nobag && per_sample_weights) return ERR_UNSUPPORTED;  // weighted nobag is not defined
  if (nobag) {
    for (int32_t t = 1; t < T; ++t)
      if (D_offsets[t + 1] - D_offsets[t] != D_offsets[1] - D_offsets[0]) return ERR_INVALID_ARG;
  }
  std::vector<Pair> pairs;
  std::vector<int64_t> bag_of;
  const int st = linearise_and_sort(T, B, hsc, indices, offsets, N, &pairs, &bag_of);
  if (st != OK) return st;
  const Runs R = encode_runs(pairs);
  const int64_t U = static_cast<int64_t>(R.keys.size());
  const int64_t row_stride = D_offsets[T];
  for (int64_t r = 0; r < U; ++r) {
    const int32_t t = table_of_key(T, hsc, R.keys[r]);
    const int32_t D = D_offsets[t + 1] - D_offsets[t];
    if (D > Dmax) return ERR_INVALID_ARG;
    double* g = G + r * static_cast<int64_t>(Dmax);
    for (int32_t d = 0; d < Dmax; ++d) g[d] = 0.0;
    for (int64_t j = R.start[r]; j < R.start[r + 1]; ++j) {
      const int64_t i = pairs[j].id;
      if (nobag) {
        for (int32_t d = 0; d < D; ++d) g[d] += load_elem(grad_output, grad_dtype, i * D + d);
      } else {
        const int64_t bt = bag_of[i];
        const int64_t b = bt % B;
        double s = per_sample_weights ? static_cast<double>(per_sample_weights[i]) : 1.0;
        if (mean_pooling) {
          const int64_t L = offsets[bt + 1] - offsets[bt];  // >= 1: the bag holds lookup i
          s *= 1.0 / static_cast<double>(L);
        }
        const int64_t base = b * row_stride + D_offsets[t];
        for (int32_t d = 0; d < D; ++d) g[d] += s * load_elem(grad_output, grad_dtype, base + d);
      }
    }
    keys_out[r] = R.keys[r];
  }
  *num_rows = U;
  return OK;
}

// Step 5-6 on one row: applies the optimizer to row `w` (storage dtype) of
// length D with gradient g (double) and its fp32 state m (one value for
// row-wise Adagrad, D values for elementwise Adagrad).
//   optimizer 0 = SGD, 1 = row-wise Adagrad, 2 = elementwise Adagrad
//   ("tt_embeddings_cuda.cu", update_tt_cores_adagrad_kernel: per element
//   m <- m + g^2, w <- w - lr * g / (sqrt(m) + eps)).
int apply_row_impl(int32_t optimizer, int32_t weight_dtype, void* weights, int64_t row_offset,
                   int32_t D, const double* g, float* m, double lr, double eps, const Rounding& rnd);

int oracle_apply_row(int32_t optimizer, int32_t weight_dtype, void* weights, int64_t row_offset,
                     int32_t D, const double* g, float* m, double lr, double eps) {
  return apply_row_impl(optimizer, weight_dtype, weights, row_offset, D, g, m, lr, eps, Rounding());
}

int apply_row_impl(int32_t optimizer, int32_t weight_dtype, void* weights, int64_t row_offset,
                   int32_t D, const double* g, float* m, double lr, double eps, const Rounding& rnd) {
  auto store = [&](int64_t i, int32_t d, double v) {
    if (rnd.on) store_elem_sr(weights, weight_dtype, i, v, sr_word(rnd.seed, rnd.call, rnd.key, d));
    else store_elem(weights, weight_dtype, i, v);
  };
  if (optimizer == 2) {
    if (!m) return ERR_INVALID_ARG;
    for (int32_t d = 0; d < D; ++d) {
      const double m_new = static_cast<double>(m[d]) + g[d] * g[d];
      const double w = load_elem(weights, weight_dtype, row_offset + d);
      store(row_offset + d, d, w - lr * g[d] / (std::sqrt(m_new) + eps));
      m[d] = static_cast<float>(m_new);
    }
    return OK;
  }
  if (optimizer == 0) {
    for (int32_t d = 0; d < D; ++d) {
      const double w = load_elem(weights, weight_dtype, row_offset + d);
      store(row_offset + d, d, w - lr * g[d]);
    }
    return OK;
  }
  if (optimizer != 1 || !m) return ERR_INVALID_ARG;
  double sum_sq = 0.0;
  for (int32_t d = 0; d < D; ++d) sum_sq += g[d] * g[d];
  const double m_new = static_cast<double>(*m) + sum_sq / static_cast<double>(D);
  const double mult = lr / (std::sqrt(m_new) + eps);
  for (int32_t d = 0; d < D; ++d) {
    const double w = load_elem(weights, weight_dtype, row_offset + d);
    store(row_offset + d, d, w - mult * g[d]);
  }
  *m = static_cast<float>(m_new);
  return OK;
}

// The whole pooled (nobag == 0) or unpooled (nobag != 0) backward with the
// optimizer applied in place to each unique touched row. Untouched rows are
// not written. Row-wise Adagrad: momentum_offsets may be NULL (then row idx of
// table t uses momentum[hash_size_cumsum[t] + idx]). Elementwise Adagrad: the
// state has the layout of the weights (momentum[weights_offsets[t] + idx*D + d]).
// momentum is ignored for SGD.
int oracle_backward(int32_t T, int32_t B, const int64_t* hsc, const int32_t* D_offsets,
                    const int64_t* weights_offsets, const int64_t* momentum_offsets,
                    int32_t weight_dtype, void* weights, float* momentum,
                    const int64_t* indices, const int64_t* offsets, int64_t N,
                    const float* per_sample_weights, int32_t mean_pooling, int32_t nobag,
                    int32_t grad_dtype, const void* grad_output, int32_t optimizer, double lr,
                    double eps, int32_t stochastic_rounding, uint64_t seed, uint64_t call) {
  if (T <= 0 || B <= 0) return ERR_INVALID_ARG;
  if (N == 0) return OK;
  int32_t Dmax = 0;
  for (int32_t t = 0; t < T; ++t) Dmax = std::max(Dmax, D_offsets[t + 1] - D_offsets[t]);
  std::vector<int64_t> keys(static_cast<size_t>(N));
  std::vector<double> G(static_cast<size_t>(N) * static_cast<size_t>(Dmax));
  int64_t U = 0;
  const int st = oracle_row_grads(T, B, hsc, D_offsets, indices, offsets, N, per_sample_weights,
                                  mean_pooling, nobag, grad_dtype, grad_output, Dmax, keys.data(),
                                  G.data(), &U);
  if (st != OK) return st;
  for (int64_t r = 0; r < U; ++r) {
    const int32_t t = table_of_key(T, hsc, keys[r]);
    const int64_t idx = keys[r] - hsc[t];
    const int32_t D = D_offsets[t + 1] - D_offsets[t];
    float* m = nullptr;
    if (optimizer == 1) {
      const int64_t mo = momentum_offsets ? momentum_offsets[t] : hsc[t];
      m = momentum + mo + idx;
    } else if (optimizer == 2) {
      m = momentum + weights_offsets[t] + idx * D;
    }
    Rounding rnd;
    rnd.on = stochastic_rounding;
    rnd.seed = seed;
    rnd.call = call;
    rnd.key = keys[r];
    const int st2 = apply_row_impl(optimizer, weight_dtype, weights, weights_offsets[t] + idx * D, D,
                                   G.data() + r * static_cast<int64_t>(Dmax), m, lr, eps, rnd);
    if (st2 != OK) return st2;
  }
  return OK;
}

// Dense-gradient mode: the de-duplicated row gradient of every touched row,
// stored (rounded once to out_dtype) into `grad_weights`, which has the layout of
// the weights and is zeroed first over [0, extent) ("embedding_backward_split_
// template.cu", the dense variant: grad_dev_weights = zeros_like(dev_weights),
// then grad_sum stored at weights_offset + idx * D per touched row).
int oracle_dense_grad(int32_t T, int32_t B, const int64_t* hsc, const int32_t* D_offsets,
                      const int64_t* weights_offsets, int64_t extent, int32_t out_dtype,
                      void* grad_weights, const int64_t* indices, const int64_t* offsets,
                      int64_t N, const float* per_sample_weights, int32_t mean_pooling,
                      int32_t nobag, int32_t grad_dtype, const void* grad_output) {
  if (T <= 0 || B <= 0) return ERR_INVALID_ARG;
  for (int64_t e = 0; e < extent; ++e) store_elem(grad_weights, out_dtype, e, 0.0);
  if (N == 0) return OK;
  int32_t Dmax = 0;
  for (int32_t t = 0; t < T; ++t) Dmax = std::max(Dmax, D_offsets[t + 1] - D_offsets[t]);
  std::vector<int64_t> keys(static_cast<size_t>(N));
  std::vector<double> G(static_cast<size_t>(N) * static_cast<size_t>(Dmax));
  int64_t U = 0;
  const int st = oracle_row_grads(T, B, hsc, D_offsets, indices, offsets, N, per_sample_weights,
                                  mean_pooling, nobag, grad_dtype, grad_output, Dmax, keys.data(),
                                  G.data(), &U);
  if (st != OK) return st;
  for (int64_t r = 0; r < U; ++r) {
    const int32_t t = table_of_key(T, hsc, keys[r]);
    const int64_t idx = keys[r] - hsc[t];
    const int32_t D = D_offsets[t + 1] - D_offsets[t];
    for (int32_t d = 0; d < D; ++d)
      store_elem(grad_weights, out_dtype, weights_offsets[t] + idx * D + d,
                 G[static_cast<size_t>(r) * Dmax + d]);
  }
  return OK;
}

// Forward pooled lookup (EmbeddingBag forward), written from the definition:
// the output row of bag (t, b) is the sum over its lookups i of s_i times row
// indices[i] of table t, with the same per-lookup scale as the backward
// (s_i = per_sample_weight_i if weighted, times 1/L if mean pooling), so that
// the forward is the adjoint of the backward's scatter. "tt_embeddings_cuda.cu",
// cache_forward_kernel and reduce_output_kernel: a bag's output row is the sum
// of the rows it indexes. Accumulated in double, rounded once to out_dtype;
// out is [B, D_offsets[T]] and is overwritten (an empty bag gives zeros).
int oracle_forward(int32_t T, int32_t B, const int64_t* hsc, const int32_t* D_offsets,
                   const int64_t* weights_offsets, int32_t weight_dtype, const void* weights,
                   const int64_t* indices, const int64_t* offsets, int64_t N,
                   const float* per_sample_weights, int32_t mean_pooling, int32_t out_dtype,
                   void* out) {
  if (T <= 0 || B <= 0 || !valid_tables(T, hsc, D_offsets)) return ERR_INVALID_ARG;
  const int64_t BT = static_cast<int64_t>(T) * B;
  if (offsets[0] != 0 || offsets[BT] != N) return ERR_INVALID_ARG;
  for (int64_t bt = 0; bt < BT; ++bt)
    if (offsets[bt + 1] < offsets[bt]) return ERR_INVALID_ARG;
  for (int64_t bt = 0; bt < BT; ++bt) {
    const int32_t t = static_cast<int32_t>(bt / B);
    for (int64_t i = offsets[bt]; i < offsets[bt + 1]; ++i)
      if (indices[i] < 0 || indices[i] >= hsc[t + 1] - hsc[t]) return ERR_INDEX_OUT_OF_RANGE;
  }
  const int64_t row_stride = D_offsets[T];
  std::vector<double> acc;
  for (int64_t bt = 0; bt < BT; ++bt) {
    const int32_t t = static_cast<int32_t>(bt / B);
    const int64_t b = bt % B;
    const int32_t D = D_offsets[t + 1] - D_offsets[t];
    const int64_t L = offsets[bt + 1] - offsets[bt];
    acc.assign(static_cast<size_t>(D), 0.0);
    for (int64_t i = offsets[bt]; i < offsets[bt + 1]; ++i) {
      double s = per_sample_weights ? static_cast<double>(per_sample_weights[i]) : 1.0;
      if (mean_pooling) s *= 1.0 / static_cast<double>(L);
      const int64_t row = weights_offsets[t] + indices[i] * D;
      for (int32_t d = 0; d < D; ++d) acc[d] += s * load_elem(weights, weight_dtype, row + d);
    }
    for (int32_t d = 0; d < D; ++d) store_elem(out, out_dtype, b * row_stride + D_offsets[t] + d, acc[d]);
  }
  return OK;
}

// ---- row-wise sharding with an exchange step.
// W ranks each own a contiguous row range of every table: rank r holds rows
// [row_bounds[t*(W+1) + r], row_bounds[t*(W+1) + r + 1]) of table t, the
// vocabulary sharding of "Function _embedding_bwd_kernel" (tinygrad: a device
// owns one slice of the rows, lookups outside it add nothing there). Under
// data-parallel batches every rank sends each of its lookups to the rank that
// owns its row (an all-to-all) and gathers the gradient rows of all ranks' bags
// (an all-gather); each owner then runs the backward on the lookups it received,
// the batches of all ranks side by side, and updates its rows only.

// Cyclic map (cyclic != 0): rank r owns the rows congruent to r modulo W of every
// table instead, local row = row / W (only row_bounds[t*(W+1) + W], the rows of
// table t, is read); a skewed id distribution then spreads over all ranks.
//
// The bucketing a rank does before the exchange: its batch (T tables x B bags,
// CSR offsets, table-major) split by owner. Owner r's part lists, bag by bag
// and in lookup order, the row relative to r's range and the lookup's scale:
// its per-sample weight (1 if none) and, under mean pooling, divided by the
// length L of its whole bag (both in fp32, one rounding, as the backward scales
// a lookup), so that the owner can run the weighted-sum backward on it.
//   send_offsets [W][T*B+1]: owner r's bag offsets, counted from its first lookup;
//   send_indices, send_scales [N]: owner 0's lookups first, then owner 1's, ...;
//   send_counts [W]: lookups per owner.
int oracle_bucketize(int32_t T, int32_t B, int32_t W, const int64_t* row_bounds, int32_t cyclic,
                     const int64_t* indices, const int64_t* offsets, int64_t N,
                     const float* per_sample_weights, int32_t mean_pooling,
                     int64_t* send_offsets, int64_t* send_indices, float* send_scales,
                     int64_t* send_counts) {
  if (T <= 0 || B <= 0 || W <= 0) return ERR_INVALID_ARG;
  const int64_t BT = static_cast<int64_t>(T) * B;
  for (int32_t t = 0; t < T; ++t) {
    const int64_t* rb = row_bounds + static_cast<int64_t>(t) * (W + 1);
    if (cyclic) {
      if (rb[W] <= 0) return ERR_INVALID_ARG;
      continue;
    }
    if (rb[0] != 0) return ERR_INVALID_ARG;
    for (int32_t r = 0; r < W; ++r)
      if (rb[r + 1] < rb[r]) return ERR_INVALID_ARG;
  }
  if (offsets[0] != 0 || offsets[BT] != N) return ERR_INVALID_ARG;
  for (int64_t bt = 0; bt < BT; ++bt)
    if (offsets[bt + 1] < offsets[bt]) return ERR_INVALID_ARG;
  std::vector<std::vector<int64_t>> idx(static_cast<size_t>(W));
  std::vector<std::vector<float>> scale(static_cast<size_t>(W));
  for (int32_t r = 0; r < W; ++r) send_offsets[static_cast<int64_t>(r) * (BT + 1)] = 0;
  for (int64_t bt = 0; bt < BT; ++bt) {
    const int32_t t = static_cast<int32_t>(bt / B);
    const int64_t* rb = row_bounds + static_cast<int64_t>(t) * (W + 1);
    const int64_t L = offsets[bt + 1] - offsets[bt];
    for (int64_t i = offsets[bt]; i < offsets[bt + 1]; ++i) {
      const int64_t row = indices[i];
      if (row < 0 || row >= rb[W]) return ERR_INDEX_OUT_OF_RANGE;
      int32_t r = 0;
      int64_t local = 0;
      if (cyclic) {
        r = static_cast<int32_t>(row % W);
        local = row / W;
      } else {
        while (!(row >= rb[r] && row < rb[r + 1])) ++r;  // empty ranges never match
        local = row - rb[r];
      }
      float s = per_sample_weights ? per_sample_weights[i] : 1.0f;
      // fp32 quotient, rounded once: the double quotient of two floats rounds to
      // the same fp32 value (53 >= 2 * 24 + 2 bits)
      if (mean_pooling) s = static_cast<float>(static_cast<double>(s) / static_cast<double>(static_cast<float>(L)));
      idx[r].push_back(local);
      scale[r].push_back(s);
    }
    for (int32_t r = 0; r < W; ++r)
      send_offsets[static_cast<int64_t>(r) * (BT + 1) + bt + 1] = static_cast<int64_t>(idx[r].size());
  }
  int64_t pos = 0;
  for (int32_t r = 0; r < W; ++r) {
    send_counts[r] = static_cast<int64_t>(idx[r].size());
    for (size_t k = 0; k < idx[r].size(); ++k, ++pos) {
      send_indices[pos] = idx[r][k];
      send_scales[pos] = scale[r][k];
    }
  }
  return OK;
}

// The owner's side after the exchange: the parts received from the W sources
// (source s's bag offsets recv_offsets[s][T*B+1], counted from its first lookup;
// the lookups of all sources concatenated in source order) laid out as one batch
// of W*B bags per table, table-major, bag s*B + b of table t holding source s's
// bag (t, b): the layout whose gradient rows are the sources' grad_output rows
// gathered in source order ([W*B, sum D]).
//   merged_offsets [T*W*B+1], merged_indices and merged_scales [sum of lookups].
int oracle_merge(int32_t T, int32_t B, int32_t W, const int64_t* recv_offsets,
                 const int64_t* recv_indices, const float* recv_scales,
                 int64_t* merged_offsets, int64_t* merged_indices, float* merged_scales) {
  if (T <= 0 || B <= 0 || W <= 0) return ERR_INVALID_ARG;
  const int64_t BT = static_cast<int64_t>(T) * B;
  std::vector<int64_t> first(static_cast<size_t>(W) + 1, 0);  // first lookup of each source
  for (int32_t s = 0; s < W; ++s) {
    const int64_t* off = recv_offsets + static_cast<int64_t>(s) * (BT + 1);
    if (off[0] != 0) return ERR_INVALID_ARG;
    for (int64_t bt = 0; bt < BT; ++bt)
      if (off[bt + 1] < off[bt]) return ERR_INVALID_ARG;
    first[s + 1] = first[s] + off[BT];
  }
  int64_t pos = 0;
  merged_offsets[0] = 0;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t s = 0; s < W; ++s)
      for (int32_t b = 0; b < B; ++b) {
        const int64_t* off = recv_offsets + static_cast<int64_t>(s) * (BT + 1);
        const int64_t bt = static_cast<int64_t>(t) * B + b;
        for (int64_t i = off[bt]; i < off[bt + 1]; ++i, ++pos) {
          merged_indices[pos] = recv_indices[first[s] + i];
          merged_scales[pos] = recv_scales[first[s] + i];
        }
        merged_offsets[(static_cast<int64_t>(t) * W + s) * B + b + 1] = pos;
      }
  return OK;
}

// Stochastic rounding pieces, exported for the pin tests.
void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}
uint16_t oracle_sr_bf16(float x, uint32_t r) { return sr_bf16(x, r); }
uint16_t oracle_sr_half(float x, uint32_t r) { return sr_half(x, r); }

// Storage conversions, exported for the pin tests.
uint16_t oracle_double_to_half(double x) { return double_to_half(x); }
double oracle_half_to_double(uint16_t h) { return half_to_double(h); }
uint16_t oracle_double_to_bf16(double x) { return double_to_bf16(x); }
double oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

}  // extern "C"
