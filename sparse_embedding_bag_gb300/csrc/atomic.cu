// Unpooled backward + SGD by atomic scatter: every lookup l adds -lr * g_l to
// its row with vector float atomics, without sorting. Same operation as
// "tinygrad/nn/__init__.py" _embedding_bwd_kernel (a relaxed atomic add per
// element into the row the token indexed) and "tt_embeddings_cuda.cu"
// cache_backward_sgd_kernel (w -= lr * g by atomics), here one 16-byte
// red.global.add.v4.f32 per 4 elements. The order of the adds is not fixed, so
// the result is not bitwise reproducible; fp32 weights only.
//
// Before this kernel runs, k_hist (with no radix passes) checks every index
// against its table and the CSR offsets; on failure nothing is written.
#include "decode.cuh"

namespace embbwd {

namespace {

constexpr int kAtomicTile = 64;  // lookups per block

template <typename grad_t>
__global__ void __launch_bounds__(kThreads) k_nobag_atomic(AtomicArgs a) {
  __shared__ uint32_t s_bag[kAtomicTile];
  __shared__ int64_t s_off[2 * kAtomicTile];
  pdl_wait();
  pdl_trigger();
  if (*(volatile uint32_t*)&a.ctl->err) return;
  const DecodeArgs& d = a.d;
  const int64_t i0 = (int64_t)blockIdx.x * kAtomicTile;
  const int64_t i1 = min(i0 + kAtomicTile, d.N);
  if (d.T > 1) expand_tile_bags(d, i0, i1, s_bag, nullptr, s_off, 2 * kAtomicTile);
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t nvec = a.D >> 2;
  const grad_t* grad = static_cast<const grad_t*>(a.grad);
  for (int64_t l = i0 + warp; l < i1; l += kWarps) {
    uint32_t t = 0;
    if (d.T > 1) {
      t = div_by_B(s_bag[l - i0], d.B, d.invB);
      if (t >= d.T) t = d.T - 1;
    }
    const int64_t idx = d.indices[l];
    float* row = a.weights + __ldg(&a.weights_offsets[t]) + idx * (int64_t)a.D;
    const grad_t* g = grad + l * (int64_t)a.D;
    for (uint32_t u = lane; u < nvec; u += 32) {
      const float4 x = Vec4<grad_t>::load(g + (int64_t)u * 4);
      atomicAdd(reinterpret_cast<float4*>(row + (int64_t)u * 4),
                make_float4(-a.lr * x.x, -a.lr * x.y, -a.lr * x.z, -a.lr * x.w));
    }
  }
}

}  // namespace

cudaError_t atomic_configure() { return cudaSuccess; }

cudaError_t launch_nobag_atomic(const AtomicArgs& a, int grad_dtype, int T, cudaStream_t s, bool pdl) {
  (void)T;
  const unsigned grid = (unsigned)((a.d.N + kAtomicTile - 1) / kAtomicTile);
  AtomicArgs arg = a;
  void* args[] = {&arg};
  const void* fn = grad_dtype == 0   ? reinterpret_cast<const void*>(&k_nobag_atomic<float>)
                   : grad_dtype == 1 ? reinterpret_cast<const void*>(&k_nobag_atomic<__half>)
                                     : reinterpret_cast<const void*>(&k_nobag_atomic<__nv_bfloat16>);
  return launch_kernel(fn, dim3(grid), dim3(kThreads), 0, s, args, pdl);
}

}  // namespace embbwd
