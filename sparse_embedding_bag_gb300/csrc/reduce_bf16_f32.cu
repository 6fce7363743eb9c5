// Instantiations of the fused reduce + optimizer kernel for __nv_bfloat16 weights and
// float gradients (one file per type pair so the variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_bf16_f32(const ReduceKey& k) { return pick_reduce<__nv_bfloat16, float>(k); }

}  // namespace embbwd
