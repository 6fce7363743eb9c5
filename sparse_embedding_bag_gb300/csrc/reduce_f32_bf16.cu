// Instantiations of the fused reduce + optimizer kernel for float weights and
// __nv_bfloat16 gradients (one file per type pair so the variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_f32_bf16(const ReduceKey& k) { return pick_reduce<float, __nv_bfloat16>(k); }

}  // namespace embbwd
