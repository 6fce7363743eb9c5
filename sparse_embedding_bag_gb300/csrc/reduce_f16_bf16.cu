// Instantiations of the fused reduce + optimizer kernel for __half weights and
// __nv_bfloat16 gradients (one file per type pair so the variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_f16_bf16(const ReduceKey& k) { return pick_reduce<__half, __nv_bfloat16>(k); }

}  // namespace embbwd
