// Instantiations of the fused reduce + optimizer kernel for __nv_bfloat16 weights
// (split per weight type so the kernel variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_bf16(const ReduceKey& k) { return pick_reduce<__nv_bfloat16>(k); }

}  // namespace embbwd
