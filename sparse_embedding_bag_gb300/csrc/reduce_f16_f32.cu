// Instantiations of the fused reduce + optimizer kernel for __half weights and
// float gradients (one file per type pair so the variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_f16_f32(const ReduceKey& k) { return pick_reduce<__half, float>(k); }

}  // namespace embbwd
