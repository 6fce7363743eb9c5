// Instantiations of the fused reduce + optimizer kernel for float weights
// (split per weight type so the kernel variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_f32(const ReduceKey& k) { return pick_reduce<float>(k); }

}  // namespace embbwd
