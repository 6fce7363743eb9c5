// Instantiations of the fused reduce + optimizer kernel for __half weights
// (split per weight type so the kernel variants compile in parallel).
#include "reduce.cuh"

namespace embbwd {

const void* reduce_kernel_f16(const ReduceKey& k) { return pick_reduce<__half>(k); }

}  // namespace embbwd
