// fp32 instantiations of the direct-load reduce-scatter / allreduce kernels.
#include "reduce_kernels.cuh"

VCOLL_DEFINE_REDUCE_TABLE(float, reduce_kernel_f32)
