// bf16 instantiations of the direct-load reduce-scatter / allreduce kernels
// (fp32 accumulation, one round-to-nearest-even cast on output).
#include "reduce_kernels.cuh"

VCOLL_DEFINE_REDUCE_TABLE(__nv_bfloat16, reduce_kernel_bf16)
