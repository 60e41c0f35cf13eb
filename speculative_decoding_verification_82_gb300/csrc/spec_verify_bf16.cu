// bf16 instantiations of the verification kernels.
#include "verify_kernel.cuh"
template cudaError_t specv::launch_verify<__nv_bfloat16>(int, const specv::Params&, const specv::LaunchPlan&, cudaStream_t);
