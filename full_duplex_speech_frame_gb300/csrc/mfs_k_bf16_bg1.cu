// Kernel instantiation: bf16 weights and key/value ring, batch group of 1.
#include "mfs_kernels.cuh"

namespace mfs {
const void* kernel_bf16_1() { return (const void*)&step_kernel<__nv_bfloat16, __nv_bfloat16, 1>; }
}  // namespace mfs
