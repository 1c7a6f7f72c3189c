// Kernel instantiation: bf16 weights and key/value ring, tensor-core weight pass (5..32 slots).
#include "mfs_kernels.cuh"

namespace mfs {
const void* kernel_bf16_mma() { return (const void*)&step_kernel<__nv_bfloat16, __nv_bfloat16, BG_MMA>; }
}  // namespace mfs
