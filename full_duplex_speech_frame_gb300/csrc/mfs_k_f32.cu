// Kernel instantiations: fp32 weights and key/value ring, batch groups 1, 2, 4.
#include "mfs_kernels.cuh"

namespace mfs {
const void* kernel_f32_1() { return (const void*)&step_kernel<float, float, 1>; }
const void* kernel_f32_2() { return (const void*)&step_kernel<float, float, 2>; }
const void* kernel_f32_4() { return (const void*)&step_kernel<float, float, 4>; }
}  // namespace mfs
