// mfs_rvq_encode: the encoder-side argmin quantizer of Mimi's split residual
// vector quantizer, for a batch of frames.  Codebook 0 quantizes each frame's
// semantic latent; codebooks 1..7 quantize its acoustic latent and then the
// residual each stage leaves.  Nearest codeword by squared Euclidean distance,
// ties to the lower index.
//
// This file holds the CUDA-core form, used when D is not a multiple of 8 (the
// tensor-core form in mfs_rvq_mma.cu takes the rest).  One CTA takes up to 16
// frames and keeps their residuals in shared memory.
// Each thread owns codewords c, c + 256, ...: it streams a codeword row once
// (float4 loads, L1-resident while it is used) and accumulates its distance to
// every frame of the tile, whose residual chunks all threads read at the same
// address (a shared-memory broadcast).  A frame's argmin is reduced across the
// CTA in thread order, so the result is deterministic.
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include "../../include/mfs.h"

namespace mfs {
void set_thread_error(const char* msg);  // defined with mfs_last_error
int rvq_encode_mma(const float* z_sem, const float* z_ac, int T, int D, const float* codebooks, int Cb, int32_t* codes,
                   cudaStream_t st);  // the tensor-core form (mfs_rvq_mma.cu)
}

namespace {

constexpr int RV_THREADS = 256;
constexpr int RV_FT = 16;  // frames per CTA
constexpr int RV_WARPS = RV_THREADS / 32;

__device__ __forceinline__ bool rv_better(float d1, int i1, float d2, int i2)
{
    return d1 < d2 || (d1 == d2 && i1 < i2);
}

__global__ void __launch_bounds__(RV_THREADS, 2) rvq_kernel(const float* __restrict__ z_sem, const float* __restrict__ z_ac,
                                                            int T, int D, const float* __restrict__ cb, int Cb,
                                                            int* __restrict__ codes)
{
    extern __shared__ float4 rv_r[];  // [RV_FT][D / 4] residuals
    __shared__ float sbd[RV_WARPS][RV_FT];
    __shared__ int sbi[RV_WARPS][RV_FT];
    __shared__ int scode[RV_FT];
    const int D4 = D / 4;
    const int t0 = blockIdx.x * RV_FT;
    const int nf = min(RV_FT, T - t0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int q = 0; q < 8; ++q) {
        if (q <= 1) {
            const float4* z = reinterpret_cast<const float4*>(q == 0 ? z_sem : z_ac);
            for (int k = threadIdx.x; k < RV_FT * D4; k += RV_THREADS) {
                const int f = k / D4;
                rv_r[k] = f < nf ? __ldg(z + (size_t)(t0 + f) * D4 + k % D4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncthreads();
        }
        const float4* book = reinterpret_cast<const float4*>(cb + (size_t)q * Cb * D);
        float bd[RV_FT];
        int bi[RV_FT];
#pragma unroll
        for (int f = 0; f < RV_FT; ++f) {
            bd[f] = INFINITY;
            bi[f] = 0x7fffffff;
        }
        for (int c = threadIdx.x; c < Cb; c += RV_THREADS) {
            float acc[RV_FT];
#pragma unroll
            for (int f = 0; f < RV_FT; ++f) acc[f] = 0.f;
            const float4* row = book + (size_t)c * D4;
            for (int e = 0; e < D4; ++e) {
                const float4 w = __ldg(row + e);
#pragma unroll
                for (int f = 0; f < RV_FT; ++f) {
                    if (f < nf) {
                        const float4 x = rv_r[f * D4 + e];
                        const float a = x.x - w.x, b = x.y - w.y, cc = x.z - w.z, dd = x.w - w.w;
                        acc[f] = fmaf(a, a, acc[f]);
                        acc[f] = fmaf(b, b, acc[f]);
                        acc[f] = fmaf(cc, cc, acc[f]);
                        acc[f] = fmaf(dd, dd, acc[f]);
                    }
                }
            }
#pragma unroll
            for (int f = 0; f < RV_FT; ++f)
                if (rv_better(acc[f], c, bd[f], bi[f])) {
                    bd[f] = acc[f];
                    bi[f] = c;
                }
        }
        // argmin per frame: warps, then the CTA in warp order
#pragma unroll
        for (int f = 0; f < RV_FT; ++f) {
            float v = bd[f];
            int i = bi[f];
            for (int o = 16; o; o >>= 1) {
                const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
                const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
                if (rv_better(v2, i2, v, i)) {
                    v = v2;
                    i = i2;
                }
            }
            if (lane == 0) {
                sbd[warp][f] = v;
                sbi[warp][f] = i;
            }
        }
        __syncthreads();
        if (threadIdx.x < RV_FT) {
            const int f = threadIdx.x;
            float v = sbd[0][f];
            int i = sbi[0][f];
            for (int w = 1; w < RV_WARPS; ++w)
                if (rv_better(sbd[w][f], sbi[w][f], v, i)) {
                    v = sbd[w][f];
                    i = sbi[w][f];
                }
            scode[f] = i;
            if (f < nf) codes[(size_t)(t0 + f) * 8 + q] = i;
        }
        __syncthreads();
        if (q >= 1 && q < 7) {  // the residual for the next acoustic stage
            for (int k = threadIdx.x; k < nf * D4; k += RV_THREADS) {
                const int f = k / D4, e = k % D4;
                const int cw = scode[f] < Cb ? scode[f] : 0;  // no codeword chosen: NaN distances
                const float4 w = __ldg(book + (size_t)cw * D4 + e);
                float4 x = rv_r[k];
                x.x -= w.x;
                x.y -= w.y;
                x.z -= w.z;
                x.w -= w.w;
                rv_r[k] = x;
            }
            __syncthreads();
        }
    }
}

int fail(int code, const char* msg)
{
    mfs::set_thread_error(msg);
    return code;
}

}  // namespace

extern "C" int mfs_rvq_encode(const float* z_sem, const float* z_ac, int T, int D, const float* codebooks, int Cb,
                              int32_t* codes, void* cuda_stream)
{
    if (T < 0 || D < 4 || D % 4 != 0 || D > MFS_RVQ_MAX_DIM || Cb < 1)
        return fail(MFS_E_ARG, "rvq: need T >= 0, D a multiple of 4 in [4, 1024], Cb >= 1");
    if (T == 0) return MFS_OK;
    if (!z_sem || !z_ac || !codebooks || !codes) return fail(MFS_E_ARG, "rvq: null pointer");
    if (((uintptr_t)z_sem | (uintptr_t)z_ac | (uintptr_t)codebooks) & 15u)
        return fail(MFS_E_ARG, "rvq: latents and codebooks must be 16-byte aligned");
    if (D % 8 == 0 && Cb < (1 << 24))
        return mfs::rvq_encode_mma(z_sem, z_ac, T, D, codebooks, Cb, codes, (cudaStream_t)cuda_stream);
    const size_t smem = (size_t)RV_FT * D * sizeof(float);
    if (smem > 48 * 1024) {  // the residual tile needs more than the default shared memory
        const cudaError_t a = cudaFuncSetAttribute(rvq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (a != cudaSuccess) return fail(MFS_E_CUDA, "rvq: cannot raise the shared memory limit");
    }
    const int grid = (T + RV_FT - 1) / RV_FT;
    rvq_kernel<<<grid, RV_THREADS, smem, (cudaStream_t)cuda_stream>>>(z_sem, z_ac, T, D, codebooks, Cb, codes);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char buf[160];
        snprintf(buf, sizeof buf, "rvq launch failed: %s", cudaGetErrorString(e));
        return fail(MFS_E_CUDA, buf);
    }
    return MFS_OK;
}
