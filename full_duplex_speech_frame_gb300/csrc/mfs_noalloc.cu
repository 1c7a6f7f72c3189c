// mfs_argmax_rows_noalloc: greedy argmax over rows of logits with no device
// allocation at all.  It is the frame step's argmax stage (per-block partial
// maxima in global scratch, reduced by the last block to finish) as a stand-alone
// kernel whose scratch is a fixed static device array of this file instead of
// memory from cudaMalloc.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "../../include/mfs.h"

namespace mfs {
void set_thread_error(const char* msg);  // defined with mfs_last_error
}

namespace {

constexpr int AM_THREADS = 256;
constexpr int AM_CHUNK = 4096;  // columns scanned by one block

struct AmScratch {
    unsigned int done[MFS_ARGMAX_MAX_ROWS];           // blocks finished, per row: must start at zero
    float part_val[MFS_ARGMAX_MAX_PARTIALS];           // per (row, block) maximum
    int part_idx[MFS_ARGMAX_MAX_PARTIALS];             // and its lowest column index
};
static_assert(sizeof(AmScratch) <= MFS_ARGMAX_SCRATCH_BYTES, "scratch layout exceeds its stated size");

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_argmax_scratch[MFS_ARGMAX_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
static void* g_scratch_addr[MAX_DEVICES];
static std::mutex g_scratch_mu;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void block_argmax(float& v, int& i, float* sv, int* si)
{
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sv[warp] = v; si[warp] = i; }
    __syncthreads();
    if (warp == 0) {
        v = lane < AM_THREADS / 32 ? sv[lane] : -INFINITY;
        i = lane < AM_THREADS / 32 ? si[lane] : 0x7fffffff;
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            if (better(ov, oi, v, i)) { v = ov; i = oi; }
        }
    }
}

// grid (nblk, rows).  Block b of row r scans columns [b * AM_CHUNK, ...) and
// leaves its partial in the scratch; the last block of the row to finish
// reduces the row's partials in block order and writes out[r].
__global__ void __launch_bounds__(AM_THREADS) argmax_rows_kernel(const float* __restrict__ logits, int cols,
                                                                 long long ld, int nblk, int* __restrict__ out,
                                                                 AmScratch* sc)
{
    __shared__ float sv[AM_THREADS / 32];
    __shared__ int si[AM_THREADS / 32];
    __shared__ int last;
    const int r = blockIdx.y, b = blockIdx.x;
    const float* row = logits + (long long)r * ld;
    const int c0 = b * AM_CHUNK, c1 = min(cols, c0 + AM_CHUNK);
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int c = c0 + threadIdx.x; c < c1; c += AM_THREADS) {
        const float x = __ldg(row + c);
        if (better(x, c, v, i)) { v = x; i = c; }
    }
    block_argmax(v, i, sv, si);
    if (threadIdx.x == 0) {
        const size_t k = (size_t)r * nblk + b;
        sc->part_val[k] = v;
        sc->part_idx[k] = i;
        __threadfence();
        last = atomicAdd(&sc->done[r], 1u) == (unsigned)(nblk - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    v = -INFINITY;
    i = 0x7fffffff;
    for (int k = threadIdx.x; k < nblk; k += AM_THREADS) {
        const float pv = __ldcg(sc->part_val + (size_t)r * nblk + k);
        const int pi = __ldcg(sc->part_idx + (size_t)r * nblk + k);
        if (better(pv, pi, v, i)) { v = pv; i = pi; }
    }
    block_argmax(v, i, sv, si);
    if (threadIdx.x == 0) {
        out[r] = i == 0x7fffffff ? 0 : i;  // a row with no comparable value (all NaN) gives 0
        sc->done[r] = 0;                    // leave the counter as the next call expects it
    }
}

int fail(int code, const char* msg)
{
    mfs::set_thread_error(msg);
    return code;
}

// The device address of the scratch array on the current device, looked up
// once per device (the array's name is only a stand-in in host code).
int scratch_address(int dev, void** addr)
{
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_argmax_scratch);
        if (e != cudaSuccess || !p) {
            char buf[160];
            snprintf(buf, sizeof buf, "cudaGetSymbolAddress of the argmax scratch failed: %s", cudaGetErrorString(e));
            return fail(MFS_E_CUDA, buf);
        }
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return MFS_OK;
}

}  // namespace

extern "C" int mfs_argmax_rows_noalloc(const float* logits, int rows, int cols, long long ld, int32_t* out,
                                       void* cuda_stream)
{
    if (rows < 0 || cols < 1 || ld < cols) return fail(MFS_E_ARG, "argmax: need rows >= 0, cols >= 1, ld >= cols");
    if (rows == 0) return MFS_OK;
    if (!logits || !out) return fail(MFS_E_ARG, "argmax: null logits or out");
    const long long nblk = (cols + (long long)AM_CHUNK - 1) / AM_CHUNK;
    if (rows > MFS_ARGMAX_MAX_ROWS || (long long)rows * nblk > MFS_ARGMAX_MAX_PARTIALS) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "argmax: %d rows x %lld column blocks of %d exceed the fixed scratch (at most %d rows and %d "
                 "row-blocks)", rows, nblk, AM_CHUNK, MFS_ARGMAX_MAX_ROWS, MFS_ARGMAX_MAX_PARTIALS);
        return fail(MFS_E_RANGE, buf);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return fail(MFS_E_CUDA, "argmax: no usable current CUDA device");
    void* addr = nullptr;
    const int rc = scratch_address(dev, &addr);
    if (rc != MFS_OK) return rc;
    AmScratch* sc = (AmScratch*)addr;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    // The row counters must start at zero.  Each call leaves them at zero, but a
    // call cut short by an earlier error may not have: clear them first.
    cudaError_t e = cudaMemsetAsync(sc->done, 0, (size_t)rows * sizeof(unsigned int), st);
    if (e == cudaSuccess) {
        argmax_rows_kernel<<<dim3((unsigned)nblk, (unsigned)rows), AM_THREADS, 0, st>>>(logits, cols, ld, (int)nblk,
                                                                                     out, sc);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        char buf[160];
        snprintf(buf, sizeof buf, "argmax launch failed: %s", cudaGetErrorString(e));
        return fail(MFS_E_CUDA, buf);
    }
    return MFS_OK;
}
