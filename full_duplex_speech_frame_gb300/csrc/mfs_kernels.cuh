// Device code of the lockstep frame step.
//
// One persistent cooperative kernel runs every phase of a step (embedding sum,
// 32 temporal layers, text head, 16 depformer substeps, write-back) with a
// grid-wide barrier between phases; the same kernel can also be launched once
// per phase (no barriers) for diagnosis.  One CTA per SM, 16 warps.
//
// Matrix-vector phases stream bf16 (or fp32) weight rows with 128-bit
// non-allocating loads.  A CTA owns a contiguous block of row pairs; its 16
// warps split K into contiguous slices so that each warp keeps its slice of
// the (normalised) activations in registers for the whole phase.  Partial dot
// products are reduced lane-wise with a fixed shuffle tree, then across the
// K-slices in slice order: the arithmetic of one slot never depends on the
// other slots of the batch, on the batch size or on the CTA that owns a row.
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "mfs_internal.h"

namespace mfs {
namespace {  // internal linkage: every kernel translation unit has its own copy

// ------------------------------------------------------------------ memory

__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// L2-only load for data written by other CTAs during the same launch.
__device__ __forceinline__ uint4 ld_cg16(const void* p)
{
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
    return r;
}

__device__ __forceinline__ int ld_cg_int(const int* p) { return __ldcg(p); }
__device__ __forceinline__ float ld_cg_f(const float* p) { return __ldcg(p); }

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// A "vector" is 8 consecutive weights.
template <typename TW>
struct WV;

template <>
struct WV<__nv_bfloat16> {
    struct raw { uint4 a; };
    static __device__ __forceinline__ raw load(const __nv_bfloat16* p) { return {ld_stream16(p)}; }
    static __device__ __forceinline__ raw zero() { return {make_uint4(0u, 0u, 0u, 0u)}; }
    static __device__ __forceinline__ void cvt(const raw& r, float f[8])
    {
        f[0] = bf_lo(r.a.x); f[1] = bf_hi(r.a.x); f[2] = bf_lo(r.a.y); f[3] = bf_hi(r.a.y);
        f[4] = bf_lo(r.a.z); f[5] = bf_hi(r.a.z); f[6] = bf_lo(r.a.w); f[7] = bf_hi(r.a.w);
    }
    static __device__ __forceinline__ float at(const void* base, long long i)
    {
        return __uint_as_float((uint32_t)((const unsigned short*)base)[i] << 16);
    }
};

template <>
struct WV<float> {
    struct raw { uint4 a, b; };
    static __device__ __forceinline__ raw load(const float* p) { return {ld_stream16(p), ld_stream16(p + 4)}; }
    static __device__ __forceinline__ raw zero() { return {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)}; }
    static __device__ __forceinline__ void cvt(const raw& r, float f[8])
    {
        f[0] = __uint_as_float(r.a.x); f[1] = __uint_as_float(r.a.y);
        f[2] = __uint_as_float(r.a.z); f[3] = __uint_as_float(r.a.w);
        f[4] = __uint_as_float(r.b.x); f[5] = __uint_as_float(r.b.y);
        f[6] = __uint_as_float(r.b.z); f[7] = __uint_as_float(r.b.w);
    }
    static __device__ __forceinline__ float at(const void* base, long long i) { return ((const float*)base)[i]; }
};

// Key/value ring element type.
template <typename TKV>
struct KV;

template <>
struct KV<__nv_bfloat16> {
    static __device__ __forceinline__ void store2(void* base, long long i, float a, float b)
    {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        *reinterpret_cast<__nv_bfloat162*>((__nv_bfloat16*)base + i) = v;
    }
    static __device__ __forceinline__ void load8(const void* base, long long i, float f[8])
    {
        uint4 r = ld_cg16((const __nv_bfloat16*)base + i);
        f[0] = bf_lo(r.x); f[1] = bf_hi(r.x); f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
        f[4] = bf_lo(r.z); f[5] = bf_hi(r.z); f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
    }
};

template <>
struct KV<float> {
    static __device__ __forceinline__ void store2(void* base, long long i, float a, float b)
    {
        *reinterpret_cast<float2*>((float*)base + i) = make_float2(a, b);
    }
    static __device__ __forceinline__ void load8(const void* base, long long i, float f[8])
    {
        uint4 r0 = ld_cg16((const float*)base + i), r1 = ld_cg16((const float*)base + i + 4);
        f[0] = __uint_as_float(r0.x); f[1] = __uint_as_float(r0.y); f[2] = __uint_as_float(r0.z); f[3] = __uint_as_float(r0.w);
        f[4] = __uint_as_float(r1.x); f[5] = __uint_as_float(r1.y); f[6] = __uint_as_float(r1.z); f[7] = __uint_as_float(r1.w);
    }
};

// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// argmax order: larger value wins, lower index on ties (NaN never wins)
__device__ __forceinline__ bool am_better(float v1, int i1, float v2, int i2)
{
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (am_better(v2, i2, v, i)) { v = v2; i = i2; }
    }
}

// Sum over the block, same bits in every thread (fixed order).  scratch >= NWARP floats.
__device__ __forceinline__ float block_sum(float v, float* scratch)
{
    v = warp_sum(v);
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < NWARP; ++k) t += scratch[k];
    return t;
}

// ------------------------------------------------------------------ grid barrier

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// All CTAs arrive; returns false (and leaves the error flag set) if the wait
// gave up after 2 s or another CTA reported an error.
__device__ bool grid_barrier(unsigned* bar, unsigned target, int* err)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(bar, 1u);
        int ok = 1;
        const unsigned long long t0 = globaltimer_ns();
        unsigned spins = 0;
        while (ld_acquire_u32(bar) < target) {
            if ((++spins & 63u) == 0u) {
                if (*(volatile int*)err != 0) { ok = 0; break; }
                if (globaltimer_ns() - t0 > 2000000000ull) {
                    atomicCAS(err, 0, (int)DERR_BARRIER);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ------------------------------------------------------------------ shared memory map

struct Smem {
    float* red;    // [maxrows][BG][16]  per-K-slice partial sums
    float* yf;     // [maxrows][BG]      final row values of the CTA
    float* r;      // [BG] RMSNorm factors
    int* prev;     // [BG] depformer input token per batch row
    float* sred;   // [NWARP * 4] block-reduction scratch
    float* amv;    // [NWARP]
    int* ami;      // [NWARP]
    int* X;        // [MFS_MAX_SLOTS][17] embedding rows of this step
    int* att;      // [MFS_MAX_SLOTS][4]  len, chunks, prefix, pad
};

constexpr int SCRATCH_FLOATS = 4096;

__device__ __forceinline__ Smem smem_map(float* base, int maxrows, int BG)
{
    Smem s;
    s.red = base;
    s.yf = s.red + (size_t)maxrows * BG * 16;
    float* sc = s.yf + (size_t)maxrows * BG;
    s.r = sc;
    s.prev = (int*)(sc + 16);
    s.sred = sc + 64;
    s.amv = sc + 128;
    s.ami = (int*)(sc + 160);
    s.X = (int*)(sc + 256);
    s.att = (int*)(sc + 256 + MFS_MAX_SLOTS * NSTREAM);
    return s;
}

// ------------------------------------------------------------------ GEMV engine

struct GemvCfg {
    int nwk, nwr, nvw, vpl;
};

// K-slices per row: the largest power of two <= 16 that leaves >= 32 vectors
// (of 8 weights) per slice.
__device__ __forceinline__ GemvCfg gemv_cfg(int K)
{
    const int NV = K / 8;
    int nwk = 16;
    while (nwk > 1 && NV / nwk < 32) nwk >>= 1;
    GemvCfg c;
    c.nwk = nwk;
    c.nwr = NWARP / nwk;
    c.nvw = (NV + nwk - 1) / nwk;
    c.vpl = (c.nvw + 31) / 32;
    return c;
}

// Where the input vector of a matrix-vector phase comes from.
struct XSrc {
    const float* base;    // batch row i at base + i * stride
    long long stride;
    const float* g;       // RMSNorm gain, or nullptr for no norm
    const void* add;      // depformer embedding table (weight dtype) or nullptr
    long long add_stride; // row length of that table (elements)
    float* store;         // CTA 0 stores base + add here (depformer residual), or nullptr
};

template <typename TW, int VPL, int BGV, int UP>
__device__ __forceinline__ void gemv_rows(const TW* __restrict__ W, int K, const GemvCfg& c, int kw, int rw,
                                          int lane, int pair_lo, int pair_hi, const float (&xr)[VPL][BGV][8],
                                          float* red)
{
    using V = WV<TW>;
    const int NV = K / 8;
    const int v_begin = kw * c.nvw;
    const int v_end = min(NV, v_begin + c.nvw);
    for (int pp0 = pair_lo + rw; pp0 < pair_hi; pp0 += c.nwr * UP) {
        typename V::raw wv[UP][2][VPL];
#pragma unroll
        for (int u = 0; u < UP; ++u) {
            const int pp = pp0 + u * c.nwr;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const TW* row = W + (size_t)(2 * pp + h) * (size_t)K;
#pragma unroll
                for (int t = 0; t < VPL; ++t) {
                    const int v = v_begin + lane + 32 * t;
                    wv[u][h][t] = (pp < pair_hi && v < v_end) ? V::load(row + (size_t)v * 8) : V::zero();
                }
            }
        }
        float acc[UP][2][BGV];
#pragma unroll
        for (int u = 0; u < UP; ++u)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int b = 0; b < BGV; ++b) acc[u][h][b] = 0.f;
#pragma unroll
        for (int u = 0; u < UP; ++u)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int t = 0; t < VPL; ++t) {
                    float f[8];
                    V::cvt(wv[u][h][t], f);
#pragma unroll
                    for (int b = 0; b < BGV; ++b)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[u][h][b] = fmaf(f[e], xr[t][b][e], acc[u][h][b]);
                }
#pragma unroll
        for (int u = 0; u < UP; ++u) {
            const int pp = pp0 + u * c.nwr;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int b = 0; b < BGV; ++b) {
                    const float s = warp_sum(acc[u][h][b]);
                    if (lane == 0 && pp < pair_hi)
                        red[((size_t)((pp - pair_lo) * 2 + h) * BGV + b) * 16 + kw] = s;
                }
        }
    }
}

// Runs one batch group [b0, b0+nb) of a matrix-vector phase and leaves the
// CTA's row results in sm.yf[row_local][b] (layout stride BGV).
template <typename TW, int VPL, int BGV, int UP>
__device__ void gemv_group(const Params& P, const TW* __restrict__ W, int K, const GemvCfg& c, int pair_lo,
                           int pair_hi, const XSrc& xs, int b0, int nb, const Smem& sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kw = warp % c.nwk, rw = warp / c.nwk;
    const TW* add_rows[BGV];
#pragma unroll
    for (int b = 0; b < BGV; ++b)
        add_rows[b] = (xs.add && b < nb) ? (const TW*)xs.add + (size_t)sm.prev[b] * (size_t)xs.add_stride : nullptr;

    // RMSNorm factors (every CTA computes the same bits)
    if (xs.g) {
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            if (b >= nb) break;
            const float* xb = xs.base + (size_t)(b0 + b) * xs.stride;
            float ss = 0.f;
            for (int k = tid; k < K; k += NT) {
                float v = ld_cg_f(xb + k);
                if (add_rows[b]) v += WV<TW>::at(add_rows[b], k);
                ss = fmaf(v, v, ss);
            }
            const float tot = block_sum(ss, sm.sred);
            if (tid == 0) sm.r[b] = rsqrtf(tot / (float)K + P.eps);
        }
        __syncthreads();
    }
    // the depformer residual u = in-projection + embedding, written once
    if (xs.store && blockIdx.x == 0) {
        for (int b = 0; b < nb; ++b) {
            const float* xb = xs.base + (size_t)(b0 + b) * xs.stride;
            float* ub = xs.store + (size_t)(b0 + b) * K;
            for (int k = tid; k < K; k += NT) {
                float v = ld_cg_f(xb + k);
                if (add_rows[b]) v += WV<TW>::at(add_rows[b], k);
                ub[k] = v;
            }
        }
    }
    // this warp's K-slice of the input, normalised, in registers
    float xr[VPL][BGV][8];
    const int NV = K / 8;
    const int v_begin = kw * c.nvw;
    const int v_end = min(NV, v_begin + c.nvw);
#pragma unroll
    for (int t = 0; t < VPL; ++t) {
        const int v = v_begin + lane + 32 * t;
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            const bool ok = v < v_end && b < nb;
            float rb = 1.f;
            if (xs.g && ok) rb = sm.r[b];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float val = 0.f;
                if (ok) {
                    const int k = v * 8 + e;
                    val = ld_cg_f(xs.base + (size_t)(b0 + b) * xs.stride + k);
                    if (add_rows[b]) val += WV<TW>::at(add_rows[b], k);
                    if (xs.g) val = val * rb * xs.g[k];
                }
                xr[t][b][e] = val;
            }
        }
    }
    gemv_rows<TW, VPL, BGV, UP>(W, K, c, kw, rw, lane, pair_lo, pair_hi, xr, sm.red);
    __syncthreads();
    // sum the K-slices in slice order
    const int rows = (pair_hi - pair_lo) * 2;
    for (int it = tid; it < rows * nb; it += NT) {
        const int r = it / nb, b = it % nb;
        const float* rp = sm.red + ((size_t)r * BGV + b) * 16;
        float y = 0.f;
        for (int k = 0; k < c.nwk; ++k) y += rp[k];
        sm.yf[(size_t)r * BGV + b] = y;
    }
    __syncthreads();
}

// ------------------------------------------------------------------ epilogues

// Each epilogue sees the CTA's rows [2*pair_lo, 2*pair_hi) for batch rows
// b0..b0+nb-1, values in sm.yf[(row - 2*pair_lo) * bgv + b].

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

template <typename TKV>
__device__ void epi_qkv(const Params& P, int l, int pair_lo, int pair_hi, int b0, int nb, int bgv, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int d = P.d, hd = P.hd;
    const int npair = pair_hi - pair_lo;
    for (int it = threadIdx.x; it < npair * nb; it += NT) {
        const int pl = it / nb, b = it % nb;
        const int i = b0 + b;
        const int r = 2 * (pair_lo + pl);
        float y0 = sm.yf[(size_t)(2 * pl) * bgv + b], y1 = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
        const int part = r / d, e = r - part * d;
        const int p = D->pos[i];
        if (part < 2) {
            const float2 cs = P.rope[(size_t)p * (hd / 2) + (e % hd) / 2];
            const float a = y0, c = y1;
            y0 = a * cs.x - c * cs.y;
            y1 = a * cs.y + c * cs.x;
        }
        if (part == 0) {
            P.q[(size_t)i * d + e] = y0;
            P.q[(size_t)i * d + e + 1] = y1;
        } else {
            const int slot = D->slot[i];
            const long long idx = (((long long)slot * P.L + l) * P.W + (p % P.W)) * (long long)d + e;
            KV<TKV>::store2(part == 1 ? P.kc : P.vc, idx, y0, y1);
        }
    }
}

__device__ void epi_resid(float* dst, long long stride, int pair_lo, int pair_hi, int b0, int nb, int bgv,
                          const Smem& sm)
{
    const int npair = pair_hi - pair_lo;
    for (int it = threadIdx.x; it < npair * nb; it += NT) {
        const int pl = it / nb, b = it % nb;
        float* row = dst + (size_t)(b0 + b) * stride + 2 * (pair_lo + pl);
        row[0] += sm.yf[(size_t)(2 * pl) * bgv + b];
        row[1] += sm.yf[(size_t)(2 * pl + 1) * bgv + b];
    }
}

// rows are (gate m, up m) pairs
__device__ void epi_swiglu(float* dst, long long stride, int pair_lo, int pair_hi, int b0, int nb, int bgv,
                           const Smem& sm)
{
    const int npair = pair_hi - pair_lo;
    for (int it = threadIdx.x; it < npair * nb; it += NT) {
        const int pl = it / nb, b = it % nb;
        const float g = sm.yf[(size_t)(2 * pl) * bgv + b], u = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
        dst[(size_t)(b0 + b) * stride + pair_lo + pl] = silu(g) * u;
    }
}

// Rows [0, nlog) are logits (stored, and the CTA's argmax per batch row goes
// to amax_*[i][cta]); rows >= nlog go to extra[i][row - nlog] (may be null).
__device__ void epi_logits(const Params& P, float* lg, long long lg_stride, int nlog, float* extra,
                           long long extra_stride, int pair_lo, int pair_hi, int b0, int nb, int bgv,
                           const Smem& sm)
{
    const int npair = pair_hi - pair_lo;
    const int rows = 2 * npair, r0 = 2 * pair_lo;
    for (int it = threadIdx.x; it < rows * nb; it += NT) {
        const int rl = it / nb, b = it % nb;
        const int r = r0 + rl;
        const float y = sm.yf[(size_t)rl * bgv + b];
        if (r < nlog) lg[(size_t)(b0 + b) * lg_stride + r] = y;
        else if (extra) extra[(size_t)(b0 + b) * extra_stride + (r - nlog)] = y;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int b = 0; b < nb; ++b) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int rl = threadIdx.x; rl < rows; rl += NT) {
            const int r = r0 + rl;
            if (r >= nlog) break;
            const float y = sm.yf[(size_t)rl * bgv + b];
            if (am_better(y, r, bv, bi)) { bv = y; bi = r; }
        }
        warp_argmax(bv, bi);
        __syncthreads();
        if (lane == 0) { sm.amv[warp] = bv; sm.ami[warp] = bi; }
        __syncthreads();
        if (threadIdx.x == 0) {
            float v = sm.amv[0];
            int ix = sm.ami[0];
            for (int k = 1; k < NWARP; ++k)
                if (am_better(sm.amv[k], sm.ami[k], v, ix)) { v = sm.amv[k]; ix = sm.ami[k]; }
            P.amax_v[(size_t)(b0 + b) * P.G + blockIdx.x] = v;
            P.amax_i[(size_t)(b0 + b) * P.G + blockIdx.x] = ix;
        }
    }
}

// Reduce the per-CTA argmax partials of batch row i with one warp (every lane
// gets the same result; the tie rule makes the combine order irrelevant).
__device__ __forceinline__ int argmax_partials_warp(const Params& P, int i)
{
    const int lane = threadIdx.x & 31;
    float v = -INFINITY;
    int ix = 0x7fffffff;
    for (int c = lane; c < P.G; c += 32) {
        const float v2 = ld_cg_f(P.amax_v + (size_t)i * P.G + c);
        const int i2 = ld_cg_int(P.amax_i + (size_t)i * P.G + c);
        if (am_better(v2, i2, v, ix)) { v = v2; ix = i2; }
    }
    warp_argmax(v, ix);
    return ix == 0x7fffffff ? 0 : ix;
}

// ------------------------------------------------------------------ GEMV phase driver

// Picks, for depformer substep j, each batch row's input token (the text token
// for j = 0, else the code chosen for stream j), from the previous head's
// argmax partials unless the token was supplied.  CTA 0 records it.
__device__ void dep_select_inputs(const Params& P, int j, int b0, int nb, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < nb) {
        const int i = b0 + warp;
        const int a = argmax_partials_warp(P, i);
        int chosen;
        if (j == 0) {
            const int forced = D->codes[i][0];
            chosen = forced >= 0 ? forced : a;
            if (blockIdx.x == 0 && lane == 0) { P.text_argmax[i] = a; P.chosen[i * NSTREAM + 0] = chosen; }
        } else {
            const int p = D->pos[i], f = p - P.delays[j];
            const int forced =
                f >= 0 ? ld_cg_int(P.hist + ((size_t)D->slot[i] * NSTREAM + j) * HIST + f % HIST) : -1;
            chosen = forced >= 0 ? forced : a;
            if (blockIdx.x == 0 && lane == 0) { P.code_argmax[i * 16 + (j - 1)] = a; P.chosen[i * NSTREAM + j] = chosen; }
        }
        const int lim = j == 0 ? P.V : P.C;
        if (lane == 0) sm.prev[warp] = (chosen >= 0 && chosen < lim) ? chosen : 0;  // keeps the embedding read in range
    }
    __syncthreads();
}

// One matrix-vector phase: rows [0, N) of W [N][K] times the input vector of
// each batch row; epi(pair_lo, pair_hi, b0, nb, bgv) consumes the CTA's rows.
// dep_j >= 0 selects the depformer layer-0 input tokens first.
template <typename TW, int BG, class Epi>
__device__ void gemv_phase(const Params& P, const TW* W, int N, int K, const XSrc& xs, int dep_j, int n,
                           const Smem& sm, Epi epi)
{
    const int npairs = N / 2;
    const int pair_lo = (int)((long long)npairs * blockIdx.x / P.G);
    const int pair_hi = (int)((long long)npairs * (blockIdx.x + 1) / P.G);
    const GemvCfg c = gemv_cfg(K);
    const int bgv = c.vpl == 3 ? (BG < 2 ? BG : 2) : BG;
    for (int b0 = 0; b0 < n; b0 += bgv) {
        const int nb = min(bgv, n - b0);
        if (dep_j >= 0) dep_select_inputs(P, dep_j, b0, nb, sm);
        if (pair_hi > pair_lo || xs.store) {
            switch (c.vpl) {
                case 1: gemv_group<TW, 1, BG, 4>(P, W, K, c, pair_lo, pair_hi, xs, b0, nb, sm); break;
                case 2: gemv_group<TW, 2, BG, 2>(P, W, K, c, pair_lo, pair_hi, xs, b0, nb, sm); break;
                default: gemv_group<TW, 3, (BG < 2 ? BG : 2), 2>(P, W, K, c, pair_lo, pair_hi, xs, b0, nb, sm); break;
            }
        }
        epi(pair_lo, pair_hi, b0, nb, bgv);
        __syncthreads();
    }
}

// ------------------------------------------------------------------ S0 + S1

template <typename TW>
__device__ void phase_embed(const Params& P, int n, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int d = P.d;
    // embedding rows read by each stream: token of frame p-1-delay[k], or INIT
    for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
        const int i = it / NSTREAM, k = it % NSTREAM;
        const int f = D->pos[i] - 1 - P.delays[k];
        const int init = k == 0 ? P.V : P.C;
        int tok = f < 0 ? init : ld_cg_int(P.hist + ((size_t)D->slot[i] * NSTREAM + k) * HIST + f % HIST);
        if (tok < 0 || tok > init) tok = init;  // never taken for a consistent history; keeps reads in the table
        sm.X[it] = tok;
    }
    __syncthreads();
    // frame p's tokens into the history (column p mod 3, disjoint from the reads above)
    if (blockIdx.x == 0) {
        for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
            const int i = it / NSTREAM, k = it % NSTREAM;
            P.hist[((size_t)D->slot[i] * NSTREAM + k) * HIST + D->pos[i] % HIST] = D->codes[i][k];
        }
    }
    // x[i] = sum over streams in stream order
    const int per = d / 8;
    for (int it = blockIdx.x * NT + threadIdx.x; it < n * per; it += P.G * NT) {
        const int i = it / per, e0 = (it % per) * 8;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int k = 0; k < NSTREAM; ++k) {
            const int tok = sm.X[i * NSTREAM + k];
            const TW* row = k == 0 ? (const TW*)P.emb_text + (size_t)tok * d
                                   : (const TW*)P.emb_audio + ((size_t)(k - 1) * (P.C + 1) + tok) * d;
            float f[8];
            WV<TW>::cvt(WV<TW>::load(row + e0), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += f[e];
        }
        float4* dst = reinterpret_cast<float4*>(P.x + (size_t)i * d + e0);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// ------------------------------------------------------------------ S5 attention

// Chunks of the window of a slot of window length len: depends on len only.
__device__ __forceinline__ int attn_chunks(int len)
{
    const int c = (len + 15) / 16;
    return c < NCHUNK_MAX ? c : NCHUNK_MAX;
}

template <typename TKV>
__device__ void phase_attn(const Params& P, int l, int n, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int H = P.H, hd = P.hd, d = P.d, W = P.W;
    if (threadIdx.x == 0) {
        int pref = 0;
        for (int i = 0; i < n; ++i) {
            const int p = D->pos[i];
            const int len = p + 1 < W ? p + 1 : W;
            const int nc = attn_chunks(len);
            sm.att[i * 4 + 0] = len;
            sm.att[i * 4 + 1] = nc;
            sm.att[i * 4 + 2] = pref;
            pref += nc * H;
        }
        sm.att[n * 4 + 2] = pref;
    }
    __syncthreads();
    const int total = sm.att[n * 4 + 2];
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * NWARP + (threadIdx.x >> 5);
    const int LPP = hd / 8;            // lanes per key
    const int PPI = 32 / LPP;          // keys per warp iteration
    const int grp = lane / LPP, gl = lane % LPP;
    const float scale = rsqrtf((float)hd);
    const int pstride = hd + 4;
    for (int item = gwarp; item < total; item += P.G * NWARP) {
        int i = 0;
        while (i + 1 < n && sm.att[(i + 1) * 4 + 2] <= item) ++i;
        const int len = sm.att[i * 4 + 0], nc = sm.att[i * 4 + 1];
        const int rem = item - sm.att[i * 4 + 2];
        const int h = rem / nc, c = rem % nc;
        const int p = D->pos[i], slot = D->slot[i];
        const int CH = (len + nc - 1) / nc;
        const int j0 = c * CH, j1 = min(len, j0 + CH);
        const int start = p - len + 1;
        float qv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] = ld_cg_f(P.q + (size_t)i * d + h * hd + gl * 8 + e) * scale;
        const long long kvbase = ((long long)slot * P.L + l) * (long long)W * d + h * hd + gl * 8;
        float m = -INFINITY, lsum = 0.f, acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        constexpr int UNR = 4;
        // warp-uniform trip count: every lane runs every iteration (shuffles below)
        for (int jb = j0; jb < j1; jb += PPI * UNR) {
            const int jj = jb + grp;
            float kf[UNR][8], vf[UNR][8], s[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int j = jj + u * PPI;
                if (j < j1) {
                    const long long row = (long long)((start + j) % W) * d;
                    KV<TKV>::load8(P.kc, kvbase + row, kf[u]);
                    KV<TKV>::load8(P.vc, kvbase + row, vf[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) { kf[u][e] = 0.f; vf[u][e] = 0.f; }
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                float t = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) t = fmaf(qv[e], kf[u][e], t);
                for (int o = LPP / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                s[u] = (jj + u * PPI < j1) ? t : -INFINITY;
            }
            float mn = m;
#pragma unroll
            for (int u = 0; u < UNR; ++u) mn = fmaxf(mn, s[u]);
            if (mn == -INFINITY) continue;
            const float corr = expf(m - mn);
            lsum *= corr;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= corr;
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const float pu = expf(s[u] - mn);
                lsum += pu;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(pu, vf[u][e], acc[e]);
            }
            m = mn;
        }
        // merge the key groups of the warp (same bits on both partners)
        for (int o = LPP; o < 32; o <<= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, lsum, o);
            float a2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, acc[e], o);
            const float M = fmaxf(m, m2);
            const float c1 = m == -INFINITY ? 0.f : expf(m - M);
            const float c2 = m2 == -INFINITY ? 0.f : expf(m2 - M);
            lsum = lsum * c1 + l2 * c2;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = acc[e] * c1 + a2[e] * c2;
            m = M;
        }
        float* part = P.apart + (((size_t)i * H + h) * NCHUNK_MAX + c) * pstride;
        if (lane < LPP) {
            if (lane == 0) { part[0] = m; part[1] = lsum; }
            float4* dst = reinterpret_cast<float4*>(part + 4 + gl * 8);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        // the warp that completes (i, h) merges its chunks in chunk order
        __syncwarp();
        int old = 0;
        if (lane == 0) {
            __threadfence();
            old = atomicAdd(P.acnt + i * H + h, 1);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == nc - 1) {
            __threadfence();
            const float* pb = P.apart + ((size_t)i * H + h) * NCHUNK_MAX * pstride;
            const float mc = lane < nc ? ld_cg_f(pb + (size_t)lane * pstride) : -INFINITY;
            const float lc = lane < nc ? ld_cg_f(pb + (size_t)lane * pstride + 1) : 0.f;
            const float M = warp_max(mc);
            const float wc = mc == -INFINITY ? 0.f : expf(mc - M);
            const float invL = 1.f / warp_sum(lc * wc);
            for (int e = lane; e < hd; e += 32) {
                float a = 0.f;
#pragma unroll 4
                for (int cc = 0; cc < nc; ++cc) {
                    const float wcc = __shfl_sync(0xffffffffu, wc, cc);
                    a = fmaf(wcc, ld_cg_f(pb + (size_t)cc * pstride + 4 + e), a);
                }
                P.o[(size_t)i * d + h * hd + e] = a * invL;
            }
            if (lane == 0) P.acnt[i * H + h] = 0;
        }
    }
}

// ------------------------------------------------------------------ S9 depformer attention

__device__ void phase_dattn(const Params& P, int l, int j, int n)
{
    const int dd = P.dd, dH = P.dH, dhd = P.dhd, S = P.S;
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * NWARP + (threadIdx.x >> 5);
    const int npos = j + 1;
    const float scale = rsqrtf((float)dhd);
    for (int item = gwarp; item < n * dH; item += P.G * NWARP) {
        const int i = item / dH, h = item % dH;
        const float* q = P.dq + (size_t)i * dd + h * dhd;
        const float* kv = P.dkv + ((size_t)i * P.dL + l) * S * 2 * dd;
        float s = -INFINITY;
        if (lane < npos) {
            const float* kr = kv + (size_t)lane * 2 * dd + h * dhd;
            float t = 0.f;
            for (int e = 0; e < dhd; ++e) t = fmaf(ld_cg_f(q + e), ld_cg_f(kr + e), t);
            s = t * scale;
        }
        const float M = warp_max(s);
        const float pe = lane < npos ? expf(s - M) : 0.f;
        const float Z = warp_sum(pe);
        const float inv = 1.f / Z;
        for (int e = lane; e < dhd; e += 32) {
            float a = 0.f;
            for (int t = 0; t < npos; ++t) {
                const float pt = __shfl_sync(0xffffffffu, pe, t);
                a = fmaf(pt, ld_cg_f(kv + ((size_t)t * 2 + 1) * dd + h * dhd + e), a);
            }
            P.dat[(size_t)i * dd + h * dhd + e] = a * inv;
        }
        // lanes >= 32 of dhd handled by the loop above; all lanes shuffle uniformly
    }
}

// ------------------------------------------------------------------ S10

__device__ void phase_final(const Params& P, int n)
{
    if (blockIdx.x != 0) return;
    const StepDesc* D = P.desc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < n; i += NWARP) {
        const int S = P.S;
        const int a = argmax_partials_warp(P, i);
        if (lane != 0) continue;
        const int p = D->pos[i], slot = D->slot[i];
        {
            const int f = p - P.delays[S];
            const int forced = f >= 0 ? ld_cg_int(P.hist + ((size_t)slot * NSTREAM + S) * HIST + f % HIST) : -1;
            P.code_argmax[i * 16 + (S - 1)] = a;
            P.chosen[i * NSTREAM + S] = forced >= 0 ? forced : a;
        }
        for (int k = 0; k < NSTREAM; ++k) {
            const int f = p - P.delays[k];
            const int c = P.chosen[i * NSTREAM + k];
            if (f >= 0) P.hist[((size_t)slot * NSTREAM + k) * HIST + f % HIST] = c;
            if (k == 0) P.text_out[i] = c;
            else P.codes_out[i * 16 + (k - 1)] = f >= 0 ? c : -1;
        }
    }
}

// ------------------------------------------------------------------ phase dispatch

template <typename TW, typename TKV, int BG>
__device__ void run_phase(const Params& P, const Phase ph, int n, const Smem& sm)
{
    const int d = P.d, F = P.F, dd = P.dd, dF = P.dF;
    const TW* tl = (const TW*)P.tw + (size_t)ph.l * P.t_layer;
    const TW* dl = (const TW*)P.dw + (size_t)ph.j * P.d_sub + (size_t)ph.l * P.d_layer;
    XSrc xs{nullptr, 0, nullptr, nullptr, 0, nullptr};
    switch (ph.type) {
        case PH_EMBED: phase_embed<TW>(P, n, sm); break;
        case PH_QKV:
            xs = XSrc{P.x, d, P.attn_norm + (size_t)ph.l * d, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, tl, 3 * d, d, xs, -1, n, sm, [&](int lo, int hi, int b0, int nb, int bgv) {
                epi_qkv<TKV>(P, ph.l, lo, hi, b0, nb, bgv, sm);
            });
            break;
        case PH_ATTN: phase_attn<TKV>(P, ph.l, n, sm); break;
        case PH_O:
            xs = XSrc{P.o, d, nullptr, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, tl + (size_t)3 * d * d, d, d, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) { epi_resid(P.x, d, lo, hi, b0, nb, bgv, sm); });
            break;
        case PH_GU:
            xs = XSrc{P.x, d, P.ffn_norm + (size_t)ph.l * d, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, tl + (size_t)4 * d * d, 2 * F, d, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) { epi_swiglu(P.s, F, lo, hi, b0, nb, bgv, sm); });
            break;
        case PH_DOWN:
            xs = XSrc{P.s, F, nullptr, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, tl + (size_t)4 * d * d + (size_t)2 * F * d, d, F, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) { epi_resid(P.x, d, lo, hi, b0, nb, bgv, sm); });
            break;
        case PH_HEAD:
            xs = XSrc{P.x, d, P.out_norm, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, (const TW*)P.head, P.V + P.S * dd, d, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) {
                                   epi_logits(P, P.logits, P.V, P.V, P.yin, (long long)P.S * dd, lo, hi, b0, nb, bgv, sm);
                               });
            break;
        case PH_DQKV: {
            if (ph.l == 0) {
                const void* add = ph.j == 0 ? P.dep_emb_text
                                            : (const void*)((const TW*)P.dep_emb_audio + (size_t)(ph.j - 1) * P.C * dd);
                xs = XSrc{P.yin + (size_t)ph.j * dd, (long long)P.S * dd, P.dep_attn_norm, add, dd, P.u};
            } else {
                xs = XSrc{P.u, dd, P.dep_attn_norm + (size_t)ph.l * dd, nullptr, 0, nullptr};
            }
            gemv_phase<TW, BG>(P, dl, 3 * dd, dd, xs, ph.l == 0 ? ph.j : -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) {
                                   const int npair = hi - lo;
                                   for (int it = threadIdx.x; it < npair * nb; it += NT) {
                                       const int pl = it / nb, b = it % nb, i = b0 + b;
                                       const int r = 2 * (lo + pl);
                                       const int part = r / dd, e = r - part * dd;
                                       const float y0 = sm.yf[(size_t)(2 * pl) * bgv + b];
                                       const float y1 = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
                                       float* dst = part == 0 ? P.dq + (size_t)i * dd + e
                                                              : P.dkv + ((((size_t)i * P.dL + ph.l) * P.S + ph.j) * 2 + (part - 1)) * dd + e;
                                       dst[0] = y0;
                                       dst[1] = y1;
                                   }
                               });
            break;
        }
        case PH_DATTN: phase_dattn(P, ph.l, ph.j, n); break;
        case PH_DO:
            xs = XSrc{P.dat, dd, nullptr, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, dl + (size_t)3 * dd * dd, dd, dd, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) { epi_resid(P.u, dd, lo, hi, b0, nb, bgv, sm); });
            break;
        case PH_DGU:
            xs = XSrc{P.u, dd, P.dep_ffn_norm + (size_t)ph.l * dd, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, dl + (size_t)4 * dd * dd, 2 * dF, dd, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) { epi_swiglu(P.ds, dF, lo, hi, b0, nb, bgv, sm); });
            break;
        case PH_DDOWN:
            xs = XSrc{P.ds, dF, nullptr, nullptr, 0, nullptr};
            gemv_phase<TW, BG>(P, dl + (size_t)4 * dd * dd + (size_t)2 * dF * dd, dd, dF, xs, -1, n, sm,
                               [&](int lo, int hi, int b0, int nb, int bgv) { epi_resid(P.u, dd, lo, hi, b0, nb, bgv, sm); });
            break;
        case PH_DHEAD: {
            xs = XSrc{P.u, dd, P.dep_out_norm, nullptr, 0, nullptr};
            const TW* hw = (const TW*)P.dw + (size_t)ph.j * P.d_sub + (size_t)P.dL * P.d_layer;
            gemv_phase<TW, BG>(P, hw, P.C, dd, xs, -1, n, sm, [&](int lo, int hi, int b0, int nb, int bgv) {
                epi_logits(P, P.dlogits + (size_t)ph.j * P.C, (long long)P.S * P.C, P.C, nullptr, 0, lo, hi, b0, nb, bgv, sm);
            });
            break;
        }
        case PH_FINAL: phase_final(P, n); break;
        default: break;
    }
}

// ------------------------------------------------------------------ the kernel

// Phases [ph0, ph1) of one step.  coop != 0: cooperative launch, grid barrier
// between phases.  maxrows sizes the dynamic shared memory (host computes it).
template <typename TW, typename TKV, int BG>
__global__ void __launch_bounds__(NT, 1) step_kernel(Params P, int ph0, int ph1, int coop, int maxrows)
{
    extern __shared__ __align__(16) float smem_raw[];
    const Smem sm = smem_map(smem_raw, maxrows, BG);
    if (*(volatile int*)P.err != 0) return;
    const StepDesc* D = P.desc;
    const int n = D->n;
    if (ph0 == 0) {
        // token ranges (device-resident inputs are only checked here)
        int bad = 0;
        for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
            const int k = it % NSTREAM;
            const int t = D->codes[it / NSTREAM][k];
            if (t < -1 || t >= (k == 0 ? P.V : P.C)) bad = 1;
        }
        if (__syncthreads_or(bad)) {
            if (blockIdx.x == 0 && threadIdx.x == 0) {
                if (atomicCAS(P.err, 0, (int)DERR_TOKEN) == 0) *P.err_seq = D->seq;
            }
            return;
        }
    }
    unsigned target = 0;
    for (int ph = ph0; ph < ph1; ++ph) {
        if (P.ptime && blockIdx.x == 0 && threadIdx.x == 0) P.ptime[ph] = globaltimer_ns();
        const Phase phs = P.phases[ph];
        run_phase<TW, TKV, BG>(P, phs, n, sm);
        if (coop && ph + 1 < ph1) {
            target += (unsigned)P.G;
            if (!grid_barrier(P.bar, target, P.err)) return;
        }
    }
    if (P.ptime && blockIdx.x == 0 && threadIdx.x == 0) P.ptime[ph1] = globaltimer_ns();
}

}  // namespace
}  // namespace mfs
