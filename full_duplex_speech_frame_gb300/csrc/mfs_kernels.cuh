// Device code of the lockstep frame step.
//
// One persistent cooperative kernel runs every phase of a step (embedding sum,
// 32 temporal layers, text head, 16 depformer substeps, write-back) with a
// grid-wide barrier between phases; the same kernel can also be launched once
// per phase (no barriers) for diagnosis.  One CTA per SM: 16 consumer warps
// and one producer warp.
//
// Weights move by TMA bulk copies (cp.async.bulk) into a ring of shared-memory
// stages guarded by mbarriers.  The producer walks the same phase schedule as
// the consumers and copies each phase's weight rows as soon as a stage is
// free, so it runs ahead across the grid barriers and HBM keeps streaming while
// the consumers synchronise.  A CTA owns a contiguous block of row pairs of
// every matrix; its 16 consumer warps split K into contiguous slices and keep
// their slice of the (normalised) activations in registers for the whole
// phase.  Partial dot products are reduced lane-wise with a fixed shuffle
// tree, then across K-slices in slice order: the arithmetic of one slot never
// depends on the other slots of the batch, on the batch size or on the CTA
// that owns a row.
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

// ------------------------------------------------------------------ synchronisation

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // every spin gives up after 2 s

// Barrier over the 16 consumer warps of the CTA (the producer warp never joins).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// All CTAs' consumers arrive; false (error flag set) if the wait gave up or
// another CTA reported an error.
__device__ bool grid_barrier(unsigned* bar, unsigned target, int* err, int* s_ok)
{
    csync();
    if (threadIdx.x == 0) {
        red_release_add(bar, 1u);
        int ok = 1;
        unsigned long long t0 = 0;
        unsigned spins = 0;
        while (ld_acquire_u32(bar) < target) {
            if ((++spins & 63u) == 0u) {
                if (*(volatile int*)err != 0) { ok = 0; break; }
                const unsigned long long t = globaltimer_ns();
                if (t0 == 0) t0 = t;
                else if (t - t0 > WAIT_LIMIT_NS) { atomicCAS(err, 0, (int)DERR_BARRIER); ok = 0; break; }
            }
        }
        *s_ok = ok;
    }
    csync();
    return *(volatile int*)s_ok != 0;
}

__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* b, unsigned parity)
{
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(b)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.
__device__ bool mbar_wait(uint64_t* b, unsigned parity, int* err)
{
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
        if (mbar_try(b, parity)) return true;
        if ((i & 255u) == 255u) {
            if (*(volatile int*)err != 0) return false;
            const unsigned long long t = globaltimer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > WAIT_LIMIT_NS) { atomicCAS(err, 0, (int)DERR_BARRIER); return false; }
        }
    }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Diagnostic timer stamps of CTA 0: slot k of phase ph (0 start, 1 inputs
// ready, 2 last weight stage consumed, 3 before the grid barrier).
__device__ __forceinline__ void stamp(const Params& P, int ph, int k)
{
    if (P.ptime && blockIdx.x == 0 && threadIdx.x == 0) P.ptime[(size_t)ph * 4 + k] = globaltimer_ns();
}

// phase index for stamps taken inside a phase (thread 0 writes and reads it)


// ------------------------------------------------------------------ shared memory map

struct Smem {
    uint64_t* full;   // [nstage] stage filled
    uint64_t* empty;  // [nstage] stage released
    float* r;         // [4] RMSNorm factors of the batch group
    int* prev;        // [4] depformer input token per batch row
    float* ssq;       // [4][16] per-K-slice sums of squares
    float* amv;       // [NWARP]
    int* ami;         // [NWARP]
    int* ok;          // [0] grid-barrier verdict, [1] phase index (stamps)
    char* ring;       // [nstage][STAGE_BYTES]
    float* red;       // [maxrows][BG][16] per-K-slice partial sums of the CTA's rows
    float* yf;        // [maxrows][BG] final row values of the CTA
    int* X;           // embedding rows of this step (aliases red)
    float* wbuf;      // attention partials of the 16 warps (aliases red)
};

__device__ __forceinline__ Smem smem_map(char* base, int maxrows, int BG)
{
    Smem s;
    s.full = (uint64_t*)base;
    s.empty = s.full + 8;
    s.r = (float*)(base + 256);
    s.prev = (int*)(base + 272);
    s.ssq = (float*)(base + 288);
    s.amv = (float*)(base + 544);
    s.ami = (int*)(base + 608);
    s.ok = (int*)(base + 672);
    s.ring = base + SMEM_HEAD;
    s.red = (float*)(s.ring + (size_t)nstage_for(BG) * STAGE_BYTES);
    s.yf = s.red + (size_t)maxrows * BG * 16;
    s.X = (int*)s.red;
    s.wbuf = s.red;
    return s;
}

// ------------------------------------------------------------------ GEMV schedule (producer and consumers)

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

template <int BG>
__device__ __forceinline__ int group_size(int K)
{
    return gemv_cfg(K).vpl == 3 ? (BG < 2 ? BG : 2) : BG;
}

// The weight matrix a phase streams, or false if it streams none.
template <typename TW>
__device__ __forceinline__ bool phase_matrix(const Params& P, const Phase& ph, const TW*& W, int& N, int& K)
{
    const long long d = P.d, F = P.F, dd = P.dd, dF = P.dF;
    const TW* tl = (const TW*)P.tw + (size_t)ph.l * P.t_layer;
    const TW* dl = (const TW*)P.dw + (size_t)ph.j * P.d_sub + (size_t)ph.l * P.d_layer;
    switch (ph.type) {
        case PH_QKV: W = tl; N = 3 * d; K = d; return true;
        case PH_O: W = tl + 3 * d * d; N = d; K = d; return true;
        case PH_GU: W = tl + 4 * d * d; N = 2 * F; K = d; return true;
        case PH_DOWN: W = tl + 4 * d * d + 2 * F * d; N = d; K = F; return true;
        case PH_HEAD: W = (const TW*)P.head; N = P.V + P.S * dd; K = d; return true;
        case PH_DQKV: W = dl; N = 3 * dd; K = dd; return true;
        case PH_DO: W = dl + 3 * dd * dd; N = dd; K = dd; return true;
        case PH_DGU: W = dl + 4 * dd * dd; N = 2 * dF; K = dd; return true;
        case PH_DDOWN: W = dl + 4 * dd * dd + 2 * dF * dd; N = dd; K = dF; return true;
        case PH_DHEAD: W = (const TW*)P.dw + (size_t)ph.j * P.d_sub + (size_t)P.dL * P.d_layer; N = P.C; K = dd; return true;
        default: return false;
    }
}

__device__ __forceinline__ void cta_rows(int N, int G, int& r0, int& r1)
{
    const int npairs = N / 2;
    r0 = 2 * (int)((long long)npairs * blockIdx.x / G);
    r1 = 2 * (int)((long long)npairs * (blockIdx.x + 1) / G);
}

template <typename TW>
__device__ __forceinline__ int rows_per_stage(int K)
{
    const int r = STAGE_BYTES / (K * (int)sizeof(TW));
    return r < RPS_MAX ? r : RPS_MAX;
}

// Producer: copy, for every phase of the launch, every batch group's pass over
// this CTA's rows, stage by stage, in the order the consumers use them.
template <typename TW, int BG>
__device__ void producer(const Params& P, int ph0, int ph1, int n, const Smem& sm)
{
    constexpr unsigned NS = nstage_for(BG);
    unsigned s = 0;
    bool ok = true;
    for (int ph = ph0; ph < ph1 && ok; ++ph) {
        const TW* W;
        int N, K;
        if (!phase_matrix<TW>(P, P.phases[ph], W, N, K)) continue;
        int r0, r1;
        cta_rows(N, P.G, r0, r1);
        const int rps = rows_per_stage<TW>(K);
        const int bgv = group_size<BG>(K);
        for (int b0 = 0; b0 < n && ok; b0 += bgv) {
            for (int r = r0; r < r1; r += rps, ++s) {
                const int rows = min(rps, r1 - r);
                const unsigned bytes = (unsigned)(rows * K * (int)sizeof(TW));
                const int slot = (int)(s % NS);
                if (!mbar_wait(&sm.empty[slot], ((s / NS) & 1u) ^ 1u, P.err)) { ok = false; break; }
                mbar_expect_tx(&sm.full[slot], bytes);
                bulk_g2s(sm.ring + (size_t)slot * STAGE_BYTES, W + (size_t)r * K, bytes, &sm.full[slot]);
            }
        }
    }
    if (!ok) {
        // the consumers stopped early: wait (bounded) until every issued copy has landed
        for (unsigned k = s > NS ? s - NS : 0; k < s; ++k) {
            uint64_t* b = &sm.full[k % NS];
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try(b, (k / NS) & 1u))
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) break;
        }
    }
}

// ------------------------------------------------------------------ GEMV consumers

// Where the input vector of a matrix-vector phase comes from.
struct XSrc {
    const float* base;    // batch row i at base + i * stride
    long long stride;
    const float* g;       // RMSNorm gain, or nullptr for no norm
    const void* add;      // depformer embedding table (weight dtype) or nullptr
    long long add_stride; // row length of that table (elements)
    float* store;         // CTA 0 stores base + add here (depformer residual), or nullptr
};

// Consume one batch group [b0, b0+nb) of a matrix-vector phase: leaves the
// CTA's row values in sm.yf[(r - r0) * bgv + b].  `stage` counts ring stages.
__device__ __forceinline__ void dep_select_inputs(const Params& P, int j, int b0, int nb, const Smem& sm);

template <typename TW, int VPL, int BGV, int BG_OF_STAGES>
__device__ __forceinline__ bool gemv_group(const Params& P, int K, const GemvCfg& c, int r0, int r1, const XSrc& xs, int b0,
                           int nb, int dep_j, const Smem& sm, unsigned& stage)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kw = warp % c.nwk, rw = warp / c.nwk;
    const int NV = K / 8;
    const int v_begin = kw * c.nvw;
    const int v_end = min(NV, v_begin + c.nvw);
    // this warp's K-slice of the input in registers, already multiplied by the
    // norm gain (loaded in the same round trip); sums of squares of the raw input
    float xr[VPL][BGV][8];
    float ssq[BGV];
#pragma unroll
    for (int b = 0; b < BGV; ++b) ssq[b] = 0.f;
    const bool gain_now = xs.g && !xs.add;
#pragma unroll
    for (int t = 0; t < VPL; ++t) {
        const int v = v_begin + lane + 32 * t;
        float4 g0 = make_float4(1.f, 1.f, 1.f, 1.f), g1 = g0;
        if (gain_now && v < v_end) {
            const float4* gs = reinterpret_cast<const float4*>(xs.g + v * 8);
            g0 = __ldg(gs);
            g1 = __ldg(gs + 1);
        }
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            if (v < v_end && b < nb) {
                const float4* src = reinterpret_cast<const float4*>(xs.base + (size_t)(b0 + b) * xs.stride + v * 8);
                const float4 a0 = __ldcg(src), a1 = __ldcg(src + 1);
                const float f[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    ssq[b] = fmaf(f[e], f[e], ssq[b]);
                    xr[t][b][e] = f[e] * gg[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xr[t][b][e] = 0.f;
            }
        }
    }
    // depformer layer 0: the input adds the embedding of the token chosen by the
    // previous head (its selection overlaps the loads above); then the gain
    if (xs.add) {
        dep_select_inputs(P, dep_j, b0, nb, sm);
#pragma unroll
        for (int b = 0; b < BGV; ++b) ssq[b] = 0.f;
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            if (b >= nb) break;
            const TW* row = (const TW*)xs.add + (size_t)sm.prev[b] * (size_t)xs.add_stride;
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const int v = v_begin + lane + 32 * t;
                if (v < v_end) {
                    float e8[8];
                    WV<TW>::cvt(WV<TW>::load(row + v * 8), e8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        xr[t][b][e] += e8[e];
                        ssq[b] = fmaf(xr[t][b][e], xr[t][b][e], ssq[b]);
                    }
                }
            }
        }
        if (xs.store && blockIdx.x == 0 && rw == 0) {
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const int v = v_begin + lane + 32 * t;
#pragma unroll
                for (int b = 0; b < BGV; ++b) {
                    if (v < v_end && b < nb) {
                        float4* dst = reinterpret_cast<float4*>(xs.store + (size_t)(b0 + b) * K + v * 8);
                        dst[0] = make_float4(xr[t][b][0], xr[t][b][1], xr[t][b][2], xr[t][b][3]);
                        dst[1] = make_float4(xr[t][b][4], xr[t][b][5], xr[t][b][6], xr[t][b][7]);
                    }
                }
            }
        }
        if (xs.g) {
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const int v = v_begin + lane + 32 * t;
                if (v < v_end) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float ge = __ldg(xs.g + v * 8 + e);
#pragma unroll
                        for (int b = 0; b < BGV; ++b) xr[t][b][e] *= ge;
                    }
                }
            }
        }
    }
    if (xs.g) {
        // RMSNorm factor: sums of squares per K-slice, combined in slice order
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            const float q = warp_sum(ssq[b]);
            if (lane == 0 && rw == 0) sm.ssq[b * 16 + kw] = q;
        }
        csync();
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            float tot = 0.f;
            for (int k = 0; k < c.nwk; ++k) tot += sm.ssq[b * 16 + k];
            const float rb = rsqrtf(tot / (float)K + P.eps);
#pragma unroll
            for (int t = 0; t < VPL; ++t)
#pragma unroll
                for (int e = 0; e < 8; ++e) xr[t][b][e] *= rb;
        }
    }
    if (P.ptime) stamp(P, *(volatile int*)(sm.ok + 1), 1);
    // stream the CTA's rows through the ring: each warp takes rows rw, rw+nwr, ...
    // of a stage, four at a time, and releases the stage on its own
    using Vt = WV<TW>;
    constexpr unsigned NS = nstage_for(BG_OF_STAGES);
    const int rps = rows_per_stage<TW>(K);
    for (int ra = r0; ra < r1; ra += rps, ++stage) {
        const int nr = min(rps, r1 - ra);
        const int slot = (int)(stage % NS);
        if (!mbar_wait(&sm.full[slot], (stage / NS) & 1u, P.err)) return false;
        const TW* ring = (const TW*)(sm.ring + (size_t)slot * STAGE_BYTES);
        for (int c0 = rw; c0 < nr; c0 += 4 * c.nwr) {
            float acc[4][BGV];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int b = 0; b < BGV; ++b) acc[q][b] = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = c0 + q * c.nwr;
                if (rr < nr) {
#pragma unroll
                    for (int t = 0; t < VPL; ++t) {
                        const int v = v_begin + lane + 32 * t;
                        if (v < v_end) {
                            float f[8];
                            const TW* wp = ring + (size_t)rr * K + (size_t)v * 8;
                            if (sizeof(TW) == 2) {
                                const uint4 w4 = *reinterpret_cast<const uint4*>(wp);
                                f[0] = bf_lo(w4.x); f[1] = bf_hi(w4.x); f[2] = bf_lo(w4.y); f[3] = bf_hi(w4.y);
                                f[4] = bf_lo(w4.z); f[5] = bf_hi(w4.z); f[6] = bf_lo(w4.w); f[7] = bf_hi(w4.w);
                            } else {
                                const uint4 q0 = *reinterpret_cast<const uint4*>(wp);
                                const uint4 q1 = *reinterpret_cast<const uint4*>((const float*)wp + 4);
                                f[0] = __uint_as_float(q0.x); f[1] = __uint_as_float(q0.y); f[2] = __uint_as_float(q0.z); f[3] = __uint_as_float(q0.w);
                                f[4] = __uint_as_float(q1.x); f[5] = __uint_as_float(q1.y); f[6] = __uint_as_float(q1.z); f[7] = __uint_as_float(q1.w);
                            }
#pragma unroll
                            for (int b = 0; b < BGV; ++b)
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[q][b] = fmaf(f[e], xr[t][b][e], acc[q][b]);
                        }
                    }
                }
            }
            // transposed butterfly: lanes 0, 8, 16, 24 end with the sums of rows 0..3
            const int myq = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            const int rr = c0 + myq * c.nwr;
#pragma unroll
            for (int b = 0; b < BGV; ++b) {
                const bool hi16 = (lane & 16) != 0;
                float s0 = hi16 ? acc[2][b] : acc[0][b], s1 = hi16 ? acc[3][b] : acc[1][b];
                const float o0 = hi16 ? acc[0][b] : acc[2][b], o1 = hi16 ? acc[1][b] : acc[3][b];
                s0 += __shfl_xor_sync(0xffffffffu, o0, 16);
                s1 += __shfl_xor_sync(0xffffffffu, o1, 16);
                const bool hi8 = (lane & 8) != 0;
                float t = hi8 ? s1 : s0;
                const float u = hi8 ? s0 : s1;
                t += __shfl_xor_sync(0xffffffffu, u, 8);
                t += __shfl_xor_sync(0xffffffffu, t, 4);
                t += __shfl_xor_sync(0xffffffffu, t, 2);
                t += __shfl_xor_sync(0xffffffffu, t, 1);
                if ((lane & 7) == 0 && rr < nr)
                    sm.red[((size_t)(ra - r0 + rr) * BGV + b) * 16 + kw] = t;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    if (P.ptime) stamp(P, *(volatile int*)(sm.ok + 1), 2);
    csync();
    // sum the K-slices in slice order
    for (int it = tid; it < (r1 - r0) * nb; it += NT) {
        const int rl = it / nb, b = it % nb;
        const float* rp = sm.red + ((size_t)rl * BGV + b) * 16;
        float y = 0.f;
        for (int k = 0; k < c.nwk; ++k) y += rp[k];
        sm.yf[(size_t)rl * BGV + b] = y;
    }
    csync();
    return true;
}

// ------------------------------------------------------------------ epilogues

// An epilogue sees the CTA's rows [r0, r1) for batch rows b0..b0+nb-1, values
// in sm.yf[(row - r0) * bgv + b].  pre() runs before the weight stages and
// loads what apply() needs from memory (up to two items per thread), so the
// epilogue itself does not wait on a round trip.
struct Pre {
    float a[2], b[2];
};

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

template <typename TKV>
struct EpiQKV {
    int l;
    __device__ Pre pre(const Params& P, int r0, int r1, int b0, int nb) const
    {
        Pre q{{0.f, 0.f}, {0.f, 0.f}};
        const int npair = (r1 - r0) / 2;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int it = threadIdx.x + k * NT;
            if (it < npair * nb) {
                const int pl = it / nb, b = it % nb;
                const int r = r0 + 2 * pl, part = r / P.d, e = r - part * P.d;
                if (part < 2) {
                    const float2 cs = __ldg(P.rope + (size_t)P.desc->pos[b0 + b] * (P.hd / 2) + (e % P.hd) / 2);
                    q.a[k] = cs.x;
                    q.b[k] = cs.y;
                }
            }
        }
        return q;
    }
    __device__ void apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre& q) const
    {
        const StepDesc* D = P.desc;
        const int d = P.d, hd = P.hd;
        const int npair = (r1 - r0) / 2;
        for (int it = threadIdx.x; it < npair * nb; it += NT) {
            const int pl = it / nb, b = it % nb;
            const int i = b0 + b;
            const int r = r0 + 2 * pl;
            float y0 = sm.yf[(size_t)(2 * pl) * bgv + b], y1 = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
            const int part = r / d, e = r - part * d;
            const int p = D->pos[i];
            if (part < 2) {
                const int k = it / NT;
                const float2 cs = k < 2 ? make_float2(q.a[k], q.b[k]) : __ldg(P.rope + (size_t)p * (hd / 2) + (e % hd) / 2);
                const float a = y0, c = y1;
                y0 = a * cs.x - c * cs.y;
                y1 = a * cs.y + c * cs.x;
            }
            if (part == 0) {
                *reinterpret_cast<float2*>(P.q + (size_t)i * d + e) = make_float2(y0, y1);
            } else {
                const int slot = D->slot[i];
                const long long idx = (((long long)slot * P.L + l) * P.W + (p % P.W)) * (long long)d + e;
                KV<TKV>::store2(part == 1 ? P.kc : P.vc, idx, y0, y1);
            }
        }
    }
};

// dst[row] = residual + row value; the residual is read in pre()
struct EpiResid {
    float* dst;
    long long stride;
    __device__ Pre pre(const Params&, int r0, int r1, int b0, int nb) const
    {
        Pre q{{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int it = threadIdx.x + k * NT;
            if (it < (r1 - r0) * nb) q.a[k] = __ldcg(dst + (size_t)(b0 + it % nb) * stride + r0 + it / nb);
        }
        return q;
    }
    __device__ void apply(const Params&, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre& q) const
    {
        for (int it = threadIdx.x; it < (r1 - r0) * nb; it += NT) {
            const int rl = it / nb, b = it % nb;
            float* p = dst + (size_t)(b0 + b) * stride + r0 + rl;
            const int k = it / NT;
            *p = (k < 2 ? q.a[k] : __ldcg(p)) + sm.yf[(size_t)rl * bgv + b];
        }
    }
};

// rows are (gate m, up m) pairs
struct EpiSwiglu {
    float* dst;
    long long stride;
    __device__ Pre pre(const Params&, int, int, int, int) const { return Pre{{0.f, 0.f}, {0.f, 0.f}}; }
    __device__ void apply(const Params&, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre&) const
    {
        const int npair = (r1 - r0) / 2;
        for (int it = threadIdx.x; it < npair * nb; it += NT) {
            const int pl = it / nb, b = it % nb;
            const float g = sm.yf[(size_t)(2 * pl) * bgv + b], u = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
            dst[(size_t)(b0 + b) * stride + r0 / 2 + pl] = silu(g) * u;
        }
    }
};

// Rows [0, nlog) are logits (stored, and the CTA's argmax per batch row goes
// to amax_*[i][cta]); rows >= nlog go to extra[i][row - nlog] (may be null).
struct EpiLogits {
    float* lg;
    long long lg_stride;
    int nlog;
    float* extra;
    long long extra_stride;
    __device__ Pre pre(const Params&, int, int, int, int) const { return Pre{{0.f, 0.f}, {0.f, 0.f}}; }
    __device__ void apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre&) const
    {
        const int rows = r1 - r0;
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
            csync();
            if (lane == 0) { sm.amv[warp] = bv; sm.ami[warp] = bi; }
            csync();
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
};

// depformer q to dq, k and v of substep j to the layer's substep cache
struct EpiDQKV {
    int l, j;
    __device__ Pre pre(const Params&, int, int, int, int) const { return Pre{{0.f, 0.f}, {0.f, 0.f}}; }
    __device__ void apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre&) const
    {
        const int dd = P.dd;
        const int npair = (r1 - r0) / 2;
        for (int it = threadIdx.x; it < npair * nb; it += NT) {
            const int pl = it / nb, b = it % nb, i = b0 + b;
            const int r = r0 + 2 * pl;
            const int part = r / dd, e = r - part * dd;
            const float y0 = sm.yf[(size_t)(2 * pl) * bgv + b];
            const float y1 = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
            float* dst = part == 0 ? P.dq + (size_t)i * dd + e
                                   : P.dkv + ((((size_t)i * P.dL + l) * P.S + j) * 2 + (part - 1)) * dd + e;
            *reinterpret_cast<float2*>(dst) = make_float2(y0, y1);
        }
    }
};

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

// Picks, for depformer substep j, each batch row's input token (the text token
// for j = 0, else the code chosen for stream j), from the previous head's
// argmax partials unless the token was supplied.  CTA 0 records it.
__device__ __forceinline__ void dep_select_inputs(const Params& P, int j, int b0, int nb, const Smem& sm)
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
    csync();
}

// One matrix-vector phase; the epilogue consumes the CTA's rows.  dep_j >= 0
// selects the depformer layer-0 input tokens (xs.add set).
template <typename TW, int BG, class Epi>
__device__ bool gemv_phase(const Params& P, const Phase& ph, const XSrc& xs, int dep_j, int n, const Smem& sm,
                           unsigned& stage, const Epi& epi)
{
    const TW* W;
    int N, K;
    phase_matrix<TW>(P, ph, W, N, K);
    int r0, r1;
    cta_rows(N, P.G, r0, r1);
    const GemvCfg c = gemv_cfg(K);
    const int bgv = group_size<BG>(K);
    for (int b0 = 0; b0 < n; b0 += bgv) {
        const int nb = min(bgv, n - b0);
        if (r1 > r0 || xs.store) {
            const Pre pre = epi.pre(P, r0, r1, b0, nb);
            bool ok;
            switch (c.vpl) {
                case 1: ok = gemv_group<TW, 1, BG, BG>(P, K, c, r0, r1, xs, b0, nb, dep_j, sm, stage); break;
                case 2: ok = gemv_group<TW, 2, BG, BG>(P, K, c, r0, r1, xs, b0, nb, dep_j, sm, stage); break;
                default: ok = gemv_group<TW, 3, (BG < 2 ? BG : 2), BG>(P, K, c, r0, r1, xs, b0, nb, dep_j, sm, stage); break;
            }
            if (!ok) return false;
            epi.apply(P, sm, r0, r1, b0, nb, bgv, pre);
        } else if (dep_j >= 0) {
            dep_select_inputs(P, dep_j, b0, nb, sm);  // keeps the CTA's records consistent
        }
        csync();
    }
    return true;
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
    csync();
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
        // loads in batches of 6 rows (in flight together), summed in stream order
#pragma unroll
        for (int k0 = 0; k0 < NSTREAM; k0 += 6) {
            typename WV<TW>::raw rows[6];
#pragma unroll
            for (int q = 0; q < 6; ++q) {
                const int k = k0 + q;
                if (k < NSTREAM) {
                    const int tok = sm.X[i * NSTREAM + k];
                    const TW* row = k == 0 ? (const TW*)P.emb_text + (size_t)tok * d
                                           : (const TW*)P.emb_audio + ((size_t)(k - 1) * (P.C + 1) + tok) * d;
                    rows[q] = WV<TW>::load(row + e0);
                }
            }
#pragma unroll
            for (int q = 0; q < 6; ++q) {
                if (k0 + q < NSTREAM) {
                    float f[8];
                    WV<TW>::cvt(rows[q], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] += f[e];
                }
            }
        }
        float4* dst = reinterpret_cast<float4*>(P.x + (size_t)i * d + e0);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    csync();
}

// ------------------------------------------------------------------ S5 attention

// One CTA per (batch row, head); its 16 warps split the window into 16
// contiguous runs of keys (a split that depends on the window length only),
// and the partial softmax states are merged in shared memory in warp order.
template <typename TKV>
__device__ void phase_attn(const Params& P, int l, int n, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int H = P.H, hd = P.hd, d = P.d, W = P.W;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int LPP = hd / 8;            // lanes per key
    const int PPI = 32 / LPP;          // keys per warp iteration
    const int grp = lane / LPP, gl = lane % LPP;
    const float scale = rsqrtf((float)hd);
    const int wstride = hd + 4;
    for (int item = blockIdx.x; item < n * H; item += P.G) {
        const int i = item / H, h = item % H;
        const int p = D->pos[i], slot = D->slot[i];
        const int len = p + 1 < W ? p + 1 : W;
        const int start = p - len + 1;
        const int j0 = (int)((long long)len * warp / NWARP), j1 = (int)((long long)len * (warp + 1) / NWARP);
        float qv[8];
        {
            const float4* qs = reinterpret_cast<const float4*>(P.q + (size_t)i * d + h * hd + gl * 8);
            const float4 a0 = __ldcg(qs), a1 = __ldcg(qs + 1);
            qv[0] = a0.x * scale; qv[1] = a0.y * scale; qv[2] = a0.z * scale; qv[3] = a0.w * scale;
            qv[4] = a1.x * scale; qv[5] = a1.y * scale; qv[6] = a1.z * scale; qv[7] = a1.w * scale;
        }
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
        float* wb = sm.wbuf + (size_t)warp * wstride;
        if (lane < LPP) {
            if (lane == 0) { wb[0] = m; wb[1] = lsum; }
#pragma unroll
            for (int e = 0; e < 8; ++e) wb[4 + gl * 8 + e] = acc[e];
        }
        csync();
        // merge the 16 warps in warp order
        for (int e = threadIdx.x; e < hd; e += NT) {
            float M = -INFINITY;
            for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sm.wbuf[(size_t)w * wstride]);
            float L = 0.f, a = 0.f;
            for (int w = 0; w < NWARP; ++w) {
                const float mw = sm.wbuf[(size_t)w * wstride];
                if (mw == -INFINITY) continue;
                const float f = expf(mw - M);
                L += sm.wbuf[(size_t)w * wstride + 1] * f;
                a += sm.wbuf[(size_t)w * wstride + 4 + e] * f;
            }
            P.o[(size_t)i * d + h * hd + e] = a / L;
        }
        csync();
    }
}

// ------------------------------------------------------------------ S9 depformer attention

// One warp per (batch row, head): keys of substeps 0..j, no rotation.
__device__ void phase_dattn(const Params& P, int l, int j, int n)
{
    const int dd = P.dd, dH = P.dH, S = P.S;  // head dim is 64
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * NWARP + (threadIdx.x >> 5);
    const int npos = j + 1;
    const float scale = 0.125f;  // 1 / sqrt(64)
    for (int item = gwarp; item < n * dH; item += P.G * NWARP) {
        const int i = item / dH, h = item % dH;
        const float* q = P.dq + (size_t)i * dd + h * 64;
        const float* kv = P.dkv + ((size_t)i * P.dL + l) * S * 2 * dd + h * 64;
        // lane covers dims 2*lane, 2*lane+1; all key loads first, then one warp sum per key
        const float2 qq = __ldcg(reinterpret_cast<const float2*>(q) + lane);
        float2 k2[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            k2[t] = t < npos ? __ldcg(reinterpret_cast<const float2*>(kv + (size_t)t * 2 * dd) + lane) : make_float2(0.f, 0.f);
        float s = -INFINITY;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const float part = warp_sum(fmaf(qq.x, k2[t].x, qq.y * k2[t].y));
            if (t == lane && t < npos) s = part * scale;
        }
        const float M = warp_max(s);
        const float pe = lane < npos ? expf(s - M) : 0.f;
        const float inv = 1.f / warp_sum(pe);
        // this lane's two output dims: all value loads first, then the sum in key order
        float2 v[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            v[t] = t < npos ? __ldcg(reinterpret_cast<const float2*>(kv + ((size_t)t * 2 + 1) * dd) + lane)
                            : make_float2(0.f, 0.f);
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const float pt = __shfl_sync(0xffffffffu, pe, t);
            a0 = fmaf(pt, v[t].x, a0);
            a1 = fmaf(pt, v[t].y, a1);
        }
        reinterpret_cast<float2*>(P.dat + (size_t)i * dd + h * 64)[lane] = make_float2(a0 * inv, a1 * inv);
    }
}

// ------------------------------------------------------------------ S10

__device__ void phase_final(const Params& P, int n)
{
    if (blockIdx.x != 0) return;
    const StepDesc* D = P.desc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = P.S;
    for (int i = warp; i < n; i += NWARP) {
        const int a = argmax_partials_warp(P, i);
        const int p = D->pos[i], slot = D->slot[i];
        if (lane < NSTREAM) {
            const int k = lane;
            const int f = p - P.delays[k];
            int c;
            if (k == S) {
                const int forced = f >= 0 ? ld_cg_int(P.hist + ((size_t)slot * NSTREAM + S) * HIST + f % HIST) : -1;
                c = forced >= 0 ? forced : a;
                P.code_argmax[i * 16 + (S - 1)] = a;
            } else {
                c = P.chosen[i * NSTREAM + k];
            }
            if (f >= 0) P.hist[((size_t)slot * NSTREAM + k) * HIST + f % HIST] = c;
            if (k == 0) P.text_out[i] = c;
            else P.codes_out[i * 16 + (k - 1)] = f >= 0 ? c : -1;
        }
    }
}

// ------------------------------------------------------------------ phase dispatch

template <typename TW, typename TKV, int BG>
__device__ bool run_phase(const Params& P, const Phase ph, int n, const Smem& sm, unsigned& stage)
{
    const int d = P.d, F = P.F, dd = P.dd, dF = P.dF;
    switch (ph.type) {
        case PH_EMBED: phase_embed<TW>(P, n, sm); return true;
        case PH_QKV:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.x, d, P.attn_norm + (size_t)ph.l * d, nullptr, 0, nullptr}, -1, n,
                                      sm, stage, EpiQKV<TKV>{ph.l});
        case PH_ATTN: phase_attn<TKV>(P, ph.l, n, sm); return true;
        case PH_O:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.o, d, nullptr, nullptr, 0, nullptr}, -1, n, sm, stage,
                                      EpiResid{P.x, d});
        case PH_GU:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.x, d, P.ffn_norm + (size_t)ph.l * d, nullptr, 0, nullptr}, -1, n,
                                      sm, stage, EpiSwiglu{P.s, F});
        case PH_DOWN:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.s, F, nullptr, nullptr, 0, nullptr}, -1, n, sm, stage,
                                      EpiResid{P.x, d});
        case PH_HEAD:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.x, d, P.out_norm, nullptr, 0, nullptr}, -1, n, sm, stage,
                                      EpiLogits{P.logits, P.V, P.V, P.yin, (long long)P.S * dd});
        case PH_DQKV: {
            XSrc xs;
            if (ph.l == 0) {
                const void* add = ph.j == 0 ? P.dep_emb_text
                                            : (const void*)((const TW*)P.dep_emb_audio + (size_t)(ph.j - 1) * P.C * dd);
                xs = XSrc{P.yin + (size_t)ph.j * dd, (long long)P.S * dd, P.dep_attn_norm, add, dd, P.u};
            } else {
                xs = XSrc{P.u, dd, P.dep_attn_norm + (size_t)ph.l * dd, nullptr, 0, nullptr};
            }
            return gemv_phase<TW, BG>(P, ph, xs, ph.l == 0 ? ph.j : -1, n, sm, stage, EpiDQKV{ph.l, ph.j});
        }
        case PH_DATTN: phase_dattn(P, ph.l, ph.j, n); return true;
        case PH_DO:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.dat, dd, nullptr, nullptr, 0, nullptr}, -1, n, sm, stage,
                                      EpiResid{P.u, dd});
        case PH_DGU:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.u, dd, P.dep_ffn_norm + (size_t)ph.l * dd, nullptr, 0, nullptr}, -1,
                                      n, sm, stage, EpiSwiglu{P.ds, dF});
        case PH_DDOWN:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.ds, dF, nullptr, nullptr, 0, nullptr}, -1, n, sm, stage,
                                      EpiResid{P.u, dd});
        case PH_DHEAD:
            return gemv_phase<TW, BG>(P, ph, XSrc{P.u, dd, P.dep_out_norm, nullptr, 0, nullptr}, -1, n, sm, stage,
                                      EpiLogits{P.dlogits + (size_t)ph.j * P.C, (long long)P.S * P.C, P.C, nullptr, 0});
        case PH_FINAL: phase_final(P, n); return true;
        default: return true;
    }
}

// ------------------------------------------------------------------ the kernel

// Phases [ph0, ph1) of one step.  coop != 0: cooperative launch, grid barrier
// between phases.  maxrows sizes the dynamic shared memory (host computes it).
template <typename TW, typename TKV, int BG>
__global__ void __launch_bounds__(NT + 32, 1) step_kernel(Params P, int ph0, int ph1, int coop, int maxrows)
{
    extern __shared__ __align__(1024) char smem_raw[];
    const Smem sm = smem_map(smem_raw, maxrows, BG);
    if (threadIdx.x == 0) {
        for (int k = 0; k < (int)nstage_for(BG); ++k) {
            mbar_init(&sm.full[k], 1);
            mbar_init(&sm.empty[k], NWARP);  // every consumer warp releases every stage
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const StepDesc* D = P.desc;
    const int n = D->n;
    int bad = *(volatile int*)P.err != 0;
    if (ph0 == 0 && !bad) {
        // token ranges (device-resident inputs are only checked here)
        int tb = 0;
        for (int it = threadIdx.x; it < n * NSTREAM; it += blockDim.x) {
            const int k = it % NSTREAM;
            const int t = D->codes[it / NSTREAM][k];
            if (t < -1 || t >= (k == 0 ? P.V : P.C)) tb = 1;
        }
        if (__syncthreads_or(tb)) {
            if (blockIdx.x == 0 && threadIdx.x == 0) {
                if (atomicCAS(P.err, 0, (int)DERR_TOKEN) == 0) *P.err_seq = D->seq;
            }
            bad = 1;
        }
    }
    __syncthreads();  // barrier init visible to every thread; all threads agree on `bad`
    if (bad) return;
    if ((threadIdx.x >> 5) == NWARP) {
        if ((threadIdx.x & 31) == 0) producer<TW, BG>(P, ph0, ph1, n, sm);
        return;
    }
    unsigned target = 0, stage = 0;
    for (int ph = ph0; ph < ph1; ++ph) {
        if (threadIdx.x == 0) sm.ok[1] = ph;  // phase index for the in-phase stamps
        stamp(P, ph, 0);
        const Phase phs = P.phases[ph];
        if (!run_phase<TW, TKV, BG>(P, phs, n, sm, stage)) return;
        stamp(P, ph, 3);
        if (coop && ph + 1 < ph1) {
            target += (unsigned)P.G;
            if (!grid_barrier(P.bar, target, P.err, sm.ok)) return;
        }
    }
    stamp(P, ph1, 0);
}

}  // namespace
}  // namespace mfs
