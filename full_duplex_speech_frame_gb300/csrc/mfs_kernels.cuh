// Device code of the lockstep frame step.
//
// One persistent cooperative kernel runs every phase of a step (embedding sum,
// 32 temporal layers, text head, 16 depformer substeps, write-back); the same
// kernel can also be launched once per phase for diagnosis.  One CTA per SM:
// 8 consumer warps and one producer warp.
//
// Weights move by TMA bulk copies (cp.async.bulk) into a ring of shared-memory
// stages guarded by mbarriers.  The producer walks the same phase schedule as
// the consumers and copies each phase's weight rows as soon as a stage is
// free, so HBM keeps streaming while the consumers wait for their inputs.
//
// Phases do not meet at grid barriers.  Every activation element that crosses
// CTAs is a 64-bit word {value, tag} written with one single-copy-atomic
// store; the tag is (step sequence << 10 | writer phase).  A consumer reads
// exactly the elements it needs and re-reads until the tags match, so a phase
// starts as soon as its inputs exist, and a stale value can never be consumed
// (a wait that cannot complete gives up after 2 s and sets the error flag).
// Buffers are reused only after every reader of the previous value has
// produced an output that the next writer itself waits for.
//
// A CTA owns a contiguous block of row pairs of every matrix; its 8 consumer
// warps split K into contiguous slices and keep their slice of the
// (normalised) activations in registers for the whole phase.  Partial dot
// products are reduced with a fixed shuffle tree, then across K-slices in
// slice order: the arithmetic of one slot never depends on the other slots of
// the batch, on the batch size or on the CTA that owns a row.
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

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

// L2-only load of keys/values written by earlier launches (no ordering
// constraint, so the compiler keeps many of these in flight).
__device__ __forceinline__ uint4 ld_cg16(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ int ld_cg_int(const int* p) { return __ldcg(p); }

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// A "vector" is 8 consecutive weights.
template <typename TW>
struct WV;

template <>
struct WV<__nv_bfloat16> {
    struct raw { uint4 a; };
    static __device__ __forceinline__ raw load(const __nv_bfloat16* p) { return {ld_stream16(p)}; }
    static __device__ __forceinline__ void cvt(const raw& r, float f[8])
    {
        f[0] = bf_lo(r.a.x); f[1] = bf_hi(r.a.x); f[2] = bf_lo(r.a.y); f[3] = bf_hi(r.a.y);
        f[4] = bf_lo(r.a.z); f[5] = bf_hi(r.a.z); f[6] = bf_lo(r.a.w); f[7] = bf_hi(r.a.w);
    }
    // 8 weights from shared memory
    static __device__ __forceinline__ void lds8(const __nv_bfloat16* p, float f[8])
    {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        f[0] = bf_lo(w.x); f[1] = bf_hi(w.x); f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
        f[4] = bf_lo(w.z); f[5] = bf_hi(w.z); f[6] = bf_lo(w.w); f[7] = bf_hi(w.w);
    }
};

template <>
struct WV<float> {
    struct raw { uint4 a, b; };
    static __device__ __forceinline__ raw load(const float* p) { return {ld_stream16(p), ld_stream16(p + 4)}; }
    static __device__ __forceinline__ void cvt(const raw& r, float f[8])
    {
        f[0] = __uint_as_float(r.a.x); f[1] = __uint_as_float(r.a.y);
        f[2] = __uint_as_float(r.a.z); f[3] = __uint_as_float(r.a.w);
        f[4] = __uint_as_float(r.b.x); f[5] = __uint_as_float(r.b.y);
        f[6] = __uint_as_float(r.b.z); f[7] = __uint_as_float(r.b.w);
    }
    static __device__ __forceinline__ void lds8(const float* p, float f[8])
    {
        const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

// Key/value ring element type.
template <typename TKV>
struct KV;

template <>
struct KV<__nv_bfloat16> {
    // 8 consecutive elements as loaded (kept packed in registers until used)
    struct raw { uint4 a; };
    static __device__ __forceinline__ raw load_raw(const void* base, long long i)
    {
        return {ld_cg16((const __nv_bfloat16*)base + i)};
    }
    static __device__ __forceinline__ void unpack(const raw& r, float f[8])
    {
        f[0] = bf_lo(r.a.x); f[1] = bf_hi(r.a.x); f[2] = bf_lo(r.a.y); f[3] = bf_hi(r.a.y);
        f[4] = bf_lo(r.a.z); f[5] = bf_hi(r.a.z); f[6] = bf_lo(r.a.w); f[7] = bf_hi(r.a.w);
    }
    // values already rounded to bf16 pack exactly
    static __device__ __forceinline__ raw pack(const float f[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[e], f[e + 1]);
            w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return {make_uint4(w[0], w[1], w[2], w[3])};
    }
    static __device__ __forceinline__ float round(float a) { return __bfloat162float(__float2bfloat16_rn(a)); }
    static __device__ __forceinline__ void store2(void* base, long long i, float a, float b)
    {
        *reinterpret_cast<__nv_bfloat162*>((__nv_bfloat16*)base + i) = __floats2bfloat162_rn(a, b);
    }
    static __device__ __forceinline__ void load8(const void* base, long long i, float f[8])
    {
        const uint4 r = ld_cg16((const __nv_bfloat16*)base + i);
        f[0] = bf_lo(r.x); f[1] = bf_hi(r.x); f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
        f[4] = bf_lo(r.z); f[5] = bf_hi(r.z); f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
    }
};

template <>
struct KV<float> {
    struct raw { uint4 a, b; };
    static __device__ __forceinline__ raw load_raw(const void* base, long long i)
    {
        return {ld_cg16((const float*)base + i), ld_cg16((const float*)base + i + 4)};
    }
    static __device__ __forceinline__ void unpack(const raw& r, float f[8])
    {
        f[0] = __uint_as_float(r.a.x); f[1] = __uint_as_float(r.a.y); f[2] = __uint_as_float(r.a.z); f[3] = __uint_as_float(r.a.w);
        f[4] = __uint_as_float(r.b.x); f[5] = __uint_as_float(r.b.y); f[6] = __uint_as_float(r.b.z); f[7] = __uint_as_float(r.b.w);
    }
    static __device__ __forceinline__ raw pack(const float f[8])
    {
        return {make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3])),
                make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]), __float_as_uint(f[7]))};
    }
    static __device__ __forceinline__ float round(float a) { return a; }
    static __device__ __forceinline__ void store2(void* base, long long i, float a, float b)
    {
        *reinterpret_cast<float2*>((float*)base + i) = make_float2(a, b);
    }
    static __device__ __forceinline__ void load8(const void* base, long long i, float f[8])
    {
        const uint4 r0 = ld_cg16((const float*)base + i), r1 = ld_cg16((const float*)base + i + 4);
        f[0] = __uint_as_float(r0.x); f[1] = __uint_as_float(r0.y); f[2] = __uint_as_float(r0.z); f[3] = __uint_as_float(r0.w);
        f[4] = __uint_as_float(r1.x); f[5] = __uint_as_float(r1.y); f[6] = __uint_as_float(r1.z); f[7] = __uint_as_float(r1.w);
    }
};

// ------------------------------------------------------------------ timers, errors

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // every wait gives up after 2 s (default)

// Spin bookkeeping: every 64 spins look at the clock and the error flag.
// false: give up.  The first waiter to give up records where (err[2..6]:
// wait site, expected and observed tag or parity, CTA, thread).  err[7], when
// positive, replaces the 2 s limit (microseconds).
enum WaitSite : int { WS_TAG1 = 1, WS_TAG8 = 2, WS_FULL = 3, WS_EMPTY = 4, WS_DQ = 5, WS_DKV = 6 };

struct Spin {
    unsigned n = 0;
    unsigned long long t0 = 0, lim = WAIT_LIMIT_NS;
    __device__ __forceinline__ bool ok(int* err, int site, unsigned want, unsigned seen)
    {
        if ((++n & 63u) != 0u) return true;
        if (*(volatile int*)err != 0) return false;
        const unsigned long long t = globaltimer_ns();
        if (t0 == 0) {
            t0 = t;
            const int us = *(volatile int*)(err + 7);
            if (us > 0) lim = (unsigned long long)us * 1000ull;
            return true;
        }
        if (t - t0 > lim) {
            if (atomicCAS(err, 0, (int)DERR_WAIT) == 0) {
                err[2] = site;
                err[3] = (int)want;
                err[4] = (int)seen;
                err[5] = (int)blockIdx.x;
                err[6] = (int)threadIdx.x;
            }
            return false;
        }
        return true;
    }
};

// ------------------------------------------------------------------ tagged values

__device__ __forceinline__ unsigned phase_tag(const StepDesc* D, int ph)
{
    return ((unsigned)D->seq << 10) | (unsigned)ph;
}

// Tagged elements are read and written with relaxed gpu-scope (morally strong)
// operations: weak loads may keep returning a stale copy of a line written by
// another SM, strong ones observe the coherent value.
// Two tagged elements (16 bytes; each 64-bit half is single-copy atomic).
__device__ __forceinline__ void ld_tag2(const uint2* p, uint2& a, uint2& b)
{
    unsigned long long x, y;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
    a = make_uint2((unsigned)x, (unsigned)(x >> 32));
    b = make_uint2((unsigned)y, (unsigned)(y >> 32));
}

__device__ __forceinline__ uint2 ld_tag1(const uint2* p)
{
    unsigned long long x;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
    return make_uint2((unsigned)x, (unsigned)(x >> 32));
}

__device__ __forceinline__ void st_tag2(uint2* p, float a, float b, unsigned tag)
{
    const unsigned long long x = ((unsigned long long)tag << 32) | __float_as_uint(a);
    const unsigned long long y = ((unsigned long long)tag << 32) | __float_as_uint(b);
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(x), "l"(y) : "memory");
}

__device__ __forceinline__ void st_tag1(uint2* p, unsigned bits, unsigned tag)
{
    const unsigned long long x = ((unsigned long long)tag << 32) | bits;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(x) : "memory");
}

// one element, waiting for its tag
__device__ __forceinline__ bool wait_tag1(const uint2* p, unsigned tag, unsigned& bits, int* err)
{
    Spin sp;
    for (;;) {
        const uint2 e = ld_tag1(p);
        if (e.y == tag) { bits = e.x; return true; }
        if (!sp.ok(err, WS_TAG1, tag, e.y)) return false;
    }
}

// 8 consecutive elements, waiting for their tags
__device__ __forceinline__ bool wait_tag8(const uint2* p, unsigned tag, float f[8], int* err)
{
    Spin sp;
    for (;;) {
        uint2 e[8];
        ld_tag2(p, e[0], e[1]);
        ld_tag2(p + 2, e[2], e[3]);
        ld_tag2(p + 4, e[4], e[5]);
        ld_tag2(p + 6, e[6], e[7]);
        bool ok = true;
        unsigned seen = tag;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            ok = ok && e[k].y == tag;
            if (e[k].y != tag) seen = e[k].y;
        }
        if (ok) {
#pragma unroll
            for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(e[k].x);
            return true;
        }
        if (!sp.ok(err, WS_TAG8, tag, seen)) return false;
    }
}

// Issue the loads of 8 tagged elements without waiting (values and tags land
// in e[]); tag8_take() checks them and falls back to wait_tag8 if needed.
__device__ __forceinline__ void tag8_issue(const uint2* p, uint2 (&e)[8])
{
    ld_tag2(p, e[0], e[1]);
    ld_tag2(p + 2, e[2], e[3]);
    ld_tag2(p + 4, e[4], e[5]);
    ld_tag2(p + 6, e[6], e[7]);
}

__device__ __forceinline__ bool tag8_take(const uint2 (&e)[8], const uint2* p, unsigned tag, float f[8], int* err)
{
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 8; ++k) ok = ok && e[k].y == tag;
    if (ok) {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(e[k].x);
        return true;
    }
    return wait_tag8(p, tag, f, err);
}

// Two IEEE fp32 FMAs in one instruction: c = a * b + c lane by lane.
__device__ __forceinline__ void ffma2(float2& c, float a0, float a1, float b0, float b1)
{
    unsigned long long ra, rb, rc;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(rc) : "l"(ra), "l"(rb));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(c.x), "=f"(c.y) : "l"(rc));
}

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
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (am_better(v2, i2, v, i)) { v = v2; i = i2; }
    }
}

// ------------------------------------------------------------------ synchronisation

// Barrier over the consumer warps of the CTA (the producer warp never joins).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

// Same barrier, returning whether the predicate held in every consumer thread.
__device__ __forceinline__ bool csync_and(int pred)
{
    int r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"(pred), "n"(NT) : "memory");
    return r != 0;
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

// test_wait: a poll that never suspends the thread (waiters see a completed phase at once)
__device__ __forceinline__ bool mbar_try(uint64_t* b, unsigned parity)
{
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(b)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, unsigned parity, int* err, int site)
{
    Spin sp;
    for (;;) {
        if (mbar_try(b, parity)) return true;
        if (!sp.ok(err, site, parity, 0)) return false;
    }
}

// L2 policies: streamed weights are evicted first, so that activations and
// prefetched keys/values stay resident.
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

// ------------------------------------------------------------------ shared memory map

struct Smem {
    uint64_t* full;   // [nstage] stage filled
    uint64_t* empty;  // [nstage] stage released
    float* ssq;       // [4][16] per-K-slice sums of squares
    int* prev;        // [4] (tensor-core path: [32]) depformer input token per batch row
    float* amv;       // [NWARP]
    int* ami;         // [NWARP]
    int* misc;        // [0] phase index (diagnostic stamps)
    char* ring;       // [nstage][STAGE_BYTES]
    float* red;       // [maxrows][BG][NWARP] per-K-slice partial sums of the CTA's rows
    float* yf;        // [maxrows][BG] final row values of the CTA
    int* X;           // embedding rows of this step (aliases red)
    float* wbuf;      // attention partials of the consumer warps (aliases red)
    // tensor-core path (null in the matrix-vector instantiations)
    uint64_t* wfull;  // [MMA_NSTAGE] weight chunk landed (TMA)
    uint64_t* bfull;  // [MMA_NSTAGE] activation chunk written (one arrival per consumer warp)
    uint64_t* sempty; // [MMA_NSTAGE] stage consumed by the MMAs (tcgen05.commit)
    uint64_t* accf;   // [MMA_URING] (tdone) a unit's products are in its tensor-memory slot (tcgen05.commit)
    uint64_t* tfree;  // [MMA_URING] the consumer warps have read that slot (one arrival per warp)
    uint64_t* adone;  // the consumers are past every stage of an attention phase (thread 0, once per phase)
    uint64_t* mdone;  // every MMA the CTA issued has completed (before TMEM is freed)
    uint32_t* tslot;  // TMEM base address from tcgen05.alloc
    float* pssq;      // [MMA_MAX_TILES][32] this CTA's sums of squares of its inputs per tile part
    float* bestv;     // [32] deferred argmax partials over the tiles a CTA owns
    int* besti;       // [32]
    char* mring;      // [MMA_NSTAGE][MMA_STAGE], 1024-byte aligned
};

__device__ __forceinline__ Smem smem_map(char* base, int maxrows, int BG)
{
    Smem s;
    s.full = (uint64_t*)base;
    s.empty = s.full + 8;
    s.ssq = (float*)(base + 256);
    s.prev = (int*)(base + 512);
    s.amv = (float*)(base + 544);
    s.ami = (int*)(base + 608);
    s.misc = (int*)(base + 672);
    s.ring = base + SMEM_HEAD;
    s.red = (float*)(s.ring + (size_t)nstage_for(BG) * STAGE_BYTES);
    s.yf = s.red + (size_t)maxrows * BG * NWARP;
    s.X = (int*)s.red;
    s.wbuf = s.red;
    s.wfull = s.bfull = s.sempty = s.accf = s.tfree = s.adone = s.mdone = nullptr;
    s.tslot = nullptr;
    s.pssq = s.bestv = nullptr;
    s.besti = nullptr;
    s.mring = nullptr;
    return s;
}

// Tensor-core instantiation: barriers and scalars in the first MMA_HEAD bytes
// of a 1024-byte aligned base, then the stages, then one region shared by the
// tile values of an epilogue, the attention partials, the embedding rows and
// the sampler (never live at the same time).
__device__ __forceinline__ Smem smem_map_mma(char* base)
{
    Smem s;
    s.wfull = (uint64_t*)base;
    s.bfull = s.wfull + 8;
    s.sempty = s.wfull + 16;
    s.accf = s.wfull + 24;
    s.adone = s.wfull + 32;
    s.mdone = s.wfull + 33;
    s.tslot = (uint32_t*)(base + 272);
    s.full = s.empty = nullptr;
    s.ssq = (float*)(base + 320);     // [4][16], unused here
    s.prev = (int*)(base + 576);      // [32]
    s.amv = (float*)(base + 704);     // [NWARP]
    s.ami = (int*)(base + 736);       // [NWARP]
    s.misc = (int*)(base + 768);      // [64]
    s.tfree = (uint64_t*)(base + 1024);  // [MMA_URING]
    s.pssq = nullptr;
    s.bestv = (float*)(base + 2048);  // [32]
    s.besti = (int*)(base + 2176);    // [32]
    s.mring = base + MMA_HEAD;
    s.ring = nullptr;
    s.red = (float*)(s.mring + (size_t)MMA_NSTAGE * MMA_STAGE);
    s.yf = s.red;
    s.X = (int*)s.red;
    s.wbuf = s.red;
    return s;
}

// Diagnostic timer stamps of CTA 0: slot k of phase ph (0 start, 1 inputs
// ready, 2 last weight stage consumed, 3 end of the phase).
__device__ __forceinline__ void stamp(const Params& P, int ph, int k)
{
    if (P.ptime && blockIdx.x == 0 && threadIdx.x == 0) P.ptime[(size_t)ph * 8 + k] = globaltimer_ns();
}

// ------------------------------------------------------------------ GEMV schedule (producer and consumers)

struct GemvCfg {
    int nwk, nwr, nvw, vpl;
};

// K-slices per row: the largest power of two <= NWARP that leaves >= 32
// vectors (of 8 weights) per slice.
__device__ __forceinline__ GemvCfg gemv_cfg(int K)
{
    const int NV = K / 8;
    const int nwk = slice_warps(K);
    GemvCfg c;
    c.nwk = nwk;
    c.nwr = NWARP / nwk;
    c.nvw = (NV + nwk - 1) / nwk;
    c.vpl = (c.nvw + 31) / 32;
    return c;
}

// vectors per lane, rounded up to an instantiated width
__device__ __forceinline__ int vpl_class(int vpl) { return vpl_class_of(vpl); }

// batch rows per pass: the input slice (8 * vpl * rows floats) stays in registers
template <int BG>
__device__ __forceinline__ int group_size(int K)
{
    return vpl_class(gemv_cfg(K).vpl) <= 2 ? BG : (BG < 2 ? BG : 2);
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

// Rows [r0, r1) of an N-row matrix for CTA c of the cnt that share it (row pairs stay together).
__device__ __forceinline__ void cta_rows(int N, int cnt, int c, int& r0, int& r1)
{
    const int npairs = N / 2;
    r0 = 2 * (int)((long long)npairs * c / cnt);
    r1 = 2 * (int)((long long)npairs * (c + 1) / cnt);
}

// ------------------------------------------------------------------ depformer substep groups
// A substep whose input token is supplied for every slot of the step (forced
// this frame, or the frame before for a delayed stream) needs nothing from the
// substep before it except that layer's keys and values, so it runs with that
// substep in one wide pass per layer; at most MAXGW substeps form a group.
// `starts` has bit j set where a group begins (always bit 0).

// Token of stream k for frame p - delay[k] supplied by the caller, or -1.
__device__ __forceinline__ int supplied_token(const Params& P, int i, int k)
{
    const StepDesc* D = P.desc;
    const int p = D->pos[i], f = p - P.delays[k];
    if (f == p) return D->codes[i][k];
    if (f >= 0) return __ldcg(P.hist + ((size_t)D->slot[i] * NSTREAM + k) * HIST + f % HIST);
    return -1;
}

// `starts` packs the group boundaries (bits 0..15: a group begins at substep j;
// a set bit past the last group that runs marks where the run stops) and, in
// bits 24..28, the number of groups that run this step.
__device__ __forceinline__ int n_groups(unsigned starts) { return (int)((starts >> 24) & 31u); }
__device__ __forceinline__ int group_of(unsigned starts, int t) { return __popc(starts & 0xFFFFu & ((2u << t) - 1u)) - 1; }

// first substep j0 and width nj of group g
__device__ __forceinline__ void group_bounds(unsigned starts, int S, int g, int& j0, int& nj)
{
    unsigned m = starts & 0xFFFFu;
    for (int k = 0; k < g; ++k) m &= m - 1u;
    j0 = __ffs(m) - 1;
    m &= m - 1u;
    nj = (m ? __ffs(m) - 1 : S) - j0;
}

// CTAs [b0, b1) of the G work on substep s of an nj-wide group
__device__ __forceinline__ void substep_ctas(int G, int nj, int s, int& b0, int& b1)
{
    b0 = (int)(((long long)s * G + nj - 1) / nj);
    b1 = (int)(((long long)(s + 1) * G + nj - 1) / nj);
}

__device__ __forceinline__ bool is_dep_gemv(int type) { return type == PH_DQKV || type == PH_DO || type == PH_DGU || type == PH_DDOWN || type == PH_DHEAD; }

// This CTA's share of a phase: CTA c of the cnt that share its matrix.  A
// depformer phase's Phase.j names its group; resolve() turns it into this
// CTA's substep (q.j) and records the group's first substep (q.pad0) and
// width (q.pad1).  False when the group does not exist this step.
__device__ __forceinline__ bool resolve(const Params& P, unsigned starts, Phase& q, int& c, int& cnt)
{
    c = blockIdx.x;
    cnt = P.G;
    if (q.type >= PH_DQKV && q.type <= PH_DHEAD) {
        if (q.j >= n_groups(starts)) return false;
        int j0, nj;
        group_bounds(starts, P.S, q.j, j0, nj);
        q.pad0 = j0;
        q.pad1 = nj;
        if (is_dep_gemv(q.type)) {
            const int s = (int)((long long)blockIdx.x * nj / P.G);
            int b0, b1;
            substep_ctas(P.G, nj, s, b0, b1);
            c = blockIdx.x - b0;
            cnt = b1 - b0;
            q.j = j0 + s;
        }
    }
    return true;
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
__device__ __forceinline__ void producer(const Params& P, int ph0, int ph1, int n, unsigned starts, const Smem& sm)
{
    constexpr unsigned NS = nstage_for(BG);
    const uint64_t pol = l2_evict_first();
    unsigned s = 0;
    bool ok = true;
    const int dep_end = P.dep_ph0 + n_groups(starts) * P.dep_ph_stride;
    const int dep_all = P.dep_ph0 + P.S * P.dep_ph_stride;
    for (int ph = ph0; ph < ph1 && ok; ++ph) {
        if (ph == dep_end && dep_end < dep_all) {
            ph = dep_all - 1;  // nothing to stream for absent groups
            continue;
        }
        const TW* W;
        int N, K, c, cnt;
        Phase q = P.phases[ph];
        if (!resolve(P, starts, q, c, cnt)) continue;
        if (!phase_matrix<TW>(P, q, W, N, K)) continue;
        int r0, r1;
        cta_rows(N, cnt, c, r0, r1);
        const int rps = rows_per_stage<TW>(K);
        const int bgv = group_size<BG>(K);
        for (int b0 = 0; b0 < n && ok; b0 += bgv) {
            for (int r = r0; r < r1; r += rps, ++s) {
                const int rows = min(rps, r1 - r);
                const unsigned bytes = (unsigned)(rows * K * (int)sizeof(TW));
                const int slot = (int)(s % NS);
                if (!mbar_wait(&sm.empty[slot], ((s / NS) & 1u) ^ 1u, P.err, WS_EMPTY)) { ok = false; break; }
                mbar_expect_tx(&sm.full[slot], bytes);
                bulk_g2s(sm.ring + (size_t)slot * STAGE_BYTES, W + (size_t)r * K, bytes, &sm.full[slot], pol);
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
    const uint2* base;    // batch row i at base + i * stride (tagged)
    long long stride;
    unsigned tag;         // tag the input must carry
    const float* g;       // RMSNorm gain, or nullptr for no norm
    const void* add;      // depformer embedding table (weight dtype) or nullptr
    long long add_stride; // row length of that table (elements)
    uint2* store;         // stores base + add here (depformer residual; one CTA per substep), or nullptr
    unsigned store_tag;
    long long store_stride;
    int dj, dj0;          // depformer substep and its group's first substep (when add != nullptr)
    unsigned am_tag;      // tag of the argmax partials the group's first substep reads
    int am_cnt;           // and their count
};

// argmax partials of batch row i from every CTA (one warp; every lane gets the
// same result; the tie rule makes the combine order irrelevant).  -1: gave up.
__device__ __forceinline__ int argmax_partials_warp(const Params& P, const uint2* parts, int cnt, unsigned tag)
{
    const int lane = threadIdx.x & 31;
    float v = -INFINITY;
    int ix = 0x7fffffff;
    bool ok = true;
    for (int c = lane; c < cnt && ok; c += 32) {
        const uint2* e = parts + (size_t)c * 2;
        unsigned vb = 0, ib = 0;
        ok = wait_tag1(e, tag, vb, P.err) && wait_tag1(e + 1, tag, ib, P.err);
        if (ok && am_better(__uint_as_float(vb), (int)ib, v, ix)) { v = __uint_as_float(vb); ix = (int)ib; }
    }
    if (!__all_sync(0xffffffffu, ok)) return -1;
    warp_argmax(v, ix);
    return ix == 0x7fffffff ? 0 : ix;
}

// ------------------------------------------------------------------ sampling heads
// Temperature + top-k draw for one logit row, by every consumer thread of the
// CTA: candidates are the k largest logits (ties to the lower index), weighted
// exp((logit - max) / T); the token is the first candidate, in ascending index
// order, at which the running sum of weights exceeds u times their total.  The
// k-th largest key comes from a three-level radix select (11, 11, 10 bits);
// each thread owns a contiguous run of indices, so thread order is index order.

__device__ __forceinline__ unsigned order_key(float f)
{
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// exclusive scan of one value per consumer thread, in thread order
template <typename T>
__device__ __forceinline__ T cta_exclusive_scan(T v, T& total, T* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    csync();
    T before = 0, tot = 0;
    for (int w = 0; w < NWARP; ++w) {
        const T sw = scratch[w];
        if (w < warp) before += sw;
        tot += sw;
    }
    csync();
    total = tot;
    return before + x - v;
}

// Among the keys whose bits above pre_shift equal `pre` (pre_shift 32: all),
// the digit of width `bits` at `shift` holding the rank-th largest (1-based);
// rank becomes the rank inside that digit.
__device__ __forceinline__ int radix_level(const float* lg, int c0, int c1, unsigned pre, int pre_shift, int shift, int bits,
                                           int& rank, unsigned* hist, unsigned* scratch, int* misc)
{
    const int nb = 1 << bits;
    for (int b = threadIdx.x; b < nb; b += NT) hist[b] = 0u;
    csync();
    for (int i = c0; i < c1; ++i) {
        const unsigned key = order_key(__ldcg(lg + i));
        if (pre_shift >= 32 || (key >> pre_shift) == pre) atomicAdd(&hist[(key >> shift) & (unsigned)(nb - 1)], 1u);
    }
    csync();
    const int per = nb / NT;                      // digits per thread; thread 0 owns the largest
    const int d0 = nb - (threadIdx.x + 1) * per;
    unsigned sum = 0u;
    for (int q = 0; q < per; ++q) sum += hist[d0 + q];
    unsigned total;
    const unsigned above = cta_exclusive_scan(sum, total, scratch);
    if (above < (unsigned)rank && (unsigned)rank <= above + sum) {
        unsigned acc = above;
        for (int q = per - 1; q >= 0; --q) {
            const unsigned h = hist[d0 + q];
            if ((unsigned)rank <= acc + h) {
                misc[0] = d0 + q;
                misc[1] = rank - (int)acc;
                break;
            }
            acc += h;
        }
    }
    csync();
    rank = misc[1];
    return misc[0];
}

__device__ __noinline__ int sample_topk_cta(const float* lg, int N, float inv_t, int k, float u, const Smem& sm)
{
    unsigned* hist = (unsigned*)sm.red;         // [2048]
    unsigned* su = (unsigned*)sm.amv;           // [NWARP] scan scratch
    float* sf = sm.amv;
    int* misc = sm.misc + 4;                    // [4]
    const int CH = (N + NT - 1) / NT;
    const int c0 = min(N, (int)threadIdx.x * CH), c1 = min(N, c0 + CH);
    if (k > N) k = N;
    float mx = -INFINITY;
    for (int i = c0; i < c1; ++i) mx = fmaxf(mx, __ldcg(lg + i));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) sf[threadIdx.x >> 5] = mx;
    csync();
    mx = sf[0];
    for (int w = 1; w < NWARP; ++w) mx = fmaxf(mx, sf[w]);
    csync();
    int rank = k;
    const unsigned b1 = (unsigned)radix_level(lg, c0, c1, 0u, 32, 21, 11, rank, hist, su, misc);
    const unsigned b2 = (unsigned)radix_level(lg, c0, c1, b1, 21, 10, 11, rank, hist, su, misc);
    const unsigned b3 = (unsigned)radix_level(lg, c0, c1, (b1 << 11) | b2, 10, 0, 10, rank, hist, su, misc);
    const unsigned kth = (b1 << 21) | (b2 << 10) | b3;
    const unsigned need_eq = (unsigned)rank;    // candidates among the keys equal to kth, lowest indices first
    unsigned ceq = 0u;
    for (int i = c0; i < c1; ++i) ceq += order_key(__ldcg(lg + i)) == kth;
    unsigned eq_tot;
    const unsigned eq_before = cta_exclusive_scan(ceq, eq_tot, su);
    float ws = 0.f;
    int last = -1;
    {
        unsigned e = eq_before;
        for (int i = c0; i < c1; ++i) {
            const float v = __ldcg(lg + i);
            const unsigned key = order_key(v);
            bool in = key > kth;
            if (key == kth) in = e++ < need_eq;
            if (in) {
                ws += expf((v - mx) * inv_t);
                last = i;
            }
        }
    }
    float wtot;
    const float wbefore = cta_exclusive_scan(ws, wtot, sf);
    const float target = u * wtot;
    if (threadIdx.x == 0) { misc[2] = 0x7fffffff; misc[3] = -1; }
    csync();
    if (last >= 0) atomicMax(&misc[3], last);
    if (ws > 0.f && wbefore + ws > target) {
        float run = wbefore;
        unsigned e = eq_before;
        for (int i = c0; i < c1; ++i) {
            const float v = __ldcg(lg + i);
            const unsigned key = order_key(v);
            bool in = key > kth;
            if (key == kth) in = e++ < need_eq;
            if (in) {
                run += expf((v - mx) * inv_t);
                if (run > target) {
                    atomicMin(&misc[2], i);
                    break;
                }
            }
        }
    }
    csync();
    const int tok = misc[2] != 0x7fffffff ? misc[2] : misc[3];  // u * total rounded up to the total: the last candidate
    csync();
    return tok;
}

// Sampling of row i's head for stream k (0: text) in this step, or false for greedy.
__device__ __forceinline__ bool sampling_on(const Params& P, int i, int k, float& inv_t, int& topk)
{
    const StepDesc* D = P.desc;
    if (!D->sampled) return false;
    const SampleCfg cfg = P.samp[D->slot[i]];
    inv_t = k == 0 ? cfg.text_inv_t : cfg.audio_inv_t;
    topk = k == 0 ? cfg.text_k : cfg.audio_k;
    return topk > 1 && inv_t > 0.f;
}

// Logits of row i's head for stream k (0: the text head; k >= 1: substep k-1's head).
__device__ __forceinline__ const float* head_logits(const Params& P, int i, int k, int& N)
{
    if (k == 0) {
        N = P.V;
        return P.logits + (size_t)i * P.V;
    }
    N = P.C;
    return P.dlogits + ((size_t)i * P.S + (k - 1)) * P.C;
}

// Input token of depformer substep j for each batch row: the token supplied
// for stream j (this frame, or the frame before for a delayed stream) if any,
// else, at a group's first substep only, the argmax of the head before it (the
// text head for j = 0).  Rows b0 .. b0+nb-1 (nb <= NWARP) land in
// sm.prev[poff ..].  Every consumer thread calls it; false if a wait gave up.
__device__ __forceinline__ bool dep_select_inputs(const Params& P, const XSrc& xs, int b0, int nb, const Smem& sm,
                                                  int poff = 0)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = xs.dj;
    int ok = 1;
    const bool sampled = P.desc->sampled != 0;
    if (warp < nb) {
        const int i = b0 + warp;
        int chosen = supplied_token(P, i, j);
        const bool generated = chosen < 0;
        if (chosen < 0 && j == xs.dj0) {
            const uint2* parts = j == 0 ? P.amax + (size_t)i * P.G * 2 : P.damax + ((size_t)i * P.S + (j - 1)) * P.G * 2;
            chosen = argmax_partials_warp(P, parts, xs.am_cnt, xs.am_tag);
            ok = chosen >= 0;
        }
        const int lim = j == 0 ? P.V : P.C;
        if (lane == 0) sm.prev[poff + warp] = (chosen >= 0 && chosen < lim) ? chosen : 0;  // keeps the embedding read in range
        float it_;
        int ik_;
        if (lane == 0) sm.misc[8 + poff + warp] = sampled && generated && j == xs.dj0 && sampling_on(P, i, j, it_, ik_);
    }
    if (!csync_and(ok)) return false;
    // rows that draw their token: every CTA draws the same one from the head's logits
    // (written before the partials were published, which the argmax wait saw)
    for (int b = 0; b < nb && sampled; ++b) {
        if (!sm.misc[8 + poff + b]) continue;
        __threadfence();
        const int i = b0 + b;
        float inv_t;
        int topk, N;
        sampling_on(P, i, j, inv_t, topk);
        const float* lg = head_logits(P, i, j, N);
        const int tok = sample_topk_cta(lg, N, inv_t, topk, P.unif[(size_t)i * NSTREAM + j], sm);
        if (threadIdx.x == 0) {
            const int lim = j == 0 ? P.V : P.C;
            sm.prev[poff + b] = (tok >= 0 && tok < lim) ? tok : 0;
            if (blockIdx.x == 0) P.drawn[(size_t)i * NSTREAM + j] = tok;
        }
        csync();
    }
    return true;
}

// Consume one batch group [b0, b0+nb) of a matrix-vector phase: leaves the
// CTA's row values in sm.yf[(r - r0) * bgv + b].  `stage` counts ring stages.
template <typename TW, int VPL, int BGV, int BG_OF_STAGES>
__device__ __forceinline__ bool gemv_group(const Params& P, const Phase& ph, int K, const GemvCfg& c, int r0, int r1,
                                           const XSrc& xs, int b0, int nb, const Smem& sm, unsigned& stage)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kw = warp % c.nwk, rw = warp / c.nwk;
    const int NV = K / 8;
    const int v_begin = kw * c.nvw;
    const int v_end = min(NV, v_begin + c.nvw);
    // this warp's K-slice of the input in registers, waiting for its tags and
    // multiplied by the norm gain; sums of squares of the raw input
    float xr[VPL][BGV][8];
    float ssq[BGV];
#pragma unroll
    for (int b = 0; b < BGV; ++b) ssq[b] = 0.f;
    const bool gain_now = xs.g && !xs.add;
    int ok = 1;
    // first pass issues every vector's loads (in chunks of 4 vectors), then checks
    constexpr int NVEC = VPL * BGV;
    constexpr int CH = NVEC < 4 ? NVEC : 4;
#pragma unroll
    for (int c0 = 0; c0 < NVEC; c0 += CH) {
        uint2 pend[CH][8];
#pragma unroll
        for (int q = 0; q < CH; ++q) {
            const int t = (c0 + q) / BGV, b = (c0 + q) % BGV;
            const int v = v_begin + lane + 32 * t;
#pragma unroll
            for (int k = 0; k < 8; ++k) pend[q][k] = make_uint2(0u, 0u);
            if (c0 + q < NVEC && v < v_end && b < nb) tag8_issue(xs.base + (size_t)(b0 + b) * xs.stride + v * 8, pend[q]);
        }
#pragma unroll
        for (int q = 0; q < CH; ++q) {
            if (c0 + q >= NVEC) break;
            const int t = (c0 + q) / BGV, b = (c0 + q) % BGV;
            const int v = v_begin + lane + 32 * t;
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 0.f;
            if (v < v_end && b < nb && ok) ok = tag8_take(pend[q], xs.base + (size_t)(b0 + b) * xs.stride + v * 8, xs.tag, f, P.err);
            float gg[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) gg[e] = 1.f;
            if (gain_now && v < v_end) {
                const float4* gs = reinterpret_cast<const float4*>(xs.g + v * 8);
                const float4 g0 = __ldg(gs), g1 = __ldg(gs + 1);
                gg[0] = g0.x; gg[1] = g0.y; gg[2] = g0.z; gg[3] = g0.w; gg[4] = g1.x; gg[5] = g1.y; gg[6] = g1.z; gg[7] = g1.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ssq[b] = fmaf(f[e], f[e], ssq[b]);
                xr[t][b][e] = f[e] * gg[e];
            }
        }
    }
    // depformer layer 0: the input adds the embedding of the token chosen by the
    // previous head; then the gain
    if (xs.add) {
        if (!dep_select_inputs(P, xs, b0, nb, sm)) ok = 0;
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
        if (xs.store && rw == 0) {
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const int v = v_begin + lane + 32 * t;
#pragma unroll
                for (int b = 0; b < BGV; ++b) {
                    if (v < v_end && b < nb) {
                        uint2* dst = xs.store + (size_t)(b0 + b) * xs.store_stride + v * 8;
#pragma unroll
                        for (int e = 0; e < 8; e += 2) st_tag2(dst + e, xr[t][b][e], xr[t][b][e + 1], xs.store_tag);
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
        // RMSNorm: sums of squares per K-slice; the factor (a scalar per batch
        // row) multiplies the row sums after the weight stages, so no warp waits
        // for the others' inputs before streaming
#pragma unroll
        for (int b = 0; b < BGV; ++b) {
            const float q = warp_sum(ssq[b]);
            if (lane == 0 && rw == 0) sm.ssq[b * 16 + kw] = q;
        }
    }
    if (P.ptime) stamp(P, sm.misc[0], 1);

    // stream the CTA's rows through the ring: each warp takes rows rw, rw+nwr, ...
    // of a stage, four at a time, and releases the stage on its own
    constexpr unsigned NS = nstage_for(BG_OF_STAGES);
    const int rps = rows_per_stage<TW>(K);
    for (int ra = r0; ra < r1; ra += rps, ++stage) {
        const int nr = min(rps, r1 - ra);
        const int slot = (int)(stage % NS);
        const unsigned long long tw0 = P.ptime ? globaltimer_ns() : 0ull;
        if (!mbar_wait(&sm.full[slot], (stage / NS) & 1u, P.err, WS_FULL)) {
            ok = 0;  // every thread leaves through the barrier below, whichever stage it reached
            break;
        }
        if (P.ptime && blockIdx.x == 0 && threadIdx.x == 0) {
            // diagnostics: time CTA 0 spent waiting for weight stages, and their count
            // (fire-and-forget reductions: the warp does not wait on them)
            atomicAdd(P.ptime + (size_t)sm.misc[0] * 8 + 4, globaltimer_ns() - tw0);
            atomicAdd(P.ptime + (size_t)sm.misc[0] * 8 + 5, 1ull);
        }
        const TW* ring = (const TW*)(sm.ring + (size_t)slot * STAGE_BYTES);
        // copy this warp's rows of the stage into registers, release the stage at
        // once (the producer refills it while the arithmetic runs), then compute
        constexpr int RW = rows_per_warp_cap(VPL);  // rows per warp per stage, at most (checked at create)
        constexpr int U4 = sizeof(TW) == 2 ? 1 : 2;  // 16-byte words per vector of 8 weights
        uint4 wv[RW][VPL][U4];
#pragma unroll
        for (int q = 0; q < RW; ++q) {
            const int rr = rw + q * c.nwr;
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const int v = v_begin + lane + 32 * t;
#pragma unroll
                for (int h = 0; h < U4; ++h) {
                    wv[q][t][h] = make_uint4(0u, 0u, 0u, 0u);
                    if (rr < nr && v < v_end)
                        wv[q][t][h] = *reinterpret_cast<const uint4*>(ring + (size_t)rr * K + (size_t)v * 8 + h * 4);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
#pragma unroll
        for (int q0 = 0; q0 < RW; q0 += 4) {
            if (rw + q0 * c.nwr < nr) {  // warp-uniform
            // independent packed accumulators per (row, vector): even and odd
            // elements of each vector accumulate separately, combined in fixed order
            float2 acc2[4][BGV];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int b = 0; b < BGV; ++b) acc2[q][b] = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = rw + (q0 + q) * c.nwr;
                if (rr < nr) {
#pragma unroll
                    for (int t = 0; t < VPL; ++t) {
                        const int v = v_begin + lane + 32 * t;
                        if (v < v_end) {
                            float f[8];
                            if (U4 == 1) {
                                const uint4 w4 = wv[q0 + q][t][0];
                                f[0] = bf_lo(w4.x); f[1] = bf_hi(w4.x); f[2] = bf_lo(w4.y); f[3] = bf_hi(w4.y);
                                f[4] = bf_lo(w4.z); f[5] = bf_hi(w4.z); f[6] = bf_lo(w4.w); f[7] = bf_hi(w4.w);
                            } else {
                                const uint4 a = wv[q0 + q][t][0], b4 = wv[q0 + q][t][U4 - 1];
                                f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y); f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
                                f[4] = __uint_as_float(b4.x); f[5] = __uint_as_float(b4.y); f[6] = __uint_as_float(b4.z); f[7] = __uint_as_float(b4.w);
                            }
#pragma unroll
                            for (int b = 0; b < BGV; ++b)
#pragma unroll
                                for (int e = 0; e < 8; e += 2) ffma2(acc2[q][b], f[e], f[e + 1], xr[t][b][e], xr[t][b][e + 1]);
                        }
                    }
                }
            }
            float acc[4][BGV];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int b = 0; b < BGV; ++b) {
                    acc[q][b] = acc2[q][b].x + acc2[q][b].y;
                }
            // transposed butterfly: lanes 0, 8, 16, 24 end with the sums of rows q0..q0+3
            const int myq = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            const int rr = rw + (q0 + myq) * c.nwr;
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
                if ((lane & 7) == 0 && rr < nr) sm.red[((size_t)(ra - r0 + rr) * BGV + b) * NWARP + kw] = t;
            }
            }
        }
    }
    if (P.ptime) stamp(P, sm.misc[0], 2);
    if (!csync_and(ok)) return false;
    // sum the K-slices in slice order; then the RMSNorm factor, its sums of
    // squares also combined in slice order
    for (int it = tid; it < (r1 - r0) * nb; it += NT) {
        const int rl = it / nb, b = it % nb;
        const float* rp = sm.red + ((size_t)rl * BGV + b) * NWARP;
        float y = 0.f;
        for (int k = 0; k < c.nwk; ++k) y += rp[k];
        if (xs.g) {
            float tot = 0.f;
            for (int k = 0; k < c.nwk; ++k) tot += sm.ssq[b * 16 + k];
            y *= rsqrtf(tot / (float)K + P.eps);
        }
        sm.yf[(size_t)rl * BGV + b] = y;
    }
    csync();
    return true;
}

// ------------------------------------------------------------------ epilogues

// An epilogue sees the CTA's rows [r0, r1) for batch rows b0..b0+nb-1, values
// in sm.yf[(row - r0) * bgv + b].  pre() runs before the weight stages and
// loads what apply() needs (up to two items per thread) so that the epilogue
// rarely waits on memory; empty() publishes what a CTA without rows owes.
struct Pre {
    float a[2], b[2];
    int ok;
};

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

template <typename TKV>
struct EpiQKV {
    int l;
    unsigned tag;
    __device__ Pre pre(const Params& P, int r0, int r1, int b0, int nb) const
    {
        Pre q{{0.f, 0.f}, {0.f, 0.f}, 1};
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
    __device__ void empty(const Params&, int, int) const {}
    __device__ bool apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre& q) const
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
                st_tag2(P.q + (size_t)i * d + e, y0, y1, tag);
            } else {
                // the ring keeps the key/value for later steps; this step's attention reads
                // the same (rounded) numbers from the tagged copy
                const int slot = D->slot[i];
                // ring [slot][layer][head][position mod W][hd]: a head's window is one contiguous run
                const long long idx = ((((long long)slot * P.L + l) * P.H + e / hd) * P.W + (p % P.W)) * (long long)hd + e % hd;
                KV<TKV>::store2(part == 1 ? P.kc : P.vc, idx, y0, y1);
                st_tag2((part == 1 ? P.kcur : P.vcur) + (size_t)i * d + e, KV<TKV>::round(y0), KV<TKV>::round(y1), tag);
            }
        }
        return true;
    }
};

// dst[row] = residual + row value; the residual (tag res_tag) is read in pre()
struct EpiResid {
    uint2* dst;
    long long stride;
    unsigned res_tag, tag;
    __device__ Pre pre(const Params& P, int r0, int r1, int b0, int nb) const
    {
        Pre q{{0.f, 0.f}, {0.f, 0.f}, 1};
        uint2 e[2] = {make_uint2(0u, res_tag), make_uint2(0u, res_tag)};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int it = threadIdx.x + k * NT;
            if (it < (r1 - r0) * nb) e[k] = ld_tag1(dst + (size_t)(b0 + it % nb) * stride + r0 + it / nb);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int it = threadIdx.x + k * NT;
            unsigned bits = e[k].x;
            if (it < (r1 - r0) * nb && e[k].y != res_tag && q.ok)
                q.ok = wait_tag1(dst + (size_t)(b0 + it % nb) * stride + r0 + it / nb, res_tag, bits, P.err);
            q.a[k] = __uint_as_float(bits);
        }
        return q;
    }
    __device__ void empty(const Params&, int, int) const {}
    // Tensor-core tiles (up to MMA_M rows x 32 batch rows): every residual of the
    // thread in flight at once, rows consecutive across threads.
    __device__ bool apply_all(const Params& P, const Smem& sm, int r0, int r1, int nb, int bgv) const
    {
        constexpr int MAXI = MMA_M * 32 / NT;
        const int rows = r1 - r0, items = rows * nb;
        uint2 e[MAXI];
#pragma unroll
        for (int k = 0; k < MAXI; ++k) {
            const int it = threadIdx.x + k * NT;
            e[k] = make_uint2(0u, res_tag);
            if (it < items) e[k] = ld_tag1(dst + (size_t)(it / rows) * stride + r0 + it % rows);
        }
        bool ok = true;
#pragma unroll
        for (int k = 0; k < MAXI; ++k) {
            const int it = threadIdx.x + k * NT;
            if (it < items) {
                const int b = it / rows, rl = it % rows;
                uint2* p = dst + (size_t)b * stride + r0 + rl;
                unsigned bits = e[k].x;
                if (e[k].y != res_tag && ok) ok = wait_tag1(p, res_tag, bits, P.err);
                st_tag1(p, __float_as_uint(__uint_as_float(bits) + sm.yf[(size_t)rl * bgv + b]), tag);
            }
        }
        return ok;
    }
    __device__ bool apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre& q) const
    {
        bool ok = true;
        for (int it = threadIdx.x; it < (r1 - r0) * nb && ok; it += NT) {
            const int rl = it / nb, b = it % nb;
            uint2* p = dst + (size_t)(b0 + b) * stride + r0 + rl;
            const int k = it / NT;
            float res = q.a[k < 2 ? k : 0];
            if (k >= 2) {
                unsigned bits = 0;
                ok = wait_tag1(p, res_tag, bits, P.err);
                res = __uint_as_float(bits);
            }
            st_tag1(p, __float_as_uint(res + sm.yf[(size_t)rl * bgv + b]), tag);
        }
        return ok;
    }
};

// rows are (gate m, up m) pairs
struct EpiSwiglu {
    uint2* dst;
    long long stride;
    unsigned tag;
    __device__ Pre pre(const Params&, int, int, int, int) const { return Pre{{0.f, 0.f}, {0.f, 0.f}, 1}; }
    __device__ void empty(const Params&, int, int) const {}
    __device__ bool apply(const Params&, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre&) const
    {
        const int npair = (r1 - r0) / 2;
        for (int it = threadIdx.x; it < npair * nb; it += NT) {
            const int pl = it / nb, b = it % nb;
            const float g = sm.yf[(size_t)(2 * pl) * bgv + b], u = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
            st_tag1(dst + (size_t)(b0 + b) * stride + r0 / 2 + pl, __float_as_uint(silu(g) * u), tag);
        }
        return true;
    }
};

// Rows [0, nlog) are logits (stored for diagnostics; the CTA's argmax per
// batch row goes to amax[i][cta], tagged); rows >= nlog go to extra[i][row - nlog].
struct EpiLogits {
    float* lg;
    long long lg_stride;
    int nlog;
    uint2* extra;
    long long extra_stride;
    unsigned tag;
    uint2* am;            // argmax partials: batch row i, this CTA at am + i * am_stride + am_idx * 2
    long long am_stride;
    int am_idx;
    float* dv = nullptr;  // deferred (several tiles per CTA): best value / index per batch row, published by flush()
    int* di = nullptr;
    __device__ Pre pre(const Params&, int, int, int, int) const { return Pre{{0.f, 0.f}, {0.f, 0.f}, 1}; }
    __device__ void flush(const Params& P, int b0, int nb) const
    {
        if (P.desc->sampled) __threadfence();
        if (threadIdx.x < nb) publish(P, b0 + threadIdx.x, dv[threadIdx.x], di[threadIdx.x]);
    }
    __device__ void publish(const Params& P, int i, float v, int ix) const
    {
        uint2* e = am + (size_t)i * am_stride + (size_t)am_idx * 2;
        st_tag1(e, __float_as_uint(v), tag);
        st_tag1(e + 1, (unsigned)ix, tag);
    }
    __device__ void empty(const Params& P, int b0, int nb) const
    {
        if (threadIdx.x < nb) publish(P, b0 + threadIdx.x, -INFINITY, 0x7fffffff);
    }
    // Tensor-core tile (deferred mode): store the tile's logits / extra rows, then
    // warp w merges the tile's argmax of batch rows w, w + NWARP, ... into dv / di.
    __device__ bool apply_tile(const Params& P, const Smem& sm, int r0, int r1, int nb, int bgv) const
    {
        const int rows = r1 - r0;
        for (int it = threadIdx.x; it < rows * nb; it += NT) {
            const int b = it / rows, rl = it % rows, r = r0 + rl;
            const float y = sm.yf[(size_t)rl * bgv + b];
            if (r < nlog) lg[(size_t)b * lg_stride + r] = y;
            else if (extra) st_tag1(extra + (size_t)b * extra_stride + (r - nlog), __float_as_uint(y), tag);
        }
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int b = warp; b < nb; b += NWARP) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int rl = lane; rl < rows; rl += 32) {
                const int r = r0 + rl;
                if (r >= nlog) break;
                const float y = sm.yf[(size_t)rl * bgv + b];
                if (am_better(y, r, bv, bi)) { bv = y; bi = r; }
            }
            warp_argmax(bv, bi);
            if (lane == 0 && am_better(bv, bi, dv[b], di[b])) { dv[b] = bv; di[b] = bi; }
        }
        return true;
    }
    __device__ bool apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre&) const
    {
        const int rows = r1 - r0;
        for (int it = threadIdx.x; it < rows * nb; it += NT) {
            const int rl = it / nb, b = it % nb;
            const int r = r0 + rl;
            const float y = sm.yf[(size_t)rl * bgv + b];
            if (r < nlog) lg[(size_t)(b0 + b) * lg_stride + r] = y;
            else if (extra) st_tag1(extra + (size_t)(b0 + b) * extra_stride + (r - nlog), __float_as_uint(y), tag);
        }
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        if (P.desc->sampled) __threadfence();  // a sampled step reads the logits once the partials announce them
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
                if (dv) {
                    if (am_better(v, ix, dv[b], di[b])) { dv[b] = v; di[b] = ix; }
                } else {
                    publish(P, b0 + b, v, ix);
                }
            }
        }
        return true;
    }
};

// depformer q to dq, k and v of substep j to the layer's substep cache
struct EpiDQKV {
    int l, j;
    unsigned tag;
    __device__ Pre pre(const Params&, int, int, int, int) const { return Pre{{0.f, 0.f}, {0.f, 0.f}, 1}; }
    __device__ void empty(const Params&, int, int) const {}
    __device__ bool apply(const Params& P, const Smem& sm, int r0, int r1, int b0, int nb, int bgv, const Pre&) const
    {
        const int dd = P.dd;
        const int npair = (r1 - r0) / 2;
        for (int it = threadIdx.x; it < npair * nb; it += NT) {
            const int pl = it / nb, b = it % nb, i = b0 + b;
            const int r = r0 + 2 * pl;
            const int part = r / dd, e = r - part * dd;
            const float y0 = sm.yf[(size_t)(2 * pl) * bgv + b];
            const float y1 = sm.yf[(size_t)(2 * pl + 1) * bgv + b];
            uint2* dst = part == 0 ? P.dq + ((size_t)i * P.S + j) * dd + e
                                   : P.dkv + ((((size_t)i * P.dL + l) * P.S + j) * 2 + (part - 1)) * dd + e;
            st_tag2(dst, y0, y1, tag);
        }
        return true;
    }
};

// One matrix-vector phase; the epilogue consumes the CTA's rows.
template <typename TW, int BG, class Epi>
__device__ __forceinline__ bool gemv_phase(const Params& P, const Phase& ph, int cta, int cnt, const XSrc& xs, int n,
                                           const Smem& sm, unsigned& stage, const Epi& epi)
{
    const TW* W;
    int N, K;
    phase_matrix<TW>(P, ph, W, N, K);
    int r0, r1;
    cta_rows(N, cnt, cta, r0, r1);
    const GemvCfg c = gemv_cfg(K);
    const int bgv = group_size<BG>(K);
    for (int b0 = 0; b0 < n; b0 += bgv) {
        const int nb = min(bgv, n - b0);
        if (r1 > r0 || xs.store) {
            const Pre pre = epi.pre(P, r0, r1, b0, nb);
            bool ok;
            switch (vpl_class(c.vpl)) {
                case 1: ok = gemv_group<TW, 1, BG, BG>(P, ph, K, c, r0, r1, xs, b0, nb, sm, stage); break;
                case 2: ok = gemv_group<TW, 2, BG, BG>(P, ph, K, c, r0, r1, xs, b0, nb, sm, stage); break;
                default: ok = gemv_group<TW, 6, (BG < 2 ? BG : 2), BG>(P, ph, K, c, r0, r1, xs, b0, nb, sm, stage); break;
            }
            if (!csync_and(ok && pre.ok)) return false;
            if (!csync_and(epi.apply(P, sm, r0, r1, b0, nb, bgv, pre))) return false;
        } else {
            epi.empty(P, b0, nb);
        }
    }
    return true;
}

// ------------------------------------------------------------------ rows and attention items

// First and last row of row i's slot (rows of a slot are consecutive).
__device__ __forceinline__ int slot_first_row(const StepDesc* D, int i)
{
    while (i > 0 && D->slot[i - 1] == D->slot[i]) --i;
    return i;
}

__device__ __forceinline__ int slot_last_row(const StepDesc* D, int n, int i)
{
    while (i + 1 < n && D->slot[i + 1] == D->slot[i]) ++i;
    return i;
}

// Chunks of a window of len keys: about 64 keys each, but no more than the
// grid holds for one slot's heads at once (G / H), nor NCHUNK_MAX.  A function
// of the slot's own window and the context's shape only, so a slot's result
// never depends on the other slots of the step.
__device__ __forceinline__ int attn_chunks(int len, int G, int H)
{
    int c = (len + 63) / 64;
    const int cap = G / H > 1 ? G / H : 1;
    c = c < cap ? c : cap;
    // long windows: chunks of at most about 384 keys (more, shorter items keep
    // every CTA busy when the windows of many slots are long)
    const int clong = (len + 383) / 384;
    c = c > clong ? c : clong;
    return c < NCHUNK_MAX ? c : NCHUNK_MAX;
}

// Keys per stage when the producer streams a head's keys and values through the
// tensor-core stages (keys, then values, bf16), and stages per item.
__device__ __forceinline__ int attn_stage_keys(int hd) { return MMA_STAGE / (2 * hd * 2); }
constexpr int ATTN_STAGES_PER_ITEM = 7;

// Chunks of a window when its keys are streamed through the stages: at most
// ATTN_STAGES_PER_ITEM stages each, at most NCHUNK_MAX.  A function of the window only.
__device__ __forceinline__ int attn_chunks_stream(int len, int hd, int ipc)
{
    const int per = attn_stage_keys(hd) * ipc;
    const int c = (len + per - 1) / per;
    return c < NCHUNK_MAX ? c : NCHUNK_MAX;
}

enum AttnMode : int { ATTN_CTA = 0, ATTN_STREAM = 2 };

// Work items of the step's attention: (batch row i, head h, chunk c), row-major.
__device__ __forceinline__ int attn_nchunks(int mode, int len, int G, int H, int hd, int ipc)
{
    return mode == ATTN_STREAM ? attn_chunks_stream(len, hd, ipc) : attn_chunks(len, G, H);
}

// Stages per streamed attention item: the phase's stages spread over about six
// items per CTA (fewer items, fewer per-item costs; enough of them to balance
// the CTAs), at least ATTN_STAGES_PER_ITEM.  Every caller computes the same value.
__device__ __forceinline__ int attn_stream_ipc(const StepDesc* D, int n, int W, int H, int hd, int G)
{
    const int kps = attn_stage_keys(hd);
    long long st = 0;
    for (int i = 0; i < n; ++i) {
        const int p = D->pos[i];
        st += ((p + 1 < W ? p + 1 : W) + kps - 1) / kps;
    }
    const long long want = (st * H + 6LL * G - 1) / (6LL * G);
    return (int)(want < ATTN_STAGES_PER_ITEM ? ATTN_STAGES_PER_ITEM : (want > 4096 ? 4096 : want));
}

__device__ __forceinline__ void attn_item(const StepDesc* D, int n, int H, int W, int G, int item, int& i, int& h,
                                          int& c, int& nch, int& len, int mode = ATTN_CTA, int hd = 0, int ipc = 0)
{
    int base = 0;
    for (i = 0; i < n; ++i) {
        const int p = D->pos[i];
        len = p + 1 < W ? p + 1 : W;
        nch = attn_nchunks(mode, len, G, H, hd, ipc);
        if (item < base + nch * H) break;
        base += nch * H;
    }
    const int r = item - base;
    h = r / nch;
    c = r % nch;
}

// A key range of one attention item streamed through the stages: item's
// chunk [k0, k1) minus this launch's keys (the last mcur of the window, which
// come from the tagged copies).
__device__ __forceinline__ void attn_stream_range(const StepDesc* D, int i, int len, int c, int nch, int& k0, int& k1,
                                                  int& kend, int& mcur)
{
    mcur = D->pos[i] - D->pos[slot_first_row(D, i)] + 1;
    k0 = (int)((long long)len * c / nch);
    k1 = (int)((long long)len * (c + 1) / nch);
    kend = min(k1, len - mcur);
}

// ------------------------------------------------------------------ tensor-core weight pass
// Batches of 5..32 rows with bf16 weights: every matrix phase is a product of
// the weight matrix (A, M rows x K) with the rows' activations (B, N rows x K,
// N = 3 x rows padded to 16 or 32: each activation is split into three bf16
// parts, so the product keeps about 27 significant bits of the fp32 input and
// the weights are read once for all rows).  tcgen05.mma accumulates in fp32 in
// tensor memory.
//
// Activations: at the start of a phase the CTAs sharing the matrix convert the
// input's 64-column K-chunks, each chunk once, into a global panel in the
// operand layout (gain applied, split, 128-byte swizzle), with the chunk's
// sums of squares per row, and publish a ready tag per chunk.
//
// A matrix is cut into units (tile of 128 rows, K-chunk of 64); CTA c of the
// cnt sharing the matrix takes the contiguous units [U c / cnt, U (c+1) / cnt)
// in tile-major order.  Per unit the producer warp loads the weight chunk with
// a 2-D TMA copy (128-byte swizzle) and the activation chunk with a 1-D bulk
// copy from the panel once its tag is there; the MMA warp issues 4 MMAs of
// K = 16.  A CTA owns the tiles whose last chunk lies in its range; the CTAs
// before it that hold earlier chunks of an owned tile leave partial sums
// tagged in global memory, and the owner adds them in K order, applies the
// RMSNorm factor from the chunks' sums of squares, and runs the epilogue.  The
// partition is a function of the shapes and the grid only, so results never
// depend on data outside the row.
//
// Buffer reuse: every chunk of a phase's input is converted once, and a tile's
// owner needs all of K, so any output of a phase follows every read of its
// input; each later writer of a buffer depends on such an output.  The panel
// and partial buffers rotate over MMA_ROT = 4 phases: a phase's buffers are
// rewritten four phases later, by which time every unit of the phase has
// completed (the chain through the phases in between needs every tile of it,
// attention phases included).  The one phase whose inputs need not depend on
// the phase before, a depformer group's first layer after another group, first
// waits until every CTA has finished that group's head (P.done).

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One warp, all lanes.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, unsigned ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, unsigned ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory operand descriptor: K-major rows of 128 bytes with the 128-byte
// swizzle, groups of 8 rows 1024 bytes apart (the layout a 2-D TMA copy of a
// 64-wide bf16 box writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(unsigned saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                             // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;                   // stride byte offset
    d |= (uint64_t)1 << 46;                             // descriptor version
    d |= (uint64_t)2 << 61;                             // 128-byte swizzle
    return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, A and B K-major, M = 128, N = ncol.
__device__ __forceinline__ uint32_t mma_idesc(int ncol)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(ncol >> 3) << 17) | ((uint32_t)(MMA_M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// The barrier completes once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3}], [%4], %5;"
                 ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

// nc consecutive fp32 columns of this warp's 32 lanes (one lane per thread).
template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[NC]);

template <>
__device__ __forceinline__ void tmem_ld<4>(uint32_t taddr, float (&v)[4])
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(r[e]);
}

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[e]);
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
}

// nc fp32 columns into this warp's 32 lanes of tensor memory.
template <int NC>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[16]);

template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                   "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])) : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                   "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                   "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                   "r"(__float_as_uint(v[15])) : "memory");
}

// This CTA's units of an M x K matrix.
struct MmaPart {
    int KC, T;
    int u0, u1;        // units [u0, u1) of T * KC, tile-major
    int t0, nt;        // first tile touched, tiles touched (0: none)
    bool last_owned;   // the last tile touched ends inside the range
};

__device__ __forceinline__ int mma_unit0(long long U, int c, int cnt) { return (int)(U * c / cnt); }

__device__ __forceinline__ MmaPart mma_part(int M, int K, int c, int cnt)
{
    MmaPart p;
    p.KC = (K + MMA_KC - 1) / MMA_KC;
    p.T = (M + MMA_M - 1) / MMA_M;
    const long long U = (long long)p.T * p.KC;
    p.u0 = mma_unit0(U, c, cnt);
    p.u1 = mma_unit0(U, c + 1, cnt);
    if (p.u1 > p.u0) {
        p.t0 = p.u0 / p.KC;
        const int tl = (p.u1 - 1) / p.KC;
        p.nt = tl - p.t0 + 1;
        p.last_owned = p.u1 == (tl + 1) * p.KC;
    } else {
        p.t0 = 0;
        p.nt = 0;
        p.last_owned = false;
    }
    return p;
}

// Activation chunk kc of substep slot `sub` (0 for temporal phases) in the panel of parity par.
__device__ __forceinline__ size_t panel_index(const Params& P, int par, int sub, int kc)
{
    return ((size_t)par * MAXGW + (size_t)sub) * (size_t)P.pchunks + (size_t)kc;
}

__device__ __forceinline__ int phase_sub(const Phase& q) { return q.type >= PH_DQKV && q.type <= PH_DHEAD ? q.j - q.pad0 : 0; }

// Producer warp (one lane), tensor-core instantiation: for every unit of every
// matrix phase of the launch, in the consumers' order, the weight chunk (2-D TMA
// from the tensor map) and the activation chunk (1-D bulk copy from the panel,
// once the CTA that converts it has published its tag).  Weights run ahead as
// soon as a stage is free; activation copies follow as their chunks appear.
template <typename TW>
__device__ __forceinline__ void producer_mma(const Params& P, int ph0, int ph1, int n, unsigned starts, const Smem& sm)
{
    const uint64_t pol_w = l2_evict_first();
    const uint64_t pol_b = l2_evict_last();  // a chunk serves every CTA whose range holds its K
    const unsigned bbytes = (unsigned)(MMA_PARTS * mma_nbp(n) * MMA_KC * 2);
    unsigned s = 0;
    bool ok = true;
    const int dep_end = P.dep_ph0 + n_groups(starts) * P.dep_ph_stride;
    const int dep_all = P.dep_ph0 + P.S * P.dep_ph_stride;
    for (int ph = ph0; ph < ph1 && ok; ++ph) {
        if (ph == dep_end && dep_end < dep_all) {
            ph = dep_all - 1;
            continue;
        }
        const TW* W;
        int M, K, c, cnt;
        Phase q = P.phases[ph];
        if (!resolve(P, starts, q, c, cnt)) continue;
        if (q.type == PH_ATTN) {
            // keys then values of every item of this CTA, one stage per attn_stage_keys positions
            // (read once: evict-first, like the weights)
            const StepDesc* D = P.desc;
            const int H = P.H, hd = P.hd, Wn = P.W, KPS = attn_stage_keys(hd);
            const int ipc = attn_stream_ipc(D, n, P.Wa, H, hd, P.G);
            int total = 0;
            for (int i = 0; i < n; ++i) total += attn_chunks_stream(D->pos[i] + 1 < P.Wa ? D->pos[i] + 1 : P.Wa, hd, ipc) * H;
            for (int item = blockIdx.x; item < total && ok; item += P.G) {
                int i, h, ci, nch, len, k0, k1, kend, mcur;
                attn_item(D, n, H, P.Wa, P.G, item, i, h, ci, nch, len, ATTN_STREAM, hd, ipc);
                attn_stream_range(D, i, len, ci, nch, k0, k1, kend, mcur);
                const int start = D->pos[i] - len + 1;
                const size_t hbase = (((size_t)D->slot[i] * P.L + q.l) * H + h) * (size_t)Wn * hd;
                for (int kb = k0; kb < kend; kb += KPS, ++s) {
                    const int nk = min(KPS, kend - kb);
                    const int slot = (int)(s % MMA_NSTAGE);
                    if (!mbar_wait(&sm.sempty[slot], ((s / MMA_NSTAGE) & 1u) ^ 1u, P.err, WS_EMPTY)) { ok = false; break; }
                    const unsigned kbytes = (unsigned)(nk * hd * sizeof(TW));
                    // the activation barrier's phase stays in step with the stage; it completes
                    // before the copies are issued, so the consumers that see the keys land have
                    // passed a completed phase of it too
                    mbar_arrive(&sm.bfull[slot]);
                    mbar_expect_tx(&sm.wfull[slot], 2 * kbytes);
                    const int r0 = (start + kb) % Wn, n1 = min(nk, Wn - r0);
                    char* dst = sm.mring + (size_t)slot * MMA_STAGE;
                    for (int t = 0; t < 2; ++t) {  // keys, then values at KPS keys' offset
                        const TW* ring = (const TW*)(t == 0 ? P.kc : P.vc) + hbase;
                        char* dt = dst + (size_t)t * KPS * hd * sizeof(TW);
                        bulk_g2s(dt, ring + (size_t)r0 * hd, (unsigned)(n1 * hd * sizeof(TW)), &sm.wfull[slot], pol_w);
                        if (n1 < nk)
                            bulk_g2s(dt + (size_t)n1 * hd * sizeof(TW), ring, (unsigned)((nk - n1) * hd * sizeof(TW)),
                                     &sm.wfull[slot], pol_w);
                    }
                }
            }
            continue;
        }
        if (!phase_matrix<TW>(P, q, W, M, K)) continue;
        const CUtensorMap* map = P.tmaps + tmap_index(q.type, q.l, q.j, P.L, P.dL);
        const MmaPart mp = mma_part(M, K, c, cnt);
        const size_t pbase = panel_index(P, ph % MMA_ROT, phase_sub(q), 0);
        const unsigned* flags = P.pflag + pbase;
        const char* chunks = P.panel + pbase * MMA_B_BYTES;
        const unsigned tag = phase_tag(P.desc, ph);
        int w = mp.u0, bq = mp.u0;  // next unit for the weights / for the activations
        const unsigned s0 = s;
        unsigned ready[(MAX_PCHUNKS + 31) / 32];  // bit kc: chunk kc seen ready in this phase
#pragma unroll
        for (int k = 0; k < (MAX_PCHUNKS + 31) / 32; ++k) ready[k] = 0u;
        Spin sp;
        while (bq < mp.u1) {
            bool progress = false;
            if (w < mp.u1 && w - bq < MMA_NSTAGE) {
                const unsigned sw = s0 + (unsigned)(w - mp.u0);
                const int slot = (int)(sw % MMA_NSTAGE);
                if (mbar_try(&sm.sempty[slot], ((sw / MMA_NSTAGE) & 1u) ^ 1u)) {
                    mbar_expect_tx(&sm.wfull[slot], MMA_W_BYTES);
                    tma_load_2d(sm.mring + (size_t)slot * MMA_STAGE, map, (w % mp.KC) * MMA_KC, (w / mp.KC) * MMA_M,
                                &sm.wfull[slot], pol_w);
                    ++w;
                    progress = true;
                }
            }
            if (bq < w) {
                const int kc = bq % mp.KC;
                if (!((ready[kc >> 5] >> (kc & 31)) & 1u)) {
                    // poll the 32 flags of kc's word at once (one round trip), then acquire
                    const int k0 = kc & ~31;
                    unsigned f[32], got = 0u;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        f[e] = 0u;
                        if (k0 + e < mp.KC)
                            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(f[e]) : "l"(flags + k0 + e) : "memory");
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) got |= (f[e] == tag ? 1u : 0u) << e;
                    if (got & ~ready[kc >> 5]) {
                        asm volatile("fence.acq_rel.gpu;" ::: "memory");
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        ready[kc >> 5] |= got;
                    }
                }
                if ((ready[kc >> 5] >> (kc & 31)) & 1u) {
                    const int slot = (int)((s0 + (unsigned)(bq - mp.u0)) % MMA_NSTAGE);
                    mbar_expect_tx(&sm.bfull[slot], bbytes);
                    bulk_g2s(sm.mring + (size_t)slot * MMA_STAGE + MMA_W_BYTES, chunks + (size_t)kc * MMA_B_BYTES, bbytes,
                             &sm.bfull[slot], pol_b);
                    ++bq;
                    progress = true;
                }
            }
            if (!progress && !sp.ok(P.err, WS_EMPTY, tag, 0)) { ok = false; break; }
        }
        s = s0 + (unsigned)(w - mp.u0);
    }
    if (!ok) {
        // stopped early: wait (bounded) until every issued copy has landed
        for (unsigned k = s > MMA_NSTAGE ? s - MMA_NSTAGE : 0; k < s; ++k) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try(&sm.wfull[k % MMA_NSTAGE], (k / MMA_NSTAGE) & 1u) ||
                   !mbar_try(&sm.bfull[k % MMA_NSTAGE], (k / MMA_NSTAGE) & 1u))
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) break;
        }
    }
}

// MMA warp (one lane): per unit, wait for the weight and activation chunks and
// for a free slot of the tensor-memory ring, issue the unit's four MMAs into
// that slot (fresh: short fp32 chains on the tensor cores), release the stage
// and signal the slot.
template <typename TW>
__device__ __forceinline__ void mma_issuer(const Params& P, int ph0, int ph1, int n, unsigned starts, const Smem& sm,
                                           uint32_t tbase)
{
    const int ncol = MMA_PARTS * mma_nbp(n);
    const uint32_t idesc = mma_idesc(ncol);
    unsigned s = 0, uc = 0, na = 0;  // stages, units, attention phases
    bool ok = true;
    const int dep_end = P.dep_ph0 + n_groups(starts) * P.dep_ph_stride;
    const int dep_all = P.dep_ph0 + P.S * P.dep_ph_stride;
    for (int ph = ph0; ph < ph1 && ok; ++ph) {
        if (ph == dep_end && dep_end < dep_all) {
            ph = dep_all - 1;
            continue;
        }
        const TW* W;
        int M, K, c, cnt;
        Phase q = P.phases[ph];
        if (!resolve(P, starts, q, c, cnt)) continue;
        if (q.type == PH_ATTN) {
            // attention stages go to the consumers: count them, then wait until the consumers
            // are past all of them (every stage's barrier phases complete), so that the next
            // parity wait on a slot cannot match an older phase
            const StepDesc* D = P.desc;
            const int H = P.H, hd = P.hd, Wn = P.W, KPS = attn_stage_keys(hd);
            const int ipc = attn_stream_ipc(D, n, P.Wa, H, hd, P.G);
            int total = 0;
            for (int i = 0; i < n; ++i) total += attn_chunks_stream(D->pos[i] + 1 < P.Wa ? D->pos[i] + 1 : P.Wa, hd, ipc) * H;
            for (int item = blockIdx.x; item < total; item += P.G) {
                int i, h, ci, nch, len, k0, k1, kend, mcur;
                attn_item(D, n, H, P.Wa, P.G, item, i, h, ci, nch, len, ATTN_STREAM, hd, ipc);
                attn_stream_range(D, i, len, ci, nch, k0, k1, kend, mcur);
                if (kend > k0) s += (unsigned)((kend - k0 + KPS - 1) / KPS);
            }
            if (!mbar_wait(sm.adone, na & 1u, P.err, WS_FULL)) ok = false;
            ++na;
            continue;
        }
        if (!phase_matrix<TW>(P, q, W, M, K)) continue;
        const MmaPart mp = mma_part(M, K, c, cnt);
        for (int u = mp.u0; u < mp.u1; ++u, ++s, ++uc) {
            const int slot = (int)(s % MMA_NSTAGE);
            const unsigned par = (s / MMA_NSTAGE) & 1u;
            const unsigned long long tw0 = P.ptime ? globaltimer_ns() : 0ull;
            if (!mbar_wait(&sm.wfull[slot], par, P.err, WS_FULL)) { ok = false; break; }
            const unsigned long long tw1 = P.ptime ? globaltimer_ns() : 0ull;
            if (!mbar_wait(&sm.bfull[slot], par, P.err, WS_FULL)) { ok = false; break; }
            if (P.ptime && blockIdx.x == 0) {
                // diagnostics: CTA 0's MMA warp waiting for weight chunks, then for activation chunks
                P.ptime[(size_t)ph * 8 + 4] += tw1 - tw0;
                P.ptime[(size_t)ph * 8 + 5] += globaltimer_ns() - tw1;
            }
            // the unit's products go to a fresh slot of the ring (K = 64: four MMAs);
            // the consumers add them to the tile's sum in fp32 on the CUDA cores
            const int r = (int)(uc % MMA_URING);
            if (!mbar_wait(&sm.tfree[r], ((uc / MMA_URING) & 1u) ^ 1u, P.err, WS_FULL)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tbase + (uint32_t)(r * ncol);
            const unsigned sa = smem_u32(sm.mring + (size_t)slot * MMA_STAGE);
            const uint64_t ad = sw128_desc(sa), bd = sw128_desc(sa + MMA_W_BYTES);
#pragma unroll
            for (int kk = 0; kk < MMA_KC / 16; ++kk)
                mma_bf16(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, kk > 0 ? 1u : 0u);
            mma_commit(&sm.sempty[slot]);
            mma_commit(&sm.accf[r]);
        }
    }
    // every MMA issued has completed before tensor memory is freed
    mma_commit(sm.mdone);
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try(sm.mdone, 0u))
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) break;
}

// Every CTA of the grid has finished phase ph (one warp polls every flag, then the CTA meets).
__device__ __forceinline__ bool wait_phase_done(const Params& P, int ph)
{
    const unsigned tag = phase_tag(P.desc, ph);
    int ok = 1;
    if ((threadIdx.x >> 5) == 0) {
        const unsigned* flags = P.done + (size_t)ph * P.G;
        for (int k0 = 0; k0 < P.G && ok; k0 += 32 * 5) {
            unsigned v[5];  // every flag of the batch in flight at once, then the stragglers
#pragma unroll
            for (int q = 0; q < 5; ++q) {
                const int k = k0 + threadIdx.x + 32 * q;
                v[q] = tag;
                if (k < P.G) asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v[q]) : "l"(flags + k) : "memory");
            }
#pragma unroll
            for (int q = 0; q < 5; ++q) {
                const int k = k0 + threadIdx.x + 32 * q;
                Spin sp;
                while (ok && v[q] != tag) {
                    if (!sp.ok(P.err, WS_TAG1, tag, v[q])) { ok = 0; break; }
                    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v[q]) : "l"(flags + k) : "memory");
                }
            }
        }
        __threadfence();
    }
    return csync_and(ok);
}

__device__ __forceinline__ void mark_phase_done(const Params& P, int ph)
{
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned tag = phase_tag(P.desc, ph);
        asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(P.done + (size_t)ph * P.G + blockIdx.x), "r"(tag) : "memory");
    }
}

// Per-thread state of the consumers across tensor-core phases.
struct MmaState {
    uint32_t tbase;
    unsigned uc;      // units read so far in this launch (position in the tensor-memory ring)
    int ph0;          // first phase of the launch
};

// Tile sum j of this warp's rows and batch rows (see mma_read_tile), stored in /
// read from the columns after the ring: MMA_URING x 3 nbp, then nbp per tile.
template <int NC>
__device__ __forceinline__ uint32_t tile_sum_addr(uint32_t tbase, int j, int nbp)
{
    const int warp = threadIdx.x >> 5;
    return tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(MMA_URING * MMA_PARTS * nbp + j * nbp) +
           (uint32_t)((warp >> 2) * NC);
}

__device__ __forceinline__ void tile_sum_store(uint32_t tbase, int j, int nbp, const float (&y)[16])
{
    if (nbp == 16) tmem_st<8>(tile_sum_addr<8>(tbase, j, nbp), y);
    else tmem_st<16>(tile_sum_addr<16>(tbase, j, nbp), y);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tile_sum_load(uint32_t tbase, int j, int nbp, float (&y)[16])
{
#pragma unroll
    for (int e = 0; e < 16; ++e) y[e] = 0.f;
    if (nbp == 16) {
        float v[8];
        tmem_ld<8>(tile_sum_addr<8>(tbase, j, nbp), v);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = v[e];
    } else {
        tmem_ld<16>(tile_sum_addr<16>(tbase, j, nbp), y);
    }
}

// This warp's accumulator values of tile slot j: rows 32 (warp % 4) + lane,
// batch rows [h * nbp / 2, (h + 1) * nbp / 2) with h = warp / 4; the products
// of the three activation parts are added in part order.
template <int NC>
__device__ __forceinline__ void mma_read_tile(uint32_t tbase, int j, int nbp, float (&y)[16])
{
    const int warp = threadIdx.x >> 5;
    const uint32_t base = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(j * MMA_PARTS * nbp) +
                          (uint32_t)((warp >> 2) * NC);
    float p0[NC], p1[NC], p2[NC];
    tmem_ld<NC>(base, p0);
    tmem_ld<NC>(base + (uint32_t)nbp, p1);
    tmem_ld<NC>(base + (uint32_t)(2 * nbp), p2);
#pragma unroll
    for (int e = 0; e < 16; ++e) y[e] = e < NC ? (p0[e] + p1[e]) + p2[e] : 0.f;
}

__device__ __forceinline__ void mma_read(uint32_t tbase, int j, int nbp, float (&y)[16])
{
    if (nbp == 16) mma_read_tile<8>(tbase, j, nbp, y);
    else mma_read_tile<16>(tbase, j, nbp, y);
}



// Consumers of one tensor-core matrix phase: stage the activation chunks of
// the CTA's units, then the partial of the tile it does not own, then, per
// owned tile, the sum over the tile's contributors in K order, the RMSNorm
// factor, and the epilogue.
template <typename TW, class Epi>
__device__ __noinline__ bool mma_phase(const Params& P, const Phase& ph, int phi, int c, int cnt, const XSrc& xs, int n,
                                       const Smem& sm, unsigned& stage, MmaState& ms, Epi epi)
{
    const TW* W;
    int M, K;
    phase_matrix<TW>(P, ph, W, M, K);
    const MmaPart mp = mma_part(M, K, c, cnt);
    const int nbp = mma_nbp(n);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta0 = (int)blockIdx.x - c;  // first CTA of the set sharing this matrix
    const unsigned tag = phase_tag(P.desc, phi);
    const int par = phi % MMA_ROT;
    int ok = 1;
    // A group's first depformer layer after another group: its inputs need not depend
    // on that group's last phases (supplied tokens), so every CTA must have left the
    // previous group before this phase reuses its rotating buffers.
    if (ph.type == PH_DQKV && ph.l == 0 && phi - 1 >= ms.ph0 && P.phases[phi - 1].type == PH_DHEAD &&
        !wait_phase_done(P, phi - 1))
        return false;
    // depformer layer 0: the input token of every batch row (all CTAs take the same)
    if (xs.add) {
        for (int b0 = 0; b0 < n; b0 += NWARP)
            if (!dep_select_inputs(P, xs, b0, min(NWARP, n - b0), sm, b0)) return false;
    }
    // activation chunks of the panel: this CTA converts chunks c, c + cnt, ... of the
    // phase's input (every CTA that shares the matrix does its share).  Thread
    // (b, c16) takes 8 consecutive K of batch row b: waits for their tags, adds the
    // depformer embedding (layer 0), applies the gain, splits each value into
    // three bf16 parts and writes them to operand rows b, nbp + b and 2 nbp + b in
    // the swizzled K-major layout; rows of padding batch rows are zero.  Then the
    // chunk's sums of squares per row, a proxy fence, and the chunk's ready tag.
    stage += (unsigned)(mp.u1 - mp.u0);  // the stages of this phase's units (the producer's and MMA warp's count)
    const int b = tid >> 3, c16 = tid & 7;
    const bool active = b < n;
    const int sub = phase_sub(ph);
    const size_t pbase = panel_index(P, par, sub, 0);
    for (int kc = c; kc < mp.KC && ok; kc += cnt) {
        const int k0 = kc * MMA_KC + c16 * 8;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
        float q = 0.f;
        if (active && k0 < K) {
            const uint2* src = xs.base + (size_t)b * xs.stride + k0;
            uint2 pend[8];
            tag8_issue(src, pend);
            typename WV<TW>::raw er;
            if (xs.add) er = WV<TW>::load((const TW*)xs.add + (size_t)sm.prev[b] * (size_t)xs.add_stride + k0);
            if (!tag8_take(pend, src, xs.tag, f, P.err)) ok = 0;
            if (xs.add) {
                float e8[8];
                WV<TW>::cvt(er, e8);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] += e8[e];
                if (xs.store) {
                    uint2* dst = xs.store + (size_t)b * xs.store_stride + k0;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) st_tag2(dst + e, f[e], f[e + 1], xs.store_tag);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) q = fmaf(f[e], f[e], q);
            if (xs.g) {
                const float4* gs = reinterpret_cast<const float4*>(xs.g + k0);
                const float4 g0 = __ldg(gs), g1 = __ldg(gs + 1);
                f[0] *= g0.x; f[1] *= g0.y; f[2] *= g0.z; f[3] *= g0.w;
                f[4] *= g1.x; f[5] *= g1.y; f[6] *= g1.z; f[7] *= g1.w;
            }
        }
        if (b < nbp) {
            // f = p0 + p1 + p2 + r with bf16 parts and |r| <= 2^-27 |f| (each difference is exact in fp32)
            uint32_t w0[4], w1[4], w2[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const __nv_bfloat162 h0 = __floats2bfloat162_rn(f[e], f[e + 1]);
                const float2 g0 = __bfloat1622float2(h0);
                const float r0 = f[e] - g0.x, r1 = f[e + 1] - g0.y;
                const __nv_bfloat162 h1 = __floats2bfloat162_rn(r0, r1);
                const float2 g1 = __bfloat1622float2(h1);
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(r0 - g1.x, r1 - g1.y);
                w0[e / 2] = *reinterpret_cast<const uint32_t*>(&h0);
                w1[e / 2] = *reinterpret_cast<const uint32_t*>(&h1);
                w2[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            char* ch = P.panel + (pbase + (size_t)kc) * MMA_B_BYTES;
            const int ra = b, rb = nbp + b, rc = 2 * nbp + b;
            *reinterpret_cast<uint4*>(ch + (ra >> 3) * 1024 + (ra & 7) * 128 + ((c16 ^ (ra & 7)) << 4)) =
                make_uint4(w0[0], w0[1], w0[2], w0[3]);
            *reinterpret_cast<uint4*>(ch + (rb >> 3) * 1024 + (rb & 7) * 128 + ((c16 ^ (rb & 7)) << 4)) =
                make_uint4(w1[0], w1[1], w1[2], w1[3]);
            *reinterpret_cast<uint4*>(ch + (rc >> 3) * 1024 + (rc & 7) * 128 + ((c16 ^ (rc & 7)) << 4)) =
                make_uint4(w2[0], w2[1], w2[2], w2[3]);
        }
        q += __shfl_xor_sync(0xffffffffu, q, 1);
        q += __shfl_xor_sync(0xffffffffu, q, 2);
        q += __shfl_xor_sync(0xffffffffu, q, 4);
        if (active && c16 == 0) st_tag1(P.pssq + (pbase + (size_t)kc) * 32 + b, __float_as_uint(q), tag);
        asm volatile("fence.proxy.async.global;" ::: "memory");  // the chunk is read by bulk copies (async proxy)
        if (!csync_and(ok)) return false;
        if (tid == 0) {
            __threadfence();
            asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(P.pflag + pbase + kc), "r"(tag) : "memory");
        }
    }
    if (!csync_and(ok)) return false;
    if (P.ptime) stamp(P, sm.misc[0], 1);
    const int row = 32 * (warp & 3) + lane;  // this thread's tile row
    const int bh = (warp >> 2) * (nbp / 2);  // and its first batch row
    const int nh = nbp / 2;
    // the units' products in order: each unit's slot of the ring is read, its three
    // parts added, and the result added to the tile's sum in fp32 (round to
    // nearest, K order); a finished tile's sum goes to its columns
    {
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        for (int u = mp.u0; u < mp.u1; ++u, ++ms.uc) {
            const int r = (int)(ms.uc % MMA_URING);
            if (ok && !mbar_wait(&sm.accf[r], (ms.uc / MMA_URING) & 1u, P.err, WS_FULL)) ok = 0;
            if (!__all_sync(0xffffffffu, ok)) { ok = 0; break; }
            tc_fence_after();
            float y[16];
            mma_read(ms.tbase, r, nbp, y);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tfree[r]);
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] += y[e];
            if (u == mp.u1 - 1 || (u + 1) % mp.KC == 0) {
                tile_sum_store(ms.tbase, u / mp.KC - mp.t0, nbp, acc);
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            }
        }
    }
    if (!csync_and(ok)) return false;
    // the partial of the tile this CTA does not own
    if (mp.nt > 0 && !mp.last_owned) {
        const int j = mp.nt - 1;
        float y[16];
        tile_sum_load(ms.tbase, j, nbp, y);
        uint2* dst = P.mpart + (((size_t)par * P.G + blockIdx.x) * MMA_M + row) * 32 + bh;  // par: phase mod MMA_ROT
#pragma unroll
        for (int e = 0; e < 16; e += 2)
            if (e < nh) st_tag2(dst + e, y[e], y[e + 1], tag);
    }
    // owned tiles
    const int nown = mp.nt - (mp.last_owned ? 0 : 1);
    constexpr bool is_logits = std::is_same<Epi, EpiLogits>::value;
    if constexpr (is_logits) {
        epi.dv = sm.bestv;
        epi.di = sm.besti;
    }
    // RMSNorm factor per batch row from the chunks' sums of squares (8 threads per
    // row take every 8th chunk, then a fixed reduction: the same for every tile).
    // Only the owners of tiles need it, after their units: the MMAs do not wait for it.
    if (xs.g && nown > 0) {
        float tq = 0.f;
        if (active) {
            const uint2* ps = P.pssq + pbase * 32 + b;
            for (int k0 = c16; k0 < mp.KC && ok; k0 += 64) {
                uint2 v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int kc = k0 + 8 * e;
                    v[e] = make_uint2(0u, tag);
                    if (kc < mp.KC) v[e] = ld_tag1(ps + (size_t)kc * 32);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int kc = k0 + 8 * e;
                    if (kc < mp.KC) {
                        unsigned bits = v[e].x;
                        if (v[e].y != tag && ok) ok = wait_tag1(ps + (size_t)kc * 32, tag, bits, P.err);
                        tq += __uint_as_float(bits);
                    }
                }
            }
        }
        tq += __shfl_xor_sync(0xffffffffu, tq, 1);
        tq += __shfl_xor_sync(0xffffffffu, tq, 2);
        tq += __shfl_xor_sync(0xffffffffu, tq, 4);
        if (active && c16 == 0) sm.ssq[b] = rsqrtf(tq / (float)K + P.eps);
    }
    if (!csync_and(ok)) return false;
    if (P.ptime) stamp(P, sm.misc[0], 2);
    if (nown > 0) {
        if (is_logits && tid < n) {
            sm.bestv[tid] = -INFINITY;
            sm.besti[tid] = 0x7fffffff;
        }
        const long long U = (long long)mp.T * mp.KC;
        for (int j = 0; j < nown && ok; ++j) {
            const int t = mp.t0 + j;
            float y[16], acc[16];
            tile_sum_load(ms.tbase, j, nbp, y);
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            // contributors: the CTAs before this one whose ranges reach into tile t, in K order
            int cs = c;
            while (cs > 0 && mma_unit0(U, cs, cnt) > t * mp.KC) --cs;  // cs: the CTA holding the tile's first unit
            for (int cc = cs; cc < c && ok; ++cc) {
                if (mma_unit0(U, cc + 1, cnt) <= mma_unit0(U, cc, cnt)) continue;  // empty range
                const uint2* src = P.mpart + (((size_t)par * P.G + cta0 + cc) * MMA_M + row) * 32 + bh;
                uint2 v[16];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {  // every element in flight at once, then the stragglers
                    v[e] = v[e + 1] = make_uint2(0u, tag);
                    if (e < nh) ld_tag2(src + e, v[e], v[e + 1]);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    if (e < nh && bh + e < n) {
                        unsigned bits = v[e].x;
                        if (v[e].y != tag && ok) ok = wait_tag1(src + e, tag, bits, P.err);
                        acc[e] += __uint_as_float(bits);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] += y[e];
            if (!csync_and(ok)) return false;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int bb = bh + e;
                if (e < nh && bb < n) sm.yf[(size_t)row * nbp + bb] = acc[e] * (xs.g ? sm.ssq[bb] : 1.f);
            }
            csync();
            const int r0 = t * MMA_M, r1 = min(M, r0 + MMA_M);
            if constexpr (std::is_same<Epi, EpiResid>::value) {
                if (!csync_and(epi.apply_all(P, sm, r0, r1, n, nbp))) return false;
            } else if constexpr (is_logits) {
                if (!csync_and(epi.apply_tile(P, sm, r0, r1, n, nbp))) return false;
            } else {
                const Pre pre = epi.pre(P, r0, r1, 0, n);
                if (!csync_and(pre.ok)) return false;
                if (!csync_and(epi.apply(P, sm, r0, r1, 0, n, nbp, pre))) return false;
            }
        }
        if (!ok) return false;
        if constexpr (is_logits) {
            csync();
            epi.flush(P, 0, n);
        }
    } else {
        epi.empty(P, 0, n);
    }
    return true;
}

// ------------------------------------------------------------------ S0 + S1

template <typename TW>
__device__ __forceinline__ bool phase_embed(const Params& P, int n, unsigned tag, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int d = P.d;
    if (!D->prompt_rows) {
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
    } else if (blockIdx.x == 0) {
        // prompt chunk: CTA 0 alone reads the history.  A frame of this chunk comes from
        // its row's tokens, an earlier one from the history; the rows are published to
        // the other CTAs, then the last three frames of each slot go into the history
        // (their columns may hold frames other rows read: CTA 0 read them already).
        for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
            const int i = it / NSTREAM, k = it % NSTREAM;
            const int f = D->pos[i] - 1 - P.delays[k];
            const int init = k == 0 ? P.V : P.C;
            const int r0 = slot_first_row(D, i);
            int tok;
            if (f < 0) tok = init;
            else if (f >= D->pos[r0]) tok = D->codes[i - (D->pos[i] - f)][k];
            else tok = ld_cg_int(P.hist + ((size_t)D->slot[i] * NSTREAM + k) * HIST + f % HIST);
            if (tok < 0 || tok > init) tok = init;
            sm.X[it] = tok;
        }
        csync();
        for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
            st_tag1(P.xtok + it, (unsigned)sm.X[it], tag);
            const int i = it / NSTREAM, k = it % NSTREAM;
            if (D->pos[i] >= D->pos[slot_last_row(D, n, i)] - (HIST - 1))
                P.hist[((size_t)D->slot[i] * NSTREAM + k) * HIST + D->pos[i] % HIST] = D->codes[i][k];
        }
    } else {
        int ok = 1;
        for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
            unsigned bits = 0;
            if (ok) ok = wait_tag1(P.xtok + it, tag, bits, P.err);
            sm.X[it] = ok ? (int)bits : 0;
        }
        if (!csync_and(ok)) return false;
    }
    // x[i] = sum over streams in stream order; rows loaded 6 at a time
    const int per = d / 8;
    for (int it = blockIdx.x * NT + threadIdx.x; it < n * per; it += P.G * NT) {
        const int i = it / per, e0 = (it % per) * 8;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
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
        uint2* dst = P.x + (size_t)i * d + e0;
#pragma unroll
        for (int e = 0; e < 8; e += 2) st_tag2(dst + e, acc[e], acc[e + 1], tag);
    }
    csync();
    return true;
}

// ------------------------------------------------------------------ S5 attention

__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes, uint64_t pol)
{
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(pol) : "memory");
}

// While the QKV phase of layer l runs, the older keys/values of every slot's
// window are pulled into L2: per (slot, head, tensor) the window is one or two
// contiguous runs of the head-major ring, prefetched 32 positions at a time and
// spread evenly over the CTAs of the grid, so that the attention reads hit L2
// instead of queueing behind the weight stream.  Only for windows small enough
// to sit in L2 (at most 32 MB per layer).
template <typename TKV>
__device__ __forceinline__ void prefetch_kv_windows(const Params& P, int l, int n)
{
    const StepDesc* D = P.desc;
    const int d = P.d, W = P.W, H = P.H, hd = P.hd;
    constexpr int PCS = 32;  // positions per prefetch
    long long total = 0;
    for (int i = 0; i < n; ++i) total += (long long)(D->pos[i] + 1 < P.Wa ? D->pos[i] : P.Wa - 1);
    if (total * d * (long long)sizeof(TKV) * 2 > (32ll << 20)) return;
    const uint64_t pol = l2_evict_last();
    // items (slot, head, piece, tensor), slot-major; item k goes to CTA k mod G
    int i = 0;
    long long base = 0;
    auto older = [&](int ii) { return D->pos[ii] + 1 < P.Wa ? D->pos[ii] : P.Wa - 1; };
    auto items = [&](int ii) { return (long long)H * ((older(ii) + PCS - 1) / PCS) * 2; };
    long long cnt = n > 0 ? items(0) : 0;
    for (long long k = blockIdx.x + (long long)P.G * threadIdx.x;; k += (long long)P.G * NT) {
        while (i < n && k >= base + cnt) {  // k only grows: walk the slots forward
            base += cnt;
            if (++i < n) cnt = items(i);
        }
        if (i >= n) break;
        const long long r = k - base;
        const int len = older(i), npc = (len + PCS - 1) / PCS;
        const int h = (int)((r >> 1) / npc), pc = (int)((r >> 1) % npc);
        const int q0 = D->pos[i] - len + pc * PCS, c = min(PCS, D->pos[i] - q0);  // positions [q0, q0 + c)
        const TKV* run = (const TKV*)((r & 1) ? P.vc : P.kc) + (((long long)D->slot[i] * P.L + l) * H + h) * (long long)W * hd;
        const int r0 = q0 % W;
        if (r0 + c <= W) {
            prefetch_l2(run + (long long)r0 * hd, (unsigned)(c * hd * sizeof(TKV)), pol);
        } else {
            prefetch_l2(run + (long long)r0 * hd, (unsigned)((W - r0) * hd * sizeof(TKV)), pol);
            prefetch_l2(run, (unsigned)((r0 + c - W) * hd * sizeof(TKV)), pol);
        }
    }
}

// One CTA per (batch row, head, chunk of the window): its warps split the
// chunk into contiguous runs of keys, merged in shared memory in warp order.
// A window of one chunk writes the output directly; otherwise each chunk
// leaves {max, sum, unnormalised output} tagged in P.attp and the CTA that ran
// chunk 0 merges the chunks in order once every CTA has run its chunks (no CTA
// waits for another's chunk before finishing its own, so the waits end).
// The newest key/value (this step's) comes from the tagged copy.
// Keys [j0, j1) of the window of batch row i, head h (len keys from absolute
// position start; the last mcur of them are this launch's and come from the
// tagged copies): scores in fp32, an online softmax over groups of PPI x UNR
// keys, then the warp's key groups merged.  Every lane ends with the running
// max m, the sum lsum and the unnormalised outputs acc of its 8 elements
// (lanes gl, gl + LPP, ... hold the same values).  ok turns 0 if a wait gave up.
template <typename TKV>
__device__ __forceinline__ void attn_keys(const Params& P, int i, int h, int len, int start, int mcur, int j0, int j1,
                                          long long kvbase, const float qv[8], const float kcur[8], const float vcur[8],
                                          unsigned in_tag, int& ok, float& m, float& lsum, float acc[8])
{
    const int hd = P.hd, d = P.d, W = P.W;
    const int lane = threadIdx.x & 31;
    const int LPP = hd / 8;            // lanes per key
    const int PPI = 32 / LPP;          // keys per warp iteration
    const int grp = lane / LPP, gl = lane % LPP;
    m = -INFINITY;
    lsum = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    // keys in flight per lane: kept packed until used, so that bf16 rings keep 8
    constexpr int UNR = sizeof(TKV) == 2 ? 8 : 4;
    // warp-uniform trip count: every lane runs every iteration (shuffles below)
    for (int jb = j0; jb < j1; jb += PPI * UNR) {
        const int jj = jb + grp;
        typename KV<TKV>::raw kr[UNR], vr[UNR];
        float s[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int j = jj + u * PPI;
            if (j < j1 && j < len - mcur) {
                const long long row = (long long)((start + j) % W) * hd;
                kr[u] = KV<TKV>::load_raw(P.kc, kvbase + row);
                vr[u] = KV<TKV>::load_raw(P.vc, kvbase + row);
            } else {
                float kf[8], vf[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) { kf[e] = 0.f; vf[e] = 0.f; }
                if (j == len - 1) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) { kf[e] = kcur[e]; vf[e] = vcur[e]; }
                } else if (j < j1) {
                    // an earlier frame of this prompt chunk: row i - (len - 1 - j)
                    const size_t ro = (size_t)(i - (len - 1 - j)) * d + h * hd + gl * 8;
                    if (ok) ok = wait_tag8(P.kcur + ro, in_tag, kf, P.err) && wait_tag8(P.vcur + ro, in_tag, vf, P.err);
                }
                kr[u] = KV<TKV>::pack(kf);
                vr[u] = KV<TKV>::pack(vf);
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            float kf[8];
            KV<TKV>::unpack(kr[u], kf);
            float t = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) t = fmaf(qv[e], kf[e], t);
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
            float vf[8];
            KV<TKV>::unpack(vr[u], vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(pu, vf[e], acc[e]);
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
}

template <typename TKV>
__device__ __forceinline__ bool phase_attn(const Params& P, int l, int n, unsigned in_tag, unsigned tag, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int H = P.H, hd = P.hd, d = P.d, W = P.W;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int LPP = hd / 8;            // lanes per key
    const int PPI = 32 / LPP;          // keys per warp iteration
    const int grp = lane / LPP, gl = lane % LPP;
    const float scale = rsqrtf((float)hd);
    const int wstride = hd + 4;
    const size_t pstride = (size_t)hd + 2;  // partial: max, sum, hd outputs
    int total = 0;
    for (int i = 0; i < n; ++i) {
        const int p = D->pos[i];
        total += attn_chunks(p + 1 < P.Wa ? p + 1 : P.Wa, P.G, H) * H;
    }
    for (int item = blockIdx.x; item < total; item += P.G) {
        int i, h, c, nch, len;
        attn_item(D, n, H, P.Wa, P.G, item, i, h, c, nch, len);
        const int p = D->pos[i], slot = D->slot[i];
        const int start = p - len + 1;
        // keys of this launch: the last mcur of the window (the current one, and in a prompt
        // chunk those of the slot's earlier rows), read from the tagged copies
        const int mcur = p - D->pos[slot_first_row(D, i)] + 1;
        const int k0 = (int)((long long)len * c / nch), k1 = (int)((long long)len * (c + 1) / nch);
        const int j0 = k0 + (int)((long long)(k1 - k0) * warp / NWARP), j1 = k0 + (int)((long long)(k1 - k0) * (warp + 1) / NWARP);
        const long long kvbase = (((long long)slot * P.L + l) * H + h) * (long long)W * hd + gl * 8;
        // the query and this step's key/value are polled while the first ring loads are in flight
        uint2 qt[8], kt[8], vt[8];
        tag8_issue(P.q + (size_t)i * d + h * hd + gl * 8, qt);
        const bool has_cur = len - 1 >= j0 && len - 1 < j1;
        if (has_cur) {
            tag8_issue(P.kcur + (size_t)i * d + h * hd + gl * 8, kt);
            tag8_issue(P.vcur + (size_t)i * d + h * hd + gl * 8, vt);
        }
        float qv[8], kcur[8], vcur[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) { kcur[e] = 0.f; vcur[e] = 0.f; }
        int ok = tag8_take(qt, P.q + (size_t)i * d + h * hd + gl * 8, in_tag, qv, P.err);
        if (has_cur && ok)
            ok = tag8_take(kt, P.kcur + (size_t)i * d + h * hd + gl * 8, in_tag, kcur, P.err) &&
                 tag8_take(vt, P.vcur + (size_t)i * d + h * hd + gl * 8, in_tag, vcur, P.err);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] *= scale;
        if (P.ptime && item == blockIdx.x) stamp(P, sm.misc[0], 1);
        float m, lsum, acc[8];
        attn_keys<TKV>(P, i, h, len, start, mcur, j0, j1, kvbase, qv, kcur, vcur, in_tag, ok, m, lsum, acc);
        if (P.ptime && item == blockIdx.x) stamp(P, sm.misc[0], 2);
        float* wb = sm.wbuf + (size_t)warp * wstride;
        if (lane < LPP) {
            if (lane == 0) { wb[0] = m; wb[1] = lsum; }
#pragma unroll
            for (int e = 0; e < 8; ++e) wb[4 + gl * 8 + e] = acc[e];
        }
        if (!csync_and(ok)) return false;
        // merge the warps in warp order
        float M = -INFINITY;
        for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sm.wbuf[(size_t)w * wstride]);
        uint2* part = P.attp + (((size_t)i * H + h) * NCHUNK_MAX + c) * pstride;
        for (int e = threadIdx.x; e < hd; e += NT) {
            float L = 0.f, a = 0.f;
            for (int w = 0; w < NWARP; ++w) {
                const float mw = sm.wbuf[(size_t)w * wstride];
                if (mw == -INFINITY) continue;
                const float f = expf(mw - M);
                L += sm.wbuf[(size_t)w * wstride + 1] * f;
                a += sm.wbuf[(size_t)w * wstride + 4 + e] * f;
            }
            if (nch == 1) {
                st_tag1(P.o + (size_t)i * d + h * hd + e, __float_as_uint(a / L), tag);
            } else {
                st_tag1(part + 2 + e, __float_as_uint(a), tag);
                if (e == 0) {
                    st_tag1(part, __float_as_uint(M), tag);
                    st_tag1(part + 1, __float_as_uint(L), tag);
                }
            }
        }
        csync();
    }
    // merges: the CTA that ran chunk 0 of a split window combines its chunks in order
    for (int item = blockIdx.x; item < total; item += P.G) {
        int i, h, c, nch, len;
        attn_item(D, n, H, P.Wa, P.G, item, i, h, c, nch, len);
        if (c != 0 || nch == 1) continue;
        const uint2* part = P.attp + ((size_t)i * H + h) * NCHUNK_MAX * pstride;
        // every chunk's partial into shared memory, four loads in flight per thread
        float* mb = sm.wbuf;  // [nch][hd + 2]
        const int cnt = nch * (int)pstride;
        int ok = 1;
        for (int x0 = threadIdx.x; x0 < cnt && ok; x0 += 4 * NT) {
            uint2 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NT;
                v[u] = x < cnt ? ld_tag1(part + (x / pstride) * pstride + x % pstride) : make_uint2(0u, tag);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NT;
                unsigned bits = v[u].x;
                if (x < cnt && v[u].y != tag && ok) ok = wait_tag1(part + (x / pstride) * pstride + x % pstride, tag, bits, P.err);
                if (x < cnt) mb[x] = __uint_as_float(bits);
            }
        }
        if (!csync_and(ok)) return false;
        for (int e = threadIdx.x; e < hd; e += NT) {
            float M = -INFINITY;
            for (int k = 0; k < nch; ++k) M = fmaxf(M, mb[k * pstride]);
            float L = 0.f, a = 0.f;
            for (int k = 0; k < nch; ++k) {
                const float mk = mb[k * pstride];
                if (mk == -INFINITY) continue;
                const float f = expf(mk - M);
                L += mb[k * pstride + 1] * f;
                a += mb[k * pstride + 2 + e] * f;
            }
            st_tag1(P.o + (size_t)i * d + h * hd + e, __float_as_uint(a / L), tag);
        }
        csync();
    }
    return true;
}

// Attention of the tensor-core instantiation with keys and values streamed by the
// producer warp: one CTA per item (batch row, head, chunk of the window; about six
// items per CTA).  A stage holds up to attn_stage_keys(hd) keys, then as many values,
// bf16, copied from the head-major ring.  A key belongs to a group of hd / 8 lanes
// (8 elements each, so a warp reads 512 contiguous bytes at once); a stage is
// ATTN_R passes, and a lane group's ATTN_R partial scores are reduced together
// (each butterfly level halves the values a lane carries), then broadcast.  Scores
// carry a factor log2(e), so the softmax runs on exp2; a group rescales its sums
// only when a stage raises its maximum.  At the end of an item the groups, then the
// warps, merge in order.  This launch's keys (the current one, and a prompt chunk's
// earlier rows) come from the tagged copies.  Chunks merge as in phase_attn.
constexpr int ATTN_R = 4;  // passes per stage: ATTN_R x NWARP x (256 / hd) >= attn_stage_keys(hd)

template <typename TKV>
__device__ __noinline__ bool phase_attn_stream(const Params& P, int l, int n, unsigned in_tag, unsigned tag, const Smem& sm,
                                               unsigned& stage)
{
    const StepDesc* D = P.desc;
    const int H = P.H, hd = P.hd, d = P.d, W = P.W;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int LPP = hd / 8, PPI = 32 / LPP;  // lanes per key, keys per warp and pass
    const int grp = lane / LPP, gl = lane % LPP;
    const int KPS = attn_stage_keys(hd);
    const float scale = 1.4426950408889634f * rsqrtf((float)hd);  // log2(e) / sqrt(hd)
    const int wstride = hd + 4;
    const size_t pstride = (size_t)hd + 2;
    const int ipc = attn_stream_ipc(D, n, P.Wa, H, hd, P.G);
    int total = 0;
    for (int i = 0; i < n; ++i) {
        const int p = D->pos[i];
        total += attn_chunks_stream(p + 1 < P.Wa ? p + 1 : P.Wa, hd, ipc) * H;
    }
    int ok = 1;
    for (int item = blockIdx.x; item < total; item += P.G) {
        int i, h, c, nch, len;
        attn_item(D, n, H, P.Wa, P.G, item, i, h, c, nch, len, ATTN_STREAM, hd, ipc);
        int k0, k1, kend, mcur;
        attn_stream_range(D, i, len, c, nch, k0, k1, kend, mcur);
        float qv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (ok && !wait_tag8(P.q + (size_t)i * d + h * hd + gl * 8, in_tag, qv, P.err)) ok = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] *= scale;
        float m = -INFINITY, lsum = 0.f, acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        // the lane's 8-element share of q.k (two chains)
        auto dot8 = [&](const uint4& k) {
            float2 t2 = make_float2(0.f, 0.f);
            ffma2(t2, qv[0], qv[1], bf_lo(k.x), bf_hi(k.x));
            ffma2(t2, qv[2], qv[3], bf_lo(k.y), bf_hi(k.y));
            ffma2(t2, qv[4], qv[5], bf_lo(k.z), bf_hi(k.z));
            ffma2(t2, qv[6], qv[7], bf_lo(k.w), bf_hi(k.w));
            return t2.x + t2.y;
        };
        auto addv = [&](float pu, const uint4& v) {
            float2 a0 = make_float2(acc[0], acc[1]), a1 = make_float2(acc[2], acc[3]);
            float2 a2 = make_float2(acc[4], acc[5]), a3 = make_float2(acc[6], acc[7]);
            ffma2(a0, pu, pu, bf_lo(v.x), bf_hi(v.x));
            ffma2(a1, pu, pu, bf_lo(v.y), bf_hi(v.y));
            ffma2(a2, pu, pu, bf_lo(v.z), bf_hi(v.z));
            ffma2(a3, pu, pu, bf_lo(v.w), bf_hi(v.w));
            acc[0] = a0.x; acc[1] = a0.y; acc[2] = a1.x; acc[3] = a1.y;
            acc[4] = a2.x; acc[5] = a2.y; acc[6] = a3.x; acc[7] = a3.y;
        };
        // raise the group's maximum to mn (rescaling its sums) if mn is above it
        auto raise = [&](float mn) {
            if (mn > m) {
                const float corr = exp2f(m - mn);
                lsum *= corr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] *= corr;
                m = mn;
            }
        };
        // streamed keys, stage by stage (every warp passes every stage's barrier, also
        // after a failed wait, so that no barrier waits for a warp that has left)
        for (int kb = k0; kb < kend; kb += KPS, ++stage) {
            const int nk = min(KPS, kend - kb);
            const int slot = (int)(stage % MMA_NSTAGE);
            if (ok && !mbar_wait(&sm.wfull[slot], (stage / MMA_NSTAGE) & 1u, P.err, WS_FULL)) ok = 0;
            if (__all_sync(0xffffffffu, ok)) {
                const __nv_bfloat16* ks = (const __nv_bfloat16*)(sm.mring + (size_t)slot * MMA_STAGE);
                const __nv_bfloat16* vs = ks + (size_t)KPS * hd;
                uint4 kr[ATTN_R], vr[ATTN_R];
                float t[ATTN_R];
#pragma unroll
                for (int r = 0; r < ATTN_R; ++r) {
                    const int kk = r * NWARP * PPI + warp * PPI + grp;
                    const size_t off = (size_t)(kk < nk ? kk : 0) * hd + gl * 8;
                    kr[r] = *reinterpret_cast<const uint4*>(ks + off);
                    vr[r] = *reinterpret_cast<const uint4*>(vs + off);
                }
#pragma unroll
                for (int r = 0; r < ATTN_R; ++r) t[r] = dot8(kr[r]);
                // reduce the four partial scores over the group: lane gl ends with key
                // 2 [gl & LPP/2] + [gl & LPP/4], then every lane takes all four
                const bool hi1 = (gl & (LPP / 2)) != 0, hi2 = (gl & (LPP / 4)) != 0;
                const float u0 = (hi1 ? t[2] : t[0]) + __shfl_xor_sync(0xffffffffu, hi1 ? t[0] : t[2], LPP / 2);
                const float u1 = (hi1 ? t[3] : t[1]) + __shfl_xor_sync(0xffffffffu, hi1 ? t[1] : t[3], LPP / 2);
                float sk = (hi2 ? u1 : u0) + __shfl_xor_sync(0xffffffffu, hi2 ? u0 : u1, LPP / 4);
                for (int o = LPP / 8; o > 0; o >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, o);
                float sc[ATTN_R], mn = m;
#pragma unroll
                for (int r = 0; r < ATTN_R; ++r) {
                    const int src = grp * LPP + (r >> 1) * (LPP / 2) + (r & 1) * (LPP / 4);
                    const float v = __shfl_sync(0xffffffffu, sk, src);
                    sc[r] = r * NWARP * PPI + warp * PPI + grp < nk ? v : -INFINITY;
                    mn = fmaxf(mn, sc[r]);
                }
                raise(mn);
#pragma unroll
                for (int r = 0; r < ATTN_R; ++r) {
                    const float pu = sc[r] == -INFINITY ? 0.f : exp2f(sc[r] - m);  // a key past the stage adds 0
                    lsum += pu;
                    addv(pu, vr[r]);
                }
            } else {
                ok = 0;
            }
            csync();  // every warp is done with the stage
            if (threadIdx.x == 0) mbar_arrive(&sm.sempty[slot]);
        }
        // this launch's keys (from the tagged copies): key j is row i - (len - 1 - j)
        const int jl0 = max(k0, len - mcur);
        for (int jb = jl0; jb < k1; jb += NWARP * PPI) {
            const int j = jb + warp * PPI + grp;
            float kf[8], vf[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) { kf[e] = 0.f; vf[e] = 0.f; }
            if (j < k1 && ok) {
                const size_t ro = (size_t)(i - (len - 1 - j)) * d + h * hd + gl * 8;
                ok = wait_tag8(P.kcur + ro, in_tag, kf, P.err) && wait_tag8(P.vcur + ro, in_tag, vf, P.err);
            }
            // the tagged copies hold values already rounded to bf16: they pack exactly
            const uint4 kp = KV<__nv_bfloat16>::pack(kf).a, vp = KV<__nv_bfloat16>::pack(vf).a;
            float tk = dot8(kp);
            for (int o = LPP / 2; o > 0; o >>= 1) tk += __shfl_xor_sync(0xffffffffu, tk, o);
            if (j < k1) {
                raise(tk);
                const float pu = exp2f(tk - m);
                lsum += pu;
                addv(pu, vp);
            }
        }
        // merge the key groups of the warp, then the warps in warp order
        for (int o = LPP; o < 32; o <<= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, lsum, o);
            float a2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, acc[e], o);
            const float M = fmaxf(m, m2);
            const float c1 = m == -INFINITY ? 0.f : exp2f(m - M);
            const float c2 = m2 == -INFINITY ? 0.f : exp2f(m2 - M);
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
        if (!csync_and(ok)) return false;
        float M = -INFINITY;
        for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sm.wbuf[(size_t)w * wstride]);
        uint2* part = P.attp + (((size_t)i * H + h) * NCHUNK_MAX + c) * pstride;
        for (int e = threadIdx.x; e < hd; e += NT) {
            float L = 0.f, a = 0.f;
            for (int w = 0; w < NWARP; ++w) {
                const float mw = sm.wbuf[(size_t)w * wstride];
                if (mw == -INFINITY) continue;
                const float f = exp2f(mw - M);
                L += sm.wbuf[(size_t)w * wstride + 1] * f;
                a += sm.wbuf[(size_t)w * wstride + 4 + e] * f;
            }
            if (nch == 1) {
                st_tag1(P.o + (size_t)i * d + h * hd + e, __float_as_uint(a / L), tag);
            } else {
                st_tag1(part + 2 + e, __float_as_uint(a), tag);
                if (e == 0) {
                    st_tag1(part, __float_as_uint(M), tag);
                    st_tag1(part + 1, __float_as_uint(L), tag);
                }
            }
        }
        csync();
    }
    if (!csync_and(ok)) return false;
    // every stage of the phase is consumed: the MMA warp may go on to the next phase's stages
    if (threadIdx.x == 0) mbar_arrive(sm.adone);
    // merges: the CTA that ran chunk 0 of a split window combines its chunks in order
    for (int item = blockIdx.x; item < total; item += P.G) {
        int i, h, c, nch, len;
        attn_item(D, n, H, P.Wa, P.G, item, i, h, c, nch, len, ATTN_STREAM, hd, ipc);
        if (c != 0 || nch == 1) continue;
        const uint2* part = P.attp + ((size_t)i * H + h) * NCHUNK_MAX * pstride;
        float* mb = sm.wbuf;  // [nch][hd + 2]
        const int cnt = nch * (int)pstride;
        for (int x0 = threadIdx.x; x0 < cnt && ok; x0 += 4 * NT) {
            uint2 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NT;
                v[u] = x < cnt ? ld_tag1(part + (x / pstride) * pstride + x % pstride) : make_uint2(0u, tag);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NT;
                unsigned bits = v[u].x;
                if (x < cnt && v[u].y != tag && ok) ok = wait_tag1(part + (x / pstride) * pstride + x % pstride, tag, bits, P.err);
                if (x < cnt) mb[x] = __uint_as_float(bits);
            }
        }
        if (!csync_and(ok)) return false;
        for (int e = threadIdx.x; e < hd; e += NT) {
            float M = -INFINITY;
            for (int k = 0; k < nch; ++k) M = fmaxf(M, mb[k * pstride]);
            float L = 0.f, a = 0.f;
            for (int k = 0; k < nch; ++k) {
                const float mk = mb[k * pstride];
                if (mk == -INFINITY) continue;
                const float f = exp2f(mk - M);  // maxima carry the factor log2(e)
                L += mb[k * pstride + 1] * f;
                a += mb[k * pstride + 2 + e] * f;
            }
            st_tag1(P.o + (size_t)i * d + h * hd + e, __float_as_uint(a / L), tag);
        }
        csync();
    }
    return true;
}

// ------------------------------------------------------------------ S9 depformer attention

// One CTA per (batch row, head): keys of substeps 0..j, no rotation.  Warp w
// loads keys/values w and w + NWARP (tag of that substep's QKV phase) with the
// query, so the loads of the item are in flight together; the softmax and the
// weighted sum run in key order in shared memory.
__device__ __forceinline__ bool phase_dattn(const Params& P, int l, int j0, int nj, unsigned starts, int n, unsigned in_tag,
                                            unsigned tag, const Smem& sm)
{
    const StepDesc* D = P.desc;
    const int dd = P.dd, dH = P.dH, S = P.S;  // head dim is 64
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float scale = 0.125f;  // 1 / sqrt(64)
    float* sc = sm.wbuf;         // [16] scores
    float* pv = sm.wbuf + 16;    // [16][64] p_t * v_t
    // items: (batch row, substep of the group, head)
    for (int item = blockIdx.x; item < n * nj * dH; item += P.G) {
        const int i = item / (nj * dH), j = j0 + (item / dH) % nj, h = item % dH;
        const int npos = j + 1;
        const uint2* q = P.dq + ((size_t)i * S + j) * dd + h * 64 + 2 * lane;
        const uint2* kv = P.dkv + ((size_t)i * P.dL + l) * S * 2 * dd + h * 64 + 2 * lane;
        int ok = 1;
        constexpr int TPW = 16 / NWARP;  // keys per warp
        float2 vt[TPW];
#pragma unroll
        for (int k = 0; k < TPW; ++k) {
            const int t = warp + k * NWARP;
            vt[k] = make_float2(0.f, 0.f);
            if (t < npos && ok) {
                const unsigned tt = phase_tag(D, P.dep_ph0 + group_of(starts, t) * P.dep_ph_stride + l * 5);
                const uint2* kp = kv + (size_t)t * 2 * dd;
                const uint2* vp = kv + ((size_t)t * 2 + 1) * dd;
                uint2 qa, qb, ka, kb, va, vb;
                ld_tag2(q, qa, qb);
                ld_tag2(kp, ka, kb);
                ld_tag2(vp, va, vb);
                Spin sp;
                while (!(qa.y == in_tag && qb.y == in_tag)) {
                    if (!sp.ok(P.err, WS_DQ, in_tag, qa.y)) { ok = 0; break; }
                    ld_tag2(q, qa, qb);
                }
                while (ok && !(ka.y == tt && kb.y == tt && va.y == tt && vb.y == tt)) {
                    if (!sp.ok(P.err, WS_DKV, tt, ka.y)) { ok = 0; break; }
                    ld_tag2(kp, ka, kb);
                    ld_tag2(vp, va, vb);
                }
                const float part = warp_sum(fmaf(__uint_as_float(qa.x), __uint_as_float(ka.x),
                                                 __uint_as_float(qb.x) * __uint_as_float(kb.x)));
                if (lane == 0) sc[t] = part * scale;
                vt[k] = make_float2(__uint_as_float(va.x), __uint_as_float(vb.x));
            }
        }
        if (!csync_and(ok)) return false;
#pragma unroll
        for (int k = 0; k < TPW; ++k) {
            const int t = warp + k * NWARP;
            if (t < npos) {
                float M = -INFINITY;
                for (int u = 0; u < npos; ++u) M = fmaxf(M, sc[u]);
                const float pt = expf(sc[t] - M);
                pv[t * 64 + 2 * lane] = pt * vt[k].x;
                pv[t * 64 + 2 * lane + 1] = pt * vt[k].y;
            }
        }
        csync();
        if (threadIdx.x < 64) {
            const int e = threadIdx.x;
            float M = -INFINITY;
            for (int u = 0; u < npos; ++u) M = fmaxf(M, sc[u]);
            float Z = 0.f, a = 0.f;
            for (int u = 0; u < npos; ++u) {
                Z += expf(sc[u] - M);
                a += pv[u * 64 + e];
            }
            st_tag1(P.dat + ((size_t)i * S + j) * dd + h * 64 + e, __float_as_uint(a / Z), tag);
        }
        csync();
    }
    return true;
}

// ------------------------------------------------------------------ S10

// CTA 0: the argmax of the text head and of every depformer head, the token
// chosen per stream (the supplied one, else that argmax), the history
// write-back for frames p - delay[k] >= 0, and the outputs.
__device__ __forceinline__ bool phase_final(const Params& P, int n, unsigned starts, const Smem& sm)
{
    if (blockIdx.x != 0) return true;
    const StepDesc* D = P.desc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = P.S, G = P.G;
    int* am = sm.X + 2048;  // [n][S + 1]: text head, then the head of substep 0 .. S-1 (after the sampler's histogram)
    int ok = 1;
    for (int it = warp; it < n * (S + 1) && ok; it += NWARP) {
        const int i = it / (S + 1), t = it % (S + 1) - 1;
        int a;
        if (t < 0) {
            a = argmax_partials_warp(P, P.amax + (size_t)i * G * 2, G, phase_tag(D, P.dep_ph0 - 1));
        } else if (group_of(starts, t) >= n_groups(starts)) {
            a = -1;  // substep skipped: its stream's output is settled without it
        } else {
            const int g = group_of(starts, t);
            int j0, nj, b0, b1;
            group_bounds(starts, S, g, j0, nj);
            substep_ctas(G, nj, t - j0, b0, b1);
            a = argmax_partials_warp(P, P.damax + ((size_t)i * S + t) * G * 2, b1 - b0,
                                     phase_tag(D, P.dep_ph0 + (g + 1) * P.dep_ph_stride - 1));
        }
        ok = a >= 0 || (t >= 0 && group_of(starts, t) >= n_groups(starts));
        if (lane == 0) am[it] = a;
    }
    if (!csync_and(ok)) return false;
    // sampled rows: streams drawn at a group's first substep were recorded then; the
    // stream of the last substep that ran (and the text when no substep ran) is drawn here
    const int ngr = n_groups(starts);
    int klast = 0;
    if (ngr > 0) {
        int j0, nj;
        group_bounds(starts, S, ngr - 1, j0, nj);
        klast = j0 + nj;
    }
    if (D->sampled) {
        __threadfence();
        for (int i = 0; i < n; ++i) {
            float inv_t;
            int topk, N;
            if (klast <= S && supplied_token(P, i, klast) < 0 && sampling_on(P, i, klast, inv_t, topk)) {
                const int tok = sample_topk_cta(head_logits(P, i, klast, N), N, inv_t, topk,
                                                P.unif[(size_t)i * NSTREAM + klast], sm);
                if (threadIdx.x == 0) P.drawn[(size_t)i * NSTREAM + klast] = tok;
            }
        }
        csync();
    }
    for (int it = threadIdx.x; it < n * NSTREAM; it += NT) {
        const int i = it / NSTREAM, k = it % NSTREAM;
        const int p = D->pos[i], slot = D->slot[i];
        const int f = p - P.delays[k];
        int a = am[i * (S + 1) + k];  // stream k's head: the text head, or substep k-1's
        const int sup = supplied_token(P, i, k);
        float inv_t;
        int topk;
        if (sup < 0 && k <= klast && sampling_on(P, i, k, inv_t, topk)) a = P.drawn[(size_t)i * NSTREAM + k];
        const int c = sup >= 0 ? sup : a;
        const int raw = am[i * (S + 1) + k];
        if (k == 0) P.text_argmax[i] = raw;
        else P.code_argmax[i * 16 + (k - 1)] = raw;
        if (f >= 0) P.hist[((size_t)slot * NSTREAM + k) * HIST + f % HIST] = c;
        if (k == 0) P.text_out[i] = c;
        else P.codes_out[i * 16 + (k - 1)] = f >= 0 ? c : -1;
    }
    return true;
}

// ------------------------------------------------------------------ phase dispatch

// A matrix phase: tensor cores in the tensor-core instantiation, CUDA-core
// matrix-vector passes otherwise.
template <typename TW, int BG, class Epi>
__device__ __forceinline__ bool matrix_phase(const Params& P, const Phase& ph, int phi, int c, int cnt, const XSrc& xs,
                                             int n, const Smem& sm, unsigned& stage, MmaState& ms, const Epi& epi)
{
    if constexpr (is_mma(BG)) return mma_phase<TW>(P, ph, phi, c, cnt, xs, n, sm, stage, ms, epi);
    else return gemv_phase<TW, BG>(P, ph, c, cnt, xs, n, sm, stage, epi);
}

template <typename TW, typename TKV, int BG>
__device__ __forceinline__ bool run_phase(const Params& P, Phase ph, int phi, int n, unsigned starts, const Smem& sm,
                                          unsigned& stage, MmaState& ms)
{
    const int d = P.d, F = P.F, dd = P.dd, dF = P.dF, S = P.S;
    const StepDesc* D = P.desc;
    const unsigned tag = phase_tag(D, phi);
    const unsigned in_tag = ph.in_ph >= 0 ? phase_tag(D, ph.in_ph) : 0u;
    const unsigned res_tag = ph.res_ph >= 0 ? phase_tag(D, ph.res_ph) : 0u;
    int c, cnt;
    if (!resolve(P, starts, ph, c, cnt)) return true;
    const int j = ph.j;  // depformer: this CTA's substep
    switch (ph.type) {
        case PH_EMBED: return phase_embed<TW>(P, n, tag, sm);
        case PH_QKV:
            prefetch_kv_windows<TKV>(P, ph.l, n);
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.x, d, in_tag, P.attn_norm + (size_t)ph.l * d},
                                      n, sm, stage, ms, EpiQKV<TKV>{ph.l, tag});
        case PH_ATTN:
            if constexpr (is_mma(BG)) return phase_attn_stream<TKV>(P, ph.l, n, in_tag, tag, sm, stage);
            else return phase_attn<TKV>(P, ph.l, n, in_tag, tag, sm);
        case PH_O:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.o, d, in_tag}, n, sm, stage, ms, EpiResid{P.x, d, res_tag, tag});
        case PH_GU:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.x, d, in_tag, P.ffn_norm + (size_t)ph.l * d},
                                      n, sm, stage, ms, EpiSwiglu{P.s, F, tag});
        case PH_DOWN:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.s, F, in_tag}, n, sm, stage, ms, EpiResid{P.x, d, res_tag, tag});
        case PH_HEAD:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.x, d, in_tag, P.out_norm}, n, sm, stage, ms,
                                      EpiLogits{P.logits, P.V, P.V, P.yin, (long long)S * dd, tag, P.amax,
                                                (long long)P.G * 2, (int)blockIdx.x});
        case PH_DQKV: {
            const long long us = (long long)S * dd;
            XSrc xs;
            if (ph.l == 0) {
                // the residual starts as in-projection + embedding of the substep's input token
                const void* add = j == 0 ? P.dep_emb_text : (const void*)((const TW*)P.dep_emb_audio + (size_t)(j - 1) * P.C * dd);
                xs = XSrc{P.yin + (size_t)j * dd, us, in_tag, P.dep_attn_norm, add, dd, (c == 0 || is_mma(BG)) ? P.u + (size_t)j * dd : nullptr,
                          tag, us, j, ph.pad0, 0u, 0};
                if (j == ph.pad0) {
                    if (j == 0) {
                        xs.am_tag = phase_tag(D, P.dep_ph0 - 1);  // the text head
                        xs.am_cnt = P.G;
                    } else {
                        // the last substep of the group before: its head's partials
                        const int g = group_of(starts, j);
                        int pj0, pnj, b0, b1;
                        group_bounds(starts, S, g - 1, pj0, pnj);
                        substep_ctas(P.G, pnj, pnj - 1, b0, b1);
                        xs.am_tag = phase_tag(D, P.dep_ph0 + g * P.dep_ph_stride - 1);
                        xs.am_cnt = b1 - b0;
                    }
                }
            } else {
                xs = XSrc{P.u + (size_t)j * dd, us, in_tag, P.dep_attn_norm + (size_t)ph.l * dd};
            }
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, xs, n, sm, stage, ms, EpiDQKV{ph.l, j, tag});
        }
        case PH_DATTN: return phase_dattn(P, ph.l, ph.pad0, ph.pad1, starts, n, in_tag, tag, sm);
        case PH_DO:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.dat + (size_t)j * dd, (long long)S * dd, in_tag}, n, sm, stage,
                                      ms, EpiResid{P.u + (size_t)j * dd, (long long)S * dd, res_tag, tag});
        case PH_DGU:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt,
                                      XSrc{P.u + (size_t)j * dd, (long long)S * dd, in_tag, P.dep_ffn_norm + (size_t)ph.l * dd},
                                      n, sm, stage, ms, EpiSwiglu{P.ds + (size_t)j * dF, (long long)S * dF, tag});
        case PH_DDOWN:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.ds + (size_t)j * dF, (long long)S * dF, in_tag}, n, sm, stage,
                                      ms, EpiResid{P.u + (size_t)j * dd, (long long)S * dd, res_tag, tag});
        case PH_DHEAD:
            return matrix_phase<TW, BG>(P, ph, phi, c, cnt, XSrc{P.u + (size_t)j * dd, (long long)S * dd, in_tag, P.dep_out_norm}, n, sm,
                                      stage, ms, EpiLogits{P.dlogits + (size_t)j * P.C, (long long)S * P.C, P.C, nullptr, 0, tag,
                                                       P.damax + (size_t)j * P.G * 2, (long long)S * P.G * 2, c});
        case PH_FINAL: return phase_final(P, n, starts, sm);
        default: return true;
    }
}

// ------------------------------------------------------------------ the kernel

// Phases [ph0, ph1) of one step.  When the launch spans more than one phase,
// every CTA must be resident at once (cooperative launch), because CTAs wait
// for each other's tagged outputs.  maxrows sizes the shared memory.
template <typename TW, typename TKV, int BG>
__global__ void __launch_bounds__(is_mma(BG) ? MMA_THREADS : NT + 32, 1) step_kernel(Params P, int ph0, int ph1, int maxrows)
{
    extern __shared__ __align__(1024) char smem_raw[];
    // the tensor-core stages need 1024-byte alignment (the host adds the slack)
    char* abase = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Smem sm = is_mma(BG) ? smem_map_mma(abase) : smem_map(smem_raw, maxrows, BG);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        if constexpr (is_mma(BG)) {
            for (int k = 0; k < MMA_NSTAGE; ++k) {
                mbar_init(&sm.wfull[k], 1);
                mbar_init(&sm.bfull[k], 1);      // the producer's bulk copy of the activation chunk
                mbar_init(&sm.sempty[k], 1);
            }
            for (int k = 0; k < MMA_URING; ++k) {
                mbar_init(&sm.accf[k], 1);      // the MMA warp's commit of a unit
                mbar_init(&sm.tfree[k], NWARP);  // every consumer warp has read the unit's slot
            }
            mbar_init(sm.mdone, 1);
            mbar_init(sm.adone, 1);
        } else {
            for (int k = 0; k < (int)nstage_for(BG); ++k) {
                mbar_init(&sm.full[k], 1);
                mbar_init(&sm.empty[k], NWARP);  // every consumer warp releases every stage
            }
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (is_mma(BG)) {
        if (warp == NWARP + 1) tmem_alloc(sm.tslot, MMA_TMEM_COLS);
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
    // depformer groups of this step: bit j of `known` stays set while every
    // slot supplies stream j's input token (read before any history write of
    // the step; the fence orders these reads before this CTA's later stores)
    // Bit k of `given` stays set while every slot's output for stream k is
    // settled without the depformer: supplied, or for a frame before 0.
    if (threadIdx.x == 0) {
        sm.misc[1] = 0xFFFF;
        sm.misc[2] = 0x1FFFE;
    }
    __syncthreads();
    if (ph1 > P.dep_ph0 && !bad) {
        for (int it = threadIdx.x; it < n * P.S; it += blockDim.x) {
            const int i = it / P.S, k = 1 + it % P.S;
            const int t = supplied_token(P, i, k);
            if (t < 0 && k < P.S) atomicAnd((unsigned*)&sm.misc[1], ~(1u << k));
            if (t < 0 && D->pos[i] - P.delays[k] >= 0) atomicAnd((unsigned*)&sm.misc[2], ~(1u << k));
        }
    }
    __threadfence();
    if constexpr (is_mma(BG)) tc_fence_before();
    __syncthreads();  // barrier init and the TMEM address visible to every thread; all threads agree on `bad`
    if constexpr (is_mma(BG)) tc_fence_after();
    if (bad) {
        if constexpr (is_mma(BG)) {
            if (warp == NWARP + 1) tmem_dealloc(*sm.tslot, MMA_TMEM_COLS);
        }
        return;
    }
    unsigned starts = 1u;
    {
        const unsigned known = (unsigned)sm.misc[1], given = (unsigned)sm.misc[2];
        // substeps [jend, S) only produce settled outputs: skipped when the context allows
        int jend = P.S;
        if (P.skip_settled)
            while (jend > 0 && ((given >> jend) & 1u)) --jend;
        int j0 = 0;
        for (int k = 1; k < P.S; ++k)
            if (k == jend || !((known >> k) & 1u) || k - j0 >= MAXGW) { starts |= 1u << k; j0 = k; }
        const int ngr = jend == 0 ? 0 : __popc(starts & ((1u << jend) - 1u));
        starts |= (unsigned)ngr << 24;
    }
    if (warp == NWARP) {
        if ((threadIdx.x & 31) == 0) {
            if constexpr (is_mma(BG)) producer_mma<TW>(P, ph0, ph1, n, starts, sm);
            else producer<TW, BG>(P, ph0, ph1, n, starts, sm);
        }
        return;
    }
    MmaState ms;
    ms.tbase = 0;
    ms.uc = 0;
    ms.ph0 = ph0;
    if constexpr (is_mma(BG)) {
        const uint32_t tbase = *sm.tslot;
        if (warp == NWARP + 1) {
            if ((threadIdx.x & 31) == 0) mma_issuer<TW>(P, ph0, ph1, n, starts, sm, tbase);
            __syncwarp();
            // tensor memory is freed once the consumers have read their last accumulator
            asm volatile("bar.sync 2, %0;" ::"n"(NT + 32) : "memory");
            tc_fence_after();
            tmem_dealloc(tbase, MMA_TMEM_COLS);
            return;
        }
        ms.tbase = tbase;
    }
    unsigned stage = 0;
    // depformer phases of groups that do not exist this step are skipped as a block
    const int dep_end = P.dep_ph0 + n_groups(starts) * P.dep_ph_stride;
    const int dep_all = P.dep_ph0 + P.S * P.dep_ph_stride;
    for (int ph = ph0; ph < ph1; ++ph) {
        if (ph == dep_end && dep_end < dep_all) {
            ph = dep_all;
            if (ph >= ph1) break;
        }
        if (threadIdx.x == 0) sm.misc[0] = ph;  // phase index for the in-phase stamps
        stamp(P, ph, 0);
        const Phase phs = P.phases[ph];
        if (!run_phase<TW, TKV, BG>(P, phs, ph, n, starts, sm, stage, ms)) break;
        if constexpr (is_mma(BG)) {
            if (phs.type == PH_DHEAD) {  // the next group's first phase waits for every CTA to get here
                csync();
                mark_phase_done(P, ph);
            }
        }
        stamp(P, ph, 3);
        // diagnostics: the latest end of this phase over all CTAs
        if (P.ptime && threadIdx.x == 0) atomicMax(P.ptime + (size_t)ph * 8 + 6, globaltimer_ns());
    }
    if constexpr (is_mma(BG)) {
        tc_fence_before();
        asm volatile("bar.arrive 2, %0;" ::"n"(NT + 32) : "memory");
    }
    stamp(P, ph1, 0);
}

}  // namespace
}  // namespace mfs
