// Tensor-core form of mfs_rvq_encode (Mimi's split RVQ argmin quantizer).
//
// Per stage, the squared distance |r - c|^2 = |r|^2 - 2 r.c + |c|^2 ranks the
// codewords of a frame by |c|^2 - 2 r.c, and r.c over all codewords and a
// tile of frames is a product [codewords x D] x [D x frames].  It runs on the
// tensor cores (tcgen05.mma, bf16 operands, fp32 accumulation): the codebook
// and the residuals are each split into a bf16 high part and the bf16 rounding
// of the rest, and the products hi.hi + hi.lo + lo.hi + lo.lo keep about 16
// significant bits (score error a few 1e-5 of sum_i |r_i c_i|), enough to pick
// candidates.  A frame's codewords fall into 8 classes by index mod 8; the best
// 2 of each class by that score (16 per frame) are then re-ranked by their
// exact fp32 distances, computed in the order of the CUDA-core kernel
// (mfs_rvq.cu: float4 chunks, one fmaf per component); the smallest wins, lower
// index on ties.  So the code equals the CUDA-core kernel's whenever the
// nearest codeword is among the 16, i.e. unless two codewords of its class score
// within that error of it (identical codewords score identically and keep the
// lower index first, so exact duplicates cannot push it out).
//
// A CTA takes 16 frames through all 8 stages.  Warp 4 (one lane) loads
// codebook tiles (128 codewords x 64 dimensions, high and low parts) with 2-D
// TMA copies into a ring of stages; warp 5 (one lane) issues the MMAs into one
// of two tensor-memory accumulators per codeword tile; warps 0-3 build the
// residuals' operand panel in shared memory, read each tile's scores (one
// codeword per thread), keep the best two of each class per frame, re-rank
// them exactly, and update the residuals.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/mfs.h"

namespace mfs {
void set_thread_error(const char* msg);  // defined with mfs_last_error
}

namespace {

constexpr int RQ_NF = 16;            // frames per CTA
constexpr int RQ_CW = 128;           // codewords per tile (tensor-memory lanes)
constexpr int RQ_KC = 64;            // dimensions per chunk (one 128-byte swizzle row of bf16)
constexpr int RQ_TILE = RQ_CW * RQ_KC * 2;  // 16 KB: one part of a codebook tile chunk
constexpr int RQ_STAGE = 2 * RQ_TILE;       // high and low parts
constexpr int RQ_CONS = 128;         // consumer threads (warps 0-3)
constexpr int RQ_THREADS = RQ_CONS + 64;
constexpr int RQ_KEEP = 2;           // best codewords kept per sub-list (8 sub-lists, one thread each, per frame)
constexpr int RQ_NCOL = 64;          // accumulator block: [A_hi x (B_hi | B_lo) | A_lo x (B_hi | B_lo)] columns
constexpr int RQ_NSPLIT = 1;         // blocks per accumulator: chunk kc accumulates into block kc % RQ_NSPLIT
constexpr int RQ_NACC = 2;           // accumulators (codeword tiles in flight between the MMAs and the consumers)
constexpr int RQ_TMEM = RQ_NACC * RQ_NSPLIT * RQ_NCOL;  // tensor-memory columns (a power of 2, 32..512)
constexpr int RQ_SCS = RQ_CW + 8;    // score row stride: the candidate scan's 32 lanes hit 32 banks
constexpr int RQ_MAXST = 6;          // ring stages at most
constexpr unsigned long long RQ_WAIT_NS = 2000000000ull;

__device__ __forceinline__ unsigned su32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint64_t* b, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_expect(uint64_t* b, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t* b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ unsigned long long gtime()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of parity `par`; false (and the error flag set) on timeout.
// The error flag and the clock are looked at every 256 polls (a global load per poll
// would put its latency on every hand-off).
__device__ __forceinline__ bool bar_wait(uint64_t* b, unsigned par, int* flag)
{
    unsigned long long t0 = 0;
    for (unsigned n = 0;; ++n) {
        unsigned ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
        if (ok) return true;
        if ((n & 255u) != 255u) continue;
        if (*(volatile int*)flag) return false;
        const unsigned long long t = gtime();
        if (t0 == 0) {
            t0 = t;
        } else if (t - t0 > RQ_WAIT_NS) {
            atomicExch(flag, 1);
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t sw128(unsigned saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void commit(uint64_t* b)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 columns of this warp's 32 tensor-memory lanes
__device__ __forceinline__ void tld16(uint32_t taddr, float (&v)[16])
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

// candidate order: smaller score first, lower index on ties
__device__ __forceinline__ bool cbetter(float s1, int i1, float s2, int i2) { return s1 < s2 || (s1 == s2 && i1 < i2); }

// Split fp32 codebooks [8][Cb][D] into bf16 high / low parts and |c|^2 per codeword.
__global__ void rq_split(const float* __restrict__ cb, long long n, int D, __nv_bfloat16* __restrict__ hi,
                         __nv_bfloat16* __restrict__ lo, float* __restrict__ norm)
{
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
        const float x = cb[k];
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        hi[k] = h;
        lo[k] = __float2bfloat16_rn(x - __bfloat162float(h));
    }
    // one warp per codeword for the norms
    const long long ncw = n / D;
    const int lane = threadIdx.x & 31;
    for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; w < ncw;
         w += (long long)gridDim.x * blockDim.x / 32) {
        float s = 0.f;
        for (int e = lane; e < D; e += 32) s = fmaf(cb[w * D + e], cb[w * D + e], s);
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) norm[w] = s;
    }
}

struct RqSmem {
    uint64_t full[RQ_MAXST], empty[RQ_MAXST], accf[RQ_NACC], accfree[RQ_NACC], bready, mdone;
    uint32_t tslot;
};

// Dynamic shared memory: [RqSmem | pad to 1024] stages [nst][32 KB] | operand panel [D/64][32 rows][128 B]
// | residuals [16][D] fp32 | scores [16][RQ_SCS] fp32 | chosen codes [16].
__global__ void __launch_bounds__(RQ_THREADS, 1) rq_kernel(const __grid_constant__ CUtensorMap mhi,
                                                           const __grid_constant__ CUtensorMap mlo,
                                                           const float* __restrict__ z_sem, const float* __restrict__ z_ac,
                                                           int T, int D, const float* __restrict__ cb, const float* __restrict__ norm,
                                                           int Cb, int nst, int32_t* __restrict__ codes, int* flag)
{
    extern __shared__ __align__(1024) char rq_raw[];
    char* base = (char*)(((uintptr_t)rq_raw + 1023) & ~(uintptr_t)1023);
    RqSmem* H = (RqSmem*)base;
    char* stages = base + 1024;
    const int KC = (D + RQ_KC - 1) / RQ_KC;
    char* panel = stages + (size_t)nst * RQ_STAGE;              // KC x 4 KB
    float* res = (float*)(panel + (size_t)KC * 4096);           // [16][D]
    float* sc = res + (size_t)RQ_NF * D;                         // [16][128]
    int* scode = (int*)(sc + RQ_NF * RQ_SCS);                    // [16]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * RQ_NF, nf = min(RQ_NF, T - t0);
    const int CT = (Cb + RQ_CW - 1) / RQ_CW;
    if (tid == 0) {
        for (int k = 0; k < nst; ++k) {
            bar_init(&H->full[k], 1);
            bar_init(&H->empty[k], 1);
        }
        for (int k = 0; k < RQ_NACC; ++k) {
            bar_init(&H->accf[k], 1);
            bar_init(&H->accfree[k], 4);  // one arrival per consumer warp
        }
        bar_init(&H->bready, RQ_CONS);
        bar_init(&H->mdone, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&H->tslot)), "r"((unsigned)RQ_TMEM) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = H->tslot;

    if (warp == 4) {
        // producer: codebook tiles of every stage, in the MMA warp's order
        if (lane == 0) {
            unsigned s = 0;
            bool ok = true;
            for (int q = 0; q < 8 && ok; ++q)
                for (int ct = 0; ct < CT && ok; ++ct)
                    for (int kc = 0; kc < KC; ++kc, ++s) {
                        const int slot = (int)(s % nst);
                        if (!bar_wait(&H->empty[slot], ((s / nst) & 1u) ^ 1u, flag)) { ok = false; break; }
                        bar_expect(&H->full[slot], RQ_STAGE);
                        char* dst = stages + (size_t)slot * RQ_STAGE;
                        const int x = kc * RQ_KC, y = q * Cb + ct * RQ_CW;
                        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                                     ::"r"(su32(dst)), "l"(&mhi), "r"(x), "r"(y), "r"(su32(&H->full[slot])) : "memory");
                        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                                     ::"r"(su32(dst + RQ_TILE)), "l"(&mlo), "r"(x), "r"(y), "r"(su32(&H->full[slot])) : "memory");
                    }
            if (!ok)  // wait (bounded) for the copies in flight
                for (unsigned k = s > (unsigned)nst ? s - nst : 0; k < s; ++k) {
                    const unsigned long long tw = gtime();
                    for (;;) {
                        unsigned d;
                        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                                     : "=r"(d) : "r"(su32(&H->full[k % nst])), "r"((k / nst) & 1u) : "memory");
                        if (d || gtime() - tw > RQ_WAIT_NS) break;
                    }
                }
        }
        return;
    }
    if (warp == 5) {
        // MMA: tiles take the accumulators in turn; per chunk 4 K-steps x (A_hi, A_lo) x B (hi | lo rows)
        // into block kc % RQ_NSPLIT of the tile's accumulator
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(32 >> 3) << 17) | ((uint32_t)(RQ_CW >> 4) << 24);
            unsigned s = 0, tcount = 0;
            bool ok = true;
            for (int q = 0; q < 8 && ok; ++q) {
                if (!bar_wait(&H->bready, (unsigned)q & 1u, flag)) { ok = false; break; }
                for (int ct = 0; ct < CT && ok; ++ct, ++tcount) {
                    const int ab = (int)(tcount % RQ_NACC);
                    if (!bar_wait(&H->accfree[ab], ((tcount / RQ_NACC) & 1u) ^ 1u, flag)) { ok = false; break; }
                    fence_after();
                    for (int kc = 0; kc < KC; ++kc, ++s) {
                        const uint32_t d = tbase + (uint32_t)((ab * RQ_NSPLIT + kc % RQ_NSPLIT) * RQ_NCOL);
                        const int slot = (int)(s % nst);
                        if (!bar_wait(&H->full[slot], (s / nst) & 1u, flag)) { ok = false; break; }
                        fence_after();
                        const unsigned sa = su32(stages + (size_t)slot * RQ_STAGE);
                        const uint64_t ahi = sw128(sa), alo = sw128(sa + RQ_TILE), bd = sw128(su32(panel + (size_t)kc * 4096));
#pragma unroll
                        for (int kk = 0; kk < RQ_KC / 16; ++kk) {
                            const uint32_t acc = (kc >= RQ_NSPLIT || kk > 0) ? 1u : 0u;
                            mma(d, ahi + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, acc);
                            mma(d + 32, alo + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, acc);
                        }
                        commit(&H->empty[slot]);
                    }
                    commit(&H->accf[ab]);
                }
            }
            // every MMA issued has completed before tensor memory is freed (a barrier of
            // its own: an extra phase on an accumulator barrier could pass a consumer by)
            commit(&H->mdone);
            const unsigned long long tw = gtime();
            for (;;) {
                unsigned dn;
                asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                             : "=r"(dn) : "r"(su32(&H->mdone)), "r"(0u) : "memory");
                if (dn || gtime() - tw > RQ_WAIT_NS) break;
            }
        }
        __syncwarp();
        asm volatile("bar.sync 1, %0;" ::"n"(RQ_CONS + 32) : "memory");
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"((unsigned)RQ_TMEM) : "memory");
        return;
    }

    // consumers (warps 0-3): tensor-memory lane = codeword of the tile = 32 warp + lane
    const int D4 = D / 4;
    const int f8 = tid >> 3, s8 = tid & 7;  // candidate lists: frame f8 (< 16), sub-list s8
    const int nsb = KC < RQ_NSPLIT ? KC : RQ_NSPLIT;  // blocks of an accumulator in use
    unsigned tcount = 0;
    int ok = 1;
    for (int q = 0; q < 8; ++q) {
        if (q <= 1) {
            const float4* z = reinterpret_cast<const float4*>(q == 0 ? z_sem : z_ac);
            for (int k = tid; k < RQ_NF * D4; k += RQ_CONS) {
                const int f = k / D4;
                reinterpret_cast<float4*>(res)[k] = f < nf ? __ldg(z + (size_t)(t0 + f) * D4 + k % D4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        }
        // operand panel: rows 0..15 the residuals' high parts, 16..31 the low parts
        for (int it = tid; it < KC * 32 * 8; it += RQ_CONS) {
            const int kc = it / 256, row = (it / 8) % 32, c16 = it % 8;
            const int f = row % 16, k0 = kc * RQ_KC + c16 * 8;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float a = 0.f, b = 0.f;
                if (k0 + e < D) a = res[f * D + k0 + e];
                if (k0 + e + 1 < D) b = res[f * D + k0 + e + 1];
                __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                if (row >= 16) {
                    const float2 hf = __bfloat1622float2(h);
                    h = __floats2bfloat162_rn(a - hf.x, b - hf.y);
                }
                w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(panel + (size_t)kc * 4096 + (row >> 3) * 1024 + (row & 7) * 128 + ((c16 ^ (row & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive(&H->bready);
        // candidates of frame f8, sub-list s8 (codewords c with c % 8 == s8 within each tile)
        float cs[RQ_KEEP];
        int ci[RQ_KEEP];
#pragma unroll
        for (int k = 0; k < RQ_KEEP; ++k) { cs[k] = INFINITY; ci[k] = 0x7fffffff; }
        for (int ct = 0; ct < CT; ++ct, ++tcount) {
            const int c = ct * RQ_CW + 32 * warp + lane;
            const float nc = c < Cb ? __ldg(norm + (size_t)q * Cb + c) : 0.f;  // in flight during the wait
            const int ab = (int)(tcount % RQ_NACC);
            if (ok && !bar_wait(&H->accf[ab], (tcount / RQ_NACC) & 1u, flag)) ok = 0;
            fence_after();
            float v0[16], v1[16], v2[16], v3[16];
            const uint32_t ta = tbase + ((uint32_t)(32 * warp) << 16) + (uint32_t)(ab * RQ_NSPLIT * RQ_NCOL);
            tld16(ta, v0);       // A_hi x B_hi
            tld16(ta + 16, v1);  // A_hi x B_lo
            tld16(ta + 32, v2);  // A_lo x B_hi
            tld16(ta + 48, v3);  // A_lo x B_lo
            for (int b = 1; b < nsb; ++b) {  // the other blocks of the tile's K
                float w[16];
                tld16(ta + b * RQ_NCOL, w);
#pragma unroll
                for (int e = 0; e < 16; ++e) v0[e] += w[e];
                tld16(ta + b * RQ_NCOL + 16, w);
#pragma unroll
                for (int e = 0; e < 16; ++e) v1[e] += w[e];
                tld16(ta + b * RQ_NCOL + 32, w);
#pragma unroll
                for (int e = 0; e < 16; ++e) v2[e] += w[e];
                tld16(ta + b * RQ_NCOL + 48, w);
#pragma unroll
                for (int e = 0; e < 16; ++e) v3[e] += w[e];
            }
            fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&H->accfree[ab]);
#pragma unroll
            for (int f = 0; f < RQ_NF; ++f)
                sc[f * RQ_SCS + 32 * warp + lane] = c < Cb ? nc - 2.f * ((v0[f] + v1[f]) + (v2[f] + v3[f])) : INFINITY;
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
            for (int k = s8; k < RQ_CW; k += 8) {  // keep the sub-list's best two (cs[0] <= cs[1])
                const float v = sc[f8 * RQ_SCS + k];
                const int ix = ct * RQ_CW + k;
                if (cbetter(v, ix, cs[1], ci[1])) {
                    const bool first = cbetter(v, ix, cs[0], ci[0]);
                    cs[1] = first ? cs[0] : v;
                    ci[1] = first ? ci[0] : ix;
                    cs[0] = first ? v : cs[0];
                    ci[0] = first ? ix : ci[0];
                }
            }
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        }
        // exact fp32 distances of the lane's two candidates (the CUDA-core kernel's arithmetic:
        // float4 chunks in order, one fmaf per component; the two chains interleave), then the
        // least over the frame's 16 candidates (8 lanes)
        const float4* book = reinterpret_cast<const float4*>(cb + (size_t)q * Cb * D);
        const float4* r4 = reinterpret_cast<const float4*>(res + (size_t)f8 * D);
        const float4* row0 = book + (size_t)(ci[0] < Cb ? ci[0] : 0) * D4;
        const float4* row1 = book + (size_t)(ci[1] < Cb ? ci[1] : 0) * D4;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
        for (int e = 0; e < D4; ++e) {
            const float4 x = r4[e], w0 = __ldg(row0 + e), w1 = __ldg(row1 + e);
            const float a0 = x.x - w0.x, b0 = x.y - w0.y, c0 = x.z - w0.z, d0 = x.w - w0.w;
            const float a1 = x.x - w1.x, b1 = x.y - w1.y, c1 = x.z - w1.z, d1 = x.w - w1.w;
            acc0 = fmaf(a0, a0, acc0);
            acc1 = fmaf(a1, a1, acc1);
            acc0 = fmaf(b0, b0, acc0);
            acc1 = fmaf(b1, b1, acc1);
            acc0 = fmaf(c0, c0, acc0);
            acc1 = fmaf(c1, c1, acc1);
            acc0 = fmaf(d0, d0, acc0);
            acc1 = fmaf(d1, d1, acc1);
        }
        float bd = INFINITY;
        int bi = 0x7fffffff;
        if (ci[0] < Cb && cbetter(acc0, ci[0], bd, bi)) { bd = acc0; bi = ci[0]; }
        if (ci[1] < Cb && cbetter(acc1, ci[1], bd, bi)) { bd = acc1; bi = ci[1]; }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {  // the frame's 8 lanes
            const float v2 = __shfl_xor_sync(0xffffffffu, bd, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
            if (cbetter(v2, i2, bd, bi)) { bd = v2; bi = i2; }
        }
        if (s8 == 0) {
            scode[f8] = bi;
            if (f8 < nf) codes[(size_t)(t0 + f8) * 8 + q] = bi;
        }
        asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        if (q >= 1 && q < 7) {  // the residual for the next acoustic stage
            for (int k = tid; k < RQ_NF * D4; k += RQ_CONS) {
                const int f = k / D4, e = k % D4;
                const int cw = scode[f] < Cb ? scode[f] : 0;
                const float4 w = __ldg(book + (size_t)cw * D4 + e);
                float4 x = reinterpret_cast<float4*>(res)[k];
                x.x -= w.x;
                x.y -= w.y;
                x.z -= w.z;
                x.w -= w.w;
                reinterpret_cast<float4*>(res)[k] = x;
            }
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        }
    }
    // a wait that gave up (here or in another CTA) leaves this CTA's frames with code -1
    if (*(volatile int*)flag)
        for (int k = tid; k < nf * 8; k += RQ_CONS) codes[(size_t)t0 * 8 + k] = -1;
    fence_before();
    asm volatile("bar.arrive 1, %0;" ::"n"(RQ_CONS + 32) : "memory");
}

int fail(int code, const char* msg)
{
    mfs::set_thread_error(msg);
    return code;
}

size_t rq_smem(int D, int nst)
{
    const int KC = (D + RQ_KC - 1) / RQ_KC;
    return 1024 + 1024 + (size_t)nst * RQ_STAGE + (size_t)KC * 4096 + (size_t)RQ_NF * D * 4 + RQ_NF * RQ_SCS * 4 + 64;
}

}  // namespace

namespace mfs {

// The tensor-core path of mfs_rvq_encode (D a multiple of 8); returns MFS_OK or
// an error after setting the thread's message.  Scratch (the split codebooks
// and their norms, 4 Cb D + 4 Cb bytes per codebook, and an error flag) comes
// from the stream-ordered pool and is released on the stream.
int rvq_encode_mma(const float* z_sem, const float* z_ac, int T, int D, const float* codebooks, int Cb, int32_t* codes,
                   cudaStream_t st)
{
    int nst = RQ_MAXST;
    while (nst > 2 && rq_smem(D, nst) > 227 * 1024) --nst;
    const size_t smem = rq_smem(D, nst);
    if (smem > 227 * 1024) return fail(MFS_E_ARG, "rvq: dimension too large for the tensor-core path");
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess || !fn)
            return fail(MFS_E_CUDA, "rvq: cuTensorMapEncodeTiled is not available");
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    const long long n = 8LL * Cb * D;
    char* scratch = nullptr;
    const size_t bytes = (size_t)n * 2 * 2 + (size_t)8 * Cb * 4 + 256;
    cudaError_t e = cudaMallocAsync((void**)&scratch, bytes, st);
    if (e != cudaSuccess) return fail(MFS_E_CUDA, "rvq: scratch allocation failed");
    __nv_bfloat16* hi = (__nv_bfloat16*)scratch;
    __nv_bfloat16* lo = hi + n;
    float* norm = (float*)(lo + n);
    int* flag = (int*)(norm + (size_t)8 * Cb);
    CUtensorMap mhi, mlo;
    const cuuint64_t dim[2] = {(cuuint64_t)D, (cuuint64_t)(8LL * Cb)};
    const cuuint64_t stride[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {(cuuint32_t)RQ_KC, (cuuint32_t)RQ_CW};
    const cuuint32_t es[2] = {1, 1};
    CUresult r1 = encode(&mhi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hi, dim, stride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = encode(&mlo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lo, dim, stride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    int rc = MFS_OK;
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) rc = fail(MFS_E_CUDA, "rvq: tensor map encoding failed");
    if (rc == MFS_OK) e = cudaMemsetAsync(flag, 0, sizeof(int), st);
    if (rc == MFS_OK && e == cudaSuccess) {
        rq_split<<<304, 256, 0, st>>>(codebooks, n, D, hi, lo, norm);
        e = cudaGetLastError();
    }
    if (rc == MFS_OK && e == cudaSuccess) e = cudaFuncSetAttribute(rq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (rc == MFS_OK && e == cudaSuccess) {
        rq_kernel<<<(T + RQ_NF - 1) / RQ_NF, RQ_THREADS, smem, st>>>(mhi, mlo, z_sem, z_ac, T, D, codebooks, norm, Cb, nst, codes,
                                                                     flag);
        e = cudaGetLastError();
    }
    if (rc == MFS_OK && e != cudaSuccess) {
        char buf[160];
        snprintf(buf, sizeof buf, "rvq (tensor cores) launch failed: %s", cudaGetErrorString(e));
        rc = fail(MFS_E_CUDA, buf);
    }
    cudaFreeAsync(scratch, st);
    return rc;
}

}  // namespace mfs
