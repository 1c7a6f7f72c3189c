// Tensor-core form of mfs_rvq_encode (Mimi's split RVQ argmin quantizer).
//
// Per stage, the squared distance |r - c|^2 = |r|^2 - 2 r.c + |c|^2 ranks the
// codewords of a frame by |c|^2 - 2 r.c, and r.c over all codewords and a
// tile of frames is a product [codewords x D] x [D x frames].  It runs on the
// tensor cores (tcgen05.mma, bf16 operands, fp32 accumulation): the codebook
// and the residuals are each split into a bf16 high part and the bf16 rounding
// of the rest, and the products hi.hi + hi.lo + lo.hi + lo.lo keep about 16
// significant bits (score error below 2^-14 |r| |c|), enough to pick
// candidates.  A frame's codewords fall into 8 classes by index mod 8; the best
// 2 of each class by that score are the candidates, and those whose score is
// within 2^-12 (|r|^2 + |c|^2) of the frame's best score (a band four times the
// error bound, so no other candidate can have the least distance) are re-ranked
// by their fp32 distances: a warp per codeword, each lane summing the squared
// differences of its float4 chunks in order, then a fixed tree over the lanes.
// The smallest wins, lower index on ties.  So the code is the fp32 argmin
// (with this summation order) unless two codewords of the nearest's class
// score within that error of it (identical codewords score identically and
// keep the lower index first, so exact duplicates cannot push it out).
//
// A pair of CTAs takes 32 frames through all 8 stages (while its shared memory
// fits, D up to about 520; larger D: one CTA per 16 frames), each CTA every other
// 128-codeword tile: a tensor-core
// instruction costs about the same for 32 and 64 columns, so 32 frames per
// instruction halve the instructions per frame, and the pair keeps every SM
// busy.  In a CTA, warp 4 (one lane) loads codebook tiles (128 codewords x 64
// dimensions, high and low parts) with 2-D TMA copies into a ring of stages;
// warp 5 (one lane) issues the MMAs into one of two tensor-memory accumulators
// per tile; warps 0-3 build the residuals' operand panel in shared memory, read
// each tile's scores (one codeword per thread), keep the best two of each class
// per frame, and re-rank those in the band.  The two CTAs of a pair then exchange
// each frame's best (distance, index) through tagged words in global memory,
// take the same winner, and update their copies of the residuals.
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

constexpr int RQ_CW = 128;           // codewords per tile (tensor-memory lanes)
constexpr int RQ_KC = 64;            // dimensions per chunk (one 128-byte swizzle row of bf16)
constexpr int RQ_TILE = RQ_CW * RQ_KC * 2;  // 16 KB: one part of a codebook tile chunk
constexpr int RQ_STAGE = 2 * RQ_TILE;       // high and low parts
constexpr int RQ_CONS = 128;         // consumer threads (warps 0-3)
constexpr int RQ_THREADS = RQ_CONS + 64;
constexpr int RQ_NACC = 2;           // accumulators (codeword tiles in flight between the MMAs and the consumers)
constexpr int RQ_SCS = RQ_CW + 8;    // score row stride (shared-memory banks of the candidate scan)
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

__device__ __forceinline__ bool bar_try(uint64_t* b, unsigned par)
{
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `par`; false (and the error flag set) on timeout.
// The error flag and the clock are looked at every 256 polls (a global load per poll
// would put its latency on every hand-off).
__device__ __forceinline__ bool bar_wait(uint64_t* b, unsigned par, int* flag)
{
    unsigned long long t0 = 0;
    for (unsigned n = 0;; ++n) {
        if (bar_try(b, par)) return true;
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

// Bounded wait (no error flag: used only to drain before leaving)
__device__ __forceinline__ void bar_drain(uint64_t* b, unsigned par)
{
    const unsigned long long t0 = gtime();
    while (!bar_try(b, par) && gtime() - t0 <= RQ_WAIT_NS) {
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

__device__ __forceinline__ void st_tagged(uint2* p, unsigned bits, unsigned tag)
{
    const unsigned long long x = ((unsigned long long)tag << 32) | bits;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(x) : "memory");
}

__device__ __forceinline__ uint2 ld_tagged(const uint2* p)
{
    unsigned long long x;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
    return make_uint2((unsigned)x, (unsigned)(x >> 32));
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

// NF frames per frame group (16 or 32: the MMAs' N is 2 NF, high and low parts of
// the residuals), G CTAs per group (1 or 2; CTA r takes tiles r, r + G, ...).
template <int NF>
struct RqShape {
    static constexpr int NCOL = 4 * NF;         // accumulator: [A_hi B_hi | A_hi B_lo | A_lo B_hi | A_lo B_lo]
    static constexpr int TMEM = RQ_NACC * NCOL;  // tensor-memory columns (128 or 256)
    static constexpr int PB = 2 * NF * 128;      // panel bytes per 64-dimension chunk
    static constexpr int TPF = RQ_CONS / NF;     // scan threads per frame (8 or 4)
    static constexpr int CPT = 8 / TPF;          // index classes (mod 8) per scan thread (1 or 2)
};

size_t rq_smem_of(int NF, int D, int nst)
{
    const int KC = (D + RQ_KC - 1) / RQ_KC;
    return 1024 + 1024 + (size_t)nst * RQ_STAGE + (size_t)KC * 2 * NF * 128 + (size_t)NF * D * 4 +
           (size_t)NF * RQ_SCS * 4 + (size_t)NF * 4 + RQ_CW * 4 + (size_t)NF * 4;
}

// Dynamic shared memory: [RqSmem | pad to 1024] stages [nst][32 KB] | operand panel [D/64][2 NF rows][128 B]
// | residuals [NF][D] fp32 | scores [NF][RQ_SCS] fp32 | chosen codes [NF] | the tile's |c|^2 [128]
// | |r|^2 per frame [NF].
// xb (G = 2): [groups][2][NF][2] tagged words, the pair's per-frame best {distance}, {index}.
template <int NF, int G>
__global__ void __launch_bounds__(RQ_THREADS, 1) rq_kernel(const __grid_constant__ CUtensorMap mhi,
                                                           const __grid_constant__ CUtensorMap mlo,
                                                           const float* __restrict__ z_sem, const float* __restrict__ z_ac,
                                                           int T, int D, const float* __restrict__ cb, const float* __restrict__ norm,
                                                           int Cb, int nst, int32_t* __restrict__ codes, int* flag, uint2* xb,
                                                           unsigned tag0)
{
    using S = RqShape<NF>;
    extern __shared__ __align__(1024) char rq_raw[];
    char* base = (char*)(((uintptr_t)rq_raw + 1023) & ~(uintptr_t)1023);
    RqSmem* H = (RqSmem*)base;
    char* stages = base + 1024;
    const int KC = (D + RQ_KC - 1) / RQ_KC;
    char* panel = stages + (size_t)nst * RQ_STAGE;              // KC x PB
    float* res = (float*)(panel + (size_t)KC * S::PB);           // [NF][D]
    float* sc = res + (size_t)NF * D;                            // [NF][RQ_SCS]
    int* scode = (int*)(sc + NF * RQ_SCS);                       // [NF]
    float* scn = (float*)(scode + NF);                           // [RQ_CW] the tile's codeword norms
    float* srr = scn + RQ_CW;                                    // [NF] |r|^2 of each frame
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = (int)blockIdx.x / G, rk = (int)blockIdx.x % G;
    const int t0 = grp * NF, nf = min(NF, T - t0);
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
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&H->tslot)), "r"((unsigned)S::TMEM) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = H->tslot;

    if (warp == 4) {
        // producer: this CTA's codebook tiles of every stage, in the MMA warp's order
        if (lane == 0) {
            unsigned s = 0;
            bool ok = true;
            for (int q = 0; q < 8 && ok; ++q)
                for (int ct = rk; ct < CT && ok; ct += G)
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
                for (unsigned k = s > (unsigned)nst ? s - nst : 0; k < s; ++k) bar_drain(&H->full[k % nst], (k / nst) & 1u);
        }
        return;
    }
    if (warp == 5) {
        // MMA: tiles take the accumulators in turn; per chunk 4 K-steps x (A_hi, A_lo) x B (hi | lo rows)
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)((2 * NF) >> 3) << 17) |
                                   ((uint32_t)(RQ_CW >> 4) << 24);
            unsigned s = 0, tcount = 0;
            bool ok = true;
            for (int q = 0; q < 8 && ok; ++q) {
                if (!bar_wait(&H->bready, (unsigned)q & 1u, flag)) { ok = false; break; }
                for (int ct = rk; ct < CT && ok; ct += G, ++tcount) {
                    const int ab = (int)(tcount % RQ_NACC);
                    if (!bar_wait(&H->accfree[ab], ((tcount / RQ_NACC) & 1u) ^ 1u, flag)) { ok = false; break; }
                    fence_after();
                    const uint32_t d = tbase + (uint32_t)(ab * S::NCOL);
                    for (int kc = 0; kc < KC; ++kc, ++s) {
                        const int slot = (int)(s % nst);
                        if (!bar_wait(&H->full[slot], (s / nst) & 1u, flag)) { ok = false; break; }
                        fence_after();
                        const unsigned sa = su32(stages + (size_t)slot * RQ_STAGE);
                        const uint64_t ahi = sw128(sa), alo = sw128(sa + RQ_TILE), bd = sw128(su32(panel + (size_t)kc * S::PB));
#pragma unroll
                        for (int kk = 0; kk < RQ_KC / 16; ++kk) {
                            const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
                            mma(d, ahi + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, acc);
                            mma(d + 2 * NF, alo + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, acc);
                        }
                        commit(&H->empty[slot]);
                    }
                    commit(&H->accf[ab]);
                }
            }
            // every MMA issued has completed before tensor memory is freed (a barrier of
            // its own: an extra phase on an accumulator barrier could pass a consumer by)
            commit(&H->mdone);
            bar_drain(&H->mdone, 0u);
        }
        __syncwarp();
        asm volatile("bar.sync 1, %0;" ::"n"(RQ_CONS + 32) : "memory");
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"((unsigned)S::TMEM) : "memory");
        return;
    }

    // consumers (warps 0-3): tensor-memory lane = codeword of the tile = 32 warp + lane
    const int D4 = D / 4;
    const int fs = tid / S::TPF, js = tid % S::TPF;  // scan: frame fs, index classes js CPT .. js CPT + CPT - 1
    unsigned tcount = 0;
    int ok = 1;
    for (int q = 0; q < 8; ++q) {
        if (q <= 1) {
            const float4* z = reinterpret_cast<const float4*>(q == 0 ? z_sem : z_ac);
            for (int k0 = tid; k0 < NF * D4; k0 += 4 * RQ_CONS) {  // four loads in flight
                float4 x[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k = k0 + j * RQ_CONS;
                    x[j] = k < NF * D4 && k / D4 < nf ? __ldg(z + (size_t)(t0 + k / D4) * D4 + k % D4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (k0 + j * RQ_CONS < NF * D4) reinterpret_cast<float4*>(res)[k0 + j * RQ_CONS] = x[j];
            }
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        }
        // operand panel: rows 0 .. NF-1 the residuals' high parts, NF .. 2 NF-1 the low parts
        for (int it = tid; it < KC * 2 * NF * 8; it += RQ_CONS) {
            const int kc = it / (2 * NF * 8), row = (it / 8) % (2 * NF), c16 = it % 8;
            const int f = row % NF, k0 = kc * RQ_KC + c16 * 8;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float a = 0.f, b = 0.f;
                if (k0 + e < D) a = res[f * D + k0 + e];
                if (k0 + e + 1 < D) b = res[f * D + k0 + e + 1];
                __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                if (row >= NF) {
                    const float2 hf = __bfloat1622float2(h);
                    h = __floats2bfloat162_rn(a - hf.x, b - hf.y);
                }
                w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(panel + (size_t)kc * S::PB + (row >> 3) * 1024 + (row & 7) * 128 + ((c16 ^ (row & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive(&H->bready);
        for (int f = warp; f < NF; f += RQ_CONS / 32) {  // |r|^2 per frame (for the re-rank's band)
            float rr = 0.f;
            for (int v = lane; v < D4; v += 32) {
                const float4 x = reinterpret_cast<const float4*>(res + (size_t)f * D)[v];
                rr = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, rr))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) rr += __shfl_xor_sync(0xffffffffu, rr, o);
            if (lane == 0) srr[f] = rr;
        }
        // the best two codewords of frame fs in each of its classes (cs[u][0] <= cs[u][1])
        float cs[S::CPT][2], cn[S::CPT][2];  // scores and |c|^2 of the kept codewords
        int ci[S::CPT][2];
#pragma unroll
        for (int u = 0; u < S::CPT; ++u) {
            cs[u][0] = cs[u][1] = INFINITY;
            cn[u][0] = cn[u][1] = 0.f;
            ci[u][0] = ci[u][1] = 0x7fffffff;
        }
        for (int ct = rk; ct < CT; ct += G, ++tcount) {
            const int c = ct * RQ_CW + 32 * warp + lane;
            const float nc = c < Cb ? __ldg(norm + (size_t)q * Cb + c) : 0.f;  // in flight during the wait
            const int ab = (int)(tcount % RQ_NACC);
            if (ok && !bar_wait(&H->accf[ab], (tcount / RQ_NACC) & 1u, flag)) ok = 0;
            fence_after();
            const uint32_t ta = tbase + ((uint32_t)(32 * warp) << 16) + (uint32_t)(ab * S::NCOL);
#pragma unroll
            for (int h = 0; h < NF / 16; ++h) {
                float v0[16], v1[16], v2[16], v3[16];
                tld16(ta + 16 * h, v0);           // A_hi x B_hi
                tld16(ta + NF + 16 * h, v1);      // A_hi x B_lo
                tld16(ta + 2 * NF + 16 * h, v2);  // A_lo x B_hi
                tld16(ta + 3 * NF + 16 * h, v3);  // A_lo x B_lo
#pragma unroll
                for (int f = 0; f < 16; ++f)
                    sc[(16 * h + f) * RQ_SCS + 32 * warp + lane] = c < Cb ? nc - 2.f * ((v0[f] + v1[f]) + (v2[f] + v3[f])) : INFINITY;
            }
            scn[32 * warp + lane] = nc;
            fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&H->accfree[ab]);
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
#pragma unroll
            for (int u = 0; u < S::CPT; ++u)
                for (int k = js * S::CPT + u; k < RQ_CW; k += 8) {
                    const float v = sc[fs * RQ_SCS + k];
                    const int ix = ct * RQ_CW + k;
                    if (cbetter(v, ix, cs[u][1], ci[u][1])) {
                        const bool first = cbetter(v, ix, cs[u][0], ci[u][0]);
                        const float nv = scn[k];
                        cs[u][1] = first ? cs[u][0] : v;
                        ci[u][1] = first ? ci[u][0] : ix;
                        cn[u][1] = first ? cn[u][0] : nv;
                        cs[u][0] = first ? v : cs[u][0];
                        ci[u][0] = first ? ix : ci[u][0];
                        cn[u][0] = first ? nv : cn[u][0];
                    }
                }
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        }
        // the frame's candidates (16 per frame and CTA) that can still hold its least distance:
        // scores within 2^-12 (|r|^2 + |c|^2) of the frame's best score (the score's error is
        // below 2^-14 |r| |c|, so no candidate outside the band can win); the rest are dropped
        constexpr int NCAND = 2 * S::CPT;
        int* cand = reinterpret_cast<int*>(sc);               // [NF][16] indices (0x7fffffff: none)
        int* wl = cand + NF * 16;                             // [4 warps][NF * 4] the warp's candidates: frame << 24 | index
        float* fbd = sc + NF * 16 + NF * 16;                  // [NF] the CTA's best distance per frame
        int* fbi = reinterpret_cast<int*>(fbd + NF);          // [NF] and its index
        {
            float smin = cs[0][0];
#pragma unroll
            for (int u = 1; u < S::CPT; ++u) smin = fminf(smin, cs[u][0]);
#pragma unroll
            for (int o = 1; o < S::TPF; o <<= 1) smin = fminf(smin, __shfl_xor_sync(0xffffffffu, smin, o));
            const float rr = srr[fs];
#pragma unroll
            for (int k = 0; k < NCAND; ++k) {
                const int ix = ci[k / 2][k % 2];
                const bool keep = ix < Cb && !(cs[k / 2][k % 2] > smin + 0x1p-12f * (rr + cn[k / 2][k % 2]));
                cand[fs * 16 + js * NCAND + k] = keep ? ix : 0x7fffffff;
            }
        }
        if (tid < NF) { fbd[tid] = INFINITY; fbi[tid] = 0x7fffffff; }
        asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        // each warp gathers the kept candidates of its frames (f = warp + 4 i) into a list, then
        // computes their fp32 distances four at a time: lane L sums the squared differences of
        // float4 chunks L, L + 32, ... in order (coalesced rows), then a fixed tree over the
        // lanes; the smallest per frame wins, lower index on ties
        const float4* book = reinterpret_cast<const float4*>(cb + (size_t)q * Cb * D);
        {
            int* mylist = wl + warp * (NF * 4);
            int cnt = 0;
            for (int s0 = 0; s0 < NF * 4; s0 += 32) {  // the warp's NF / 4 frames x 16 slots
                const int sl = s0 + lane, f = warp + 4 * (sl / 16);
                const int ix = cand[f * 16 + sl % 16];
                const bool valid = ix < Cb;
                const unsigned m = __ballot_sync(0xffffffffu, valid);
                if (valid) mylist[cnt + __popc(m & ((1u << lane) - 1u))] = (f << 24) | ix;
                cnt += __popc(m);
            }
            __syncwarp();
            for (int e0 = 0; e0 < cnt; e0 += 4) {
                int ent[4];
                float acc[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ent[j] = e0 + j < cnt ? mylist[e0 + j] : -1;
                    acc[j] = 0.f;
                }
                for (int v = lane; v < D4; v += 32) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (ent[j] < 0) continue;
                        const float4 x = reinterpret_cast<const float4*>(res + (size_t)(ent[j] >> 24) * D)[v];
                        const float4 w = __ldg(book + (size_t)(ent[j] & 0xffffff) * D4 + v);
                        const float a = x.x - w.x, bb = x.y - w.y, c2 = x.z - w.z, d2 = x.w - w.w;
                        acc[j] = fmaf(a, a, acc[j]);
                        acc[j] = fmaf(bb, bb, acc[j]);
                        acc[j] = fmaf(c2, c2, acc[j]);
                        acc[j] = fmaf(d2, d2, acc[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
                if (lane == 0)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (ent[j] < 0) continue;
                        const int f = ent[j] >> 24, ix = ent[j] & 0xffffff;
                        if (cbetter(acc[j], ix, fbd[f], fbi[f])) { fbd[f] = acc[j]; fbi[f] = ix; }
                    }
            }
        }
        asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        if (tid < NF) {
            const int f = tid;
            float bd = fbd[f];
            int bi = fbi[f];
            if (G == 2) {
                // the pair's other half: publish this CTA's best, take the other's (same rule, so
                // both CTAs choose the same codeword)
                const unsigned tag = tag0 + (unsigned)q;
                uint2* mine = xb + (((size_t)grp * 2 + rk) * NF + f) * 2;
                const uint2* peer = xb + (((size_t)grp * 2 + (1 - rk)) * NF + f) * 2;
                st_tagged(mine, __float_as_uint(bd), tag);
                st_tagged(mine + 1, (unsigned)bi, tag);
                unsigned long long tw = 0;
                for (unsigned n = 0; ok; ++n) {
                    const uint2 pa = ld_tagged(peer), pb = ld_tagged(peer + 1);
                    if (pa.y == tag && pb.y == tag) {
                        const float pd = __uint_as_float(pa.x);
                        const int pi = (int)pb.x;
                        if (cbetter(pd, pi, bd, bi)) { bd = pd; bi = pi; }
                        break;
                    }
                    if ((n & 63u) != 63u) continue;
                    if (*(volatile int*)flag) { ok = 0; break; }
                    const unsigned long long t = gtime();
                    if (tw == 0) {
                        tw = t;
                    } else if (t - tw > RQ_WAIT_NS) {
                        atomicExch(flag, 1);
                        ok = 0;
                    }
                }
            }
            scode[f] = bi;
            if (rk == 0 && f < nf) codes[(size_t)(t0 + f) * 8 + q] = bi;
        }
        asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        if (q >= 1 && q < 7) {  // the residual for the next acoustic stage (four rows' loads in flight)
            for (int k0 = tid; k0 < NF * D4; k0 += 4 * RQ_CONS) {
                float4 w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k = k0 + j * RQ_CONS;
                    w[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (k < NF * D4) {
                        const int cw = scode[k / D4] < Cb ? scode[k / D4] : 0;
                        w[j] = __ldg(book + (size_t)cw * D4 + k % D4);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k = k0 + j * RQ_CONS;
                    if (k < NF * D4) {
                        float4 x = reinterpret_cast<float4*>(res)[k];
                        x.x -= w[j].x;
                        x.y -= w[j].y;
                        x.z -= w[j].z;
                        x.w -= w[j].w;
                        reinterpret_cast<float4*>(res)[k] = x;
                    }
                }
            }
            asm volatile("bar.sync 2, %0;" ::"n"(RQ_CONS) : "memory");
        }
    }
    // a wait that gave up (here or in another CTA) leaves this group's frames with code -1
    if (rk == 0 && *(volatile int*)flag)
        for (int k = tid; k < nf * 8; k += RQ_CONS) codes[(size_t)t0 * 8 + k] = -1;
    fence_before();
    asm volatile("bar.arrive 1, %0;" ::"n"(RQ_CONS + 32) : "memory");
}

int fail(int code, const char* msg)
{
    mfs::set_thread_error(msg);
    return code;
}

}  // namespace

namespace mfs {

// The tensor-core path of mfs_rvq_encode (D a multiple of 8); returns MFS_OK or
// an error after setting the thread's message.  Scratch (the split codebooks
// and their norms, 4 Cb D + 4 Cb bytes per codebook, an error flag and the pairs'
// exchange words) comes from the stream-ordered pool and is released on the
// stream.  With the CTA pairs (D <= 512) the frames go in launches of at most the
// co-resident grid (a cooperative launch: a CTA waits for its partner's words).
int rvq_encode_mma(const float* z_sem, const float* z_ac, int T, int D, const float* codebooks, int Cb, int32_t* codes,
                   cudaStream_t st)
{
    const size_t cap = 227 * 1024;
    int nst2 = RQ_MAXST, nst1 = RQ_MAXST;
    while (nst2 > 2 && rq_smem_of(32, D, nst2) > cap) --nst2;
    while (nst1 > 2 && rq_smem_of(16, D, nst1) > cap) --nst1;
    const bool pairs = rq_smem_of(32, D, nst2) <= cap;
    const int nst = pairs ? nst2 : nst1;
    const size_t smem = pairs ? rq_smem_of(32, D, nst2) : rq_smem_of(16, D, nst1);
    if (smem > cap) return fail(MFS_E_ARG, "rvq: dimension too large for the tensor-core path");
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess || !fn)
            return fail(MFS_E_CUDA, "rvq: cuTensorMapEncodeTiled is not available");
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    void* kfn = pairs ? (void*)rq_kernel<32, 2> : (void*)rq_kernel<16, 1>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(MFS_E_CUDA, "rvq: cannot raise the shared memory limit");
    // frame groups per launch: with pairs, every CTA of a launch must be resident at once
    long long groups_per_launch = (T + 15) / 16;
    if (pairs) {
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, RQ_THREADS, smem) != cudaSuccess || per_sm < 1)
            return fail(MFS_E_CUDA, "rvq: cannot size the co-resident grid");
        groups_per_launch = (long long)sms * per_sm / 2;
        if (groups_per_launch < 1) return fail(MFS_E_CUDA, "rvq: a CTA pair does not fit on the device");
    }
    const int NF = pairs ? 32 : 16;
    const long long xwords = pairs ? groups_per_launch * 2 * NF * 2 : 0;
    const long long n = 8LL * Cb * D;
    char* scratch = nullptr;
    const size_t xoff = ((size_t)n * 2 * 2 + (size_t)8 * Cb * 4 + 16 + 255) & ~(size_t)255;
    const size_t bytes = xoff + (size_t)xwords * sizeof(uint2) + 256;
    e = cudaMallocAsync((void**)&scratch, bytes, st);
    if (e != cudaSuccess) return fail(MFS_E_CUDA, "rvq: scratch allocation failed");
    __nv_bfloat16* hi = (__nv_bfloat16*)scratch;
    __nv_bfloat16* lo = hi + n;
    float* norm = (float*)(lo + n);
    int* flag = (int*)(norm + (size_t)8 * Cb);
    uint2* xb = (uint2*)(scratch + xoff);
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
    if (rc == MFS_OK && e == cudaSuccess && xwords) e = cudaMemsetAsync(xb, 0, (size_t)xwords * sizeof(uint2), st);
    if (rc == MFS_OK && e == cudaSuccess) {
        rq_split<<<304, 256, 0, st>>>(codebooks, n, D, hi, lo, norm);
        e = cudaGetLastError();
    }
    // launches of up to groups_per_launch frame groups; exchange tags 8 c + 1 .. 8 c + 8
    unsigned c = 0;
    for (long long g0 = 0; rc == MFS_OK && e == cudaSuccess && g0 * NF < T; g0 += groups_per_launch, ++c) {
        const long long f0 = g0 * NF;
        int Tc = (int)(T - f0 < groups_per_launch * NF ? T - f0 : groups_per_launch * NF);
        const float* zs = z_sem + (size_t)f0 * D;
        const float* za = z_ac + (size_t)f0 * D;
        int32_t* cc = codes + (size_t)f0 * 8;
        const unsigned tag0 = 8u * c + 1u;
        const int grid = pairs ? 2 * ((Tc + NF - 1) / NF) : (Tc + NF - 1) / NF;
        int Cbv = Cb, Dv = D, nstv = nst;
        void* args[] = {(void*)&mhi, (void*)&mlo, (void*)&zs, (void*)&za, (void*)&Tc, (void*)&Dv, (void*)&codebooks,
                        (void*)&norm, (void*)&Cbv, (void*)&nstv, (void*)&cc, (void*)&flag, (void*)&xb, (void*)&tag0};
        e = pairs ? cudaLaunchCooperativeKernel(kfn, dim3(grid), dim3(RQ_THREADS), args, smem, st)
                  : cudaLaunchKernel(kfn, dim3(grid), dim3(RQ_THREADS), args, smem, st);
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
