// Internal layout shared by the host side of the library and its kernels.
#pragma once
#include <stdint.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mfs.h"

namespace mfs {

constexpr int NT = 256;          // consumer threads per CTA (8 warps); one more warp produces
constexpr int NWARP = NT / 32;
// One weight ring stage.  Large stages amortise the consumers' per-stage cost
// (barrier, copy to registers, row reductions); four of them keep 192 KB of
// weights in flight per SM.
constexpr int STAGE_BYTES = 49152;
constexpr int RPS_MAX = 16;      // rows per stage at most
// Ring depth per batch group: the per-row partial sums grow with the group, the ring shrinks.
__host__ __device__ constexpr unsigned nstage_for(int bg) { return bg <= 2 ? 4u : 3u; }
constexpr int SMEM_HEAD = 1024;  // mbarriers and scalars before the ring

// Matrix-vector K-slicing, shared by the kernels and the host's config check:
// nwk warps split K (the largest power of two <= NWARP that leaves >= 32
// vectors of 8 weights per slice), NWARP / nwk warps split the rows of a stage.
__host__ __device__ inline int slice_warps(int K)
{
    int nwk = NWARP;
    while (nwk > 1 && (K / 8) / nwk < 32) nwk >>= 1;
    return nwk;
}
// vectors per lane, rounded up to an instantiated width (1, 2 or 6)
__host__ __device__ constexpr int vpl_class_of(int vpl) { return vpl <= 1 ? 1 : (vpl == 2 ? 2 : 6); }
// rows of one stage a warp holds in registers at most, per width
__host__ __device__ constexpr int rows_per_warp_cap(int vplc) { return vplc <= 2 ? 8 : 2; }
constexpr int NSTREAM = MFS_N_STREAMS;
constexpr int NCHUNK_MAX = 32;   // attention split over the window, per (slot, head)
constexpr int HIST = 3;          // frames of token history per stream
constexpr int MAXGW = 8;         // depformer substeps run together as one group, at most

// Tensor-core weight pass (batches of 5..32 rows, bf16 weights): a matrix is
// cut into tiles of MMA_M rows and K-chunks of MMA_KC columns; one stage holds
// a weight tile chunk (TMA, 128-byte swizzle) and the rows' activations split
// into three bf16 parts (up to 96 operand rows).
constexpr int BG_MMA = 32;                            // instantiation marker: up to 32 rows per weight pass
__host__ __device__ constexpr bool is_mma(int bg) { return bg >= 8; }
constexpr int MMA_M = 128;
constexpr int MMA_KC = 64;
constexpr int MMA_PARTS = 3;                          // bf16 parts of an activation (about 27 significant bits)
constexpr int MMA_W_BYTES = MMA_M * MMA_KC * 2;       // 16 KB
constexpr int MMA_B_BYTES = MMA_PARTS * 32 * MMA_KC * 2;  // 12 KB
constexpr int MMA_STAGE = MMA_W_BYTES + MMA_B_BYTES;  // 28 KB
constexpr int MMA_NSTAGE = 7;
constexpr int MMA_HEAD = 3072;                        // barriers and scalars before the stages
constexpr int MMA_TMEM_COLS = 512;
constexpr int MMA_MAX_TILES = 5;                      // tile sums a CTA keeps (tiles it touches in one phase)
constexpr int MMA_URING = 3;                          // tensor-memory slots of per-unit products (a ring)
constexpr int MMA_THREADS = 32 * (8 + 2);             // 8 consumer warps, the producer warp, the MMA warp
constexpr int MMA_ROT = 4;                            // phases a panel / partial buffer serves before its reuse
constexpr int MAX_PCHUNKS = 192;                      // K-chunks of a matrix input at most (K <= 12288)
// rows padded to 16 or 32 (three operand rows each: N = 48 or 96)
__host__ __device__ constexpr int mma_nbp(int n) { return n <= 16 ? 16 : 32; }

// Weight matrices that have a tensor map (index into Params.tmaps): per
// temporal layer QKV, O, GU, DOWN; the text head (+ depformer in-projections);
// per depformer substep and layer DQKV, DO, DGU, DDOWN, then the substep's head.
__host__ __device__ inline int tmap_index(int type, int l, int j, int L, int dL)
{
    // PhaseType values are below; kept as ints so the host can use this too
    switch (type) {
        case 1: return 4 * l + 0;   // PH_QKV
        case 3: return 4 * l + 1;   // PH_O
        case 4: return 4 * l + 2;   // PH_GU
        case 5: return 4 * l + 3;   // PH_DOWN
        case 6: return 4 * L;       // PH_HEAD
        case 7: return 4 * L + 1 + j * (4 * dL + 1) + 4 * l + 0;  // PH_DQKV
        case 9: return 4 * L + 1 + j * (4 * dL + 1) + 4 * l + 1;  // PH_DO
        case 10: return 4 * L + 1 + j * (4 * dL + 1) + 4 * l + 2; // PH_DGU
        case 11: return 4 * L + 1 + j * (4 * dL + 1) + 4 * l + 3; // PH_DDOWN
        case 12: return 4 * L + 1 + j * (4 * dL + 1) + 4 * dL;    // PH_DHEAD
        default: return -1;
    }
}

enum PhaseType : int {
    PH_EMBED = 0,  // S0 + S1: record frame p's tokens, delayed embedding sum
    PH_QKV,        // S2: RMSNorm + QKV + RoPE + ring write
    PH_ATTN,       // S5: split flash-decode over the ring window + merge
    PH_O,          // S6: out projection + residual
    PH_GU,         // S7: RMSNorm + gate/up + SwiGLU
    PH_DOWN,       // S8: down projection + residual
    PH_HEAD,       // S4: final norm + text logits (+ argmax partials) + depformer in-projections
    PH_DQKV,       // S9: depformer layer QKV (layer 0 also forms u = in-proj + embedding)
    PH_DATTN,      // S9: depformer attention over substeps 0..j
    PH_DO,
    PH_DGU,
    PH_DDOWN,
    PH_DHEAD,      // S9: depformer head + argmax partials
    PH_FINAL,      // S10: last argmax, history write-back, outputs
};

// One phase of the step.  in_ph / res_ph / am_ph: index of the phase that
// writes this phase's input vector / residual / argmax partials (-1: none);
// the consumer waits for that phase's tag.
struct Phase {
    int type, l, j, in_ph, res_ph, am_ph, pad0, pad1;
};

// Written by the host before each launch.  A row is one frame of one slot.  In
// a normal step every row is a different slot.  In a prompt chunk
// (prompt_rows = 1, temporal phases only, every token supplied) a slot may have
// several rows, consecutive and in frame order, all at positions below the
// window (no ring row a later row writes is still in an earlier row's window).
struct StepDesc {
    int n, seq;
    int sampled;      // 1: generated tokens of slots with sampling on are drawn with P.unif
    int prompt_rows;  // 1: rows may share a slot (prompt chunk)
    int slot[MFS_MAX_SLOTS];
    int pos[MFS_MAX_SLOTS];
    int codes[MFS_MAX_SLOTS][NSTREAM];
};
constexpr int PROMPT_ROWS = 32;  // rows of a prompt chunk at most (one tensor-core pass)
// Batched steps of at most this many rows run the depformer on the CUDA-core
// instantiation (second launch); larger ones keep it on the tensor-core pass.
constexpr int DEP_GEMV_MAX_ROWS = 8;

enum DeviceError : int { DERR_NONE = 0, DERR_TOKEN = 1, DERR_WAIT = 2 };

// Per-slot sampling: temperature as its inverse, top-k (k <= 1 or inv_t <= 0: greedy).
struct SampleCfg {
    float text_inv_t;
    int text_k;
    float audio_inv_t;
    int audio_k;
};

struct Params {
    // shape
    int d, L, H, hd, F, V, C, W, dd, dL, dH, dhd, dF, S;
    int Wa;                     // keys a step attends to at most: W, or W - 1 with the oldest ring slot masked
    int delays[NSTREAM];
    float eps;
    int G;  // CTAs in the grid
    // weights (element pointers into the arena; "W" = weight dtype)
    const void* emb_text;       // [V+1][d]
    const void* emb_audio;      // [16][C+1][d]
    const void* dep_emb_text;   // [V][dd]
    const void* dep_emb_audio;  // [S-1][C][dd]
    const void* tw;             // per layer: wqkv [3d][d] | wo [d][d] | wgu [2F][d] (gate/up rows interleaved) | wdown [d][F]
    long long t_layer;          // elements per temporal layer block
    const void* head;           // text head [V][d] then depformer in-proj [S*dd][d]
    const void* dw;             // per substep j: per layer l': dqkv | dwo | dgu (interleaved) | ddown; then head [C][dd]
    long long d_layer, d_sub;   // elements per depformer layer block / per substep block
    const float* attn_norm;     // [L][d]
    const float* ffn_norm;      // [L][d]
    const float* out_norm;      // [d]
    const float* dep_attn_norm; // [dL][dd]
    const float* dep_ffn_norm;  // [dL][dd]
    const float* dep_out_norm;  // [dd]
    const float2* rope;         // [max_pos][hd/2] (cos, sin)
    // per-slot state
    void* kc;                   // [MS][L][H][W][hd] keys (kv dtype), head-major: a head's window is contiguous
    void* vc;                   // [MS][L][H][W][hd] values
    int* hist;                  // [MS][17][3]
    const StepDesc* desc;
    // activations, row = position in the step's row list (MS here: max(max_slots,
    // PROMPT_ROWS) rows).  Elements that cross CTAs are tagged 64-bit words {float bits, tag}.
    uint2* xtok;     // [MS][17] embedding rows of a prompt chunk, resolved by CTA 0 (tagged)
    uint2* x;        // [MS][d]  residual stream
    uint2* q;        // [MS][d]  rotated queries
    uint2* kcur;     // [MS][d]  this step's rotated keys (rounded to the ring's type)
    uint2* vcur;     // [MS][d]  this step's values (rounded to the ring's type)
    uint2* o;        // [MS][d]  attention output
    uint2* attp;     // [MS][H][NCHUNK_MAX][hd + 2] per-chunk attention partials: max, sum, outputs
    uint2* s;        // [MS][F]  SwiGLU output
    float* logits;   // [MS][V]  (diagnostics)
    uint2* yin;      // [MS][S][dd]  depformer in-projections
    uint2* u;        // [MS][S][dd] depformer residual stream, per substep
    uint2* dq;       // [MS][S][dd]
    uint2* dkv;      // [MS][dL][S][2][dd]
    uint2* dat;      // [MS][S][dd] depformer attention output
    uint2* ds;       // [MS][S][dF]
    float* dlogits;  // [MS][S][C]  (diagnostics)
    uint2* amax;     // [MS][G][2] text head argmax partials per CTA: {value, tag}, {index, tag}
    uint2* damax;    // [MS][S][G][2] depformer head argmax partials per substep and CTA
    const SampleCfg* samp;  // [max_slots] by slot
    const float* unif;      // [MS][17] this step's uniforms in [0, 1), by row (sampled steps)
    int* drawn;             // [MS][17] tokens drawn this step (CTA 0), by row
    int* text_out;   // [MS]
    int* codes_out;  // [MS][16]
    int* text_argmax;  // [MS]
    int* code_argmax;  // [MS][16]
    int skip_settled;  // skip trailing depformer substeps whose outputs are all settled
    int dep_ph0;       // index of the first depformer phase
    int dep_ph_stride; // phases per depformer group (dL x 5 + head)
    // control
    int* err;        // sticky device error (DeviceError)
    int* err_seq;    // step sequence number that raised it
    const Phase* phases;
    unsigned long long* ptime;  // optional: CTA 0 timer stamps and stage-wait sums, [nphase + 1][8]
    // tensor-core path
    const CUtensorMap* tmaps;   // per weight matrix (tmap_index), bf16 [rows][K], box 64 x 128, 128-byte swizzle
    unsigned* done;             // [nphase][G] tag of a depformer head phase each CTA finished
    // the next four buffers rotate over MMA_ROT phases (phase index mod MMA_ROT)
    uint2* mpart;               // [MMA_ROT][G][MMA_M][32] partial tile sums a CTA leaves for a tile's owner (tagged)
    char* panel;                // [MMA_ROT][MAXGW][pchunks][MMA_B_BYTES] activation chunks in the operand layout (by substep)
    uint2* pssq;                // [MMA_ROT][MAXGW][pchunks][32] sums of squares of a chunk's inputs per row (tagged)
    unsigned* pflag;            // [MMA_ROT][MAXGW][pchunks] tag of the phase whose chunk is written
    int pchunks;                // K-chunks of the widest matrix input
};

// Kernel entry points, one per (weight dtype, batch group).  Defined in the
// per-instantiation translation units.
const void* kernel_f32(int bg);
const void* kernel_bf16(int bg);
const void* kernel_bf16_mma();

}  // namespace mfs
