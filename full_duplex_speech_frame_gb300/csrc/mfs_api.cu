// Host side of the C ABI declared in include/mfs.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <map>
#include <new>
#include <cstddef>
#include <string>
#include <vector>

#include "mfs_internal.h"

using namespace mfs;

namespace {

constexpr int PREF_CHUNK = 256;       // prompt frames staged per copy
constexpr int DESC_RING = 8;          // pinned step descriptors in flight

struct CopyOp {
    size_t dst_off;    // bytes from the region base
    size_t src_off;    // bytes from the caller's pointer
    size_t width;      // bytes per row
    size_t rows;       // rows (1 = plain copy)
    size_t dst_pitch;  // bytes between destination rows
    size_t src_pitch;
};

struct TensorInfo {
    int region;        // 0 = weight arena, 1 = gain arena
    size_t bytes;
    std::vector<CopyOp> ops;
    bool loaded = false;
};

struct Pending {
    int seq;
    std::vector<int> slots;
    std::vector<int> old_pos;
};

}  // namespace

struct mfs_ctx {
    mfs_config cfg;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    int device = 0, G = 0;
    size_t wb = 2, kvb = 2;
    // device memory
    char* arena = nullptr;
    size_t arena_bytes = 0;
    float* gains = nullptr;
    size_t gain_bytes = 0;
    void* kc = nullptr;
    void* vc = nullptr;
    int* hist = nullptr;
    char* act = nullptr;
    float2* rope = nullptr;
    Phase* d_phases = nullptr;
    StepDesc* d_desc = nullptr;
    StepDesc* d_pref = nullptr;
    int* d_err = nullptr;
    // pinned host memory
    StepDesc* h_desc = nullptr;  // DESC_RING entries
    cudaEvent_t desc_ev[DESC_RING] = {};
    int desc_next = 0;
    StepDesc* h_pref = nullptr;
    int* h_out = nullptr;        // text [MS] | codes [MS*16] | err | err_seq
    float* h_unif = nullptr;     // pinned staging of a sampled step's uniforms [MS][17]
    // state
    Params P;
    int nphase = 0, nphase_prefill = 0;
    int maxrows = 0;
    // kernels: batch groups of 1, 2, 4 slots (CUDA cores), then the tensor-core pass (bf16 weights only)
    size_t smem[4] = {0, 0, 0, 0};
    const void* kfn[4] = {nullptr, nullptr, nullptr, nullptr};
    int threads[4] = {0, 0, 0, 0};
    CUtensorMap* d_tmaps = nullptr;
    int ntmaps = 0;
    char* mma_buf = nullptr;      // tensor-core pass: partial tile sums, activation panel
    std::vector<int> pos;
    std::map<std::string, TensorInfo> tensors;
    int mode = 0;
    int launches = 0;
    unsigned seq = 0;            // step sequence number (tags use its low 22 bits)
    size_t tag_off = 0, tag_bytes = 0;  // the tagged region of the activation arena
    size_t mma_bytes = 0;        // the tensor-core pass's tagged buffers
    int last_n = 0;
    bool last_full = false;
    std::vector<Pending> pending;
    std::string err;
    // kernel timing
    bool timing = false;
    bool stamps = false;
    unsigned long long* d_ptime = nullptr;
    int last_nph = 0;
    std::vector<cudaEvent_t> ev_pool;
    size_t ev_used = 0;
};

static int fail(mfs_ctx* c, int code, const char* fmt, ...)
{
    if (c) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        c->err = buf;
    }
    return code;
}

#define CK(call)                                                                                 \
    do {                                                                                         \
        cudaError_t e_ = (call);                                                                 \
        if (e_ != cudaSuccess) return fail(c, MFS_E_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

namespace mfs {
const void* kernel_f32_1();
const void* kernel_f32_2();
const void* kernel_f32_4();
const void* kernel_bf16_1();
const void* kernel_bf16_2();
const void* kernel_bf16_4();
const void* kernel_f32(int bg) { return bg == 1 ? kernel_f32_1() : bg == 2 ? kernel_f32_2() : kernel_f32_4(); }
const void* kernel_bf16(int bg) { return bg == 1 ? kernel_bf16_1() : bg == 2 ? kernel_bf16_2() : kernel_bf16_4(); }
}  // namespace mfs

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Kernel for a step of n rows: matrix-vector passes over groups of 1, 2 or 4
// rows, or (bf16 weights, 5 <= n <= 32) one tensor-core pass for all of them
// (the pass holds at most 32 rows: 64 operand rows of high and low halves).
static int kernel_index(const mfs_ctx* c, int n)
{
    if (n >= 5 && n <= 32 && c->kfn[3]) return 3;
    return n <= 1 ? 0 : (n == 2 ? 1 : 2);
}
static int bg_value(int idx) { return idx == 0 ? 1 : (idx == 1 ? 2 : 4); }

// ------------------------------------------------------------------ create

static int check_config(mfs_ctx* c, const mfs_config& g)
{
    if (g.d <= 0 || g.n_layers <= 0 || g.n_heads <= 0 || g.ffn <= 0 || g.text_vocab <= 0 || g.card <= 0 ||
        g.window <= 0 || g.max_pos <= 0 || g.dep_d <= 0 || g.dep_layers <= 0 || g.dep_heads <= 0 ||
        g.dep_ffn <= 0)
        return fail(c, MFS_E_ARG, "config: non-positive dimension");
    if (g.n_q != 16 || g.dep_steps != 16) return fail(c, MFS_E_ARG, "config: n_q and dep_steps must be 16");
    if (g.head_dim != 64 && g.head_dim != 128) return fail(c, MFS_E_ARG, "config: head_dim must be 64 or 128");
    if (g.n_heads * g.head_dim != g.d) return fail(c, MFS_E_ARG, "config: n_heads * head_dim != d");
    if (g.dep_head_dim != 64 || g.dep_heads * g.dep_head_dim != g.dep_d)
        return fail(c, MFS_E_ARG, "config: dep_head_dim must be 64 and dep_heads * 64 == dep_d");
    const int Ks[4] = {g.d, g.ffn, g.dep_d, g.dep_ffn};
    const int wbytes = g.weight_dtype == MFS_DTYPE_BF16 ? 2 : 4;
    for (int K : Ks) {
        if (K % 8 != 0 || K > 12288 || K * wbytes > STAGE_BYTES)
            return fail(c, MFS_E_ARG, "config: K dimension %d not a multiple of 8, or a row exceeds %d bytes", K, STAGE_BYTES);
        // every row of a stage must fit the registers of the warp that takes it
        const int nwk = slice_warps(K), nwr = NWARP / nwk;
        const int nvw = (K / 8 + nwk - 1) / nwk, vpl = (nvw + 31) / 32;
        int rps = STAGE_BYTES / (K * wbytes);
        rps = rps < RPS_MAX ? rps : RPS_MAX;
        if ((rps + nwr - 1) / nwr > rows_per_warp_cap(vpl_class_of(vpl)))
            return fail(c, MFS_E_ARG, "config: K dimension %d gives %d rows per warp and stage (at most %d)", K,
                        (rps + nwr - 1) / nwr, rows_per_warp_cap(vpl_class_of(vpl)));
    }
    if (g.text_vocab % 2 || g.card % 2) return fail(c, MFS_E_ARG, "config: vocabularies must be even");
    if (g.max_slots < 1 || g.max_slots > MFS_MAX_SLOTS) return fail(c, MFS_E_ARG, "config: max_slots out of range");
    if (g.weight_dtype != MFS_DTYPE_F32 && g.weight_dtype != MFS_DTYPE_BF16) return fail(c, MFS_E_ARG, "config: weight_dtype");
    if (g.kv_dtype != g.weight_dtype) return fail(c, MFS_E_ARG, "config: kv_dtype must equal weight_dtype");
    for (int k = 0; k < NSTREAM; ++k)
        if (g.delays[k] < 0 || g.delays[k] > 1) return fail(c, MFS_E_ARG, "config: delays must be 0 or 1");
    if (g.eps <= 0 || g.rope_theta <= 0) return fail(c, MFS_E_ARG, "config: eps and rope_theta must be positive");
    return MFS_OK;
}

static void add_tensor(mfs_ctx* c, const std::string& name, int region, size_t bytes, std::vector<CopyOp> ops)
{
    TensorInfo t;
    t.region = region;
    t.bytes = bytes;
    t.ops = std::move(ops);
    c->tensors[name] = t;
}

static CopyOp plain(size_t dst, size_t src, size_t bytes) { return CopyOp{dst, src, bytes, 1, bytes, bytes}; }

// Gate rows go to even destination rows, up rows to odd ones.
static void interleave(std::vector<CopyOp>& ops, size_t dst, size_t src, size_t rows_half, size_t row_bytes)
{
    ops.push_back(CopyOp{dst, src, row_bytes, rows_half, 2 * row_bytes, row_bytes});
    ops.push_back(CopyOp{dst + row_bytes, src + rows_half * row_bytes, row_bytes, rows_half, 2 * row_bytes, row_bytes});
}

static int build_layout(mfs_ctx* c)
{
    const mfs_config& g = c->cfg;
    const size_t wb = c->wb;
    const size_t d = g.d, F = g.ffn, V = g.text_vocab, C = g.card, S = g.dep_steps, L = g.n_layers;
    const size_t dd = g.dep_d, dF = g.dep_ffn, dL = g.dep_layers;
    size_t off = 0;
    auto region = [&](size_t elems) {
        size_t o = off;
        off = align_up(off + elems * wb, 256);
        return o;
    };
    const size_t o_emb_text = region((V + 1) * d);
    const size_t o_emb_audio = region(16 * (C + 1) * d);
    const size_t o_dep_emb_text = region(V * dd);
    const size_t o_dep_emb_audio = region((S - 1) * C * dd);
    const size_t t_layer = 4 * d * d + 3 * F * d;
    const size_t o_tw = region(L * t_layer);
    const size_t o_head = region((V + S * dd) * d);
    const size_t d_layer = 4 * dd * dd + 3 * dd * dF;
    const size_t d_sub = dL * d_layer + C * dd;
    const size_t o_dw = region(S * d_sub);
    c->arena_bytes = off;

    // gains (fp32)
    size_t go = 0;
    auto gregion = [&](size_t elems) {
        size_t o = go;
        go = align_up(go + elems * 4, 256);
        return o;
    };
    const size_t g_attn = gregion(L * d), g_ffn = gregion(L * d), g_out = gregion(d);
    const size_t g_dattn = gregion(dL * dd), g_dffn = gregion(dL * dd), g_dout = gregion(dd);
    c->gain_bytes = go;

    add_tensor(c, "emb.text", 0, (V + 1) * d * wb, {plain(o_emb_text, 0, (V + 1) * d * wb)});
    add_tensor(c, "emb.audio", 0, 16 * (C + 1) * d * wb, {plain(o_emb_audio, 0, 16 * (C + 1) * d * wb)});
    add_tensor(c, "dep.emb.text", 0, V * dd * wb, {plain(o_dep_emb_text, 0, V * dd * wb)});
    add_tensor(c, "dep.emb.audio", 0, (S - 1) * C * dd * wb, {plain(o_dep_emb_audio, 0, (S - 1) * C * dd * wb)});
    for (size_t l = 0; l < L; ++l) {
        const size_t base = o_tw + l * t_layer * wb;
        const std::string p = "layers." + std::to_string(l) + ".";
        add_tensor(c, p + "wqkv", 0, 3 * d * d * wb, {plain(base, 0, 3 * d * d * wb)});
        add_tensor(c, p + "wo", 0, d * d * wb, {plain(base + 3 * d * d * wb, 0, d * d * wb)});
        std::vector<CopyOp> gu;
        interleave(gu, base + 4 * d * d * wb, 0, F, d * wb);
        add_tensor(c, p + "wgu", 0, 2 * F * d * wb, gu);
        add_tensor(c, p + "wdown", 0, d * F * wb, {plain(base + (4 * d * d + 2 * F * d) * wb, 0, d * F * wb)});
        add_tensor(c, p + "attn_norm", 1, d * 4, {plain(g_attn + l * d * 4, 0, d * 4)});
        add_tensor(c, p + "ffn_norm", 1, d * 4, {plain(g_ffn + l * d * 4, 0, d * 4)});
    }
    add_tensor(c, "out_norm", 1, d * 4, {plain(g_out, 0, d * 4)});
    add_tensor(c, "text_head", 0, V * d * wb, {plain(o_head, 0, V * d * wb)});
    add_tensor(c, "dep.in", 0, S * dd * d * wb, {plain(o_head + V * d * wb, 0, S * dd * d * wb)});
    for (size_t l = 0; l < dL; ++l) {
        const std::string p = "dep.layers." + std::to_string(l) + ".";
        std::vector<CopyOp> qkv, wo, gu, down;
        for (size_t s = 0; s < S; ++s) {
            const size_t base = o_dw + (s * d_sub + l * d_layer) * wb;
            qkv.push_back(plain(base, s * 3 * dd * dd * wb, 3 * dd * dd * wb));
            wo.push_back(plain(base + 3 * dd * dd * wb, s * dd * dd * wb, dd * dd * wb));
            interleave(gu, base + 4 * dd * dd * wb, s * 2 * dF * dd * wb, dF, dd * wb);
            down.push_back(plain(base + (4 * dd * dd + 2 * dF * dd) * wb, s * dd * dF * wb, dd * dF * wb));
        }
        add_tensor(c, p + "wqkv", 0, S * 3 * dd * dd * wb, qkv);
        add_tensor(c, p + "wo", 0, S * dd * dd * wb, wo);
        add_tensor(c, p + "wgu", 0, S * 2 * dF * dd * wb, gu);
        add_tensor(c, p + "wdown", 0, S * dd * dF * wb, down);
        add_tensor(c, p + "attn_norm", 1, dd * 4, {plain(g_dattn + l * dd * 4, 0, dd * 4)});
        add_tensor(c, p + "ffn_norm", 1, dd * 4, {plain(g_dffn + l * dd * 4, 0, dd * 4)});
    }
    add_tensor(c, "dep.out_norm", 1, dd * 4, {plain(g_dout, 0, dd * 4)});
    {
        std::vector<CopyOp> hd;
        for (size_t s = 0; s < S; ++s) hd.push_back(plain(o_dw + (s * d_sub + dL * d_layer) * wb, s * C * dd * wb, C * dd * wb));
        add_tensor(c, "dep.head", 0, S * C * dd * wb, hd);
    }

    // device pointers (filled once the arenas exist)
    Params& P = c->P;
    P.emb_text = (void*)o_emb_text;
    P.emb_audio = (void*)o_emb_audio;
    P.dep_emb_text = (void*)o_dep_emb_text;
    P.dep_emb_audio = (void*)o_dep_emb_audio;
    P.tw = (void*)o_tw;
    P.t_layer = (long long)t_layer;
    P.head = (void*)o_head;
    P.dw = (void*)o_dw;
    P.d_layer = (long long)d_layer;
    P.d_sub = (long long)d_sub;
    P.attn_norm = (float*)g_attn;
    P.ffn_norm = (float*)g_ffn;
    P.out_norm = (float*)g_out;
    P.dep_attn_norm = (float*)g_dattn;
    P.dep_ffn_norm = (float*)g_dffn;
    P.dep_out_norm = (float*)g_dout;
    return MFS_OK;
}

static void rebase(const void*& p, char* base) { p = base + (size_t)p; }
static void rebasef(const float*& p, float* base) { p = (const float*)((char*)base + (size_t)p); }

static int max_rows(const mfs_config& g, int G)
{
    // temporal matrices are shared by all G CTAs; a depformer matrix by at
    // least G / MAXGW of them (a group of up to MAXGW substeps splits the grid)
    const long long tpairs[] = {3LL * g.d / 2, g.d / 2, g.ffn, g.d / 2, (g.text_vocab + 16LL * g.dep_d) / 2};
    const long long dpairs[] = {3LL * g.dep_d / 2, g.dep_d / 2, g.dep_ffn, g.dep_d / 2, g.card / 2};
    const long long Gd = G / MAXGW;
    long long m = 0;
    for (long long np : tpairs) m = (np + G - 1) / G > m ? (np + G - 1) / G : m;
    for (long long np : dpairs) m = (np + Gd - 1) / Gd > m ? (np + Gd - 1) / Gd : m;
    return (int)(2 * m);
}

static thread_local std::string g_create_error;

// Tiles of one matrix a CTA can touch in one phase, at most (cnt CTAs share it).
static int tiles_touched(long long M, long long K, long long cnt)
{
    const long long KC = (K + MMA_KC - 1) / MMA_KC, T = (M + MMA_M - 1) / MMA_M;
    const long long per = (T * KC + cnt - 1) / cnt;
    return (int)((per + KC - 1) / KC + 1);
}

// Shared memory of the tensor-core instantiation: alignment slack, barriers,
// stages, then one region for epilogue tile values, attention partials,
// embedding rows or the sampler, whichever phase runs.
static size_t mma_smem(const mfs_config& g)
{
    const size_t tile = (size_t)MMA_M * 32 * sizeof(float);
    const size_t attn_w = (size_t)NWARP * (g.head_dim + 4) * sizeof(float);
    const size_t attn_m = (size_t)NCHUNK_MAX * (g.head_dim + 2) * sizeof(float);
    const size_t emb = (size_t)MFS_MAX_SLOTS * NSTREAM * sizeof(int);
    const size_t samp = (size_t)(2048 + MFS_MAX_SLOTS * NSTREAM) * sizeof(int);
    size_t region = tile;
    for (size_t r : {attn_w, attn_m, emb, samp}) region = r > region ? r : region;
    return 1024 + (size_t)MMA_HEAD + (size_t)MMA_NSTAGE * MMA_STAGE + region;
}

// One tensor map per weight matrix (tmap_index order): bf16 [rows][K], boxes of
// 64 columns x 128 rows with the 128-byte swizzle the MMA operand layout expects.
static int setup_tensor_core_pass(mfs_ctx* c)
{
    const mfs_config& g = c->cfg;
    const long long d = g.d, F = g.ffn, dd = g.dep_d, dF = g.dep_ffn, V = g.text_vocab, C = g.card, S = g.dep_steps;
    const int L = g.n_layers, dL = g.dep_layers;
    // every matrix must leave a CTA at most MMA_MAX_TILES accumulator slots
    struct Mat { long long M, K; };
    const Mat tm[] = {{3 * d, d}, {d, d}, {2 * F, d}, {d, F}, {V + S * dd, d}};
    const Mat dm[] = {{3 * dd, dd}, {dd, dd}, {2 * dF, dd}, {dd, dF}, {C, dd}};
    for (const Mat& m : tm)
        if (tiles_touched(m.M, m.K, c->G) > MMA_MAX_TILES) return MFS_OK;  // shape unsuited: batches stay on CUDA cores
    for (const Mat& m : dm)
        if (tiles_touched(m.M, m.K, c->G / MAXGW) > MMA_MAX_TILES) return MFS_OK;
    const size_t smem = mma_smem(g);
    if (smem > 227 * 1024) return MFS_OK;

    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    if (!fn || q != cudaDriverEntryPointSuccess) return fail(c, MFS_E_CUDA, "cuTensorMapEncodeTiled is not available");
    auto encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    c->ntmaps = 4 * L + 1 + (int)S * (4 * dL + 1);
    std::vector<CUtensorMap> maps((size_t)c->ntmaps);
    auto make = [&](int idx, const void* base, long long M, long long K) -> int {
        if (((uintptr_t)base & 15u) != 0 || (K * 2) % 16 != 0) return fail(c, MFS_E_ARG, "tensor map: misaligned matrix");
        const cuuint64_t dim[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t stride[1] = {(cuuint64_t)(K * 2)};
        const cuuint32_t box[2] = {(cuuint32_t)MMA_KC, (cuuint32_t)MMA_M};
        const cuuint32_t es[2] = {1, 1};
        const CUresult r = encode(&maps[(size_t)idx], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dim,
                                  stride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(c, MFS_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return MFS_OK;
    };
    const uint16_t* tw = (const uint16_t*)c->P.tw;
    const size_t tl = (size_t)c->P.t_layer;
    int rc = MFS_OK;
    for (int l = 0; l < L && rc == MFS_OK; ++l) {
        const uint16_t* b = tw + (size_t)l * tl;
        if (!rc) rc = make(tmap_index(PH_QKV, l, 0, L, dL), b, 3 * d, d);
        if (!rc) rc = make(tmap_index(PH_O, l, 0, L, dL), b + 3 * d * d, d, d);
        if (!rc) rc = make(tmap_index(PH_GU, l, 0, L, dL), b + 4 * d * d, 2 * F, d);
        if (!rc) rc = make(tmap_index(PH_DOWN, l, 0, L, dL), b + 4 * d * d + 2 * F * d, d, F);
    }
    if (!rc) rc = make(tmap_index(PH_HEAD, 0, 0, L, dL), c->P.head, V + S * dd, d);
    const uint16_t* dw = (const uint16_t*)c->P.dw;
    for (int j = 0; j < S && rc == MFS_OK; ++j)
        for (int l = 0; l < dL && rc == MFS_OK; ++l) {
            const uint16_t* b = dw + (size_t)j * c->P.d_sub + (size_t)l * c->P.d_layer;
            if (!rc) rc = make(tmap_index(PH_DQKV, l, j, L, dL), b, 3 * dd, dd);
            if (!rc) rc = make(tmap_index(PH_DO, l, j, L, dL), b + 3 * dd * dd, dd, dd);
            if (!rc) rc = make(tmap_index(PH_DGU, l, j, L, dL), b + 4 * dd * dd, 2 * dF, dd);
            if (!rc) rc = make(tmap_index(PH_DDOWN, l, j, L, dL), b + 4 * dd * dd + 2 * dF * dd, dd, dF);
            if (!rc && l == dL - 1) rc = make(tmap_index(PH_DHEAD, 0, j, L, dL), dw + (size_t)j * c->P.d_sub + (size_t)dL * c->P.d_layer, C, dd);
        }
    if (rc != MFS_OK) return rc;
    CK(cudaMalloc((void**)&c->d_tmaps, maps.size() * sizeof(CUtensorMap)));
    CK(cudaMemcpy(c->d_tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice));
    c->P.tmaps = c->d_tmaps;
    // partial tile sums, phase completion tags, and the activation panel (chunks
    // of every matrix input in the operand layout, by phase parity and substep)
    long long kmax = d > F ? d : F;
    kmax = kmax > dd ? kmax : dd;
    kmax = kmax > dF ? kmax : dF;
    c->P.pchunks = (int)((kmax + MMA_KC - 1) / MMA_KC);
    if (c->P.pchunks > MAX_PCHUNKS) return MFS_OK;  // (K <= 12288 is checked at create)
    const size_t nch = (size_t)MMA_ROT * MAXGW * c->P.pchunks;
    const size_t part = align_up((size_t)MMA_ROT * c->G * MMA_M * 32 * sizeof(uint2), 256);
    const size_t panel = nch * MMA_B_BYTES, pssq = align_up(nch * 32 * sizeof(uint2), 256), pflag = nch * sizeof(unsigned);
    const size_t done = align_up((size_t)c->nphase * c->G * sizeof(unsigned), 256);
    const size_t total = part + panel + pssq + align_up(pflag, 256) + done;
    c->mma_bytes = total;
    CK(cudaMalloc((void**)&c->mma_buf, total));
    CK(cudaMemset(c->mma_buf, 0, total));
    c->P.mpart = (uint2*)c->mma_buf;
    c->P.panel = c->mma_buf + part;
    c->P.pssq = (uint2*)(c->mma_buf + part + panel);
    c->P.pflag = (unsigned*)(c->mma_buf + part + panel + pssq);
    c->P.done = (unsigned*)(c->mma_buf + part + panel + pssq + align_up(pflag, 256));
    c->kfn[3] = kernel_bf16_mma();
    c->threads[3] = MMA_THREADS;
    c->smem[3] = smem;
    CK(cudaFuncSetAttribute(c->kfn[3], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    int per_sm = 0;
    CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c->kfn[3], MMA_THREADS, smem));
    if (per_sm < 1) return fail(c, MFS_E_CUDA, "tensor-core kernel does not fit on an SM");
    return MFS_OK;
}

static int create_impl(mfs_ctx* c, void* cuda_stream)
{
    int rc = check_config(c, c->cfg);
    if (rc != MFS_OK) return rc;
    const mfs_config& g = c->cfg;
    c->wb = g.weight_dtype == MFS_DTYPE_BF16 ? 2 : 4;
    c->kvb = g.kv_dtype == MFS_DTYPE_BF16 ? 2 : 4;
    CK(cudaGetDevice(&c->device));
    int nsm = 0;
    CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, c->device));
    int coop = 0;
    CK(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device));
    if (!coop) return fail(c, MFS_E_CUDA, "device lacks cooperative launch");
    c->G = nsm;
    if (cuda_stream) c->stream = (cudaStream_t)cuda_stream;
    else {
        CK(cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking));
        c->own_stream = true;
    }

    build_layout(c);
    const size_t MS = g.max_slots, d = g.d, F = g.ffn, V = g.text_vocab, C = g.card, S = g.dep_steps;
    const size_t dd = g.dep_d, dF = g.dep_ffn, dL = g.dep_layers, H = g.n_heads, hd = g.head_dim;

    CK(cudaMalloc((void**)&c->arena, c->arena_bytes));
    CK(cudaMalloc((void**)&c->gains, c->gain_bytes));
    CK(cudaMemset(c->gains, 0, c->gain_bytes));
    const size_t kv = MS * g.n_layers * (size_t)g.window * d * c->kvb;
    CK(cudaMalloc(&c->kc, kv));
    CK(cudaMalloc(&c->vc, kv));
    CK(cudaMalloc((void**)&c->hist, MS * NSTREAM * HIST * sizeof(int)));
    CK(cudaMemset(c->hist, 0xFF, MS * NSTREAM * HIST * sizeof(int)));

    // activations: one row per slot of a step, or per frame of a prompt chunk
    const size_t AR = MS > (size_t)PROMPT_ROWS ? MS : (size_t)PROMPT_ROWS;
    size_t ao = 0;
    auto areg = [&](size_t bytes) {
        size_t o = ao;
        ao = align_up(ao + bytes, 256);
        return o;
    };
    const size_t T8 = sizeof(uint2);  // tagged element
    const size_t a_x = areg(AR * d * T8), a_q = areg(AR * d * T8), a_kc = areg(AR * d * T8), a_vc = areg(AR * d * T8);
    const size_t a_o = areg(AR * d * T8), a_s = areg(AR * F * T8);
    const size_t a_ap = areg(AR * H * NCHUNK_MAX * (hd + 2) * T8);
    const size_t a_xt = areg(AR * NSTREAM * T8);
    const size_t a_lg = areg(MS * V * 4), a_yin = areg(MS * S * dd * T8), a_u = areg(MS * S * dd * T8);
    const size_t a_dq = areg(MS * S * dd * T8), a_dkv = areg(MS * dL * S * 2 * dd * T8), a_dat = areg(MS * S * dd * T8);
    const size_t a_ds = areg(MS * S * dF * T8), a_dlg = areg(MS * S * C * 4);
    const size_t a_am = areg(MS * c->G * 2 * T8), a_dam = areg(MS * S * c->G * 2 * T8);
    const size_t a_to = areg(MS * 4), a_co = areg(MS * 16 * 4), a_ta = areg(MS * 4), a_ca = areg(MS * 16 * 4);
    const size_t a_sc = areg(MS * sizeof(SampleCfg)), a_un = areg(MS * NSTREAM * 4), a_dr = areg(MS * NSTREAM * 4);
    c->tag_off = a_x;  // [a_x, a_to): every tagged buffer (and the logits); a_to on are outputs and settings
    c->tag_bytes = a_to - a_x;
    CK(cudaMalloc((void**)&c->act, ao));
    CK(cudaMemset(c->act, 0, ao));

    // RoPE table: angle p * theta^(-2i/hd), in double, rounded to fp32
    {
        const size_t half = hd / 2;
        std::vector<float2> tab((size_t)g.max_pos * half);
        for (size_t p = 0; p < (size_t)g.max_pos; ++p)
            for (size_t i = 0; i < half; ++i) {
                const double a = (double)p * pow(g.rope_theta, -2.0 * (double)i / (double)hd);
                tab[p * half + i] = make_float2((float)cos(a), (float)sin(a));
            }
        CK(cudaMalloc((void**)&c->rope, tab.size() * sizeof(float2)));
        CK(cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
    }

    // phase list: embed, L x 5, head, S x (dL x 5 + 1), final; each phase names
    // the phases whose tagged outputs it consumes
    std::vector<Phase> ph;
    auto add = [&](int type, int l, int j, int in, int res, int am) {
        ph.push_back(Phase{type, l, j, in, res, am, 0, 0});
        return (int)ph.size() - 1;
    };
    int x_ph = add(PH_EMBED, 0, 0, -1, -1, -1);  // last writer of the residual stream
    for (int l = 0; l < g.n_layers; ++l) {
        const int qkv = add(PH_QKV, l, 0, x_ph, -1, -1);
        const int att = add(PH_ATTN, l, 0, qkv, -1, -1);
        const int o = add(PH_O, l, 0, att, x_ph, -1);
        const int gu = add(PH_GU, l, 0, o, -1, -1);
        x_ph = add(PH_DOWN, l, 0, gu, o, -1);
    }
    c->nphase_prefill = (int)ph.size();
    const int head = add(PH_HEAD, 0, 0, x_ph, -1, -1);
    int am_ph = head;
    c->P.dep_ph0 = (int)ph.size();
    c->P.dep_ph_stride = 5 * g.dep_layers + 1;
    for (int j = 0; j < g.dep_steps; ++j) {
        int u_ph = -1;  // last writer of the depformer residual
        for (int l = 0; l < g.dep_layers; ++l) {
            const int qkv = add(PH_DQKV, l, j, l == 0 ? head : u_ph, -1, l == 0 ? am_ph : -1);
            if (l == 0) u_ph = qkv;  // layer 0 also writes the residual (in-projection + embedding)
            const int att = add(PH_DATTN, l, j, qkv, -1, -1);
            const int o = add(PH_DO, l, j, att, u_ph, -1);
            const int gu = add(PH_DGU, l, j, o, -1, -1);
            u_ph = add(PH_DDOWN, l, j, gu, o, -1);
        }
        am_ph = add(PH_DHEAD, 0, j, u_ph, -1, -1);
    }
    add(PH_FINAL, 0, 0, -1, -1, am_ph);
    c->nphase = (int)ph.size();
    if (c->nphase >= 1024) return fail(c, MFS_E_ARG, "config: %d phases per step (at most 1023)", c->nphase);
    CK(cudaMalloc((void**)&c->d_phases, ph.size() * sizeof(Phase)));
    CK(cudaMemcpy(c->d_phases, ph.data(), ph.size() * sizeof(Phase), cudaMemcpyHostToDevice));

    CK(cudaMalloc((void**)&c->d_desc, sizeof(StepDesc)));
    CK(cudaMemset(c->d_desc, 0, sizeof(StepDesc)));
    CK(cudaMalloc((void**)&c->d_pref, PREF_CHUNK * sizeof(StepDesc)));
    CK(cudaMalloc((void**)&c->d_err, 256));
    CK(cudaMemset(c->d_err, 0, 256));
    CK(cudaHostAlloc((void**)&c->h_desc, DESC_RING * sizeof(StepDesc), cudaHostAllocDefault));
    for (int i = 0; i < DESC_RING; ++i) CK(cudaEventCreateWithFlags(&c->desc_ev[i], cudaEventDisableTiming));
    CK(cudaHostAlloc((void**)&c->h_pref, PREF_CHUNK * sizeof(StepDesc), cudaHostAllocDefault));
    CK(cudaHostAlloc((void**)&c->h_out, (MFS_MAX_SLOTS * 17 + 2) * sizeof(int), cudaHostAllocDefault));
    CK(cudaHostAlloc((void**)&c->h_unif, MFS_MAX_SLOTS * NSTREAM * sizeof(float), cudaHostAllocDefault));

    Params& P = c->P;
    P.d = g.d; P.L = g.n_layers; P.H = g.n_heads; P.hd = g.head_dim; P.F = g.ffn; P.V = g.text_vocab;
    P.C = g.card; P.W = g.window; P.dd = g.dep_d; P.dL = g.dep_layers; P.dH = g.dep_heads;
    P.Wa = g.window;
    P.dhd = g.dep_head_dim; P.dF = g.dep_ffn; P.S = g.dep_steps;
    for (int k = 0; k < NSTREAM; ++k) P.delays[k] = g.delays[k];
    P.eps = (float)g.eps;
    P.G = c->G;
    rebase(P.emb_text, c->arena); rebase(P.emb_audio, c->arena);
    rebase(P.dep_emb_text, c->arena); rebase(P.dep_emb_audio, c->arena);
    rebase(P.tw, c->arena); rebase(P.head, c->arena); rebase(P.dw, c->arena);
    rebasef(P.attn_norm, c->gains); rebasef(P.ffn_norm, c->gains); rebasef(P.out_norm, c->gains);
    rebasef(P.dep_attn_norm, c->gains); rebasef(P.dep_ffn_norm, c->gains); rebasef(P.dep_out_norm, c->gains);
    P.rope = c->rope;
    P.kc = c->kc; P.vc = c->vc; P.hist = c->hist; P.desc = c->d_desc;
    char* A = c->act;
    P.x = (uint2*)(A + a_x); P.q = (uint2*)(A + a_q); P.kcur = (uint2*)(A + a_kc); P.vcur = (uint2*)(A + a_vc);
    P.o = (uint2*)(A + a_o); P.s = (uint2*)(A + a_s); P.attp = (uint2*)(A + a_ap); P.xtok = (uint2*)(A + a_xt);
    P.logits = (float*)(A + a_lg); P.yin = (uint2*)(A + a_yin); P.u = (uint2*)(A + a_u);
    P.dq = (uint2*)(A + a_dq); P.dkv = (uint2*)(A + a_dkv); P.dat = (uint2*)(A + a_dat);
    P.ds = (uint2*)(A + a_ds); P.dlogits = (float*)(A + a_dlg); P.amax = (uint2*)(A + a_am);
    P.damax = (uint2*)(A + a_dam); P.text_out = (int*)(A + a_to); P.codes_out = (int*)(A + a_co);
    P.text_argmax = (int*)(A + a_ta); P.code_argmax = (int*)(A + a_ca);
    P.samp = (const SampleCfg*)(A + a_sc); P.unif = (const float*)(A + a_un); P.drawn = (int*)(A + a_dr);
    P.err = c->d_err; P.err_seq = c->d_err + 1;
    P.phases = c->d_phases;

    // kernels: one per batch group; shared memory for the largest row block
    c->maxrows = max_rows(g, c->G);
    for (int i = 0; i < 4; ++i) c->threads[i] = NT + 32;
    if (g.weight_dtype == MFS_DTYPE_BF16) {
        int rc2 = setup_tensor_core_pass(c);
        if (rc2 != MFS_OK) return rc2;
    }
    for (int i = 0; i < 3; ++i) {
        const int bg = bg_value(i);
        c->kfn[i] = g.weight_dtype == MFS_DTYPE_BF16 ? kernel_bf16(bg) : kernel_f32(bg);
        // ring, then one region used as GEMV partials + row values, attention
        // partials, or the step's embedding rows, whichever phase runs
        const size_t gemv = (size_t)c->maxrows * bg * (NWARP + 1) * sizeof(float);
        const size_t attn_w = (size_t)NWARP * (g.head_dim + 4) * sizeof(float);
        const size_t attn_m = (size_t)NCHUNK_MAX * (g.head_dim + 2) * sizeof(float);  // chunk merge
        const size_t attn = attn_w > attn_m ? attn_w : attn_m;
        const size_t emb = (size_t)MFS_MAX_SLOTS * NSTREAM * sizeof(int);
        const size_t samp = (size_t)(2048 + MFS_MAX_SLOTS * NSTREAM) * sizeof(int);  // sampler histogram + final argmaxes
        size_t region = gemv > attn ? gemv : attn;
        region = region > emb ? region : emb;
        region = region > samp ? region : samp;
        c->smem[i] = SMEM_HEAD + (size_t)nstage_for(bg) * STAGE_BYTES + region;
        if (c->smem[i] > 227 * 1024) return fail(c, MFS_E_ARG, "shape needs %zu B of shared memory", c->smem[i]);
        CK(cudaFuncSetAttribute(c->kfn[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c->smem[i]));
        int per_sm = 0;
        CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c->kfn[i], NT + 32, c->smem[i]));
        if (per_sm < 1) return fail(c, MFS_E_CUDA, "kernel does not fit on an SM");
    }
    c->pos.assign(MS, 0);
    return MFS_OK;
}

extern "C" int mfs_create(const mfs_config* cfg, void* cuda_stream, mfs_ctx** out)
{
    if (!out) return MFS_E_ARG;
    *out = nullptr;
    if (!cfg) {
        g_create_error = "null config";
        return MFS_E_ARG;
    }
    mfs_ctx* c = new (std::nothrow) mfs_ctx();
    if (!c) {
        g_create_error = "out of host memory";
        return MFS_E_NOMEM;
    }
    c->cfg = *cfg;
    const int rc = create_impl(c, cuda_stream);
    if (rc != MFS_OK) {
        g_create_error = c->err;
        mfs_destroy(c);
        return rc;
    }
    *out = c;
    return MFS_OK;
}

extern "C" void mfs_destroy(mfs_ctx* c)
{
    if (!c) return;
    if (c->stream) cudaStreamSynchronize(c->stream);
    cudaFree(c->arena); cudaFree(c->gains); cudaFree(c->kc); cudaFree(c->vc); cudaFree(c->hist);
    cudaFree(c->act); cudaFree(c->rope); cudaFree(c->d_phases); cudaFree(c->d_desc); cudaFree(c->d_pref);
    cudaFree(c->d_err);
    cudaFree(c->d_ptime);
    cudaFree(c->d_tmaps);
    cudaFree(c->mma_buf);
    for (int i = 0; i < DESC_RING; ++i)
        if (c->desc_ev[i]) cudaEventDestroy(c->desc_ev[i]);
    for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
    cudaFreeHost(c->h_desc); cudaFreeHost(c->h_pref); cudaFreeHost(c->h_out); cudaFreeHost(c->h_unif);
    if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
    delete c;
}

namespace mfs {
// Message for mfs_last_error(NULL) from an entry point that takes no context.
void set_thread_error(const char* msg) { g_create_error = msg ? msg : ""; }
}  // namespace mfs

extern "C" const char* mfs_last_error(const mfs_ctx* c)
{
    if (!c) return g_create_error.c_str();
    return c->err.c_str();
}

// ------------------------------------------------------------------ weights

extern "C" int mfs_load_weights(mfs_ctx* c, const char* name, const void* src, size_t bytes, int on_device)
{
    if (!c || !name || !src) return fail(c, MFS_E_ARG, "null argument");
    if (!c->arena) return fail(c, MFS_E_STATE, "context not created");
    auto it = c->tensors.find(name);
    if (it == c->tensors.end()) return fail(c, MFS_E_STATE, "unknown tensor %s", name);
    TensorInfo& t = it->second;
    if (bytes != t.bytes) return fail(c, MFS_E_STATE, "%s: %zu bytes, expected %zu", name, bytes, t.bytes);
    CK(cudaStreamSynchronize(c->stream));
    char* base = t.region == 0 ? c->arena : (char*)c->gains;
    const cudaMemcpyKind kind = on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    for (const CopyOp& op : t.ops) {
        if (op.rows == 1) CK(cudaMemcpy(base + op.dst_off, (const char*)src + op.src_off, op.width, kind));
        else CK(cudaMemcpy2D(base + op.dst_off, op.dst_pitch, (const char*)src + op.src_off, op.src_pitch, op.width, op.rows, kind));
    }
    t.loaded = true;
    return MFS_OK;
}

static int weights_ready(mfs_ctx* c)
{
    for (auto& kv : c->tensors)
        if (!kv.second.loaded) return fail(c, MFS_E_STATE, "tensor %s not loaded", kv.first.c_str());
    return MFS_OK;
}

// ------------------------------------------------------------------ steps

static int check_slots(mfs_ctx* c, int n, const int32_t* slots, int advance)
{
    if (n < 1 || n > c->cfg.max_slots) return fail(c, MFS_E_ARG, "n = %d outside [1, %d]", n, c->cfg.max_slots);
    if (!slots) return fail(c, MFS_E_ARG, "null slots");
    std::vector<char> seen(c->cfg.max_slots, 0);
    for (int i = 0; i < n; ++i) {
        const int s = slots[i];
        if (s < 0 || s >= c->cfg.max_slots) return fail(c, MFS_E_SLOT, "slot %d outside [0, %d)", s, c->cfg.max_slots);
        if (seen[s]) return fail(c, MFS_E_ARG, "slot %d listed twice", s);
        seen[s] = 1;
        if (c->pos[s] + advance > c->cfg.max_pos)
            return fail(c, MFS_E_RANGE, "slot %d at frame %d would pass max_pos %d", s, c->pos[s], c->cfg.max_pos);
    }
    return MFS_OK;
}

static int check_tokens(mfs_ctx* c, const int32_t* codes, int rows, int lo)
{
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < NSTREAM; ++k) {
            const int t = codes[(size_t)r * NSTREAM + k];
            const int hi = k == 0 ? c->cfg.text_vocab : c->cfg.card;
            if (t < lo || t >= hi) return fail(c, MFS_E_TOKEN, "token %d of stream %d outside [%d, %d)", t, k, lo, hi);
        }
    return MFS_OK;
}

// Enqueue the kernel(s) for phases [0, nph) of the step described by desc.
static int launch(mfs_ctx* c, int n, int nph, const StepDesc* desc)
{
    Params P = c->P;
    P.desc = desc;
    P.ptime = c->stamps ? c->d_ptime : nullptr;
    c->last_nph = nph;
    const int bi = kernel_index(c, n);
    int maxrows = c->maxrows;
    cudaEvent_t ev1 = nullptr;
    if (c->timing) {
        if (c->ev_used + 2 > c->ev_pool.size()) {
            for (int k = 0; k < 64; ++k) {
                cudaEvent_t e;
                CK(cudaEventCreate(&e));
                c->ev_pool.push_back(e);
            }
        }
        CK(cudaEventRecord(c->ev_pool[c->ev_used], c->stream));
        ev1 = c->ev_pool[c->ev_used + 1];
        c->ev_used += 2;
    }
    // With the tensor-core pass and up to DEP_GEMV_MAX_ROWS rows, the depformer phases
    // (small matrices, one dependent phase after another) run on the CUDA-core
    // instantiation in groups of 4 rows, as a second launch: [0, dep_ph0) tensor cores,
    // [dep_ph0, nph) CUDA cores.  Above that the groups of 4 cost more passes than the
    // tensor-core phases' hand-offs, and one launch runs every phase.
    const int split = (bi == 3 && nph > c->P.dep_ph0 && n <= DEP_GEMV_MAX_ROWS) ? c->P.dep_ph0 : nph;
    if (c->mode == 0) {
        int ph0 = 0, ph1 = split;
        void* args[] = {&P, &ph0, &ph1, &maxrows};
        CK(cudaLaunchCooperativeKernel(c->kfn[bi], dim3(c->G), dim3(c->threads[bi]), args, c->smem[bi], c->stream));
        c->launches = 1;
        if (split < nph) {
            int q0 = split, q1 = nph;
            void* args2[] = {&P, &q0, &q1, &maxrows};
            CK(cudaLaunchCooperativeKernel(c->kfn[2], dim3(c->G), dim3(c->threads[2]), args2, c->smem[2], c->stream));
            c->launches = 2;
        }
    } else {
        for (int ph = 0; ph < nph; ++ph) {
            const int k = ph < split ? bi : 2;
            int ph0 = ph, ph1 = ph + 1;
            void* args[] = {&P, &ph0, &ph1, &maxrows};
            CK(cudaLaunchKernel(c->kfn[k], dim3(c->G), dim3(c->threads[k]), args, c->smem[k], c->stream));
        }
        c->launches = nph;
    }
    if (ev1) CK(cudaEventRecord(ev1, c->stream));
    return MFS_OK;
}

static StepDesc* next_desc(mfs_ctx* c, int* idx)
{
    const int i = c->desc_next;
    c->desc_next = (i + 1) % DESC_RING;
    cudaEventSynchronize(c->desc_ev[i]);
    *idx = i;
    return &c->h_desc[i];
}

// Read the device error flag (stream must be idle); rolls back positions of
// steps that a device-side token check turned into no-ops.
static int collect_device_error(mfs_ctx* c)
{
    int e[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    CK(cudaMemcpy(e, c->d_err, sizeof e, cudaMemcpyDeviceToHost));
    int rc = MFS_OK;
    if (e[0] != 0) {
        if (e[0] == DERR_TOKEN) {
            for (auto it = c->pending.rbegin(); it != c->pending.rend(); ++it)
                if (it->seq >= e[1])
                    for (size_t k = 0; k < it->slots.size(); ++k) c->pos[it->slots[k]] = it->old_pos[k];
            rc = fail(c, MFS_E_TOKEN, "a device-side token was out of range (step %d); those steps did nothing", e[1]);
        } else {
            static const char* sites[] = {"?", "tagged element", "tagged vector", "weight stage", "ring slot release",
                                          "depformer query", "depformer key/value"};
            const unsigned want = (unsigned)e[3], seen = (unsigned)e[4];
            rc = fail(c, MFS_E_DEVICE,
                      "device wait gave up at %s (expected step %u phase %u, saw step %u phase %u; CTA %d thread %d); "
                      "slot state is undefined",
                      sites[e[2] >= 1 && e[2] <= 6 ? e[2] : 0], want >> 10, want & 1023u, seen >> 10, seen & 1023u,
                      e[5], e[6]);
        }
        CK(cudaMemset(c->d_err, 0, 7 * sizeof(int)));  // err[7] (the wait limit) stays
    }
    c->pending.clear();
    return rc;
}

extern "C" int mfs_sync(mfs_ctx* c)
{
    if (!c) return MFS_E_ARG;
    CK(cudaStreamSynchronize(c->stream));
    return collect_device_error(c);
}

// The next step's sequence number.  A tag is (seq << 10) | phase in 32 bits, so tags
// repeat every 2^22 steps.  Before the step that starts a period, every tagged word is
// set to 0xFFFFFFFF (phase 1023), which no step writes (at most 1023 phases), so no word
// left from an earlier period can match a tag (the reset is ordered after every
// launch of the earlier steps on the stream).
static int next_seq(mfs_ctx* c, int& seq)
{
    ++c->seq;
    if ((c->seq & 0x3FFFFFu) == 0u) {
        CK(cudaMemsetAsync(c->act + c->tag_off, 0xFF, c->tag_bytes, c->stream));
        if (c->mma_buf) CK(cudaMemsetAsync(c->mma_buf, 0xFF, c->mma_bytes, c->stream));
    }
    seq = (int)(c->seq & 0x7FFFFFFFu);
    return MFS_OK;
}

static int fill_desc(mfs_ctx* c, StepDesc* h, int n, const int32_t* slots, const int32_t* codes, int frame_off)
{
    h->n = n;
    if (next_seq(c, h->seq) != MFS_OK) return MFS_E_CUDA;
    h->sampled = 0;
    h->prompt_rows = 0;
    for (int i = 0; i < n; ++i) {
        h->slot[i] = slots[i];
        h->pos[i] = c->pos[slots[i]] + frame_off;
        if (codes) memcpy(h->codes[i], codes + (size_t)i * NSTREAM, NSTREAM * sizeof(int));
    }
    return MFS_OK;
}

static int step_host(mfs_ctx* c, int n, const int32_t* slots, const int32_t* in_codes, const float* uniforms,
                     int32_t* text_tok, int32_t* codes);

extern "C" int mfs_step(mfs_ctx* c, int n, const int32_t* slots, const int32_t* in_codes, int32_t* text_tok,
                        int32_t* codes)
{
    return step_host(c, n, slots, in_codes, nullptr, text_tok, codes);
}

extern "C" int mfs_step_sampled(mfs_ctx* c, int n, const int32_t* slots, const int32_t* in_codes, const float* uniforms,
                                int32_t* text_tok, int32_t* codes)
{
    if (!c) return MFS_E_ARG;
    if (!uniforms) return fail(c, MFS_E_ARG, "null uniforms");
    for (int i = 0; i < n * NSTREAM; ++i)
        if (!(uniforms[i] >= 0.f && uniforms[i] < 1.f)) return fail(c, MFS_E_ARG, "uniform %d outside [0, 1)", i);
    return step_host(c, n, slots, in_codes, uniforms, text_tok, codes);
}

extern "C" int mfs_set_sampling(mfs_ctx* c, int slot, float text_temp, int text_topk, float audio_temp, int audio_topk)
{
    if (!c) return MFS_E_ARG;
    if (slot < 0 || slot >= c->cfg.max_slots) return fail(c, MFS_E_SLOT, "slot %d outside [0, %d)", slot, c->cfg.max_slots);
    if (text_topk < 0 || audio_topk < 0 || !(text_temp >= 0.f) || !(audio_temp >= 0.f))
        return fail(c, MFS_E_ARG, "sampling: temperatures and top-k must be >= 0");
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    SampleCfg cfg;
    cfg.text_inv_t = text_temp > 0.f ? 1.f / text_temp : 0.f;
    cfg.text_k = text_topk;
    cfg.audio_inv_t = audio_temp > 0.f ? 1.f / audio_temp : 0.f;
    cfg.audio_k = audio_topk;
    CK(cudaMemcpy((SampleCfg*)c->P.samp + slot, &cfg, sizeof cfg, cudaMemcpyHostToDevice));
    return MFS_OK;
}

static int step_host(mfs_ctx* c, int n, const int32_t* slots, const int32_t* in_codes, const float* uniforms,
                     int32_t* text_tok, int32_t* codes)
{
    if (!c) return MFS_E_ARG;
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    int rc = weights_ready(c);
    if (rc) return rc;
    if ((rc = check_slots(c, n, slots, 1))) return rc;
    if (!in_codes || !text_tok || !codes) return fail(c, MFS_E_ARG, "null buffer");
    if ((rc = check_tokens(c, in_codes, n, -1))) return rc;
    int di;
    StepDesc* h = next_desc(c, &di);
    if ((rc = fill_desc(c, h, n, slots, in_codes, 0))) return rc;
    if (uniforms) {
        h->sampled = 1;
        memcpy(c->h_unif, uniforms, (size_t)n * NSTREAM * sizeof(float));
        CK(cudaMemcpyAsync((float*)c->P.unif, c->h_unif, (size_t)n * NSTREAM * sizeof(float), cudaMemcpyHostToDevice,
                           c->stream));
    }
    CK(cudaMemcpyAsync(c->d_desc, h, sizeof(StepDesc), cudaMemcpyHostToDevice, c->stream));
    CK(cudaEventRecord(c->desc_ev[di], c->stream));
    if ((rc = launch(c, n, c->nphase, c->d_desc))) return rc;
    int* ho = c->h_out;
    CK(cudaMemcpyAsync(ho, c->P.text_out, n * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaMemcpyAsync(ho + MFS_MAX_SLOTS, c->P.codes_out, n * 16 * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaMemcpyAsync(ho + MFS_MAX_SLOTS * 17, c->d_err, 2 * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    if (ho[MFS_MAX_SLOTS * 17] != 0) return collect_device_error(c);
    memcpy(text_tok, ho, n * sizeof(int));
    memcpy(codes, ho + MFS_MAX_SLOTS, n * 16 * sizeof(int));
    for (int i = 0; i < n; ++i) c->pos[slots[i]] += 1;
    c->last_n = n;
    c->last_full = true;
    return MFS_OK;
}

extern "C" int mfs_step_device(mfs_ctx* c, int n, const int32_t* slots, const int32_t* d_in_codes,
                               int32_t* d_text_tok, int32_t* d_codes)
{
    if (!c) return MFS_E_ARG;
    int rc = weights_ready(c);
    if (rc) return rc;
    if ((rc = check_slots(c, n, slots, 1))) return rc;
    if (!d_in_codes) return fail(c, MFS_E_ARG, "null device codes");
    int di;
    StepDesc* h = next_desc(c, &di);
    if ((rc = fill_desc(c, h, n, slots, nullptr, 0))) return rc;
    const size_t head = offsetof(StepDesc, codes);
    CK(cudaMemcpyAsync(c->d_desc, h, head, cudaMemcpyHostToDevice, c->stream));
    CK(cudaEventRecord(c->desc_ev[di], c->stream));
    CK(cudaMemcpyAsync(c->d_desc->codes, d_in_codes, (size_t)n * NSTREAM * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
    if ((rc = launch(c, n, c->nphase, c->d_desc))) return rc;
    if (d_text_tok) CK(cudaMemcpyAsync(d_text_tok, c->P.text_out, n * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
    if (d_codes) CK(cudaMemcpyAsync(d_codes, c->P.codes_out, n * 16 * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
    Pending pd;
    pd.seq = h->seq;
    for (int i = 0; i < n; ++i) {
        pd.slots.push_back(slots[i]);
        pd.old_pos.push_back(c->pos[slots[i]]);
        c->pos[slots[i]] += 1;
    }
    c->pending.push_back(pd);
    c->last_n = n;
    c->last_full = true;
    return MFS_OK;
}

extern "C" int mfs_prefill(mfs_ctx* c, int n, const int32_t* slots, int T, const int32_t* codes)
{
    if (!c) return MFS_E_ARG;
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    int rc = weights_ready(c);
    if (rc) return rc;
    if (T < 0) return fail(c, MFS_E_ARG, "T < 0");
    if ((rc = check_slots(c, n, slots, T))) return rc;
    if (T == 0) return MFS_OK;
    if (!codes) return fail(c, MFS_E_ARG, "null codes");
    if ((rc = check_tokens(c, codes, n * T, 0))) return rc;
    // Launches of up to PROMPT_ROWS rows: a chunk takes tc consecutive frames of every
    // slot (rows of a slot consecutive, in frame order) while every position of the
    // chunk stays below the window, so that no ring row it writes is still read;
    // otherwise one frame per launch.
    int maxpos = 0;
    for (int i = 0; i < n; ++i) maxpos = c->pos[slots[i]] > maxpos ? c->pos[slots[i]] : maxpos;
    const int tc_max = n <= PROMPT_ROWS ? PROMPT_ROWS / n : 1;
    std::vector<int> chunk_t0, chunk_tc;
    for (int t0 = 0; t0 < T;) {
        int tc = tc_max < T - t0 ? tc_max : T - t0;
        if (maxpos + t0 + tc > c->cfg.window) tc = 1;
        chunk_t0.push_back(t0);
        chunk_tc.push_back(tc);
        t0 += tc;
    }
    for (size_t q0 = 0; q0 < chunk_t0.size(); q0 += PREF_CHUNK) {
        const size_t qn = chunk_t0.size() - q0 < (size_t)PREF_CHUNK ? chunk_t0.size() - q0 : (size_t)PREF_CHUNK;
        CK(cudaStreamSynchronize(c->stream));  // the pinned staging is reused
        for (size_t q = 0; q < qn; ++q) {
            const int t0 = chunk_t0[q0 + q], tc = chunk_tc[q0 + q];
            StepDesc* h = &c->h_pref[q];
            h->n = n * tc;
            if (next_seq(c, h->seq) != MFS_OK) return MFS_E_CUDA;
            h->sampled = 0;
            h->prompt_rows = tc > 1;
            for (int i = 0; i < n; ++i)
                for (int t = 0; t < tc; ++t) {
                    const int r = i * tc + t;
                    h->slot[r] = slots[i];
                    h->pos[r] = c->pos[slots[i]] + t0 + t;
                    memcpy(h->codes[r], codes + ((size_t)i * T + t0 + t) * NSTREAM, NSTREAM * sizeof(int));
                }
        }
        CK(cudaMemcpyAsync(c->d_pref, c->h_pref, qn * sizeof(StepDesc), cudaMemcpyHostToDevice, c->stream));
        for (size_t q = 0; q < qn; ++q)
            if ((rc = launch(c, n * chunk_tc[q0 + q], c->nphase_prefill, c->d_pref + q))) return rc;
    }
    CK(cudaMemcpyAsync(c->h_out + MFS_MAX_SLOTS * 17, c->d_err, 2 * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    if (c->h_out[MFS_MAX_SLOTS * 17] != 0) return collect_device_error(c);
    for (int i = 0; i < n; ++i) c->pos[slots[i]] += T;
    c->last_full = false;
    return MFS_OK;
}

extern "C" int mfs_reset_slot(mfs_ctx* c, int slot)
{
    if (!c) return MFS_E_ARG;
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    if (slot < 0 || slot >= c->cfg.max_slots) return fail(c, MFS_E_SLOT, "slot %d outside [0, %d)", slot, c->cfg.max_slots);
    CK(cudaMemsetAsync(c->hist + (size_t)slot * NSTREAM * HIST, 0xFF, NSTREAM * HIST * sizeof(int), c->stream));
    CK(cudaStreamSynchronize(c->stream));
    c->pos[slot] = 0;
    return MFS_OK;
}

// ------------------------------------------------------------------ slot state

static size_t ring_bytes(const mfs_ctx* c)
{
    return (size_t)c->cfg.n_layers * c->cfg.window * c->cfg.d * c->kvb;
}

// A slot's key and value rings between the device layout [L][H][W][hd] and the
// slot-state layout [L][W][d] (keys, then values) of a host buffer: one
// contiguous host copy per tensor through a device staging buffer, transposed
// there by pitched device copies (one per layer and head).  Exactly one of
// out (export) and in (import) is set.
static int ring_transfer(mfs_ctx* c, int slot, char* out, const char* in)
{
    const size_t L = c->cfg.n_layers, W = c->cfg.window, d = c->cfg.d, H = c->cfg.n_heads, hd = c->cfg.head_dim;
    const size_t kvb = c->kvb, rb = ring_bytes(c);
    char* stage = nullptr;
    CK(cudaMalloc((void**)&stage, rb));
    int rc = MFS_OK;
    for (int t = 0; t < 2 && rc == MFS_OK; ++t) {
        char* ring = (char*)(t == 0 ? c->kc : c->vc) + (size_t)slot * rb;
        cudaError_t e = cudaSuccess;
        if (in) e = cudaMemcpy(stage, in + (size_t)t * rb, rb, cudaMemcpyHostToDevice);
        for (size_t l = 0; l < L && e == cudaSuccess; ++l)
            for (size_t h = 0; h < H && e == cudaSuccess; ++h) {
                char* dev = ring + ((l * H + h) * W * hd) * kvb;    // [W][hd], rows hd apart
                char* flat = stage + (l * W * d + h * hd) * kvb;   // [W] rows of the head, d apart
                e = in ? cudaMemcpy2D(dev, hd * kvb, flat, d * kvb, hd * kvb, W, cudaMemcpyDeviceToDevice)
                       : cudaMemcpy2D(flat, d * kvb, dev, hd * kvb, hd * kvb, W, cudaMemcpyDeviceToDevice);
            }
        if (e == cudaSuccess && out) e = cudaMemcpy(out + (size_t)t * rb, stage, rb, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) rc = fail(c, MFS_E_CUDA, "slot state copy: %s", cudaGetErrorString(e));
    }
    cudaFree(stage);
    return rc;
}

extern "C" size_t mfs_slot_state_bytes(const mfs_ctx* c)
{
    if (!c) return 0;
    return MFS_SLOT_HEADER_BYTES + 2 * ring_bytes(c);
}

extern "C" int mfs_export_slot(mfs_ctx* c, int slot, void* buf, size_t bytes)
{
    if (!c || !buf) return MFS_E_ARG;
    if (slot < 0 || slot >= c->cfg.max_slots) return fail(c, MFS_E_SLOT, "slot %d outside [0, %d)", slot, c->cfg.max_slots);
    if (bytes != mfs_slot_state_bytes(c)) return fail(c, MFS_E_ARG, "slot state is %zu bytes, not %zu", mfs_slot_state_bytes(c), bytes);
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    CK(cudaStreamSynchronize(c->stream));
    char* out = (char*)buf;
    memset(out, 0, MFS_SLOT_HEADER_BYTES);
    int32_t head[4] = {1, c->pos[slot], c->cfg.window, c->cfg.kv_dtype};
    memcpy(out, head, sizeof head);
    CK(cudaMemcpy(out + sizeof head, c->hist + (size_t)slot * NSTREAM * HIST, NSTREAM * HIST * sizeof(int),
                  cudaMemcpyDeviceToHost));
    return ring_transfer(c, slot, out + MFS_SLOT_HEADER_BYTES, nullptr);
}

extern "C" int mfs_import_slot(mfs_ctx* c, int slot, const void* buf, size_t bytes)
{
    if (!c || !buf) return MFS_E_ARG;
    if (slot < 0 || slot >= c->cfg.max_slots) return fail(c, MFS_E_SLOT, "slot %d outside [0, %d)", slot, c->cfg.max_slots);
    if (bytes != mfs_slot_state_bytes(c)) return fail(c, MFS_E_ARG, "slot state is %zu bytes, not %zu", mfs_slot_state_bytes(c), bytes);
    const char* in = (const char*)buf;
    int32_t head[4];
    memcpy(head, in, sizeof head);
    if (head[0] != 1 || head[2] != c->cfg.window || head[3] != c->cfg.kv_dtype)
        return fail(c, MFS_E_ARG, "slot state header (version %d, window %d, kv dtype %d) does not match this context",
                    head[0], head[2], head[3]);
    if (head[1] < 0 || head[1] > c->cfg.max_pos) return fail(c, MFS_E_ARG, "slot state position %d outside [0, %d]", head[1], c->cfg.max_pos);
    int32_t hist[NSTREAM * HIST];
    memcpy(hist, in + sizeof head, sizeof hist);
    for (int k = 0; k < NSTREAM; ++k)
        for (int t = 0; t < HIST; ++t) {
            const int v = hist[k * HIST + t], lim = k == 0 ? c->cfg.text_vocab : c->cfg.card;
            if (v < -1 || v >= lim) return fail(c, MFS_E_ARG, "slot state history: stream %d holds token %d", k, v);
        }
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    CK(cudaStreamSynchronize(c->stream));
    CK(cudaMemcpy(c->hist + (size_t)slot * NSTREAM * HIST, hist, sizeof hist, cudaMemcpyHostToDevice));
    const int rc = ring_transfer(c, slot, nullptr, in + MFS_SLOT_HEADER_BYTES);
    if (rc != MFS_OK) return rc;
    c->pos[slot] = head[1];
    return MFS_OK;
}

extern "C" int mfs_position(const mfs_ctx* c, int slot)
{
    if (!c) return MFS_E_ARG;
    if (slot < 0 || slot >= c->cfg.max_slots) return MFS_E_SLOT;
    return c->pos[slot];
}

extern "C" int mfs_read_debug(mfs_ctx* c, float* text_logits, float* dep_logits, int32_t* text_argmax,
                              int32_t* code_argmax)
{
    if (!c) return MFS_E_ARG;
    if (!c->last_full || c->last_n == 0) return fail(c, MFS_E_STATE, "no full step to report");
    CK(cudaStreamSynchronize(c->stream));
    const size_t n = c->last_n;
    if (text_logits) CK(cudaMemcpy(text_logits, c->P.logits, n * c->cfg.text_vocab * 4, cudaMemcpyDeviceToHost));
    if (dep_logits) CK(cudaMemcpy(dep_logits, c->P.dlogits, n * 16 * c->cfg.card * 4, cudaMemcpyDeviceToHost));
    if (text_argmax) CK(cudaMemcpy(text_argmax, c->P.text_argmax, n * 4, cudaMemcpyDeviceToHost));
    if (code_argmax) CK(cudaMemcpy(code_argmax, c->P.code_argmax, n * 16 * 4, cudaMemcpyDeviceToHost));
    return MFS_OK;
}

extern "C" int mfs_set_ring_mask_oldest(mfs_ctx* c, int on)
{
    if (!c) return MFS_E_ARG;
    if (on != 0 && on != 1) return fail(c, MFS_E_ARG, "on must be 0 or 1");
    if (on && c->cfg.window < 2) return fail(c, MFS_E_ARG, "masking the oldest slot needs a window of at least 2");
    CK(cudaStreamSynchronize(c->stream));
    c->P.Wa = on ? c->cfg.window - 1 : c->cfg.window;
    return MFS_OK;
}

extern "C" int mfs_debug_set_seq(mfs_ctx* c, uint32_t seq)
{
    if (!c) return MFS_E_ARG;
    CK(cudaStreamSynchronize(c->stream));
    c->seq = seq;
    return MFS_OK;
}

extern "C" int mfs_set_mode(mfs_ctx* c, int mode)
{
    if (!c) return MFS_E_ARG;
    if (mode != 0 && mode != 1) return fail(c, MFS_E_ARG, "mode must be 0 or 1");
    c->mode = mode;
    return MFS_OK;
}

extern "C" int mfs_set_wait_limit(mfs_ctx* c, int ms)
{
    if (!c) return MFS_E_ARG;
    if (ms < 1 || ms > 60000) return fail(c, MFS_E_ARG, "wait limit %d ms outside [1, 60000]", ms);
    if (!c->pending.empty()) {
        int rc = mfs_sync(c);
        if (rc != MFS_OK) return rc;
    }
    const int us = ms * 1000;
    CK(cudaMemcpy(c->d_err + 7, &us, sizeof us, cudaMemcpyHostToDevice));
    return MFS_OK;
}

extern "C" int mfs_debug_stall(mfs_ctx* c, int slot)
{
    if (!c) return MFS_E_ARG;
    int rc = weights_ready(c);
    if (rc) return rc;
    if (!c->pending.empty() && (rc = mfs_sync(c)) != MFS_OK) return rc;
    if (slot < 0 || slot >= c->cfg.max_slots) return fail(c, MFS_E_SLOT, "slot %d outside [0, %d)", slot, c->cfg.max_slots);
    if (c->pos[slot] >= c->cfg.max_pos) return fail(c, MFS_E_RANGE, "slot %d is at max_pos", slot);
    int di;
    StepDesc* h = next_desc(c, &di);
    if ((rc = fill_desc(c, h, 1, &slot, nullptr, 0))) return rc;
    for (int k = 0; k < NSTREAM; ++k) h->codes[0][k] = -1;
    CK(cudaMemcpyAsync(c->d_desc, h, sizeof(StepDesc), cudaMemcpyHostToDevice, c->stream));
    CK(cudaEventRecord(c->desc_ev[di], c->stream));
    // the first QKV phase alone: its input (this step's embedding sum) is never produced
    Params P = c->P;
    P.desc = c->d_desc;
    P.ptime = nullptr;
    int ph0 = 1, ph1 = 2, maxrows = c->maxrows;
    void* args[] = {&P, &ph0, &ph1, &maxrows};
    CK(cudaLaunchKernel(c->kfn[0], dim3(c->G), dim3(NT + 32), args, c->smem[0], c->stream));
    CK(cudaStreamSynchronize(c->stream));
    int e0 = 0;
    CK(cudaMemcpy(&e0, c->d_err, sizeof e0, cudaMemcpyDeviceToHost));
    if (e0 == 0) return fail(c, MFS_E_STATE, "the stalled phase did not give up");
    c->last_full = false;
    return collect_device_error(c);
}

extern "C" int mfs_set_skip_settled(mfs_ctx* c, int on)
{
    if (!c) return MFS_E_ARG;
    if (on != 0 && on != 1) return fail(c, MFS_E_ARG, "skip_settled must be 0 or 1");
    c->P.skip_settled = on;
    return MFS_OK;
}

extern "C" int mfs_launches_per_step(const mfs_ctx* c)
{
    if (!c) return MFS_E_ARG;
    return c->launches;
}

extern "C" int mfs_set_timing(mfs_ctx* c, int flags)
{
    if (!c) return MFS_E_ARG;
    c->timing = (flags & 1) != 0;
    c->stamps = (flags & 2) != 0;
    if (c->stamps && !c->d_ptime) {
        CK(cudaMalloc((void**)&c->d_ptime, (size_t)(c->nphase + 1) * 8 * sizeof(unsigned long long)));
        CK(cudaMemset(c->d_ptime, 0, (size_t)(c->nphase + 1) * 8 * sizeof(unsigned long long)));
    }
    return MFS_OK;
}

extern "C" int mfs_phase_times(mfs_ctx* c, uint64_t* ns, int cap)
{
    if (!c || !ns) return MFS_E_ARG;
    if (!c->d_ptime) return fail(c, MFS_E_STATE, "phase stamps were never enabled");
    CK(cudaStreamSynchronize(c->stream));
    const int cnt = (c->last_nph + 1) * 8;
    if (cap < cnt) return fail(c, MFS_E_ARG, "need room for %d stamps", cnt);
    CK(cudaMemcpy(ns, c->d_ptime, (size_t)cnt * sizeof(uint64_t), cudaMemcpyDeviceToHost));
    CK(cudaMemset(c->d_ptime, 0, (size_t)cnt * sizeof(uint64_t)));  // the wait totals restart
    return cnt;
}

extern "C" int mfs_kernel_time(mfs_ctx* c, double* total_ms, int* steps)
{
    if (!c || !total_ms || !steps) return MFS_E_ARG;
    CK(cudaStreamSynchronize(c->stream));
    double tot = 0.0;
    for (size_t k = 0; k + 1 < c->ev_used; k += 2) {
        float ms = 0.f;
        CK(cudaEventElapsedTime(&ms, c->ev_pool[k], c->ev_pool[k + 1]));
        tot += ms;
    }
    *total_ms = tot;
    *steps = (int)(c->ev_used / 2);
    c->ev_used = 0;
    return MFS_OK;
}
