/*
 * mfs_oracle.c -- plain CPU definition of the Moshi/PersonaPlex lockstep frame
 * step, in fp64.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and
 * the bench's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * What it computes, per slot and one slot at a time (no batching, no fusion):
 *
 *  S0  the caller's 17 tokens for frame p go into the slot's token history
 *      (-1 = generate).  History keeps 3 frames, indexed by frame mod 3.
 *  S1  the temporal input is the sum of 17 embedding rows.  Stream k reads the
 *      token of frame p-1-delay[k]; frames before 0 read an extra INIT row
 *      (row V of the text table, row C of each audio table).  Delays are
 *      [0, 0, 1 x 7, 0, 1 x 7] (mobius PR #368, "P3 - ONNX Runtime example":
 *      ring cache with per-codebook delays; Kyutai moshi README, "Model
 *      architecture": 80 ms of acoustic delay).
 *  S2..S8  32 pre-norm temporal layers (mobius PR #368, "P2 - Moshi LM":
 *      RoPE, sliding-window causal attention, SwiGLU via FusedGateUpMLP,
 *      RMSNorm eps 1e-8): a = rmsnorm(x); q|k|v = Wqkv a; q and k rotated by
 *      the absolute frame position p (interleaved pairs, theta 10000); keys and
 *      values of positions max(0, p-W+1) .. p (W = 3000 window, vLLM-Omni
 *      PersonaPlex recipe, "Architecture"; with mask_oldest W-1 positions,
 *      the masked oldest slot of SGLang-Omni cookbook, PersonaPlex, "Known
 *      limitations") with a max-subtracted softmax at
 *      scale 1/sqrt(hd); x += Wo o; a = rmsnorm(x); gate|up = Wgu a;
 *      x += Wdown (silu(gate) * up).
 *  S4  h = rmsnorm(x, out_norm); text logits = Wtext h; greedy argmax (lowest
 *      index on ties).  A token the caller supplied (>= 0) replaces it.
 *  S9  depformer (mobius PR #368, "P2 - Moshi LM": 1024-d, 6 layers, no RoPE,
 *      full causal over substeps, 16 per-substep weight sets selected by the
 *      substep index): for substep j = 0..15 (stream k = j+1),
 *      u = Win[j] h + Edep_j[prev] (prev = text token for j = 0, else the
 *      chosen code of stream j), then pre-norm layers with per-substep
 *      linears and shared gains, attention over substeps 0..j, then
 *      rmsnorm(dep out_norm), logits = Head[j] z, argmax.  The code chosen
 *      for frame p-delay[k] is the caller's token if one was supplied, else
 *      the argmax; it is stored into the history when that frame is >= 0.
 *  S10 outputs: the text token of frame p and, per audio stream, the code of
 *      frame p-delay[k] (-1 for frames before 0); p advances by one.
 *
 * Follow mode (a test input, not part of the method): orc_step can be given,
 * per slot and stream, a token to adopt in place of its own argmax (or draw)
 * wherever that stream's token is generated this step.  A comparison with
 * another implementation passes that implementation's chosen tokens, so the
 * two keep the same token history after a legal flip at a near tie (greedy
 * agreement is only required above a top-2 margin: SGLang-Omni cookbook,
 * PersonaPlex, "Reference parity").  A supplied token still takes precedence,
 * and the arithmetic of every logit is unchanged.
 *
 * Keys (after rotation) and values are cached in the cache's dtype: fp64, or
 * bf16 (round to nearest even) as the model's own KV cache is held
 * (SGLang-Omni cookbook, PersonaPlex, "Known limitations": BF16 KV per request);
 * every key, the current position's included, is read back from the cache.
 *
 * The ring of keys/values is kept two ways: storage at position mod W (the
 * default), or a full history of every position masked to the last W
 * (brute_force = 1).  Both read keys in ascending absolute position.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#define ORC_STREAMS 17
#define ORC_HIST 3

typedef struct {
    int d, n_layers, n_heads, head_dim, ffn, text_vocab, card, n_q, window, max_pos;
    int dep_d, dep_layers, dep_heads, dep_head_dim, dep_ffn, dep_steps;
    int delays[ORC_STREAMS];
    double rope_theta, eps;
    int weight_dtype; /* 0 = fp32, 1 = bf16 */
    int max_slots;
    int brute_force;  /* 1: keep every position, mask to the last W */
    int kv_dtype;     /* 0 = fp64 cache, 1 = keys and values rounded to bf16 when cached */
    int mask_oldest;  /* 1: once the ring holds W positions its oldest is masked (W - 1 keys) */
} orc_config;

typedef struct {
    const void* attn_norm; const void* wqkv; const void* wo;
    const void* ffn_norm; const void* wgu; const void* wdown;
} orc_layer;

typedef struct {
    int pos;
    int hist[ORC_STREAMS][ORC_HIST];
    double* K; /* [n_layers][cap][d] */
    double* V;
    /* sampling (k <= 1 or temperature <= 0: greedy) */
    double text_temp, audio_temp;
    int text_k, audio_k;
} orc_slot;

typedef struct {
    orc_config c;
    int cap; /* positions held per layer */
    const void* emb_text; const void* emb_audio; const void* out_norm; const void* text_head;
    const void* dep_in; const void* dep_emb_text; const void* dep_emb_audio;
    const void* dep_out_norm; const void* dep_head;
    orc_layer* L;
    orc_layer* DL;
    orc_slot* slots;
    char err[256];
} orc;

/* ------------------------------------------------------------------ elements */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* x rounded to the nearest bfloat16 (8 significant bits, ties to even), as a
 * double.  Only normal bf16 magnitudes occur in a key or value cache. */
static double round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    double m = frexp(x, &e);          /* x = m * 2^e, 0.5 <= |m| < 1 */
    double r = nearbyint(ldexp(m, 8)); /* default rounding mode: to nearest, ties to even */
    return ldexp(r, e - 8);
}

/* element i of a weight tensor stored in the model's weight dtype */
static double w_at(const orc* o, const void* base, size_t i)
{
    if (o->c.weight_dtype == 1) return bf16_bits_to_double(((const uint16_t*)base)[i]);
    return (double)((const float*)base)[i];
}

static size_t wbytes(const orc* o) { return o->c.weight_dtype == 1 ? 2 : 4; }

/* ------------------------------------------------------------------ pieces */

/* y[n] = sum_k W[row0+n][k] x[k] for n < N; each row summed in ascending k.
 * Rows are handled four at a time only to give the CPU independent chains;
 * every row's own sum is the plain left-to-right sum. */
static void matvec(const orc* o, const void* W, size_t row0, int N, int K,
                   const double* x, double* y)
{
    if (o->c.weight_dtype == 1) {
        const uint16_t* w = (const uint16_t*)W;
#pragma omp parallel for schedule(static)
        for (int n0 = 0; n0 < N; n0 += 4) {
            int m = N - n0 < 4 ? N - n0 : 4;
            double acc[4] = {0, 0, 0, 0};
            const uint16_t* r[4];
            for (int t = 0; t < 4; ++t) r[t] = w + (row0 + (size_t)(n0 + (t < m ? t : 0))) * (size_t)K;
            for (int k = 0; k < K; ++k) {
                double xv = x[k];
                for (int t = 0; t < 4; ++t) acc[t] += bf16_bits_to_double(r[t][k]) * xv;
            }
            for (int t = 0; t < m; ++t) y[n0 + t] = acc[t];
        }
    } else {
        const float* w = (const float*)W;
#pragma omp parallel for schedule(static)
        for (int n0 = 0; n0 < N; n0 += 4) {
            int m = N - n0 < 4 ? N - n0 : 4;
            double acc[4] = {0, 0, 0, 0};
            const float* r[4];
            for (int t = 0; t < 4; ++t) r[t] = w + (row0 + (size_t)(n0 + (t < m ? t : 0))) * (size_t)K;
            for (int k = 0; k < K; ++k) {
                double xv = x[k];
                for (int t = 0; t < 4; ++t) acc[t] += (double)r[t][k] * xv;
            }
            for (int t = 0; t < m; ++t) y[n0 + t] = acc[t];
        }
    }
}

/* Y[t][n] = sum_k W[n][k] X[t][k] for T frames (prompt path).  Every entry
 * is the same ascending-k sum as matvec(); rows are taken 32 at a time with
 * the frames innermost only so that one pass over W serves all T frames. */
static void matmul_frames(const orc* o, const void* W, int N, int K, const double* X, int T, double* Y)
{
    double* XT = (double*)malloc(sizeof(double) * (size_t)K * (size_t)T);
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) XT[(size_t)k * T + t] = X[(size_t)t * K + k];
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * 32 * (size_t)T);
#pragma omp for schedule(dynamic)
        for (int n0 = 0; n0 < N; n0 += 32) {
            int m = N - n0 < 32 ? N - n0 : 32;
            for (size_t i = 0; i < (size_t)m * T; ++i) acc[i] = 0.0;
            for (int k = 0; k < K; ++k) {
                const double* x = XT + (size_t)k * T;
                for (int r = 0; r < m; ++r) {
                    double w = w_at(o, W, (size_t)(n0 + r) * (size_t)K + (size_t)k);
                    double* a = acc + (size_t)r * T;
                    for (int t = 0; t < T; ++t) a[t] += w * x[t];
                }
            }
            for (int r = 0; r < m; ++r)
                for (int t = 0; t < T; ++t) Y[(size_t)t * N + n0 + r] = acc[(size_t)r * T + t];
        }
        free(acc);
    }
    free(XT);
}

/* RMSNorm: out = x / sqrt(mean(x^2) + eps) * g  (g fp32) */
void orc_rmsnorm(const double* x, const float* g, int n, double eps, double* out)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * r * (double)g[i];
}

/* Rotate one head vector v[hd] by position p: pair (2i, 2i+1) turns by angle
 * p * theta^(-2i/hd). */
void orc_rope(double* v, int hd, int p, double theta)
{
    for (int i = 0; i < hd / 2; ++i) {
        double freq = pow(theta, -2.0 * (double)i / (double)hd);
        double ang = (double)p * freq;
        double c = cos(ang), s = sin(ang);
        double a = v[2 * i], b = v[2 * i + 1];
        v[2 * i] = a * c - b * s;
        v[2 * i + 1] = a * s + b * c;
    }
}

/* softmax(q . k_j / sqrt(hd)) weighted sum of v_j over npos keys.
 * K and V rows are at K + j*stride (head slice already applied). */
void orc_attention(const double* q, const double* K, const double* V, int npos, int hd,
                   long stride, double* out)
{
    double* s = (double*)malloc(sizeof(double) * (size_t)(npos > 0 ? npos : 1));
    double scale = 1.0 / sqrt((double)hd);
    double m = -INFINITY;
    for (int j = 0; j < npos; ++j) {
        double acc = 0.0;
        for (int e = 0; e < hd; ++e) acc += q[e] * K[(long)j * stride + e];
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < npos; ++j) { s[j] = exp(s[j] - m); z += s[j]; }
    for (int e = 0; e < hd; ++e) out[e] = 0.0;
    for (int j = 0; j < npos; ++j) {
        double wgt = s[j] / z;
        for (int e = 0; e < hd; ++e) out[e] += wgt * V[(long)j * stride + e];
    }
    free(s);
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* greedy pick: largest value, lowest index on ties */
static int argmax(const double* v, int n)
{
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

static int mod(int a, int m) { int r = a % m; return r < 0 ? r + m : r; }

/* Temperature + top-k sampling (mobius PR #368, commit note replacing greedy
 * argmax: text temperature 0.7 / top_k 25, audio 0.8 / 250; SGLang-Omni
 * cookbook, PersonaPlex, "Stage sampling": each request draws from its own
 * generator).  The candidates are the k largest logits (ties: lower index
 * first), weighted exp((logit - max) / temp).  With u in [0, 1) the token is
 * the first candidate, in ascending index order, at which the running sum of
 * weights exceeds u times their total; a draw from the candidates'
 * distribution for uniform u.  k <= 1 or temp <= 0 is the argmax. */
int orc_sample_topk(const double* lg, int n, double temp, int k, double u)
{
    if (k <= 1 || temp <= 0.0) return argmax(lg, n);
    if (k > n) k = n;
    /* membership: logit greater, or equal with a lower index, than fewer than k others */
    unsigned char* in = (unsigned char*)calloc((size_t)n, 1);
    /* partial selection sort on (value desc, index asc): k passes */
    for (int r = 0; r < k; ++r) {
        int best = -1;
        for (int i = 0; i < n; ++i) {
            if (in[i]) continue;
            if (best < 0 || lg[i] > lg[best]) best = i;
        }
        in[best] = 1;
    }
    double mx = lg[argmax(lg, n)];
    double tot = 0.0;
    for (int i = 0; i < n; ++i)
        if (in[i]) tot += exp((lg[i] - mx) / temp);
    double target = u * tot, run = 0.0;
    int tok = -1;
    for (int i = 0; i < n && tok < 0; ++i) {
        if (!in[i]) continue;
        run += exp((lg[i] - mx) / temp);
        if (run > target) tok = i;
    }
    if (tok < 0) /* u * tot rounded up to tot: the last candidate */
        for (int i = n - 1; i >= 0 && tok < 0; --i)
            if (in[i]) tok = i;
    free(in);
    return tok;
}

/* ------------------------------------------------------------------ lifecycle */

orc* orc_create(const orc_config* c)
{
    if (c->mask_oldest && c->window < 2) return NULL;
    orc* o = (orc*)calloc(1, sizeof(orc));
    if (!o) return NULL;
    o->c = *c;
    o->cap = c->brute_force ? c->max_pos : c->window;
    o->L = (orc_layer*)calloc((size_t)c->n_layers, sizeof(orc_layer));
    o->DL = (orc_layer*)calloc((size_t)c->dep_layers, sizeof(orc_layer));
    o->slots = (orc_slot*)calloc((size_t)c->max_slots, sizeof(orc_slot));
    for (int s = 0; s < c->max_slots; ++s) {
        o->slots[s].pos = 0;
        for (int k = 0; k < ORC_STREAMS; ++k)
            for (int t = 0; t < ORC_HIST; ++t) o->slots[s].hist[k][t] = -1;
    }
    return o;
}

void orc_destroy(orc* o)
{
    if (!o) return;
    for (int s = 0; s < o->c.max_slots; ++s) { free(o->slots[s].K); free(o->slots[s].V); }
    free(o->slots); free(o->L); free(o->DL); free(o);
}

const char* orc_last_error(orc* o) { return o->err; }

int orc_position(orc* o, int slot) { return o->slots[slot].pos; }

int orc_reset_slot(orc* o, int slot)
{
    if (slot < 0 || slot >= o->c.max_slots) return -1;
    o->slots[slot].pos = 0;
    for (int k = 0; k < ORC_STREAMS; ++k)
        for (int t = 0; t < ORC_HIST; ++t) o->slots[slot].hist[k][t] = -1;
    return 0;
}

/* Replace a slot's state with a buffer in the CUDA library's slot-state layout
 * (its header documents it): 256 bytes of header (int32 version 1, position,
 * window, kv dtype, then history [17][3]), then keys and values
 * [n_layers][W][d] in the kv dtype, row r holding the position q with
 * q mod W == r.  Ring storage only (not brute_force).  Returns 0 or -1. */
static int ensure_kv(orc* o, orc_slot* s);

int orc_import_slot(orc* o, int slot, const void* buf, long long nbytes)
{
    const orc_config* c = &o->c;
    if (slot < 0 || slot >= c->max_slots || c->brute_force) return -1;
    size_t kvb = c->kv_dtype == 1 ? 2 : 4;
    size_t ring = (size_t)c->n_layers * (size_t)c->window * (size_t)c->d;
    if (nbytes != (long long)(256 + 2 * ring * kvb)) return -1;
    const unsigned char* in = (const unsigned char*)buf;
    int32_t head[4 + ORC_STREAMS * ORC_HIST];
    memcpy(head, in, sizeof head);
    if (head[0] != 1 || head[2] != c->window || head[3] != c->kv_dtype || head[1] < 0 || head[1] > c->max_pos) return -1;
    orc_slot* s = &o->slots[slot];
    if (ensure_kv(o, s) != 0) return -1;
    s->pos = head[1];
    for (int k = 0; k < ORC_STREAMS; ++k)
        for (int t = 0; t < ORC_HIST; ++t) s->hist[k][t] = head[4 + k * ORC_HIST + t];
    const unsigned char* kin = in + 256;
    const unsigned char* vin = kin + ring * kvb;
    for (size_t i = 0; i < ring; ++i) {
        if (kvb == 2) {
            uint16_t kb, vb;
            memcpy(&kb, kin + 2 * i, 2);
            memcpy(&vb, vin + 2 * i, 2);
            s->K[i] = bf16_bits_to_double(kb);
            s->V[i] = bf16_bits_to_double(vb);
        } else {
            float kf, vf;
            memcpy(&kf, kin + 4 * i, 4);
            memcpy(&vf, vin + 4 * i, 4);
            s->K[i] = kf;
            s->V[i] = vf;
        }
    }
    return 0;
}

/* The slot's state in the same layout (ring storage only); keys and values
 * are converted to the kv dtype (exact for a bf16 cache, which holds bf16
 * values already).  Returns 0 or -1. */
int orc_export_slot(orc* o, int slot, void* buf, long long nbytes)
{
    const orc_config* c = &o->c;
    if (slot < 0 || slot >= c->max_slots || c->brute_force) return -1;
    size_t kvb = c->kv_dtype == 1 ? 2 : 4;
    size_t ring = (size_t)c->n_layers * (size_t)c->window * (size_t)c->d;
    if (nbytes != (long long)(256 + 2 * ring * kvb)) return -1;
    orc_slot* s = &o->slots[slot];
    if (ensure_kv(o, s) != 0) return -1;
    unsigned char* out = (unsigned char*)buf;
    memset(out, 0, 256);
    int32_t head[4 + ORC_STREAMS * ORC_HIST];
    head[0] = 1; head[1] = s->pos; head[2] = c->window; head[3] = c->kv_dtype;
    for (int k = 0; k < ORC_STREAMS; ++k)
        for (int t = 0; t < ORC_HIST; ++t) head[4 + k * ORC_HIST + t] = s->hist[k][t];
    memcpy(out, head, sizeof head);
    unsigned char* kout = out + 256;
    unsigned char* vout = kout + ring * kvb;
    for (size_t i = 0; i < ring; ++i) {
        if (kvb == 2) {
            /* the cache values are bf16 already: keep the top 16 bits of the float */
            float kf = (float)s->K[i], vf = (float)s->V[i];
            uint32_t ku, vu;
            memcpy(&ku, &kf, 4);
            memcpy(&vu, &vf, 4);
            uint16_t kb = (uint16_t)(ku >> 16), vb = (uint16_t)(vu >> 16);
            memcpy(kout + 2 * i, &kb, 2);
            memcpy(vout + 2 * i, &vb, 2);
        } else {
            float kf = (float)s->K[i], vf = (float)s->V[i];
            memcpy(kout + 4 * i, &kf, 4);
            memcpy(vout + 4 * i, &vf, 4);
        }
    }
    return 0;
}

/* Sampling parameters of a slot (k <= 1 or temp <= 0: greedy); used by
 * orc_step when it is given uniforms. */
int orc_set_sampling(orc* o, int slot, double text_temp, int text_k, double audio_temp, int audio_k)
{
    if (slot < 0 || slot >= o->c.max_slots) return -1;
    orc_slot* s = &o->slots[slot];
    s->text_temp = text_temp; s->text_k = text_k;
    s->audio_temp = audio_temp; s->audio_k = audio_k;
    return 0;
}

/* Borrow a host tensor by name; size must match the shape the config implies. */
int orc_set_weight(orc* o, const char* name, const void* data, long long nbytes)
{
    const orc_config* c = &o->c;
    size_t wb = wbytes(o);
    long long d = c->d, F = c->ffn, V = c->text_vocab, C = c->card, S = c->dep_steps;
    long long dd = c->dep_d, dF = c->dep_ffn;
    int l = -1;
    char tail[64];
    const void** slot = NULL;
    long long want = -1;
    if (!strcmp(name, "emb.text")) { slot = &o->emb_text; want = (V + 1) * d * wb; }
    else if (!strcmp(name, "emb.audio")) { slot = &o->emb_audio; want = c->n_q * (C + 1) * d * wb; }
    else if (!strcmp(name, "out_norm")) { slot = &o->out_norm; want = d * 4; }
    else if (!strcmp(name, "text_head")) { slot = &o->text_head; want = V * d * wb; }
    else if (!strcmp(name, "dep.in")) { slot = &o->dep_in; want = S * dd * d * wb; }
    else if (!strcmp(name, "dep.emb.text")) { slot = &o->dep_emb_text; want = V * dd * wb; }
    else if (!strcmp(name, "dep.emb.audio")) { slot = &o->dep_emb_audio; want = (S - 1) * C * dd * wb; }
    else if (!strcmp(name, "dep.out_norm")) { slot = &o->dep_out_norm; want = dd * 4; }
    else if (!strcmp(name, "dep.head")) { slot = &o->dep_head; want = S * C * dd * wb; }
    else if (sscanf(name, "dep.layers.%d.%63s", &l, tail) == 2) {
        if (l < 0 || l >= c->dep_layers) goto bad;
        orc_layer* Ly = &o->DL[l];
        if (!strcmp(tail, "attn_norm")) { slot = &Ly->attn_norm; want = dd * 4; }
        else if (!strcmp(tail, "ffn_norm")) { slot = &Ly->ffn_norm; want = dd * 4; }
        else if (!strcmp(tail, "wqkv")) { slot = &Ly->wqkv; want = S * 3 * dd * dd * wb; }
        else if (!strcmp(tail, "wo")) { slot = &Ly->wo; want = S * dd * dd * wb; }
        else if (!strcmp(tail, "wgu")) { slot = &Ly->wgu; want = S * 2 * dF * dd * wb; }
        else if (!strcmp(tail, "wdown")) { slot = &Ly->wdown; want = S * dd * dF * wb; }
    } else if (sscanf(name, "layers.%d.%63s", &l, tail) == 2) {
        if (l < 0 || l >= c->n_layers) goto bad;
        orc_layer* Ly = &o->L[l];
        if (!strcmp(tail, "attn_norm")) { slot = &Ly->attn_norm; want = d * 4; }
        else if (!strcmp(tail, "ffn_norm")) { slot = &Ly->ffn_norm; want = d * 4; }
        else if (!strcmp(tail, "wqkv")) { slot = &Ly->wqkv; want = 3 * d * d * wb; }
        else if (!strcmp(tail, "wo")) { slot = &Ly->wo; want = d * d * wb; }
        else if (!strcmp(tail, "wgu")) { slot = &Ly->wgu; want = 2 * F * d * wb; }
        else if (!strcmp(tail, "wdown")) { slot = &Ly->wdown; want = d * F * wb; }
    }
    if (!slot) goto bad;
    if (want != nbytes) {
        snprintf(o->err, sizeof o->err, "%s: %lld bytes, expected %lld", name, nbytes, want);
        return -2;
    }
    *slot = data;
    return 0;
bad:
    snprintf(o->err, sizeof o->err, "unknown tensor %s", name);
    return -1;
}

static int weights_ready(orc* o)
{
    const void* need[] = {o->emb_text, o->emb_audio, o->out_norm, o->text_head, o->dep_in,
                          o->dep_emb_text, o->dep_emb_audio, o->dep_out_norm, o->dep_head};
    for (size_t i = 0; i < sizeof need / sizeof need[0]; ++i)
        if (!need[i]) return 0;
    for (int l = 0; l < o->c.n_layers; ++l) {
        orc_layer* y = &o->L[l];
        if (!y->attn_norm || !y->wqkv || !y->wo || !y->ffn_norm || !y->wgu || !y->wdown) return 0;
    }
    for (int l = 0; l < o->c.dep_layers; ++l) {
        orc_layer* y = &o->DL[l];
        if (!y->attn_norm || !y->wqkv || !y->wo || !y->ffn_norm || !y->wgu || !y->wdown) return 0;
    }
    return 1;
}

static int ensure_kv(orc* o, orc_slot* s)
{
    if (s->K) return 0;
    size_t n = (size_t)o->c.n_layers * (size_t)o->cap * (size_t)o->c.d;
    s->K = (double*)calloc(n, sizeof(double));
    s->V = (double*)calloc(n, sizeof(double));
    return (s->K && s->V) ? 0 : -1;
}

/* ------------------------------------------------------------------ the step */

/* S1: token index read by stream k at step p (INIT row when that frame is < 0). */
static int input_token(const orc* o, const orc_slot* s, int k, int p)
{
    int f = p - 1 - o->c.delays[k];
    if (f < 0) return k == 0 ? o->c.text_vocab : o->c.card;
    return s->hist[k][mod(f, ORC_HIST)];
}

/* Rotate q and k of one position, store k and v at the ring row of position p,
 * and attend over the window of p (keys in ascending absolute position): the last
 * W positions, or with mask_oldest the last W - 1 (SGLang-Omni cookbook,
 * PersonaPlex, "Known limitations": the oldest slot of a full ring is masked). */
static void attend(orc* o, orc_slot* s, int l, int p, double* q, double* k, const double* v, double* att)
{
    const orc_config* c = &o->c;
    int d = c->d, H = c->n_heads, hd = c->head_dim, W = c->window;
    int Wa = c->mask_oldest ? W - 1 : W;
    int len = p + 1 < Wa ? p + 1 : Wa;
    int start = p - len + 1;
    size_t layer_stride = (size_t)o->cap * (size_t)d;
    for (int hh = 0; hh < H; ++hh) {
        orc_rope(q + hh * hd, hd, p, c->rope_theta);
        orc_rope(k + hh * hd, hd, p, c->rope_theta);
    }
    if (c->kv_dtype == 1) {
        /* the cache holds keys and values in bf16: the current position is read
         * back from it like every other */
        for (int i = 0; i < d; ++i) { k[i] = round_bf16(k[i]); }
    }
    int row = c->brute_force ? p : mod(p, W);
    double* Kl = s->K + (size_t)l * layer_stride;
    double* Vl = s->V + (size_t)l * layer_stride;
    memcpy(Kl + (size_t)row * d, k, sizeof(double) * (size_t)d);
    memcpy(Vl + (size_t)row * d, v, sizeof(double) * (size_t)d);
    if (c->kv_dtype == 1)
        for (int i = 0; i < d; ++i) Vl[(size_t)row * d + i] = round_bf16(Vl[(size_t)row * d + i]);
    double* Kw = (double*)malloc(sizeof(double) * (size_t)len * (size_t)d);
    double* Vw = (double*)malloc(sizeof(double) * (size_t)len * (size_t)d);
    /* the window in ascending position; heads are independent (threads only share
     * the work, each head's sums keep their order) */
#pragma omp parallel for schedule(static)
    for (int j = 0; j < len; ++j) {
        int pos = start + j;
        int r = c->brute_force ? pos : mod(pos, W);
        memcpy(Kw + (size_t)j * d, Kl + (size_t)r * d, sizeof(double) * (size_t)d);
        memcpy(Vw + (size_t)j * d, Vl + (size_t)r * d, sizeof(double) * (size_t)d);
    }
#pragma omp parallel for schedule(static)
    for (int hh = 0; hh < H; ++hh)
        orc_attention(q + hh * hd, Kw + hh * hd, Vw + hh * hd, len, hd, d, att + hh * hd);
    free(Kw); free(Vw);
}

/* temporal stack for one slot at position p; x[d] in, h[d] (post final norm) out
 * when h != NULL. */
static void temporal(orc* o, orc_slot* s, int p, double* x, double* h)
{
    const orc_config* c = &o->c;
    int d = c->d, F = c->ffn;
    double* a = (double*)malloc(sizeof(double) * (size_t)d);
    double* qkv = (double*)malloc(sizeof(double) * (size_t)(3 * d));
    double* att = (double*)malloc(sizeof(double) * (size_t)d);
    double* y = (double*)malloc(sizeof(double) * (size_t)d);
    double* gu = (double*)malloc(sizeof(double) * (size_t)(2 * F));
    double* act = (double*)malloc(sizeof(double) * (size_t)F);
    for (int l = 0; l < c->n_layers; ++l) {
        const orc_layer* Ly = &o->L[l];
        orc_rmsnorm(x, (const float*)Ly->attn_norm, d, c->eps, a);
        matvec(o, Ly->wqkv, 0, 3 * d, d, a, qkv);
        attend(o, s, l, p, qkv, qkv + d, qkv + 2 * d, att);
        matvec(o, Ly->wo, 0, d, d, att, y);
        for (int i = 0; i < d; ++i) x[i] += y[i];
        orc_rmsnorm(x, (const float*)Ly->ffn_norm, d, c->eps, a);
        matvec(o, Ly->wgu, 0, 2 * F, d, a, gu);
        for (int i = 0; i < F; ++i) act[i] = silu(gu[i]) * gu[F + i];
        matvec(o, Ly->wdown, 0, d, F, act, y);
        for (int i = 0; i < d; ++i) x[i] += y[i];
    }
    if (h) orc_rmsnorm(x, (const float*)o->out_norm, d, c->eps, h);
    free(a); free(qkv); free(att); free(y); free(gu); free(act);
}

/* S0 + S1 for one slot: record frame p's tokens, build the embedding sum. */
static void embed(orc* o, orc_slot* s, const int* codes, double* x, int* x_tokens)
{
    const orc_config* c = &o->c;
    int p = s->pos, d = c->d;
    for (int k = 0; k < ORC_STREAMS; ++k) s->hist[k][mod(p, ORC_HIST)] = codes[k];
    for (int i = 0; i < d; ++i) x[i] = 0.0;
    for (int k = 0; k < ORC_STREAMS; ++k) {
        int tok = input_token(o, s, k, p);
        if (x_tokens) x_tokens[k] = tok;
        size_t base;
        const void* table;
        if (k == 0) { table = o->emb_text; base = (size_t)tok * (size_t)d; }
        else { table = o->emb_audio; base = ((size_t)(k - 1) * (size_t)(c->card + 1) + (size_t)tok) * (size_t)d; }
        for (int i = 0; i < d; ++i) x[i] += w_at(o, table, base + (size_t)i);
    }
}

/* depformer for one slot; h[d] is the temporal output, t the text token. */
static void depformer(orc* o, orc_slot* s, const double* h, int t, int* codes_out,
                      double* logits_out, int* argmax_out, const double* unif, const int* follow)
{
    const orc_config* c = &o->c;
    int p = s->pos, d = c->d, dd = c->dep_d, dF = c->dep_ffn, C = c->card, S = c->dep_steps;
    int Hd = c->dep_heads, hd = c->dep_head_dim, Ld = c->dep_layers;
    double* u = (double*)malloc(sizeof(double) * (size_t)dd);
    double* a = (double*)malloc(sizeof(double) * (size_t)dd);
    double* qkv = (double*)malloc(sizeof(double) * (size_t)(3 * dd));
    double* att = (double*)malloc(sizeof(double) * (size_t)dd);
    double* y = (double*)malloc(sizeof(double) * (size_t)dd);
    double* gu = (double*)malloc(sizeof(double) * (size_t)(2 * dF));
    double* act = (double*)malloc(sizeof(double) * (size_t)dF);
    double* lg = (double*)malloc(sizeof(double) * (size_t)C);
    /* keys/values of substeps 0..j for every layer: [Ld][S][dd] */
    double* DK = (double*)calloc((size_t)Ld * (size_t)S * (size_t)dd, sizeof(double));
    double* DV = (double*)calloc((size_t)Ld * (size_t)S * (size_t)dd, sizeof(double));
    int prev = t;
    for (int j = 0; j < S; ++j) {
        int k = j + 1;
        /* u = Win[j] h + Edep_j[prev] */
        matvec(o, o->dep_in, (size_t)j * (size_t)dd, dd, d, h, u);
        if (j == 0) {
            for (int i = 0; i < dd; ++i) u[i] += w_at(o, o->dep_emb_text, (size_t)prev * dd + (size_t)i);
        } else {
            size_t base = ((size_t)(j - 1) * (size_t)C + (size_t)prev) * (size_t)dd;
            for (int i = 0; i < dd; ++i) u[i] += w_at(o, o->dep_emb_audio, base + (size_t)i);
        }
        for (int l = 0; l < Ld; ++l) {
            const orc_layer* Ly = &o->DL[l];
            orc_rmsnorm(u, (const float*)Ly->attn_norm, dd, c->eps, a);
            matvec(o, Ly->wqkv, (size_t)j * (size_t)(3 * dd), 3 * dd, dd, a, qkv);
            double* Kl = DK + (size_t)l * (size_t)S * (size_t)dd;
            double* Vl = DV + (size_t)l * (size_t)S * (size_t)dd;
            memcpy(Kl + (size_t)j * dd, qkv + dd, sizeof(double) * (size_t)dd);
            memcpy(Vl + (size_t)j * dd, qkv + 2 * dd, sizeof(double) * (size_t)dd);
            for (int hh = 0; hh < Hd; ++hh)
                orc_attention(qkv + hh * hd, Kl + hh * hd, Vl + hh * hd, j + 1, hd, dd, att + hh * hd);
            matvec(o, Ly->wo, (size_t)j * (size_t)dd, dd, dd, att, y);
            for (int i = 0; i < dd; ++i) u[i] += y[i];
            orc_rmsnorm(u, (const float*)Ly->ffn_norm, dd, c->eps, a);
            matvec(o, Ly->wgu, (size_t)j * (size_t)(2 * dF), 2 * dF, dd, a, gu);
            for (int i = 0; i < dF; ++i) act[i] = silu(gu[i]) * gu[dF + i];
            matvec(o, Ly->wdown, (size_t)j * (size_t)dd, dd, dF, act, y);
            for (int i = 0; i < dd; ++i) u[i] += y[i];
        }
        orc_rmsnorm(u, (const float*)o->dep_out_norm, dd, c->eps, a);
        matvec(o, o->dep_head, (size_t)j * (size_t)C, C, dd, a, lg);
        if (logits_out) memcpy(logits_out + (size_t)j * C, lg, sizeof(double) * (size_t)C);
        int chat = argmax(lg, C);
        if (argmax_out) argmax_out[j] = chat;
        int f = p - c->delays[k];
        int forced = f >= 0 ? s->hist[k][mod(f, ORC_HIST)] : -1;
        int drawn = unif ? orc_sample_topk(lg, C, s->audio_temp, s->audio_k, unif[k]) : chat;
        if (follow && follow[k] >= 0) drawn = follow[k];  /* follow mode: adopt the given token */
        int chosen = forced >= 0 ? forced : drawn;
        if (f >= 0) {
            s->hist[k][mod(f, ORC_HIST)] = chosen;
            codes_out[j] = chosen;
        } else {
            codes_out[j] = -1;
        }
        prev = chosen;
    }
    free(u); free(a); free(qkv); free(att); free(y); free(gu); free(act); free(lg);
    free(DK); free(DV);
}

static int check_tokens(orc* o, const int* codes, int allow_generate)
{
    int lo = allow_generate ? -1 : 0;
    if (codes[0] < lo || codes[0] >= o->c.text_vocab) return -1;
    for (int k = 1; k < ORC_STREAMS; ++k)
        if (codes[k] < lo || codes[k] >= o->c.card) return -1;
    return 0;
}

/* One frame step for n slots (processed one after another).
 * codes [n][17] (-1 = generate); text_out [n]; codes_out [n][16];
 * optional: text_logits [n][V], dep_logits [n][16][C], text_argmax [n],
 * code_argmax [n][16], x_tokens [n][17] (embedding rows read by S1),
 * unif [n][17] (sampling), follow [n][17] (follow mode: token adopted for a
 * generated stream, -1 = the oracle's own choice). */
int orc_step(orc* o, int n, const int* slots, const int* codes, int* text_out, int* codes_out,
             double* text_logits, double* dep_logits, int* text_argmax, int* code_argmax,
             int* x_tokens, const double* unif, const int* follow)
{
    const orc_config* c = &o->c;
    if (!weights_ready(o)) { snprintf(o->err, sizeof o->err, "weights missing"); return -3; }
    for (int i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= c->max_slots) { snprintf(o->err, sizeof o->err, "bad slot"); return -1; }
        if (check_tokens(o, codes + (size_t)i * ORC_STREAMS, 1)) { snprintf(o->err, sizeof o->err, "bad token"); return -4; }
        if (follow && check_tokens(o, follow + (size_t)i * ORC_STREAMS, 1)) { snprintf(o->err, sizeof o->err, "bad follow token"); return -4; }
        if (o->slots[slots[i]].pos >= c->max_pos) { snprintf(o->err, sizeof o->err, "position limit"); return -5; }
    }
    int d = c->d, V = c->text_vocab;
    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)d);
    double* lg = (double*)malloc(sizeof(double) * (size_t)V);
    for (int i = 0; i < n; ++i) {
        orc_slot* s = &o->slots[slots[i]];
        const int* cd = codes + (size_t)i * ORC_STREAMS;
        if (ensure_kv(o, s)) { free(x); free(h); free(lg); return -6; }
        embed(o, s, cd, x, x_tokens ? x_tokens + (size_t)i * ORC_STREAMS : NULL);
        temporal(o, s, s->pos, x, h);
        matvec(o, o->text_head, 0, V, d, h, lg);
        if (text_logits) memcpy(text_logits + (size_t)i * V, lg, sizeof(double) * (size_t)V);
        int that = argmax(lg, V);
        if (text_argmax) text_argmax[i] = that;
        const double* ui = unif ? unif + (size_t)i * ORC_STREAMS : NULL;
        int tdraw = ui ? orc_sample_topk(lg, V, s->text_temp, s->text_k, ui[0]) : that;
        const int* fi = follow ? follow + (size_t)i * ORC_STREAMS : NULL;
        if (fi && fi[0] >= 0) tdraw = fi[0];  /* follow mode */
        int t = cd[0] >= 0 ? cd[0] : tdraw;
        s->hist[0][mod(s->pos, ORC_HIST)] = t;
        text_out[i] = t;
        depformer(o, s, h, t, codes_out + (size_t)i * (ORC_STREAMS - 1),
                  dep_logits ? dep_logits + (size_t)i * c->dep_steps * c->card : NULL,
                  code_argmax ? code_argmax + (size_t)i * c->dep_steps : NULL, ui, fi);
        s->pos += 1;
    }
    free(x); free(h); free(lg);
    return 0;
}

/* T frames of one slot with every token supplied: the temporal stack only.
 * With all 17 rows forced the text head and the depformer change nothing in
 * the slot's state, so they are not run.  Frames are taken layer by layer
 * (each layer's products for a block of frames at once, then the frames'
 * attention in frame order, so a frame only sees keys of earlier positions);
 * the arithmetic of every frame is that of orc_step. */
#define ORC_PREFILL_BLOCK 256
int orc_prefill(orc* o, int slot, int T, const int* codes)
{
    const orc_config* c = &o->c;
    if (!weights_ready(o)) { snprintf(o->err, sizeof o->err, "weights missing"); return -3; }
    if (slot < 0 || slot >= c->max_slots) return -1;
    orc_slot* s = &o->slots[slot];
    if (s->pos + T > c->max_pos) { snprintf(o->err, sizeof o->err, "position limit"); return -5; }
    for (int t = 0; t < T; ++t)
        if (check_tokens(o, codes + (size_t)t * ORC_STREAMS, 0)) { snprintf(o->err, sizeof o->err, "bad token"); return -4; }
    if (ensure_kv(o, s)) return -6;
    int d = c->d, F = c->ffn;
    for (int t0 = 0; t0 < T; t0 += ORC_PREFILL_BLOCK) {
        int nt = T - t0 < ORC_PREFILL_BLOCK ? T - t0 : ORC_PREFILL_BLOCK;
        int p0 = s->pos;
        double* X = (double*)malloc(sizeof(double) * (size_t)nt * d);
        double* A = (double*)malloc(sizeof(double) * (size_t)nt * d);
        double* QKV = (double*)malloc(sizeof(double) * (size_t)nt * 3 * d);
        double* ATT = (double*)malloc(sizeof(double) * (size_t)nt * d);
        double* Y = (double*)malloc(sizeof(double) * (size_t)nt * d);
        double* GU = (double*)malloc(sizeof(double) * (size_t)nt * 2 * F);
        double* ACT = (double*)malloc(sizeof(double) * (size_t)nt * F);
        for (int t = 0; t < nt; ++t) {
            s->pos = p0 + t;
            embed(o, s, codes + (size_t)(t0 + t) * ORC_STREAMS, X + (size_t)t * d, NULL);
        }
        for (int l = 0; l < c->n_layers; ++l) {
            const orc_layer* Ly = &o->L[l];
            for (int t = 0; t < nt; ++t)
                orc_rmsnorm(X + (size_t)t * d, (const float*)Ly->attn_norm, d, c->eps, A + (size_t)t * d);
            matmul_frames(o, Ly->wqkv, 3 * d, d, A, nt, QKV);
            for (int t = 0; t < nt; ++t) {
                double* q = QKV + (size_t)t * 3 * d;
                attend(o, s, l, p0 + t, q, q + d, q + 2 * d, ATT + (size_t)t * d);
            }
            matmul_frames(o, Ly->wo, d, d, ATT, nt, Y);
            for (size_t i = 0; i < (size_t)nt * d; ++i) X[i] += Y[i];
            for (int t = 0; t < nt; ++t)
                orc_rmsnorm(X + (size_t)t * d, (const float*)Ly->ffn_norm, d, c->eps, A + (size_t)t * d);
            matmul_frames(o, Ly->wgu, 2 * F, d, A, nt, GU);
            for (int t = 0; t < nt; ++t)
                for (int i = 0; i < F; ++i)
                    ACT[(size_t)t * F + i] = silu(GU[(size_t)t * 2 * F + i]) * GU[(size_t)t * 2 * F + F + i];
            matmul_frames(o, Ly->wdown, d, F, ACT, nt, Y);
            for (size_t i = 0; i < (size_t)nt * d; ++i) X[i] += Y[i];
        }
        s->pos = p0 + nt;
        free(X); free(A); free(QKV); free(ATT); free(Y); free(GU); free(ACT);
    }
    return 0;
}

/* ------------------------------------------------------------------ Mimi split RVQ encode */

/* The encoder-side argmin quantizer of Mimi's split residual VQ (mobius PR
 * #368, "P1 - Mimi": SplitResidualVectorQuantizer, encoder-side argmin
 * quantizer, 8 RVQ codes per 80 ms frame; kyutai-labs/moshi, "Mimi": the
 * first codebook is semantic, the rest acoustic).  Frame t's semantic latent
 * z_sem[t] takes the nearest codeword (squared Euclidean distance, ties to the
 * lower index) of codebook 0; its acoustic latent z_ac[t] is quantized by
 * codebooks 1..7 in turn, each on the residual the stage before left
 * (r <- r - chosen codeword).  Codebooks cb [8][Cb][D] fp32; codes [T][8].
 * gap (optional) [T][8]: second-best minus best distance of each stage, for
 * comparisons with an implementation in another precision. */
void orc_rvq_encode(const float* z_sem, const float* z_ac, int T, int D, const float* cb, int Cb, int* codes,
                    double* gap)
{
    double* r = (double*)malloc(sizeof(double) * (size_t)D);
    for (int t = 0; t < T; ++t) {
        for (int q = 0; q < 8; ++q) {
            if (q == 0)
                for (int e = 0; e < D; ++e) r[e] = z_sem[(size_t)t * D + e];
            else if (q == 1)
                for (int e = 0; e < D; ++e) r[e] = z_ac[(size_t)t * D + e];
            const float* book = cb + (size_t)q * Cb * D;
            int best = 0;
            double bd = INFINITY, second = INFINITY;
            for (int c = 0; c < Cb; ++c) {
                double dist = 0.0;
                for (int e = 0; e < D; ++e) {
                    const double diff = r[e] - (double)book[(size_t)c * D + e];
                    dist += diff * diff;
                }
                if (dist < bd) { second = bd; bd = dist; best = c; }
                else if (dist < second) second = dist;
            }
            codes[(size_t)t * 8 + q] = best;
            if (gap) gap[(size_t)t * 8 + q] = second - bd;
            if (q >= 1)
                for (int e = 0; e < D; ++e) r[e] -= (double)book[(size_t)best * D + e];
        }
    }
    free(r);
}
