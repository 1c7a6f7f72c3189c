/*
 * mfs.h -- C ABI of the GB300 lockstep frame step of a Moshi-class
 * full-duplex speech model (PersonaPlex / Moshi RQ-Transformer).
 *
 * One frame step (80 ms of audio per session) for B concurrent sessions
 * ("slots") runs, on one GPU:
 *   - the 17-stream delayed embedding sum (1 text row + 16 audio codebooks,
 *     delays [0, 0, 1 x 7, 0, 1 x 7]: mobius PR #368 "Add PersonaPlex / Moshi
 *     full-duplex S2S support", section "P3 - ONNX Runtime example"; token
 *     column layout: vLLM-Omni PersonaPlex recipe, section "Architecture");
 *   - one decode step of the temporal transformer (RMSNorm, RoPE, sliding-
 *     window causal attention over a per-slot ring of keys/values, SwiGLU:
 *     mobius PR #368, "P2 - Moshi LM"; 3000-frame ring window: vLLM-Omni
 *     PersonaPlex recipe, "Architecture" and "Notes") and a greedy text argmax;
 *   - the 16-substep autoregressive depformer with per-substep weights and a
 *     greedy code argmax per substep (mobius PR #368, "P2 - Moshi LM");
 *     optionally temperature + top-k sampling instead of the argmaxes.
 *
 * Conventions for every entry point:
 *   - Return value: MFS_OK (0) or a negative MFS_E_* status.  An argument
 *     error is detected on the host before anything is launched and leaves
 *     every slot's state unchanged; mfs_last_error() gives a one-line reason.
 *   - Host pointers are read or written only during the call; the library
 *     keeps no reference to them.  Device pointers must be device memory of
 *     the context's GPU.
 *   - All GPU work runs on the stream given to mfs_create().
 *   - A context is not thread-safe: one host thread at a time.
 */
#ifndef MFS_H
#define MFS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MFS_OK 0
#define MFS_E_ARG (-1)     /* null pointer, n out of range, duplicate slot, bad config */
#define MFS_E_SLOT (-2)    /* slot id outside [0, max_slots) */
#define MFS_E_TOKEN (-3)   /* token outside [-1, vocab) (text) or [-1, card) (audio) */
#define MFS_E_RANGE (-4)   /* a slot would pass max_pos frames (context limit) */
#define MFS_E_STATE (-5)   /* weights missing, unknown tensor name or wrong size */
#define MFS_E_CUDA (-6)    /* a CUDA runtime call failed */
#define MFS_E_DEVICE (-7)  /* a device-side wait gave up (bounded spin); state undefined */
#define MFS_E_NOMEM (-8)   /* device or host allocation failed */

#define MFS_DTYPE_F32 0
#define MFS_DTYPE_BF16 1

#define MFS_MAX_SLOTS 64
#define MFS_N_STREAMS 17

typedef struct mfs_ctx mfs_ctx;

/* Model shape and limits.  Stream 0 is the text row; streams 1..16 are the
 * audio codebooks (1..8 agent, 9..16 user); delays[k] is stream k's delay in
 * frames.  window = ring length W (keys of positions p-W+1..p are attended);
 * max_pos = largest frame count a slot may reach (RoPE range).  n_q and
 * dep_steps must be 16.  Limits: head_dim in {64, 128}, dep_head_dim = 64,
 * every K dimension (d, ffn, dep_d, dep_ffn) a multiple of 8 and at most
 * 12288, max_slots <= MFS_MAX_SLOTS. */
typedef struct {
    int d, n_layers, n_heads, head_dim, ffn, text_vocab, card, n_q, window, max_pos;
    int dep_d, dep_layers, dep_heads, dep_head_dim, dep_ffn, dep_steps;
    int delays[MFS_N_STREAMS];
    double rope_theta, eps;
    int weight_dtype; /* MFS_DTYPE_F32 | MFS_DTYPE_BF16: linears and embedding tables */
    int kv_dtype;     /* MFS_DTYPE_F32 | MFS_DTYPE_BF16: the ring of keys/values */
    int max_slots;
} mfs_config;

/* Create a context on the current CUDA device: allocates the weight arena,
 * the per-slot key/value rings (max_slots x n_layers x window x d, for keys
 * and for values), the token histories and the activations.  cuda_stream is a
 * cudaStream_t (NULL: the library creates its own).  Every slot starts fresh
 * (position 0, empty history).  On success *out owns all of it. */
int mfs_create(const mfs_config* cfg, void* cuda_stream, mfs_ctx** out);

/* Synchronize and free everything the context owns. NULL is accepted. */
void mfs_destroy(mfs_ctx* ctx);

/* Reason for the last non-OK status of this context (never NULL); with a
 * NULL context, the reason the last mfs_create() on this thread failed. */
const char* mfs_last_error(const mfs_ctx* ctx);

/* Copy one named tensor into the weight arena (the caller keeps ownership).
 * src: host memory (on_device = 0) or device memory (on_device = 1); bytes
 * must equal the tensor's size.  Names and row-major shapes (W = weight
 * dtype, gains always fp32; V = text_vocab, C = card, S = dep_steps,
 * d' = dep_d, F' = dep_ffn):
 *   emb.text [V+1, d] W        emb.audio [16, C+1, d] W   (row V / C = INIT)
 *   layers.{l}.attn_norm [d]   layers.{l}.wqkv [3d, d] W   (rows q | k | v)
 *   layers.{l}.wo [d, d] W     layers.{l}.ffn_norm [d]
 *   layers.{l}.wgu [2F, d] W   (rows: gate then up)      layers.{l}.wdown [d, F] W
 *   out_norm [d]               text_head [V, d] W
 *   dep.in [S, d', d] W        dep.emb.text [V, d'] W      dep.emb.audio [S-1, C, d'] W
 *   dep.layers.{l}.attn_norm [d']   dep.layers.{l}.wqkv [S, 3d', d'] W
 *   dep.layers.{l}.wo [S, d', d'] W dep.layers.{l}.ffn_norm [d']
 *   dep.layers.{l}.wgu [S, 2F', d'] W   dep.layers.{l}.wdown [S, d', F'] W
 *   dep.out_norm [d']          dep.head [S, C, d'] W
 * Blocking.  Returns MFS_E_STATE for an unknown name or a size mismatch. */
int mfs_load_weights(mfs_ctx* ctx, const char* name, const void* src, size_t bytes, int on_device);

/* One frame step for n slots (1 <= n <= max_slots): the lockstep step with
 * per-codebook delays and delayed output collection (mobius PR #368, "P3 -
 * ONNX Runtime example"), all listed sessions advancing together in one 80 ms
 * tick (vLLM-Omni PersonaPlex recipe, "Notes": batched ticks).
 *   slots    [n]      distinct slot ids (host)
 *   in_codes [n, 17]  frame p's tokens for each slot (host): -1 = generate,
 *                     else the token is forced (text < text_vocab, audio < card)
 *   text_tok [n]      out (host): text token of frame p
 *   codes    [n, 16]  out (host): code of stream k (k = 1..16) for frame
 *                     p - delays[k], or -1 when that frame is before 0
 * Slots not listed are untouched.  Each listed slot advances by one frame.
 * Blocks until the results are on the host. */
int mfs_step(mfs_ctx* ctx, int n, const int32_t* slots, const int32_t* in_codes,
             int32_t* text_tok, int32_t* codes);

/* Same step with device-resident tokens; returns without waiting.
 *   slots (host) [n]; d_in_codes [n, 17], d_text_tok [n], d_codes [n, 16]
 *   (device; may be NULL for outputs that are not wanted).
 * Token ranges are checked on the device: a bad token makes the whole step
 * (and any later step enqueued before the next mfs_sync) a no-op, and the
 * next mfs_sync (or blocking call) returns MFS_E_TOKEN with the positions of
 * those steps rolled back. */
int mfs_step_device(mfs_ctx* ctx, int n, const int32_t* slots, const int32_t* d_in_codes,
                    int32_t* d_text_tok, int32_t* d_codes);

/* Wait for enqueued steps; report a deferred device-side error (see above). */
int mfs_sync(mfs_ctx* ctx);

/* Teacher-forced prompt of T frames for n slots: codes [n, T, 17] (host), every
 * token >= 0 (persona and voice go in through the same lockstep step with their
 * rows supplied: vLLM-Omni PersonaPlex recipe, "Architecture").  Runs the temporal stack only (the text head and depformer
 * cannot change a slot whose every stream is supplied) and advances each slot
 * by T frames.  Blocking. */
int mfs_prefill(mfs_ctx* ctx, int n, const int32_t* slots, int T, const int32_t* codes);

/* Return a slot to the fresh state: position 0, empty history, so that a new
 * session can take it (vLLM-Omni PersonaPlex recipe, "Notes": a recycled slot
 * matches a fresh engine for the same inputs).  Its ring is not cleared:
 * positions are only ever read after being rewritten. */
int mfs_reset_slot(mfs_ctx* ctx, int slot);

/* Frame count of a slot (its next position), or a negative status. */
int mfs_position(const mfs_ctx* ctx, int slot);

/* ---------------------------------------------------------------- slot state
 * A slot's whole decode state as one host buffer, so that a session can be
 * checkpointed, moved to another context, or checked against an independent
 * implementation without replaying its history (SGLang-Omni cookbook,
 * PersonaPlex, "Known limitations": decode states are resident per request).
 * Layout, little-endian, MFS_SLOT_HEADER_BYTES of header then the ring:
 *   int32 version (1), position p, window W, kv dtype (MFS_DTYPE_*),
 *   int32 hist[17][3]: token of stream k for frame f at [k][f mod 3], -1 = none,
 *   zero padding to MFS_SLOT_HEADER_BYTES,
 *   keys [n_layers][W][d] then values [n_layers][W][d] in the kv dtype; row r
 *   holds the position q < p with q mod W == r among the last W positions
 *   (rows of positions never written are unspecified).
 * mfs_slot_state_bytes: the buffer size for this context.  Export copies the
 * slot's state out (waits for the stream); import replaces it after checking
 * the header (version, window, dtype, 0 <= p <= max_pos, every history token
 * -1 or inside its stream's vocabulary), else MFS_E_ARG and nothing changes. */
#define MFS_SLOT_HEADER_BYTES 256
size_t mfs_slot_state_bytes(const mfs_ctx* ctx);
int mfs_export_slot(mfs_ctx* ctx, int slot, void* buf, size_t bytes);
int mfs_import_slot(mfs_ctx* ctx, int slot, const void* buf, size_t bytes);

/* Diagnostics of the last step, rows in that step's slot order (any pointer
 * may be NULL): text logits [n, V], depformer logits [n, 16, C] (fp32), and
 * the raw argmaxes before forcing, text [n] and per substep [n, 16]. */
int mfs_read_debug(mfs_ctx* ctx, float* text_logits, float* dep_logits,
                   int32_t* text_argmax, int32_t* code_argmax);

/* Ring window variant (SGLang-Omni cookbook, PersonaPlex, "Known limitations":
 * the window follows the streaming ring, including the masked oldest slot once
 * the ring fills).  on = 1: a step at position p attends to positions
 * max(0, p - W + 2) .. p, i.e. W - 1 keys once the ring holds W; the ring keeps
 * its capacity W.  on = 0 (default): positions max(0, p - W + 1) .. p.  Applies
 * from the next step on; waits for the context's stream.  MFS_E_ARG if on is not
 * 0 or 1, or W < 2. */
int mfs_set_ring_mask_oldest(mfs_ctx* ctx, int on);

/* Testing: the next step (or prompt launch) takes sequence number seq + 1.
 * Phases hand values over as words tagged (sequence << 10) | phase in 32 bits,
 * so tags repeat every 2^22 steps; before the step whose sequence number is a
 * multiple of 2^22 the library sets every tagged word to a value no step
 * writes.  This call lets a test cross that point without 4 million steps.
 * Waits for the context's stream first; MFS_E_ARG on a null context. */
int mfs_debug_set_seq(mfs_ctx* ctx, uint32_t seq);

/* Execution mode: 0 (default) = one persistent cooperative launch per step,
 * in which a phase waits for the tagged outputs of the phases it reads (no
 * grid-wide barrier); 1 = one launch per phase (same arithmetic, bit for bit,
 * for diagnosis). */
int mfs_set_mode(mfs_ctx* ctx, int mode);

/* Sampling heads (mobius PR #368, commit note replacing greedy argmax with
 * temperature + top-k sampling: text 0.7 / 25, audio 0.8 / 250; SGLang-Omni
 * cookbook, PersonaPlex, "Stage sampling": every request draws from its own
 * generator).  mfs_set_sampling sets a slot's temperatures and top-k (k <= 1
 * or temperature 0: greedy, the default for every slot).  mfs_step_sampled is
 * mfs_step plus uniforms [n, 17] in [0, 1) from the caller's per-session
 * generator: row i's token of stream k (0: text) that is not supplied is drawn
 * with uniforms[i][k] as follows.  The candidates are the k largest logits
 * (ties: lower index first), weighted exp((logit - max) / temperature); the
 * token is the first candidate, in ascending index order, at which the running
 * sum of weights exceeds u times their total.  A drawn token feeds the next
 * substep like a greedy one.  mfs_read_debug still reports the raw argmaxes.
 * Uniforms outside [0, 1) give MFS_E_ARG.  mfs_step and mfs_step_device stay
 * greedy. */
int mfs_set_sampling(mfs_ctx* ctx, int slot, float text_temp, int text_topk, float audio_temp, int audio_topk);
int mfs_step_sampled(mfs_ctx* ctx, int n, const int32_t* slots, const int32_t* in_codes, const float* uniforms,
                     int32_t* text_tok, int32_t* codes);

/* Depformer substeps whose every output is settled without them (mobius PR
 * #368, "P3 - ONNX Runtime example": substep j yields the code of stream j+1;
 * SGLang-Omni cookbook, PersonaPlex, "Known limitations": the depformer steps
 * run after the backbone each frame).  With on = 1, a step skips the trailing
 * substeps j..15 when, for every slot, the tokens of streams j+1..16 are
 * supplied (or belong to frames before 0): the substeps are causal, so the
 * earlier substeps and every output are unchanged.  In decode with the user
 * streams supplied this skips substeps 8..15 (about 1.3 GB of weights per
 * step).  Skipped substeps leave no logits and report argmax -1 in
 * mfs_read_debug.  Default 0: all 16 substeps run. */
int mfs_set_skip_settled(mfs_ctx* ctx, int on);

/* Failure detection (the pages detect failures on the host only, e.g. sessions
 * beyond the batch size are refused: vLLM-Omni PersonaPlex recipe, "Notes";
 * the device-side limit below has no counterpart there).  Every wait inside the step kernel (on another CTA's
 * tagged output, on a weight stage) gives up after a limit, records where,
 * and the call returns MFS_E_DEVICE with that place in mfs_last_error; the
 * context stays usable, the state of the step's slots is undefined (reset or
 * import them).  mfs_set_wait_limit sets the limit (1 .. 60000 ms; default
 * 2000).  mfs_debug_stall checks the mechanism: it launches the slot's first
 * attention-projection phase alone, whose input is never produced, so its
 * waits run out; it returns MFS_E_DEVICE (or MFS_E_STATE if nothing gave up)
 * and leaves the slot's state undefined. */
int mfs_set_wait_limit(mfs_ctx* ctx, int ms);
int mfs_debug_stall(mfs_ctx* ctx, int slot);

/* Kernel launches made by the last step (for accounting). */
int mfs_launches_per_step(const mfs_ctx* ctx);

/* Kernel timing.  flags bit 0: every step records a CUDA event pair on the
 * context's stream around its kernel launch(es); mfs_kernel_time waits for
 * the stream, returns the summed device time (ms) and the number of steps
 * timed since the previous call, and starts a new sum.  flags bit 1: CTA 0
 * records, per phase, 8 values: GPU timer stamps (ns) at the start, when the
 * inputs are ready, when the last weight stage is consumed, at the end (0
 * where a point does not apply), then the ns spent waiting for weight stages
 * and the number of stages, summed since the last read, then the latest end
 * of the phase over all CTAs (timer ns, the maximum since the last read); mfs_phase_times
 * copies [phases + 1][8] values into ns, restarts the sums and returns the
 * count, or a negative status. */
int mfs_set_timing(mfs_ctx* ctx, int flags);
int mfs_kernel_time(mfs_ctx* ctx, double* total_ms, int* steps);
int mfs_phase_times(mfs_ctx* ctx, uint64_t* ns, int cap);

/* ---------------------------------------------------------------- Mimi RVQ
 * Encoder-side argmin quantizer of Mimi's split residual vector quantizer
 * (mobius PR #368, "P1 - Mimi": SplitResidualVectorQuantizer and the
 * encoder-side argmin quantizer, 8 codes per 80 ms frame; kyutai-labs/moshi,
 * "Mimi": the first codebook is semantic).  For each of T frames: codebook 0
 * takes the nearest codeword to z_sem[t]; codebooks 1..7 quantize z_ac[t] and
 * then, in turn, the residual the stage before leaves (r -= chosen codeword).
 * Nearest = least squared Euclidean distance (fp32), ties to the lower index.
 *   z_sem, z_ac  device, [T][D] fp32, 16-byte aligned (the quantizer's input
 *                latents; the codec's trained projections are not part of it)
 *   codebooks    device, [8][Cb][D] fp32, 16-byte aligned
 *   codes        device, [T][8] int32 out
 *   D            multiple of 4 in [4, MFS_RVQ_MAX_DIM]; stream as elsewhere
 * D a multiple of 8: the distances' cross terms r.c run on the tensor cores
 * (bf16 high/low parts of r and c, fp32 accumulation, about 16 significant
 * bits); per frame, the best 2 codewords by that score of each class of
 * indices mod 8 are candidates, and those within a band of four times the
 * score's error bound (2^-14 |r| |c|) of the best score are re-ranked by their
 * fp32 distance (a fixed summation order), so the code is the exhaustive fp32
 * argmin (up to that order's rounding) unless two codewords of the nearest's
 * class score within that error of it.  Up to D of about 520, CTAs work in
 * pairs (32 frames per pair, every other codeword tile per CTA) that exchange
 * each frame's winner through global memory, in cooperative launches of at
 * most the device's co-resident grid (2432 frames per launch on 152 SMs); a
 * larger D takes one CTA per 16 frames.  Codebooks of 2^24 or more codewords
 * use the CUDA-core form.  The tensor-core form takes about 4 * 8 * Cb * D +
 * 32 * Cb bytes of scratch (plus 1 KB per CTA pair) from the device's
 * stream-ordered pool and frees it on the stream.  Otherwise every distance is
 * computed exactly in fp32 on the CUDA cores.
 * Enqueues and returns; MFS_E_ARG on bad sizes, alignment or NULL pointers;
 * MFS_E_CUDA if the scratch or a launch fails (mfs_last_error(NULL) gives the
 * reason).  A frame whose distances are all NaN gets code 0x7fffffff; on the
 * tensor-core form, if one of the kernel's internal waits gives up (about 2 s:
 * a stalled device), the frames of the groups that saw it get code -1. */
#define MFS_RVQ_MAX_DIM 1024
int mfs_rvq_encode(const float* z_sem, const float* z_ac, int T, int D, const float* codebooks, int Cb,
                   int32_t* codes, void* cuda_stream);

/* ---------------------------------------------------------------- no-alloc
 * Greedy argmax over rows of fp32 logits that allocates no device memory.
 * The pages describe no such call: it exists for callers that cannot call
 * cudaMalloc at the point where they pick tokens, for example code running
 * inside a serving engine whose allocator has already reserved all free
 * device memory (a cudaMalloc there fails or takes memory the engine counts
 * on), or a real-time loop that must not block on the allocator.
 *
 * It is the frame step's argmax stage as a stand-alone kernel: blocks of 4096
 * columns leave partial maxima in scratch memory and the last block of each
 * row reduces them.  That scratch is a fixed static array of
 * MFS_ARGMAX_SCRATCH_BYTES (528 KiB) inside this library, held on every GPU
 * that loads the library until the process exits.
 *
 *   logits  device pointer, row r at logits + r * ld (fp32, read only)
 *   rows    0 .. MFS_ARGMAX_MAX_ROWS; 0 returns MFS_OK and launches nothing
 *   cols    >= 1, with rows * ceil(cols / 4096) <= MFS_ARGMAX_MAX_PARTIALS
 *   ld      row stride in elements, >= cols
 *   out     device pointer to rows int32: the lowest column holding the
 *           row's maximum (NaN never wins; a row of only NaN gives 0), the
 *           same rule as the step's text and code argmax
 *   stream  cudaStream_t (NULL = legacy default stream); the call only
 *           enqueues work and returns without waiting
 * Returns MFS_OK, MFS_E_ARG (bad sizes or NULL pointers), MFS_E_RANGE (sizes
 * beyond the fixed scratch), or MFS_E_CUDA; mfs_last_error(NULL) then gives
 * the reason.  MFS_E_ARG and MFS_E_RANGE are found before anything is
 * enqueued.  MFS_E_CUDA from the launch itself can come after the clear of the
 * row counters (a memset of the scratch) was already enqueued on the stream;
 * the argmax kernel then did not run and `out` is unchanged.
 *
 * The first call on each device looks up the device address of the scratch
 * array (cudaGetSymbolAddress) with that device current: make that first call
 * before any stream capture on the device.  The address is cached per device
 * for the life of the process and is not looked up again: after a
 * cudaDeviceReset of that device the cached address is stale, so do not call
 * this entry point on a device that was reset.  Every call on a device shares the
 * one array; each call first clears the per-row counters that must start at
 * zero.  Calls whose work overlaps on the GPU (other streams, other host
 * threads) race on the array and may return wrong indices: order them on one
 * stream or synchronise between them. */
#define MFS_ARGMAX_MAX_ROWS 4096
#define MFS_ARGMAX_MAX_PARTIALS 65536
#define MFS_ARGMAX_SCRATCH_BYTES (MFS_ARGMAX_MAX_ROWS * 4 + MFS_ARGMAX_MAX_PARTIALS * 8)
int mfs_argmax_rows_noalloc(const float* logits, int rows, int cols, long long ld, int32_t* out,
                            void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* MFS_H */
