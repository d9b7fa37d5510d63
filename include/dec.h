/*
 * dec.h -- C ABI of the GB300 (sm_103a) single-token autoregressive decode library.
 *
 * One call of dec_step advances m independent decode streams by one position through a
 * stack of transformer layers of one of two kinds:
 *
 *   DEC_QWEN3_TALKER   the Qwen3-style TTS talker layer (Qwen3-TTS talker on wgpu,
 *                      inferencelayer qwen3tts_gpu.rs, build_step_plan): RMSNorm, q/k/v
 *                      row-major GEMVs, per-head q/k RMSNorm, 1-D rotate_half RoPE (or its
 *                      multimodal form, dec_step_mrope), KV append, causal GQA attention over
 *                      the whole cache, o-proj + residual, RMSNorm, gate/up GEMVs + SwiGLU,
 *                      down-proj + residual; final RMSNorm.
 *   DEC_CODEC_WINDOWED the codec-style layer over a KV ring (Mimi on wgpu, inferencelayer
 *                      mimi_gpu.rs, transformer_shaped): LayerNorm, qkv GEMV, interleaved
 *                      RoPE + ring push + position stamp, windowed attention, out-proj with
 *                      LayerScale residual, LayerNorm, lin1 + GELU(erf), lin2 with LayerScale
 *                      residual; the output is the residual stream (no final norm), or with
 *                      the FlowLM head (Pocket TTS on wgpu) its final LayerNorm and EOS logit.
 *
 * Beside the step: batched causal prefill of talker blocks (dec_prefill), the flow head
 * (dec_flow_*), and stateless GEMV / attention entry points.
 *
 * Every step of the path runs in this library's CUDA kernels.  Pointers are plain host or
 * device addresses as stated per argument; `void* stream` is a cudaStream_t (0 = legacy
 * default stream).  Sizes are in elements unless they say bytes.  All functions return a
 * dec_status; on failure dec_last_error(ctx) holds a one-line reason and the context's
 * state is unchanged, except for DEC_E_CUDA / DEC_E_DEVICE_CHECK, after which the context
 * should be destroyed.  A context is not thread-safe: one host thread at a time.
 */
#ifndef DEC_H
#define DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DEC_ABI_VERSION 1

typedef enum {
    DEC_OK = 0,
    DEC_E_ARG = 1,          /* null pointer, out-of-range size, inconsistent configuration */
    DEC_E_POS = 2,          /* pos[i] differs from the current length of stream i */
    DEC_E_CAPACITY = 3,     /* a position would reach max_pos, or a prefill exceeds capacity */
    DEC_E_UNSUPPORTED = 4,  /* a shape or dtype outside what the kernels implement */
    DEC_E_CUDA = 5,         /* a CUDA runtime call failed (text in dec_last_error) */
    DEC_E_DEVICE_CHECK = 6  /* a kernel's own bounds or wait-limit check fired */
} dec_status;

typedef enum { DEC_QWEN3_TALKER = 0, DEC_CODEC_WINDOWED = 1 } dec_kind;
typedef enum { DEC_F32 = 0, DEC_BF16 = 1 } dec_dtype;

/* flags */
#define DEC_FLAG_TAPS 1u     /* keep the residual stream after every layer (dec_read_tap) */
#define DEC_FLAG_NO_GRAPH 2u /* launch kernels one by one instead of replaying a CUDA graph */
#define DEC_FLAG_PERSISTENT 4u /* steps of m <= 2 rows run as one persistent cooperative kernel
                                  (the streamed step: every SM streams its share of the weights
                                  and K/V through a shared-memory ring while its consumer warps
                                  wait on tagged activations) instead of the chain of kernels;
                                  results agree within floating-point rounding */
#define DEC_FLAG_TENSOR_GEMV 8u /* GEMVs of 3..8 rows over bf16 weights (steps of 3..8 streams,
                                   prefill blocks) run on the tensor cores: tcgen05.mma with
                                   TMEM accumulators, weight tiles by TMA, x split into three
                                   bf16 terms (f32 accuracy); otherwise the FMA kernels serve
                                   them.  Results agree within floating-point rounding.  On the
                                   28-layer 2048-wide shapes it measured slower than the FMA
                                   kernels, which stay the default */

/*
 * Model geometry.  Talker fields follow the talker's Dims (Qwen3-TTS talker on wgpu, `Dims`
 * and load()); codec fields follow TrShape (Mimi on wgpu, `TrShape`).
 *   hidden      h (talker) or d_model (codec); multiple of 8
 *   q_heads     H; kv_heads G; H % G == 0 (codec: G == H and H * head_dim == hidden)
 *   head_dim    d: 64 or 128 (the talker page bounds it by 128, load())
 *   inter       SwiGLU width (talker) or MLP width (codec); multiple of 8
 *   norm_eps    RMSNorm eps (talker, 1e-6) or LayerNorm eps (codec, 1e-5)
 *   rope_theta  RoPE base: 1e6 (talker, rotate_half), 1e4 (codec, interleaved pairs)
 *   weight_dtype storage type of every matrix: DEC_F32 or DEC_BF16 (widened to f32 exactly
 *               in-kernel); norm weights, biases and LayerScale vectors are always f32
 *   max_pos     talker: KV capacity per stream (a step at pos needs pos + 1 <= max_pos);
 *               codec: positions must stay below max_pos (length of the RoPE table)
 *   ring        codec: KV ring slots per layer and stream; window: attention window,
 *               1 <= window <= ring (window == ring means unbounded within the ring)
 *   max_streams number of decode streams (rows) the context holds state for: 1..8
 */
typedef struct {
    int32_t kind;          /* dec_kind */
    int32_t layers;
    int32_t hidden;
    int32_t q_heads;
    int32_t kv_heads;
    int32_t head_dim;
    int32_t inter;
    float norm_eps;
    double rope_theta;
    int32_t weight_dtype;  /* dec_dtype */
    int32_t max_pos;
    int32_t ring;
    int32_t window;
    int32_t max_streams;
    uint32_t flags;        /* DEC_FLAG_* */
} dec_config;

/*
 * Per-layer weights: DEVICE pointers, read only during dec_create (the library copies them
 * into its own arena, so the caller may free them afterwards).  Matrices are row-major
 * [out][in], exactly as a Linear stores them and as the talker page uploads them
 * (Qwen3-TTS talker on wgpu, load(): "row-major [n,k] -- uploaded as-is"), 16-byte aligned.
 * Talker: q [H*d][h], k [G*d][h], v [G*d][h], o [h][H*d], gate [inter][h], up [inter][h],
 *         down [h][inter]; in_norm [h], q_norm [d], k_norm [d], post_norm [h] (f32).
 * Codec:  in_proj [3*hidden][hidden] with rows [q | k | v], each head-major; out_proj
 *         [hidden][hidden]; lin1 [inter][hidden]; lin2 [hidden][inter]; ln1_w, ln1_b,
 *         ln2_w, ln2_b, ls1, ls2 [hidden] (f32); ls1 / ls2 may be NULL (no LayerScale, as in
 *         the FlowLM backbone).  Fields of the other kind are ignored.
 */
typedef struct {
    const void *q, *k, *v, *o, *gate, *up, *down;
    const float *in_norm, *q_norm, *k_norm, *post_norm;
    const void *in_proj, *out_proj, *lin1, *lin2;
    const float *ln1_w, *ln1_b, *ln2_w, *ln2_b, *ls1, *ls2;
} dec_layer_weights;

typedef struct {
    const dec_layer_weights* layers; /* HOST array of `layers` entries */
    const float* final_norm;         /* talker: the final RMSNorm weight, DEVICE [h] f32.
                                        codec: NULL (the output is the residual stream, as in
                                        Mimi) or the FlowLM backbone's out_norm LayerNorm weight */
    const float* final_norm_b;       /* codec with final_norm: out_norm bias, DEVICE [h] f32 */
    const float* eos_w;              /* codec, optional: the EOS row, DEVICE [h] f32; each step
                                        then computes eos_w . output (Pocket TTS on wgpu,
                                        PocketBackboneGpu: out_eos) */
    float eos_b;                     /* the EOS bias, added when the logits are read */
} dec_weights;

typedef struct dec_ctx dec_ctx;

/* Create a context on the current CUDA device: validates the configuration, allocates the
 * weight arena, KV caches (talker: [layers][streams][G][max_pos][d] f32; codec: rings
 * [layers][streams][H][ring][d] f32 plus u32 position rings, all stamped empty), RoPE
 * tables and scratch, and copies the weights.  The talker page's load() sizes the same
 * state (Qwen3-TTS talker on wgpu, load() and new_state()).  `stream` is where every later
 * step is enqueued.  On success *out owns all of it until dec_destroy. */
dec_status dec_create(const dec_config* cfg, const dec_weights* w, void* stream, dec_ctx** out);

/* Free everything the context owns.  Waits for the context's stream first.  NULL is a no-op. */
void dec_destroy(dec_ctx* ctx);

/* One-line text of the last failure on this context (empty string if none).  With ctx ==
 * NULL, the last failure of dec_create on this thread. */
const char* dec_last_error(const dec_ctx* ctx);

/* Replace the stream later calls enqueue on. */
dec_status dec_set_stream(dec_ctx* ctx, void* stream);

/* Load a stream's cache from prefilled keys and values, as the backbone's voice load does
 * (Pocket TTS on wgpu, load_voice(): the stored keys already carry RoPE, so it is a copy).
 * k, v: DEVICE [layers][n_pos][kv_heads][head_dim] f32.  The stream is reset first; then
 * talker: cache rows 0..n_pos-1; codec: ring slots 0..n_pos-1 stamped with positions
 * 0..n_pos-1 (n_pos <= ring).  The stream's length becomes n_pos.  Asynchronous on the
 * context's stream; k and v must stay valid until it has run.
 * Errors: DEC_E_ARG (stream out of range, n_pos < 0, null with n_pos > 0), DEC_E_CAPACITY
 * (n_pos > max_pos for the talker, n_pos > ring for the codec). */
dec_status dec_prefill_kv(dec_ctx* ctx, int stream, const float* k, const float* v, int n_pos);

/* Batched causal prefill (Qwen3-TTS talker on wgpu, prefill() / forward_rows()): append the n
 * rows of x to stream `stream` at positions len .. len + n - 1 and return every position's
 * final-norm hidden.  Row r attends to keys 0 .. len + r: the block's own K/V rows are appended
 * before its attention, so the block is causal within itself, and the result equals n single
 * steps up to the order of floating-point sums.  Talker only.
 *   x    DEVICE [n][hidden] f32 (16-byte aligned)
 *   out  DEVICE [n][hidden] f32, must not overlap x
 * Asynchronous on the context's stream; runs in blocks of up to 8 rows (each weight matrix is
 * read once per block), launched directly (no graph).  The stream's length advances by n.
 * Errors: DEC_E_ARG (stream, n < 1, NULL), DEC_E_UNSUPPORTED (codec: a KV ring takes one position
 * per step), DEC_E_CAPACITY (len + n > max_pos); the state is unchanged on these. */
dec_status dec_prefill(dec_ctx* ctx, int stream, int n, const float* x, float* out);

/* Rows per dec_prefill block (each block reads every weight matrix once); 0 when the context
 * does not serve prefill (codec) or ctx is NULL. */
int dec_prefill_block_rows(const dec_ctx* ctx);

/* One decode step of streams 0..m-1 (Qwen3-TTS talker on wgpu, step(): the new K/V row is
 * appended at `pos`, attention covers pos + 1 keys, the final-norm hidden is returned;
 * Pocket TTS on wgpu, step_device(): the output stays on the device).
 *   m           rows = streams 0..m-1, 1 <= m <= max_streams
 *   x_in        DEVICE [m][hidden] f32, the input embeddings
 *   pos         HOST [m]; pos[i] must equal stream i's current length (contiguous
 *               positions, as step() demands) and pos[i] + 1 <= max_pos (talker) or
 *               pos[i] < max_pos (codec)
 *   hidden_out  DEVICE [m][hidden] f32: talker final-norm hidden, codec residual stream;
 *               must not overlap x_in
 * Asynchronous: enqueued on the context's stream, returns without waiting; x_in must not
 * change and hidden_out must not be read until the stream reaches this point.  The first
 * step of a given m captures a CUDA graph (milliseconds); later steps replay it, with new
 * x_in / hidden_out pointers written into the graph's nodes that take them (up to 8 graphs
 * are kept).  Lengths advance by one on success; nothing changes on
 * an error. */
dec_status dec_step(dec_ctx* ctx, int m, const float* x_in, const int32_t* pos, float* hidden_out);

/* Multimodal rope of the talker (Qwen3-TTS talker on wgpu, module notes: the talker's rope is
 * interleaved MRoPE; with equal positions on its three axes it is the 1-D rope the tables hold).
 * axis_host HOST [n], n = head_dim / 2: the axis (0 t, 1 h, 2 w) whose rotary position turns
 * rope frequency i; the pages give no section split, so the caller supplies the map (an
 * interleaved split puts h on i = 1, 4, 7, ... and w on i = 2, 5, 8, ... up to their sections).
 * NULL sets every frequency to axis t.  The map is used only by the steps and prefills given
 * per-axis rotary positions (dec_step_mrope, dec_prefill_mrope).  Synchronous (waits for the
 * context's stream).  Errors: DEC_E_ARG (n, an entry outside 0..2), DEC_E_UNSUPPORTED (codec). */
dec_status dec_set_mrope(dec_ctx* ctx, const int32_t* axis_host, int n);

/* dec_step with per-axis rotary positions (talker).
 *   rope_pos  DEVICE [m][3] int32 (4-byte aligned): row i's t, h, w rotary positions, each in
 *             0..max_pos-1; NULL is dec_step.  The K/V row still goes to cache row pos[i].
 * The buffer is read when the step runs (like x_in), so it may be rewritten between steps; its
 * pointer is part of the captured graph's key.  Steps with rope_pos always run the multi-kernel
 * plan (6 * layers + 1 kernels, also with DEC_FLAG_PERSISTENT).  A position outside 0..max_pos-1
 * leaves that row's attention undone and is reported as DEC_E_DEVICE_CHECK by the next dec_sync.
 * Errors as dec_step, plus DEC_E_ARG (alignment) and DEC_E_UNSUPPORTED (codec with rope_pos). */
dec_status dec_step_mrope(dec_ctx* ctx, int m, const float* x_in, const int32_t* pos,
                          const int32_t* rope_pos, float* hidden_out);

/* dec_prefill with per-axis rotary positions: rope_pos DEVICE [n][3] int32, row r's t, h, w
 * positions (NULL is dec_prefill); the rows still go to cache rows len .. len + n - 1. */
dec_status dec_prefill_mrope(dec_ctx* ctx, int stream, int n, const float* x,
                             const int32_t* rope_pos, float* out);

/* dec_step with HOST buffers, blocking, as the talker page's step() returns its hidden state
 * to the host (Qwen3-TTS talker on wgpu, step(): write_buffer, submit, blocking read).
 * x_in_host [m][hidden] and hidden_out_host [m][hidden] f32 in host memory (pinned or not);
 * copies in, runs the step, copies out and waits.  Also reports device-side check failures
 * (DEC_E_DEVICE_CHECK) like dec_sync. */
dec_status dec_step_host(dec_ctx* ctx, int m, const float* x_in_host, const int32_t* pos,
                         float* hidden_out_host);

/* Clear one stream: length 0, its K/V zeroed, and (codec) every position stamp set to
 * empty by ring capacity (Mimi on wgpu, reset(); Pocket TTS on wgpu, reset()).
 * Asynchronous on the context's stream. */
dec_status dec_reset(dec_ctx* ctx, int stream);

/* Wait for the context's stream, then read the kernels' device check word: DEC_OK, or
 * DEC_E_DEVICE_CHECK naming the check (bounds or wait limit), or DEC_E_CUDA. */
dec_status dec_sync(dec_ctx* ctx);

/* Current length (next position) of a stream as the host sees it, or -1 on a bad index. */
int dec_get_len(const dec_ctx* ctx, int stream);

/* Copy the stored key and value of (layer, stream, position) to HOST [kv_heads][head_dim]
 * f32 each (codec: the slot position % ring).  Synchronous.  For tests and inspection. */
dec_status dec_read_kv(dec_ctx* ctx, int layer, int stream, int position, float* k_host,
                       float* v_host);

/* With DEC_FLAG_TAPS: copy the residual stream after `layer` of the last step to HOST
 * [m][hidden] f32 (the pages' stage probes, Mimi on wgpu, debug_read()).  Synchronous. */
dec_status dec_read_tap(dec_ctx* ctx, int layer, int m, float* dst_host);

/* With eos_w: the EOS logits of the last step of streams 0..m-1, bias added, into HOST [m]
 * (waits for the context's stream).  Errors: DEC_E_ARG, DEC_E_UNSUPPORTED (no EOS row). */
dec_status dec_read_eos(dec_ctx* ctx, int m, float* dst_host);

/* Number of CUDA kernels one step of m rows launches (for launch accounting): 6 * layers + 1,
 * or 1 when the persistent kernel serves the step (DEC_FLAG_PERSISTENT, m <= 2). */
int dec_kernels_per_step(const dec_ctx* ctx, int m);

/* Failure-path check of the persistent kernel's bounded waits (no counterpart on the pages).
 * The NEXT step of m <= 2 rows that the persistent kernel serves runs once outside the CUDA graph
 * with the consumers of phase `phase` (0 .. 5 * layers; per layer: q/k/v, attention with the
 * merge of its partials, o-proj, gate/up, down; then the output rows) waiting for activation
 * tags that no CTA writes,
 * and with every wait of that step bounded by `polls` loads (>= 1; about a microsecond each;
 * too small a bound also cuts the step's ordinary waits short).  The wait runs out, the
 * kernel flags its check word and every CTA leaves early after its copies in flight have landed:
 * nothing faults or hangs.  That step's output and its cache rows are undefined; the next
 * dec_sync returns DEC_E_DEVICE_CHECK (wait limit) and clears the check word.  The stream length
 * still advances, so a caller rewinds with dec_truncate (talker) before stepping on.  Phases
 * that wait on no activation (layer 0's q/k/v reads the step input) do not run out.
 * Errors: DEC_E_ARG (phase or polls out of range), DEC_E_UNSUPPORTED (no persistent plan). */
dec_status dec_inject_stall(dec_ctx* ctx, int phase, int polls);

/* Talker only: shorten stream `stream` to `new_len` positions (0 <= new_len <= its length), so
 * the next step is at position new_len.  Cache rows below new_len are kept (rows at and above
 * it are overwritten by later steps), e.g. to roll back rejected positions or to replay a fixed
 * position range.  Asynchronous.  Errors: DEC_E_ARG (range), DEC_E_UNSUPPORTED (codec ring:
 * its slots are reused, so earlier positions cannot be restored). */
dec_status dec_truncate(dec_ctx* ctx, int stream, int new_len);

/* Enqueue one stage of the step plan for rows 0..m-1, on the context's stream, from the
 * context's current buffers -- for timing a kernel on its own (the per-kernel attribution of
 * the pages' bench_steps, Mimi on wgpu).  chained != 0 launches the stage as a programmatic
 * dependent of the previous kernel on the stream, as inside a step; 0 launches it alone.
 * stage: 0 norm + q/k/v GEMV, 1 attention (with its
 * prologue; two kernels: the split-K chunks, then the merge of their partials), 2 o-proj +
 * residual, 3 norm + gate/up + SwiGLU (codec: lin1 + GELU), 4 down + residual (codec: lin2);
 * every stage but 1 is exactly one kernel.  Layer 0's stages 0 and 2 read the context's internal input buffer.
 * Lengths do not advance; stage 1 writes the K/V row (ring slot) of the next position, which
 * the next step rewrites.  Not for use between a dec_step and its completion. */
dec_status dec_launch_stage(dec_ctx* ctx, int layer, int stage, int m, int chained);

/* ---------------------------------------------------------------------------------------
 * The flow head (Pocket TTS on wgpu, PocketFlowGpu: SimpleMLPAdaLN, one LSD step), reading
 * the backbone's hidden state in place on the device.  One call:
 *   x = W_ip noise + b_ip;  y = silu(t_const + W_c cond + b_c)
 *   per block: (shift, scale, gate) = W_ada y + b_ada;
 *              x += gate * (W_2 silu(W_0 (LN(x; ln_w, ln_b) (1 + scale) + shift) + b_0) + b_2)
 *   final:     (shift, scale) = W_fada y + b_fada;
 *              latent = noise + W_f (LN(x; 1, 0) (1 + scale) + shift) + b_f
 * All weights f32, row-major [out][in], 16-byte aligned DEVICE pointers; the per-block fields
 * are HOST arrays of `blocks` DEVICE pointers.  dec_flow_create copies them.
 * ------------------------------------------------------------------------------------- */
typedef struct {
    int dim;        /* the head's width (multiple of 8) */
    int latent;     /* latent / noise width (multiple of 8) */
    int cond;       /* conditioning width: the backbone's hidden (multiple of 8) */
    int blocks;     /* residual blocks (>= 0) */
    float ln_eps;   /* LayerNorm eps (1e-6 on the page) */
    int lsd_steps;  /* must be 1: the page plans one LSD step */
} dec_flow_config;

typedef struct {
    const float *ip_w, *ip_b;        /* input_proj [dim][latent], [dim] */
    const float *cond_w, *cond_b;    /* cond embedding [dim][cond], [dim] */
    const float* t_const;            /* constant timestep embedding [dim] */
    const float* const* ada_w;       /* [blocks] of [3 dim][dim]: shift | scale | gate rows */
    const float* const* ada_b;       /* [blocks] of [3 dim] */
    const float* const* ln_w;        /* [blocks] of [dim] */
    const float* const* ln_b;
    const float* const* m0_w;        /* [blocks] of [dim][dim] (SiLU after) */
    const float* const* m0_b;
    const float* const* m2_w;        /* [blocks] of [dim][dim] */
    const float* const* m2_b;
    const float *fada_w, *fada_b;    /* final adaLN [2 dim][dim] (shift | scale), [2 dim] */
    const float *f_w, *f_b;          /* final linear [latent][dim], [latent] */
} dec_flow_weights;

typedef struct dec_flow dec_flow;

/* Errors: DEC_E_ARG (NULL, bad sizes), DEC_E_UNSUPPORTED (lsd_steps != 1, widths not multiples
 * of 8), DEC_E_CUDA.  On failure *out is NULL and dec_flow_last_error(NULL) tells why. */
dec_status dec_flow_create(const dec_flow_config* cfg, const dec_flow_weights* w, void* stream,
                           dec_flow** out);
/* One LSD step on the head's stream: cond DEVICE [cond] (e.g. a dec_step hidden_out row, read
 * in place), noise DEVICE [latent], latent_out DEVICE [latent] (may not overlap noise).
 * Asynchronous; captured as a CUDA graph per (cond, noise, latent_out) and replayed. */
dec_status dec_flow_step(dec_flow* f, const float* cond, const float* noise, float* latent_out);
void dec_flow_destroy(dec_flow* f);
const char* dec_flow_last_error(const dec_flow* f);
int dec_flow_kernels_per_step(const dec_flow* f);

/* ---------------------------------------------------------------------------------------
 * Stateless kernel entry points (the same kernels the step uses, on caller buffers).
 * ------------------------------------------------------------------------------------- */

/* Row-major GEMV (Qwen3-TTS talker on wgpu, MATVEC_SRC): y[r][n] = sum_k W[n][k] x[r][k]
 * for r < m, each weight read once for all m rows.
 *   dtype  DEC_F32 or DEC_BF16 (W as bf16 bit patterns, widened exactly)
 *   W      DEVICE [N][K], 16-byte aligned, K % 8 == 0
 *   x      DEVICE [m][K] f32, 16-byte aligned;  y: DEVICE [m][N] f32;  1 <= m <= 8
 * Asynchronous on `stream`.  Errors: DEC_E_ARG, DEC_E_UNSUPPORTED (K % 8, alignment). */
dec_status dec_gemv(int dtype, const void* W, int N, int K, const float* x, int m, float* y,
                    void* stream);

/* Split-K GQA decode attention (Qwen3-TTS talker on wgpu, GQA_ATTN_SRC), one query row per
 * stream: out[r][i] = sum_j softmax_j(q[r][i] . K[r][g][j] / sqrt(d)) V[r][g][j] over
 * j < lens[r], with g = i / (H / G).
 *   q      DEVICE [m][H][d] f32 (already normalised and rotated)
 *   k, v   DEVICE [m][G][capacity][d] f32, head-major caches, 16-byte aligned
 *   lens   DEVICE [m] int32, 1 <= lens[r] <= capacity
 *   out    DEVICE [m][H][d] f32
 *   workspace  DEVICE scratch of dec_attention_workspace_bytes(...) bytes, 16-byte
 *          aligned, used for per-chunk partial results and merge tickets; its ticket words
 *          must be zero before the first call (cudaMemset) -- every call leaves them zero
 *          again.  Calls sharing one workspace must not overlap on the GPU.
 * Asynchronous on `stream`.  head_dim 64 or 128, H / G <= 8, m <= 64. */
size_t dec_attention_workspace_bytes(int m, int q_heads, int kv_heads, int head_dim,
                                     int capacity);
dec_status dec_attention(int m, int q_heads, int kv_heads, int head_dim, int capacity,
                         const float* q, const float* k, const float* v, const int32_t* lens,
                         float* out, void* workspace, size_t workspace_bytes, void* stream);

/* dec_attention without any allocation (no counterpart on the pages: a service of this library).
 * Some callers cannot allocate device memory: code on a real-time audio thread, where
 * cudaMalloc/cudaFree may synchronize the device and take unbounded time, and code inside a host
 * application whose own allocator owns the device-memory budget.  This entry computes exactly
 * what dec_attention computes, with the same arguments minus the workspace: its scratch is a
 * static device array of 4 MiB (4194304 bytes) that the library holds on every GPU it is
 * loaded on until the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *   Limit: the scratch dec_attention_workspace_bytes(m, q_heads, kv_heads, head_dim, capacity)
 *   reports must fit in the 4 MiB.  Example: m = 1, 16 q heads, 8 kv heads, d = 128 takes
 *   capacity up to 32256 (504 chunks of 64 keys: 4128768 bytes of partial outputs, 64512 of
 *   partial maxima and sums, 256 of merge tickets); capacity 32257 needs a 505th chunk and is
 *   rejected.  Larger requests return DEC_E_UNSUPPORTED (text in dec_last_error(NULL)).
 *   When the array is reserved: with the default lazy loading of CUDA modules, the library's
 *   module, and with it the array, is loaded on a device at the first call of this entry (or of
 *   any other entry point) on that device; that first call also looks up the array's device
 *   address.  Make that first call outside any stream capture, and early if the reservation of
 *   4 MiB must not happen on a time-critical path.
 *   Every call on a device shares the one array: calls that overlap on the GPU (other streams,
 *   other host threads) race and corrupt each other's results.  Each call clears the words that
 *   must start at zero before its kernel runs.
 *   lens[r] outside 1..capacity is not reported by this entry (it has no status word the caller
 *   could read): the rows of such a stream are left unwritten, so out[r] is undefined.
 * Asynchronous on `stream`; same layouts, limits and errors as dec_attention otherwise. */
dec_status dec_attention_noalloc(int m, int q_heads, int kv_heads, int head_dim, int capacity,
                                 const float* q, const float* k, const float* v,
                                 const int32_t* lens, float* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DEC_H */
