/*
 * oracle.h -- plain, sequential CPU restatement of the single-token decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the parity oracle for the CUDA decode
 * library.  Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it; the product path never does.  It shares no code, header, table or helper
 * with the CUDA path.
 *
 * The arithmetic type is `orc_real`, chosen at compile time:
 *   -DORC_REAL=float   (liboracle_f32.so)  the pages' precision: every page computes
 *                                          in f32 ("f32 everywhere", Mimi on wgpu,
 *                                          module doc; Qwen3-TTS talker on wgpu,
 *                                          module doc, "self-contained f32 plan").
 *   -DORC_REAL=double  (liboracle_f64.so)  an f64 shadow of the same code, used only
 *                                          to bound rounding error in the tests.
 * Every product and every sum is rounded separately (built with -ffp-contract=off),
 * dot products run in ascending k, softmax and value sums in ascending key order --
 * the "sequential dot" and "exact ascending-j order" that the talker page names as its
 * CPU reference (Qwen3-TTS talker on wgpu, "Equality standard").
 *
 * Inputs (weights, embeddings, prefilled K/V) are always f32 arrays, or bf16 bit
 * patterns (uint16) for bf16-stored matrices; outputs are returned as double (exact for
 * the f32 build).  The oracle keeps pointers to the caller's weight arrays; they must
 * outlive the model.
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_TALKER = 0, ORC_CODEC = 1 };
#define ORC_INVALID_POS 0xFFFFFFFFu /* Mimi on wgpu, constants: empty pos-ring slot */

typedef struct {
    int kind;          /* ORC_TALKER (Qwen3 talker layer) or ORC_CODEC (windowed ring layer) */
    int layers;
    int hidden;        /* h (talker) or d_model (codec) */
    int q_heads;       /* H */
    int kv_heads;      /* G (codec: == H) */
    int head_dim;      /* d */
    int inter;         /* SwiGLU width (talker) or MLP width (codec) */
    float norm_eps;    /* RMSNorm eps (talker) or LayerNorm eps (codec) */
    double rope_theta; /* 1e6 (talker, rotate_half) or 1e4 (codec, interleaved pairs) */
    int weight_bf16;   /* matrices given as bf16 bit patterns (1) or f32 (0) */
    int max_pos;       /* talker: KV capacity per stream; codec: bound on positions */
    int ring;          /* codec: ring slots per layer */
    int window;        /* codec: attention window */
    int streams;       /* independent decode streams (rows) */
} orc_config;

/* Per-layer weights.  Matrices are row-major [out][in] as a Linear stores them
 * (Qwen3-TTS talker on wgpu, `load`: "row-major [n,k] -- uploaded as-is"). */
typedef struct {
    /* talker */
    const void *wq, *wk, *wv, *wo, *wgate, *wup, *wdown;
    const float *in_norm, *q_norm, *k_norm, *post_norm;
    /* codec */
    const void *in_proj, *out_proj, *lin1, *lin2;
    const float *ln1_w, *ln1_b, *ln2_w, *ln2_b, *ls1, *ls2;
} orc_layer;

typedef struct orc_model orc_model;

/* ---- primitives (exported so the tests can pin each one on its own) ---- */

/* exact bf16 -> f32 widening of one bit pattern */
float orc_bf16_to_f32(uint16_t bits);
/* y[n] = sum_k W[n,k] x[k], ascending k; W f32 [N][K] */
void orc_matvec_f32(const float* W, int N, int K, const double* x, double* y);
/* same with W given as bf16 bit patterns [N][K] */
void orc_matvec_bf16(const uint16_t* W, int N, int K, const double* x, double* y);
/* MV_BIAS: y[n] = b[n] + W[n,k] x[k] accumulated from the bias in ascending k; act == 1 applies
 * SiLU to the result; W f32 [N][K] */
void orc_matvec_bias(const float* W, int N, int K, const double* x, const float* b, int act,
                     double* y);
/* y = x / sqrt(mean(x^2) + eps) * w */
void orc_rms_norm(const double* x, const float* w, int n, double eps, double* y);
/* y = (x - mean) / sqrt(var + eps) * w + b, var biased */
void orc_layer_norm(const double* x, const float* w, const float* b, int n, double eps, double* y);
/* cos/sin of pos * theta^(-2i/d) for i in [0, d/2), computed in double, rounded to orc_real */
void orc_rope_table(int d, double theta, int pos, double* cos_out, double* sin_out);
/* multimodal rope: frequency i is driven by position pos3[assign[i]] (assign[i] in 0..2) */
void orc_mrope_table(int d, double theta, const int* pos3, const int* assign, double* cos_out,
                     double* sin_out);
/* HF rotate_half rope in place on one head of width d */
void orc_rope_rotate_half(double* x, int d, const double* c, const double* s);
/* interleaved-pair rope in place on one head of width d */
void orc_rope_interleaved(double* x, int d, const double* c, const double* s);
/* silu(g) = g / (1 + exp(-g)) */
double orc_silu(double g);
/* gelu(v) = 0.5 v (1 + erf(v / sqrt 2)) */
double orc_gelu(double v);
/* causal GQA attention of H query heads over L cached keys.
 * q [H][d]; kc, vc position-major [L][G][d]; out [H][d]; kv head of q head i is i/(H/G) */
void orc_gqa_attention(const double* q, const double* kc, const double* vc, int L, int H, int G,
                       int d, double* out);
/* windowed attention over a ring of `ring` slots with position stamps pr[ring];
 * q [H][d]; kr, vr slot-major [ring][H][d] (MHA); out [H][d] */
void orc_ring_attention(const double* q, const double* kr, const double* vr, const uint32_t* pr,
                        int ring, int window, uint32_t pos, int H, int d, double* out);

/* ---- the decode stack ---- */

orc_model* orc_create(const orc_config* cfg, const orc_layer* layers, const float* final_norm);
/* copy prefilled K/V of one stream: k, v are [layers][n_pos][kv_heads][head_dim] f32, keys
 * already carrying rope.  Talker: rows 0..n_pos; codec: ring slots 0..n_pos stamped 0..n_pos. */
int orc_prefill_kv(orc_model* m, int stream, const float* k, const float* v, int n_pos);
/* one decode step of streams 0..rows-1 at positions pos[i] (must equal the stream length).
 * x_in [rows][hidden] f32; out [rows][hidden]; taps (nullable) [layers][rows][hidden] =
 * the residual stream after each layer.  Returns 0 or a negative error code. */
int orc_step(orc_model* m, int rows, const float* x_in, const int* pos, double* out, double* taps);

/* Talker multimodal rope (Qwen3-TTS talker on wgpu, module notes: "interleaved MRoPE"; uniform
 * positions reduce it to the 1-D rope).  assign [head_dim/2]: the axis (0 t, 1 h, 2 w) whose
 * position turns rope frequency i; NULL restores the 1-D rope.  Returns 0, or -1 (codec, an
 * entry outside 0..2). */
int orc_set_mrope(orc_model* m, const int* assign);
/* orc_step with per-axis rotary positions pos3 [rows][3] (each in 0..max_pos-1; NULL: the 1-D
 * rope at pos).  The K/V row still goes to cache row pos[i].  -4 for a codec model. */
int orc_step_mrope(orc_model* m, int rows, const float* x_in, const int* pos, const int* pos3,
                   double* out, double* taps);

/* Codec only: the FlowLM backbone's head (Pocket TTS on wgpu, PocketBackboneGpu): after the
 * stack, out = LayerNorm(x; norm_w, norm_b) is the step's output instead of x, and with eos_w
 * the EOS logit eos_w . out (ascending sum; its bias is added by the caller, as the page does on
 * read-back) is kept per stream for orc_eos.  A codec layer with ls1 / ls2 NULL has no
 * LayerScale.  Returns 0, or -1 on a bad argument. */
int orc_set_head(orc_model* m, const float* norm_w, const float* norm_b, const float* eos_w);
double orc_eos(const orc_model* m, int stream);

/* Causal prefill of n rows of one stream (Qwen3-TTS talker on wgpu, prefill(): the block is
 * appended at positions len .. len+n-1 and every position's final-norm hidden is returned).
 * Its plain definition is the autoregressive one: row r is one talker step of `stream` at
 * position len + r, which attends to keys 0 .. len + r -- exactly the keys a batched block with
 * a causal mask gives row r.  x_in [n][hidden], out [n][hidden].  Talker only.
 * Returns 0, or < 0 on a bad argument or capacity. */
int orc_prefill(orc_model* m, int stream, int n, const float* x_in, double* out);
/* orc_prefill with per-axis rotary positions pos3 [n][3] for the rows (NULL: 1-D rope). */
int orc_prefill_mrope(orc_model* m, int stream, int n, const float* x_in, const int* pos3,
                      double* out);
void orc_reset(orc_model* m, int stream);

/* ---- the flow head (Pocket TTS on wgpu, PocketFlowGpu: SimpleMLPAdaLN, one LSD step) ---- */
typedef struct {
    int dim, latent, cond, blocks;
    double ln_eps;
    const float *ip_w, *ip_b;       /* input_proj [dim][latent], [dim] */
    const float *cond_w, *cond_b;   /* cond embedding [dim][cond], [dim] */
    const float* t_const;           /* the constant timestep embedding [dim] */
    const float* const* ada_w;      /* per block: adaLN projection [3 dim][dim] = shift|scale|gate */
    const float* const* ada_b;      /* [3 dim] */
    const float* const* ln_w;       /* per block in_ln [dim] */
    const float* const* ln_b;
    const float* const* m0_w;       /* per block [dim][dim], [dim] (through SiLU) */
    const float* const* m0_b;
    const float* const* m2_w;
    const float* const* m2_b;
    const float *fada_w, *fada_b;   /* final adaLN [2 dim][dim] = shift|scale, [2 dim] */
    const float *f_w, *f_b;         /* final linear [latent][dim], [latent] */
} orc_flow;
/* One LSD step (steps = 1) from `noise` [latent], conditioned on `cond` [cond]:
 *   x = W_ip noise + b_ip;  y = silu(t_const + W_c cond + b_c)
 *   per block: (shift, scale, gate) = W_ada y + b_ada; u = LN(x; w, b) (1 + scale) + shift;
 *              x += gate * (W_2 silu(W_0 u + b_0) + b_2)
 *   final: (shift, scale) = W_fada y + b_fada; u = LN(x; 1, 0) (1 + scale) + shift;
 *   out = noise + (W_f u + b_f) / 1.
 * Returns 0, or -1 on a bad argument. */
int orc_flow_step(const orc_flow* f, const float* cond, const float* noise, double* out);
int orc_len(const orc_model* m, int stream);
/* read the stored key/value of (layer, stream, position) as [kv_heads][head_dim] */
int orc_read_kv(const orc_model* m, int layer, int stream, int pos, double* k, double* v);
void orc_destroy(orc_model* m);

/* threads used by the row-parallel matvec (results are bitwise independent of it) */
void orc_set_threads(int n);
int orc_get_threads(void);
/* sizeof(orc_real): 4 or 8 */
int orc_real_size(void);

#ifdef __cplusplus
}
#endif
#endif
