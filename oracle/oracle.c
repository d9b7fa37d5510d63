/*
 * oracle.c -- plain sequential CPU restatement of the decode step (TEST INFRASTRUCTURE).
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load this
 * library.  It is written from the pages' kernel descriptions, step by step, in their
 * order and notation, with no blocking, fusion or reordering:
 *
 *   Qwen3-TTS talker on wgpu (inferencelayer qwen3tts_gpu.rs):
 *     MATVEC_SRC      y[m,n] = x[m,k] W[n,k]^T, W row-major, no bias
 *     RMSNORM_SRC     y = x / sqrt(mean(x^2) + eps) * w
 *     QK_NORM_SRC     the same per head, weight [hd] shared by all heads
 *     ROPE_SRC        HF rotate_half rope from cos/sin tables at the row's position
 *     GQA_ATTN_SRC    causal GQA attention, kv head = head / group, scale 1/sqrt(hd),
 *                     single-pass softmax and value sum in ascending key order
 *     SWIGLU_SRC      silu(g) * u, silu(g) = g / (1 + exp(-g))
 *     APPEND_SRC      new K/V row written at the current length
 *     build_step_plan the layer order: rmsnorm, q/k/v, qk-norm, rope, append, attention,
 *                     o-proj + residual add, rmsnorm, gate/up, swiglu, down + residual add;
 *                     final rmsnorm
 *   Mimi on wgpu (inferencelayer mimi_gpu.rs):
 *     ln_src / LN512  LayerNorm: mean, biased variance of deviations, affine
 *     rope_push_src   interleaved-pair rope, K/V pushed into slot pos % ring, slot stamped
 *     attn_src        a key is legal iff stamp != INVALID, stamp <= pos, pos - stamp < window;
 *                     max, exp-sum, (sum e_j v_j) / den
 *     MV_LS           y += ls[n] * (W x)[n]
 *     GELU_ERF        0.5 v (1 + erf(v / sqrt 2)) -- here with the C library's erf
 *     transformer_shaped  the layer order: LN, qkv, rope+push, attention, out-proj + LS,
 *                     LN, lin1, GELU, lin2 + LS; the output is the residual stream
 *
 * Readings where the pages are silent (each is listed with its reason in the design notes):
 *   - multimodal rope (the talker's "interleaved MRoPE"): frequency i of the rotate_half table
 *     turns by the position of one of three axes (t, h, w), named by a per-frequency axis map
 *     the caller supplies (the pages give no section split); equal positions on all axes give
 *     the 1-D table (the pages' MRoPE-uniform identity).  The arithmetic for any map is pinned;
 *     which split the real model uses is parity unpinned
 *   - rope tables: angle pos * theta^(-2i/d), cos/sin computed in double, rounded to orc_real
 *     (the talker's table builder is not printed; the codec computes the same angle in-kernel)
 *   - codec rope base 10000 (the value in rope_push_src)
 *   - codec q/k/v split [q | k | v], each head-major, as rope_push_src indexes it
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <tgmath.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORC_REAL
#define ORC_REAL float
#endif
typedef ORC_REAL real;

int orc_real_size(void) { return (int)sizeof(real); }

static int g_threads = 1;
void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int orc_get_threads(void) { return g_threads; }

/* ------------------------------------------------------------------------------------- */
/* primitives on orc_real                                                                 */
/* ------------------------------------------------------------------------------------- */

float orc_bf16_to_f32(uint16_t bits) {
    /* a bf16 value is the top half of an f32 bit pattern */
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* y[n] = sum_k W[n,k] x[k]; one output row at a time, ascending k (MATVEC_SRC's contract).
 * Rows are independent, so they may be handed to several threads: each row's sum is still
 * taken in the same order and the result does not depend on the thread count. */
static void matvec_r(const void* W, int bf16, int N, int K, const real* x, real* y) {
    long long work = (long long)N * K;
    int nt = (work >= (1LL << 18)) ? g_threads : 1;
#pragma omp parallel for num_threads(nt) schedule(static)
    for (int n = 0; n < N; ++n) {
        real acc = 0;
        if (bf16) {
            const uint16_t* row = (const uint16_t*)W + (size_t)n * K;
            for (int k = 0; k < K; ++k) acc += (real)orc_bf16_to_f32(row[k]) * x[k];
        } else {
            const float* row = (const float*)W + (size_t)n * K;
            for (int k = 0; k < K; ++k) acc += (real)row[k] * x[k];
        }
        y[n] = acc;
    }
}

/* MV_BIAS (Pocket TTS on wgpu, the flow head): the accumulator starts at the bias,
 * acc = b[n], then acc += W[n,k] x[k] for ascending k; with act == 1 the result goes through
 * SiLU.  W is f32 row-major [N][K]. */
static real silu_r(real g);
static void matvec_bias_r(const float* W, int N, int K, const real* x, const float* b, int act,
                          real* y) {
    for (int n = 0; n < N; ++n) {
        const float* row = W + (size_t)n * K;
        real acc = (real)b[n];
        for (int k = 0; k < K; ++k) acc += (real)row[k] * x[k];
        y[n] = act == 1 ? silu_r(acc) : acc;
    }
}

/* RMSNORM_SRC: inv = 1 / sqrt(sum(x^2) / n + eps); y = x * inv * w */
static void rms_norm_r(const real* x, const float* w, int n, real eps, real* y) {
    real ss = 0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    real inv = (real)1 / sqrt(ss / (real)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (real)w[i];
}

/* ln_src: mean first, then the biased variance of the deviations, then the affine map */
static void layer_norm_r(const real* x, const float* w, const float* b, int n, real eps,
                         real* y) {
    real s = 0;
    for (int i = 0; i < n; ++i) s += x[i];
    real mean = s / (real)n;
    real v = 0;
    for (int i = 0; i < n; ++i) {
        real dv = x[i] - mean;
        v += dv * dv;
    }
    real inv = (real)1 / sqrt(v / (real)n + eps);
    for (int i = 0; i < n; ++i) y[i] = (x[i] - mean) * inv * (real)w[i] + (real)b[i];
}

/* angle(pos, i) = pos * theta^(-2i/d) in double; cos and sin rounded to orc_real */
static void rope_table_r(int d, double theta, int pos, real* c, real* s) {
    for (int i = 0; i < d / 2; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
        double ang = (double)pos * inv_freq;
        c[i] = (real)cos(ang);
        s[i] = (real)sin(ang);
    }
}

/* the multimodal table: angle(i) = pos3[axis(i)] * theta^(-2i/d), axis(i) = assign[i]
 * (assign NULL: every frequency follows axis 0) */
static void mrope_table_r(int d, double theta, const int* pos3, const int* assign, real* c,
                          real* s) {
    for (int i = 0; i < d / 2; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
        double ang = (double)pos3[assign ? assign[i] : 0] * inv_freq;
        c[i] = (real)cos(ang);
        s[i] = (real)sin(ang);
    }
}

/* ROPE_SRC: out[t] = x[t] c_t + rot_t s_t, rot_t = -x[t+half] (t < half), x[t-half] (t >= half);
 * the tables satisfy cos[t] == cos[t + half], so index t mod half */
static void rope_rotate_half_r(real* x, int d, const real* c, const real* s) {
    int half = d / 2;
    real tmp[512];
    for (int t = 0; t < d; ++t) tmp[t] = x[t];
    for (int t = 0; t < d; ++t) {
        real rot = (t < half) ? -tmp[t + half] : tmp[t - half];
        int i = (t < half) ? t : t - half;
        x[t] = tmp[t] * c[i] + rot * s[i];
    }
}

/* rope_push_src: pair (2j, 2j+1) -> (a c - b s, a s + b c) */
static void rope_interleaved_r(real* x, int d, const real* c, const real* s) {
    for (int j = 0; j < d / 2; ++j) {
        real a = x[2 * j], b = x[2 * j + 1];
        x[2 * j] = a * c[j] - b * s[j];
        x[2 * j + 1] = a * s[j] + b * c[j];
    }
}

static real silu_r(real g) { return g / ((real)1 + exp(-g)); }

static real gelu_r(real v) {
    return (real)0.5 * v * ((real)1 + erf(v * (real)0.70710678118654752440));
}

/* GQA_ATTN_SRC for one query row: scores in ascending j, max, exp, sum, divide, then the
 * value sum in ascending j.  kc/vc are position-major [L][G][d]. */
static void gqa_attention_r(const real* q, const real* kc, const real* vc, int L, int H, int G,
                            int d, real* out, real* sc /* scratch [L] */) {
    int group = H / G;
    real scale = (real)1 / sqrt((real)d);
    int kvw = G * d;
    for (int head = 0; head < H; ++head) {
        int kvh = head / group;
        const real* qh = q + (size_t)head * d;
        for (int j = 0; j < L; ++j) {
            const real* kj = kc + (size_t)j * kvw + (size_t)kvh * d;
            real p = 0;
            for (int t = 0; t < d; ++t) p += qh[t] * kj[t];
            sc[j] = p * scale;
        }
        real mx = sc[0];
        for (int j = 1; j < L; ++j) mx = (sc[j] > mx) ? sc[j] : mx;
        real den = 0;
        for (int j = 0; j < L; ++j) {
            real e = exp(sc[j] - mx);
            sc[j] = e;
            den += e;
        }
        for (int j = 0; j < L; ++j) sc[j] = sc[j] / den;
        for (int t = 0; t < d; ++t) {
            real acc = 0;
            for (int j = 0; j < L; ++j) acc += sc[j] * vc[(size_t)j * kvw + (size_t)kvh * d + t];
            out[(size_t)head * d + t] = acc;
        }
    }
}

/* attn_src for one query row: only legal slots take part; max over legal scores, exp-sum,
 * then (sum_j e_j v_j) / den, all in ascending slot order.  kr/vr slot-major [ring][H][d]. */
static void ring_attention_r(const real* q, const real* kr, const real* vr, const uint32_t* pr,
                             int ring, int window, uint32_t pos, int H, int d, real* out,
                             real* sc /* scratch [ring] */, unsigned char* legal /* [ring] */) {
    real scale = (real)1 / sqrt((real)d);
    int dim = H * d;
    for (int j = 0; j < ring; ++j) {
        uint32_t pj = pr[j];
        legal[j] = (pj != ORC_INVALID_POS) && (pj <= pos) && (pos - pj < (uint32_t)window);
    }
    for (int h = 0; h < H; ++h) {
        const real* qh = q + (size_t)h * d;
        int any = 0;
        real mx = 0;
        for (int j = 0; j < ring; ++j) {
            if (!legal[j]) continue;
            const real* kj = kr + (size_t)j * dim + (size_t)h * d;
            real acc = 0;
            for (int t = 0; t < d; ++t) acc += qh[t] * kj[t];
            sc[j] = acc * scale;
            if (!any || sc[j] > mx) mx = sc[j];
            any = 1;
        }
        real den = 0;
        for (int j = 0; j < ring; ++j) {
            if (!legal[j]) continue;
            sc[j] = exp(sc[j] - mx);
            den += sc[j];
        }
        for (int t = 0; t < d; ++t) {
            real acc = 0;
            for (int j = 0; j < ring; ++j) {
                if (!legal[j]) continue;
                acc += sc[j] * vr[(size_t)j * dim + (size_t)h * d + t];
            }
            out[(size_t)h * d + t] = any ? acc / den : (real)0;
        }
    }
}

/* ------------------------------------------------------------------------------------- */
/* exported primitive wrappers (double in / double out)                                   */
/* ------------------------------------------------------------------------------------- */

static real* to_real(const double* x, int n) {
    real* r = (real*)calloc((size_t)(n > 0 ? n : 1), sizeof(real));
    for (int i = 0; i < n; ++i) r[i] = (real)x[i];
    return r;
}
static void from_real(const real* r, int n, double* x) {
    for (int i = 0; i < n; ++i) x[i] = (double)r[i];
}

void orc_matvec_f32(const float* W, int N, int K, const double* x, double* y) {
    real* xr = to_real(x, K);
    real* yr = (real*)malloc(sizeof(real) * (size_t)N);
    matvec_r(W, 0, N, K, xr, yr);
    from_real(yr, N, y);
    free(xr);
    free(yr);
}

void orc_matvec_bf16(const uint16_t* W, int N, int K, const double* x, double* y) {
    real* xr = to_real(x, K);
    real* yr = (real*)malloc(sizeof(real) * (size_t)N);
    matvec_r(W, 1, N, K, xr, yr);
    from_real(yr, N, y);
    free(xr);
    free(yr);
}

void orc_matvec_bias(const float* W, int N, int K, const double* x, const float* b, int act,
                     double* y) {
    real* xr = to_real(x, K);
    real* yr = (real*)malloc(sizeof(real) * (size_t)N);
    matvec_bias_r(W, N, K, xr, b, act, yr);
    from_real(yr, N, y);
    free(xr);
    free(yr);
}

void orc_rms_norm(const double* x, const float* w, int n, double eps, double* y) {
    real* xr = to_real(x, n);
    real* yr = (real*)malloc(sizeof(real) * (size_t)n);
    rms_norm_r(xr, w, n, (real)eps, yr);
    from_real(yr, n, y);
    free(xr);
    free(yr);
}

void orc_layer_norm(const double* x, const float* w, const float* b, int n, double eps,
                    double* y) {
    real* xr = to_real(x, n);
    real* yr = (real*)malloc(sizeof(real) * (size_t)n);
    layer_norm_r(xr, w, b, n, (real)eps, yr);
    from_real(yr, n, y);
    free(xr);
    free(yr);
}

void orc_rope_table(int d, double theta, int pos, double* c, double* s) {
    real cr[256], sr[256];
    rope_table_r(d, theta, pos, cr, sr);
    from_real(cr, d / 2, c);
    from_real(sr, d / 2, s);
}

void orc_mrope_table(int d, double theta, const int* pos3, const int* assign, double* c,
                     double* s) {
    real cr[256], sr[256];
    mrope_table_r(d, theta, pos3, assign, cr, sr);
    from_real(cr, d / 2, c);
    from_real(sr, d / 2, s);
}

void orc_rope_rotate_half(double* x, int d, const double* c, const double* s) {
    real* xr = to_real(x, d);
    real* cr = to_real(c, d / 2);
    real* sr = to_real(s, d / 2);
    rope_rotate_half_r(xr, d, cr, sr);
    from_real(xr, d, x);
    free(xr);
    free(cr);
    free(sr);
}

void orc_rope_interleaved(double* x, int d, const double* c, const double* s) {
    real* xr = to_real(x, d);
    real* cr = to_real(c, d / 2);
    real* sr = to_real(s, d / 2);
    rope_interleaved_r(xr, d, cr, sr);
    from_real(xr, d, x);
    free(xr);
    free(cr);
    free(sr);
}

double orc_silu(double g) { return (double)silu_r((real)g); }
double orc_gelu(double v) { return (double)gelu_r((real)v); }

void orc_gqa_attention(const double* q, const double* kc, const double* vc, int L, int H, int G,
                       int d, double* out) {
    real* qr = to_real(q, H * d);
    real* kr = to_real(kc, L * G * d);
    real* vr = to_real(vc, L * G * d);
    real* o = (real*)malloc(sizeof(real) * (size_t)(H * d));
    real* sc = (real*)malloc(sizeof(real) * (size_t)(L > 0 ? L : 1));
    gqa_attention_r(qr, kr, vr, L, H, G, d, o, sc);
    from_real(o, H * d, out);
    free(qr);
    free(kr);
    free(vr);
    free(o);
    free(sc);
}

void orc_ring_attention(const double* q, const double* kr, const double* vr, const uint32_t* pr,
                        int ring, int window, uint32_t pos, int H, int d, double* out) {
    real* qr = to_real(q, H * d);
    real* k = to_real(kr, ring * H * d);
    real* v = to_real(vr, ring * H * d);
    real* o = (real*)malloc(sizeof(real) * (size_t)(H * d));
    real* sc = (real*)malloc(sizeof(real) * (size_t)ring);
    unsigned char* legal = (unsigned char*)malloc((size_t)ring);
    ring_attention_r(qr, k, v, pr, ring, window, pos, H, d, o, sc, legal);
    from_real(o, H * d, out);
    free(qr);
    free(k);
    free(v);
    free(o);
    free(sc);
    free(legal);
}

/* ------------------------------------------------------------------------------------- */
/* the decode stack                                                                       */
/* ------------------------------------------------------------------------------------- */

struct orc_model {
    orc_config c;
    orc_layer* layers;
    const float* final_norm;
    const float *head_w, *head_b, *eos_w;  /* codec head (FlowLM): out_norm and the EOS row */
    double* eos;    /* [streams] the last step's EOS logit (without its bias) */
    int slots;      /* KV rows per (layer, stream): max_pos (talker) or ring (codec) */
    real* kc;       /* [layers][streams][slots][kv_heads][head_dim], position- or slot-major */
    real* vc;
    uint32_t* pr;   /* codec: [layers][streams][ring] position stamps */
    int* len;       /* [streams] */
    int* rope_assign; /* talker: [head_dim/2] axis of each rope frequency, or NULL (axis 0) */
};

static size_t kv_index(const orc_model* m, int layer, int stream, int slot) {
    size_t kvw = (size_t)m->c.kv_heads * m->c.head_dim;
    return (((size_t)layer * m->c.streams + stream) * m->slots + slot) * kvw;
}

orc_model* orc_create(const orc_config* cfg, const orc_layer* layers, const float* final_norm) {
    if (!cfg || !layers) return NULL;
    if (cfg->layers < 1 || cfg->hidden < 1 || cfg->q_heads < 1 || cfg->kv_heads < 1 ||
        cfg->head_dim < 2 || (cfg->head_dim & 1) || cfg->head_dim > 512 ||
        cfg->q_heads % cfg->kv_heads || cfg->streams < 1 || cfg->max_pos < 1)
        return NULL;
    if (cfg->kind == ORC_CODEC &&
        (cfg->ring < 1 || cfg->window < 1 || cfg->window > cfg->ring ||
         cfg->q_heads != cfg->kv_heads || cfg->q_heads * cfg->head_dim != cfg->hidden))
        return NULL;
    orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
    m->c = *cfg;
    m->layers = (orc_layer*)malloc(sizeof(orc_layer) * (size_t)cfg->layers);
    memcpy(m->layers, layers, sizeof(orc_layer) * (size_t)cfg->layers);
    m->final_norm = final_norm;
    m->slots = (cfg->kind == ORC_CODEC) ? cfg->ring : cfg->max_pos;
    size_t n = (size_t)cfg->layers * cfg->streams * m->slots * cfg->kv_heads * cfg->head_dim;
    m->kc = (real*)calloc(n, sizeof(real));
    m->vc = (real*)calloc(n, sizeof(real));
    m->len = (int*)calloc((size_t)cfg->streams, sizeof(int));
    m->eos = (double*)calloc((size_t)cfg->streams, sizeof(double));
    if (cfg->kind == ORC_CODEC) {
        size_t np = (size_t)cfg->layers * cfg->streams * cfg->ring;
        m->pr = (uint32_t*)malloc(np * sizeof(uint32_t));
        for (size_t i = 0; i < np; ++i) m->pr[i] = ORC_INVALID_POS;
    }
    if (!m->kc || !m->vc || !m->len) {
        orc_destroy(m);
        return NULL;
    }
    return m;
}

void orc_destroy(orc_model* m) {
    if (!m) return;
    free(m->layers);
    free(m->kc);
    free(m->vc);
    free(m->pr);
    free(m->rope_assign);
    free(m->len);
    free(m->eos);
    free(m);
}

int orc_set_head(orc_model* m, const float* norm_w, const float* norm_b, const float* eos_w) {
    if (!m || m->c.kind != ORC_CODEC || !norm_w || !norm_b) return -1;
    m->head_w = norm_w;
    m->head_b = norm_b;
    m->eos_w = eos_w;
    return 0;
}

double orc_eos(const orc_model* m, int stream) {
    return (m && stream >= 0 && stream < m->c.streams) ? m->eos[stream] : 0.0;
}

int orc_len(const orc_model* m, int stream) {
    if (!m || stream < 0 || stream >= m->c.streams) return -1;
    return m->len[stream];
}

/* pocket_tts_gpu `reset` / mimi_gpu `reset`: zero K/V, every stamp back to INVALID */
void orc_reset(orc_model* m, int stream) {
    if (!m || stream < 0 || stream >= m->c.streams) return;
    size_t kvw = (size_t)m->c.kv_heads * m->c.head_dim;
    for (int l = 0; l < m->c.layers; ++l) {
        memset(m->kc + kv_index(m, l, stream, 0), 0, sizeof(real) * kvw * m->slots);
        memset(m->vc + kv_index(m, l, stream, 0), 0, sizeof(real) * kvw * m->slots);
        if (m->pr)
            for (int j = 0; j < m->c.ring; ++j)
                m->pr[((size_t)l * m->c.streams + stream) * m->c.ring + j] = ORC_INVALID_POS;
    }
    m->len[stream] = 0;
}

/* pocket_tts_gpu `load_voice`: the stored keys already carry rope, so this is a copy into
 * rows (slots) 0..n_pos, and (codec) the stamps become 0..n_pos */
int orc_prefill_kv(orc_model* m, int stream, const float* k, const float* v, int n_pos) {
    if (!m || stream < 0 || stream >= m->c.streams || n_pos < 0) return -1;
    if (n_pos > m->slots) return -3;
    size_t kvw = (size_t)m->c.kv_heads * m->c.head_dim;
    orc_reset(m, stream);
    for (int l = 0; l < m->c.layers; ++l) {
        for (int p = 0; p < n_pos; ++p) {
            const float* ks = k + ((size_t)l * n_pos + p) * kvw;
            const float* vs = v + ((size_t)l * n_pos + p) * kvw;
            real* kd = m->kc + kv_index(m, l, stream, p);
            real* vd = m->vc + kv_index(m, l, stream, p);
            for (size_t i = 0; i < kvw; ++i) {
                kd[i] = (real)ks[i];
                vd[i] = (real)vs[i];
            }
            if (m->pr) m->pr[((size_t)l * m->c.streams + stream) * m->c.ring + p] = (uint32_t)p;
        }
    }
    m->len[stream] = n_pos;
    return 0;
}

int orc_read_kv(const orc_model* m, int layer, int stream, int pos, double* k, double* v) {
    if (!m || layer < 0 || layer >= m->c.layers || stream < 0 || stream >= m->c.streams)
        return -1;
    int slot = (m->c.kind == ORC_CODEC) ? pos % m->c.ring : pos;
    if (pos < 0 || slot >= m->slots) return -1;
    size_t kvw = (size_t)m->c.kv_heads * m->c.head_dim;
    const real* ks = m->kc + kv_index(m, layer, stream, slot);
    const real* vs = m->vc + kv_index(m, layer, stream, slot);
    for (size_t i = 0; i < kvw; ++i) {
        k[i] = (double)ks[i];
        v[i] = (double)vs[i];
    }
    return 0;
}

/* one talker layer for one stream, in build_step_plan's order; the new K/V row goes to cache
 * row pos, and the rope turns by pos or, with pos3, by the per-axis positions pos3[0..2] */
static void talker_layer(orc_model* m, int l, int s, int pos, const int* pos3, real* x,
                         real* buf) {
    const orc_config* c = &m->c;
    const orc_layer* W = &m->layers[l];
    int h = c->hidden, d = c->head_dim, H = c->q_heads, G = c->kv_heads, ni = c->inter;
    int qw = H * d, kvw = G * d, bf = c->weight_bf16;
    real eps = (real)c->norm_eps;
    real* n = buf;             /* [h] */
    real* q = n + h;           /* [qw] */
    real* k = q + qw;          /* [kvw] */
    real* v = k + kvw;         /* [kvw] */
    real* att = v + kvw;       /* [qw] */
    real* o = att + qw;        /* [h] */
    real* g = o + h;           /* [inter] */
    real* u = g + ni;          /* [inter] */
    real* a = u + ni;          /* [inter] */
    real* dn = a + ni;         /* [h] */
    real* cs = dn + h;         /* [d/2] */
    real* sn = cs + d / 2;     /* [d/2] */
    real* sc = sn + d / 2;     /* [max_pos] */

    rms_norm_r(x, W->in_norm, h, eps, n);
    matvec_r(W->wq, bf, qw, h, n, q);
    matvec_r(W->wk, bf, kvw, h, n, k);
    matvec_r(W->wv, bf, kvw, h, n, v);
    for (int hh = 0; hh < H; ++hh) rms_norm_r(q + hh * d, W->q_norm, d, eps, q + hh * d);
    for (int gg = 0; gg < G; ++gg) rms_norm_r(k + gg * d, W->k_norm, d, eps, k + gg * d);
    if (pos3)
        mrope_table_r(d, c->rope_theta, pos3, m->rope_assign, cs, sn);
    else
        rope_table_r(d, c->rope_theta, pos, cs, sn);
    for (int hh = 0; hh < H; ++hh) rope_rotate_half_r(q + hh * d, d, cs, sn);
    for (int gg = 0; gg < G; ++gg) rope_rotate_half_r(k + gg * d, d, cs, sn);
    real* kd = m->kc + kv_index(m, l, s, pos);
    real* vd = m->vc + kv_index(m, l, s, pos);
    for (int i = 0; i < kvw; ++i) {
        kd[i] = k[i];
        vd[i] = v[i];
    }
    gqa_attention_r(q, m->kc + kv_index(m, l, s, 0), m->vc + kv_index(m, l, s, 0), pos + 1, H, G,
                    d, att, sc);
    matvec_r(W->wo, bf, h, qw, att, o);
    for (int i = 0; i < h; ++i) x[i] = x[i] + o[i];
    rms_norm_r(x, W->post_norm, h, eps, n);
    matvec_r(W->wgate, bf, ni, h, n, g);
    matvec_r(W->wup, bf, ni, h, n, u);
    for (int i = 0; i < ni; ++i) a[i] = silu_r(g[i]) * u[i];
    matvec_r(W->wdown, bf, h, ni, a, dn);
    for (int i = 0; i < h; ++i) x[i] = x[i] + dn[i];
}

/* one codec layer for one stream, in transformer_shaped's order */
static void codec_layer(orc_model* m, int l, int s, int pos, real* x, real* buf) {
    const orc_config* c = &m->c;
    const orc_layer* W = &m->layers[l];
    int D = c->hidden, d = c->head_dim, H = c->q_heads, F = c->inter, ring = c->ring;
    int bf = c->weight_bf16;
    real eps = (real)c->norm_eps;
    real* hb = buf;            /* [D] */
    real* qkv = hb + D;        /* [3D] */
    real* att = qkv + 3 * D;   /* [D] */
    real* o = att + D;         /* [D] */
    real* f = o + D;           /* [F] */
    real* y = f + F;           /* [D] */
    real* cs = y + D;          /* [d/2] */
    real* sn = cs + d / 2;     /* [d/2] */
    real* sc = sn + d / 2;     /* [ring] */
    unsigned char* legal = (unsigned char*)(sc + ring);

    layer_norm_r(x, W->ln1_w, W->ln1_b, D, eps, hb);
    matvec_r(W->in_proj, bf, 3 * D, D, hb, qkv);
    real* q = qkv;
    real* k = qkv + D;
    real* v = qkv + 2 * D;
    rope_table_r(d, c->rope_theta, pos, cs, sn);
    for (int hh = 0; hh < H; ++hh) {
        rope_interleaved_r(q + hh * d, d, cs, sn);
        rope_interleaved_r(k + hh * d, d, cs, sn);
    }
    int slot = pos % ring;
    real* kd = m->kc + kv_index(m, l, s, slot);
    real* vd = m->vc + kv_index(m, l, s, slot);
    for (int i = 0; i < D; ++i) {
        kd[i] = k[i];
        vd[i] = v[i];
    }
    uint32_t* pr = m->pr + ((size_t)l * c->streams + s) * ring;
    pr[slot] = (uint32_t)pos;
    ring_attention_r(q, m->kc + kv_index(m, l, s, 0), m->vc + kv_index(m, l, s, 0), pr, ring,
                     c->window, (uint32_t)pos, H, d, att, sc, legal);
    matvec_r(W->out_proj, bf, D, D, att, o);
    /* LayerScale multiplies the branch; the FlowLM backbone has none (a scale of one) */
    for (int i = 0; i < D; ++i) x[i] = x[i] + (W->ls1 ? (real)W->ls1[i] * o[i] : o[i]);
    layer_norm_r(x, W->ln2_w, W->ln2_b, D, eps, hb);
    matvec_r(W->lin1, bf, F, D, hb, f);
    for (int i = 0; i < F; ++i) f[i] = gelu_r(f[i]);
    matvec_r(W->lin2, bf, D, F, f, y);
    for (int i = 0; i < D; ++i) x[i] = x[i] + (W->ls2 ? (real)W->ls2[i] * y[i] : y[i]);
}

static int pos3_ok(const orc_model* m, const int* p3) {
    for (int a = 0; a < 3; ++a)
        if (p3[a] < 0 || p3[a] >= m->c.max_pos) return 0;
    return 1;
}

int orc_set_mrope(orc_model* m, const int* assign) {
    if (!m || m->c.kind != ORC_TALKER) return -1;
    const int half = m->c.head_dim / 2;
    if (assign)
        for (int i = 0; i < half; ++i)
            if (assign[i] < 0 || assign[i] > 2) return -1;
    free(m->rope_assign);
    m->rope_assign = NULL;
    if (assign) {
        m->rope_assign = (int*)malloc(sizeof(int) * (size_t)half);
        memcpy(m->rope_assign, assign, sizeof(int) * (size_t)half);
    }
    return 0;
}

int orc_step(orc_model* m, int rows, const float* x_in, const int* pos, double* out,
             double* taps) {
    return orc_step_mrope(m, rows, x_in, pos, NULL, out, taps);
}

int orc_step_mrope(orc_model* m, int rows, const float* x_in, const int* pos, const int* pos3,
                   double* out, double* taps) {
    if (!m || rows < 1 || rows > m->c.streams || !x_in || !pos || !out) return -1;
    const orc_config* c = &m->c;
    if (pos3 && c->kind != ORC_TALKER) return -4;
    for (int s = 0; s < rows; ++s) {
        if (pos[s] != m->len[s]) return -2;
        if (pos[s] >= c->max_pos) return -3;
        if (pos3 && !pos3_ok(m, pos3 + 3 * s)) return -3;
    }
    int h = c->hidden;
    size_t nbuf = (size_t)8 * h + 4 * (size_t)c->q_heads * c->head_dim +
                  4 * (size_t)c->inter + (size_t)c->head_dim + 2 * (size_t)m->slots + 64;
    real* buf = (real*)malloc(sizeof(real) * nbuf);
    real* x = (real*)malloc(sizeof(real) * (size_t)h);
    real* y = (real*)malloc(sizeof(real) * (size_t)h);
    for (int s = 0; s < rows; ++s) {
        for (int i = 0; i < h; ++i) x[i] = (real)x_in[(size_t)s * h + i];
        for (int l = 0; l < c->layers; ++l) {
            if (c->kind == ORC_TALKER)
                talker_layer(m, l, s, pos[s], pos3 ? pos3 + 3 * s : NULL, x, buf);
            else
                codec_layer(m, l, s, pos[s], x, buf);
            if (taps) from_real(x, h, taps + ((size_t)l * rows + s) * h);
        }
        if (c->kind == ORC_TALKER) {
            rms_norm_r(x, m->final_norm, h, (real)c->norm_eps, y);
            from_real(y, h, out + (size_t)s * h);
        } else if (m->head_w) {
            /* FlowLM backbone: out_norm, then the EOS logit of the normalized row */
            layer_norm_r(x, m->head_w, m->head_b, h, (real)c->norm_eps, y);
            from_real(y, h, out + (size_t)s * h);
            if (m->eos_w) {
                real e = 0;
                for (int i = 0; i < h; ++i) e += (real)m->eos_w[i] * y[i];
                m->eos[s] = (double)e;
            }
        } else {
            from_real(x, h, out + (size_t)s * h);
        }
        m->len[s] += 1;
    }
    free(buf);
    free(x);
    free(y);
    return 0;
}

int orc_flow_step(const orc_flow* f, const float* cond, const float* noise, double* out) {
    if (!f || !cond || !noise || !out || f->dim < 1 || f->latent < 1 || f->cond < 1 ||
        f->blocks < 0)
        return -1;
    const int D = f->dim, Lt = f->latent, C = f->cond;
    const real eps = (real)f->ln_eps;
    real* x = (real*)malloc(sizeof(real) * (size_t)D);
    real* y = (real*)malloc(sizeof(real) * (size_t)D);
    real* m = (real*)malloc(sizeof(real) * 3 * (size_t)D);
    real* u = (real*)malloc(sizeof(real) * (size_t)D);
    real* t = (real*)malloc(sizeof(real) * (size_t)(D > C ? D : C));
    real* h = (real*)malloc(sizeof(real) * (size_t)D);
    float* one = (float*)malloc(sizeof(float) * (size_t)D);
    float* zero = (float*)malloc(sizeof(float) * (size_t)D);
    real* dir = (real*)malloc(sizeof(real) * (size_t)Lt);
    for (int i = 0; i < D; ++i) {
        one[i] = 1.0f;
        zero[i] = 0.0f;
    }
    /* x = input_proj(noise) (MV_BIAS) */
    for (int i = 0; i < Lt; ++i) t[i] = (real)noise[i];
    matvec_bias_r(f->ip_w, D, Lt, t, f->ip_b, 0, x);
    /* y = silu(t_const + cond_embed(cond)) (MV_BIAS, then ADD_SILU: the constant first) */
    for (int i = 0; i < C; ++i) t[i] = (real)cond[i];
    matvec_bias_r(f->cond_w, D, C, t, f->cond_b, 0, y);
    for (int i = 0; i < D; ++i) y[i] = silu_r((real)f->t_const[i] + y[i]);
    for (int bl = 0; bl < f->blocks; ++bl) {
        /* the fused adaLN projection [shift | scale | gate] */
        matvec_bias_r(f->ada_w[bl], 3 * D, D, y, f->ada_b[bl], 0, m);
        layer_norm_r(x, f->ln_w[bl], f->ln_b[bl], D, eps, u);
        for (int i = 0; i < D; ++i) u[i] = u[i] * ((real)1 + m[D + i]) + m[i];  /* modulate */
        matvec_bias_r(f->m0_w[bl], D, D, u, f->m0_b[bl], 1, h);
        matvec_bias_r(f->m2_w[bl], D, D, h, f->m2_b[bl], 0, u);
        for (int i = 0; i < D; ++i) x[i] += m[2 * D + i] * u[i];  /* GATED_ADD, third chunk */
    }
    /* final layer: [shift | scale] over a LayerNorm without affine weights */
    matvec_bias_r(f->fada_w, 2 * D, D, y, f->fada_b, 0, m);
    layer_norm_r(x, one, zero, D, eps, u);
    for (int i = 0; i < D; ++i) u[i] = u[i] * ((real)1 + m[D + i]) + m[i];  /* final modulate */
    matvec_bias_r(f->f_w, Lt, D, u, f->f_b, 0, dir);
    /* LSD_STEP with one step: x1 = x0 + dir * (1 / steps) */
    const real inv_steps = (real)1 / (real)1;
    for (int i = 0; i < Lt; ++i) out[i] = (double)((real)noise[i] + dir[i] * inv_steps);
    free(x); free(y); free(m); free(u); free(t); free(h); free(one); free(zero); free(dir);
    return 0;
}

int orc_prefill(orc_model* m, int stream, int n, const float* x_in, double* out) {
    return orc_prefill_mrope(m, stream, n, x_in, NULL, out);
}

int orc_prefill_mrope(orc_model* m, int stream, int n, const float* x_in, const int* pos3,
                      double* out) {
    if (!m || stream < 0 || stream >= m->c.streams || n < 1 || !x_in || !out) return -1;
    const orc_config* c = &m->c;
    if (c->kind != ORC_TALKER) return -4;
    if (m->len[stream] + n > c->max_pos) return -3;
    if (pos3)
        for (int r = 0; r < n; ++r)
            if (!pos3_ok(m, pos3 + 3 * r)) return -3;
    const int h = c->hidden;
    size_t nbuf = (size_t)8 * h + 4 * (size_t)c->q_heads * c->head_dim +
                  4 * (size_t)c->inter + (size_t)c->head_dim + 2 * (size_t)m->slots + 64;
    real* buf = (real*)malloc(sizeof(real) * nbuf);
    real* x = (real*)malloc(sizeof(real) * (size_t)h);
    real* y = (real*)malloc(sizeof(real) * (size_t)h);
    for (int r = 0; r < n; ++r) {  /* row r: one step at position len + r */
        const int pos = m->len[stream];
        for (int i = 0; i < h; ++i) x[i] = (real)x_in[(size_t)r * h + i];
        for (int l = 0; l < c->layers; ++l)
            talker_layer(m, l, stream, pos, pos3 ? pos3 + 3 * r : NULL, x, buf);
        rms_norm_r(x, m->final_norm, h, (real)c->norm_eps, y);
        from_real(y, h, out + (size_t)r * h);
        m->len[stream] += 1;
    }
    free(buf);
    free(x);
    free(y);
    return 0;
}
