// dec_api.cu -- the C ABI (include/dec.h): context state, the step plan, CUDA-graph replay.
//
// Plan of one step of m rows (per layer, six kernels chained with programmatic dependent
// launch, then one final kernel):
//   talker: [RMSNorm + QKV GEMV] -> [qk-norm + rope + append + split-K GQA attention chunks]
//           -> [merge of the chunks] -> [o-proj GEMV + residual]
//           -> [RMSNorm + gate/up GEMV + SwiGLU] -> [down GEMV + residual];
//           final RMSNorm (+ length advance)
//   codec:  [LayerNorm + qkv GEMV] -> [rope + ring push + windowed attention chunks] -> [merge]
//           -> [out-proj GEMV + LayerScale residual] -> [LayerNorm + lin1 GEMV + GELU]
//           -> [lin2 GEMV + LayerScale residual]; copy-out (+ length advance)
// The sequence is the talker's build_step_plan and Mimi's transformer_shaped with the
// elementwise passes folded into the GEMV prologues/epilogues and the attention prologue.
// It is captured once per step width m as a CUDA graph and replayed, with the step's input and
// output pointers patched into the few nodes that take them; the per-step positions live on
// the device and the graph's last kernel advances them, so a step needs no host-to-device
// traffic beyond the caller's own input.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dec.h"
#include "gemv_rows.cuh"
#include "kernels.h"

using namespace dec;

namespace {

thread_local std::string g_create_error;

struct LayerW {
    // talker
    const void *qkv, *o, *gu, *down;
    const float *in_norm, *post_norm, *q_norm, *k_norm;
    // codec
    const void *in_proj, *out_proj, *lin1, *lin2;
    const float *ln1_w, *ln1_b, *ln2_w, *ln2_b, *ls1, *ls2;
};

// A step plan, one per (m, rotary-position buffer): it serves every input/output pair.  The
// step's input and output pointers are arguments of a few kernel nodes of the captured graph,
// updated in place when they change: the streamed kernel's single node, or in the multi-kernel
// plan the three launches that take them (layer 0's q/k/v GEMV reads x_in, its o-proj adds
// x_in as the residual, the final kernel writes the output).  exec is null with
// DEC_FLAG_NO_GRAPH (the kernels are launched with the step's pointers each time).
struct PlanEntry {
    int m;
    const float* x_in;       // the pointers the graph's nodes hold now
    float* out;
    const int32_t* rope;     // per-axis rotary positions of the rows (multi-kernel plans), or null
    SPhase* phases;          // streamed plan: its phase list (device), or null (multi-kernel plan)
    char* sbuf;              // streamed plan: its tagged activation buffers and StreamState
    size_t sbuf_bytes;
    StreamState* st;
    unsigned* cnt;           // streamed plan: its per-phase completion counters
    long long launches;      // streamed plan: launches since sbuf was last cleared
    cudaGraphExec_t exec;
    cudaGraph_t graph;       // the captured graph, owner of the node handles below
    cudaGraphNode_t node;    // streamed plan: the kernel node
    cudaKernelNodeParams kp; // its launch parameters (kernelParams points at a StreamParams)
    cudaGraphNode_t io_node[3];       // multi-kernel plan: q/k/v GEMV, o-proj, final kernel
    cudaKernelNodeParams io_kp[3];    // their launch parameters
    GemvParams io_g[2];               // the two GEMVs' captured arguments
    TmapBytes io_tm[2];               // ... and, for the tensor-core GEMV, its second argument
    bool io_has_tm[2] = {false, false};
    FinalParams io_f;                 // the final kernel's captured arguments
};

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

namespace dec {
cudaError_t configure_kernels() {
    static std::mutex mu;
    static uint64_t done = 0;  // bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && (done >> dev & 1u)) return cudaSuccess;
    if ((e = gemv_configure()) != cudaSuccess) return e;
    if ((e = gemv_tc_configure()) != cudaSuccess) return e;
    if ((e = attention_configure()) != cudaSuccess) return e;
    if ((e = stream_configure()) != cudaSuccess) return e;
    if (dev < 64) done |= (uint64_t)1 << dev;
    return cudaSuccess;
}
}  // namespace dec

namespace {

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

struct dec_ctx {
    dec_config cfg{};
    cudaStream_t stream = nullptr;
    cudaStream_t cap_stream = nullptr;
    int num_sms = 0;
    int S = 0;              // streams
    int R = 0;              // rows of the activation scratch: max(S, prefill block rows)
    int prefill_rows = 0;   // rows of a prefill block (0: prefill not served)
    int slots = 0;          // KV rows per (layer, stream, kv head)
    int qkv_rows = 0;       // rows of the fused q/k/v matrix
    int max_chunks = 0;     // attention chunks per (stream, kv head)
    int step_grid[3] = {};  // CTAs of the streamed step kernel for m = 1, 2 (0: not used)
    char* arena = nullptr;  // weights
    std::vector<LayerW> L;
    const float* final_norm = nullptr;
    const float* final_norm_b = nullptr;  // codec head: out_norm bias
    const float* eos_w = nullptr;         // codec head: EOS row
    float eos_b = 0.f;
    float* eos = nullptr;                 // [S] the last step's EOS logits (no bias)
    char* state = nullptr;  // caches, tables, scratch
    float *kc = nullptr, *vc = nullptr;
    uint32_t* pr = nullptr;
    float *rope_cos = nullptr, *rope_sin = nullptr;
    int32_t* rope_axis = nullptr;  // [d/2] multimodal rope: the axis of each frequency
    float *xres = nullptr, *qkv = nullptr, *attn = nullptr, *act = nullptr;
    float *part = nullptr, *part_ml = nullptr;  // attention chunk partials
    float* mpart = nullptr;       // tensor-core GEMV: partial sums of split tiles
    size_t mpart_floats = 0;
    unsigned* mtick = nullptr;    // ... and its tickets, one per 8-row tile
    int mtick_n = 0;
    int32_t* len_dev = nullptr;
    unsigned* status = nullptr;
    int stall_phase = -1;   // dec_inject_stall: the next step's stalled phase and its poll bound
    int stall_polls = 0;
    float* taps = nullptr;
    float *io_in = nullptr, *io_out = nullptr;
    unsigned* status_host = nullptr;  // pinned
    std::vector<int> len_host;
    std::vector<TmapBytes> tmaps;     // TMA descriptors of the GEMV matrices [layer][4] (bf16, > 2 rows)
    std::vector<uint8_t> tmap_ok;     // ... and which of them were made
    std::vector<PlanEntry> plans;
    std::string err;
};

namespace {

dec_status fail(dec_ctx* ctx, dec_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (ctx)
        ctx->err = buf;
    else
        g_create_error = buf;
    return st;
}

dec_status cuda_fail(dec_ctx* ctx, cudaError_t e, const char* what) {
    return fail(ctx, DEC_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CUDA_TRY(ctx, call, what)                          \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, what); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dec_status validate_config(const dec_config* c) {
    if (!c) return fail(nullptr, DEC_E_ARG, "config is NULL");
    if (c->kind != DEC_QWEN3_TALKER && c->kind != DEC_CODEC_WINDOWED)
        return fail(nullptr, DEC_E_ARG, "unknown kind %d", c->kind);
    if (c->layers < 1 || c->hidden < 8 || c->inter < 8 || c->q_heads < 1 || c->kv_heads < 1)
        return fail(nullptr, DEC_E_ARG, "layers/hidden/inter/heads must be positive");
    if (c->hidden % 8 || c->inter % 8)
        return fail(nullptr, DEC_E_UNSUPPORTED, "hidden and inter must be multiples of 8");
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(nullptr, DEC_E_UNSUPPORTED, "head_dim %d: kernels take 64 or 128", c->head_dim);
    if (c->q_heads % c->kv_heads)
        return fail(nullptr, DEC_E_ARG, "q_heads %% kv_heads != 0");
    if (c->q_heads / c->kv_heads > kMaxGroup)
        return fail(nullptr, DEC_E_UNSUPPORTED, "GQA group above %d", kMaxGroup);
    if (c->weight_dtype != DEC_F32 && c->weight_dtype != DEC_BF16)
        return fail(nullptr, DEC_E_ARG, "unknown weight dtype %d", c->weight_dtype);
    if (c->max_pos < 1) return fail(nullptr, DEC_E_ARG, "max_pos must be >= 1");
    if (c->max_streams < 1 || c->max_streams > 8)
        return fail(nullptr, DEC_E_ARG, "max_streams must be in 1..8");
    if (!(c->norm_eps >= 0.f) || !std::isfinite(c->norm_eps))
        return fail(nullptr, DEC_E_ARG, "norm_eps must be finite and >= 0");
    if (!(c->rope_theta > 0.0) || !std::isfinite(c->rope_theta))
        return fail(nullptr, DEC_E_ARG, "rope_theta must be finite and > 0");
    if (c->kind == DEC_CODEC_WINDOWED) {
        if (c->kv_heads != c->q_heads)
            return fail(nullptr, DEC_E_ARG, "codec layers are multi-head: kv_heads == q_heads");
        if (c->q_heads * c->head_dim != c->hidden)
            return fail(nullptr, DEC_E_ARG, "codec: q_heads * head_dim must equal hidden");
        if (c->ring < 1 || c->window < 1 || c->window > c->ring)
            return fail(nullptr, DEC_E_ARG, "codec: need 1 <= window <= ring");
    }
    if ((c->kind == DEC_QWEN3_TALKER ? c->max_pos : c->ring) > kMaxSlots)
        return fail(nullptr, DEC_E_UNSUPPORTED, "KV capacity above %d positions", kMaxSlots);
    const int widest = std::max(std::max(c->hidden, c->inter), c->q_heads * c->head_dim);
    if (gemv_smem_bytes(c->max_streams, widest) > 200 * 1024)
        return fail(nullptr, DEC_E_UNSUPPORTED,
                    "max_streams * widest row (%d) exceeds the GEMV's shared-memory stage", widest);
    return DEC_OK;
}

// cos/sin of pos * theta^(-2i/d) for i < d/2, computed in double and rounded to f32.  The
// talker page builds its table on the host (Qwen3-TTS talker on wgpu, load(): cos/sin
// [max_pos x hd]); the same angle drives the codec's interleaved pairs.
void build_rope_tables(int max_pos, int d, double theta, std::vector<float>& c,
                       std::vector<float>& s) {
    const int half = d / 2;
    c.resize((size_t)max_pos * half);
    s.resize((size_t)max_pos * half);
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) inv[i] = std::pow(theta, -2.0 * (double)i / (double)d);
    for (int p = 0; p < max_pos; ++p)
        for (int i = 0; i < half; ++i) {
            const double a = (double)p * inv[i];
            c[(size_t)p * half + i] = (float)std::cos(a);
            s[(size_t)p * half + i] = (float)std::sin(a);
        }
}

void destroy_plan(PlanEntry& e) {
    if (e.exec) cudaGraphExecDestroy(e.exec);
    if (e.graph) cudaGraphDestroy(e.graph);
    if (e.phases) cudaFree(e.phases);
    if (e.sbuf) cudaFree(e.sbuf);
    e.exec = nullptr;
    e.graph = nullptr;
    e.phases = nullptr;
    e.sbuf = nullptr;
}

void destroy_plans(dec_ctx* ctx) {
    for (auto& e : ctx->plans) destroy_plan(e);
    ctx->plans.clear();
}

// Parameters of stage `stage` of layer `l` for rows 0..m-1 (see dec_launch_stage for the
// stages): a GEMV (returns false) or, for stage 1, the attention (returns true; `a` is filled).
bool stage_params(dec_ctx* ctx, int l, int stage, int m, const float* x_in, GemvParams& g,
                  AttnParams& a, const int32_t* rope_pos = nullptr) {
    const dec_config& c = ctx->cfg;
    const bool talker = c.kind == DEC_QWEN3_TALKER;
    const int h = c.hidden, d = c.head_dim, H = c.q_heads, G = c.kv_heads, I = c.inter;
    const int S = ctx->S;
    const int qw = H * d;
    const size_t kv_layer = (size_t)S * G * ctx->slots * d;
    const LayerW& W = ctx->L[l];
    const float* xr = (l == 0) ? x_in : ctx->xres;  // residual stream entering layer l
    g = GemvParams{};
    g.m = m;
    g.eps = c.norm_eps;
    g.status = ctx->status;
    g.unit = 1;
    if (stage != 1 && !ctx->tmaps.empty()) {  // q/k/v, o-proj, gate/up, down: slots 0..3
        const size_t slot = (size_t)l * 4 + (stage == 0 ? 0 : stage - 1);
        g.tmap = ctx->tmap_ok[slot] ? ctx->tmaps[slot].b : nullptr;
    }
    g.mpart = ctx->mpart;
    g.mpart_floats = ctx->mpart_floats;
    g.mtick = ctx->mtick;
    g.mtick_n = ctx->mtick_n;
    switch (stage) {
        case 0:  // norm + q/k/v
            g.W = talker ? W.qkv : W.in_proj;
            g.N = ctx->qkv_rows;
            g.K = h;
            g.x = xr;
            g.ldx = h;
            g.pro = talker ? PRO_RMS : PRO_LN;
            g.nw = talker ? W.in_norm : W.ln1_w;
            g.nb = talker ? nullptr : W.ln1_b;
            g.epi = EPI_STORE;
            g.y = ctx->qkv;
            g.ldy = ctx->qkv_rows;
            return false;
        case 1:  // attention with its prologue
            a = AttnParams{};
            a.mode = talker ? ATTN_TALKER : ATTN_RING;
            a.m = m;
            a.H = H;
            a.G = G;
            a.d = d;
            a.slots = ctx->slots;
            a.window = c.window;
            a.qkv = ctx->qkv;
            a.ldqkv = ctx->qkv_rows;
            a.kc = ctx->kc + (size_t)l * kv_layer;
            a.vc = ctx->vc + (size_t)l * kv_layer;
            a.pr = talker ? nullptr : ctx->pr + (size_t)l * S * ctx->slots;
            a.len = ctx->len_dev;
            a.qn = W.q_norm;
            a.kn = W.k_norm;
            a.eps = c.norm_eps;
            a.rope_cos = ctx->rope_cos;
            a.rope_sin = ctx->rope_sin;
            a.max_pos = c.max_pos;
            a.rope_pos = talker ? rope_pos : nullptr;
            a.rope_axis = ctx->rope_axis;
            a.part = ctx->part;
            a.part_ml = ctx->part_ml;
            a.tickets = nullptr;  // the partials are merged by k_attn_merge (or a merge phase)
            a.max_chunks = ctx->max_chunks;
            // two chunks per CTA when that grid is one wave at one CTA per SM (a short cache,
            // few streams); otherwise one chunk per CTA, up to three CTAs per SM
            a.paired = attention_pair_ctas(a) <= ctx->num_sms ? 1 : 0;
            a.out = ctx->attn;
            a.status = ctx->status;
            return true;
        case 2:  // o-proj + residual (codec: LayerScale)
            g.W = talker ? W.o : W.out_proj;
            g.N = h;
            g.K = qw;
            g.x = ctx->attn;
            g.ldx = qw;
            g.pro = PRO_NONE;
            g.epi = EPI_RESID;
            g.y = ctx->xres;
            g.ldy = h;
            g.res = xr;
            g.ldres = h;
            g.ls = talker ? nullptr : W.ls1;
            return false;
        case 3:  // norm + gate/up + SwiGLU (codec: lin1 + GELU)
            g.W = talker ? W.gu : W.lin1;
            g.N = talker ? 2 * I : I;
            g.K = h;
            g.x = ctx->xres;
            g.ldx = h;
            g.pro = talker ? PRO_RMS : PRO_LN;
            g.nw = talker ? W.post_norm : W.ln2_w;
            g.nb = talker ? nullptr : W.ln2_b;
            g.epi = talker ? EPI_SWIGLU : EPI_GELU;
            g.unit = talker ? 2 : 1;
            g.y = ctx->act;
            g.ldy = I;
            return false;
        default:  // 4: down + residual (codec: lin2 + LayerScale)
            g.W = talker ? W.down : W.lin2;
            g.N = h;
            g.K = I;
            g.x = ctx->act;
            g.ldx = I;
            g.pro = PRO_NONE;
            g.epi = EPI_RESID;
            g.y = ctx->xres;
            g.ldy = h;
            g.res = ctx->xres;
            g.ldres = h;
            g.ls = talker ? nullptr : W.ls2;
            g.tap = ctx->taps ? ctx->taps + (size_t)l * S * h : nullptr;
            g.ldtap = h;
            return false;
    }
}

// Launch stage `stage` of layer `l` for rows 0..m-1: one GEMV kernel, or for stage 1 the
// attention chunks and the merge of their partials.
cudaError_t launch_stage(dec_ctx* ctx, int l, int stage, int m, const float* x_in, cudaStream_t s,
                         bool pdl, const int32_t* rope_pos = nullptr) {
    if (stage < 0 || stage > 4) return cudaErrorInvalidValue;
    GemvParams g;
    AttnParams a;
    if (!stage_params(ctx, l, stage, m, x_in, g, a, rope_pos))
        return launch_gemv(g, ctx->cfg.weight_dtype, ctx->num_sms, s, pdl);
    cudaError_t e = launch_attention(a, s, pdl);
    if (e != cudaSuccess) return e;
    return launch_attention_merge(a, s, true);
}

FinalParams final_params(dec_ctx* ctx, int m, float* out) {
    const dec_config& c = ctx->cfg;
    FinalParams f = {};
    f.m = m;
    f.h = c.hidden;
    f.x = ctx->xres;
    f.w = ctx->final_norm;  // talker RMSNorm; codec: the head's LayerNorm, or NULL (copy)
    f.b = ctx->final_norm_b;
    f.eos_w = ctx->eos_w;
    f.eos = ctx->eos;
    f.eps = c.norm_eps;
    f.out = out;
    f.len = ctx->len_dev;
    f.advance_stream = -1;
    return f;
}

// The streamed kernel's plan of a step of m rows: its tagged activation buffers (allocated into
// pe.sbuf, zeroed) and its phase list (per layer: q/k/v, attention with the merge of its
// partials, o-proj, gate/up, down; then the output rows).  Layer 0 reads the step input, which
// is a kernel argument.
cudaError_t build_stream_plan(dec_ctx* ctx, int m, PlanEntry& pe, std::vector<SPhase>& ph) {
    const dec_config& c = ctx->cfg;
    const bool talker = c.kind == DEC_QWEN3_TALKER;
    const int h = c.hidden, d = c.head_dim, H = c.q_heads, G = c.kv_heads, I = c.inter;
    const int qw = H * d, P = ctx->step_grid[m];
    const size_t kv_layer = (size_t)ctx->S * G * ctx->slots * d;
    size_t tot = 0;
    auto take = [&](size_t words) {
        const size_t o = tot;
        tot += align_up(words * sizeof(uint64_t));
        return o;
    };
    const size_t o_qkv = take((size_t)m * ctx->qkv_rows), o_att = take((size_t)m * qw);
    const size_t o_mid = take((size_t)m * h), o_act = take((size_t)m * I), o_res = take((size_t)m * h);
    const size_t o_part = take((size_t)m * H * P * d), o_ml = take((size_t)m * H * P * 2);
    const size_t o_st = tot;
    tot += align_up(sizeof(StreamState));
    const size_t o_cnt = tot;
    tot += align_up((size_t)(5 * c.layers + 1) * sizeof(unsigned));
    const size_t o_arr = tot;
    tot += align_up((size_t)c.layers * m * G * sizeof(unsigned));
    cudaError_t e = cudaMalloc(&pe.sbuf, tot);
    if (e != cudaSuccess) return e;
    pe.sbuf_bytes = tot;
    // (on the context's stream: the plan's first launch is ordered after the clear)
    if ((e = cudaMemsetAsync(pe.sbuf, 0, tot, ctx->stream)) != cudaSuccess) return e;
    auto buf = [&](size_t o) { return reinterpret_cast<uint64_t*>(pe.sbuf + o); };
    uint64_t *qkv = buf(o_qkv), *att = buf(o_att), *mid = buf(o_mid), *act = buf(o_act),
             *res = buf(o_res), *part = buf(o_part), *ml = buf(o_ml);
    pe.st = reinterpret_cast<StreamState*>(pe.sbuf + o_st);
    pe.cnt = reinterpret_cast<unsigned*>(pe.sbuf + o_cnt);
    unsigned* arr = reinterpret_cast<unsigned*>(pe.sbuf + o_arr);
    const int es = c.weight_dtype == DEC_BF16 ? 2 : 4, vec = c.weight_dtype == DEC_BF16 ? 8 : 4;
    auto nj = [&](int K) { return (K / vec + 255) / 256; };

    ph.clear();
    for (int l = 0; l < c.layers; ++l) {
        const LayerW& W = ctx->L[l];
        SPhase p = {};
        // norm + q/k/v
        p.type = SP_GEMV;
        SGemv& g = p.g;
        g.W = talker ? W.qkv : W.in_proj;
        g.N = ctx->qkv_rows;
        g.K = h;
        g.unit = 1;
        g.pro = talker ? PRO_RMS : PRO_LN;
        g.nw = talker ? W.in_norm : W.ln1_w;
        g.nb = talker ? nullptr : W.ln1_b;
        g.eps = c.norm_eps;
        g.epi = EPI_STORE;
        g.x = l == 0 ? nullptr : res;
        g.ldx = h;
        g.x_layer = l - 1;
        g.y = qkv;
        g.ldy = ctx->qkv_rows;
        g.layer = l;
        p.nj = nj(g.K);
        ph.push_back(p);
        // attention, then the merge of its partials
        p = {};
        p.type = SP_ATTN;
        SAttn& a = p.a;
        a.mode = talker ? ATTN_TALKER : ATTN_RING;
        a.H = H;
        a.G = G;
        a.slots = ctx->slots;
        a.window = c.window;
        a.layer = l;
        a.qkv = qkv;
        a.ldqkv = ctx->qkv_rows;
        a.kc = ctx->kc + (size_t)l * kv_layer;
        a.vc = ctx->vc + (size_t)l * kv_layer;
        a.pr = talker ? nullptr : ctx->pr + (size_t)l * ctx->S * ctx->slots;
        a.qn = W.q_norm;
        a.kn = W.k_norm;
        a.eps = c.norm_eps;
        a.rope_cos = ctx->rope_cos;
        a.rope_sin = ctx->rope_sin;
        a.part = part;
        a.ml = ml;
        a.out = att;
        a.arr = arr + (size_t)l * m * G;
        ph.push_back(p);
        // o-proj + residual (codec: LayerScale)
        p = {};
        p.type = SP_GEMV;
        g = SGemv{};
        g.W = talker ? W.o : W.out_proj;
        g.N = h;
        g.K = qw;
        g.unit = 1;
        g.pro = PRO_NONE;
        g.epi = EPI_RESID;
        g.ls = talker ? nullptr : W.ls1;
        g.x = att;
        g.ldx = qw;
        g.x_layer = l;
        g.res = l == 0 ? nullptr : res;
        g.ldres = h;
        g.res_layer = l - 1;
        g.y = mid;
        g.ldy = h;
        g.layer = l;
        p.nj = nj(g.K);
        ph.push_back(p);
        // norm + gate/up + SwiGLU (codec: lin1 + GELU)
        p = {};
        p.type = SP_GEMV;
        g = SGemv{};
        g.W = talker ? W.gu : W.lin1;
        g.N = talker ? 2 * I : I;
        g.K = h;
        g.unit = talker ? 2 : 1;
        g.pro = talker ? PRO_RMS : PRO_LN;
        g.nw = talker ? W.post_norm : W.ln2_w;
        g.nb = talker ? nullptr : W.ln2_b;
        g.eps = c.norm_eps;
        g.epi = talker ? EPI_SWIGLU : EPI_GELU;
        g.x = mid;
        g.ldx = h;
        g.x_layer = l;
        g.y = act;
        g.ldy = I;
        g.layer = l;
        p.nj = nj(g.K);
        ph.push_back(p);
        // down + residual (codec: lin2 + LayerScale)
        p = {};
        p.type = SP_GEMV;
        g = SGemv{};
        g.W = talker ? W.down : W.lin2;
        g.N = h;
        g.K = I;
        g.unit = 1;
        g.pro = PRO_NONE;
        g.epi = EPI_RESID;
        g.ls = talker ? nullptr : W.ls2;
        g.x = act;
        g.ldx = I;
        g.x_layer = l;
        g.res = mid;
        g.ldres = h;
        g.res_layer = l;
        g.y = res;
        g.ldy = h;
        g.layer = l;
        g.tap = ctx->taps ? ctx->taps + (size_t)l * ctx->S * h : nullptr;
        g.ldtap = h;
        p.nj = nj(g.K);
        ph.push_back(p);
    }
    SPhase f = {};
    f.type = SP_FINAL;
    f.f.x = res;
    f.f.layer = c.layers - 1;
    f.f.h = h;
    f.f.w = ctx->final_norm;
    f.f.b = ctx->final_norm_b;
    f.f.eos_w = ctx->eos_w;
    f.f.eos = ctx->eos;
    f.f.eps = c.norm_eps;
    ph.push_back(f);
    (void)es;
    return cudaSuccess;
}

// The graph node the last launch captured on `s` became (null when `s` is not capturing).
cudaGraphNode_t last_captured(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t* deps = nullptr;
    size_t n = 0;
    if (cudaStreamGetCaptureInfo(s, &st, nullptr, nullptr, &deps, nullptr, &n) != cudaSuccess ||
        st != cudaStreamCaptureStatusActive || n != 1)
        return nullptr;
    return deps[0];
}

// Enqueue the multi-kernel plan of one step on `s`: six kernels per layer, then the final
// kernel.  Every kernel but the step's first is launched as a programmatic dependent of its
// predecessor.  With `io` (under stream capture) the nodes of the three launches that take the
// step's pointers are recorded in it.
cudaError_t enqueue_kernels(dec_ctx* ctx, int m, const float* x_in, float* out, cudaStream_t s,
                            const int32_t* rope_pos, PlanEntry* io = nullptr) {
    const dec_config& c = ctx->cfg;
    cudaError_t e;
    for (int l = 0; l < c.layers; ++l)
        for (int stage = 0; stage < 5; ++stage) {
            if ((e = launch_stage(ctx, l, stage, m, x_in, s, l > 0 || stage > 0, rope_pos)) !=
                cudaSuccess)
                return e;
            if (io && l == 0 && (stage == 0 || stage == 2)) io->io_node[stage / 2] = last_captured(s);
        }
    if ((e = launch_final(final_params(ctx, m, out), s, true)) != cudaSuccess) return e;
    if (io) io->io_node[2] = last_captured(s);
    return cudaSuccess;
}

// After the capture of a multi-kernel plan: the recorded nodes' launch parameters and captured
// arguments, checked against the pointers they must hold.
cudaError_t record_io_nodes(PlanEntry& pe) {
    for (int i = 0; i < 3; ++i) {
        if (!pe.io_node[i]) return cudaErrorInvalidValue;
        cudaError_t e = cudaGraphKernelNodeGetParams(pe.io_node[i], &pe.io_kp[i]);
        if (e != cudaSuccess) return e;
        if (!pe.io_kp[i].kernelParams || !pe.io_kp[i].kernelParams[0]) return cudaErrorInvalidValue;
    }
    for (int i = 0; i < 2; ++i) {
        memcpy(&pe.io_g[i], pe.io_kp[i].kernelParams[0], sizeof(GemvParams));
        // the tensor-core GEMV takes its TMA descriptor as a second argument
        pe.io_has_tm[i] = pe.io_kp[i].func == gemv_tc_kernel();
        if (pe.io_has_tm[i]) {
            if (!pe.io_kp[i].kernelParams[1]) return cudaErrorInvalidValue;
            memcpy(&pe.io_tm[i], pe.io_kp[i].kernelParams[1], sizeof(TmapBytes));
        }
    }
    memcpy(&pe.io_f, pe.io_kp[2].kernelParams[0], sizeof(FinalParams));
    if (pe.io_g[0].x != pe.x_in || pe.io_g[1].res != pe.x_in || pe.io_f.out != pe.out)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

// Point a multi-kernel plan's graph at new input/output buffers.
cudaError_t update_io_nodes(PlanEntry& pe, const float* x_in, float* out) {
    GemvParams g0 = pe.io_g[0], g1 = pe.io_g[1];
    FinalParams f = pe.io_f;
    g0.x = x_in;
    g1.res = x_in;
    f.out = out;
    TmapBytes t0 = pe.io_tm[0], t1 = pe.io_tm[1];
    void* a0[] = {&g0, &t0};  // the second entry only for the tensor-core GEMV
    void* a1[] = {&g1, &t1};
    void* a2[] = {&f};
    void** args[3] = {a0, a1, a2};
    for (int i = 0; i < 3; ++i) {
        cudaKernelNodeParams kp = pe.io_kp[i];
        kp.kernelParams = args[i];
        kp.extra = nullptr;
        cudaError_t e = cudaGraphExecKernelNodeSetParams(pe.exec, pe.io_node[i], &kp);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

StreamParams stream_params(dec_ctx* ctx, const PlanEntry& pe, const float* x_in, float* out,
                           int stall_phase = -1, int stall_polls = 0) {
    StreamParams sp = {};
    sp.phases = pe.phases;
    sp.n_phases = 5 * ctx->cfg.layers + 1;
    sp.m = pe.m;
    sp.x_in = x_in;
    sp.out = out;
    sp.len = ctx->len_dev;
    sp.max_pos = ctx->cfg.max_pos;
    sp.st = pe.st;
    sp.cnt = pe.cnt;
    sp.status = ctx->status;
    sp.wait_polls = stall_polls;
    sp.stall_phase = stall_phase;
    return sp;
}

// Enqueue one prefill block of m rows of stream `stream` (Qwen3-TTS talker on wgpu,
// forward_rows): the step's kernels with m rows of one stream, plus the append of the block's
// K/V rows before its attention, which then runs in ATTN_PREFILL mode (row r sees keys up to
// len + r).  The final kernel advances the stream by m.
cudaError_t enqueue_prefill_block(dec_ctx* ctx, int stream, int m, const float* x_in, float* out,
                                  cudaStream_t s, const int32_t* rope_pos) {
    const dec_config& c = ctx->cfg;
    cudaError_t e;
    for (int l = 0; l < c.layers; ++l)
        for (int stage = 0; stage < 5; ++stage) {
            const bool pdl = l > 0 || stage > 0;
            GemvParams g;
            AttnParams a;
            if (!stage_params(ctx, l, stage, m, x_in, g, a, rope_pos)) {
                g.tap = nullptr;  // taps hold the last step's rows, not a block's
                if ((e = launch_gemv(g, c.weight_dtype, ctx->num_sms, s, pdl)) != cudaSuccess) return e;
                continue;
            }
            a.mode = ATTN_PREFILL;
            a.stream = stream;
            if ((e = launch_prefill_append(a, s, pdl)) != cudaSuccess) return e;
            // not a programmatic dependent: the attention stages cache rows before its
            // griddepcontrol.wait, and the append above writes this block's rows
            if ((e = launch_attention(a, s, false)) != cudaSuccess) return e;
            if ((e = launch_attention_merge(a, s, true)) != cudaSuccess) return e;
        }
    FinalParams f = final_params(ctx, m, out);
    f.advance_stream = stream;
    return launch_final(f, s, true);
}

// Enqueue one step of a plan: the streamed kernel when the plan has a phase list, else the
// kernels one by one.
cudaError_t enqueue_step(dec_ctx* ctx, PlanEntry& pe, const float* x_in, float* out,
                         cudaStream_t s, bool record = false, int stall_phase = -1,
                         int stall_polls = 0) {
    if (!pe.phases) return enqueue_kernels(ctx, pe.m, x_in, out, s, pe.rope, record ? &pe : nullptr);
    return launch_stream_step(stream_params(ctx, pe, x_in, out, stall_phase, stall_polls),
                              ctx->cfg.weight_dtype, pe.m, ctx->cfg.head_dim, ctx->step_grid[pe.m], s);
}

// Whether steps of m rows take the streamed kernel: m <= 2, the kernel launchable here, and
// every GEMV, head group and output row within its limits.
bool uses_stream(const dec_ctx* ctx, int m) {
    if (m < 1 || m > 2 || ctx->step_grid[m] <= 0) return false;
    const dec_config& c = ctx->cfg;
    const int dt = c.weight_dtype;
    // the attention key split is 32-bit: keys of all streams and kv heads times (grid + 1)
    if ((uint64_t)m * c.kv_heads * ctx->slots * (uint64_t)(ctx->step_grid[m] + 1) >= (1ull << 32))
        return false;
    return c.layers <= kStreamMaxLayers && c.hidden <= 8192 && c.q_heads / c.kv_heads <= kMaxGroup &&
           stream_gemv_ok(dt, c.hidden) && stream_gemv_ok(dt, c.inter) &&
           stream_gemv_ok(dt, c.q_heads * c.head_dim);
}

// The plan for (m, x_in, out, rope): found in the cache or built (phase list uploaded, graph
// captured).  Steps with per-axis rotary positions take the multi-kernel plan.
PlanEntry* get_plan(dec_ctx* ctx, int m, const float* x_in, float* out, const int32_t* rope,
                    cudaError_t* err) {
    for (auto& e : ctx->plans)
        if (e.m == m && e.rope == rope) return &e;
    PlanEntry pe = {};
    pe.m = m;
    pe.x_in = x_in;
    pe.out = out;
    pe.rope = rope;
    if (!rope && uses_stream(ctx, m)) {
        std::vector<SPhase> ph;
        if ((*err = build_stream_plan(ctx, m, pe, ph)) != cudaSuccess) {
            destroy_plan(pe);
            return nullptr;
        }
        const size_t bytes = ph.size() * sizeof(SPhase);
        if ((*err = cudaMalloc(&pe.phases, bytes)) != cudaSuccess ||
            (*err = cudaMemcpy(pe.phases, ph.data(), bytes, cudaMemcpyHostToDevice)) != cudaSuccess) {
            destroy_plan(pe);
            return nullptr;
        }
    }
    if (!(ctx->cfg.flags & DEC_FLAG_NO_GRAPH)) {
        *err = cudaStreamBeginCapture(ctx->cap_stream, cudaStreamCaptureModeThreadLocal);
        if (*err != cudaSuccess) {
            destroy_plan(pe);
            return nullptr;
        }
        cudaError_t e = enqueue_step(ctx, pe, x_in, out, ctx->cap_stream, true);
        cudaGraph_t graph = nullptr;
        cudaError_t e2 = cudaStreamEndCapture(ctx->cap_stream, &graph);
        if (e != cudaSuccess || e2 != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            *err = e != cudaSuccess ? e : e2;
            destroy_plan(pe);
            return nullptr;
        }
        if (pe.phases) {  // the single kernel node, for in-place pointer updates
            size_t n = 1;
            *err = cudaGraphGetNodes(graph, &pe.node, &n);
            if (*err == cudaSuccess && n != 1) *err = cudaErrorInvalidValue;
            if (*err == cudaSuccess) *err = cudaGraphKernelNodeGetParams(pe.node, &pe.kp);
        } else {
            *err = record_io_nodes(pe);
        }
        if (*err == cudaSuccess) *err = cudaGraphInstantiate(&pe.exec, graph, 0);
        pe.graph = graph;  // keeps the node handles valid for updates
        if (*err != cudaSuccess) {
            destroy_plan(pe);
            return nullptr;
        }
    }
    if (ctx->plans.size() >= 8) {
        // a graph still queued on the stream is freed when it completes; a phase list is not
        // (cudaFree waits for the device)
        destroy_plan(ctx->plans.front());
        ctx->plans.erase(ctx->plans.begin());
    }
    ctx->plans.push_back(pe);
    return &ctx->plans.back();
}

dec_status check_step_args(dec_ctx* ctx, int m, const int32_t* pos) {
    if (m < 1 || m > ctx->S) return fail(ctx, DEC_E_ARG, "m=%d outside 1..%d", m, ctx->S);
    if (!pos) return fail(ctx, DEC_E_ARG, "pos is NULL");
    for (int i = 0; i < m; ++i) {
        if (pos[i] != ctx->len_host[i])
            return fail(ctx, DEC_E_POS, "stream %d: pos %d != length %d (positions must be contiguous)",
                        i, pos[i], ctx->len_host[i]);
        if (ctx->cfg.kind == DEC_QWEN3_TALKER && pos[i] + 1 > ctx->cfg.max_pos)
            return fail(ctx, DEC_E_CAPACITY, "stream %d: cache length %d exceeds max_pos %d", i,
                        pos[i] + 1, ctx->cfg.max_pos);
        if (ctx->cfg.kind == DEC_CODEC_WINDOWED && pos[i] >= ctx->cfg.max_pos)
            return fail(ctx, DEC_E_CAPACITY, "stream %d: position %d reaches max_pos %d", i, pos[i],
                        ctx->cfg.max_pos);
    }
    return DEC_OK;
}

dec_status run_step(dec_ctx* ctx, int m, const float* x_in, float* out,
                    const int32_t* rope = nullptr) {
    cudaError_t e = cudaSuccess;
    PlanEntry* pe = get_plan(ctx, m, x_in, out, rope, &e);
    if (!pe) return cuda_fail(ctx, e, "step plan");
    if (pe->exec && (pe->x_in != x_in || pe->out != out)) {
        // new input/output buffers: update the kernel nodes' arguments in place
        if (pe->phases) {
            StreamParams sp = stream_params(ctx, *pe, x_in, out);
            void* args[] = {&sp};
            cudaKernelNodeParams kp = pe->kp;
            kp.kernelParams = args;
            kp.extra = nullptr;
            e = cudaGraphExecKernelNodeSetParams(pe->exec, pe->node, &kp);
        } else {
            e = update_io_nodes(*pe, x_in, out);
        }
        if (e != cudaSuccess) {  // the graph may hold a mix of old and new pointers: drop it
            destroy_plan(*pe);
            ctx->plans.erase(ctx->plans.begin() + (pe - ctx->plans.data()));
            return cuda_fail(ctx, e, "step graph update");
        }
        pe->x_in = x_in;
        pe->out = out;
    }
    if (pe->phases) {
        // the tags of the streamed plan hold (launches + 1) << 8 in 32 bits: start the buffers
        // and the count over long before the tag could come round to an old value
        if (++pe->launches >= (1LL << 22)) {
            e = cudaMemsetAsync(pe->sbuf, 0, pe->sbuf_bytes, ctx->stream);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "tag reset");
            pe->launches = 1;
        }
    }
    if (pe->phases && ctx->stall_phase >= 0) {
        // dec_inject_stall: this one step runs outside the graph with its stalled phase
        e = enqueue_step(ctx, *pe, x_in, out, ctx->stream, false, ctx->stall_phase, ctx->stall_polls);
        ctx->stall_phase = -1;
    } else {
        e = pe->exec ? cudaGraphLaunch(pe->exec, ctx->stream) : enqueue_step(ctx, *pe, x_in, out, ctx->stream);
    }
    if (e != cudaSuccess) return cuda_fail(ctx, e, "step launch");
    for (int i = 0; i < m; ++i) ctx->len_host[i] += 1;
    return DEC_OK;
}

dec_status read_status(dec_ctx* ctx) {
    const unsigned st = *ctx->status_host;
    if (st == 0) return DEC_OK;
    *ctx->status_host = 0;
    cudaMemset(ctx->status, 0, sizeof(unsigned));
    return fail(ctx, DEC_E_DEVICE_CHECK, "device check fired:%s%s",
                (st & CHECK_WAIT_LIMIT) ? " wait-limit" : "", (st & CHECK_BOUNDS) ? " bounds" : "");
}

}  // namespace

namespace dec {
// record a failure of a context-free entry point (read back with dec_last_error(NULL))
dec_status stateless_fail(dec_status st, const char* msg) { return fail(nullptr, st, "%s", msg); }
}  // namespace dec

// =============================================================================================
// exported entry points
// =============================================================================================
extern "C" {

dec_status dec_create(const dec_config* cfg, const dec_weights* w, void* stream, dec_ctx** out) {
    g_create_error.clear();
    if (!out) return fail(nullptr, DEC_E_ARG, "out is NULL");
    *out = nullptr;
    dec_status st = validate_config(cfg);
    if (st != DEC_OK) return st;
    if (!w || !w->layers) return fail(nullptr, DEC_E_ARG, "weights are NULL");
    const dec_config c = *cfg;
    const bool talker = c.kind == DEC_QWEN3_TALKER;
    const int h = c.hidden, d = c.head_dim, H = c.q_heads, G = c.kv_heads, I = c.inter;
    for (int l = 0; l < c.layers; ++l) {
        const dec_layer_weights& lw = w->layers[l];
        const void* need_t[] = {lw.q, lw.k, lw.v, lw.o, lw.gate, lw.up, lw.down,
                                lw.in_norm, lw.q_norm, lw.k_norm, lw.post_norm};
        const void* need_c[] = {lw.in_proj, lw.out_proj, lw.lin1, lw.lin2, lw.ln1_w,
                                lw.ln1_b, lw.ln2_w, lw.ln2_b};  // ls1 / ls2 optional
        if (talker) {
            for (const void* p : need_t)
                if (!p) return fail(nullptr, DEC_E_ARG, "layer %d: a talker weight is NULL", l);
        } else {
            for (const void* p : need_c)
                if (!p) return fail(nullptr, DEC_E_ARG, "layer %d: a codec weight is NULL", l);
        }
    }
    if (talker && !w->final_norm) return fail(nullptr, DEC_E_ARG, "final_norm is NULL");
    if (!talker && w->final_norm && !w->final_norm_b)
        return fail(nullptr, DEC_E_ARG, "codec final_norm (LayerNorm) needs final_norm_b");

    dec_ctx* ctx = new dec_ctx();
    ctx->cfg = c;
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->S = c.max_streams;
    ctx->slots = talker ? c.max_pos : c.ring;
    ctx->qkv_rows = talker ? (H + 2 * G) * d : 3 * h;
    ctx->num_sms = device_sm_count();
    ctx->len_host.assign(ctx->S, 0);
    auto bail = [&](dec_status s) {
        g_create_error = ctx->err;
        dec_destroy(ctx);
        return s;
    };
    if (ctx->num_sms <= 0) {
        fail(ctx, DEC_E_CUDA, "no CUDA device");
        return bail(DEC_E_CUDA);
    }
    cudaError_t e = configure_kernels();
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "kernel attributes"));
    ctx->max_chunks = (ctx->slots + kAttnChunk - 1) / kAttnChunk;
    if (c.flags & DEC_FLAG_PERSISTENT)
        for (int mm = 1; mm <= std::min(2, ctx->S); ++mm)
            ctx->step_grid[mm] = stream_grid(c.weight_dtype, mm, d, ctx->num_sms);
    e = cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "capture stream"));
    if ((e = cudaMallocHost(&ctx->status_host, sizeof(unsigned))) != cudaSuccess)
        return bail(cuda_fail(ctx, e, "pinned status word"));
    *ctx->status_host = 0;

    // ---- weight arena ------------------------------------------------------------------------
    const size_t es = c.weight_dtype == DEC_BF16 ? 2 : 4;
    const int qw = H * d, kvw = G * d;
    struct Off {
        size_t a, b, cc, dd, f[6];
    };
    std::vector<Off> offs(c.layers);
    size_t tot = 0;
    auto take = [&](size_t bytes) {
        const size_t o = tot;
        tot += align_up(bytes);
        return o;
    };
    for (int l = 0; l < c.layers; ++l) {
        Off& o = offs[l];
        if (talker) {
            o.a = take((size_t)(qw + 2 * kvw) * h * es);
            o.b = take((size_t)h * qw * es);
            o.cc = take((size_t)2 * I * h * es);
            o.dd = take((size_t)h * I * es);
            o.f[0] = take(h * 4);
            o.f[1] = take(h * 4);
            o.f[2] = take(d * 4);
            o.f[3] = take(d * 4);
        } else {
            o.a = take((size_t)3 * h * h * es);
            o.b = take((size_t)h * h * es);
            o.cc = take((size_t)I * h * es);
            o.dd = take((size_t)h * I * es);
            for (int j = 0; j < 6; ++j) o.f[j] = take(h * 4);
        }
    }
    const size_t fn_off = take(h * 4), fnb_off = take(h * 4), eos_off = take(h * 4);
    if ((e = cudaMalloc(&ctx->arena, tot)) != cudaSuccess) return bail(cuda_fail(ctx, e, "weight arena"));
    cudaStream_t s = ctx->stream;
    auto cp = [&](size_t off, const void* src, size_t bytes) {
        return cudaMemcpyAsync(ctx->arena + off, src, bytes, cudaMemcpyDeviceToDevice, s);
    };
    ctx->L.resize(c.layers);
    for (int l = 0; l < c.layers; ++l) {
        const dec_layer_weights& lw = w->layers[l];
        const Off& o = offs[l];
        LayerW& L = ctx->L[l];
        L = LayerW{};
        if (talker) {
            const size_t rb = (size_t)h * es;
            if ((e = cp(o.a, lw.q, (size_t)qw * rb)) != cudaSuccess ||
                (e = cp(o.a + (size_t)qw * rb, lw.k, (size_t)kvw * rb)) != cudaSuccess ||
                (e = cp(o.a + (size_t)(qw + kvw) * rb, lw.v, (size_t)kvw * rb)) != cudaSuccess ||
                (e = cp(o.b, lw.o, (size_t)h * qw * es)) != cudaSuccess ||
                // gate row j -> row 2j, up row j -> row 2j+1
                (e = cudaMemcpy2DAsync(ctx->arena + o.cc, 2 * rb, lw.gate, rb, rb, I,
                                       cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
                (e = cudaMemcpy2DAsync(ctx->arena + o.cc + rb, 2 * rb, lw.up, rb, rb, I,
                                       cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
                (e = cp(o.dd, lw.down, (size_t)h * I * es)) != cudaSuccess ||
                (e = cp(o.f[0], lw.in_norm, h * 4)) != cudaSuccess ||
                (e = cp(o.f[1], lw.post_norm, h * 4)) != cudaSuccess ||
                (e = cp(o.f[2], lw.q_norm, d * 4)) != cudaSuccess ||
                (e = cp(o.f[3], lw.k_norm, d * 4)) != cudaSuccess)
                return bail(cuda_fail(ctx, e, "weight copy"));
            L.qkv = ctx->arena + o.a;
            L.o = ctx->arena + o.b;
            L.gu = ctx->arena + o.cc;
            L.down = ctx->arena + o.dd;
            L.in_norm = reinterpret_cast<const float*>(ctx->arena + o.f[0]);
            L.post_norm = reinterpret_cast<const float*>(ctx->arena + o.f[1]);
            L.q_norm = reinterpret_cast<const float*>(ctx->arena + o.f[2]);
            L.k_norm = reinterpret_cast<const float*>(ctx->arena + o.f[3]);
        } else {
            const float* vecs[6] = {lw.ln1_w, lw.ln1_b, lw.ln2_w, lw.ln2_b, lw.ls1, lw.ls2};
            if ((e = cp(o.a, lw.in_proj, (size_t)3 * h * h * es)) != cudaSuccess ||
                (e = cp(o.b, lw.out_proj, (size_t)h * h * es)) != cudaSuccess ||
                (e = cp(o.cc, lw.lin1, (size_t)I * h * es)) != cudaSuccess ||
                (e = cp(o.dd, lw.lin2, (size_t)h * I * es)) != cudaSuccess)
                return bail(cuda_fail(ctx, e, "weight copy"));
            for (int j = 0; j < 6; ++j)
                if (vecs[j] && (e = cp(o.f[j], vecs[j], h * 4)) != cudaSuccess)
                    return bail(cuda_fail(ctx, e, "weight copy"));
            L.in_proj = ctx->arena + o.a;
            L.out_proj = ctx->arena + o.b;
            L.lin1 = ctx->arena + o.cc;
            L.lin2 = ctx->arena + o.dd;
            const float** dst[6] = {&L.ln1_w, &L.ln1_b, &L.ln2_w, &L.ln2_b, &L.ls1, &L.ls2};
            for (int j = 0; j < 6; ++j)  // a missing LayerScale stays NULL (a scale of one)
                *dst[j] = vecs[j] ? reinterpret_cast<const float*>(ctx->arena + o.f[j]) : nullptr;
        }
    }
    if (w->final_norm) {  // talker: final RMSNorm; codec: the FlowLM head's out_norm
        if ((e = cp(fn_off, w->final_norm, h * 4)) != cudaSuccess)
            return bail(cuda_fail(ctx, e, "weight copy"));
        ctx->final_norm = reinterpret_cast<const float*>(ctx->arena + fn_off);
    }
    if (!talker && w->final_norm) {
        if ((e = cp(fnb_off, w->final_norm_b, h * 4)) != cudaSuccess)
            return bail(cuda_fail(ctx, e, "weight copy"));
        ctx->final_norm_b = reinterpret_cast<const float*>(ctx->arena + fnb_off);
    }
    if (!talker && w->eos_w) {
        if ((e = cp(eos_off, w->eos_w, h * 4)) != cudaSuccess)
            return bail(cuda_fail(ctx, e, "weight copy"));
        ctx->eos_w = reinterpret_cast<const float*>(ctx->arena + eos_off);
        ctx->eos_b = w->eos_b;
    }

    // ---- state: caches, stamps, tables, scratch -------------------------------------------------
    const int S = ctx->S;
    const size_t kv_elems = (size_t)c.layers * S * G * ctx->slots * d;
    tot = 0;
    const size_t o_kc = take(kv_elems * 4), o_vc = take(kv_elems * 4);
    const size_t o_pr = talker ? 0 : take((size_t)c.layers * S * ctx->slots * 4);
    const size_t half = d / 2;
    const size_t o_cos = take((size_t)c.max_pos * half * 4), o_sin = take((size_t)c.max_pos * half * 4);
    const size_t o_axis = take(half * 4);
    // a prefill block takes up to 8 rows, as many as the m > 2 GEMV's shared-memory stage allows
    if (talker) {
        const int widest = std::max(std::max(h, I), qw);
        for (int rows = 8; rows >= 1 && !ctx->prefill_rows; --rows)
            if (gemv_smem_bytes(rows, widest) <= (size_t)kGemvMaxSmem) ctx->prefill_rows = rows;
    }
    const int R = ctx->R = std::max(S, ctx->prefill_rows);
    const size_t o_x = take((size_t)R * h * 4), o_qkv = take((size_t)R * ctx->qkv_rows * 4);
    const size_t o_att = take((size_t)R * qw * 4), o_act = take((size_t)R * I * 4);
    const size_t o_part = take(attention_part_bytes(R, H, ctx->max_chunks, d));
    const size_t o_ml = take(attention_ml_bytes(R, H, ctx->max_chunks));
    const size_t o_len = take((size_t)S * 4), o_st = take(4);
    const size_t o_eos = take((size_t)S * 4);
    const size_t o_taps = (c.flags & DEC_FLAG_TAPS) ? take((size_t)c.layers * S * h * 4) : 0;
    const size_t o_in = take((size_t)S * h * 4), o_out = take((size_t)S * h * 4);
    // tensor-core GEMV scratch (more than two rows): partial tiles of the CTAs and one ticket per
    // 128-row tile
    size_t o_mpart = 0, o_mtick = 0;
    if (R > 2) {
        const size_t shapes[4][2] = {{(size_t)ctx->qkv_rows, (size_t)h},
                                     {(size_t)h, (size_t)qw},
                                     {(size_t)(talker ? 2 * I : I), (size_t)h},
                                     {(size_t)h, (size_t)I}};
        size_t most = 0, rows = 0;
        for (auto& sh : shapes) {
            most = std::max(most, sh[0] * sh[1]);
            rows = std::max(rows, sh[0]);
        }
        // the tensor-core GEMV: up to 16 partial tiles of 128 rows x 8 streams per CTA
        ctx->mpart_floats = std::max(most / 32, (size_t)ctx->num_sms * 16 * 128 * 8);
        ctx->mtick_n = (int)(rows / 8 + 1);
        o_mpart = take(ctx->mpart_floats * 4);
        o_mtick = take((size_t)ctx->mtick_n * 4);
    }
    if ((e = cudaMalloc(&ctx->state, tot)) != cudaSuccess) return bail(cuda_fail(ctx, e, "state"));
    char* b = ctx->state;
    ctx->kc = reinterpret_cast<float*>(b + o_kc);
    ctx->vc = reinterpret_cast<float*>(b + o_vc);
    ctx->pr = talker ? nullptr : reinterpret_cast<uint32_t*>(b + o_pr);
    ctx->rope_cos = reinterpret_cast<float*>(b + o_cos);
    ctx->rope_sin = reinterpret_cast<float*>(b + o_sin);
    ctx->rope_axis = reinterpret_cast<int32_t*>(b + o_axis);  // zero: every frequency on axis t
    ctx->xres = reinterpret_cast<float*>(b + o_x);
    ctx->qkv = reinterpret_cast<float*>(b + o_qkv);
    ctx->attn = reinterpret_cast<float*>(b + o_att);
    ctx->act = reinterpret_cast<float*>(b + o_act);
    ctx->part = reinterpret_cast<float*>(b + o_part);
    ctx->part_ml = reinterpret_cast<float*>(b + o_ml);
    ctx->len_dev = reinterpret_cast<int32_t*>(b + o_len);
    ctx->status = reinterpret_cast<unsigned*>(b + o_st);
    ctx->eos = reinterpret_cast<float*>(b + o_eos);
    ctx->taps = (c.flags & DEC_FLAG_TAPS) ? reinterpret_cast<float*>(b + o_taps) : nullptr;
    ctx->io_in = reinterpret_cast<float*>(b + o_in);
    ctx->io_out = reinterpret_cast<float*>(b + o_out);
    if (R > 2) {
        ctx->mpart = reinterpret_cast<float*>(b + o_mpart);
        ctx->mtick = reinterpret_cast<unsigned*>(b + o_mtick);  // zeroed with the state below
    }
    // everything zero (K/V, scratch, lengths, status), then the stamps to empty
    if ((e = cudaMemsetAsync(ctx->state, 0, tot, s)) != cudaSuccess)
        return bail(cuda_fail(ctx, e, "state clear"));
    if (!talker && (e = cudaMemsetAsync(ctx->pr, 0xFF, (size_t)c.layers * S * ctx->slots * 4, s)) !=
                       cudaSuccess)
        return bail(cuda_fail(ctx, e, "stamp clear"));
    std::vector<float> tc, ts;
    build_rope_tables(c.max_pos, d, c.rope_theta, tc, ts);
    if ((e = cudaMemcpyAsync(ctx->rope_cos, tc.data(), tc.size() * 4, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(ctx->rope_sin, ts.data(), ts.size() * 4, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess)
        return bail(cuda_fail(ctx, e, "rope tables"));
    // TMA descriptors for the tensor-core GEMV (DEC_FLAG_TENSOR_GEMV: steps or prefill blocks of
    // more than two rows over bf16 weights)
    if ((c.flags & DEC_FLAG_TENSOR_GEMV) && R > 2 && c.weight_dtype == DEC_BF16) {
        const size_t n = (size_t)c.layers * 4;
        std::vector<TmapBytes> maps(n);
        std::vector<uint8_t> ok(n, 0);
        for (int l = 0; l < c.layers; ++l)
            for (int st : {0, 2, 3, 4}) {
                GemvParams g;
                AttnParams a;
                stage_params(ctx, l, st, R, ctx->io_in, g, a);
                const size_t slot = (size_t)l * 4 + (st == 0 ? 0 : st - 1);
                ok[slot] = gemv_tc_encode(g.W, g.N, g.K, maps[slot].b) == cudaSuccess;
            }
        (void)cudaGetLastError();  // a matrix the descriptors do not serve is not an error
        ctx->tmaps.swap(maps);
        ctx->tmap_ok.swap(ok);
    }
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return bail(cuda_fail(ctx, e, "create sync"));
    *out = ctx;
    return DEC_OK;
}

void dec_destroy(dec_ctx* ctx) {
    if (!ctx) return;
    if (ctx->stream || ctx->cap_stream) cudaStreamSynchronize(ctx->stream);
    destroy_plans(ctx);
    if (ctx->cap_stream) cudaStreamDestroy(ctx->cap_stream);
    if (ctx->arena) cudaFree(ctx->arena);
    if (ctx->state) cudaFree(ctx->state);
    if (ctx->status_host) cudaFreeHost(ctx->status_host);
    delete ctx;
}

const char* dec_last_error(const dec_ctx* ctx) {
    return ctx ? ctx->err.c_str() : g_create_error.c_str();
}

dec_status dec_set_stream(dec_ctx* ctx, void* stream) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    ctx->stream = static_cast<cudaStream_t>(stream);
    return DEC_OK;
}

dec_status dec_reset(dec_ctx* ctx, int stream) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (stream < 0 || stream >= ctx->S)
        return fail(ctx, DEC_E_ARG, "stream %d outside 0..%d", stream, ctx->S - 1);
    const dec_config& c = ctx->cfg;
    const size_t per = (size_t)c.kv_heads * ctx->slots * c.head_dim * 4;
    for (int l = 0; l < c.layers; ++l) {
        const size_t off = ((size_t)l * ctx->S + stream) * per;
        CUDA_TRY(ctx, cudaMemsetAsync(reinterpret_cast<char*>(ctx->kc) + off, 0, per, ctx->stream),
                 "reset K");
        CUDA_TRY(ctx, cudaMemsetAsync(reinterpret_cast<char*>(ctx->vc) + off, 0, per, ctx->stream),
                 "reset V");
    }
    ResetParams rp = {c.layers, ctx->S, stream, ctx->slots, ctx->pr, ctx->len_dev};
    CUDA_TRY(ctx, launch_reset_stamps(rp, ctx->stream), "reset stamps");
    ctx->len_host[stream] = 0;
    return DEC_OK;
}

dec_status dec_prefill_kv(dec_ctx* ctx, int stream, const float* k, const float* v, int n_pos) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (stream < 0 || stream >= ctx->S)
        return fail(ctx, DEC_E_ARG, "stream %d outside 0..%d", stream, ctx->S - 1);
    if (n_pos < 0) return fail(ctx, DEC_E_ARG, "n_pos < 0");
    if (n_pos > 0 && (!k || !v)) return fail(ctx, DEC_E_ARG, "k or v is NULL");
    const dec_config& c = ctx->cfg;
    if (c.kind == DEC_QWEN3_TALKER && n_pos > c.max_pos)
        return fail(ctx, DEC_E_CAPACITY, "prefill of %d positions exceeds max_pos %d", n_pos, c.max_pos);
    if (c.kind == DEC_CODEC_WINDOWED && n_pos > c.ring)
        return fail(ctx, DEC_E_CAPACITY, "prefill of %d positions exceeds the %d-slot ring", n_pos,
                    c.ring);
    if (c.kind == DEC_CODEC_WINDOWED && n_pos > c.max_pos)
        return fail(ctx, DEC_E_CAPACITY, "prefill of %d positions reaches max_pos %d", n_pos,
                    c.max_pos);
    dec_status st = dec_reset(ctx, stream);
    if (st != DEC_OK) return st;
    if (n_pos > 0) {
        PrefillParams p = {c.layers, n_pos, c.kv_heads, c.head_dim, ctx->slots, ctx->S, stream,
                           k, v, ctx->kc, ctx->vc, ctx->pr, ctx->len_dev};
        CUDA_TRY(ctx, launch_prefill(p, ctx->stream), "prefill");
    }
    ctx->len_host[stream] = n_pos;
    return DEC_OK;
}

dec_status dec_prefill(dec_ctx* ctx, int stream, int n, const float* x, float* out) {
    return dec_prefill_mrope(ctx, stream, n, x, nullptr, out);
}

dec_status dec_prefill_mrope(dec_ctx* ctx, int stream, int n, const float* x,
                             const int32_t* rope_pos, float* out) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (ctx->cfg.kind != DEC_QWEN3_TALKER || ctx->prefill_rows < 1)
        return fail(ctx, DEC_E_UNSUPPORTED, "prefill blocks are a talker operation (a KV ring takes one position per step)");
    if (stream < 0 || stream >= ctx->S)
        return fail(ctx, DEC_E_ARG, "stream %d outside 0..%d", stream, ctx->S - 1);
    if (n < 1 || !x || !out) return fail(ctx, DEC_E_ARG, "n < 1 or a NULL buffer");
    if (!aligned16(x) || !aligned16(out)) return fail(ctx, DEC_E_ARG, "x and out must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(rope_pos) & 3u)
        return fail(ctx, DEC_E_ARG, "rope_pos must be 4-byte aligned");
    if ((long long)ctx->len_host[stream] + n > ctx->cfg.max_pos)
        return fail(ctx, DEC_E_CAPACITY, "stream %d: length %d + %d exceeds max_pos %d", stream,
                    ctx->len_host[stream], n, ctx->cfg.max_pos);
    const size_t h = (size_t)ctx->cfg.hidden;
    for (int r0 = 0; r0 < n; r0 += ctx->prefill_rows) {
        const int m = std::min(ctx->prefill_rows, n - r0);
        CUDA_TRY(ctx, enqueue_prefill_block(ctx, stream, m, x + (size_t)r0 * h, out + (size_t)r0 * h,
                                            ctx->stream, rope_pos ? rope_pos + 3 * (size_t)r0 : nullptr),
                 "prefill launch");
    }
    ctx->len_host[stream] += n;
    return DEC_OK;
}

int dec_prefill_block_rows(const dec_ctx* ctx) { return ctx ? ctx->prefill_rows : 0; }

dec_status dec_read_eos(dec_ctx* ctx, int m, float* dst_host) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (!ctx->eos_w) return fail(ctx, DEC_E_UNSUPPORTED, "the context has no EOS row");
    if (m < 1 || m > ctx->S || !dst_host) return fail(ctx, DEC_E_ARG, "bad m or NULL dst");
    CUDA_TRY(ctx, cudaStreamSynchronize(ctx->stream), "stream sync");
    CUDA_TRY(ctx, cudaMemcpy(dst_host, ctx->eos, (size_t)m * 4, cudaMemcpyDeviceToHost), "eos read");
    for (int i = 0; i < m; ++i) dst_host[i] += ctx->eos_b;
    return DEC_OK;
}

dec_status dec_step(dec_ctx* ctx, int m, const float* x_in, const int32_t* pos, float* hidden_out) {
    return dec_step_mrope(ctx, m, x_in, pos, nullptr, hidden_out);
}

dec_status dec_set_mrope(dec_ctx* ctx, const int32_t* axis_host, int n) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (ctx->cfg.kind != DEC_QWEN3_TALKER)
        return fail(ctx, DEC_E_UNSUPPORTED, "multimodal rope is a talker operation");
    const int half = ctx->cfg.head_dim / 2;
    std::vector<int32_t> axis(half, 0);
    if (axis_host) {
        if (n != half) return fail(ctx, DEC_E_ARG, "the axis map has %d entries, head_dim/2 = %d", n, half);
        for (int i = 0; i < half; ++i) {
            if (axis_host[i] < 0 || axis_host[i] > 2)
                return fail(ctx, DEC_E_ARG, "axis[%d] = %d outside 0..2", i, axis_host[i]);
            axis[i] = axis_host[i];
        }
    }
    CUDA_TRY(ctx, cudaMemcpyAsync(ctx->rope_axis, axis.data(), (size_t)half * 4,
                                  cudaMemcpyHostToDevice, ctx->stream),
             "axis map copy");
    CUDA_TRY(ctx, cudaStreamSynchronize(ctx->stream), "axis map sync");
    return DEC_OK;
}

dec_status dec_step_mrope(dec_ctx* ctx, int m, const float* x_in, const int32_t* pos,
                          const int32_t* rope_pos, float* hidden_out) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (rope_pos && ctx->cfg.kind != DEC_QWEN3_TALKER)
        return fail(ctx, DEC_E_UNSUPPORTED, "multimodal rope is a talker operation");
    if (reinterpret_cast<uintptr_t>(rope_pos) & 3u)
        return fail(ctx, DEC_E_ARG, "rope_pos must be 4-byte aligned");
    dec_status st = check_step_args(ctx, m, pos);
    if (st != DEC_OK) return st;
    if (!x_in || !hidden_out) return fail(ctx, DEC_E_ARG, "x_in or hidden_out is NULL");
    if (!aligned16(x_in)) return fail(ctx, DEC_E_ARG, "x_in must be 16-byte aligned");
    const size_t bytes = (size_t)m * ctx->cfg.hidden * 4;
    const char* a = reinterpret_cast<const char*>(x_in);
    const char* o = reinterpret_cast<const char*>(hidden_out);
    if (a < o + bytes && o < a + bytes) return fail(ctx, DEC_E_ARG, "x_in and hidden_out overlap");
    return run_step(ctx, m, x_in, hidden_out, rope_pos);
}

dec_status dec_step_host(dec_ctx* ctx, int m, const float* x_in_host, const int32_t* pos,
                         float* hidden_out_host) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    dec_status st = check_step_args(ctx, m, pos);
    if (st != DEC_OK) return st;
    if (!x_in_host || !hidden_out_host) return fail(ctx, DEC_E_ARG, "x_in or hidden_out is NULL");
    const size_t bytes = (size_t)m * ctx->cfg.hidden * 4;
    CUDA_TRY(ctx, cudaMemcpyAsync(ctx->io_in, x_in_host, bytes, cudaMemcpyHostToDevice, ctx->stream),
             "input copy");
    st = run_step(ctx, m, ctx->io_in, ctx->io_out);
    if (st != DEC_OK) return st;
    CUDA_TRY(ctx, cudaMemcpyAsync(hidden_out_host, ctx->io_out, bytes, cudaMemcpyDeviceToHost,
                                  ctx->stream),
             "output copy");
    CUDA_TRY(ctx, cudaMemcpyAsync(ctx->status_host, ctx->status, sizeof(unsigned),
                                  cudaMemcpyDeviceToHost, ctx->stream),
             "status copy");
    CUDA_TRY(ctx, cudaStreamSynchronize(ctx->stream), "step sync");
    return read_status(ctx);
}

dec_status dec_sync(dec_ctx* ctx) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    CUDA_TRY(ctx, cudaStreamSynchronize(ctx->stream), "stream sync");
    CUDA_TRY(ctx, cudaMemcpy(ctx->status_host, ctx->status, sizeof(unsigned), cudaMemcpyDeviceToHost),
             "status read");
    return read_status(ctx);
}

int dec_get_len(const dec_ctx* ctx, int stream) {
    if (!ctx || stream < 0 || stream >= ctx->S) return -1;
    return ctx->len_host[stream];
}

dec_status dec_read_kv(dec_ctx* ctx, int layer, int stream, int position, float* k_host,
                       float* v_host) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    const dec_config& c = ctx->cfg;
    if (layer < 0 || layer >= c.layers || stream < 0 || stream >= ctx->S || position < 0 ||
        !k_host || !v_host)
        return fail(ctx, DEC_E_ARG, "bad layer/stream/position or NULL destination");
    const int slot = c.kind == DEC_CODEC_WINDOWED ? position % ctx->slots : position;
    if (slot >= ctx->slots) return fail(ctx, DEC_E_ARG, "position %d outside the cache", position);
    CUDA_TRY(ctx, cudaStreamSynchronize(ctx->stream), "stream sync");
    const size_t d = c.head_dim;
    const size_t base = (((size_t)layer * ctx->S + stream) * c.kv_heads) * ctx->slots * d + slot * d;
    CUDA_TRY(ctx, cudaMemcpy2D(k_host, d * 4, ctx->kc + base, ctx->slots * d * 4, d * 4, c.kv_heads,
                               cudaMemcpyDeviceToHost),
             "read K");
    CUDA_TRY(ctx, cudaMemcpy2D(v_host, d * 4, ctx->vc + base, ctx->slots * d * 4, d * 4, c.kv_heads,
                               cudaMemcpyDeviceToHost),
             "read V");
    return DEC_OK;
}

dec_status dec_read_tap(dec_ctx* ctx, int layer, int m, float* dst_host) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (!ctx->taps) return fail(ctx, DEC_E_ARG, "context was created without DEC_FLAG_TAPS");
    if (layer < 0 || layer >= ctx->cfg.layers || m < 1 || m > ctx->S || !dst_host)
        return fail(ctx, DEC_E_ARG, "bad layer or m, or NULL destination");
    CUDA_TRY(ctx, cudaStreamSynchronize(ctx->stream), "stream sync");
    const size_t h = ctx->cfg.hidden;
    CUDA_TRY(ctx, cudaMemcpy(dst_host, ctx->taps + (size_t)layer * ctx->S * h, (size_t)m * h * 4,
                             cudaMemcpyDeviceToHost),
             "read tap");
    return DEC_OK;
}

int dec_kernels_per_step(const dec_ctx* ctx, int m) {
    if (!ctx || m < 1 || m > ctx->S) return -1;
    if (uses_stream(ctx, m)) return 1;
    return 6 * ctx->cfg.layers + 1;
}

dec_status dec_inject_stall(dec_ctx* ctx, int phase, int polls) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (ctx->step_grid[1] <= 0 && ctx->step_grid[2] <= 0)
        return fail(ctx, DEC_E_UNSUPPORTED, "the context has no persistent plan");
    if (phase < 0 || phase > 5 * ctx->cfg.layers || polls < 1)
        return fail(ctx, DEC_E_ARG, "phase %d outside 0..%d or polls < 1", phase, 5 * ctx->cfg.layers);
    ctx->stall_phase = phase;
    ctx->stall_polls = polls;
    return DEC_OK;
}

dec_status dec_truncate(dec_ctx* ctx, int stream, int new_len) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (ctx->cfg.kind != DEC_QWEN3_TALKER)
        return fail(ctx, DEC_E_UNSUPPORTED, "a KV ring cannot be truncated");
    if (stream < 0 || stream >= ctx->S)
        return fail(ctx, DEC_E_ARG, "stream %d outside 0..%d", stream, ctx->S - 1);
    if (new_len < 0 || new_len > ctx->len_host[stream])
        return fail(ctx, DEC_E_ARG, "new length %d outside 0..%d", new_len, ctx->len_host[stream]);
    CUDA_TRY(ctx, launch_set_len(ctx->len_dev, stream, new_len, ctx->stream), "truncate");
    ctx->len_host[stream] = new_len;
    return DEC_OK;
}

dec_status dec_launch_stage(dec_ctx* ctx, int layer, int stage, int m, int chained) {
    if (!ctx) return fail(nullptr, DEC_E_ARG, "ctx is NULL");
    if (layer < 0 || layer >= ctx->cfg.layers || stage < 0 || stage > 4 || m < 1 || m > ctx->S)
        return fail(ctx, DEC_E_ARG, "bad layer, stage or m");
    for (int i = 0; i < m; ++i) {
        const int pos = ctx->len_host[i];
        if ((ctx->cfg.kind == DEC_QWEN3_TALKER && pos + 1 > ctx->cfg.max_pos) ||
            (ctx->cfg.kind == DEC_CODEC_WINDOWED && pos >= ctx->cfg.max_pos))
            return fail(ctx, DEC_E_CAPACITY, "stream %d is full", i);
    }
    CUDA_TRY(ctx, launch_stage(ctx, layer, stage, m, ctx->io_in, ctx->stream, chained != 0),
             "stage launch");
    return DEC_OK;
}

dec_status dec_gemv(int dtype, const void* W, int N, int K, const float* x, int m, float* y,
                    void* stream) {
    if (dtype != DEC_F32 && dtype != DEC_BF16) return fail(nullptr, DEC_E_ARG, "unknown dtype");
    if (!W || !x || !y) return fail(nullptr, DEC_E_ARG, "NULL pointer");
    if (N < 1 || K < 8 || m < 1 || m > 8) return fail(nullptr, DEC_E_ARG, "need N >= 1, K >= 8, 1 <= m <= 8");
    if (K % 8) return fail(nullptr, DEC_E_UNSUPPORTED, "K must be a multiple of 8");
    if (!aligned16(W) || !aligned16(x)) return fail(nullptr, DEC_E_UNSUPPORTED, "W and x must be 16-byte aligned");
    if (gemv_smem_bytes(m, K) > 200 * 1024) return fail(nullptr, DEC_E_UNSUPPORTED, "m * K too large");
    const int sms = device_sm_count();
    if (sms <= 0) return fail(nullptr, DEC_E_CUDA, "no CUDA device");
    cudaError_t ce = configure_kernels();
    if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "kernel attributes");
    GemvParams p = {};
    p.W = W;
    p.N = N;
    p.K = K;
    p.m = m;
    p.x = x;
    p.ldx = K;
    p.pro = PRO_NONE;
    p.epi = EPI_STORE;
    p.y = y;
    p.ldy = N;
    cudaError_t e = launch_gemv(p, dtype, sms, static_cast<cudaStream_t>(stream), false);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "gemv launch");
    return DEC_OK;
}

size_t dec_attention_workspace_bytes(int m, int q_heads, int kv_heads, int head_dim, int capacity) {
    if (m < 1 || q_heads < 1 || kv_heads < 1 || head_dim < 1 || capacity < 1) return 0;
    const int mc = (capacity + kAttnChunk - 1) / kAttnChunk;
    return align_up(attention_part_bytes(m, q_heads, mc, head_dim)) +
           align_up(attention_ml_bytes(m, q_heads, mc)) + align_up((size_t)m * kv_heads * 4);
}

dec_status dec_attention(int m, int q_heads, int kv_heads, int head_dim, int capacity,
                         const float* q, const float* k, const float* v, const int32_t* lens,
                         float* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !lens || !out || !workspace) return fail(nullptr, DEC_E_ARG, "NULL pointer");
    if (m < 1 || m > 64 || capacity < 1 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads)
        return fail(nullptr, DEC_E_ARG, "bad m, capacity or head counts");
    if (capacity > kMaxSlots) return fail(nullptr, DEC_E_UNSUPPORTED, "capacity above %d", kMaxSlots);
    if (head_dim != 64 && head_dim != 128) return fail(nullptr, DEC_E_UNSUPPORTED, "head_dim 64 or 128");
    if (q_heads / kv_heads > kMaxGroup) return fail(nullptr, DEC_E_UNSUPPORTED, "GQA group above 8");
    if (!aligned16(k) || !aligned16(v) || !aligned16(workspace))
        return fail(nullptr, DEC_E_UNSUPPORTED, "k, v and workspace must be 16-byte aligned");
    const size_t need = dec_attention_workspace_bytes(m, q_heads, kv_heads, head_dim, capacity);
    if (workspace_bytes < need)
        return fail(nullptr, DEC_E_ARG, "workspace of %zu bytes, need %zu", workspace_bytes, need);
    const int mc = (capacity + kAttnChunk - 1) / kAttnChunk;
    cudaError_t ce = configure_kernels();
    if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "kernel attributes");
    char* ws = static_cast<char*>(workspace);
    AttnParams a = {};
    a.mode = ATTN_PLAIN;
    a.m = m;
    a.H = q_heads;
    a.G = kv_heads;
    a.d = head_dim;
    a.slots = capacity;
    a.qkv = q;
    a.kc = const_cast<float*>(k);
    a.vc = const_cast<float*>(v);
    a.len = lens;
    a.max_pos = capacity;
    a.part = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float*>(ws + align_up(attention_part_bytes(m, q_heads, mc, head_dim)));
    a.tickets = reinterpret_cast<unsigned*>(ws + align_up(attention_part_bytes(m, q_heads, mc, head_dim)) +
                                            align_up(attention_ml_bytes(m, q_heads, mc)));
    a.max_chunks = mc;
    a.out = out;
    cudaError_t e = launch_attention(a, static_cast<cudaStream_t>(stream), false);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "attention launch");
    return DEC_OK;
}

}  // extern "C"
