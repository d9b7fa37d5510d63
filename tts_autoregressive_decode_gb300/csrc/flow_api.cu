// flow_api.cu -- the flow head's C ABI (include/dec.h): SimpleMLPAdaLN with one LSD step
// (Pocket TTS on wgpu, PocketFlowGpu), as a chain of split-K GEMVs on the device.
//
// Plan of one call (3 + 2 blocks + 1 kernels, chained with programmatic dependent launch and
// captured as a CUDA graph):
//   [input_proj + bias -> x]  [cond embedding + (bias + time constant), SiLU -> y]
//   [the adaLN projections of every block and of the final layer, stacked: one GEMV of y]
//   per block: [LayerNorm(x) + modulate prologue, m0 + bias, SiLU -> h]
//              [m2 + bias, gated residual into x]
//   [non-affine LayerNorm(x) + modulate prologue, final linear + bias, + noise -> latent]
// The elementwise passes of the page's plan (MV_BIAS's bias and SiLU, ADD_SILU, MODULATE,
// GATED_ADD, LSD_STEP) are folded into the GEMVs' prologues and epilogues; the page's
// per-block adaLN projections all read the same y, so they run as one GEMV over the stacked
// rows.  The time constant is folded into the cond bias once, at creation.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <string>
#include <vector>

#include "../../include/dec.h"
#include "gemv_rows.cuh"
#include "kernels.h"

using namespace dec;

namespace {

thread_local std::string g_flow_error;

struct FlowGraph {
    const float *cond, *noise;
    float* out;
    cudaGraphExec_t exec;
};

}  // namespace

struct dec_flow {
    dec_flow_config cfg{};
    cudaStream_t stream = nullptr;
    cudaStream_t cap_stream = nullptr;
    int num_sms = 0;
    int ada_rows = 0;            // blocks * 3 dim + 2 dim
    char* arena = nullptr;       // weights and scratch
    const float *ip_w = nullptr, *ip_b = nullptr, *cond_w = nullptr, *cond_bt = nullptr;
    const float *ada_w = nullptr, *ada_b = nullptr, *f_w = nullptr, *f_b = nullptr;
    std::vector<const float*> ln_w, ln_b, m0_w, m0_b, m2_w, m2_b;
    float *x = nullptr, *y = nullptr, *m = nullptr, *h = nullptr;
    std::vector<FlowGraph> graphs;
    std::string err;
};

namespace {

dec_status flow_fail(dec_flow* f, dec_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    (f ? f->err : g_flow_error) = buf;
    return st;
}

GemvParams flow_gemv(const dec_flow* f, const float* W, int N, int K, const float* x,
                     const float* bias, float* y) {
    GemvParams g = {};
    g.W = W;
    g.N = N;
    g.K = K;
    g.m = 1;
    g.x = x;
    g.ldx = K;
    g.pro = PRO_NONE;
    g.eps = f->cfg.ln_eps;
    g.epi = EPI_STORE;
    g.bias = bias;
    g.y = y;
    g.ldy = N;
    g.unit = 1;
    return g;
}

cudaError_t flow_enqueue(dec_flow* f, const float* cond, const float* noise, float* out,
                         cudaStream_t s) {
    const dec_flow_config& c = f->cfg;
    const int D = c.dim;
    cudaError_t e;
    auto run = [&](const GemvParams& g, bool pdl) { return launch_gemv(g, DEC_F32, f->num_sms, s, pdl); };

    if ((e = run(flow_gemv(f, f->ip_w, D, c.latent, noise, f->ip_b, f->x), false)) != cudaSuccess) return e;
    GemvParams g = flow_gemv(f, f->cond_w, D, c.cond, cond, f->cond_bt, f->y);
    g.act = 1;
    if ((e = run(g, true)) != cudaSuccess) return e;
    if ((e = run(flow_gemv(f, f->ada_w, f->ada_rows, D, f->y, f->ada_b, f->m), true)) != cudaSuccess)
        return e;
    for (int b = 0; b < c.blocks; ++b) {
        const float* mb = f->m + (size_t)b * 3 * D;  // shift | scale | gate of block b
        g = flow_gemv(f, f->m0_w[b], D, D, f->x, f->m0_b[b], f->h);
        g.pro = PRO_LN_MOD;
        g.nw = f->ln_w[b];
        g.nb = f->ln_b[b];
        g.mod = mb;
        g.act = 1;
        if ((e = run(g, true)) != cudaSuccess) return e;
        g = flow_gemv(f, f->m2_w[b], D, D, f->h, f->m2_b[b], f->x);
        g.epi = EPI_RESID;
        g.res = f->x;
        g.ldres = D;
        g.ls = mb + 2 * D;  // the gate scales the branch
        if ((e = run(g, true)) != cudaSuccess) return e;
    }
    // final layer: non-affine LayerNorm, modulate, linear, and the LSD update on the noise
    g = flow_gemv(f, f->f_w, c.latent, D, f->x, f->f_b, out);
    g.pro = PRO_LN_MOD;
    g.mod = f->m + (size_t)c.blocks * 3 * D;
    g.epi = EPI_RESID;
    g.res = noise;
    g.ldres = c.latent;
    return run(g, true);
}

}  // namespace

extern "C" {

dec_status dec_flow_create(const dec_flow_config* cfg, const dec_flow_weights* w, void* stream,
                           dec_flow** out) {
    g_flow_error.clear();
    if (!out) return flow_fail(nullptr, DEC_E_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg || !w) return flow_fail(nullptr, DEC_E_ARG, "config or weights NULL");
    const dec_flow_config c = *cfg;
    if (c.dim < 8 || c.latent < 8 || c.cond < 8 || c.blocks < 0 || !(c.ln_eps >= 0.f))
        return flow_fail(nullptr, DEC_E_ARG, "bad flow head sizes");
    if (c.dim % 8 || c.latent % 8 || c.cond % 8)
        return flow_fail(nullptr, DEC_E_UNSUPPORTED, "dim, latent and cond must be multiples of 8");
    if (c.lsd_steps != 1)
        return flow_fail(nullptr, DEC_E_UNSUPPORTED, "only one LSD step is planned (lsd_steps = 1)");
    if (rows_gemv_nj(std::max(c.dim, c.cond), 1, DEC_F32) == 0)
        return flow_fail(nullptr, DEC_E_UNSUPPORTED, "dim / cond too wide for the split-K GEMV");
    if (!w->ip_w || !w->ip_b || !w->cond_w || !w->cond_b || !w->t_const || !w->fada_w ||
        !w->fada_b || !w->f_w || !w->f_b)
        return flow_fail(nullptr, DEC_E_ARG, "a flow head weight is NULL");
    if (c.blocks > 0 && (!w->ada_w || !w->ada_b || !w->ln_w || !w->ln_b || !w->m0_w || !w->m0_b ||
                         !w->m2_w || !w->m2_b))
        return flow_fail(nullptr, DEC_E_ARG, "a block weight array is NULL");
    for (int b = 0; b < c.blocks; ++b)
        if (!w->ada_w[b] || !w->ada_b[b] || !w->ln_w[b] || !w->ln_b[b] || !w->m0_w[b] ||
            !w->m0_b[b] || !w->m2_w[b] || !w->m2_b[b])
            return flow_fail(nullptr, DEC_E_ARG, "block %d: a weight is NULL", b);

    dec_flow* f = new dec_flow();
    f->cfg = c;
    f->stream = static_cast<cudaStream_t>(stream);
    const int D = c.dim;
    f->ada_rows = c.blocks * 3 * D + 2 * D;
    auto bail = [&](cudaError_t e, const char* what) {
        flow_fail(nullptr, DEC_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
        dec_flow_destroy(f);
        return DEC_E_CUDA;
    };
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&f->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return bail(e, "device");
    if ((e = configure_kernels()) != cudaSuccess) return bail(e, "kernel attributes");
    if ((e = cudaStreamCreateWithFlags(&f->cap_stream, cudaStreamNonBlocking)) != cudaSuccess)
        return bail(e, "capture stream");

    // ---- arena: weights (the adaLN projections stacked) and scratch ---------------------------
    size_t tot = 0;
    auto take = [&](size_t floats) {
        const size_t o = tot;
        tot += (floats * 4 + 255) / 256 * 256;
        return o;
    };
    const size_t o_ipw = take((size_t)D * c.latent), o_ipb = take(D);
    const size_t o_cw = take((size_t)D * c.cond), o_cb = take(D);
    const size_t o_aw = take((size_t)f->ada_rows * D), o_ab = take(f->ada_rows);
    std::vector<size_t> o_blk;
    for (int b = 0; b < c.blocks; ++b) {
        o_blk.push_back(take(D));                 // ln_w
        o_blk.push_back(take(D));                 // ln_b
        o_blk.push_back(take((size_t)D * D));     // m0_w
        o_blk.push_back(take(D));                 // m0_b
        o_blk.push_back(take((size_t)D * D));     // m2_w
        o_blk.push_back(take(D));                 // m2_b
    }
    const size_t o_fw = take((size_t)c.latent * D), o_fb = take(c.latent);
    const size_t o_x = take(D), o_y = take(D), o_m = take(f->ada_rows), o_h = take(D);
    if ((e = cudaMalloc(&f->arena, tot)) != cudaSuccess) return bail(e, "flow arena");
    char* a = f->arena;
    cudaStream_t s = f->stream;
    auto cp = [&](size_t off, const float* src, size_t floats) {
        return cudaMemcpyAsync(a + off, src, floats * 4, cudaMemcpyDeviceToDevice, s);
    };
    auto fp = [&](size_t off) { return reinterpret_cast<float*>(a + off); };
    if ((e = cp(o_ipw, w->ip_w, (size_t)D * c.latent)) != cudaSuccess ||
        (e = cp(o_ipb, w->ip_b, D)) != cudaSuccess ||
        (e = cp(o_cw, w->cond_w, (size_t)D * c.cond)) != cudaSuccess ||
        (e = cp(o_fw, w->f_w, (size_t)c.latent * D)) != cudaSuccess ||
        (e = cp(o_fb, w->f_b, c.latent)) != cudaSuccess)
        return bail(e, "weight copy");
    for (int b = 0; b < c.blocks; ++b) {
        // byte offsets of block b's rows in the stacked projection
        if ((e = cp(o_aw + (size_t)b * 3 * D * D * 4, w->ada_w[b], (size_t)3 * D * D)) != cudaSuccess ||
            (e = cp(o_ab + (size_t)b * 3 * D * 4, w->ada_b[b], (size_t)3 * D)) != cudaSuccess)
            return bail(e, "weight copy");
    }
    if ((e = cp(o_aw + (size_t)c.blocks * 3 * D * D * 4, w->fada_w, (size_t)2 * D * D)) != cudaSuccess ||
        (e = cp(o_ab + (size_t)c.blocks * 3 * D * 4, w->fada_b, (size_t)2 * D)) != cudaSuccess)
        return bail(e, "weight copy");
    const float* const* srcs[6] = {w->ln_w, w->ln_b, w->m0_w, w->m0_b, w->m2_w, w->m2_b};
    const size_t sizes[6] = {(size_t)D, (size_t)D, (size_t)D * D, (size_t)D, (size_t)D * D, (size_t)D};
    for (int b = 0; b < c.blocks; ++b)
        for (int j = 0; j < 6; ++j)
            if ((e = cp(o_blk[(size_t)b * 6 + j], srcs[j][b], sizes[j])) != cudaSuccess)
                return bail(e, "weight copy");
    // cond bias + time constant, once (the page's ADD_SILU adds the constant every call)
    std::vector<float> hb(D), ht(D);
    if ((e = cudaMemcpyAsync(hb.data(), w->cond_b, (size_t)D * 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(ht.data(), w->t_const, (size_t)D * 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return bail(e, "cond bias read");
    for (int i = 0; i < D; ++i) hb[i] += ht[i];
    if ((e = cudaMemcpyAsync(a + o_cb, hb.data(), (size_t)D * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return bail(e, "cond bias write");

    f->ip_w = fp(o_ipw);
    f->ip_b = fp(o_ipb);
    f->cond_w = fp(o_cw);
    f->cond_bt = fp(o_cb);
    f->ada_w = fp(o_aw);
    f->ada_b = fp(o_ab);
    f->f_w = fp(o_fw);
    f->f_b = fp(o_fb);
    for (int b = 0; b < c.blocks; ++b) {
        f->ln_w.push_back(fp(o_blk[(size_t)b * 6 + 0]));
        f->ln_b.push_back(fp(o_blk[(size_t)b * 6 + 1]));
        f->m0_w.push_back(fp(o_blk[(size_t)b * 6 + 2]));
        f->m0_b.push_back(fp(o_blk[(size_t)b * 6 + 3]));
        f->m2_w.push_back(fp(o_blk[(size_t)b * 6 + 4]));
        f->m2_b.push_back(fp(o_blk[(size_t)b * 6 + 5]));
    }
    f->x = fp(o_x);
    f->y = fp(o_y);
    f->m = fp(o_m);
    f->h = fp(o_h);
    *out = f;
    return DEC_OK;
}

dec_status dec_flow_step(dec_flow* f, const float* cond, const float* noise, float* latent_out) {
    if (!f) return flow_fail(nullptr, DEC_E_ARG, "flow head is NULL");
    if (!cond || !noise || !latent_out) return flow_fail(f, DEC_E_ARG, "NULL buffer");
    if ((reinterpret_cast<uintptr_t>(cond) | reinterpret_cast<uintptr_t>(noise) |
         reinterpret_cast<uintptr_t>(latent_out)) & 15u)
        return flow_fail(f, DEC_E_ARG, "buffers must be 16-byte aligned");
    cudaGraphExec_t exec = nullptr;
    for (auto& g : f->graphs)
        if (g.cond == cond && g.noise == noise && g.out == latent_out) exec = g.exec;
    cudaError_t e = cudaSuccess;
    if (!exec) {
        if ((e = cudaStreamBeginCapture(f->cap_stream, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
            return flow_fail(f, DEC_E_CUDA, "capture: %s", cudaGetErrorString(e));
        const cudaError_t e1 = flow_enqueue(f, cond, noise, latent_out, f->cap_stream);
        cudaGraph_t graph = nullptr;
        const cudaError_t e2 = cudaStreamEndCapture(f->cap_stream, &graph);
        if (e1 == cudaSuccess && e2 == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (e1 != cudaSuccess || e2 != cudaSuccess || e != cudaSuccess)
            return flow_fail(f, DEC_E_CUDA, "flow graph: %s",
                             cudaGetErrorString(e1 != cudaSuccess ? e1 : e2 != cudaSuccess ? e2 : e));
        if (f->graphs.size() >= 8) {  // a queued graph is freed when it completes
            cudaGraphExecDestroy(f->graphs.front().exec);
            f->graphs.erase(f->graphs.begin());
        }
        f->graphs.push_back({cond, noise, latent_out, exec});
    }
    if ((e = cudaGraphLaunch(exec, f->stream)) != cudaSuccess)
        return flow_fail(f, DEC_E_CUDA, "flow launch: %s", cudaGetErrorString(e));
    return DEC_OK;
}

void dec_flow_destroy(dec_flow* f) {
    if (!f) return;
    if (f->stream || f->cap_stream) cudaStreamSynchronize(f->stream);
    for (auto& g : f->graphs) cudaGraphExecDestroy(g.exec);
    if (f->cap_stream) cudaStreamDestroy(f->cap_stream);
    if (f->arena) cudaFree(f->arena);
    delete f;
}

const char* dec_flow_last_error(const dec_flow* f) { return f ? f->err.c_str() : g_flow_error.c_str(); }

int dec_flow_kernels_per_step(const dec_flow* f) { return f ? 3 + 2 * f->cfg.blocks + 1 : -1; }

}  // extern "C"
