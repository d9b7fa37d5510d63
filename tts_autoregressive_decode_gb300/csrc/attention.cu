// attention.cu -- split-K decode attention with the step's q/k prologue fused in (sm_103a).
//
// One CTA per (key chunk c, kv head g, stream r).  It serves every q head of the GQA group of g
// (kv head of q head i is i / (H/G), Qwen3-TTS talker on wgpu, GQA_ATTN_SRC), so each K/V
// element is read from HBM once per step.  The chunk's cached K and V rows (64 keys, head-major
// cache, contiguous) are staged into shared memory by two 1-D bulk copies (cp.async.bulk) on an
// mbarrier; they are issued BEFORE griddepcontrol.wait because cached rows never change during
// the step.
//
// Prologue, after the wait (the QKV GEMV's raw output is then visible):
//   ATTN_TALKER  per-head RMSNorm of q and of the new k with the shared [d] weights (QK_NORM_SRC),
//                rotate_half rope from the cos/sin table at pos (ROPE_SRC), and the KV append
//                (APPEND_SRC) done by the CTA whose chunk holds pos.
//   ATTN_RING    interleaved-pair rope (rope_push_src); the CTA whose chunk holds slot pos % ring
//                writes k, v and the position stamp into the ring.  A slot is legal iff its stamp
//                is not empty, not after pos, and pos - stamp < window (attn_src).
//   ATTN_PLAIN   q is taken as given; keys 0..len-1.
// Each CTA produces, per q head, the chunk's max score m_c, sum l_c = sum_j exp(s_j - m_c) and
// o_c = sum_j exp(s_j - m_c) v_j.  The last CTA of a (stream, kv head) to finish -- found with an
// atomic ticket, no waiting -- merges them: out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c,
// the running-max rescaling of the online softmax (prior art: REL_POS_ATTN on the Parakeet page).
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace dec {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;

size_t attention_smem_bytes(int d, int group) {
    (void)group;
    // K tile, V tile, q [kMaxGroup][d], scores [kMaxGroup][chunk], new k and v [d] each,
    // stamps [chunk]
    return sizeof(float) * ((size_t)2 * kAttnChunk * d + (size_t)kMaxGroup * d +
                            (size_t)kMaxGroup * kAttnChunk + 2 * (size_t)d) +
           sizeof(uint32_t) * kAttnChunk;
}

size_t attention_part_bytes(int m, int H, int max_chunks, int d) {
    return sizeof(float) * (size_t)m * H * max_chunks * d;
}
size_t attention_ml_bytes(int m, int H, int max_chunks) {
    return sizeof(float) * 2 * (size_t)m * H * max_chunks;
}

// v[0..7] per lane -> lane l returns the warp-wide sum of v[(l >> 2) & 7]
__device__ __forceinline__ float butterfly8_attn(const float v[8], int lane) {
    const bool hi16 = lane & 16, hi8 = lane & 8, hi4 = lane & 4;
    float a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = hi16 ? v[i] : v[i + 4];
        const float keep = hi16 ? v[i + 4] : v[i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = hi8 ? a[i] : a[i + 2];
        const float keep = hi8 ? a[i + 2] : a[i];
        b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = hi4 ? b[0] : b[1];
    float c = (hi4 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) k_attention(const AttnParams p) {
    constexpr int CH = kAttnChunk;
    constexpr int HALF = D / 2;
    extern __shared__ __align__(128) float smem[];
    float* Ks = smem;                          // [CH][D]
    float* Vs = Ks + CH * D;                   // [CH][D]
    float* qs = Vs + CH * D;                   // [kMaxGroup][D]
    float* sc = qs + kMaxGroup * D;            // [kMaxGroup][CH]
    float* knew = sc + kMaxGroup * CH;         // [D]
    float* vnew = knew + D;                    // [D]
    uint32_t* stamp = reinterpret_cast<uint32_t*>(vnew + D);  // [CH]
    __shared__ __align__(8) uint64_t bar;
    __shared__ float s_m[kMaxGroup], s_l[kMaxGroup];
    __shared__ int s_last;

    const int c = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mode = p.mode;
    const int group = p.H / p.G;
    const float scale = 1.0f / sqrtf((float)D);

    // ---- which keys this CTA owns ---------------------------------------------------------
    int pos = 0, nch, k0 = c * CH, nk, ncached, newrow = -1;
    if (mode == ATTN_PLAIN) {
        const int L = p.len[r];
        nch = (L + CH - 1) / CH;
        nk = min(CH, L - k0);
        ncached = nk;
    } else if (mode == ATTN_TALKER) {
        pos = p.len[r];
        const int L = pos + 1;
        nch = (L + CH - 1) / CH;
        nk = min(CH, L - k0);
        ncached = min(nk, pos - k0);
        if (pos >= k0 && pos < k0 + CH) newrow = pos - k0;
    } else {
        pos = p.len[r];
        nch = (p.slots + CH - 1) / CH;
        nk = min(CH, p.slots - k0);
        ncached = nk;
        const int slot = pos % p.slots;
        if (slot >= k0 && slot < k0 + CH) newrow = slot - k0;
    }
    const bool bad = (mode != ATTN_PLAIN && (pos < 0 || pos >= p.max_pos ||
                                             (mode == ATTN_TALKER && pos >= p.slots))) ||
                     (mode == ATTN_PLAIN && (nch > p.max_chunks || p.len[r] > p.slots ||
                                             p.len[r] < 1));
    if (bad || c >= nch) {
        if (bad && c == 0 && g == 0 && tid == 0) flag_check(p.status, CHECK_BOUNDS);
        pdl_trigger();
        pdl_wait();
        return;
    }

    // ---- stage the cached rows of the chunk (independent of the previous kernel) ------------
    const size_t head_base = ((size_t)r * p.G + g) * p.slots;
    const uint32_t bar_a = smem_u32(&bar);
    if (tid == 0) {
        mbar_init(bar_a, 1);
        const uint32_t bytes = (uint32_t)(ncached > 0 ? ncached : 0) * D * sizeof(float);
        mbar_arrive_expect_tx(bar_a, 2 * bytes);
        if (bytes) {
            bulk_g2s(smem_u32(Ks), p.kc + (head_base + k0) * D, bytes, bar_a);
            bulk_g2s(smem_u32(Vs), p.vc + (head_base + k0) * D, bytes, bar_a);
        }
    }
    __syncthreads();  // the barrier is initialised before any thread waits on it
    pdl_trigger();
    pdl_wait();

    // ---- prologue: q heads of the group (and the new key) -----------------------------------
    for (int i = warp; i < group; i += kAttnWarps) {
        const int hq = g * group + i;
        if (mode == ATTN_PLAIN) {
            for (int t = lane; t < D; t += 32) qs[i * D + t] = p.qkv[((size_t)r * p.H + hq) * D + t];
        } else if (mode == ATTN_TALKER) {
            const float* src = p.qkv + (size_t)r * p.ldqkv + (size_t)hq * D;
            float v[D / 32];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                v[j] = src[lane + 32 * j];
                ss += v[j] * v[j];
            }
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)D + p.eps);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) v[j] = v[j] * inv * p.qn[lane + 32 * j];
            const float* cs = p.rope_cos + (size_t)pos * HALF;
            const float* sn = p.rope_sin + (size_t)pos * HALF;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const int t = lane + 32 * j;
                const int jj = (j + D / 64) % (D / 32);       // element t +- D/2, same lane
                const float rot = (t < HALF) ? -v[jj] : v[jj];
                const int f = t < HALF ? t : t - HALF;
                qs[i * D + t] = v[j] * cs[f] + rot * sn[f];
            }
        } else {
            const float* src = p.qkv + (size_t)r * p.ldqkv + (size_t)hq * D;
            const float* cs = p.rope_cos + (size_t)pos * HALF;
            const float* sn = p.rope_sin + (size_t)pos * HALF;
            for (int j = lane; j < HALF; j += 32) {
                const float a = src[2 * j], b = src[2 * j + 1];
                qs[i * D + 2 * j] = a * cs[j] - b * sn[j];
                qs[i * D + 2 * j + 1] = a * sn[j] + b * cs[j];
            }
        }
    }
    if (newrow >= 0 && warp == (group % kAttnWarps)) {
        // the new key and value of kv head g at position pos
        if (mode == ATTN_TALKER) {
            const float* ksrc = p.qkv + (size_t)r * p.ldqkv + (size_t)p.H * D + (size_t)g * D;
            const float* vsrc = ksrc + (size_t)p.G * D;
            float v[D / 32];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                v[j] = ksrc[lane + 32 * j];
                ss += v[j] * v[j];
            }
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)D + p.eps);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) v[j] = v[j] * inv * p.kn[lane + 32 * j];
            const float* cs = p.rope_cos + (size_t)pos * HALF;
            const float* sn = p.rope_sin + (size_t)pos * HALF;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const int t = lane + 32 * j;
                const int jj = (j + D / 64) % (D / 32);
                const float rot = (t < HALF) ? -v[jj] : v[jj];
                const int f = t < HALF ? t : t - HALF;
                knew[t] = v[j] * cs[f] + rot * sn[f];
                vnew[t] = vsrc[t];
            }
        } else {
            const int D_model = p.H * D;
            const float* ksrc = p.qkv + (size_t)r * p.ldqkv + D_model + (size_t)g * D;
            const float* vsrc = ksrc + D_model;
            const float* cs = p.rope_cos + (size_t)pos * HALF;
            const float* sn = p.rope_sin + (size_t)pos * HALF;
            for (int j = lane; j < HALF; j += 32) {
                const float a = ksrc[2 * j], b = ksrc[2 * j + 1];
                knew[2 * j] = a * cs[j] - b * sn[j];
                knew[2 * j + 1] = a * sn[j] + b * cs[j];
                vnew[2 * j] = vsrc[2 * j];
                vnew[2 * j + 1] = vsrc[2 * j + 1];
            }
        }
    }
    if (mode == ATTN_RING)
        for (int j = tid; j < nk; j += kAttnThreads)
            stamp[j] = p.pr[(size_t)r * p.slots + k0 + j];

    // ---- wait for the staged rows (bounded) ---------------------------------------------------
    const bool ok = mbar_wait_bounded(bar_a, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) flag_check(p.status, CHECK_WAIT_LIMIT);
        mbar_wait_bounded(bar_a, 0);  // let copies still in flight land before the CTA leaves
        return;
    }
    if (newrow >= 0) {
        for (int t = tid; t < D; t += kAttnThreads) {
            Ks[newrow * D + t] = knew[t];
            Vs[newrow * D + t] = vnew[t];
        }
        if (tid == 0 && mode == ATTN_RING) stamp[newrow] = (uint32_t)pos;
        // append to the cache (after the staged copy has landed: no read/write overlap)
        float* kd = p.kc + (head_base + k0 + newrow) * D;
        float* vd = p.vc + (head_base + k0 + newrow) * D;
        for (int t = tid; t < D; t += kAttnThreads) {
            kd[t] = knew[t];
            vd[t] = vnew[t];
        }
        if (tid == 0 && mode == ATTN_RING) p.pr[(size_t)r * p.slots + k0 + newrow] = (uint32_t)pos;
    }
    __syncthreads();

    // ---- scores: a warp takes 8 keys at a time, lanes split d, one butterfly per head ------------
    constexpr int PER = D / 32;  // dims per lane (contiguous)
    for (int j0 = warp * 8; j0 < nk; j0 += kAttnWarps * 8) {
        float kv[8][PER];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (j0 + u < nk)
                load_vec<PER>(kv[u], Ks + (j0 + u) * D + lane * PER);
            else
#pragma unroll
                for (int e = 0; e < PER; ++e) kv[u][e] = 0.f;
        }
        for (int i = 0; i < group; ++i) {
            float qv[PER];
            load_vec<PER>(qv, qs + i * D + lane * PER);
            float part[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < PER; ++e) a += qv[e] * kv[u][e];
                part[u] = a;
            }
            const float sum = butterfly8_attn(part, lane);   // lanes 4u..4u+3 hold key j0 + u
            const int u = (lane >> 2) & 7;
            if ((lane & 3) == 0 && j0 + u < nk) {
                bool legal = true;
                if (mode == ATTN_RING) {
                    const uint32_t pj = stamp[j0 + u];
                    legal = (pj != 0xFFFFFFFFu) && (pj <= (uint32_t)pos) &&
                            ((uint32_t)pos - pj < (uint32_t)p.window);
                }
                sc[i * CH + j0 + u] = legal ? sum * scale : -CUDART_INF_F;
            }
        }
    }
    __syncthreads();

    // ---- chunk softmax statistics: warp per q head ---------------------------------------------
    for (int i = warp; i < group; i += kAttnWarps) {
        float mx = -CUDART_INF_F;
        for (int j = lane; j < nk; j += 32) mx = fmaxf(mx, sc[i * CH + j]);
        mx = warp_max(mx);
        float l = 0.f;
        for (int j = lane; j < nk; j += 32) {
            const float e = (mx == -CUDART_INF_F) ? 0.f : expf(sc[i * CH + j] - mx);
            sc[i * CH + j] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            s_m[i] = mx;
            s_l[i] = l;
        }
    }
    __syncthreads();

    // ---- o_c = sum_j e_j v_j (ascending j), then write the partial ----------------------------
    for (int o = tid; o < group * D; o += kAttnThreads) {
        const int i = o / D, t = o - i * D;
        // masked keys weigh exactly 0 and their V rows hold finite values (zeroed at creation)
        float acc = 0.f;
        const float* w = sc + i * CH;
#pragma unroll 8
        for (int j = 0; j < nk; ++j) acc += w[j] * Vs[j * D + t];
        const int hq = g * group + i;
        if (nch == 1) {
            p.out[((size_t)r * p.H + hq) * D + t] = acc / s_l[i];
        } else {
            const size_t pi = ((size_t)r * p.H + hq) * p.max_chunks + c;
            p.part[pi * D + t] = acc;
            if (t == 0) {
                p.part_ml[2 * pi] = s_m[i];
                p.part_ml[2 * pi + 1] = s_l[i];
            }
        }
    }
    // with no ticket array the partials are merged by the separate merge kernel
    if (nch == 1 || !p.tickets) return;

    // ---- ticket: the last CTA of (r, g) merges the chunks ---------------------------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&p.tickets[r * p.G + g], 1u);
        s_last = (prev == (unsigned)(nch - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Stage every chunk's (m, l) of the group's heads in shared memory with independent loads
    // (the K/V tiles are no longer needed), then the per-head max M, denominator and chunk
    // weights w_c = exp(m_c - M); chunks without a legal key (l == 0) weigh 0.
    float* wsc = Ks;                               // [group][nch] chunk weights
    float* buf = Ks + kMaxGroup * ((p.max_chunks + 3) & ~3);  // partial outputs, batched
    for (int idx = tid; idx < group * nch; idx += kAttnThreads) {
        const int i = idx / nch, cc = idx - i * nch;
        const size_t pi = ((size_t)r * p.H + g * group + i) * p.max_chunks + cc;
        const float mc = __ldcg(p.part_ml + 2 * pi), lc = __ldcg(p.part_ml + 2 * pi + 1);
        wsc[i * nch + cc] = lc > 0.f ? mc : -CUDART_INF_F;
        buf[idx] = lc;
    }
    __syncthreads();
    for (int i = warp; i < group; i += kAttnWarps) {
        float M = -CUDART_INF_F;
        for (int cc = lane; cc < nch; cc += 32) M = fmaxf(M, wsc[i * nch + cc]);
        M = warp_max(M);
        float den = 0.f;
        for (int cc = lane; cc < nch; cc += 32) {
            const float mc = wsc[i * nch + cc];
            const float wc = (mc == -CUDART_INF_F) ? 0.f : expf(mc - M);
            wsc[i * nch + cc] = wc;
            den += wc * buf[i * nch + cc];
        }
        den = warp_sum(den);
        if (lane == 0) s_l[i] = den;
    }
    __syncthreads();
    // out = sum_c w_c o_c / den, the partial rows fetched in batches of whole chunks
    const int per_batch = (int)((2 * CH * D - kMaxGroup * ((p.max_chunks + 3) & ~3)) / (group * D));
    float num[(kMaxGroup * D + kAttnThreads - 1) / kAttnThreads];
#pragma unroll
    for (int q = 0; q < (kMaxGroup * D + kAttnThreads - 1) / kAttnThreads; ++q) num[q] = 0.f;
    for (int c0 = 0; c0 < nch; c0 += per_batch) {
        const int nb = min(per_batch, nch - c0);
        const int total = nb * group * D;
        constexpr int UNR = 16;  // independent loads in flight per thread
        for (int base = 0; base < total; base += kAttnThreads * UNR) {
            float tmp[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int idx = base + u * kAttnThreads + tid;
                tmp[u] = 0.f;
                if (idx < total) {
                    const int cc = idx / (group * D), rem = idx - cc * group * D;
                    const int i = rem / D, t = rem - i * D;
                    const size_t pi = ((size_t)r * p.H + g * group + i) * p.max_chunks + c0 + cc;
                    tmp[u] = __ldcg(p.part + pi * D + t);
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int idx = base + u * kAttnThreads + tid;
                if (idx < total) buf[idx] = tmp[u];
            }
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < (kMaxGroup * D + kAttnThreads - 1) / kAttnThreads; ++q) {
            const int o = tid + q * kAttnThreads;
            if (o < group * D) {
                const int i = o / D;
                for (int cc = 0; cc < nb; ++cc)
                    num[q] += wsc[i * nch + c0 + cc] * buf[cc * group * D + o];
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < (kMaxGroup * D + kAttnThreads - 1) / kAttnThreads; ++q) {
        const int o = tid + q * kAttnThreads;
        if (o < group * D) {
            const int i = o / D, t = o - i * D;
            p.out[((size_t)r * p.H + g * group + i) * D + t] = num[q] / s_l[i];
        }
    }
    if (tid == 0) p.tickets[r * p.G + g] = 0u;
}

template <int D>
static cudaError_t launch_t(const AttnParams& p, cudaStream_t s, bool pdl) {
    const size_t smem = attention_smem_bytes(D, p.H / p.G);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.max_chunks, p.G, p.m);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_attention<D>, p);
}

// ---------------------------------------------------------------------------------------------
// Merge of the chunk partials, one CTA per (q head, stream), d threads:
// out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c over the chunks with a legal key (l_c > 0).
// Launched after k_attention (programmatic dependent); the chunking is k_attention's.
// ---------------------------------------------------------------------------------------------
constexpr int kMergeBatch = 64;  // partial rows in flight per thread

template <int D>
__global__ void __launch_bounds__(D) k_attn_merge(const AttnParams p) {
    constexpr int CH = kAttnChunk;
    __shared__ float sm[kMaxSlots / kAttnChunk], sw[kMaxSlots / kAttnChunk];
    const int hq = blockIdx.x, r = blockIdx.y, t = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    int L;
    if (p.mode == ATTN_PLAIN) L = p.len[r];
    else L = (p.mode == ATTN_TALKER) ? p.len[r] + 1 : p.slots;
    const int nch = (L + CH - 1) / CH;
    if (L < 1 || nch <= 1 || nch > p.max_chunks) return;  // one chunk: k_attention wrote out
    const size_t base = ((size_t)r * p.H + hq) * p.max_chunks;
    for (int c = t; c < nch; c += D) {
        const float l = __ldcg(p.part_ml + 2 * (base + c) + 1);
        sm[c] = l > 0.f ? __ldcg(p.part_ml + 2 * (base + c)) : -CUDART_INF_F;
        sw[c] = l;
    }
    __syncthreads();
    float M = -CUDART_INF_F;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, sm[c]);
    __syncthreads();
    for (int c = t; c < nch; c += D) {  // weight of chunk c, and its share of the denominator
        const float w = sm[c] == -CUDART_INF_F ? 0.f : expf(sm[c] - M);
        sm[c] = w;
        sw[c] = w * sw[c];
    }
    __syncthreads();
    float den = 0.f, num = 0.f;
    for (int c = 0; c < nch; ++c) den += sw[c];
    for (int c0 = 0; c0 < nch; c0 += kMergeBatch) {
        float v[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
            v[u] = c0 + u < nch ? __ldcg(p.part + (base + c0 + u) * D + t) : 0.f;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
            if (c0 + u < nch) num += sm[c0 + u] * v[u];
    }
    p.out[((size_t)r * p.H + hq) * D + t] = num / den;
}

template <int D>
static cudaError_t launch_merge_t(const AttnParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.H, p.m);
    cfg.blockDim = dim3(D);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_attn_merge<D>, p);
}

cudaError_t launch_attention_merge(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.max_chunks > kMaxSlots / kAttnChunk) return cudaErrorInvalidValue;
    if (p.d == 64) return launch_merge_t<64>(p, s, pdl);
    if (p.d == 128) return launch_merge_t<128>(p, s, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t attention_configure() {
    cudaError_t e = cudaFuncSetAttribute(k_attention<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)attention_smem_bytes(64, kMaxGroup));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_attention<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attention_smem_bytes(128, kMaxGroup));
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.d == 64) return launch_t<64>(p, s, pdl);
    if (p.d == 128) return launch_t<128>(p, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace dec
