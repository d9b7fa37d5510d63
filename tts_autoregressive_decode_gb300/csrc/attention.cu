// attention.cu -- the stand-alone split-K decode attention kernels (sm_103a).
//
// k_attention: one CTA per (key chunk c, kv head g, stream r) runs one work item of
// attention_chunk.cuh: its cached K/V rows are staged by bulk copies issued BEFORE
// griddepcontrol.wait (cached rows never change during a step), then the fused q/k prologue,
// scores and the chunk's softmax partial.  With a ticket array the last CTA of a (stream, kv
// head) to finish -- found with an atomic ticket, no waiting -- merges the chunks itself (the
// stateless entry points); without one the partials are left for k_attn_merge, a small
// programmatic-dependent kernel with one CTA per (q head, stream).
#include <math_constants.h>

#include "attention_chunk.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dec {

constexpr int kAttnThreads = kChunkThreads;
constexpr int kAttnWarps = kAttnThreads / 32;

size_t attention_smem_bytes(int d, int group) {
    (void)group;
    return chunk_smem_bytes(d);
}

size_t attention_part_bytes(int m, int H, int max_chunks, int d) {
    return sizeof(float) * (size_t)m * H * max_chunks * d;
}
size_t attention_ml_bytes(int m, int H, int max_chunks) {
    return sizeof(float) * 2 * (size_t)m * H * max_chunks;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) k_attention(const AttnParams p) {
    constexpr int CH = kAttnChunk;
    extern __shared__ __align__(128) float smem[];
    const ChunkSmem sm = chunk_smem<D>(smem);
    float* const Ks = sm.Ks;
    float* const s_l = sm.s_l;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_last;

    const int c = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int group = p.H / p.G;

    const ChunkInfo ci = chunk_info(p, r, c);
    const int nch = ci.nch;
    if (ci.bad || c >= nch) {
        if (ci.bad && c == 0 && g == 0 && tid == 0) flag_check(p.status, CHECK_BOUNDS);
        pdl_trigger();
        pdl_wait();
        return;
    }

    // ---- stage the cached rows of the chunk (independent of the previous kernel) ------------
    const uint32_t bar_a = smem_u32(&bar);
    if (tid == 0) {
        mbar_init(bar_a, 1);
        chunk_issue<D>(p, r, g, ci, sm, bar_a);
    }
    __syncthreads();  // the barrier is initialised before any thread waits on it
    pdl_trigger();
    pdl_wait();
    if (!chunk_compute<D>(p, r, g, c, ci, sm, bar_a, 0)) return;

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
template <int D>
__global__ void __launch_bounds__(D) k_attn_merge(const AttnParams p) {
    __shared__ float scratch[2 * (kMaxSlots / kAttnChunk)];
    pdl_trigger();
    pdl_wait();
    merge_items<D, D>(p, blockIdx.y * p.H + blockIdx.x, scratch);
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
