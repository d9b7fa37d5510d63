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
    extern __shared__ __align__(128) float smem[];
    const ChunkSmem sm = chunk_smem<D>(smem);
    float* const Ks = sm.Ks;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_last;

    const int c = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x;
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

    // with no ticket array the partials are merged by k_attn_merge
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

    // merge the group's q heads (items r H + g group + i), kAttnThreads / D at a time; the K/V
    // tiles are no longer needed, so their area is the scratch
    for (int i0 = 0; i0 < group; i0 += kAttnThreads / D)
        merge_items<D, kAttnThreads>(p, r * p.H + g * group + i0, r * p.H + (g + 1) * group, Ks);
    if (tid == 0) p.tickets[r * p.G + g] = 0u;
}

// Two chunks per CTA: half h (128 threads, named barrier 1 + h) takes chunk 2 x + h of (kv
// head y, row z); both halves stage their K/V rows before griddepcontrol.wait.  Each chunk is
// computed as k_attention computes it; the partials are merged by k_attn_merge.
template <int D>
__global__ void __launch_bounds__(kAttnThreads) k_attention_pair(const AttnParams p) {
    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t bar[2];
    const int tid = threadIdx.x, h = tid >> 7, htid = tid & 127;
    const int c = 2 * blockIdx.x + h, g = blockIdx.y, r = blockIdx.z;
    const ChunkSmem sm = chunk_smem<D>(smem + (size_t)h * chunk_smem_floats(D));
    const ChunkInfo ci = chunk_info(p, r, c);
    const bool active = !ci.bad && c < ci.nch && c < p.max_chunks;
    const uint32_t bar_h = smem_u32(&bar[h]);
    if (htid == 0) {
        mbar_init(bar_h, 1);
        if (active) chunk_issue<D>(p, r, g, ci, sm, bar_h);
    }
    if (ci.bad && c == 0 && g == 0 && htid == 0) flag_check(p.status, CHECK_BOUNDS);
    __syncthreads();  // both barriers initialised before any thread waits
    pdl_trigger();
    pdl_wait();
    if (active) chunk_compute<D, kAttnThreads / 2>(p, r, g, c, ci, sm, bar_h, 0, htid, 1 + h);
}

// CTAs of k_attention_pair's grid: two chunks of the capacity per CTA, per kv head and row
int attention_pair_ctas(const AttnParams& p) {
    return ((p.max_chunks + 1) / 2) * p.G * p.m;
}

template <int D>
static cudaError_t launch_t(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.paired && !p.tickets) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((p.max_chunks + 1) / 2, p.G, p.m);
        cfg.blockDim = dim3(kAttnThreads);
        cfg.dynamicSmemBytes = 2 * chunk_smem_bytes(D);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, k_attention_pair<D>, p);
    }
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
    merge_items<D, D, kMergeFirstWide>(p, blockIdx.y * p.H + blockIdx.x, p.m * p.H, scratch);
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

// ---------------------------------------------------------------------------------------------
// Prefill block append: one warp per (row r, kv head g) computes the talker's new key (k-norm,
// rope at len[stream] + r) and value, as the step's attention prologue does, and writes them to
// the cache of p.stream.  The attention of the block runs after it, so every row sees the keys
// of the rows before it (causal within the block).
// ---------------------------------------------------------------------------------------------
constexpr int kAppendWarps = 4;

template <int D>
__global__ void __launch_bounds__(kAppendWarps * 32) k_prefill_append(const AttnParams p) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int idx = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (idx >= p.m * p.G) return;
    const int r = idx / p.G, g = idx - r * p.G;
    const ChunkInfo ci = chunk_info(p, r, 0);  // position len + r and its rotary positions
    if (ci.bad) {
        if (lane == 0) flag_check(p.status, CHECK_BOUNDS);
        return;
    }
    const size_t row = (((size_t)p.stream * p.G + g) * p.slots + ci.pos) * D;
    talker_new_kv<D>(p, r, g, ci, lane, p.kc + row, p.vc + row);
}

template <int D>
static cudaError_t launch_append_t(const AttnParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.m * p.G + kAppendWarps - 1) / kAppendWarps);
    cfg.blockDim = dim3(kAppendWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_prefill_append<D>, p);
}

cudaError_t launch_prefill_append(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.mode != ATTN_PREFILL) return cudaErrorInvalidValue;
    if (p.d == 64) return launch_append_t<64>(p, s, pdl);
    if (p.d == 128) return launch_append_t<128>(p, s, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t attention_configure() {
    cudaError_t e = cudaFuncSetAttribute(k_attention<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)attention_smem_bytes(64, kMaxGroup));
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_attention_pair<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)(2 * chunk_smem_bytes(64)))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(k_attention_pair<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)(2 * chunk_smem_bytes(128)))) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k_attention<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attention_smem_bytes(128, kMaxGroup));
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.d == 64) return launch_t<64>(p, s, pdl);
    if (p.d == 128) return launch_t<128>(p, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace dec
