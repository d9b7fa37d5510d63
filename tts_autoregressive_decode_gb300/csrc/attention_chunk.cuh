// attention_chunk.cuh -- one key chunk of the split-K decode attention, and the merge of the
// chunk partials, as device functions shared by the stand-alone kernels (attention.cu) and the
// persistent step kernel (step.cu).
//
// A work item is (stream r, kv head g, chunk c of kAttnChunk keys).  It serves every q head of
// the GQA group of g (kv head of q head i is i / (H/G), Qwen3-TTS talker on wgpu, GQA_ATTN_SRC),
// so each K/V element is read from HBM once per step.  The chunk's cached K and V rows
// (head-major cache, contiguous) are staged into shared memory by two 1-D bulk copies
// (cp.async.bulk) on an mbarrier; cached rows never change during a step, so the copies may be
// issued before the q/k/v projection that precedes the attention has finished.
//
// Prologue, once the q/k/v projection is visible:
//   ATTN_TALKER  per-head RMSNorm of q and of the new k with the shared [d] weights (QK_NORM_SRC),
//                rotate_half rope from the cos/sin table at pos (ROPE_SRC), and the KV append
//                (APPEND_SRC) done by the item whose chunk holds pos.
//   ATTN_RING    interleaved-pair rope (rope_push_src); the item whose chunk holds slot pos % ring
//                writes k, v and the position stamp into the ring.  A slot is legal iff its stamp
//                is not empty, not after pos, and pos - stamp < window (attn_src).
//   ATTN_PLAIN   q is taken as given; keys 0..len-1.
// Each item produces, per q head, the chunk's max score m_c, sum l_c = sum_j exp(s_j - m_c) and
// o_c = sum_j exp(s_j - m_c) v_j.  The merge is out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c,
// the running-max rescaling of the online softmax (prior art: REL_POS_ATTN on the Parakeet page).
//
// Values written earlier in the same launch (q/k/v, partials, stamps) are read with ld.global.cg.
#pragma once

#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace dec {

constexpr int kChunkThreads = 256;  // threads of the stand-alone kernel's CTA (one item)

// Barriers of the NT threads that work on one item: the whole CTA (NT == kChunkThreads) or a
// group of NT threads with its own named barrier `id` (1..15; 0 is __syncthreads).
template <int NT>
__device__ __forceinline__ void group_sync(int id) {
    if constexpr (NT == kChunkThreads) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(NT) : "memory");
    }
}
template <int NT>
__device__ __forceinline__ bool group_or(int id, bool v) {
    if constexpr (NT == kChunkThreads) {
        return __syncthreads_or(v);
    } else {
        uint32_t out;
        asm volatile(
            "{\n\t.reg .pred pv, pr;\n\t"
            "setp.ne.u32 pv, %2, 0;\n\t"
            "bar.red.or.pred pr, %1, %3, pv;\n\t"
            "selp.u32 %0, 1, 0, pr;\n\t}"
            : "=r"(out)
            : "r"(id), "r"((uint32_t)v), "r"(NT)
            : "memory");
        return out != 0;
    }
}

// shared-memory carve-up of one item (the dynamic shared memory of the attention kernels)
struct ChunkSmem {
    float* Ks;       // [CH][D]  (16-byte aligned: bulk-copy destination)
    float* Vs;       // [CH][D]
    float* qs;       // [kMaxGroup][D]
    float* sc;       // [kMaxGroup][CH] scores, then exp weights
    float* knew;     // [D]
    float* vnew;     // [D]
    float* s_m;      // [kMaxGroup] chunk max per q head
    float* s_l;      // [kMaxGroup] chunk sum per q head
    uint32_t* stamp; // [CH] ring position stamps
};

// floats of one item's area (a multiple of 32, so consecutive areas stay 128-byte aligned)
__host__ __device__ constexpr size_t chunk_smem_floats(int d) {
    return ((size_t)2 * kAttnChunk * d + (size_t)kMaxGroup * d + (size_t)kMaxGroup * kAttnChunk +
            2 * (size_t)d + 2 * kMaxGroup + kAttnChunk + 31) / 32 * 32;
}
__host__ __device__ constexpr size_t chunk_smem_bytes(int d) {
    return sizeof(float) * chunk_smem_floats(d);
}

template <int D>
__device__ __forceinline__ ChunkSmem chunk_smem(float* base) {
    ChunkSmem s;
    s.Ks = base;
    s.Vs = s.Ks + kAttnChunk * D;
    s.qs = s.Vs + kAttnChunk * D;
    s.sc = s.qs + kMaxGroup * D;
    s.knew = s.sc + kMaxGroup * kAttnChunk;
    s.vnew = s.knew + D;
    s.s_m = s.vnew + D;
    s.s_l = s.s_m + kMaxGroup;
    s.stamp = reinterpret_cast<uint32_t*>(s.s_l + kMaxGroup);
    return s;
}

// The stream whose cache row r of a launch reads: the row itself, or for a prefill block the
// block's stream.
__device__ __forceinline__ int cache_stream(const AttnParams& p, int r) {
    return p.mode == ATTN_PREFILL ? p.stream : r;
}

// Which keys chunk c of row r covers, and whether the row's position is usable.
struct ChunkInfo {
    int pos;      // TALKER/RING: the step's position
    int nch;      // chunks of the stream
    int k0;       // first key (cache row / ring slot) of the chunk
    int nk;       // keys in the chunk
    int ncached;  // rows to stage from the cache
    int newrow;   // row of the chunk that receives the new k/v (-1: none)
    int rt, rh, rw; // TALKER/PREFILL: the rotary positions of the t, h, w axes (all pos
                    // without per-axis positions)
    bool bad;     // position / length out of range: the item does nothing
};

__device__ __forceinline__ ChunkInfo chunk_info(const AttnParams& p, int r, int c) {
    constexpr int CH = kAttnChunk;
    ChunkInfo ci;
    ci.pos = 0;
    ci.k0 = c * CH;
    ci.newrow = -1;
    const int len = p.mode == ATTN_PREFILL ? 0 : __ldcg(p.len + r);
    if (p.mode == ATTN_PLAIN) {
        ci.nch = (len + CH - 1) / CH;
        ci.nk = min(CH, len - ci.k0);
        ci.ncached = ci.nk;
        ci.bad = ci.nch > p.max_chunks || len > p.slots || len < 1;
    } else if (p.mode == ATTN_PREFILL) {
        const int base = __ldcg(p.len + p.stream);  // the stream's length before the block
        ci.pos = base + r;
        const int L = ci.pos + 1;
        ci.nch = (L + CH - 1) / CH;
        ci.nk = min(CH, L - ci.k0);
        ci.ncached = ci.nk;  // the block's own rows are already in the cache
        ci.bad = base < 0 || ci.pos >= p.max_pos || ci.pos >= p.slots;
        (void)len;
    } else if (p.mode == ATTN_TALKER) {
        ci.pos = len;
        const int L = len + 1;
        ci.nch = (L + CH - 1) / CH;
        ci.nk = min(CH, L - ci.k0);
        ci.ncached = min(ci.nk, ci.pos - ci.k0);
        if (ci.pos >= ci.k0 && ci.pos < ci.k0 + CH) ci.newrow = ci.pos - ci.k0;
        ci.bad = ci.pos < 0 || ci.pos >= p.max_pos || ci.pos >= p.slots;
    } else {
        ci.pos = len;
        ci.nch = (p.slots + CH - 1) / CH;
        ci.nk = min(CH, p.slots - ci.k0);
        ci.ncached = ci.nk;
        const int slot = ci.pos % p.slots;
        if (slot >= ci.k0 && slot < ci.k0 + CH) ci.newrow = slot - ci.k0;
        ci.bad = ci.pos < 0 || ci.pos >= p.max_pos;
    }
    ci.rt = ci.rh = ci.rw = ci.pos;
    if (p.rope_pos && (p.mode == ATTN_TALKER || p.mode == ATTN_PREFILL)) {
        const int32_t* q3 = p.rope_pos + 3 * (size_t)r;
        ci.rt = __ldcg(q3);
        ci.rh = __ldcg(q3 + 1);
        ci.rw = __ldcg(q3 + 2);
        const int lo = min(ci.rt, min(ci.rh, ci.rw)), hi = max(ci.rt, max(ci.rh, ci.rw));
        if (lo < 0 || hi >= p.max_pos) ci.bad = true;
    }
    return ci;
}

// cos and sin of rotate_half rope frequency f for a row: from the table row of its cache
// position or, with per-axis rotary positions, of the position of the axis frequency f follows.
template <int HALF>
__device__ __forceinline__ void rope_cs(const AttnParams& p, const ChunkInfo& ci, int f, float& c,
                                        float& s) {
    int pf = ci.pos;
    if (p.rope_pos) {
        const int a = __ldg(p.rope_axis + f);
        pf = a == 1 ? ci.rh : (a == 2 ? ci.rw : ci.rt);
    }
    c = p.rope_cos[(size_t)pf * HALF + f];
    s = p.rope_sin[(size_t)pf * HALF + f];
}

// Thread 0 only: arm the mbarrier for the item's staged rows and start the two bulk copies.
// Exactly one phase of the barrier completes per call (also when there is nothing to copy).
template <int D>
__device__ __forceinline__ void chunk_issue(const AttnParams& p, int r, int g, const ChunkInfo& ci,
                                            const ChunkSmem& sm, uint32_t bar) {
    const size_t head_base = ((size_t)cache_stream(p, r) * p.G + g) * p.slots;
    const uint32_t bytes = (uint32_t)(ci.ncached > 0 ? ci.ncached : 0) * D * sizeof(float);
    mbar_arrive_expect_tx(bar, 2 * bytes);
    if (bytes) {
        bulk_g2s(smem_u32(sm.Ks), p.kc + (head_base + ci.k0) * D, bytes, bar);
        bulk_g2s(smem_u32(sm.Vs), p.vc + (head_base + ci.k0) * D, bytes, bar);
    }
}

// v[0..7] per lane -> lane l returns the warp-wide sum of v[(l >> 2) & 7]
__device__ __forceinline__ float butterfly8_keys(const float v[8], int lane) {
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

// The talker's new key and value of kv head g from raw q/k/v row `row` (per-head RMSNorm of k
// with the shared [d] weight, rotate_half rope at the row's positions `ci`; v as is), by one
// warp: element t = lane + 32 j of the results is written to k_out[t] and v_out[t].
template <int D>
__device__ __forceinline__ void talker_new_kv(const AttnParams& p, int row, int g,
                                              const ChunkInfo& ci, int lane, float* k_out,
                                              float* v_out) {
    constexpr int HALF = D / 2;
    const float* ksrc = p.qkv + (size_t)row * p.ldqkv + (size_t)p.H * D + (size_t)g * D;
    const float* vsrc = ksrc + (size_t)p.G * D;
    float v[D / 32];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
        v[j] = __ldcg(ksrc + lane + 32 * j);
        ss += v[j] * v[j];
    }
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)D + p.eps);
#pragma unroll
    for (int j = 0; j < D / 32; ++j) v[j] = v[j] * inv * p.kn[lane + 32 * j];
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
        const int t = lane + 32 * j;
        const int jj = (j + D / 64) % (D / 32);  // element t +- D/2, same lane
        const float rot = (t < HALF) ? -v[jj] : v[jj];
        const int f = t < HALF ? t : t - HALF;
        float c, s;
        rope_cs<HALF>(p, ci, f, c, s);
        k_out[t] = v[j] * c + rot * s;
        v_out[t] = __ldcg(vsrc + t);
    }
}

// The item's work once its copies were issued with chunk_issue (barrier phase `parity`): the
// prologue, the wait for the staged rows, the append, scores, the chunk softmax statistics and
// the partial (or, for a single-chunk stream, the final output).  The NT threads of a group call
// it (tid = index in the group, gbar = the group's named barrier); every output is computed the
// same way whatever NT is.  Returns false when the staged rows did not land within the wait
// bound (the status word then holds CHECK_WAIT_LIMIT and nothing was written).
template <int D, int NT = kChunkThreads>
__device__ bool chunk_compute(const AttnParams& p, int r, int g, int c, const ChunkInfo& ci,
                              const ChunkSmem& sm, uint32_t bar, uint32_t parity,
                              int tid = threadIdx.x, int gbar = 0) {
    constexpr int CH = kAttnChunk;
    constexpr int HALF = D / 2;
    constexpr int kChunkWarps = NT / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const int mode = p.mode;
    const int group = p.H / p.G;
    const float scale = 1.0f / sqrtf((float)D);
    const int pos = ci.pos, nk = ci.nk, k0 = ci.k0, newrow = ci.newrow, nch = ci.nch;
    float* const Ks = sm.Ks;
    float* const Vs = sm.Vs;
    float* const qs = sm.qs;
    float* const sc = sm.sc;

    // ---- prologue: q heads of the group (and the new key) -----------------------------------
    for (int i = warp; i < group; i += kChunkWarps) {
        const int hq = g * group + i;
        if (mode == ATTN_PLAIN) {
            for (int t = lane; t < D; t += 32)
                qs[i * D + t] = __ldcg(p.qkv + ((size_t)r * p.H + hq) * D + t);
        } else if (mode == ATTN_TALKER || mode == ATTN_PREFILL) {
            const float* src = p.qkv + (size_t)r * p.ldqkv + (size_t)hq * D;
            float v[D / 32];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                v[j] = __ldcg(src + lane + 32 * j);
                ss += v[j] * v[j];
            }
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)D + p.eps);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) v[j] = v[j] * inv * p.qn[lane + 32 * j];
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const int t = lane + 32 * j;
                const int jj = (j + D / 64) % (D / 32);       // element t +- D/2, same lane
                const float rot = (t < HALF) ? -v[jj] : v[jj];
                const int f = t < HALF ? t : t - HALF;
                float c, s;
                rope_cs<HALF>(p, ci, f, c, s);
                qs[i * D + t] = v[j] * c + rot * s;
            }
        } else {
            const float* src = p.qkv + (size_t)r * p.ldqkv + (size_t)hq * D;
            const float* cs = p.rope_cos + (size_t)pos * HALF;
            const float* sn = p.rope_sin + (size_t)pos * HALF;
            for (int j = lane; j < HALF; j += 32) {
                const float a = __ldcg(src + 2 * j), b = __ldcg(src + 2 * j + 1);
                qs[i * D + 2 * j] = a * cs[j] - b * sn[j];
                qs[i * D + 2 * j + 1] = a * sn[j] + b * cs[j];
            }
        }
    }
    if (newrow >= 0 && warp == (group % kChunkWarps)) {
        // the new key and value of kv head g at position pos
        if (mode == ATTN_TALKER) {
            talker_new_kv<D>(p, r, g, ci, lane, sm.knew, sm.vnew);
        } else {
            const int D_model = p.H * D;
            const float* ksrc = p.qkv + (size_t)r * p.ldqkv + D_model + (size_t)g * D;
            const float* vsrc = ksrc + D_model;
            const float* cs = p.rope_cos + (size_t)pos * HALF;
            const float* sn = p.rope_sin + (size_t)pos * HALF;
            for (int j = lane; j < HALF; j += 32) {
                const float a = __ldcg(ksrc + 2 * j), b = __ldcg(ksrc + 2 * j + 1);
                sm.knew[2 * j] = a * cs[j] - b * sn[j];
                sm.knew[2 * j + 1] = a * sn[j] + b * cs[j];
                sm.vnew[2 * j] = __ldcg(vsrc + 2 * j);
                sm.vnew[2 * j + 1] = __ldcg(vsrc + 2 * j + 1);
            }
        }
    }
    if (mode == ATTN_RING)
        for (int j = tid; j < nk; j += NT)
            sm.stamp[j] = __ldcg(p.pr + (size_t)r * p.slots + k0 + j);

    // ---- wait for the staged rows (bounded) ---------------------------------------------------
    const bool ok = mbar_wait_bounded(bar, parity);
    if (group_or<NT>(gbar, !ok)) {
        if (tid == 0) flag_check(p.status, CHECK_WAIT_LIMIT);
        mbar_wait_bounded(bar, parity);  // let copies still in flight land before moving on
        return false;
    }
    if (newrow >= 0) {
        const size_t head_base = ((size_t)cache_stream(p, r) * p.G + g) * p.slots;
        for (int t = tid; t < D; t += NT) {
            Ks[newrow * D + t] = sm.knew[t];
            Vs[newrow * D + t] = sm.vnew[t];
        }
        if (tid == 0 && mode == ATTN_RING) sm.stamp[newrow] = (uint32_t)pos;
        // append to the cache (after the staged copy has landed: no read/write overlap)
        float* kd = p.kc + (head_base + k0 + newrow) * D;
        float* vd = p.vc + (head_base + k0 + newrow) * D;
        for (int t = tid; t < D; t += NT) {
            kd[t] = sm.knew[t];
            vd[t] = sm.vnew[t];
        }
        if (tid == 0 && mode == ATTN_RING) p.pr[(size_t)r * p.slots + k0 + newrow] = (uint32_t)pos;
    }
    group_sync<NT>(gbar);

    // ---- scores: a warp takes 8 keys at a time, lanes split d, one butterfly per head ------------
    constexpr int PER = D / 32;  // dims per lane (contiguous)
    for (int j0 = warp * 8; j0 < nk; j0 += kChunkWarps * 8) {
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
            const float sum = butterfly8_keys(part, lane);   // lanes 4u..4u+3 hold key j0 + u
            const int u = (lane >> 2) & 7;
            if ((lane & 3) == 0 && j0 + u < nk) {
                bool legal = true;
                if (mode == ATTN_RING) {
                    const uint32_t pj = sm.stamp[j0 + u];
                    legal = (pj != 0xFFFFFFFFu) && (pj <= (uint32_t)pos) &&
                            ((uint32_t)pos - pj < (uint32_t)p.window);
                }
                sc[i * CH + j0 + u] = legal ? sum * scale : -CUDART_INF_F;
            }
        }
    }
    group_sync<NT>(gbar);

    // ---- chunk softmax statistics: warp per q head ---------------------------------------------
    for (int i = warp; i < group; i += kChunkWarps) {
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
            sm.s_m[i] = mx;
            sm.s_l[i] = l;
        }
    }
    group_sync<NT>(gbar);

    // ---- o_c = sum_j e_j v_j (ascending j), then write the partial ----------------------------
    for (int o = tid; o < group * D; o += NT) {
        const int i = o / D, t = o - i * D;
        // masked keys weigh exactly 0 and their V rows hold finite values (zeroed at creation)
        float acc = 0.f;
        const float* w = sc + i * CH;
#pragma unroll 8
        for (int j = 0; j < nk; ++j) acc += w[j] * Vs[j * D + t];
        const int hq = g * group + i;
        if (nch == 1) {
            p.out[((size_t)r * p.H + hq) * D + t] = acc / sm.s_l[i];
        } else {
            const size_t pi = ((size_t)r * p.H + hq) * p.max_chunks + c;
            p.part[pi * D + t] = acc;
            if (t == 0) {
                p.part_ml[2 * pi] = sm.s_m[i];
                p.part_ml[2 * pi + 1] = sm.s_l[i];
            }
        }
    }
    return true;
}

// Merge of the chunk partials of NT / D (q head, stream) items at once, D threads per item:
// items item0 .. min(item0 + NT/D, item_end) - 1 of the list r * H + hq.  Thread t of an item owns output
// dimension t and sums the chunks in ascending order.  The chunk statistics and the first
// FIRST partial values are fetched in one round of independent loads.  `scratch` holds
// 2 * max_chunks floats per item.  All NT threads call it (block-wide barriers inside).
constexpr int kMergeFirst = 48;      // partial rows of the first round (covers 3072 keys) ...
constexpr int kMergeFirstWide = 72;  // ... and in the stand-alone merge kernel (4608 keys), whose
                                     // CTAs have registers to spare
constexpr int kMergeBatch = 16;      // partial rows per later round

template <int D, int NT, int FIRST = kMergeFirst>
__device__ void merge_items(const AttnParams& p, int item0, int item_end, float* scratch) {
    constexpr int CH = kAttnChunk;
    const int sub = threadIdx.x / D, t = threadIdx.x - sub * D;
    const int item = item0 + sub;
    int nch = 0, r = 0, hq = 0;
    if (item < item_end) {
        r = item / p.H;
        hq = item - r * p.H;
        int L;
        if (p.mode == ATTN_PREFILL) L = __ldcg(p.len + p.stream) + r + 1;
        else if (p.mode == ATTN_PLAIN) L = __ldcg(p.len + r);
        else L = (p.mode == ATTN_TALKER) ? __ldcg(p.len + r) + 1 : p.slots;
        nch = (L + CH - 1) / CH;
        if (L < 1 || nch <= 1 || nch > p.max_chunks) nch = 0;  // one chunk: already final
    }
    float* sm = scratch + (size_t)sub * 2 * p.max_chunks;
    float* sw = sm + p.max_chunks;
    const size_t base = ((size_t)r * p.H + hq) * p.max_chunks;
    // first load pass: this thread's first partial values and its share of the chunk statistics
    float v0[FIRST];
#pragma unroll
    for (int u = 0; u < FIRST; ++u)
        v0[u] = u < nch ? __ldcg(p.part + (base + u) * D + t) : 0.f;
    float2 ml[(kMaxSlots / kAttnChunk + D - 1) / D];
#pragma unroll
    for (int q = 0; q < (kMaxSlots / kAttnChunk + D - 1) / D; ++q) {
        const int c = t + q * D;
        ml[q] = c < nch ? __ldcg(reinterpret_cast<const float2*>(p.part_ml) + base + c)
                        : make_float2(0.f, 0.f);
    }
    __syncthreads();  // the scratch may still be read by a previous call
#pragma unroll
    for (int q = 0; q < (kMaxSlots / kAttnChunk + D - 1) / D; ++q) {
        const int c = t + q * D;
        if (c < nch) {
            sm[c] = ml[q].y > 0.f ? ml[q].x : -CUDART_INF_F;
            sw[c] = ml[q].y;
        }
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
    if (nch == 0) return;
    float den = 0.f, num = 0.f;
    for (int c = 0; c < nch; ++c) den += sw[c];
#pragma unroll
    for (int u = 0; u < FIRST; ++u)
        if (u < nch) num += sm[u] * v0[u];
    for (int c0 = FIRST; c0 < nch; c0 += kMergeBatch) {
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

}  // namespace dec
