// gemv_rows.cuh -- the split-K row-streaming GEMV for m <= 8 rows as device functions, shared by
// the stand-alone kernel (gemv.cu) and its callers.
//
// y[r][n] = sum_k W[n][k] xin[r][k]; W row-major [N][K] (Qwen3-TTS talker on wgpu, MATVEC_SRC:
// each weight is read once for all rows), f32 or bf16 bit patterns widened exactly.
//
// All 256 threads of a CTA split K: warp w, lane l owns the 16-byte weight granules
// g = (8 j + w) 32 + l (j < NJ), so each warp-wide load is 512 contiguous bytes of one row and
// the CTA's threads together cover a whole row.  A thread's slice of x is only NJ granules wide,
// so x lives in registers; the norm prologue is a block reduction over those registers.  The
// CTA's rows are streamed in batches of RB rows, the next batch's loads in flight while the
// current one is consumed (two register buffers).  The caller issues the first two batches
// (issue()) before it waits for x -- weights never depend on earlier work -- and run() does the
// rest.  Each warp folds 8 rows' partials at a time across lanes with a transposed butterfly
// (lanes 4r..4r+3 end up holding row r): per batch of RB >= 8 rows, or, for one or two rows of x
// and smaller batches, once per 8 / RB batches; the cross-warp sum and the epilogue run once per
// segment of at most kRowsMaxRows rows.
//
// Activations (x, the residual) are read with ld.global.cg (L2): they were written by the
// previous kernel of the chain, on other SMs.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dec {

constexpr int kRowsThreads = 256;
constexpr int kRowsWarps = kRowsThreads / 32;
constexpr int kRowsMaxRows = 128;  // rows per segment the cross-warp scratch holds

// shared-memory floats run() needs: cross-warp row sums, norm partials, norm statistics
template <int MT>
__host__ __device__ constexpr int rows_smem_floats() {
    return kRowsWarps * kRowsMaxRows * MT + kRowsWarps * MT + 2 * MT;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float gelu_f(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752440f));
}

// v[0..7] per lane -> lane l returns the warp-wide sum of v[(l >> 2) & 7]
__device__ __forceinline__ float butterfly8(const float v[8], int lane) {
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

template <int DT>
struct WType;
template <>
struct WType<0> {  // f32 weights
    static constexpr int VEC = 4;
    static constexpr int ES = 4;
};
template <>
struct WType<1> {  // bf16 weights
    static constexpr int VEC = 8;
    static constexpr int ES = 2;
};

// BUF: 16-byte weight registers per buffer and thread (two buffers in flight); a batch is
// RB = BUF / NJ rows.  8 suits two CTAs per SM, 16 one CTA per SM with the larger register file.
template <int DT, int MT, int NJ, int BUF>
struct RowsGemv {
    static constexpr int VEC = WType<DT>::VEC;
    static constexpr int ES = WType<DT>::ES;
    static constexpr int RB = BUF / NJ;  // rows per batch
    static_assert(RB >= 1 && RB * NJ <= BUF, "weight buffer");

    // rows [row0, row0 + nrows) of CTA b of P: whole partition units (2 rows for SwiGLU pairs)
    __device__ static void range(const GemvParams& p, int b, int P, int& row0, int& nrows) {
        const int units = p.N / p.unit;
        const int u0 = (int)((long long)b * units / P);
        const int u1 = (int)((long long)(b + 1) * units / P);
        row0 = u0 * p.unit;
        nrows = (u1 - u0) * p.unit;
    }

    // batch of RB rows starting at row `first` of the CTA (rows at or past `lim` load zeros)
    __device__ static void load(const GemvParams& p, const char* Wb, size_t row_bytes, int first,
                                int lim, uint64_t pol, uint4 (&w)[BUF]) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int G = p.K / VEC;
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int gj = (j * kRowsWarps + warp) * 32 + lane;
                w[r * NJ + j] = (first + r < lim && gj < G)
                                    ? ld_stream16(Wb + (size_t)(first + r) * row_bytes + (size_t)gj * 16, pol)
                                    : make_uint4(0u, 0u, 0u, 0u);
            }
    }

    // the first two batches of CTA b's rows (pol: the weights' L2 policy)
    __device__ static void issue(const GemvParams& p, int b, int P, uint4 (&wa)[BUF],
                                 uint4 (&wb)[BUF], uint64_t pol) {
        int row0, nrows;
        range(p, b, P, row0, nrows);
        const size_t row_bytes = (size_t)p.K * ES;
        const char* Wb = static_cast<const char*>(p.W) + (size_t)row0 * row_bytes;
        const int lim = nrows < kRowsMaxRows ? nrows : kRowsMaxRows;
        load(p, Wb, row_bytes, 0, lim, pol, wa);
        load(p, Wb, row_bytes, RB, lim, pol, wb);
    }

    // A thread's share of one CTA's rows: the row range, its weight granules, its slice of x
    // (normalised in place by the prologue) and its prefetched residual-epilogue operands.
    struct Lane {
        int row0, nrows;
        int gj[NJ];
        bool ok[NJ];
        float2 xv[MT][NJ][VEC / 2];
        float res_v, ls_v, bias_v;
    };

    // The residual epilogue's operands of this thread's output (row tid / m, stream tid % m),
    // fetched together with x rather than after the rows are summed.  With m <= 2 a segment
    // has at most kRowsMaxRows * 2 <= kRowsThreads outputs, one per thread; wider rows read
    // them in the epilogue's loop instead.
    static constexpr bool kEpiPrefetch = MT <= 2;

    __device__ static void setup(const GemvParams& p, int b, int P, Lane& L) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        range(p, b, P, L.row0, L.nrows);
        const int G = p.K / VEC;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            L.gj[j] = (j * kRowsWarps + warp) * 32 + lane;
            L.ok[j] = L.gj[j] < G;
        }
        L.res_v = L.ls_v = L.bias_v = 0.f;
    }

    __device__ static void fetch_epi(const GemvParams& p, Lane& L, int seg) {
        if constexpr (!kEpiPrefetch) return;
        const int tid = threadIdx.x, m = p.m;
        const int srows = L.nrows - seg < kRowsMaxRows ? L.nrows - seg : kRowsMaxRows;
        if (tid < srows * m) {
            const int row = L.row0 + seg + tid / m, mm = tid % m;
            if (p.bias) L.bias_v = p.bias[row];
            if (p.epi == EPI_RESID) {
                L.res_v = __ldcg(p.res + (size_t)mm * p.ldres + row);
                if (p.ls) L.ls_v = __ldcg(p.ls + row);
            }
        }
    }

    // x slice into registers, then the norm prologue (a block reduction).  Every thread of the
    // CTA calls it (block-wide barriers inside).
    __device__ static void prologue(const GemvParams& p, Lane& L, float* sh) {
        float* nred = sh + kRowsWarps * kRowsMaxRows * MT;  // [warps][MT]
        float* stat = nred + kRowsWarps * MT;               // [2][MT]
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        const int K = p.K, m = p.m;
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float* src = p.x + (size_t)mm * p.ldx + (size_t)L.gj[j] * VEC;
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q) {
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (mm < m && L.ok[j]) a = __ldcg(reinterpret_cast<const float4*>(src + 4 * q));
                    L.xv[mm][j][2 * q] = make_float2(a.x, a.y);
                    L.xv[mm][j][2 * q + 1] = make_float2(a.z, a.w);
                }
            }
        if (p.pro == PRO_NONE) return;
        auto block_sum = [&](float (&v)[MT], int slot) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                const float t = warp_sum(v[mm]);
                if (lane == 0) nred[warp * MT + mm] = t;
            }
            __syncthreads();
            if (tid < MT) {
                float sum = 0.f;
                for (int w = 0; w < kRowsWarps; ++w) sum += nred[w * MT + tid];
                stat[slot * MT + tid] = sum / (float)K;
            }
            __syncthreads();
        };
        float part[MT];
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
            part[mm] = 0.f;
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < VEC / 2; ++e) {
                    const float2 v = L.xv[mm][j][e];
                    part[mm] += (p.pro != PRO_RMS) ? v.x + v.y : v.x * v.x + v.y * v.y;
                }
        }
        block_sum(part, 0);  // mean (LayerNorm) or mean square (RMSNorm)
        float inv[MT], mean[MT];
        if (p.pro != PRO_RMS) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                mean[mm] = stat[mm];
                part[mm] = 0.f;
#pragma unroll
                for (int j = 0; j < NJ; ++j)
#pragma unroll
                    for (int e = 0; e < VEC / 2; ++e) {
                        if (!L.ok[j]) continue;
                        const float dx = L.xv[mm][j][e].x - mean[mm], dy = L.xv[mm][j][e].y - mean[mm];
                        part[mm] += dx * dx + dy * dy;
                    }
            }
            block_sum(part, 1);
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) inv[mm] = 1.0f / sqrtf(stat[MT + mm] + p.eps);
        } else {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                mean[mm] = 0.f;
                inv[mm] = 1.0f / sqrtf(stat[mm] + p.eps);
            }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            if (!L.ok[j]) continue;
            const int k0 = L.gj[j] * VEC;
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) {
                // a LayerNorm without affine weights (the flow head's final norm) is w 1, b 0
                const float2 w = p.nw ? *reinterpret_cast<const float2*>(p.nw + k0 + 2 * e)
                                      : make_float2(1.f, 1.f);
                float2 bb = make_float2(0.f, 0.f);
                if (p.pro != PRO_RMS && p.nb) bb = *reinterpret_cast<const float2*>(p.nb + k0 + 2 * e);
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) {
                    float2& v = L.xv[mm][j][e];
                    v.x = (v.x - mean[mm]) * inv[mm] * w.x + bb.x;
                    v.y = (v.y - mean[mm]) * inv[mm] * w.y + bb.y;
                }
                if (p.pro == PRO_LN_MOD) {  // modulate: n (1 + scale) + shift
                    const float2 sh2 = __ldcg(reinterpret_cast<const float2*>(p.mod + k0 + 2 * e));
                    const float2 sc = __ldcg(reinterpret_cast<const float2*>(p.mod + K + k0 + 2 * e));
#pragma unroll
                    for (int mm = 0; mm < MT; ++mm) {
                        float2& v = L.xv[mm][j][e];
                        v.x = v.x * (1.0f + sc.x) + sh2.x;
                        v.y = v.y * (1.0f + sc.y) + sh2.y;
                    }
                }
            }
        }
    }

    // One batch of RB rows (rows b0.. of the segment; rows at or past lim are not stored): the
    // thread's partial dot products, folded across lanes, into the cross-warp scratch.
    __device__ static void consume(const uint4 (&w)[BUF], int b0, int lim, const Lane& L,
                                   float* red) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int g8 = 0; g8 < RB; g8 += 8) {  // 8 rows per transposed butterfly
            float part[MT][8];
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                for (int r = 0; r < 8; ++r) part[mm][r] = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (g8 + r >= RB) break;
                float2 acc[MT];
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) acc[mm] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const uint4 wr = w[(g8 + r) * NJ + j];
                    float2 wf[VEC / 2];
                    if constexpr (DT == 1) {
                        wf[0] = bf16x2_to_f32x2(wr.x);
                        wf[1] = bf16x2_to_f32x2(wr.y);
                        wf[2] = bf16x2_to_f32x2(wr.z);
                        wf[3] = bf16x2_to_f32x2(wr.w);
                    } else {
                        wf[0] = make_float2(__uint_as_float(wr.x), __uint_as_float(wr.y));
                        wf[1] = make_float2(__uint_as_float(wr.z), __uint_as_float(wr.w));
                    }
#pragma unroll
                    for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                        for (int e = 0; e < VEC / 2; ++e) acc[mm] = ffma2(wf[e], L.xv[mm][j][e], acc[mm]);
                }
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) part[mm][r] = acc[mm].x + acc[mm].y;
            }
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                const float v = butterfly8(part[mm], lane);
                const int r = (lane >> 2) & 7;
                if ((lane & 3) == 0 && g8 + r < RB && b0 + g8 + r < lim)
                    red[(warp * kRowsMaxRows + b0 + g8 + r) * MT + mm] = v;
            }
        }
    }

    // Batches of fewer than 8 rows (one or two rows of x): the rows of 8 / RB consecutive batches (8 rows, alternating
    // buffers, each refilled with the batch two ahead once consumed) share one transposed
    // butterfly, instead of a butterfly per batch with most of its 8 rows empty.  Rows at or past
    // lim compute on whatever the buffer holds and are not stored.
    __device__ static void consume8(const GemvParams& p, const char* Ws, size_t row_bytes,
                                    uint64_t pol, uint4 (&wa)[BUF], uint4 (&wb)[BUF], int b0,
                                    int lim, const Lane& L, float* red) {
        static_assert(RB < 8 && 8 % (2 * RB) == 0, "8 rows in pairs of batches");
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        float part[MT][8];
#pragma unroll
        for (int i = 0; i < 8 / RB; ++i) {
            uint4(&w)[BUF] = (i & 1) ? wb : wa;
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float2 acc[MT];
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) acc[mm] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const uint4 wr = w[r * NJ + j];
                    float2 wf[VEC / 2];
                    if constexpr (DT == 1) {
                        wf[0] = bf16x2_to_f32x2(wr.x);
                        wf[1] = bf16x2_to_f32x2(wr.y);
                        wf[2] = bf16x2_to_f32x2(wr.z);
                        wf[3] = bf16x2_to_f32x2(wr.w);
                    } else {
                        wf[0] = make_float2(__uint_as_float(wr.x), __uint_as_float(wr.y));
                        wf[1] = make_float2(__uint_as_float(wr.z), __uint_as_float(wr.w));
                    }
#pragma unroll
                    for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                        for (int e = 0; e < VEC / 2; ++e) acc[mm] = ffma2(wf[e], L.xv[mm][j][e], acc[mm]);
                }
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) part[mm][i * RB + r] = acc[mm].x + acc[mm].y;
            }
            const int next = b0 + i * RB + 2 * RB;  // the batch this buffer takes next
            if (next < lim) load(p, Ws, row_bytes, next, lim, pol, w);
        }
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
            const float v = butterfly8(part[mm], lane);
            const int r = (lane >> 2) & 7;
            if ((lane & 3) == 0 && b0 + r < lim) red[(warp * kRowsMaxRows + b0 + r) * MT + mm] = v;
        }
    }

    // Cross-warp sums of a segment's srows rows and the epilogue (after a block barrier).
    __device__ static void epilogue(const GemvParams& p, Lane& L, int seg, int srows,
                                    const float* red) {
        const int tid = threadIdx.x, m = p.m;
        const int rbase = L.row0 + seg;
        if (p.epi == EPI_SWIGLU) {
            for (int o = tid; o < (srows / 2) * m; o += kRowsThreads) {
                const int pr = o / m, mm = o - pr * m;
                float vg = 0.f, vu = 0.f;
                for (int w = 0; w < kRowsWarps; ++w) {
                    vg += red[(w * kRowsMaxRows + 2 * pr) * MT + mm];
                    vu += red[(w * kRowsMaxRows + 2 * pr + 1) * MT + mm];
                }
                p.y[(size_t)mm * p.ldy + rbase / 2 + pr] = silu_f(vg) * vu;
            }
            return;
        }
        for (int o = tid; o < srows * m; o += kRowsThreads) {
            const int r = o / m, mm = o - r * m;
            float v = 0.f;
            for (int w = 0; w < kRowsWarps; ++w) v += red[(w * kRowsMaxRows + r) * MT + mm];
            const int row = rbase + r;
            if constexpr (!kEpiPrefetch) {
                if (p.bias) L.bias_v = p.bias[row];
                if (p.epi == EPI_RESID) {
                    L.res_v = __ldcg(p.res + (size_t)mm * p.ldres + row);
                    if (p.ls) L.ls_v = __ldcg(p.ls + row);
                }
            }
            if (p.bias) v += L.bias_v;
            float out;
            if (p.epi == EPI_RESID) {
                const float tt = p.ls ? L.ls_v * v : v;
                out = L.res_v + tt;
                if (p.tap) p.tap[(size_t)mm * p.ldtap + row] = out;
            } else if (p.epi == EPI_GELU) {
                out = gelu_f(v);
            } else {
                out = p.act == 1 ? silu_f(v) : v;
            }
            p.y[(size_t)mm * p.ldy + row] = out;
        }
    }

    // everything after issue(): x and the norm prologue, the remaining batches, the epilogue.
    // Every thread of the CTA calls it (block-wide barriers inside).
    __device__ static void run(const GemvParams& p, int b, int P, uint4 (&wa)[BUF],
                               uint4 (&wb)[BUF], float* sh, uint64_t pol) {
        float* red = sh;  // [warps][kRowsMaxRows][MT]
        Lane L;
        setup(p, b, P, L);
        const size_t row_bytes = (size_t)p.K * ES;
        const char* Wb = static_cast<const char*>(p.W) + (size_t)L.row0 * row_bytes;
        if (L.nrows > 0) fetch_epi(p, L, 0);
        prologue(p, L, sh);

        // ---- stream the rows, segment by segment, in double-buffered batches ------------------
        for (int seg = 0; seg < L.nrows; seg += kRowsMaxRows) {
            const int srows = L.nrows - seg < kRowsMaxRows ? L.nrows - seg : kRowsMaxRows;
            const char* Ws = Wb + (size_t)seg * row_bytes;
            if (seg > 0) {  // the first segment's first two batches came from issue()
                load(p, Ws, row_bytes, 0, srows, pol, wa);
                load(p, Ws, row_bytes, RB, srows, pol, wb);
                fetch_epi(p, L, seg);
            }
            // ping-pong: while one batch is consumed the other is in flight
            // (not with four granules, nor with x of 4 or 8 rows: the 8 rows' partials would stay
            // live across the batches in a register file that is already full)
            if constexpr (RB < 8 && NJ <= 3 && MT <= 2) {
                for (int b0 = 0; b0 < srows; b0 += 8)
                    consume8(p, Ws, row_bytes, pol, wa, wb, b0, srows, L, red);
            } else {
                for (int b0 = 0; b0 < srows; b0 += 2 * RB) {
                    consume(wa, b0, srows, L, red);
                    if (b0 + 2 * RB < srows) load(p, Ws, row_bytes, b0 + 2 * RB, srows, pol, wa);
                    if (b0 + RB < srows) consume(wb, b0 + RB, srows, L, red);
                    if (b0 + 3 * RB < srows) load(p, Ws, row_bytes, b0 + 3 * RB, srows, pol, wb);
                }
            }
            __syncthreads();
            epilogue(p, L, seg, srows, red);
            if (seg + kRowsMaxRows < L.nrows) __syncthreads();  // red is reused by the next segment
        }
    }
};

// granules per lane of the split-K GEMV for this shape (0: not served by it): up to 4 for
// m <= 2; for 3..8 rows up to 3, x of at most 4 rows in registers at a time (4 rows x 3
// granules: 96 registers a thread).  With one granule x holds all 8 rows (64 registers); wider
// rows of 5..8 are two passes over the weights (k_gemv_rows2).
inline int rows_gemv_nj(int K, int m, int dtype) {
    const int vec = dtype == 1 ? 8 : 4;
    const int per_pass = kRowsThreads * vec;  // elements one pass of the CTA covers
    const int nj = (K + per_pass - 1) / per_pass;
    if (nj < 1 || m < 1) return 0;
    if (m <= 2) return nj <= 4 ? nj : 0;
    return (m <= 8 && nj <= 3) ? nj : 0;
}

}  // namespace dec
