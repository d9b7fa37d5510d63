// gemv.cu -- bandwidth-bound row-major GEMV for the decode step (sm_103a).
//
// y[r][n] = sum_k W[n][k] xin[r][k] for the m <= 8 rows of one step; W is row-major [N][K] as a
// Linear stores it (Qwen3-TTS talker on wgpu, MATVEC_SRC: "each weight is read exactly once"),
// f32 or bf16 bit patterns widened exactly in registers.
//
// Layout of the work: a warp owns two consecutive rows at a time; its 32 lanes split K in
// 16-byte pieces (8 bf16 or 4 f32 per lane per step), so every weight load is a coalesced
// 512-byte warp access issued as ld.global.nc.L1::no_allocate.v4.  Four steps per row (eight
// 16-byte loads per lane) are in flight before any arithmetic.  Row sums are finished with warp
// shuffles.  The first batch of weight loads is issued BEFORE griddepcontrol.wait: weights never
// depend on the previous kernel, so they stream in while that kernel drains.
//
// Prologue (optional): the CTA stages x in shared memory and applies RMSNorm (talker RMSNORM_SRC)
// or LayerNorm (Mimi ln_src) in place.  Epilogues: store; residual add with optional LayerScale
// (the talker's ADD after o/down, Mimi MV_LS); SwiGLU over interleaved gate/up rows (SWIGLU_SRC);
// GELU(erf) (GELU_ERF, with CUDA's erff).
#include "common.cuh"
#include "kernels.h"

namespace dec {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kRows = 2;     // rows per warp task (a gate/up pair for SwiGLU)
constexpr int kUnroll = 4;   // 16-byte steps per row in flight

template <int DT>
struct WT;
template <>
struct WT<0> {  // f32 weights
    static constexpr int VEC = 4;
    static constexpr int ES = 4;
};
template <>
struct WT<1> {  // bf16 weights
    static constexpr int VEC = 8;
    static constexpr int ES = 2;
};

// Shared-memory position of x element k.  For bf16 a lane consumes 8 consecutive k per step;
// storing each 256-wide block as [half][lane][4] lets the lane fetch its 8 values with two
// conflict-free 16-byte reads (at lane*4 and 128 + lane*4).
template <int DT>
__device__ __forceinline__ int sx_index(int k) {
    if constexpr (DT == 0) return k;
    int blk = k & ~255, w = k & 255;
    int l = w >> 3, j = w & 7;
    return blk + ((j >> 2) << 7) + (l << 2) + (j & 3);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float gelu_f(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752440f));
}

template <int DT, int MT>
__global__ void __launch_bounds__(kGemvThreads, 2) k_gemv(const GemvParams p) {
    extern __shared__ __align__(16) float sx[];  // [m][ldsx]
    __shared__ float red[kGemvWarps][MT];
    __shared__ float stat[2][MT];

    constexpr int VEC = WT<DT>::VEC;
    constexpr int ES = WT<DT>::ES;
    constexpr int KS = 32 * VEC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int N = p.N, K = p.K, m = p.m;
    const int nsteps = (K + KS - 1) / KS;
    const int ldsx = nsteps * KS;
    const int ngroups = (N + kRows - 1) / kRows;
    const int total_warps = gridDim.x * kGemvWarps;
    int g = blockIdx.x * kGemvWarps + warp;
    const char* Wb = static_cast<const char*>(p.W);
    const size_t row_bytes = (size_t)K * ES;

    uint4 wv[kUnroll][kRows];
    auto load_batch = [&](int grp, int s0) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int k = (s0 + u) * KS + lane * VEC;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int row = grp * kRows + r;
                if (k < K && row < N)
                    wv[u][r] = ld_stream16(Wb + (size_t)row * row_bytes + (size_t)k * ES);
                else
                    wv[u][r] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };

    // weights first: independent of the previous kernel
    bool preloaded = g < ngroups;
    if (preloaded) load_batch(g, 0);
    pdl_trigger();
    pdl_wait();

    // ---- stage x (rows < m), zero the padding, apply the norm prologue -------------------
    for (int i = tid; i < m * (ldsx / 4); i += kGemvThreads) {
        const int mm = i / (ldsx / 4);
        const int k = (i - mm * (ldsx / 4)) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < K) v = *reinterpret_cast<const float4*>(p.x + (size_t)mm * p.ldx + k);
        *reinterpret_cast<float4*>(sx + mm * ldsx + sx_index<DT>(k)) = v;
    }
    __syncthreads();
    if (p.pro != PRO_NONE) {
        // pass 1: LayerNorm mean (sum x) or RMSNorm sum of squares
        float part[MT];
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
            part[mm] = 0.f;
            if (mm < m)
                for (int k = tid; k < K; k += kGemvThreads) {
                    const float v = sx[mm * ldsx + sx_index<DT>(k)];
                    part[mm] += (p.pro == PRO_LN) ? v : v * v;
                }
            part[mm] = warp_sum(part[mm]);
        }
        if (lane == 0)
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) red[warp][mm] = part[mm];
        __syncthreads();
        if (tid < MT) {
            float s = 0.f;
            for (int w = 0; w < kGemvWarps; ++w) s += red[w][tid];
            stat[0][tid] = s / (float)K;  // mean (LN) or mean square (RMS)
        }
        __syncthreads();
        if (p.pro == PRO_LN) {
            // pass 2: biased variance of the deviations
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                part[mm] = 0.f;
                if (mm < m) {
                    const float mean = stat[0][mm];
                    for (int k = tid; k < K; k += kGemvThreads) {
                        const float dv = sx[mm * ldsx + sx_index<DT>(k)] - mean;
                        part[mm] += dv * dv;
                    }
                }
                part[mm] = warp_sum(part[mm]);
            }
            if (lane == 0)
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) red[warp][mm] = part[mm];
            __syncthreads();
            if (tid < MT) {
                float s = 0.f;
                for (int w = 0; w < kGemvWarps; ++w) s += red[w][tid];
                stat[1][tid] = 1.0f / sqrtf(s / (float)K + p.eps);
            }
        } else if (tid < MT) {
            stat[1][tid] = 1.0f / sqrtf(stat[0][tid] + p.eps);
        }
        __syncthreads();
        for (int i = tid; i < m * K; i += kGemvThreads) {
            const int mm = i / K, k = i - mm * K;
            float& v = sx[mm * ldsx + sx_index<DT>(k)];
            if (p.pro == PRO_LN)
                v = (v - stat[0][mm]) * stat[1][mm] * p.nw[k] + p.nb[k];
            else
                v = v * stat[1][mm] * p.nw[k];
        }
        __syncthreads();
    }

    // ---- main loop ---------------------------------------------------------------------
    for (; g < ngroups; g += total_warps) {
        float2 acc[kRows][MT];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) acc[r][mm] = make_float2(0.f, 0.f);

        for (int s0 = 0; s0 < nsteps; s0 += kUnroll) {
            if (!preloaded) load_batch(g, s0);
            preloaded = false;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int step = s0 + u;
                if (step * KS + lane * VEC >= K) continue;
                float2 wf[kRows][VEC / 2];
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    if constexpr (DT == 1) {
                        wf[r][0] = bf16x2_to_f32x2(wv[u][r].x);
                        wf[r][1] = bf16x2_to_f32x2(wv[u][r].y);
                        wf[r][2] = bf16x2_to_f32x2(wv[u][r].z);
                        wf[r][3] = bf16x2_to_f32x2(wv[u][r].w);
                    } else {
                        wf[r][0] = make_float2(__uint_as_float(wv[u][r].x),
                                               __uint_as_float(wv[u][r].y));
                        wf[r][1] = make_float2(__uint_as_float(wv[u][r].z),
                                               __uint_as_float(wv[u][r].w));
                    }
                }
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) {
                    if (mm >= m) break;
                    const float* xs = sx + mm * ldsx + step * KS;
                    float2 xv[VEC / 2];
                    if constexpr (DT == 1) {
                        const float4 a = *reinterpret_cast<const float4*>(xs + lane * 4);
                        const float4 b = *reinterpret_cast<const float4*>(xs + 128 + lane * 4);
                        xv[0] = make_float2(a.x, a.y);
                        xv[1] = make_float2(a.z, a.w);
                        xv[2] = make_float2(b.x, b.y);
                        xv[3] = make_float2(b.z, b.w);
                    } else {
                        const float4 a = *reinterpret_cast<const float4*>(xs + lane * 4);
                        xv[0] = make_float2(a.x, a.y);
                        xv[1] = make_float2(a.z, a.w);
                    }
#pragma unroll
                    for (int r = 0; r < kRows; ++r)
#pragma unroll
                        for (int j = 0; j < VEC / 2; ++j) acc[r][mm] = ffma2(wf[r][j], xv[j], acc[r][mm]);
                }
            }
        }

        // ---- reduce over lanes and run the epilogue --------------------------------------
        const int row0 = g * kRows;
        if (p.epi == EPI_SWIGLU) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                if (mm >= m) break;
                const float vg = warp_sum(acc[0][mm].x + acc[0][mm].y);
                const float vu = warp_sum(acc[1][mm].x + acc[1][mm].y);
                if (lane == mm && row0 + 1 < N) p.y[(size_t)mm * p.ldy + g] = silu_f(vg) * vu;
            }
        } else {
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) {
                    if (mm >= m) break;
                    const float v = warp_sum(acc[r][mm].x + acc[r][mm].y);
                    const int row = row0 + r;
                    if (lane != r * MT + mm || row >= N) continue;
                    float out;
                    if (p.epi == EPI_RESID) {
                        const float t = p.ls ? p.ls[row] * v : v;
                        out = p.res[(size_t)mm * p.ldres + row] + t;
                        if (p.tap) p.tap[(size_t)mm * p.ldtap + row] = out;
                    } else if (p.epi == EPI_GELU) {
                        out = gelu_f(v);
                    } else {
                        out = v;
                    }
                    p.y[(size_t)mm * p.ldy + row] = out;
                }
            }
        }
    }
}

// =============================================================================================
// Split-K row-streaming GEMV for m <= 2 (the decode step's common case).
//
// All 256 threads of a CTA split K: warp w, lane l owns the 16-byte weight granules
// g = (8 j + w) 32 + l (j < NJ), so each warp-wide load is 512 contiguous bytes of one row and
// the CTA's threads together cover a whole row.  A thread's slice of x is only NJ granules wide,
// so x lives in registers, loaded once; the norm prologue is a block reduction over those
// registers (no shared-memory staging).  The CTA's rows are streamed in batches of RB rows with
// the next batch's loads in flight while the current one is consumed (double-buffered
// registers); the first batch is issued before griddepcontrol.wait.  Per batch, each warp folds
// its RB row partials across lanes with a transposed butterfly (lanes 4r..4r+3 end up holding
// row r), and the cross-warp sum plus the epilogue run once at the end of the CTA.
// =============================================================================================
constexpr int kRowsThreads = 256;
constexpr int kRowsWarps = kRowsThreads / 32;
constexpr int kRowsMaxRows = 64;  // rows per CTA the cross-warp scratch holds

// v[0..7] per lane -> lane l returns the warp-wide sum of v[(l >> 2) & 7]
__device__ __forceinline__ float butterfly8(float v[8], int lane) {
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

template <int DT, int MT, int NJ>
__global__ void __launch_bounds__(kRowsThreads, 2) k_gemv_rows(const GemvParams p) {
    constexpr int VEC = WT<DT>::VEC;
    constexpr int ES = WT<DT>::ES;
    constexpr int RB = NJ >= 8 ? 1 : 8 / NJ;   // rows per batch (8 loads per lane in flight)
    __shared__ float red[kRowsWarps][kRowsMaxRows][MT];
    __shared__ float nred[kRowsWarps][MT];
    __shared__ float stat[2][MT];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, m = p.m;
    const int G = K / VEC;
    const size_t row_bytes = (size_t)K * ES;
    const int units = p.N / p.unit;
    const int u0 = (int)((long long)blockIdx.x * units / gridDim.x);
    const int u1 = (int)((long long)(blockIdx.x + 1) * units / gridDim.x);
    const int row0 = u0 * p.unit, nrows = (u1 - u0) * p.unit;
    const char* Wb = static_cast<const char*>(p.W) + (size_t)row0 * row_bytes;

    int gj[NJ];
    bool ok[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        gj[j] = (j * kRowsWarps + warp) * 32 + lane;
        ok[j] = gj[j] < G;
    }
    const uint64_t pol = l2_evict_first();
    uint4 wa[RB][NJ], wb[RB][NJ];
    auto load = [&](uint4 (&w)[RB][NJ], int b0) {
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int j = 0; j < NJ; ++j)
                w[r][j] = (b0 + r < nrows && ok[j])
                              ? ld_stream16(Wb + (size_t)(b0 + r) * row_bytes + (size_t)gj[j] * 16, pol)
                              : make_uint4(0u, 0u, 0u, 0u);
    };

    // weights first: independent of the previous kernel, so two batches are in flight before
    // the wait (a whole CTA's rows when it owns at most 2 * RB of them)
    load(wa, 0);
    load(wb, RB);
    pdl_trigger();
    pdl_wait();

    // ---- x slice in registers, norm prologue as a block reduction ---------------------------
    float2 xv[MT][NJ][VEC / 2];
#pragma unroll
    for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const float* src = p.x + (size_t)mm * p.ldx + (size_t)gj[j] * VEC;
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                if (mm < m && ok[j]) a = *reinterpret_cast<const float4*>(src + 4 * q);
                xv[mm][j][2 * q] = make_float2(a.x, a.y);
                xv[mm][j][2 * q + 1] = make_float2(a.z, a.w);
            }
        }
    if (p.pro != PRO_NONE) {
        auto block_sum = [&](float (&v)[MT], int slot) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                const float t = warp_sum(v[mm]);
                if (lane == 0) nred[warp][mm] = t;
            }
            __syncthreads();
            if (tid < MT) {
                float sum = 0.f;
                for (int w = 0; w < kRowsWarps; ++w) sum += nred[w][tid];
                stat[slot][tid] = sum / (float)K;
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
                    const float2 v = xv[mm][j][e];
                    part[mm] += (p.pro == PRO_LN) ? v.x + v.y : v.x * v.x + v.y * v.y;
                }
        }
        block_sum(part, 0);  // mean (LayerNorm) or mean square (RMSNorm)
        float inv[MT], mean[MT];
        if (p.pro == PRO_LN) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                mean[mm] = stat[0][mm];
                part[mm] = 0.f;
#pragma unroll
                for (int j = 0; j < NJ; ++j)
#pragma unroll
                    for (int e = 0; e < VEC / 2; ++e) {
                        if (!ok[j]) continue;
                        const float dx = xv[mm][j][e].x - mean[mm], dy = xv[mm][j][e].y - mean[mm];
                        part[mm] += dx * dx + dy * dy;
                    }
            }
            block_sum(part, 1);
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) inv[mm] = 1.0f / sqrtf(stat[1][mm] + p.eps);
        } else {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                mean[mm] = 0.f;
                inv[mm] = 1.0f / sqrtf(stat[0][mm] + p.eps);
            }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            if (!ok[j]) continue;
            const int k0 = gj[j] * VEC;
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) {
                const float2 w = *reinterpret_cast<const float2*>(p.nw + k0 + 2 * e);
                float2 b = make_float2(0.f, 0.f);
                if (p.pro == PRO_LN) b = *reinterpret_cast<const float2*>(p.nb + k0 + 2 * e);
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) {
                    float2& v = xv[mm][j][e];
                    v.x = (v.x - mean[mm]) * inv[mm] * w.x + b.x;
                    v.y = (v.y - mean[mm]) * inv[mm] * w.y + b.y;
                }
            }
        }
    }

    // ---- stream the CTA's rows in double-buffered batches --------------------------------------
    auto consume = [&](const uint4 (&w)[RB][NJ], int b0) {
        float part[MT][8];
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
            for (int r = 0; r < 8; ++r) part[mm][r] = 0.f;
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float2 acc[MT];
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) acc[mm] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                float2 wf[VEC / 2];
                if constexpr (DT == 1) {
                    wf[0] = bf16x2_to_f32x2(w[r][j].x);
                    wf[1] = bf16x2_to_f32x2(w[r][j].y);
                    wf[2] = bf16x2_to_f32x2(w[r][j].z);
                    wf[3] = bf16x2_to_f32x2(w[r][j].w);
                } else {
                    wf[0] = make_float2(__uint_as_float(w[r][j].x), __uint_as_float(w[r][j].y));
                    wf[1] = make_float2(__uint_as_float(w[r][j].z), __uint_as_float(w[r][j].w));
                }
#pragma unroll
                for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                    for (int e = 0; e < VEC / 2; ++e) acc[mm] = ffma2(wf[e], xv[mm][j][e], acc[mm]);
            }
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) part[mm][r] = acc[mm].x + acc[mm].y;
        }
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
            const float v = butterfly8(part[mm], lane);
            const int r = (lane >> 2) & 7;
            if ((lane & 3) == 0 && r < RB && b0 + r < nrows) red[warp][b0 + r][mm] = v;
        }
    };
    // ping-pong: while one batch is consumed the other is in flight
    for (int b0 = 0; b0 < nrows; b0 += 2 * RB) {
        consume(wa, b0);
        if (b0 + 2 * RB < nrows) load(wa, b0 + 2 * RB);
        if (b0 + RB < nrows) consume(wb, b0 + RB);
        if (b0 + 3 * RB < nrows) load(wb, b0 + 3 * RB);
    }
    __syncthreads();

    // ---- cross-warp sums and the epilogue --------------------------------------------------------
    if (p.epi == EPI_SWIGLU) {
        for (int t = tid; t < (nrows / 2) * m; t += kRowsThreads) {
            const int pr = t / m, mm = t - pr * m;
            float vg = 0.f, vu = 0.f;
            for (int w = 0; w < kRowsWarps; ++w) {
                vg += red[w][2 * pr][mm];
                vu += red[w][2 * pr + 1][mm];
            }
            p.y[(size_t)mm * p.ldy + row0 / 2 + pr] = silu_f(vg) * vu;
        }
    } else {
        for (int t = tid; t < nrows * m; t += kRowsThreads) {
            const int r = t / m, mm = t - r * m;
            float v = 0.f;
            for (int w = 0; w < kRowsWarps; ++w) v += red[w][r][mm];
            const int row = row0 + r;
            float out;
            if (p.epi == EPI_RESID) {
                const float tt = p.ls ? p.ls[row] * v : v;
                out = p.res[(size_t)mm * p.ldres + row] + tt;
                if (p.tap) p.tap[(size_t)mm * p.ldtap + row] = out;
            } else if (p.epi == EPI_GELU) {
                out = gelu_f(v);
            } else {
                out = v;
            }
            p.y[(size_t)mm * p.ldy + row] = out;
        }
    }
}

size_t gemv_smem_bytes(int m, int K) {
    // upper bound for both weight types: K rounded up to the 256-element bf16 warp step
    const int ldsx = ((K + 255) / 256) * 256;
    return (size_t)m * ldsx * sizeof(float);
}

template <int DT, int MT>
static cudaError_t launch_t(const GemvParams& p, int num_sms, cudaStream_t s, bool pdl) {
    constexpr int KS = 32 * WT<DT>::VEC;
    const int ldsx = ((p.K + KS - 1) / KS) * KS;
    const size_t smem = (size_t)p.m * ldsx * sizeof(float);
    const int ngroups = (p.N + kRows - 1) / kRows;
    const int per_sm = smem <= 96 * 1024 ? 2 : 1;
    int grid = (ngroups + kGemvWarps - 1) / kGemvWarps;
    if (grid > num_sms * per_sm) grid = num_sms * per_sm;
    if (grid < 1) grid = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemv<DT, MT>, p);
}

template <int DT, int MT>
static cudaError_t configure_t() {
    return cudaFuncSetAttribute(k_gemv<DT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kGemvMaxSmem);
}

cudaError_t gemv_configure() {
    cudaError_t e;

    if ((e = configure_t<0, 1>()) != cudaSuccess || (e = configure_t<0, 2>()) != cudaSuccess ||
        (e = configure_t<0, 4>()) != cudaSuccess || (e = configure_t<0, 8>()) != cudaSuccess ||
        (e = configure_t<1, 1>()) != cudaSuccess || (e = configure_t<1, 2>()) != cudaSuccess ||
        (e = configure_t<1, 4>()) != cudaSuccess || (e = configure_t<1, 8>()) != cudaSuccess)
        return e;
    return cudaSuccess;
}

template <int DT, int MT, int NJ>
static cudaError_t launch_rows_t(GemvParams p, int num_sms, cudaStream_t s, bool pdl) {
    p.unit = p.epi == EPI_SWIGLU ? 2 : 1;
    const int units = p.N / p.unit;
    int grid = 2 * num_sms;
    // at most kRowsMaxRows rows per CTA
    const int need = (p.N + kRowsMaxRows - 2) / (kRowsMaxRows - 1);
    if (grid < need) grid = need;
    if (grid > units) grid = units;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kRowsThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemv_rows<DT, MT, NJ>, p);
}

// granules per lane of the split-K kernel (0: shape not served by it)
static int rows_nj(const GemvParams& p, int dtype) {
    const int vec = dtype == 1 ? 8 : 4;
    const int per_pass = kRowsThreads * vec;  // elements one pass of the CTA covers
    const int nj = (p.K + per_pass - 1) / per_pass;
    return (p.m <= 2 && nj <= 4 && nj != 0) ? (nj == 3 ? 3 : nj == 4 ? 4 : nj) : 0;
}

template <int DT, int MT>
static cudaError_t launch_rows_nj(const GemvParams& p, int nj, int num_sms, cudaStream_t s, bool pdl) {
    switch (nj) {
        case 1: return launch_rows_t<DT, MT, 1>(p, num_sms, s, pdl);
        case 2: return launch_rows_t<DT, MT, 2>(p, num_sms, s, pdl);
        case 3: return launch_rows_t<DT, MT, 3>(p, num_sms, s, pdl);
        default: return launch_rows_t<DT, MT, 4>(p, num_sms, s, pdl);
    }
}

cudaError_t launch_gemv(const GemvParams& p, int dtype, int num_sms, cudaStream_t s, bool pdl) {
    const int nj = rows_nj(p, dtype);
    if (nj) {
        if (dtype == 1) return p.m <= 1 ? launch_rows_nj<1, 1>(p, nj, num_sms, s, pdl)
                                        : launch_rows_nj<1, 2>(p, nj, num_sms, s, pdl);
        return p.m <= 1 ? launch_rows_nj<0, 1>(p, nj, num_sms, s, pdl)
                        : launch_rows_nj<0, 2>(p, nj, num_sms, s, pdl);
    }
    const int mt = p.m <= 1 ? 1 : p.m <= 2 ? 2 : p.m <= 4 ? 4 : 8;
    if (dtype == 1) {
        switch (mt) {
            case 1: return launch_t<1, 1>(p, num_sms, s, pdl);
            case 2: return launch_t<1, 2>(p, num_sms, s, pdl);
            case 4: return launch_t<1, 4>(p, num_sms, s, pdl);
            default: return launch_t<1, 8>(p, num_sms, s, pdl);
        }
    }
    switch (mt) {
        case 1: return launch_t<0, 1>(p, num_sms, s, pdl);
        case 2: return launch_t<0, 2>(p, num_sms, s, pdl);
        case 4: return launch_t<0, 4>(p, num_sms, s, pdl);
        default: return launch_t<0, 8>(p, num_sms, s, pdl);
    }
}

}  // namespace dec
