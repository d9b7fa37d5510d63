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
#include "gemv_rows.cuh"
#include "kernels.h"

namespace dec {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kRows = 2;     // rows per warp task (a gate/up pair for SwiGLU)
constexpr int kUnroll = 4;   // 16-byte steps per row in flight

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

template <int DT, int MT>
__global__ void __launch_bounds__(kGemvThreads, 2) k_gemv(const GemvParams p) {
    extern __shared__ __align__(16) float sx[];  // [m][ldsx]
    __shared__ float red[kGemvWarps][MT];
    __shared__ float stat[2][MT];

    constexpr int VEC = WType<DT>::VEC;
    constexpr int ES = WType<DT>::ES;
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
// Split-K row-streaming GEMV for m <= 8 (the decode step's common case), on its own: the first
// two weight batches are issued before griddepcontrol.wait (see gemv_rows.cuh).  Two CTAs per
// SM for m <= 2; one for wider rows, whose x slice and partial sums fill the register file.
// =============================================================================================
template <int DT, int MT, int NJ>
__global__ void __launch_bounds__(kRowsThreads, MT <= 2 ? 2 : 1) k_gemv_rows(const GemvParams p) {
    __shared__ float sh[rows_smem_floats<MT>()];
    using R = RowsGemv<DT, MT, NJ, 8>;
    uint4 wa[8], wb[8];
    const uint64_t pol = l2_evict_first();
    R::issue(p, blockIdx.x, gridDim.x, wa, wb, pol);
    pdl_trigger();
    pdl_wait();
    R::run(p, blockIdx.x, gridDim.x, wa, wb, sh, pol);
}

// 5..8 rows of a matrix wider than one granule a lane (the down GEMV, K = 6144): x of 8 rows
// would take up to 192 registers a thread, so each CTA makes two passes over its rows, x rows
// 0..3 and then 4..m-1.  The first pass reads the weights at normal L2 priority and the second,
// which follows at once on the same CTA (a few hundred KB per CTA), finds them in L2: HBM sees
// each weight once.  Rows of different passes write disjoint rows of y.
template <int DT, int NJ>
__global__ void __launch_bounds__(kRowsThreads, 1) k_gemv_rows2(const GemvParams p) {
    __shared__ float sh[rows_smem_floats<4>()];
    using R = RowsGemv<DT, 4, NJ, 8>;
    uint4 wa[8], wb[8];
    GemvParams q = p;
    q.m = 4;
    const uint64_t keep = l2_evict_normal();
    R::issue(q, blockIdx.x, gridDim.x, wa, wb, keep);
    pdl_trigger();
    pdl_wait();
    R::run(q, blockIdx.x, gridDim.x, wa, wb, sh, keep);
    __syncthreads();  // the cross-warp scratch is reused
    q.m = p.m - 4;
    q.x = p.x + (size_t)4 * p.ldx;
    q.y = p.y + (size_t)4 * p.ldy;
    if (p.res) q.res = p.res + (size_t)4 * p.ldres;
    if (p.tap) q.tap = p.tap + (size_t)4 * p.ldtap;
    const uint64_t pol = l2_evict_first();
    R::issue(q, blockIdx.x, gridDim.x, wa, wb, pol);
    R::run(q, blockIdx.x, gridDim.x, wa, wb, sh, pol);
}

size_t gemv_smem_bytes(int m, int K) {
    // upper bound for both weight types: K rounded up to the 256-element bf16 warp step
    const int ldsx = ((K + 255) / 256) * 256;
    return (size_t)m * ldsx * sizeof(float);
}

template <int DT, int MT>
static cudaError_t launch_t(const GemvParams& p, int num_sms, cudaStream_t s, bool pdl) {
    constexpr int KS = 32 * WType<DT>::VEC;
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
static cudaError_t launch_rows_t(GemvParams p, int num_sms, cudaStream_t s, bool pdl,
                                 bool two_pass = false) {
    p.unit = p.epi == EPI_SWIGLU ? 2 : 1;
    const int units = p.N / p.unit;
    int grid = (p.per_sm > 0 ? p.per_sm : (MT <= 2 ? 2 : 1)) * num_sms;
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
    if constexpr (MT == 4 && NJ > 1)
        if (two_pass) return cudaLaunchKernelEx(&cfg, k_gemv_rows2<DT, NJ>, p);
    return cudaLaunchKernelEx(&cfg, k_gemv_rows<DT, MT, NJ>, p);
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
    const int nj = rows_gemv_nj(p.K, p.m, dtype);
    // bias, SiLU and the modulate prologue are served by the split-K kernel only
    if (!nj && (p.bias || p.act || p.pro == PRO_LN_MOD)) return cudaErrorInvalidValue;
    if (dtype == 1 && p.m > 2 && gemv_tc_ok(p, num_sms))  // 3..8 rows on the tensor cores
        return launch_gemv_tc(p, num_sms, s, pdl);
    if (nj == 1 && p.m > 2) {  // 3..8 rows, one granule a lane
        if (dtype == 1) return p.m <= 4 ? launch_rows_t<1, 4, 1>(p, num_sms, s, pdl)
                                        : launch_rows_t<1, 8, 1>(p, num_sms, s, pdl);
        return p.m <= 4 ? launch_rows_t<0, 4, 1>(p, num_sms, s, pdl)
                        : launch_rows_t<0, 8, 1>(p, num_sms, s, pdl);
    }
    if (nj && p.m > 2) {  // 3..8 rows, 2..3 granules a lane: x of 4 rows at a time
        const bool two = p.m > 4;
        if (dtype == 1) return nj == 2 ? launch_rows_t<1, 4, 2>(p, num_sms, s, pdl, two)
                                       : launch_rows_t<1, 4, 3>(p, num_sms, s, pdl, two);
        return nj == 2 ? launch_rows_t<0, 4, 2>(p, num_sms, s, pdl, two)
                       : launch_rows_t<0, 4, 3>(p, num_sms, s, pdl, two);
    }
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
