// gemv_tc.cu -- tensor-core GEMV for 3..8 rows of x against bf16 weights: tcgen05.mma with the
// accumulators in tensor memory, weight tiles by TMA (sm_103a).
//
// y[r][n] = sum_k W[n][k] x[r][k], r < m <= 8, W row-major [N][K] bf16 (Qwen3-TTS talker on
// wgpu, MATVEC_SRC: each weight is read once for all rows).  With eight rows the FMA form is bound
// by instruction issue; here the weights stream through the tensor cores.
//
// One MMA (kind::f16, M = 128, N = 32, K = 16, both operands K-major in shared memory with the
// 128-byte swizzle, f32 accumulators in TMEM):
//   A = a tile of 128 weight rows, 64 k per TMA box (16 KB), 4 MMAs per box;
//   B = x split into three bf16 terms, x = hi + mid + lo: B row n = term * 8 + stream (rows of
//       streams >= m and rows 24..31 are zero).  bf16 x bf16 products are exact and the three
//       terms hold x's 24-bit significand, so the result keeps f32 accuracy; D column n holds the
//       term's partial dot product and a row's sum for stream s is D[s] + D[8 + s] + D[16 + s].
//
// Work split (stream-K): units are (tile of 128 rows, chunk of 64 k), tile-major; CTA b of P takes
// units [b U / P, (b + 1) U / P), so every CTA streams the same bytes to within one 16 KB box.
// The matrix's TMA descriptor is a __grid_constant__ kernel parameter.  Roles: thread 0 issues the
// TMA boxes into a ring of stages (the first ones before
// griddepcontrol.wait: weights never depend on the previous kernel); thread 32 issues the MMAs,
// one TMEM accumulator of 32 columns per tile the CTA touches, and frees each stage with
// tcgen05.commit; all four warps stage the x terms (norm prologue included) and read the
// accumulators back (warp w: TMEM lanes 32 w .. 32 w + 31 = the tile's rows).  A tile whose chunks
// fall in several CTAs is finished by the last to arrive (an atomic ticket, no waiting): each
// writes its partial sums to global scratch and the last adds them in CTA order, so the result
// does not depend on which CTA came last.  Every wait is bounded; after a wait gives up the CTA
// stops issuing, waits (bounded) for what it issued, frees its TMEM and records CHECK_WAIT_LIMIT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "gemv_rows.cuh"
#include "kernels.h"

namespace dec {

constexpr int kTcThreads = 128;
constexpr int kTcRows = 128;            // weight rows per tile (MMA M, TMEM lanes)
constexpr int kTcChunk = 64;            // k per TMA box (128 bytes of bf16: one swizzle row)
constexpr int kTcBox = kTcRows * kTcChunk * 2;  // 16 KB
constexpr int kTcBBytes = 32 * 128;     // x terms of one chunk: 32 rows x 128 B
constexpr int kTcMaxSlots = 16;         // tiles one CTA may accumulate (TMEM: 32 columns each)
// (each tile takes 1, 2 or 4 accumulators: the MMAs of one accumulator run one after another)
constexpr int kTcMaxStages = 12;
constexpr int kTcMaxKSlots = 64;        // x-term chunk slots of one CTA
constexpr int kTcMinSmem = 116 * 1024;  // at least this much: one CTA per SM
constexpr int kTcMaxSmem = 220 * 1024;

// instruction descriptor: D f32, A and B bf16, both K-major, N = 32, M = 128
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((32u >> 3) << 17) |
                              ((uint32_t)(kTcRows >> 4) << 24);

// byte offset of element (r, k) (k < 64) in a K-major tile of 128-byte rows with the 128-byte
// swizzle: 16-byte chunk c of row r sits at chunk c ^ (r mod 8)
__device__ __forceinline__ uint32_t sw128(int r, int k) {
    return (uint32_t)r * 128u + ((uint32_t)((k >> 3) ^ (r & 7)) << 4) + (uint32_t)(k & 7) * 2u;
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(acc));
}

__device__ __forceinline__ unsigned tc_atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tma_box(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                        uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

// 32 consecutive f32 columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// two f32 values -> (hi, mid, lo) bf16 pairs with v = hi + mid + lo (each pair: low half first)
__device__ __forceinline__ void split3(float v0, float v1, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float r0 = v0 - __low2float(h), r1 = v1 - __high2float(h);
    const __nv_bfloat162 md = __floats2bfloat162_rn(r0, r1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(r0 - __low2float(md), r1 - __high2float(md));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    mid = *reinterpret_cast<const uint32_t*>(&md);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The split shared by host and device.  Units are (tile of 128 rows, chunk of 64 k).  Tiles are
// grouped in bands of G; units run band by band, chunk-major inside a band (chunk c of every tile
// of the band, then chunk c + 1).  CTA b of P takes units [b U / P, (b + 1) U / P): a CTA then
// needs the x terms of few chunks (about its units / G) and accumulates at most a few tiles.
struct TcSplit {
    // tiles, chunk groups per tile (a unit's k: CB chunks of 64), units, tiles per band
    int NT, NC, U, G;
    __host__ __device__ TcSplit(int N, int K, int G_, int CB)
        : NT((N + kTcRows - 1) / kTcRows), NC(K / (kTcChunk * CB)),
          U(((N + kTcRows - 1) / kTcRows) * (K / (kTcChunk * CB))), G(G_) {}
    // (32-bit: the plan keeps U P below 2^31)
    __host__ __device__ int u0(int b, int P) const { return (int)((unsigned)b * (unsigned)U / (unsigned)P); }
    __host__ __device__ int band_of(int u) const { return u / (G * NC); }
    __host__ __device__ int band_tiles(int band) const { return NT - band * G < G ? NT - band * G : G; }
    __host__ __device__ void unit(int u, int& tile, int& chunk) const {
        const int band = band_of(u), gb = band_tiles(band), w = u - band * G * NC;
        chunk = w / gb;
        tile = band * G + (w - chunk * gb);
    }
    // the unit after (tile, chunk): the next tile of the band, else chunk + 1, else the next band
    __host__ __device__ void next(int& tile, int& chunk) const {
        const int band = tile / G, gb = band_tiles(band);
        if (tile + 1 < band * G + gb) {
            ++tile;
        } else if (chunk + 1 < NC) {
            tile = band * G;
            ++chunk;
        } else {
            tile = (band + 1) * G;
            chunk = 0;
        }
    }
    // unit of (tile, chunk)
    __host__ __device__ int unit_of(int tile, int chunk) const {
        const int band = tile / G;
        return band * G * NC + chunk * band_tiles(band) + (tile - band * G);
    }
    // the CTA whose range holds unit u: the largest b with b U / P <= u
    __host__ __device__ int owner(int u, int P) const {
        return (int)(((unsigned)u * (unsigned)P + (unsigned)P - 1u) / (unsigned)U);
    }
    // CTA b: its first tile slot (accumulator j holds tile tile_base + j), the slots it may touch,
    // the first chunk of its x terms and how many consecutive chunks (mod NC) they span
    __host__ __device__ void cta(int b, int P, int& tile_base, int& slots, int& c_first, int& nchunks) const {
        const int a = u0(b, P), e = u0(b + 1, P);
        const int ba = band_of(a), be = band_of(e - 1);
        tile_base = ba * G;
        const int t_end = (be + 1) * G < NT ? (be + 1) * G : NT;
        slots = t_end - tile_base;
        int ta, tl, cl;
        unit(a, ta, c_first);
        unit(e - 1, tl, cl);
        if (e - a >= NC * band_tiles(ba) || be > ba + 1) {
            nchunks = NC;
        } else if (be == ba) {
            nchunks = cl - c_first + 1;
        } else {  // into the next band: chunks c_first .. NC - 1, then 0 .. cl
            nchunks = NC - c_first + cl + 1;
            if (nchunks > NC) nchunks = NC;
        }
    }
};

// the launch plan (host)
struct TcPlan {
    int grid, G, CB, stages, bslots, slots, acc, tcols, contrib;
    size_t smem;
    double cost;
};

__host__ __device__ inline size_t tc_smem_bytes(int stages, int bslots) {
    return 1024 + (size_t)stages * kTcBox + (size_t)bslots * kTcBBytes;
}

// The epilogue in two parts.  tc_linear: the part that is linear in the dot product, applied to a
// row's sum or to one CTA's partial of it: y <- ls (y + bias) + res, where LayerScale ls applies to
// the residual epilogue only, and bias and the residual are added once, by the caller that holds
// the tile's first unit (first).  tc_out: the rest, on the full sum: the store (and tap) of the
// residual epilogue, SiLU, GELU, or SwiGLU over rows 2j, 2j + 1 (adjacent lanes).  Every lane of
// the warp calls tc_out (SwiGLU pairs rows across lanes).
__device__ __forceinline__ void tc_linear(const GemvParams& p, int row, float (&y)[8], bool first) {
    if (row >= p.N) return;
    const float ls = (p.epi == EPI_RESID && p.ls) ? p.ls[row] : 1.0f;
    const float bias = (first && p.bias) ? p.bias[row] : 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        if (s >= p.m) break;
        y[s] = ls * (y[s] + bias);
        if (first && p.epi == EPI_RESID) y[s] += __ldcg(p.res + (size_t)s * p.ldres + row);
    }
}

__device__ __forceinline__ void tc_out(const GemvParams& p, int row, const float (&y)[8]) {
    const int m = p.m;
    if (p.epi == EPI_SWIGLU) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const float up = __shfl_down_sync(0xffffffffu, y[s], 1);
            if (s < m && !(row & 1) && row + 1 < p.N) p.y[(size_t)s * p.ldy + row / 2] = silu_f(y[s]) * up;
        }
        return;
    }
    if (row >= p.N) return;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        if (s >= m) break;
        float out = y[s];
        if (p.epi == EPI_RESID) {
            if (p.tap) p.tap[(size_t)s * p.ldtap + row] = out;
        } else if (p.epi == EPI_GELU) {
            out = gelu_f(out);
        } else if (p.act == 1) {
            out = silu_f(out);
        }
        p.y[(size_t)s * p.ldy + row] = out;
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) k_gemv_tc(const GemvParams p,
                                                             const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    __shared__ __align__(8) uint64_t full[kTcMaxStages], empty[kTcMaxStages], done_bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_issued, s_consumed, s_done;
    __shared__ float s_stat[2][8];
    __shared__ int s_cnt[kTcMaxSlots], s_last[kTcMaxSlots];
    __shared__ int s_kslot[kTcMaxKSlots];  // k offset of every x-term slot

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int CB = p.tc_cb;  // 64-k chunks per unit (one TMA box each)
    const TcSplit sp(p.N, p.K, p.tc_band, CB);
    const int P = gridDim.x, b = blockIdx.x;
    const int u0 = sp.u0(b, P), u1 = sp.u0(b + 1, P), nu = u1 - u0;
    const int S = p.tc_stages, NC = sp.NC, m = p.m, K = p.K, A = p.tc_acc;
    const uint32_t stage_bytes = (uint32_t)CB * kTcBox;
    int tile_base, nslots, g_first, ngroups;
    // x-term slot j * CB + cc: chunk cc of group (g_first + j) mod NC
    sp.cta(b, P, tile_base, nslots, g_first, ngroups);
    // RMSNorm: the MMAs take x * w and the epilogue applies 1 / rms, so the statistics are not
    // on the path to the first MMA; LayerNorm needs its mean first
    const bool defer = p.pro == PRO_RMS;
    const uint32_t raw = smem_u32(tc_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* const bsm = tc_raw + (base - raw) + (size_t)S * stage_bytes;
    const uint32_t bsm_a = base + (uint32_t)S * stage_bytes;
    const uint64_t pol = l2_evict_first();

    auto issue = [&](int i, int st) {  // the TMA boxes of unit u0 + i into stage st
        int tile, grp;
        sp.unit(u0 + i, tile, grp);
        const uint32_t bar = smem_u32(&full[st]);
        mbar_arrive_expect_tx(bar, stage_bytes);
        for (int cc = 0; cc < CB; ++cc)
            tma_box(base + (uint32_t)st * stage_bytes + (uint32_t)cc * kTcBox, &tmap,
                    (grp * CB + cc) * kTcChunk, tile * kTcRows, bar, pol);
    };
    if (tid == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(smem_u32(&full[st]), 1);
            mbar_init(smem_u32(&empty[st]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        s_abort = 0;
        s_consumed = 0;
        if (nu > 0) issue(0, 0);  // weights never depend on the previous kernel
    }
    if (tid < kTcMaxSlots) s_cnt[tid] = 0;
    __syncthreads();
    pdl_trigger();
    pdl_wait();

    // ---- warp 0: the accumulators (32 columns each), then lane 0 streams the boxes ----------
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(p.tc_cols)
                     : "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        named_bar_arrive(1, kTcThreads);  // TMEM is allocated
        if (lane == 0) {
            int i = 1, st = 1 % S;
            uint32_t ph = 0u;  // phase of the stage's release to wait for (units S, S + 1, ...)
            for (; i < nu; ++i) {
                if (s_abort) break;
                if (i >= S && !mbar_wait_bounded(smem_u32(&empty[st]), ph)) {
                    s_abort = 1;
                    break;
                }
                issue(i, st);
                if (++st == S) {
                    st = 0;
                    if (i >= S) ph ^= 1u;
                }
            }
            s_issued = i;
        }
    } else {
        // ---- warps 1..3: norm statistics (LayerNorm: before the terms), the x terms ----------
        const int t96 = tid - 32;
        auto stats = [&](int s0, int step) {  // one warp per stream, lanes over k
            for (int s = s0; s < m; s += step) {
                const float* xr = p.x + (size_t)s * p.ldx;
                float a = 0.f;
#pragma unroll 8
                for (int k = lane * 4; k < K; k += 128) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(xr + k));
                    a += (p.pro == PRO_RMS) ? v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w
                                            : v.x + v.y + v.z + v.w;
                }
                a = warp_sum(a) / (float)K;
                float mean = 0.f, inv;
                if (p.pro == PRO_RMS) {
                    inv = 1.0f / sqrtf(a + p.eps);
                } else {
                    mean = a;
                    float q = 0.f;
#pragma unroll 8
                    for (int k = lane * 4; k < K; k += 128) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(xr + k));
                        q += (v.x - mean) * (v.x - mean) + (v.y - mean) * (v.y - mean) +
                             (v.z - mean) * (v.z - mean) + (v.w - mean) * (v.w - mean);
                    }
                    inv = 1.0f / sqrtf(warp_sum(q) / (float)K + p.eps);
                }
                if (lane == 0) {
                    s_stat[0][s] = mean;
                    s_stat[1][s] = inv;
                }
            }
        };
        for (int jj = t96; jj < ngroups * CB; jj += kTcThreads - 32)
            s_kslot[jj] = (((g_first + jj / CB) % NC) * CB + jj % CB) * kTcChunk;
        if (p.pro != PRO_NONE && !defer) stats(warp - 1, 3);
        named_bar_sync(2, kTcThreads - 32);  // the slot offsets (and LayerNorm statistics) are set
        // task (x-term slot jj, stream st, k quad q), 128 per slot, over 96 threads
        const int nterm = ngroups * CB;
        for (int t0 = t96; t0 < nterm * 128; t0 += 8 * 96) {
            float4 xv[8], wv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {  // the batch's loads first
                const int t = t0 + e * 96, jj = t >> 7, st = (t >> 4) & 7, q = t & 15;
                xv[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                wv[e] = make_float4(1.f, 1.f, 1.f, 1.f);
                if (jj < nterm && st < m) {
                    const int k = s_kslot[jj] + 4 * q;
                    xv[e] = __ldcg(reinterpret_cast<const float4*>(p.x + (size_t)st * p.ldx + k));
                    if (p.pro != PRO_NONE && p.nw) wv[e] = *reinterpret_cast<const float4*>(p.nw + k);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = t0 + e * 96, jj = t >> 7, st = (t >> 4) & 7, q = t & 15;
                if (jj >= nterm) break;
                const int k = s_kslot[jj] + 4 * q;
                float v[4] = {xv[e].x, xv[e].y, xv[e].z, xv[e].w};
                if (p.pro != PRO_NONE && st < m) {
                    const float w[4] = {wv[e].x, wv[e].y, wv[e].z, wv[e].w};
                    float mean = 0.f, inv = 1.f, bb[4] = {0.f, 0.f, 0.f, 0.f};
                    if (!defer) {
                        mean = s_stat[0][st];
                        inv = s_stat[1][st];
                        if (p.nb) {
                            const float4 t4 = *reinterpret_cast<const float4*>(p.nb + k);
                            bb[0] = t4.x; bb[1] = t4.y; bb[2] = t4.z; bb[3] = t4.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = (v[i] - mean) * inv * w[i] + bb[i];
                    if (p.pro == PRO_LN_MOD) {  // modulate: n (1 + scale) + shift
                        const float4 sh = __ldcg(reinterpret_cast<const float4*>(p.mod + k));
                        const float4 sc = __ldcg(reinterpret_cast<const float4*>(p.mod + K + k));
                        v[0] = v[0] * (1.0f + sc.x) + sh.x;
                        v[1] = v[1] * (1.0f + sc.y) + sh.y;
                        v[2] = v[2] * (1.0f + sc.z) + sh.z;
                        v[3] = v[3] * (1.0f + sc.w) + sh.w;
                    }
                }
                uint32_t h0, m0, l0, h1, m1, l1;
                split3(v[0], v[1], h0, m0, l0);
                split3(v[2], v[3], h1, m1, l1);
                unsigned char* bs = bsm + (size_t)jj * kTcBBytes;
                *reinterpret_cast<uint2*>(bs + sw128(st, 4 * q)) = make_uint2(h0, h1);
                *reinterpret_cast<uint2*>(bs + sw128(8 + st, 4 * q)) = make_uint2(m0, m1);
                *reinterpret_cast<uint2*>(bs + sw128(16 + st, 4 * q)) = make_uint2(l0, l1);
                *reinterpret_cast<uint2*>(bs + sw128(24 + st, 4 * q)) = make_uint2(0u, 0u);
            }
        }
        fence_proxy_async_smem();  // the MMAs read the terms through the async proxy
        named_bar_sync(1, kTcThreads);  // the terms are written, TMEM is allocated
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (tid == 32) {
            // ---- the MMA issuer (no tcgen05 fence after the stage waits: the mbarrier orders
            // the TMA's writes before the MMAs' reads, and the fence would wait for the MMAs
            // still in flight) -----------------------------------------------------------------
            const uint32_t tmem = s_tmem;
            unsigned used = 0u;  // tile slots whose accumulators have been started
            int i = 0, st = 0, tile, grp;
            uint32_t ph = 0u;
            sp.unit(u0, tile, grp);
            for (; i < nu; ++i) {
                if (s_abort) break;
                if (!mbar_wait_bounded(smem_u32(&full[st]), ph)) {
                    s_abort = 1;
                    break;
                }
                const int slot = tile - tile_base;
                int bg = grp - g_first;
                if (bg < 0) bg += NC;
                const uint64_t da = tc_sdesc(base + (uint32_t)st * stage_bytes);
                const uint64_t db = tc_sdesc(bsm_a + (uint32_t)(bg * CB) * kTcBBytes);
                const uint32_t d = tmem + (uint32_t)(slot * A) * 32u;
                const bool first = !((used >> slot) & 1u);
                used |= 1u << slot;
                // k-step kk (chunk kk / 4, 16 k each) accumulates into accumulator kk mod A;
                // descriptors advance in 16-byte units: 32 bytes per k-step, a box per chunk
                for (int cc = 0; cc < CB; ++cc)
#pragma unroll
                    for (int ks = 0; ks < kTcChunk / 16; ++ks) {
                        const int kk = cc * 4 + ks;
                        tc_mma(d + (uint32_t)(kk & (A - 1)) * 32u,
                               da + (uint64_t)(cc * (kTcBox >> 4) + ks * 2),
                               db + (uint64_t)(cc * (kTcBBytes >> 4) + ks * 2), (first && kk < A) ? 0u : 1u);
                    }
                tc_commit(smem_u32(&empty[st]));  // the stage is free once these MMAs have read it
                ++s_cnt[slot];
                sp.next(tile, grp);
                if (++st == S) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            s_consumed = i;
            tc_commit(smem_u32(&done_bar));  // every MMA issued above has completed
        } else if (defer && warp >= 2) {
            stats(warp - 2, 2);
        }
    }
    // one thread polls for the MMAs' completion; the others wait at the block barrier
    __syncwarp();
    if (tid == 64) s_done = mbar_wait_bounded(smem_u32(&done_bar), 0u) ? 1 : 0;
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const bool ok = s_done && !s_abort;
    const uint32_t tmem = s_tmem;

    // ---- accumulators -> outputs (thread: tile row 32 warp + lane) ---------------------------
    if (ok) {
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const int r = warp * 32 + lane;
        float scale[8];
#pragma unroll
        for (int st = 0; st < 8; ++st) scale[st] = (defer && st < m) ? s_stat[1][st] : 1.0f;
        bool split = false;
        for (int j = 0; j < nslots; ++j) {
            const int cnt = s_cnt[j];
            if (!cnt) continue;
            float v[32], y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int ac = 0; ac < A; ++ac) {
                tmem_ld32(lane_base + (uint32_t)(j * A + ac) * 32u, v);
#pragma unroll
                for (int st = 0; st < 8; ++st) y[st] += v[st] + v[8 + st] + v[16 + st];
            }
#pragma unroll
            for (int st = 0; st < 8; ++st) y[st] *= scale[st];
            const int tile = tile_base + j, row = tile * kTcRows + r;
            const int u_first = sp.unit_of(tile, 0), holder = sp.owner(u_first, P);
            tc_linear(p, row, y, holder == b);  // the holder of the tile's first unit adds bias, residual
            if (cnt == NC) {
                tc_out(p, row, y);
            } else {  // a partial tile: block (tile, this CTA's ordinal among its holders)
                const int k = b - holder;
                float* dst = p.mpart + (((size_t)tile * p.tc_contrib + k) * kTcRows + r) * 8;
                *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(y[4], y[5], y[6], y[7]);
                split = true;
            }
        }
        if (__syncthreads_or(split)) {
            // The tickets: a tile's ticket counts its units; the CTA whose units complete it
            // finishes it.  The barrier above and the release of the atomic publish this CTA's
            // partials; the acquire and the barrier below order the finisher's reads after the
            // other CTAs' partials.
            if (tid < nslots) {
                const int cnt = s_cnt[tid];
                s_last[tid] = (cnt > 0 && cnt < NC) &&
                              tc_atom_add_acq_rel(&p.mtick[tile_base + tid], (unsigned)cnt) + (unsigned)cnt ==
                                  (unsigned)NC;
            }
            __syncthreads();
            // the finished tiles, four at a time; tile t's holders are CTAs owner(first unit) ..
            // owner(last unit), all of them (the plan keeps a band within every CTA's reach), and
            // their partials are blocks t * contrib + 0, 1, ...: loaded together, added in order
            const int r = warp * 32 + lane;
            int fin[4], nfin = 0;
            auto finish = [&]() {
                float yt[4][8];
                int blk[4], nc[4], most = 0;
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) yt[g4][e] = 0.f;
                    nc[g4] = 0;
                    blk[g4] = 0;
                    if (g4 < nfin) {
                        const int tile = fin[g4], band = tile / sp.G, gb = sp.band_tiles(band);
                        const int ub = band * sp.G * NC + (tile - band * sp.G);
                        nc[g4] = sp.owner(ub + (NC - 1) * gb, P) - sp.owner(ub, P) + 1;
                        blk[g4] = tile * p.tc_contrib;
                        most = nc[g4] > most ? nc[g4] : most;
                    }
                }
                for (int k0 = 0; k0 < most; k0 += 2) {  // two holders of four tiles per load round
                    float4 a4[2][4], c4[2][4];
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int g4 = 0; g4 < 4; ++g4)
                            if (k0 + h < nc[g4]) {
                                const float* src = p.mpart + ((size_t)(blk[g4] + k0 + h) * kTcRows + r) * 8;
                                a4[h][g4] = __ldcg(reinterpret_cast<const float4*>(src));
                                c4[h][g4] = __ldcg(reinterpret_cast<const float4*>(src + 4));
                            }
#pragma unroll
                    for (int h = 0; h < 2; ++h)  // holder k0, then k0 + 1: the same order as one by one
#pragma unroll
                        for (int g4 = 0; g4 < 4; ++g4)
                            if (k0 + h < nc[g4]) {
                                float* y = yt[g4];
                                y[0] += a4[h][g4].x; y[1] += a4[h][g4].y; y[2] += a4[h][g4].z; y[3] += a4[h][g4].w;
                                y[4] += c4[h][g4].x; y[5] += c4[h][g4].y; y[6] += c4[h][g4].z; y[7] += c4[h][g4].w;
                            }
                }
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4)
                    if (g4 < nfin) {
                        tc_out(p, fin[g4] * kTcRows + r, yt[g4]);
                        if (tid == 0) p.mtick[fin[g4]] = 0u;  // every unit has arrived
                    }
                nfin = 0;
            };
            for (int j = 0; j < nslots; ++j) {
                if (!s_last[j]) continue;
                fin[nfin++] = tile_base + j;
                if (nfin == 4) finish();
            }
            if (nfin) finish();
        }
    } else if (tid == 0) {
        // a wait gave up: record it, and let no box still be landing when the CTA exits
        flag_check(p.status, CHECK_WAIT_LIMIT);
        for (int i = s_consumed; i < s_issued; ++i)
            mbar_wait_bounded(smem_u32(&full[i % S]), (uint32_t)(i / S) & 1u);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tc_cols)
                     : "memory");
}

// ---------------------------------------------------------------------------------------------
// Host: the launch plan (grid, stages, x-term slots, TMEM columns), the tensor maps, the launch.
// ---------------------------------------------------------------------------------------------
static bool tc_plan_one(const GemvParams& p, int num_sms, int G, int CB, TcPlan& pl) {
    const TcSplit sp(p.N, p.K, G, CB);
    const int P = sp.U < num_sms ? sp.U : num_sms;
    if ((long long)sp.U * (P + 1) >= (1ll << 31)) return false;  // 32-bit unit arithmetic
    int max_groups = 0, max_slots = 0, max_units = 0;
    for (int b = 0; b < P; ++b) {
        int tile_base, slots, g_first, ngroups;
        sp.cta(b, P, tile_base, slots, g_first, ngroups);
        max_groups = std::max(max_groups, ngroups);
        max_slots = std::max(max_slots, slots);
        max_units = std::max(max_units, sp.u0(b + 1, P) - sp.u0(b, P));
    }
    bool split = false;  // a tile is split unless one CTA holds all its units
    int max_contrib = 1;
    for (int t = 0; t < sp.NT; ++t) {
        const int c = sp.owner(sp.unit_of(t, sp.NC - 1), P) - sp.owner(sp.unit_of(t, 0), P) + 1;
        max_contrib = std::max(max_contrib, c);
        if (c > 1) split = true;
    }
    // every CTA between a tile's first and last holder holds one of its units: a CTA's range
    // reaches across a band of G tiles
    int min_units = 1 << 30;
    for (int b = 0; b < P; ++b) min_units = std::min(min_units, sp.u0(b + 1, P) - sp.u0(b, P));
    if (split && G > min_units) return false;
    if (max_slots > kTcMaxSlots || max_groups * CB > kTcMaxKSlots) return false;
    if (split && (!p.mpart || !p.mtick || (size_t)sp.NT * max_contrib * kTcRows * 8 > p.mpart_floats ||
                  sp.NT > p.mtick_n))
        return false;
    const size_t bbytes = (size_t)max_groups * CB * kTcBBytes, sbytes = (size_t)CB * kTcBox;
    if (bbytes + 1024 + 2 * sbytes > (size_t)kTcMaxSmem) return false;
    pl.grid = P;
    pl.G = G;
    pl.CB = CB;
    pl.bslots = max_groups * CB;
    pl.stages = std::min(kTcMaxStages, (int)((kTcMaxSmem - 1024 - bbytes) / sbytes));
    pl.slots = max_slots;
    pl.contrib = max_contrib;
    // independent accumulators per tile (TMEM: 512 columns of 32 per accumulator)
    pl.acc = max_slots <= 4 ? 4 : max_slots <= 8 ? 2 : 1;
    pl.tcols = 32;
    while (pl.tcols < 32 * pl.acc * max_slots) pl.tcols <<= 1;
    pl.smem = std::max((size_t)kTcMinSmem, tc_smem_bytes(pl.stages * CB, pl.bslots));
    // estimated CTA time (us): per unit, the larger of its bytes at one SM's share of HBM and
    // the MMA thread's work; a split tile adds the fixup round trips
    const double per_unit = std::max(CB * 0.36, 0.35 + 0.1 * CB);
    pl.cost = max_units * per_unit + (split ? 1.5 : 0.0);
    return true;
}

// Among bands of 1, 2, 4, 8 tiles and units of 1, 2, 4 chunks: the lowest estimated time, then
// the most accumulators and stages.
static bool tc_plan(const GemvParams& p, int num_sms, TcPlan& pl) {
    if (!p.tmap || p.m < 3 || p.m > 8 || p.K < kTcChunk || p.K % kTcChunk || p.N < kTcRows) return false;
    auto a16 = [](const void* q) { return ((uintptr_t)q & 15u) == 0; };
    if (!a16(p.x) || (p.ldx & 3)) return false;  // float4 loads of x, norm weights, modulation
    if (p.pro != PRO_NONE && p.nw && !a16(p.nw)) return false;
    if (p.pro != PRO_NONE && p.pro != PRO_RMS && p.nb && !a16(p.nb)) return false;
    if (p.pro == PRO_LN_MOD && (!a16(p.mod) || (p.K & 3))) return false;
    if (p.epi == EPI_SWIGLU && (p.N & 1)) return false;
    // the search below takes tens of microseconds of host time: launches outside a CUDA graph
    // (prefill blocks) reuse the plan of a shape seen before
    struct Key {
        int N, K, sms;
        size_t mpart_floats;
        int mtick_n;
        bool scratch;
    };
    Key key;
    memset(&key, 0, sizeof(key));  // padding included: keys compare bytewise
    key.N = p.N;
    key.K = p.K;
    key.sms = num_sms;
    key.mpart_floats = p.mpart_floats;
    key.mtick_n = p.mtick_n;
    key.scratch = p.mpart && p.mtick;
    static std::mutex mu;
    static std::vector<std::pair<Key, TcPlan>> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (auto& e : cache)
            if (!memcmp(&e.first, &key, sizeof(Key))) {
                pl = e.second;
                return pl.grid > 0;
            }
    }
    bool found = false;
    for (int CB = 1; CB <= 4; CB *= 2) {
        if ((p.K / kTcChunk) % CB) continue;
        for (int G = 1; G <= 8; G *= 2) {
            TcPlan c;
            if (!tc_plan_one(p, num_sms, G, CB, c)) continue;
            const bool better = !found || c.cost < pl.cost - 1e-9 ||
                                (c.cost < pl.cost + 1e-9 && (c.acc > pl.acc || (c.acc == pl.acc && c.stages > pl.stages)));
            if (better) {
                pl = c;
                found = true;
            }
        }
    }
    if (!found) pl.grid = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 256) cache.push_back({key, pl});
    return found;
}

bool gemv_tc_ok(const GemvParams& p, int num_sms) {
    TcPlan pl;
    return tc_plan(p, num_sms, pl);
}

cudaError_t launch_gemv_tc(GemvParams p, int num_sms, cudaStream_t s, bool pdl) {
    TcPlan pl;
    if (!tc_plan(p, num_sms, pl)) return cudaErrorInvalidValue;
    p.tc_stages = pl.stages;
    p.tc_cols = pl.tcols;
    p.tc_band = pl.G;
    p.tc_cb = pl.CB;
    p.tc_contrib = pl.contrib;
    p.tc_acc = pl.acc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    CUtensorMap tm;  // a kernel parameter: the TMA unit reads it from parameter space
    memcpy(&tm, p.tmap, sizeof(tm));
    return cudaLaunchKernelEx(&cfg, k_gemv_tc, p, tm);
}

const void* gemv_tc_kernel() { return reinterpret_cast<const void*>(&k_gemv_tc); }

cudaError_t gemv_tc_configure() {
    return cudaFuncSetAttribute(k_gemv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem);
}

// The TMA descriptor of a row-major [N][K] bf16 matrix: boxes of 128 rows x 64 k, 128-byte
// swizzle (the layout the MMA's shared-memory descriptors assume).  Written to out (128 bytes).
cudaError_t gemv_tc_encode(const void* W, int N, int K, void* out) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (((uintptr_t)W & 15u) || N < kTcRows || K < kTcChunk || K % kTcChunk) return cudaErrorInvalidValue;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {kTcChunk, kTcRows};
    cuuint32_t es[2] = {1, 1};
    const CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                           const_cast<void*>(W), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace dec
