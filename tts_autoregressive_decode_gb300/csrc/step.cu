// step.cu -- the whole decode step of m <= 2 rows as one persistent, cooperative kernel (sm_103a).
//
// The step is the same sequence of phases as the multi-kernel plan (per layer: norm + q/k/v GEMV,
// attention chunks, their merge, o-proj GEMV, norm + gate/up GEMV, down GEMV; then the output
// rows), but every CTA stays resident for the whole step and the phases are separated by a
// grid-wide barrier instead of kernel boundaries.  What that buys on a bandwidth-bound step:
//   * each CTA issues the first two weight batches of the NEXT GEMV phase before it arrives at the
//     barrier, so HBM keeps streaming while the barrier completes -- no launch ramp, no drain;
//   * each CTA starts the bulk copy of its attention chunk's cached K/V rows into shared memory
//     while the preceding GEMV phases stream (the copy is issued at the start of layer l-1's
//     o-proj phase for layer l), so the attention phase finds its rows already staged.
// Work inside a phase is split over the CTAs exactly as the stand-alone kernels split it over
// their grids (gemv_rows.cuh, attention_chunk.cuh), so both plans give bitwise-identical
// results when the GEMV grids match.
//
// The launch is cooperative, so all CTAs are co-resident and every barrier completes; each
// barrier wait is still bounded (kGridWaitIters polls), after which the CTA flags
// CHECK_WAIT_LIMIT, waits (bounded) for its own copies in flight and leaves.  A CTA arrives at a
// barrier as soon as its part of the phase is written and only then issues the next phase's
// weight loads, so the arrival never waits for those loads.
#include "attention_chunk.cuh"
#include "common.cuh"
#include "final_row.cuh"
#include "gemv_rows.cuh"
#include "kernels.h"

namespace dec {

constexpr int kStepThreads = 256;
static_assert(kStepThreads == kRowsThreads && kStepThreads == kChunkThreads, "one CTA shape");
// One CTA per SM: each thread may hold up to 255 registers, so the GEMV keeps two buffers of 16
// 16-byte weight loads in flight (128 KB per SM) without spilling, and shared memory has room
// to stage two attention items per CTA.
constexpr int kStepBuf = 16;
constexpr int kStaged = 2;
constexpr uint32_t kGridWaitIters = 1u << 21;

// ---- grid barrier -----------------------------------------------------------------------------
// Arrival is a release reduction (no return value, so the arriving thread does not wait for it);
// the wait polls the count with acquire loads.  Between the two a CTA issues work that does not
// depend on the other CTAs (the next phase's weight loads), so the barrier latency overlaps it.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_gpu(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_gpu(unsigned* p, unsigned v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Thread 0, after a __syncthreads that follows the CTA's writes of the phase.
__device__ __forceinline__ void grid_arrive(GridBarrier* b) { red_release_add_gpu(&b->count, 1u); }

// Thread 0: wait until `target` arrivals; false when the wait bound ran out (status flagged).
__device__ __forceinline__ bool grid_wait(GridBarrier* b, unsigned target, unsigned* status) {
    uint32_t it = 0;
    while ((int)(ld_acquire_gpu(&b->count) - target) < 0) {
        if (++it > kGridWaitIters) {
            flag_check(status, CHECK_WAIT_LIMIT);
            return false;
        }
    }
    return true;
}

// ---- attention items ------------------------------------------------------------------------------
// The step's attention work list is (stream r, kv head g, chunk c) in that nesting; it depends only
// on the stream lengths at the start of the step, so it is the same for every layer.
__device__ __forceinline__ int stream_chunks(const AttnParams& a, int r) {
    const int len = __ldcg(a.len + r);
    const int L = a.mode == ATTN_TALKER ? len + 1 : a.slots;
    int nch = (L + kAttnChunk - 1) / kAttnChunk;
    // an out-of-range length still gets one item, which flags it
    if (nch < 1 || nch > a.max_chunks) nch = 1;
    return nch;
}

__device__ __forceinline__ int attn_items(const AttnParams& a) {
    int n = 0;
    for (int r = 0; r < a.m; ++r) n += a.G * stream_chunks(a, r);
    return n;
}

__device__ __forceinline__ void attn_item(const AttnParams& a, int i, int& r, int& g, int& c) {
    for (r = 0; r < a.m; ++r) {
        const int nch = stream_chunks(a, r);
        if (i < a.G * nch) break;
        i -= a.G * nch;
    }
    g = i / stream_chunks(a, r);
    c = i - g * stream_chunks(a, r);
}

// ---- GEMV dispatch on the granules per lane ---------------------------------------------------------
template <int DT, int MT>
__device__ __forceinline__ void gemv_issue(const GemvParams& g, int nj, int b, int P,
                                           uint4 (&wa)[kStepBuf], uint4 (&wb)[kStepBuf]) {
    switch (nj) {
        case 1: RowsGemv<DT, MT, 1, kStepBuf>::issue(g, b, P, wa, wb); break;
        case 2: RowsGemv<DT, MT, 2, kStepBuf>::issue(g, b, P, wa, wb); break;
        case 3: RowsGemv<DT, MT, 3, kStepBuf>::issue(g, b, P, wa, wb); break;
        default: RowsGemv<DT, MT, 4, kStepBuf>::issue(g, b, P, wa, wb); break;
    }
}

template <int DT, int MT>
__device__ __forceinline__ void gemv_run(const GemvParams& g, int nj, int b, int P,
                                         uint4 (&wa)[kStepBuf], uint4 (&wb)[kStepBuf], float* sh) {
    switch (nj) {
        case 1: RowsGemv<DT, MT, 1, kStepBuf>::run(g, b, P, wa, wb, sh); break;
        case 2: RowsGemv<DT, MT, 2, kStepBuf>::run(g, b, P, wa, wb, sh); break;
        case 3: RowsGemv<DT, MT, 3, kStepBuf>::run(g, b, P, wa, wb, sh); break;
        default: RowsGemv<DT, MT, 4, kStepBuf>::run(g, b, P, wa, wb, sh); break;
    }
}

// A phase descriptor is copied into shared memory by the CTA's threads, one word each: the load
// is issued early (fetch_phase) and stored late (store_phase), so its latency overlaps the work
// of the current phase.
constexpr int kPhaseWords = (int)(sizeof(StepPhase) / sizeof(int));
static_assert(kPhaseWords <= kStepThreads, "one descriptor word per thread");

__device__ __forceinline__ int fetch_phase(const StepPhase* src) {
    return threadIdx.x < kPhaseWords ? __ldg(reinterpret_cast<const int*>(src) + threadIdx.x) : 0;
}
__device__ __forceinline__ void store_phase(StepPhase* dst, int word) {
    if (threadIdx.x < kPhaseWords) reinterpret_cast<int*>(dst)[threadIdx.x] = word;
}

// Thread 0, once the descriptor's words are stored: the launch's input / output pointers.
__device__ __forceinline__ void patch_io(StepPhase& ph, const StepParams& sp) {
    if (ph.io & IO_X) ph.g.x = sp.x_in;
    if (ph.io & IO_RES) ph.g.res = sp.x_in;
    if (ph.io & IO_OUT) ph.f.out = sp.out;
}

// ---- the kernel -----------------------------------------------------------------------------------------
template <int DT, int MT, int D>
__global__ void __launch_bounds__(kStepThreads, 1) k_step(const __grid_constant__ StepParams sp) {
    extern __shared__ __align__(128) float dsm[];  // kStaged attention item areas; merge scratch
    __shared__ float gsh[rows_smem_floats<MT>()];
    __shared__ __align__(16) StepPhase ph[2];
    __shared__ __align__(8) uint64_t mbar[kStaged];
    __shared__ int s_flag;
    // This CTA's first kStaged attention items (b, b + P, ...), the same in every layer of the
    // step (the list depends only on the stream lengths): found once, so staging them later
    // costs no dependent loads.
    __shared__ struct {
        int r, g, c, ok;
        ChunkInfo ci;
        size_t off;  // floats from a layer's K (V) cache base to the item's first staged row
    } s_item[kStaged];
    __shared__ int s_items;  // attention items of the step

    const int b = blockIdx.x, P = gridDim.x, tid = threadIdx.x;
    uint32_t parity = 0;  // bit h: the phase area h's barrier waits for next (kept by half h)
    bool staged = false;  // block-uniform: the copies of this CTA's items are in flight
    // thread 0: the barrier count at the start of this launch (stable until every CTA has
    // passed the last barrier, after which CTA 0 advances it)
    const unsigned base = tid == 0 ? ld_relaxed_gpu(&sp.bar->base) : 0u;

    if (tid < kStaged) mbar_init(smem_u32(&mbar[tid]), 1);
    store_phase(&ph[0], fetch_phase(sp.phases));
    __syncthreads();
    if (tid == 0) {
        patch_io(ph[0], sp);
        s_items = 0;
        for (int k = 0; k < kStaged; ++k) s_item[k].ok = 0;
        if (sp.attn0 >= 0) {
            const AttnParams& a = sp.phases[sp.attn0].a;
            s_items = attn_items(a);
            for (int k = 0; k < kStaged && b + k * P < s_items; ++k) {
                int r, g, c;
                attn_item(a, b + k * P, r, g, c);
                s_item[k].r = r;
                s_item[k].g = g;
                s_item[k].c = c;
                s_item[k].ci = chunk_info(a, r, c);
                s_item[k].ok = !s_item[k].ci.bad;
                s_item[k].off = (((size_t)r * a.G + g) * a.slots + s_item[k].ci.k0) * D;
            }
        }
    }
    __syncthreads();

    uint4 wa[kStepBuf], wb[kStepBuf];
    if (ph[0].type == PH_GEMV) gemv_issue<DT, MT>(ph[0].g, ph[0].nj, b, P, wa, wb);

    for (int i = 0; i < sp.n_phases; ++i) {
        const StepPhase& cur = ph[i & 1];
        // the next phase's descriptor, in flight while this phase works
        const int next_word = i + 1 < sp.n_phases ? fetch_phase(sp.phases + i + 1) : 0;
        if (cur.type != PH_GEMV) {
            // the weight buffers are dead until the next GEMV phase issues them: say so, so that
            // they hold no registers through the attention and merge code
#pragma unroll
            for (int k = 0; k < kStepBuf; ++k) wa[k] = wb[k] = make_uint4(0u, 0u, 0u, 0u);
        }

        // start staging this CTA's attention items of a later phase (shared memory is free
        // from here until that phase)
        if (cur.stage_attn >= 0 && !staged) {
            // the areas were last read and written by threads (previous attention, merge)
            fence_proxy_async_smem();
            __syncthreads();
            if (tid < kStaged && s_item[tid].ok) {
                const ChunkSmem cs = chunk_smem<D>(dsm + (size_t)tid * chunk_smem_floats(D));
                const uint32_t bar = smem_u32(&mbar[tid]);
                const int nc = s_item[tid].ci.ncached;
                const uint32_t bytes = (uint32_t)(nc > 0 ? nc : 0) * D * sizeof(float);
                mbar_arrive_expect_tx(bar, 2 * bytes);
                if (bytes) {
                    bulk_g2s(smem_u32(cs.Ks), cur.stage_kc + s_item[tid].off, bytes, bar);
                    bulk_g2s(smem_u32(cs.Vs), cur.stage_vc + s_item[tid].off, bytes, bar);
                }
            }
            staged = true;
        }

        switch (cur.type) {
            case PH_GEMV:
                gemv_run<DT, MT>(cur.g, cur.nj, b, P, wa, wb, gsh);
                break;
            case PH_ATTN: {
                // the two halves of the CTA work on its items concurrently: half h takes items
                // b + j P for j = h, h + 2, ... in staging area h, with named barrier 1 + h
                constexpr int NT = kStepThreads / kStaged;
                const AttnParams& a = cur.a;
                const int items = s_items;
                const int h = tid / NT, gtid = tid - h * NT;
                const ChunkSmem cs = chunk_smem<D>(dsm + (size_t)h * chunk_smem_floats(D));
                const uint32_t bar = smem_u32(&mbar[h]);
                for (int j = h; b + j * P < items; j += kStaged) {
                    int r, g, c;
                    ChunkInfo ci;
                    if (j < kStaged) {
                        r = s_item[j].r;
                        g = s_item[j].g;
                        c = s_item[j].c;
                        ci = s_item[j].ci;
                    } else {
                        attn_item(a, b + j * P, r, g, c);
                        ci = chunk_info(a, r, c);
                    }
                    if (ci.bad) {
                        if (gtid == 0) flag_check(a.status, CHECK_BOUNDS);
                        continue;
                    }
                    if (!(staged && j < kStaged)) {
                        fence_proxy_async_smem();
                        group_sync<NT>(1 + h);  // the previous item is done with the area
                        if (gtid == 0) chunk_issue<D>(a, r, g, ci, cs, bar);
                    }
                    chunk_compute<D, NT>(a, r, g, c, ci, cs, bar, (parity >> h) & 1u, gtid, 1 + h);
                    parity ^= 1u << h;  // (only this half's threads use bit h)
                }
                __syncthreads();
                staged = false;
                break;
            }
            case PH_MERGE: {
                constexpr int SUB = kStepThreads / D;
                const int total = cur.a.m * cur.a.H;
                for (int base_item = b * SUB; base_item < total; base_item += P * SUB)
                    merge_items<D, kStepThreads>(cur.a, base_item, total, dsm);
                break;
            }
            default:  // PH_FINAL
                for (int r = b; r < cur.f.m; r += P) {
                    final_row(cur.f, r, gsh);
                    __syncthreads();
                    if (tid == 0) cur.f.len[r] += 1;
                }
                break;
        }

        if (i + 1 < sp.n_phases) {
            // (the next descriptor's buffer held the previous phase, which every thread has left)
            store_phase(&ph[(i + 1) & 1], next_word);
            __syncthreads();  // the phase's writes are issued; the next descriptor is in place
            if (tid == 0) {
                grid_arrive(sp.bar);
                patch_io(ph[(i + 1) & 1], sp);  // read only after the barrier's __syncthreads
            }
            const StepPhase& nxt = ph[(i + 1) & 1];
            if (nxt.type == PH_GEMV) gemv_issue<DT, MT>(nxt.g, nxt.nj, b, P, wa, wb);
            if (tid == 0)
                s_flag = grid_wait(sp.bar, base + (unsigned)(i + 1) * (unsigned)P, sp.status);
            __syncthreads();
            if (!s_flag) {
                // own copies land before leaving (each half knows its own area's phase)
                const int h = tid / (kStepThreads / kStaged);
                if (staged && s_item[h].ok) mbar_wait_bounded(smem_u32(&mbar[h]), (parity >> h) & 1u);
                return;
            }
        }
    }
    // every CTA has passed the last barrier, so all have read `base`: advance it for the next launch
    if (b == 0 && tid == 0)
        st_relaxed_gpu(&sp.bar->base, base + (unsigned)(sp.n_phases - 1) * (unsigned)P);
}

// ---- host side ---------------------------------------------------------------------------------------------
template <int DT, int MT, int D>
static size_t step_smem() {
    return kStaged * chunk_smem_floats(D) * sizeof(float);
}

template <int DT, int MT, int D>
static int step_grid_t(int num_sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_step<DT, MT, D>, kStepThreads,
                                                      step_smem<DT, MT, D>()) != cudaSuccess)
        return 0;
    return per_sm >= 1 ? num_sms : 0;  // one CTA per SM
}

template <int DT, int MT, int D>
static cudaError_t configure_t() {
    return cudaFuncSetAttribute(k_step<DT, MT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)step_smem<DT, MT, D>());
}

template <int DT, int MT, int D>
static cudaError_t launch_t(const StepParams& sp, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = step_smem<DT, MT, D>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_step<DT, MT, D>, sp);
}

#define STEP_DISPATCH(FN, ...)                                                   \
    do {                                                                         \
        const int mt = m <= 1 ? 1 : 2;                                           \
        if (dtype == 1) {                                                        \
            if (mt == 1) return d == 64 ? FN<1, 1, 64>(__VA_ARGS__) : FN<1, 1, 128>(__VA_ARGS__); \
            return d == 64 ? FN<1, 2, 64>(__VA_ARGS__) : FN<1, 2, 128>(__VA_ARGS__);             \
        }                                                                        \
        if (mt == 1) return d == 64 ? FN<0, 1, 64>(__VA_ARGS__) : FN<0, 1, 128>(__VA_ARGS__);     \
        return d == 64 ? FN<0, 2, 64>(__VA_ARGS__) : FN<0, 2, 128>(__VA_ARGS__);                 \
    } while (0)

int step_grid(int dtype, int m, int d, int num_sms) {
    if (m < 1 || m > 2 || (d != 64 && d != 128)) return 0;
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return 0;
    STEP_DISPATCH(step_grid_t, num_sms);
}

cudaError_t step_configure() {
    cudaError_t e;
    if ((e = configure_t<0, 1, 64>()) != cudaSuccess || (e = configure_t<0, 1, 128>()) != cudaSuccess ||
        (e = configure_t<0, 2, 64>()) != cudaSuccess || (e = configure_t<0, 2, 128>()) != cudaSuccess ||
        (e = configure_t<1, 1, 64>()) != cudaSuccess || (e = configure_t<1, 1, 128>()) != cudaSuccess ||
        (e = configure_t<1, 2, 64>()) != cudaSuccess || (e = configure_t<1, 2, 128>()) != cudaSuccess)
        return e;
    return cudaSuccess;
}

cudaError_t launch_step(const StepParams& sp, int dtype, int m, int d, int grid, cudaStream_t s) {
    if (m < 1 || m > 2 || (d != 64 && d != 128) || grid < 1) return cudaErrorInvalidValue;
    STEP_DISPATCH(launch_t, sp, grid, s);
}

}  // namespace dec
