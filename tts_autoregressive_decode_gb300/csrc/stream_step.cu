// stream_step.cu -- the whole decode step of m <= 2 rows as one persistent kernel (sm_103a).
//
// A step is a fixed list of phases (per layer: norm + q/k/v GEMV, attention over the cache,
// merge of the attention partials, o-proj + residual, norm + gate/up + SwiGLU, down + residual;
// then the output rows), the talker's build_step_plan and Mimi's transformer_shaped with the
// elementwise passes folded into GEMV prologues and epilogues.  What bounds a single-token step
// is HBM bandwidth, so the kernel is organised around keeping the weight stream going:
//
//   * one CTA per SM (cooperative launch, so all CTAs are resident); 8 consumer warps and one
//     producer warp;
//   * the producer walks the CTA's share of every phase in order -- its rows of each weight
//     matrix, its keys of each layer's K/V cache -- and copies them into a ring of shared-memory
//     slots with 1-D bulk copies (cp.async.bulk, completion counted on a per-slot mbarrier).  It
//     waits only for a free slot, never for an activation: weights and cached K/V rows do not
//     depend on the step, so the ring fills with the next phases' bytes while the consumers wait
//     for the current phase's input;
//   * a phase's inputs are the outputs of the phase before it (or of earlier ones, complete by
//     then).  When a CTA has written its part of phase i, its thread 0 adds 1 to the phase's
//     counter with release semantics; the consumers of phase i + 1 start once thread 0 has seen
//     the counter reach the grid size (acquire), so only one thread per CTA polls, on one word.
//     The activations themselves are tagged 64-bit words (value | tag << 32, tag = the plan's
//     launch count and the layer), read once and checked: a word with another tag (which the
//     counter makes impossible) is polled until it is right.  Every buffer is rewritten once per
//     layer; a reader of layer l can only see layer l's words or older ones, never newer (each
//     write of a buffer depends, through the phase chain, on every read of its previous contents);
//   * the attention keys of all (stream, kv head) pairs are laid end to end and split evenly over
//     the CTAs; each CTA computes an online-softmax partial for every q head of the groups it
//     touches (kv head of q head i is i / (H / G): K/V are read once), and the merge phase
//     combines the partials of each q head (out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c,
//     the running-max rescaling of REL_POS_ATTN on the Parakeet page).
//
// Every wait is bounded: mbarrier waits by try_wait rounds, tag polls by `polls` loads.  A wait
// that runs out flags CHECK_WAIT_LIMIT in the device check word and the CTA stops: its consumers
// leave the phase loop together, its producer stops issuing copies, and before the CTA exits its
// thread 0 waits (bounded) until the copies already issued have landed.
#include <math_constants.h>

#include "attention_chunk.cuh"
#include "common.cuh"
#include "gemv_rows.cuh"
#include "kernels.h"

namespace dec {

namespace {

constexpr int kSConsumerWarps = 8;
constexpr int kSConsumers = kSConsumerWarps * 32;
constexpr int kSThreads = kSConsumers + 32;     // + the producer warp
constexpr int kSlots = 6;                       // ring slots
constexpr int kSlotBytes = 32 * 1024;           // 8 rows of 2048 bf16, 2 of 6144, 32 keys of d 128
constexpr int kRedRows = 128;                   // GEMV rows per epilogue segment
constexpr int kWinKeys = 128;                   // attention keys per window (score buffer)
constexpr int kFinalPer = 32;                   // output elements per consumer thread (h <= 8192)
constexpr int kDefaultPolls = 1 << 20;
constexpr uint32_t kStallTag = 0x80000000u;

static_assert(kSConsumers == kRowsThreads, "one granule split with the split-K GEMV");

// keys of one ring slot's tile: the K rows, then the V rows
template <int D>
__host__ __device__ constexpr int tile_keys() {
    return kSlotBytes / (2 * D * (int)sizeof(float));
}
// tiles of one attention window
template <int D>
__host__ __device__ constexpr int win_tiles() {
    return kWinKeys / tile_keys<D>();
}

// ---- dynamic shared memory ---------------------------------------------------------------------
template <int MT, int D>
struct SLayout {
    static constexpr int kRing = 0;
    static constexpr int kRed = kRing + kSlots * kSlotBytes;              // [warps][kRedRows][MT]
    static constexpr int kNred = kRed + kSConsumerWarps * kRedRows * MT * 4;  // [warps][MT]
    static constexpr int kStat = kNred + kSConsumerWarps * MT * 4;        // [2][MT]
    static constexpr int kQs = (kStat + 2 * MT * 4 + 15) / 16 * 16;       // [kMaxGroup][D]
    static constexpr int kSc = kQs + kMaxGroup * D * 4;                   // [kMaxGroup][kWinKeys]
    static constexpr int kKnew = kSc + kMaxGroup * kWinKeys * 4;          // [D]
    static constexpr int kVnew = kKnew + D * 4;                           // [D]
    static constexpr int kSM = kVnew + D * 4;                             // [kMaxGroup] running max
    static constexpr int kSL = kSM + kMaxGroup * 4;                       // [kMaxGroup] running sum
    static constexpr int kSA = kSL + kMaxGroup * 4;                       // [kMaxGroup] rescale
    static constexpr int kStamp = kSA + kMaxGroup * 4;                    // [kWinKeys] u32
    static constexpr int kFlag = kStamp + kWinKeys * 4;                   // [4] int
    static constexpr int kRope = kFlag + 16;                              // cos [2][D], sin [2][D]
    static constexpr int kQKn = kRope + 4 * D * 4;                        // q / k norm weights [2][D]
    static constexpr int kBytes = kQKn + 2 * D * 4;
};

// ---- tagged words -------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t tag_of(uint32_t epoch, int layer) {
    return ((epoch + 1u) << 8) | (uint32_t)layer;
}
// Loads of tagged words for the rounds of a poll: the value and the tag of each word land in
// registers of their own, from L2 (.cg: a line another SM rewrote is never served from this
// SM's L1).  The counter protocol orders the data before these loads; the tag is a check.  A
// round issues all its loads before it checks any tag: on an in-order core a check between two
// loads would make the second wait for the first.
__device__ __forceinline__ void ld_pair(const uint64_t* p, float& v0, uint32_t& t0, float& v1,
                                        uint32_t& t1) {
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v0), "=r"(t0), "=f"(v1), "=r"(t1)
                 : "l"(p)
                 : "memory");
}
__device__ __forceinline__ void ld_one(const uint64_t* p, float& v, uint32_t& t) {
    asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=f"(v), "=r"(t) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_word(uint64_t* p, float v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_gpu(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---- waits and shared-memory loads of the hot loops ----------------------------------------------
// try_wait with a suspend-time hint: a thread whose phase has not completed sleeps (up to the
// hint) until it does, instead of spinning on the barrier and taking issue slots from the warps
// that compute.
constexpr uint32_t kSuspendNs = 2000;
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
constexpr int kHintWaits = 1 << 20;  // rounds of up to kSuspendNs each: a bound of seconds
__device__ __forceinline__ bool mbar_wait_hint(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kHintWaits; ++i)
        if (mbar_try_wait_hint(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

// Transposed butterfly over N rows (N = 2 .. 32, a power of two): v[0..N) per lane -> lane l
// returns the warp-wide sum of v[l >> (5 - log2 N)]; the 32 / N lanes of a row all hold it.
// At each exchange level the lanes whose bit is set keep the upper half of the values and
// send the lower half, so a level halves the values a lane carries; the remaining levels are a
// plain reduction.  One chain of five shuffle levels serves all N rows.
template <int N, int M>
__device__ __forceinline__ void bfly_level(float* cur, int lane) {
    if constexpr (M >= 1) {
        if constexpr (N > 1) {
            const bool hi = lane & M;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = hi ? cur[i] : cur[i + N / 2];
                const float keep = hi ? cur[i + N / 2] : cur[i];
                cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            bfly_level<N / 2, M / 2>(cur, lane);
        } else {
            cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], M);
            bfly_level<1, M / 2>(cur, lane);
        }
    }
}
template <int N>
__device__ __forceinline__ float butterfly_n(const float (&v)[N], int lane) {
    float cur[N];
#pragma unroll
    for (int i = 0; i < N; ++i) cur[i] = v[i];
    bfly_level<N, 16>(cur, lane);
    return cur[0];
}
__host__ __device__ constexpr int log2_of(int n) { return n <= 1 ? 0 : 1 + log2_of(n / 2); }

// Rows of one GEMV tile for NJ granules per consumer thread: 8 rows of <= 4 KB, 4 of <= 8 KB,
// 2 of <= 16 KB (all within a slot); the producer cuts the CTA's rows into tiles of this size.
__host__ __device__ constexpr int gemv_tile_rows(int nj) { return nj == 1 ? 8 : (nj == 2 ? 4 : 2); }

// ---- consumer-group barriers (named barrier 1 over the 256 consumer threads) -----------------
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"r"(kSConsumers) : "memory"); }
__device__ __forceinline__ bool cbar_or(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pv, pr;\n\t"
        "setp.ne.u32 pv, %1, 0;\n\t"
        "bar.red.or.pred pr, 1, %2, pv;\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(kSConsumers)
        : "memory");
    return out != 0;
}

// ---- per-launch context ------------------------------------------------------------------------
// The CTA-uniform part lives in shared memory; every phase function copies it into registers on
// entry (a context reached through a pointer to the stack would live in local memory, which the
// small L1 left beside the ring turns into L2 round trips inside the hot loops).  No arrays, so
// no indexing can push it to local memory either.
struct SCtx {
    int b, P, m;                // CTA, grid, rows
    char* ring;                 // generic address of the ring
    uint32_t full0, empty0;     // shared addresses of full[0] / empty[0] (8-byte stride)
    uint32_t epoch;
    const float* x_in;
    int polls;
    volatile int* abort;
    unsigned* status;
    bool stall;                 // this phase waits for a tag nothing writes
    int len0, len1;             // stream lengths (positions) of rows 0 and 1
    int L0, L1;                 // keys per (stream, kv head) of rows 0 and 1
    int T;                      // keys of all (stream, kv head) pairs of the attention phase
};
__device__ __forceinline__ int len_of(const SCtx& c, int r) { return r ? c.len1 : c.len0; }
__device__ __forceinline__ int keys_of(const SCtx& c, int r) { return r ? c.L1 : c.L0; }

__device__ __forceinline__ uint32_t full_bar(const SCtx& c, uint32_t t) { return c.full0 + 8u * (t % kSlots); }
__device__ __forceinline__ uint32_t empty_bar(const SCtx& c, uint32_t t) { return c.empty0 + 8u * (t % kSlots); }
__device__ __forceinline__ char* slot_ptr(const SCtx& c, uint32_t t) { return c.ring + (size_t)(t % kSlots) * kSlotBytes; }

// consumers: wait until tile t has landed; release it when every lane of the warp is done with it
__device__ __forceinline__ bool tile_wait(const SCtx& c, uint32_t t) {
    return mbar_wait_hint(full_bar(c, t), (t / kSlots) & 1u);
}
__device__ __forceinline__ uint32_t slot_addr(const SCtx& c, uint32_t t) {
    return smem_u32(c.ring) + (t % kSlots) * (uint32_t)kSlotBytes;
}
__device__ __forceinline__ void tile_release(const SCtx& c, uint32_t t) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar(c, t));
}

// Every consumer calls it after a cbar_or that came back true: flag the check word once and
// tell the producer to stop.
__device__ __forceinline__ void consumers_abort(const SCtx& c) {
    if (threadIdx.x == 0) {
        flag_check(c.status, CHECK_WAIT_LIMIT);
        *c.abort = 1;
    }
}

// ---- work split ----------------------------------------------------------------------------------
// rows [row0, row0 + nrows) of CTA b of P: whole partition units, as the split-K GEMV splits them
__device__ __forceinline__ void gemv_range(const SGemv& g, int b, int P, int& row0, int& nrows) {
    const int units = g.N / g.unit;
    const int u0 = (int)((long long)b * units / P);
    const int u1 = (int)((long long)(b + 1) * units / P);
    row0 = u0 * g.unit;
    nrows = (u1 - u0) * g.unit;
}

// The attention keys of all (stream r, kv head g) pairs laid end to end (r outer, g inner, keys
// ascending) and split evenly: CTA b takes [start(b), start(b + 1)).
// (32-bit: the host admits the plan only when T * (grid + 1) < 2^32)
__device__ __forceinline__ int key_start(const SCtx& c, int b) {
    return (int)((uint32_t)b * (uint32_t)c.T / (uint32_t)c.P);
}
// the CTA whose range holds flat key x
__device__ __forceinline__ int key_cta(const SCtx& c, int x) {
    return (int)(((uint32_t)(x + 1) * (uint32_t)c.P - 1u) / (uint32_t)c.T);
}

// One segment of a CTA's key range: keys [k0, k1) of (stream r, kv head g).
struct Seg {
    int r, g, k0, k1;
};

// The segment that starts at flat key s (s inside the CTA's range ending at s1).
__device__ __forceinline__ Seg seg_at(const SCtx& c, int G, int s, int s1) {
    Seg q;
    int off = s;
    q.r = 0;
    while (q.r + 1 < c.m && off >= G * keys_of(c, q.r)) {
        off -= G * keys_of(c, q.r);
        ++q.r;
    }
    const int L = keys_of(c, q.r);
    q.g = off / L;
    q.k0 = off - q.g * L;
    q.k1 = min(L, q.k0 + (s1 - s));
    return q;
}

// ==================================================================================================
// producer
// ==================================================================================================
struct Producer {
    const SCtx c;
    uint64_t pol;
    uint32_t t = 0;  // tiles issued
    __device__ Producer(const SCtx& cc) : c(cc), pol(l2_evict_first()) {}

    // a free slot for tile t: the consumers have released the tile kSlots before it
    __device__ bool acquire() {
        if (t < (uint32_t)kSlots) return true;
        const uint32_t bar = empty_bar(c, t), par = ((t / kSlots) - 1u) & 1u;
        for (int i = 0; i < kHintWaits; ++i) {
            if (mbar_try_wait_hint(bar, par)) return true;
            if (*c.abort) return false;
        }
        flag_check(c.status, CHECK_WAIT_LIMIT);
        *c.abort = 1;
        return false;
    }

    __device__ bool gemv(const SGemv& g, int es, int nj) {
        int row0, nrows;
        gemv_range(g, c.b, c.P, row0, nrows);
        const size_t row_bytes = (size_t)g.K * es;
        const int R = gemv_tile_rows(nj);
        const char* W = static_cast<const char*>(g.W) + (size_t)row0 * row_bytes;
        for (int i = 0; i < nrows; i += R) {
            if (!acquire()) return false;
            const uint32_t bytes = (uint32_t)(min(R, nrows - i) * row_bytes);
            const uint32_t bar = full_bar(c, t);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s_pol(smem_u32(slot_ptr(c, t)), W + (size_t)i * row_bytes, bytes, bar, pol);
            ++t;
        }
        return true;
    }

    template <int D>
    __device__ bool attn(const SAttn& a) {
        constexpr int TK = tile_keys<D>();
        const int s1 = key_start(c, c.b + 1);
        for (int s = key_start(c, c.b); s < s1;) {
            const Seg q = seg_at(c, a.G, s, s1);
            const int pos = len_of(c, q.r);
            // talker: the row at pos is being appended in this step, it is not copied
            const int cached_end = a.mode == ATTN_TALKER ? min(q.k1, pos) : q.k1;
            const size_t head = ((size_t)q.r * a.G + q.g) * a.slots;
            for (int kk = q.k0; kk < q.k1; kk += TK) {
                if (!acquire()) return false;
                const int nc = max(0, min(kk + TK, cached_end) - kk);
                const uint32_t bytes = (uint32_t)nc * D * sizeof(float);
                const uint32_t bar = full_bar(c, t);
                mbar_arrive_expect_tx(bar, 2 * bytes);
                if (bytes) {
                    const uint32_t dst = smem_u32(slot_ptr(c, t));
                    bulk_g2s_pol(dst, a.kc + (head + kk) * D, bytes, bar, pol);
                    bulk_g2s_pol(dst + TK * D * sizeof(float), a.vc + (head + kk) * D, bytes, bar, pol);
                }
                ++t;
            }
            s += q.k1 - q.k0;
        }
        return true;
    }
};

// The producer lane: every phase's tiles in order; returns the number of tiles issued.
template <int DT, int D>
__device__ __noinline__ uint32_t run_producer(const SPhase* phases, int n_phases, const SCtx* cp) {
    Producer pr(*cp);
    for (int i = 0; i < n_phases; ++i) {
        const int type = phases[i].type;
        bool ok = true;
        if (type == SP_GEMV) {
            const SGemv g = phases[i].g;
            ok = pr.gemv(g, WType<DT>::ES, phases[i].nj);
        } else if (type == SP_ATTN) {
            const SAttn a = phases[i].a;
            ok = pr.attn<D>(a);
        }
        if (!ok) break;
    }
    return pr.t;
}

// Thread 0: wait until the counter reaches `target` (acquire); false when the wait bound runs out
// or the CTA is stopping.
__device__ __noinline__ bool wait_count(const unsigned* cnt, unsigned target, const SCtx& c) {
    for (int it = 0;; ++it) {
        if ((int)(ld_acquire_gpu(cnt) - target) >= 0) return true;
        if (it >= c.polls || *c.abort) return false;
        __nanosleep(32);
    }
}

// Every consumer thread: thread 0 waits for the counter of the phase before (none for the first
// phase) while the others wait at the barrier.  Operands that depend on nothing (norm weights,
// rope tables) are loaded before the call, so their latency overlaps the wait.
__device__ __forceinline__ bool wait_inputs(const unsigned* cnt, unsigned target, const SCtx& c) {
    bool ok = true;
    if (threadIdx.x == 0 && cnt) ok = wait_count(cnt, target, c);
    return !cbar_or(!ok);
}

// ==================================================================================================
// consumers: GEMV phase
// ==================================================================================================
// y[r][n] = epi(sum_k W[n][k] xin[r][k]) for the CTA's rows.  Consumer thread ct owns the
// 16-byte granules ct + 256 j (j < NJ) of every row (its slice of x lives in registers); the
// rows come from the ring, tile after tile, and are folded across lanes 8 rows at a time.
constexpr uint32_t kFailed = 0xFFFFFFFFu;  // a phase function's return when the step stops

template <int DT, int MT, int NJ>
__device__ __noinline__ uint32_t consume_gemv(const SGemv* gp, const SCtx* cp, uint32_t tile,
                                              float* red, float* nred, float* stat,
                                              const unsigned* wcnt, unsigned wtarget) {
    const SGemv g = *gp;
    const SCtx c = *cp;
    constexpr int VEC = WType<DT>::VEC;
    constexpr int ES = WType<DT>::ES;
    const int ct = threadIdx.x, lane = ct & 31, warp = ct >> 5;
    const int K = g.K, m = c.m, Gn = K / VEC;
    int row0, nrows;
    gemv_range(g, c.b, c.P, row0, nrows);
    const int row_bytes = K * ES;
    constexpr int GR = gemv_tile_rows(NJ);  // rows of one tile
    const int R = GR;
    const int ntiles = (nrows + R - 1) / R;
    const uint32_t stall = c.stall ? kStallTag : 0u;

    int gj[NJ];
    bool ok[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        gj[j] = j * kSConsumers + ct;
        ok[j] = gj[j] < Gn;
    }
    bool bad = false;

    // the residual operand of this thread's output of the first segment, loaded with x
    const int seg_rows = max(1, kRedRows / R) * R;  // rows per epilogue segment, whole tiles
    float res_v = 0.f;
    const int first_out = min(nrows, seg_rows) * m;
    const bool pre_res = g.epi == EPI_RESID && ct < first_out && MT <= 2;

    // ---- operands that depend on nothing, then the wait for the phase before ---------------------
    // (norm weights only for one or two granules a thread: the norms run on the hidden width)
    constexpr bool kPreNorm = NJ <= 2;
    float2 nwv[kPreNorm ? NJ : 1][VEC / 2], nbv[kPreNorm ? NJ : 1][VEC / 2];
    if constexpr (kPreNorm) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) {
                nwv[j][e] = make_float2(1.f, 1.f);
                nbv[j][e] = make_float2(0.f, 0.f);
                if (g.pro != PRO_NONE && ok[j]) {
                    nwv[j][e] = __ldg(reinterpret_cast<const float2*>(g.nw + gj[j] * VEC + 2 * e));
                    if (g.pro != PRO_RMS && g.nb)
                        nbv[j][e] = __ldg(reinterpret_cast<const float2*>(g.nb + gj[j] * VEC + 2 * e));
                }
            }
    }
    const float ls_first = (pre_res && g.ls) ? __ldg(g.ls + row0 + ct / m) : 1.f;
    if (!wait_inputs(wcnt, wtarget, c)) {
        consumers_abort(c);
        return kFailed;
    }

    // ---- x (and the residual): wait until every word carries its tag --------------------------
    float2 xv[MT][NJ][VEC / 2];
    if (g.x) {
        const uint32_t tag = tag_of(c.epoch, g.x_layer) ^ stall;
        const uint32_t rtag = tag_of(c.epoch, g.res_layer) ^ stall;
        for (int it = 0;; ++it) {
            uint32_t tg[MT][NJ][VEC];
            uint32_t rt = rtag;
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                for (int j = 0; j < NJ; ++j)
#pragma unroll
                    for (int q = 0; q < VEC / 2; ++q) {
                        xv[mm][j][q] = make_float2(0.f, 0.f);
                        tg[mm][j][2 * q] = tg[mm][j][2 * q + 1] = tag;
                        if (mm < m && ok[j])
                            ld_pair(g.x + (size_t)mm * g.ldx + (size_t)gj[j] * VEC + 2 * q, xv[mm][j][q].x,
                                    tg[mm][j][2 * q], xv[mm][j][q].y, tg[mm][j][2 * q + 1]);
                    }
            if (pre_res) {
                const int row = row0 + ct / m, mm = ct % m;
                if (g.res) ld_one(g.res + (size_t)mm * g.ldres + row, res_v, rt);
                else res_v = __ldcg(c.x_in + (size_t)mm * g.ldres + row);
            }
            // the checks, once every load of the round is issued
            uint32_t diff = rt ^ rtag;
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                for (int j = 0; j < NJ; ++j)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) diff |= tg[mm][j][e] ^ tag;
            if (diff == 0) break;
            if (it >= c.polls || *c.abort) {
                bad = true;
                break;
            }
            __nanosleep(64);
        }
    } else {
        // the step's input rows, written before the launch
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q) {
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (mm < m && ok[j])
                        a = __ldcg(reinterpret_cast<const float4*>(c.x_in + (size_t)mm * g.ldx +
                                                                   (size_t)gj[j] * VEC) + q);
                    xv[mm][j][2 * q] = make_float2(a.x, a.y);
                    xv[mm][j][2 * q + 1] = make_float2(a.z, a.w);
                }
        if (pre_res) {
            const int row = row0 + ct / m, mm = ct % m;
            const uint32_t rtag = tag_of(c.epoch, g.res_layer) ^ stall;
            if (g.res) {
                for (int it = 0;; ++it) {
                    uint32_t t;
                    ld_one(g.res + (size_t)mm * g.ldres + row, res_v, t);
                    if (t == rtag) break;
                    if (it >= c.polls || *c.abort) {
                        bad = true;
                        break;
                    }
                    __nanosleep(64);
                }
            } else {
                res_v = __ldcg(c.x_in + (size_t)mm * g.ldres + row);
            }
        }
    }
    if (cbar_or(bad)) {
        consumers_abort(c);
        return kFailed;
    }

    // ---- norm prologue: a reduction over the 256 consumer threads --------------------------------
    if (g.pro != PRO_NONE) {
        auto block_sum = [&](float (&v)[MT], int slot) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                const float t = warp_sum(v[mm]);
                if (lane == 0) nred[warp * MT + mm] = t;
            }
            cbar();
            if (ct < MT) {
                float sum = 0.f;
                for (int w = 0; w < kSConsumerWarps; ++w) sum += nred[w * MT + ct];
                stat[slot * MT + ct] = sum / (float)K;
            }
            cbar();
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
                    part[mm] += (g.pro != PRO_RMS) ? v.x + v.y : v.x * v.x + v.y * v.y;
                }
        }
        block_sum(part, 0);
        float inv[MT], mean[MT];
        if (g.pro != PRO_RMS) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                mean[mm] = stat[mm];
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
            for (int mm = 0; mm < MT; ++mm) inv[mm] = 1.0f / sqrtf(stat[MT + mm] + g.eps);
        } else {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                mean[mm] = 0.f;
                inv[mm] = 1.0f / sqrtf(stat[mm] + g.eps);
            }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            if (!ok[j]) continue;
            const int k0 = gj[j] * VEC;
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) {
                float2 w, bb;
                if constexpr (kPreNorm) {
                    w = nwv[j][e];
                    bb = nbv[j][e];
                } else {
                    w = *reinterpret_cast<const float2*>(g.nw + k0 + 2 * e);
                    bb = make_float2(0.f, 0.f);
                    if (g.pro != PRO_RMS && g.nb) bb = *reinterpret_cast<const float2*>(g.nb + k0 + 2 * e);
                }
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) {
                    float2& v = xv[mm][j][e];
                    v.x = (v.x - mean[mm]) * inv[mm] * w.x + bb.x;
                    v.y = (v.y - mean[mm]) * inv[mm] * w.y + bb.y;
                }
            }
        }
    }

    // ---- the rows, tile by tile from the ring ----------------------------------------------------
    // A tile holds GR rows; every load of a tile is issued before its arithmetic.  The per-lane
    // partial sums of TPB tiles (BATCH rows) stay in registers and are folded across the lanes
    // by one transposed butterfly.  Segments (one epilogue each) are whole batches.
    constexpr int TPB = 4;
    constexpr int BATCH = GR * TPB;  // 32, 16 or 8 rows
    static_assert(kRedRows % BATCH == 0, "segments of whole batches");
    const uint32_t ytag = tag_of(c.epoch, g.layer);
    for (int seg = 0; seg < nrows; seg += seg_rows) {
        const int srows = min(seg_rows, nrows - seg);
        for (int b0 = 0; b0 < srows; b0 += BATCH) {
            float part[MT][BATCH];
#pragma unroll
            for (int k = 0; k < TPB; ++k) {
                const int t0 = b0 + k * GR;  // the tile's first row in the segment
                if (t0 < srows) {
                    const int trows = min(GR, srows - t0);
                    const uint32_t tt = tile + (uint32_t)((seg + t0) / GR);
                    if (!bad && !tile_wait(c, tt)) bad = true;
                    const uint32_t base = slot_addr(c, tt);
                    uint4 w[GR][NJ];
#pragma unroll
                    for (int r = 0; r < GR; ++r)
#pragma unroll
                        for (int j = 0; j < NJ; ++j)
                            w[r][j] = (r < trows && ok[j])
                                          ? lds128(base + (uint32_t)(r * row_bytes + gj[j] * 16))
                                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int r = 0; r < GR; ++r) {
                        float2 acc[MT];
#pragma unroll
                        for (int mm = 0; mm < MT; ++mm) acc[mm] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < NJ; ++j) {
                            const uint4 wr = w[r][j];
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
                                for (int e = 0; e < VEC / 2; ++e) acc[mm] = ffma2(wf[e], xv[mm][j][e], acc[mm]);
                        }
#pragma unroll
                        for (int mm = 0; mm < MT; ++mm) part[mm][k * GR + r] = acc[mm].x + acc[mm].y;
                    }
                    tile_release(c, tt);
                } else {
#pragma unroll
                    for (int mm = 0; mm < MT; ++mm)
#pragma unroll
                        for (int r = 0; r < GR; ++r) part[mm][k * GR + r] = 0.f;
                }
            }
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                const float v = butterfly_n<BATCH>(part[mm], lane);
                const int r = lane >> (5 - log2_of(BATCH));
                if ((lane & (32 / BATCH - 1)) == 0 && b0 + r < srows)
                    red[(warp * kRedRows + b0 + r) * MT + mm] = v;
            }
        }
        if (cbar_or(bad)) {  // (also: every warp's sums of the segment are in `red`)
            consumers_abort(c);
            return kFailed;
        }

        // ---- epilogue of the segment: cross-warp sums, tagged stores ------------------------------
        const int rbase = row0 + seg;
        if (g.epi == EPI_SWIGLU) {
            for (int o = ct; o < (srows / 2) * m; o += kSConsumers) {
                const int pr = o / m, mm = o - pr * m;
                float vg = 0.f, vu = 0.f;
                for (int w = 0; w < kSConsumerWarps; ++w) {
                    vg += red[(w * kRedRows + 2 * pr) * MT + mm];
                    vu += red[(w * kRedRows + 2 * pr + 1) * MT + mm];
                }
                st_word(g.y + (size_t)mm * g.ldy + rbase / 2 + pr, silu_f(vg) * vu, ytag);
            }
        } else {
            const uint32_t rtag = tag_of(c.epoch, g.res_layer) ^ stall;
            for (int o = ct; o < srows * m; o += kSConsumers) {
                const int r = o / m, mm = o - r * m;
                float v = 0.f;
                for (int w = 0; w < kSConsumerWarps; ++w) v += red[(w * kRedRows + r) * MT + mm];
                const int row = rbase + r;
                float out;
                if (g.epi == EPI_RESID) {
                    float rv = res_v;
                    if (!(seg == 0 && pre_res)) {
                        if (g.res) {
                            for (int it = 0;; ++it) {
                                uint32_t t;
                                ld_one(g.res + (size_t)mm * g.ldres + row, rv, t);
                                if (t == rtag) break;
                                if (it >= c.polls || *c.abort) {
                                    bad = true;
                                    break;
                                }
                                __nanosleep(64);
                            }
                        } else {
                            rv = __ldcg(c.x_in + (size_t)mm * g.ldres + row);
                        }
                    }
                    const float lsv = !g.ls ? 1.f : ((seg == 0 && pre_res) ? ls_first : g.ls[row]);
                    out = rv + (g.ls ? lsv * v : v);
                    if (g.tap) g.tap[(size_t)mm * g.ldtap + row] = out;
                } else if (g.epi == EPI_GELU) {
                    out = gelu_f(v);
                } else {
                    out = v;
                }
                st_word(g.y + (size_t)mm * g.ldy + row, out, ytag);
            }
        }
        if (cbar_or(bad)) {  // (also: `red` is free for the next segment)
            consumers_abort(c);
            return kFailed;
        }
    }
    return tile + ntiles;
}

// ==================================================================================================
// consumers: attention phase
// ==================================================================================================
template <int D>
struct AttnSmem {
    int* flag;        // [1] broadcast of thread 0's arrival result
    float* rcs;       // [2][D] cos of each element's frequency at stream r's position
    float* rsn;       // [2][D] sin
    float* qkn;       // [2][D] q norm weight, k norm weight
    float* qs;        // [kMaxGroup][D]
    float* sc;        // [kMaxGroup][kWinKeys]
    float* knew;      // [D]
    float* vnew;      // [D]
    float* sM;        // [kMaxGroup]
    float* sL;
    float* sA;
    uint32_t* stamp;  // [kWinKeys]
};

// Poll D / 32 tagged words a lane (element lane + 32 j) of a raw q/k/v head; false on timeout.
template <int D>
__device__ __forceinline__ bool poll_head(const SCtx& c, const uint64_t* src, uint32_t tag,
                                          int lane, float (&v)[D / 32]) {
    for (int it = 0;; ++it) {
        uint32_t t[D / 32];
#pragma unroll
        for (int j = 0; j < D / 32; ++j) ld_one(src + lane + 32 * j, v[j], t[j]);
        uint32_t diff = 0;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) diff |= t[j] ^ tag;
        if (__all_sync(0xffffffffu, diff == 0)) return true;
        // (a warp vote: every lane leaves the loop together)
        if (__any_sync(0xffffffffu, it >= c.polls || *c.abort)) return false;
        __nanosleep(64);
    }
}

// ==================================================================================================
// merge of the attention partials (run by the CTA that completes a (stream, kv head) pair)
// ==================================================================================================
// One warp, one unit (stream r, q head hq, 32 output dims).  The partials of (r, kv head g) are
// those of CTAs bf..bl (the CTAs whose key ranges meet g's keys): load each one's (max, sum) and
// the unit's 32 values of its output, all in one round, then
// out = sum_c w_c o_c / sum_c w_c l_c with w_c = e^(m_c - M), M the largest m_c (the running
// rescaling of REL_POS_ATTN on the Parakeet page).  False when the partials' tags did not show.
template <int D>
__device__ __noinline__ bool merge_unit(const SAttn* ap, const SCtx* cp, int r, int hq, int sl,
                                        int bf, int bl, uint32_t tag, uint32_t otag, int lane) {
    const SAttn a = *ap;
    const SCtx c = *cp;
    const bool sparse = c.T < c.P;  // some CTAs may have no keys at all
    const size_t base = ((size_t)r * a.H + hq) * c.P;
    const int dim = sl * 32 + lane;
    float M = -CUDART_INF_F, den = 0.f, num = 0.f;
    for (int b0 = bf; b0 <= bl; b0 += 32) {
        // this lane's partial (b0 + lane): its (max, sum); every lane: 32 partials' values
        const int bj = b0 + lane;
        const bool mine = bj <= bl && (!sparse || key_start(c, bj) < key_start(c, bj + 1));
        float mj = -CUDART_INF_F, lj = 0.f;
        float ov[32];
        uint32_t has = 0;  // bit jj: partial b0 + jj exists
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int bb = b0 + jj;
            if (bb <= bl && (!sparse || key_start(c, bb) < key_start(c, bb + 1))) has |= 1u << jj;
        }
        for (int it = 0;; ++it) {
            uint32_t tm0 = tag, tm1 = tag, to[32];
            if (mine) ld_pair(a.ml + 2 * (base + bj), mj, tm0, lj, tm1);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                ov[jj] = 0.f;
                to[jj] = tag;
                if (has >> jj & 1u) ld_one(a.part + (base + b0 + jj) * D + dim, ov[jj], to[jj]);
            }
            uint32_t diff = (tm0 ^ tag) | (tm1 ^ tag);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) diff |= to[jj] ^ tag;
            if (__all_sync(0xffffffffu, diff == 0)) break;
            if (__any_sync(0xffffffffu, it >= c.polls || *c.abort)) return false;  // warp-uniform
            __nanosleep(64);
        }
        if (!mine || lj <= 0.f) mj = -CUDART_INF_F;
        // fold this batch into the running (M, den, num)
        const float Mb = warp_max(mj);
        const float Mn = fmaxf(M, Mb);
        const float scale_old = M == -CUDART_INF_F ? 0.f : expf(M - Mn);
        const float wj = mj == -CUDART_INF_F ? 0.f : expf(mj - Mn);
        den = den * scale_old + warp_sum(wj * lj);
        float nb = 0.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) nb += __shfl_sync(0xffffffffu, wj, jj) * ov[jj];
        num = num * scale_old + nb;
        M = Mn;
    }
    st_word(a.out + (size_t)r * a.H * D + (size_t)hq * D + dim, num / den, otag);
    return true;
}

// rope of a head held D/32 values a lane (element lane + 32 j) with the lane's cos / sin already
// loaded (cs[j], sn[j] belong to element lane + 32 j): rotate_half (ROPE_SRC) or interleaved
// pairs (rope_push_src) -> out[t]
template <int D>
__device__ __forceinline__ void rope_store(bool half, int lane, const float (&v)[D / 32],
                                           const float* cs, const float* sn, float* out) {
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
        const int t = lane + 32 * j;
        if (half) {
            const int jj = (j + D / 64) % (D / 32);  // element t +- D/2, same lane
            const float rot = (t < D / 2) ? -v[jj] : v[jj];
            out[t] = v[j] * cs[t] + rot * sn[t];
        } else {
            // pair (2i, 2i+1) straddles lanes; even t: a c - b s, odd t: a s + b c
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            out[t] = (t & 1) ? other * sn[t] + v[j] * cs[t] : v[j] * cs[t] - other * sn[t];
        }
    }
}
// per-head RMSNorm with the shared [D] weight (QK_NORM_SRC) staged in shared memory
template <int D>
__device__ __forceinline__ void head_rms_pre(float (&v)[D / 32], const float* w, float eps, int lane) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) ss += v[j] * v[j];
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)D + eps);
#pragma unroll
    for (int j = 0; j < D / 32; ++j) v[j] = v[j] * inv * w[lane + 32 * j];
}

template <int D>
__device__ __noinline__ uint32_t consume_attn(const SAttn* ap, const SCtx* cp, uint32_t tile,
                                              const AttnSmem<D>* smp, const unsigned* wcnt,
                                              unsigned wtarget) {
    const SAttn a = *ap;
    const SCtx c = *cp;
    const AttnSmem<D> sm = *smp;
    constexpr int TK = tile_keys<D>();
    constexpr int WT = win_tiles<D>();
    constexpr int PER = D / 32;
    constexpr int NU = (kMaxGroup * D + kSConsumers - 1) / kSConsumers;
    const int ct = threadIdx.x, lane = ct & 31, warp = ct >> 5;
    const int group = a.H / a.G;
    const float scale = 1.0f / sqrtf((float)D);
    const uint32_t tag = tag_of(c.epoch, a.layer) ^ (c.stall ? kStallTag : 0u);
    const uint32_t otag = tag_of(c.epoch, a.layer);
    const int s1 = key_start(c, c.b + 1);
    bool bad = false;

    // operands that depend on nothing, staged in shared memory before the wait for the q/k/v rows:
    // cos / sin of every element's frequency at each stream's position, the q / k norm weights
    constexpr int HALF = D / 2;
    const bool half = a.mode == ATTN_TALKER;
    for (int i = ct; i < c.m * D; i += kSConsumers) {
        const int r = i / D, t = i - r * D;
        const int f = half ? (t < HALF ? t : t - HALF) : (t >> 1);
        const size_t row = (size_t)len_of(c, r) * HALF + f;
        sm.rcs[i] = __ldg(a.rope_cos + row);
        sm.rsn[i] = __ldg(a.rope_sin + row);
    }
    for (int t = ct; t < D; t += kSConsumers) {
        sm.qkn[t] = half ? __ldg(a.qn + t) : 1.f;
        sm.qkn[D + t] = half ? __ldg(a.kn + t) : 1.f;
    }
    if (!wait_inputs(wcnt, wtarget, c)) {  // (its barrier also publishes the staged operands)
        consumers_abort(c);
        return kFailed;
    }

    for (int s = key_start(c, c.b); s < s1;) {
        const Seg q = seg_at(c, a.G, s, s1);
        s += q.k1 - q.k0;
        const int r = q.r, g = q.g;
        const float* cs = sm.rcs + r * D;
        const float* sn = sm.rsn + r * D;
        const int pos = len_of(c, r);
        const int newkey = a.mode == ATTN_TALKER ? pos : pos % a.slots;
        const bool seg_new = newkey >= q.k0 && newkey < q.k1;
        const size_t head = ((size_t)r * a.G + g) * a.slots;
        const int ntiles = (q.k1 - q.k0 + TK - 1) / TK;

        // ---- prologue: q heads of the group (warp per head), the new key and value -----------
        const uint64_t* row = a.qkv + (size_t)r * a.ldqkv;
        for (int i = warp; i < group; i += kSConsumerWarps) {
            const int hq = g * group + i;
            float v[PER];
            if (!poll_head<D>(c, row + (size_t)hq * D, tag, lane, v)) {
                bad = true;
                continue;
            }
            if (half) head_rms_pre<D>(v, sm.qkn, a.eps, lane);
            rope_store<D>(half, lane, v, cs, sn, sm.qs + i * D);
        }
        if (seg_new && warp == kSConsumerWarps - 1) {
            const size_t koff = (size_t)a.H * D + (size_t)g * D;             // talker: [q | k | v]
            const size_t voff = koff + (size_t)(a.mode == ATTN_TALKER ? a.G : a.H) * D;
            float k[PER], v[PER];
            if (!poll_head<D>(c, row + koff, tag, lane, k) || !poll_head<D>(c, row + voff, tag, lane, v)) {
                bad = true;
            } else {
                if (half) head_rms_pre<D>(k, sm.qkn + D, a.eps, lane);
                rope_store<D>(half, lane, k, cs, sn, sm.knew);
#pragma unroll
                for (int j = 0; j < PER; ++j) sm.vnew[lane + 32 * j] = v[j];
            }
        }
        if (ct < group) {
            sm.sM[ct] = -CUDART_INF_F;
            sm.sL[ct] = 0.f;
        }
        if (cbar_or(bad)) {
            consumers_abort(c);
            return kFailed;
        }

        float acc[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) acc[u] = 0.f;

        for (int w0 = 0; w0 < ntiles; w0 += WT) {
            const int wt = min(WT, ntiles - w0);
            const int kw0 = q.k0 + w0 * TK;
            const int nwin = min(wt * TK, q.k1 - kw0);
            if (a.mode == ATTN_RING)
                for (int j = ct; j < nwin; j += kSConsumers)
                    sm.stamp[j] = __ldcg(a.pr + (size_t)r * a.slots + kw0 + j);
            for (int t = 0; t < wt; ++t)
                if (!bad && !tile_wait(c, tile + w0 + t)) bad = true;
            const bool win_new = seg_new && newkey >= kw0 && newkey < kw0 + nwin;
            if (win_new && !bad) {
                // the new row goes into the staged tile and is appended to the cache
                const int jn = newkey - kw0;
                float* ks = reinterpret_cast<float*>(slot_ptr(c, tile + w0 + jn / TK)) + (jn % TK) * D;
                for (int t = ct; t < D; t += kSConsumers) {
                    ks[t] = sm.knew[t];
                    ks[TK * D + t] = sm.vnew[t];
                    a.kc[(head + newkey) * D + t] = sm.knew[t];
                    a.vc[(head + newkey) * D + t] = sm.vnew[t];
                }
                if (ct == 0 && a.mode == ATTN_RING) a.pr[(size_t)r * a.slots + newkey] = (uint32_t)pos;
            }
            if (cbar_or(bad)) {
                consumers_abort(c);
                return kFailed;
            }

            // ---- scores: a warp takes 8 keys at a time, lanes split d ----------------------------
            const uint32_t qs_a = smem_u32(sm.qs);
            for (int j0 = warp * 8; j0 < nwin; j0 += kSConsumerWarps * 8) {
                float kv[8][PER];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    if (j < nwin) {
                        const uint32_t ka = slot_addr(c, tile + w0 + j / TK) +
                                            (uint32_t)(((j % TK) * D + lane * PER) * 4);
                        if constexpr (PER == 4) {
                            const float4 t4 = lds_f4(ka);
                            kv[u][0] = t4.x;
                            kv[u][1] = t4.y;
                            kv[u][2] = t4.z;
                            kv[u][3] = t4.w;
                        } else {
                            const float2 t2 = lds_f2(ka);
                            kv[u][0] = t2.x;
                            kv[u][1] = t2.y;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < PER; ++e) kv[u][e] = 0.f;
                    }
                }
                for (int i = 0; i < group; ++i) {
                    float qv[PER];
                    if constexpr (PER == 4) {
                        const float4 t4 = lds_f4(qs_a + (uint32_t)((i * D + lane * PER) * 4));
                        qv[0] = t4.x;
                        qv[1] = t4.y;
                        qv[2] = t4.z;
                        qv[3] = t4.w;
                    } else {
                        const float2 t2 = lds_f2(qs_a + (uint32_t)((i * D + lane * PER) * 4));
                        qv[0] = t2.x;
                        qv[1] = t2.y;
                    }
                    float part[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float acc_s = 0.f;
#pragma unroll
                        for (int e = 0; e < PER; ++e) acc_s += qv[e] * kv[u][e];
                        part[u] = acc_s;
                    }
                    const float sum = butterfly8_keys(part, lane);  // lanes 4u..4u+3: key j0 + u
                    const int u = (lane >> 2) & 7;
                    if ((lane & 3) == 0 && j0 + u < nwin) {
                        bool legal = true;
                        if (a.mode == ATTN_RING) {
                            const int key = kw0 + j0 + u;
                            const uint32_t pj = key == newkey ? (uint32_t)pos : sm.stamp[j0 + u];
                            legal = (pj != 0xFFFFFFFFu) && (pj <= (uint32_t)pos) &&
                                    ((uint32_t)pos - pj < (uint32_t)a.window);
                        }
                        sm.sc[i * kWinKeys + j0 + u] = legal ? sum * scale : -CUDART_INF_F;
                    }
                }
            }
            cbar();

            // ---- running softmax statistics: warp per q head ----------------------------------------
            for (int i = warp; i < group; i += kSConsumerWarps) {
                float mw = -CUDART_INF_F;
                for (int j = lane; j < nwin; j += 32) mw = fmaxf(mw, sm.sc[i * kWinKeys + j]);
                mw = warp_max(mw);
                const float Mold = sm.sM[i];
                const float Mnew = fmaxf(Mold, mw);
                const float alpha = Mold == -CUDART_INF_F ? 0.f : expf(Mold - Mnew);
                float l = 0.f;
                for (int j = lane; j < nwin; j += 32) {
                    const float e = Mnew == -CUDART_INF_F ? 0.f : expf(sm.sc[i * kWinKeys + j] - Mnew);
                    sm.sc[i * kWinKeys + j] = e;
                    l += e;
                }
                l = warp_sum(l);
                if (lane == 0) {
                    sm.sL[i] = sm.sL[i] * alpha + l;
                    sm.sM[i] = Mnew;
                    sm.sA[i] = alpha;
                }
            }
            cbar();

            // ---- o = o alpha + sum_j e_j v_j, ascending keys ------------------------------------------
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int o = ct + kSConsumers * u;
                if (o < group * D) {
                    const int i = o / D, dim = o - i * D;
                    // four independent chains over the keys (j mod 4), summed at the end
                    float av[4] = {acc[u] * sm.sA[i], 0.f, 0.f, 0.f};
                    const uint32_t p_a = smem_u32(sm.sc) + (uint32_t)(i * kWinKeys * 4);
                    for (int tw = 0; tw < wt; ++tw) {
                        const uint32_t vb = slot_addr(c, tile + w0 + tw) + (uint32_t)((TK * D + dim) * 4);
                        const int nk = min(TK, nwin - tw * TK);
                        const uint32_t pt = p_a + (uint32_t)(tw * TK * 4);
                        int j = 0;
                        for (; j + 4 <= nk; j += 4) {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                av[q4] += lds_f(pt + 4u * (j + q4)) * lds_f(vb + (uint32_t)((j + q4) * D * 4));
                        }
                        for (; j < nk; ++j) av[0] += lds_f(pt + 4u * j) * lds_f(vb + (uint32_t)(j * D * 4));
                    }
                    acc[u] = (av[0] + av[1]) + (av[2] + av[3]);
                }
            }
            // the tiles go back to the producer (after the threads' own writes to a tile are
            // ordered before the bulk copies that will overwrite it)
            if (win_new) fence_proxy_async_smem();
            for (int t = 0; t < wt; ++t) tile_release(c, tile + w0 + t);
            cbar();  // the scores are read before the next window overwrites them
        }
        tile += ntiles;

        // ---- the segment's partial for every q head of the group -----------------------------------
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int o = ct + kSConsumers * u;
            if (o < group * D) {
                const int i = o / D, dim = o - i * D;
                const int hq = g * group + i;
                const size_t pi = ((size_t)r * a.H + hq) * c.P + c.b;
                st_word(a.part + pi * D + dim, acc[u], otag);
                if (dim == 0) {
                    st_word(a.ml + 2 * pi, sm.sM[i], otag);
                    st_word(a.ml + 2 * pi + 1, sm.sL[i], otag);
                }
            }
        }
        // ---- arrival: the CTA that completes the pair merges its partials -------------------------
        // The CTAs bf..bl (those with keys) of (r, g) each add 1 with acq_rel after writing their
        // partials (the barrier before orders every thread's stores); the one that brings the count
        // to their number has seen all of them, merges, and sets the count back to zero.
        const int A = g * keys_of(c, r) + (r ? a.G * c.L0 : 0);
        const int bf = key_cta(c, A), bl = key_cta(c, A + keys_of(c, r) - 1);
        cbar();  // the partial stores precede the arrival; sM / sL / qs are free again
        if (ct == 0) {
            int nseg = bl - bf + 1;
            if (c.T < c.P) {  // CTAs without keys wrote nothing
                nseg = 0;
                for (int bb = bf; bb <= bl; ++bb) nseg += key_start(c, bb) < key_start(c, bb + 1);
            }
            unsigned* cnt = a.arr + (size_t)r * a.G + g;
            const unsigned old = atom_add_acq_rel_gpu(cnt, 1u);
            const bool last = old + 1u == (unsigned)nseg;
            if (last) *cnt = 0u;  // (every arrival of this launch has happened)
            sm.flag[0] = last;
        }
        cbar();
        if (sm.flag[0]) {
            constexpr int SL = D / 32;
            for (int u = warp; u < group * SL && !bad; u += kSConsumerWarps) {
                const int i = u / SL, sl = u - i * SL;
                if (!merge_unit<D>(ap, cp, r, g * group + i, sl, bf, bl, tag, otag, lane)) bad = true;
            }
            if (cbar_or(bad)) {
                consumers_abort(c);
                return kFailed;
            }
        }
    }
    return tile;
}

// ==================================================================================================
// consumers: the output rows
// ==================================================================================================
// Talker: out = x / sqrt(mean(x^2) + eps) * w (the final RMSNorm).  Codec: the residual stream,
// or for the FlowLM head LayerNorm(x; w, b) and eos = eos_w . out.  CTA r writes row r.
__device__ float csum(float v, float* nred) {
    const int ct = threadIdx.x;
    v = warp_sum(v);
    if ((ct & 31) == 0) nred[ct >> 5] = v;
    cbar();
    float t = 0.f;
    for (int w = 0; w < kSConsumerWarps; ++w) t += nred[w];
    cbar();
    return t;
}

__device__ __noinline__ bool consume_final(const SFinal* fp, const SCtx* cp, float* out_rows,
                                          float* nred, const unsigned* wcnt, unsigned wtarget) {
    const SFinal f = *fp;
    const SCtx c = *cp;
    if (!wait_inputs(wcnt, wtarget, c)) {
        consumers_abort(c);
        return false;
    }
    const int ct = threadIdx.x;
    const uint32_t tag = tag_of(c.epoch, f.layer) ^ (c.stall ? kStallTag : 0u);
    bool bad = false;
    for (int r = c.b; r < c.m; r += c.P) {
        float x[kFinalPer];
        const uint64_t* src = f.x + (size_t)r * f.h;
        for (int it = 0;; ++it) {
            uint32_t t[kFinalPer];
#pragma unroll
            for (int k = 0; k < kFinalPer; ++k) {
                const int i = ct + kSConsumers * k;
                x[k] = 0.f;
                t[k] = tag;
                if (i < f.h) ld_one(src + i, x[k], t[k]);
            }
            uint32_t diff = 0;
#pragma unroll
            for (int k = 0; k < kFinalPer; ++k) diff |= t[k] ^ tag;
            if (diff == 0) break;
            if (it >= c.polls || *c.abort) {
                bad = true;
                break;
            }
            __nanosleep(64);
        }
        if (cbar_or(bad)) break;
        float* out = out_rows + (size_t)r * f.h;
        float mean = 0.f, inv = 1.f;
        if (f.w && f.b) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < kFinalPer; ++k) s += x[k];
            mean = csum(s, nred) / (float)f.h;
            float v = 0.f;
#pragma unroll
            for (int k = 0; k < kFinalPer; ++k)
                if (ct + kSConsumers * k < f.h) v += (x[k] - mean) * (x[k] - mean);
            inv = 1.0f / sqrtf(csum(v, nred) / (float)f.h + f.eps);
        } else if (f.w) {
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < kFinalPer; ++k) ss += x[k] * x[k];
            inv = 1.0f / sqrtf(csum(ss, nred) / (float)f.h + f.eps);
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < kFinalPer; ++k) {
            const int i = ct + kSConsumers * k;
            if (i < f.h) {
                float o = x[k];
                if (f.w && f.b) o = (x[k] - mean) * inv * f.w[i] + f.b[i];
                else if (f.w) o = x[k] * inv * f.w[i];
                out[i] = o;
                if (f.eos_w) dot += f.eos_w[i] * o;
            }
        }
        if (f.eos_w) {
            dot = csum(dot, nred);
            if (ct == 0) f.eos[r] = dot;
        }
    }
    if (cbar_or(bad)) {
        consumers_abort(c);
        return false;
    }
    return true;
}

template <int DT, int MT>
__device__ __forceinline__ uint32_t gemv_dispatch(const SGemv* g, int nj, const SCtx* c,
                                                  uint32_t tile, float* red, float* nred,
                                                  float* stat, const unsigned* wcnt,
                                                  unsigned wtarget) {
    switch (nj) {
        case 1: return consume_gemv<DT, MT, 1>(g, c, tile, red, nred, stat, wcnt, wtarget);
        case 2: return consume_gemv<DT, MT, 2>(g, c, tile, red, nred, stat, wcnt, wtarget);
        case 3: return consume_gemv<DT, MT, 3>(g, c, tile, red, nred, stat, wcnt, wtarget);
        default: return consume_gemv<DT, MT, 4>(g, c, tile, red, nred, stat, wcnt, wtarget);
    }
}

// ==================================================================================================
// the kernel
// ==================================================================================================
// The phase descriptors reach the consumers through a double buffer in shared memory: the words
// of phase i + 1 are loaded while phase i runs and stored when it ends.
constexpr int kPhaseWords = (int)(sizeof(SPhase) / sizeof(int));
static_assert(sizeof(SPhase) % sizeof(int) == 0 && kPhaseWords <= kSConsumers, "descriptor words");

template <int DT, int MT, int D>
__global__ void __launch_bounds__(kSThreads, 1) k_stream_step(const __grid_constant__ StreamParams sp) {
    using LY = SLayout<MT, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[2 * kSlots];
    __shared__ __align__(16) SPhase s_ph[2];
    __shared__ SCtx s_ctx;
    __shared__ int s_abort, s_skip;
    __shared__ unsigned s_epoch, s_issued;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, b = blockIdx.x;
    if (tid < kSlots) {
        mbar_init(smem_u32(&bars[tid]), 1);                         // full: the producer's arrival
        mbar_init(smem_u32(&bars[kSlots + tid]), kSConsumerWarps);  // empty: one per consumer warp
    }
    if (tid < kPhaseWords) reinterpret_cast<int*>(&s_ph[0])[tid] = reinterpret_cast<const int*>(sp.phases)[tid];
    if (tid == 0) {
        s_abort = 0;
        s_issued = 0;
        s_epoch = *(volatile unsigned*)&sp.st->epoch;
        // the lengths at the step's start (every attention phase splits the same keys)
        const int len0 = __ldcg(sp.len), len1 = sp.m > 1 ? __ldcg(sp.len + 1) : 0;
        int skip = len0 < 0 || len0 >= sp.max_pos || (sp.m > 1 && (len1 < 0 || len1 >= sp.max_pos));
        if (skip && b == 0) flag_check(sp.status, CHECK_BOUNDS);
        s_skip = skip;
        int attn_mode = -1, attn_G = 1, attn_slots = 1;
        for (int i = 0; i < sp.n_phases; ++i)
            if (sp.phases[i].type == SP_ATTN) {
                attn_mode = sp.phases[i].a.mode;
                attn_G = sp.phases[i].a.G;
                attn_slots = sp.phases[i].a.slots;
                break;
            }
        SCtx c;
        c.b = b;
        c.P = P;
        c.m = sp.m;
        c.ring = reinterpret_cast<char*>(smem + LY::kRing);
        c.full0 = smem_u32(&bars[0]);
        c.empty0 = smem_u32(&bars[kSlots]);
        c.epoch = s_epoch;
        c.x_in = sp.x_in;
        c.polls = sp.wait_polls > 0 ? sp.wait_polls : kDefaultPolls;
        c.abort = &s_abort;
        c.status = sp.status;
        c.stall = false;
        c.len0 = len0;
        c.len1 = len1;
        c.L0 = attn_mode == ATTN_RING ? attn_slots : len0 + 1;
        c.L1 = sp.m > 1 ? (attn_mode == ATTN_RING ? attn_slots : len1 + 1) : 0;
        c.T = attn_G * (c.L0 + c.L1);
        s_ctx = c;
    }
    __syncthreads();

    if (!s_skip) {
        if (warp == kSConsumerWarps) {
            // ---- the producer ----------------------------------------------------------------------
            if (lane == 0) s_issued = run_producer<DT, D>(sp.phases, sp.n_phases, &s_ctx);
        } else {
            // ---- the consumers ---------------------------------------------------------------------
            float* red = reinterpret_cast<float*>(smem + LY::kRed);
            float* nred = reinterpret_cast<float*>(smem + LY::kNred);
            float* stat = reinterpret_cast<float*>(smem + LY::kStat);
            __shared__ AttnSmem<D> s_as;  // written by thread 0; the loop's first barrier orders it
            if (tid == 0) {
                AttnSmem<D>& as = s_as;
                as.qs = reinterpret_cast<float*>(smem + LY::kQs);
                as.sc = reinterpret_cast<float*>(smem + LY::kSc);
                as.knew = reinterpret_cast<float*>(smem + LY::kKnew);
                as.vnew = reinterpret_cast<float*>(smem + LY::kVnew);
                as.sM = reinterpret_cast<float*>(smem + LY::kSM);
                as.sL = reinterpret_cast<float*>(smem + LY::kSL);
                as.sA = reinterpret_cast<float*>(smem + LY::kSA);
                as.stamp = reinterpret_cast<uint32_t*>(smem + LY::kStamp);
                as.flag = reinterpret_cast<int*>(smem + LY::kFlag);
                as.rcs = reinterpret_cast<float*>(smem + LY::kRope);
                as.rsn = as.rcs + 2 * D;
                as.qkn = reinterpret_cast<float*>(smem + LY::kQKn);
            }
            uint32_t tile = 0;
            int done = 0;  // phases this CTA has completed (and counted)
            for (int i = 0; i < sp.n_phases; ++i) {
                const SPhase* ph = &s_ph[i & 1];
                // the next descriptor's words, in flight while this phase runs
                int next = 0;
                if (i + 1 < sp.n_phases && tid < kPhaseWords)
                    next = __ldg(reinterpret_cast<const int*>(sp.phases + i + 1) + tid);
                if (tid == 0) s_ctx.stall = i == sp.stall_phase;
                cbar();  // (the stall flag and this phase's descriptor are in place)
                // the phase waits for the counter of the phase before: every CTA has written it
                const unsigned* wcnt = i > 0 ? sp.cnt + i - 1 : nullptr;
                const unsigned wtarget = (s_epoch + 1u) * (unsigned)P;
                bool ok = true;
                switch (ph->type) {
                    case SP_GEMV:
                        tile = gemv_dispatch<DT, MT>(&ph->g, ph->nj, &s_ctx, tile, red, nred, stat,
                                                     wcnt, wtarget);
                        ok = tile != kFailed;
                        break;
                    case SP_ATTN:
                        tile = consume_attn<D>(&ph->a, &s_ctx, tile, &s_as, wcnt, wtarget);
                        ok = tile != kFailed;
                        break;
                    default: ok = consume_final(&ph->f, &s_ctx, sp.out, nred, wcnt, wtarget); break;
                }
                if (!ok) break;  // (every consumer: the phase functions fail together)
                // every consumer's stores of the phase precede the phase function's last barrier
                if (tid == 0) red_release_add_gpu(sp.cnt + i, 1u);
                done = i + 1;
                if (i + 1 < sp.n_phases && tid < kPhaseWords)
                    reinterpret_cast<int*>(&s_ph[(i + 1) & 1])[tid] = next;
            }
            // A CTA that stopped early still counts the phases it did not complete, so that every
            // counter ends the launch at (epoch + 1) * grid and the next launch's waits hold;
            // CTAs still waiting on them go on (on undefined data) instead of running out too.
            if (tid == 0)
                for (int j = done; j < sp.n_phases; ++j) red_release_add_gpu(sp.cnt + j, 1u);
        }
    } else if (tid == 0) {
        for (int j = 0; j < sp.n_phases; ++j) red_release_add_gpu(sp.cnt + j, 1u);
    }
    __syncthreads();

    if (tid == 0) {
        // copies still in flight land before the CTA leaves (the last kSlots tiles issued)
        const uint32_t n = s_issued;
        for (uint32_t t = n > (uint32_t)kSlots ? n - kSlots : 0u; t < n; ++t)
            mbar_wait_bounded(smem_u32(&bars[t % kSlots]), (t / kSlots) & 1u);
        // the last CTA to leave advances the launch count and the stream lengths: every CTA has
        // read both by the time it arrives here
        if (atom_add_acq_rel_gpu(&sp.st->exit_count, 1u) == (unsigned)P - 1u) {
            sp.st->exit_count = 0u;
            sp.st->epoch = s_epoch + 1u;
            sp.len[0] = s_ctx.len0 + 1;
            if (sp.m > 1) sp.len[1] = s_ctx.len1 + 1;
        }
    }
}

template <int DT, int MT, int D>
constexpr size_t stream_smem() {
    return (size_t)SLayout<MT, D>::kBytes;
}

template <int DT, int MT, int D>
int stream_grid_t(int num_sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_stream_step<DT, MT, D>, kSThreads,
                                                      stream_smem<DT, MT, D>()) != cudaSuccess)
        return 0;
    return per_sm >= 1 ? num_sms : 0;
}

template <int DT, int MT, int D>
cudaError_t configure_t() {
    return cudaFuncSetAttribute(k_stream_step<DT, MT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)stream_smem<DT, MT, D>());
}

template <int DT, int MT, int D>
cudaError_t launch_t(const StreamParams& sp, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = stream_smem<DT, MT, D>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_stream_step<DT, MT, D>, sp);
}

}  // namespace

#define STREAM_DISPATCH(FN, ...)                                                                  \
    do {                                                                                          \
        if (dtype == 1) {                                                                         \
            if (m <= 1) return d == 64 ? FN<1, 1, 64>(__VA_ARGS__) : FN<1, 1, 128>(__VA_ARGS__);  \
            return d == 64 ? FN<1, 2, 64>(__VA_ARGS__) : FN<1, 2, 128>(__VA_ARGS__);              \
        }                                                                                         \
        if (m <= 1) return d == 64 ? FN<0, 1, 64>(__VA_ARGS__) : FN<0, 1, 128>(__VA_ARGS__);      \
        return d == 64 ? FN<0, 2, 64>(__VA_ARGS__) : FN<0, 2, 128>(__VA_ARGS__);                  \
    } while (0)

int stream_grid(int dtype, int m, int d, int num_sms) {
    if (m < 1 || m > 2 || (d != 64 && d != 128)) return 0;
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return 0;
    STREAM_DISPATCH(stream_grid_t, num_sms);
}

bool stream_gemv_ok(int dtype, int K) {
    const int es = dtype == 1 ? 2 : 4, vec = dtype == 1 ? 8 : 4;
    if (K < vec || K % vec) return false;
    const int granules = K / vec;
    return (size_t)K * es <= (size_t)kSlotBytes && granules <= 4 * kSConsumers;
}

cudaError_t stream_configure() {
    cudaError_t e;
    if ((e = configure_t<0, 1, 64>()) != cudaSuccess || (e = configure_t<0, 1, 128>()) != cudaSuccess ||
        (e = configure_t<0, 2, 64>()) != cudaSuccess || (e = configure_t<0, 2, 128>()) != cudaSuccess ||
        (e = configure_t<1, 1, 64>()) != cudaSuccess || (e = configure_t<1, 1, 128>()) != cudaSuccess ||
        (e = configure_t<1, 2, 64>()) != cudaSuccess || (e = configure_t<1, 2, 128>()) != cudaSuccess)
        return e;
    return cudaSuccess;
}

cudaError_t launch_stream_step(const StreamParams& sp, int dtype, int m, int d, int grid,
                               cudaStream_t s) {
    if (m < 1 || m > 2 || (d != 64 && d != 128) || grid < 1) return cudaErrorInvalidValue;
    STREAM_DISPATCH(launch_t, sp, grid, s);
}

}  // namespace dec
