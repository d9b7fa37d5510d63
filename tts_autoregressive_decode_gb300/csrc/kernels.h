// kernels.h -- parameter blocks and launchers of the decode kernels (internal to the library).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dec {

// device check word bits (read back by dec_sync / dec_step_host)
enum : unsigned {
    CHECK_WAIT_LIMIT = 1u,   // an mbarrier wait exceeded its iteration bound
    CHECK_BOUNDS = 2u,       // a position / slot index failed its range check
};

// ---------------------------------------------------------------------------------------------
// GEMV: y[r][n] = sum_k W[n][k] * xin[r][k], W row-major [N][K], each weight read once for all
// rows.  An optional norm prologue builds xin from x; an epilogue consumes the row sums.
// ---------------------------------------------------------------------------------------------
enum Prologue : int {
    PRO_NONE = 0,
    PRO_RMS = 1,
    PRO_LN = 2,
    PRO_LN_MOD = 3,  // LayerNorm (affine when nw / nb are set), then DiT's modulate:
                     // xin = n * (1 + mod[K + k]) + mod[k]   (shift at mod[0..K), scale after)
};
enum Epilogue : int {
    EPI_STORE = 0,   // y[r][n] = v
    EPI_RESID = 1,   // y[r][n] = res[r][n] + (ls ? ls[n] * v : v)   (o-proj / down / MV_LS)
    EPI_SWIGLU = 2,  // rows interleaved (gate j, up j): y[r][j] = silu(v_2j) * v_2j+1
    EPI_GELU = 3,    // y[r][n] = 0.5 v (1 + erf(v / sqrt 2))
};
// Before any epilogue, v += bias[n] when bias is set; EPI_STORE then applies SiLU when act == 1.

struct GemvParams {
    const void* W;
    int N, K;
    int m;                 // active rows
    const float* x;        // [m][ldx]
    int ldx;
    int pro;               // Prologue
    const float* nw;       // norm weight [K]
    const float* nb;       // LayerNorm bias [K]
    float eps;
    int epi;               // Epilogue
    float* y;              // [m][ldy]
    int ldy;
    const float* res;      // residual input [m][ldres] (may alias y)
    int ldres;
    const float* ls;       // LayerScale [N] or null
    float* tap;            // optional copy of y rows [m][ldtap] (EPI_RESID)
    int ldtap;
    unsigned* status;      // device check word (bounded waits), may be null
    int unit;              // rows per partition unit (2 for SwiGLU pairs)
    int per_sm;            // split-K GEMV launch: CTAs per SM (0: 2).  One CTA per SM leaves room
                           // for the next kernel's CTAs to start and stage their loads early
    const float* bias;     // [N] or null (split-K GEMV, m <= 2, only)
    int act;               // EPI_STORE: 1 = SiLU
    const float* mod;      // PRO_LN_MOD: [2K] shift then scale
    // tensor-core GEMV (3..8 rows, bf16 weights): the matrix's TMA descriptor (host memory,
    // 128 bytes, copied into the launch's parameters; null: not served), partial sums of tiles
    // split over CTAs and one ticket per 128-row tile (zero between launches)
    const void* tmap;
    float* mpart;
    size_t mpart_floats;
    unsigned* mtick;
    int mtick_n;
    int tc_stages, tc_cols, tc_band, tc_acc, tc_cb, tc_contrib;  // set by the launch
};

// dtype: 0 f32, 1 bf16.  Launches with the programmatic-dependency attribute when pdl.
// gemv_configure() must have run on the current device first (see configure_kernels).
constexpr int kGemvMaxSmem = 200 * 1024;
cudaError_t launch_gemv(const GemvParams& p, int dtype, int num_sms, cudaStream_t s, bool pdl);
cudaError_t gemv_configure();
size_t gemv_smem_bytes(int m, int K);
// the tensor-core GEMV: whether it serves this launch (bf16 weights with a TMA descriptor, 3..8
// rows), its launch, and the descriptor of a row-major [N][K] bf16 matrix (128 bytes to out)
bool gemv_tc_ok(const GemvParams& p, int num_sms);
cudaError_t launch_gemv_tc(GemvParams p, int num_sms, cudaStream_t s, bool pdl);
cudaError_t gemv_tc_configure();
cudaError_t gemv_tc_encode(const void* W, int N, int K, void* out);
const void* gemv_tc_kernel();  // the kernel's entry (graph nodes that launch it take two arguments)
constexpr int kTmapBytes = 128;
struct alignas(64) TmapBytes {  // one TMA descriptor, as the driver encodes it
    unsigned char b[kTmapBytes];
};

// ---------------------------------------------------------------------------------------------
// Split-K decode attention with the step's prologue fused in front of it.
// ---------------------------------------------------------------------------------------------
enum AttnMode : int {
    ATTN_PLAIN = 0,   // q given; keys 0..lens[r]-1 of the cache; nothing appended
    ATTN_TALKER = 1,  // raw qkv: per-head q/k RMSNorm, rotate_half rope, append K/V at pos
    ATTN_RING = 2,    // raw qkv: interleaved rope, push K/V into slot pos % ring, stamp it;
                      // keys legal by stamp and window
    ATTN_PREFILL = 3, // a block of rows of ONE stream (`stream`) at positions len[stream] + r:
                      // raw qkv, q as ATTN_TALKER, keys 0..len[stream] + r (the block's K/V
                      // rows already appended by k_prefill_append); nothing appended here
};

constexpr int kAttnChunk = 64;   // keys per CTA
constexpr int kMaxGroup = 8;     // q heads per kv head handled by one CTA
constexpr int kMaxSlots = 32768; // cache rows per (stream, kv head): bounds the merge's staging

struct AttnParams {
    int mode;
    int m;                 // rows (streams; ATTN_PREFILL: rows of the block)
    int stream;            // ATTN_PREFILL: the stream whose cache and length the rows use
    int H, G, d;           // q heads, kv heads, head_dim
    int slots;             // cache rows per (stream, kv head): capacity or ring
    int window;            // ring: attention window
    const float* qkv;      // TALKER/RING: raw [m][ldqkv] = [q | k | v]; PLAIN: q [m][H][d]
    int ldqkv;
    float* kc;             // K cache [m][G][slots][d] (this layer)
    float* vc;             // V cache
    uint32_t* pr;          // RING: position stamps [m][slots]
    const int32_t* len;    // TALKER/RING: [m] current lengths = positions; PLAIN: keys
    const float* qn;       // TALKER: q norm weight [d]
    const float* kn;       // TALKER: k norm weight [d]
    float eps;
    const float* rope_cos; // [max_pos][d/2]
    const float* rope_sin;
    int max_pos;
    // TALKER/PREFILL, optional multimodal rope: the rows' rotary positions [rows][3] (t, h, w),
    // each in 0..max_pos-1; rope frequency f turns by the position of axis rope_axis[f] (0..2).
    // Null: every frequency turns by the row's cache position.
    const int32_t* rope_pos;
    const int32_t* rope_axis;  // [d/2]
    // 1: two chunks per CTA (k_attention_pair), for grids that then fit one wave at one CTA per
    // SM; the chunks are computed exactly as by k_attention.  Not with tickets.
    int paired;
    float* part;           // [m][H][max_chunks][d] partial outputs
    float* part_ml;        // [m][H][max_chunks][2] partial (max, sum)
    unsigned* tickets;     // [m][G] merge tickets, zero between calls; null: no in-kernel merge
    int max_chunks;
    float* out;            // [m][H*d]
    unsigned* status;
};

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl);
// CTAs of k_attention_pair's grid for these parameters
int attention_pair_ctas(const AttnParams& p);
cudaError_t attention_configure();
// Merge of k_attention's chunk partials (launch after k_attention with tickets == nullptr).
cudaError_t launch_attention_merge(const AttnParams& p, cudaStream_t s, bool pdl);
// ATTN_PREFILL blocks: q/k norm of the block's keys, rope, append to the cache of p.stream at
// positions len[stream] + r (r < p.m); launch before the attention.
cudaError_t launch_prefill_append(const AttnParams& p, cudaStream_t s, bool pdl);
size_t attention_smem_bytes(int d, int group);
// scratch sizes (bytes) for the partials and tickets
size_t attention_part_bytes(int m, int H, int max_chunks, int d);
size_t attention_ml_bytes(int m, int H, int max_chunks);

// ---------------------------------------------------------------------------------------------
// Small kernels: final norm / copy-out + length advance, prefill copy-in, stream reset.
// ---------------------------------------------------------------------------------------------
struct FinalParams {
    int m, h;
    const float* x;        // residual stream [m][h]
    const float* w;        // final norm weight [h]: RMSNorm, or LayerNorm with b; null = copy
    const float* b;        // LayerNorm bias [h] (codec head), or null
    const float* eos_w;    // EOS row [h] (codec head), or null
    float* eos;            // [m] eos_w . out, when eos_w
    float eps;
    float* out;            // [m][h]
    int32_t* len;          // [m]: incremented (row r advances stream r) ...
    int advance_stream;    // ... unless >= 0: a prefill block, which advances this stream by m
};
cudaError_t launch_final(const FinalParams& p, cudaStream_t s, bool pdl);

// ---------------------------------------------------------------------------------------------
// Streamed step kernel (m <= 2 rows): the whole step as one persistent cooperative launch, one
// CTA per SM.  Per CTA a producer warp streams the CTA's share of every phase's weights and K/V
// rows through a shared-memory ring by bulk copies, running ahead across phase boundaries; the
// consumer warps compute each phase once its input activations are there.  Activations travel
// between CTAs as tagged words: the low half is the f32 value, the high half the tag of the
// (launch, layer) that wrote it, so waiting for an input and reading it are one load.
// ---------------------------------------------------------------------------------------------
enum StreamPhaseType : int { SP_GEMV = 0, SP_ATTN = 1, SP_FINAL = 3 };

struct SGemv {
    const void* W;
    int N, K;
    int unit;               // rows per partition unit (2: SwiGLU gate/up pairs)
    int pro;                // PRO_NONE / PRO_RMS / PRO_LN
    const float* nw;        // norm weight [K]
    const float* nb;        // LayerNorm bias [K]
    float eps;
    int epi;                // EPI_STORE / EPI_RESID / EPI_SWIGLU / EPI_GELU
    const float* ls;        // LayerScale [N] or null (EPI_RESID)
    const uint64_t* x;      // tagged input [m][ldx] written at layer x_layer; null: the step input
    int ldx, x_layer;
    const uint64_t* res;    // tagged residual [m][ldres] at layer res_layer; null: the step input
    int ldres, res_layer;
    uint64_t* y;            // tagged output [m][ldy], written with tag `layer`
    int ldy, layer;
    float* tap;             // optional plain copy of the EPI_RESID output [m][ldtap]
    int ldtap;
};

struct SAttn {
    int mode;               // ATTN_TALKER or ATTN_RING
    int H, G;
    int slots, window;
    int layer;              // tag of the q/k/v rows read and of the partials written
    const uint64_t* qkv;    // tagged raw [m][ldqkv] = [q | k | v]
    int ldqkv;
    float* kc;              // K cache [m][G][slots][d] (this layer)
    float* vc;
    uint32_t* pr;           // RING: position stamps [m][slots]
    const float* qn;        // TALKER: q / k norm weights [d]
    const float* kn;
    float eps;
    const float* rope_cos;  // [max_pos][d/2]
    const float* rope_sin;
    uint64_t* part;         // tagged partial outputs [m][H][grid][d]
    uint64_t* ml;           // tagged partial (max, sum) [m][H][grid][2]
    uint64_t* out;          // tagged attention output [m][H * d] (merged partials)
    unsigned* arr;          // [m][G] arrival counts of this layer's (stream, kv head) pairs,
                            // zero between launches
};

struct SFinal {
    const uint64_t* x;      // tagged residual stream [m][h] of layer `layer`
    int layer, h;
    const float* w;         // RMSNorm weight (talker), LayerNorm weight (codec head), or null
    const float* b;         // LayerNorm bias (codec head) or null
    const float* eos_w;     // EOS row [h] or null
    float* eos;             // [m]
    float eps;
};

struct SPhase {
    int type;               // StreamPhaseType
    int nj;                 // SP_GEMV: 16-byte granules of a row per consumer thread (1..4)
    SGemv g;
    SAttn a;
    SFinal f;
};

// Per-plan device state: `epoch` counts the plan's launches (tags are (epoch + 1) << 8 | layer),
// `exit_count` the CTAs that have finished the current launch.
struct StreamState {
    unsigned epoch;
    unsigned exit_count;
};

struct StreamParams {
    const SPhase* phases;   // device array
    int n_phases;
    int m;                  // rows (streams 0..m-1)
    const float* x_in;      // the step's input rows [m][hidden]
    float* out;             // the step's output rows [m][hidden]
    int32_t* len;           // [m] stream lengths: read at the start, advanced at the end
    int max_pos;            // rows of the rope tables
    StreamState* st;
    unsigned* cnt;          // [n_phases] completion counters: each CTA adds 1 when its part of the
                            // phase is written; phase i + 1 starts once cnt[i] = (epoch + 1) * grid
    unsigned* status;       // device check word
    int wait_polls;         // bound on the polls of one wait (0: the default bound)
    int stall_phase;        // -1; else the consumers of this phase wait for a tag that no CTA
                            // writes, so the wait runs out (tests of the bounded waits)
};

// Layers the tag scheme takes.
constexpr int kStreamMaxLayers = 255;
// CTAs of the streamed kernel on this device (one per SM; 0 when it cannot be launched).
int stream_grid(int dtype, int m, int d, int num_sms);
cudaError_t stream_configure();
// Whether a GEMV of K columns fits the kernel (a row within one ring slot, at most 4 granules
// per consumer thread).
bool stream_gemv_ok(int dtype, int K);
cudaError_t launch_stream_step(const StreamParams& sp, int dtype, int m, int d, int grid,
                               cudaStream_t s);

struct PrefillParams {
    int layers, n, G, d, slots, streams, stream;
    const float* k_src;    // [layers][n][G][d]
    const float* v_src;
    float* kc;             // [layers][streams][G][slots][d]
    float* vc;
    uint32_t* pr;          // codec: [layers][streams][slots] or null
    int32_t* len;          // [streams]
};
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s);

struct ResetParams {
    int layers, streams, stream, slots;
    uint32_t* pr;          // codec stamps or null
    int32_t* len;
};
cudaError_t launch_reset_stamps(const ResetParams& p, cudaStream_t s);
// len[stream] = value (the value travels as a kernel argument, so the host may reuse it at once)
cudaError_t launch_set_len(int32_t* len, int stream, int value, cudaStream_t s);

// Set the kernels' shared-memory limits on the current device (once per device; safe to call
// from several threads).  Must run before a kernel is launched or captured on that device.
cudaError_t configure_kernels();

}  // namespace dec
