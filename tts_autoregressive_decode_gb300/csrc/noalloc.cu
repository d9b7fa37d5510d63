// noalloc.cu -- dec_attention_noalloc: the stateless split-K decode attention with its scratch
// in a fixed, library-owned device array, for callers that must not allocate device memory.
//
// dec_attention needs scratch for its per-chunk partial results and merge tickets, which the
// caller allocates.  Some callers cannot: code on a real-time audio thread, where cudaMalloc and
// cudaFree may synchronize the device and take unbounded time, and code embedded in a host
// application whose own allocator owns the whole device-memory budget.  For them this file holds
// the scratch in a file-scope __device__ array of kNoallocScratchBytes, which every GPU that
// loads the library keeps until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/dec.h"
#include "kernels.h"

namespace dec {
dec_status stateless_fail(dec_status st, const char* msg);  // dec_api.cu: sets dec_last_error(NULL)
}

using namespace dec;

namespace {

constexpr size_t kNoallocScratchBytes = 4u << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on each device.  In host code the array's name is only a
// host-side stand-in, so the address is looked up once per device, with that device current.
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

extern "C" dec_status dec_attention_noalloc(int m, int q_heads, int kv_heads, int head_dim,
                                            int capacity, const float* q, const float* k,
                                            const float* v, const int32_t* lens, float* out,
                                            void* stream) {
    if (!q || !k || !v || !lens || !out) return stateless_fail(DEC_E_ARG, "NULL pointer");
    if (m < 1 || m > 64 || capacity < 1 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads)
        return stateless_fail(DEC_E_ARG, "bad m, capacity or head counts");
    if (capacity > kMaxSlots) return stateless_fail(DEC_E_UNSUPPORTED, "capacity above 32768");
    if (head_dim != 64 && head_dim != 128)
        return stateless_fail(DEC_E_UNSUPPORTED, "head_dim 64 or 128");
    if (q_heads / kv_heads > kMaxGroup) return stateless_fail(DEC_E_UNSUPPORTED, "GQA group above 8");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
        return stateless_fail(DEC_E_UNSUPPORTED, "k and v must be 16-byte aligned");

    // the same scratch layout dec_attention uses: partial outputs, partial (max, sum), tickets
    const int mc = (capacity + kAttnChunk - 1) / kAttnChunk;
    const size_t part_bytes = align_up(attention_part_bytes(m, q_heads, mc, head_dim));
    const size_t ml_bytes = align_up(attention_ml_bytes(m, q_heads, mc));
    const size_t ticket_bytes = (size_t)m * kv_heads * sizeof(unsigned);
    const size_t need = part_bytes + ml_bytes + align_up(ticket_bytes);
    if (need > kNoallocScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof msg, "needs %zu bytes of scratch; the static scratch holds %zu",
                 need, kNoallocScratchBytes);
        return stateless_fail(DEC_E_UNSUPPORTED, msg);
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return stateless_fail(DEC_E_CUDA, "no usable current CUDA device");
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            // first call on this device: find the array's device address (must not happen while
            // a stream is being captured)
            void* ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr) {
                char msg[160];
                snprintf(msg, sizeof msg, "scratch address lookup: %s", cudaGetErrorString(e));
                return stateless_fail(DEC_E_CUDA, msg);
            }
            g_scratch_ptr[dev] = ptr;
        }
        base = g_scratch_ptr[dev];
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return stateless_fail(DEC_E_CUDA, "no CUDA device");
    cudaError_t e = configure_kernels();
    if (e != cudaSuccess) return stateless_fail(DEC_E_CUDA, "kernel attributes");

    char* ws = static_cast<char*>(base);
    unsigned* tickets = reinterpret_cast<unsigned*>(ws + part_bytes + ml_bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the merge tickets must start at zero; the array keeps whatever the last call left
    e = cudaMemsetAsync(tickets, 0, ticket_bytes, s);
    if (e != cudaSuccess) return stateless_fail(DEC_E_CUDA, "ticket clear");

    AttnParams a = {};
    a.mode = ATTN_PLAIN;
    a.m = m;
    a.H = q_heads;
    a.G = kv_heads;
    a.d = head_dim;
    a.slots = capacity;
    a.qkv = q;
    a.kc = const_cast<float*>(k);
    a.vc = const_cast<float*>(v);
    a.len = lens;
    a.max_pos = capacity;
    a.part = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float*>(ws + part_bytes);
    a.tickets = tickets;
    a.max_chunks = mc;
    a.out = out;
    e = launch_attention(a, s, false);
    if (e != cudaSuccess) return stateless_fail(DEC_E_CUDA, "attention launch");
    return DEC_OK;
}
