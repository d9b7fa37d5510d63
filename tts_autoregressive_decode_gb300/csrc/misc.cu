// misc.cu -- the step's last kernel and the state-management kernels (sm_103a).
#include "common.cuh"
#include "final_row.cuh"
#include "kernels.h"

namespace dec {

// The step's last kernel: the output row of each stream (final_row.cuh), one CTA per stream.  It
// also advances that stream's length, which no other kernel of the step reads after this one has
// passed griddepcontrol.wait.
__global__ void __launch_bounds__(256) k_final(const FinalParams p) {
    __shared__ float red[8];
    const int r = blockIdx.x, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    final_row(p, r, red);
    if (tid == 0) {
        if (p.advance_stream < 0)
            p.len[r] += 1;
        else if (r == 0)
            p.len[p.advance_stream] += p.m;
    }
}

cudaError_t launch_final(const FinalParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.m);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_final, p);
}

// Copy a prefilled position-major [layers][n][G][d] K/V block into the head-major cache of one
// stream ([layers][streams][G][slots][d]); codec: stamp slots 0..n-1 with their positions.
__global__ void k_prefill(const PrefillParams p) {
    const size_t per_layer = (size_t)p.n * p.G * p.d;
    const size_t total = (size_t)p.layers * per_layer;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int l = (int)(i / per_layer);
        size_t rem = i - (size_t)l * per_layer;
        const int pos = (int)(rem / ((size_t)p.G * p.d));
        rem -= (size_t)pos * p.G * p.d;
        const int g = (int)(rem / p.d);
        const int t = (int)(rem - (size_t)g * p.d);
        const size_t dst =
            ((((size_t)l * p.streams + p.stream) * p.G + g) * p.slots + pos) * p.d + t;
        p.kc[dst] = p.k_src[i];
        p.vc[dst] = p.v_src[i];
    }
    if (p.pr) {
        const size_t ns = (size_t)p.layers * p.slots;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < ns;
             i += (size_t)gridDim.x * blockDim.x) {
            const int l = (int)(i / p.slots), j = (int)(i - (size_t)l * p.slots);
            p.pr[((size_t)l * p.streams + p.stream) * p.slots + j] =
                j < p.n ? (uint32_t)j : 0xFFFFFFFFu;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) p.len[p.stream] = p.n;
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s) {
    const size_t total = (size_t)p.layers * p.n * p.G * p.d;
    int grid = (int)((total + 255) / 256);
    if (grid > 4096) grid = 4096;
    if (grid < 1) grid = 1;
    k_prefill<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// Every stamp of one stream back to empty, its length to 0 (the K/V bytes are cleared with
// cudaMemsetAsync by the caller).
__global__ void k_reset_stamps(const ResetParams p) {
    if (p.pr) {
        const size_t ns = (size_t)p.layers * p.slots;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < ns;
             i += (size_t)gridDim.x * blockDim.x) {
            const int l = (int)(i / p.slots), j = (int)(i - (size_t)l * p.slots);
            p.pr[((size_t)l * p.streams + p.stream) * p.slots + j] = 0xFFFFFFFFu;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) p.len[p.stream] = 0;
}

cudaError_t launch_reset_stamps(const ResetParams& p, cudaStream_t s) {
    k_reset_stamps<<<64, 256, 0, s>>>(p);
    return cudaGetLastError();
}

__global__ void k_set_len(int32_t* len, int stream, int value) { len[stream] = value; }

cudaError_t launch_set_len(int32_t* len, int stream, int value, cudaStream_t s) {
    k_set_len<<<1, 1, 0, s>>>(len, stream, value);
    return cudaGetLastError();
}

}  // namespace dec
