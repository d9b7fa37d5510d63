// final_row.cuh -- the step's output row, shared by k_final (misc.cu) and the persistent step
// kernel (step.cu).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dec {

// Talker: out = x / sqrt(mean(x^2) + eps) * w (the final RMSNorm, RMSNORM_SRC); codec: the
// residual stream is the output (Pocket TTS on wgpu: the codec transformer has no final norm).
// Row r of the residual stream, by the 256 threads of one CTA; red: 8 floats of shared memory.
// The residual stream is read with ld.global.cg (other CTAs of the same launch may have written it).
__device__ __forceinline__ void final_row(const FinalParams& p, int r, float* red) {
    const int tid = threadIdx.x;
    const float* x = p.x + (size_t)r * p.h;
    float* out = p.out + (size_t)r * p.h;
    if (p.w) {
        float ss = 0.f;
        for (int i = tid; i < p.h; i += 256) {
            const float v = __ldcg(x + i);
            ss += v * v;
        }
        ss = warp_sum(ss);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int w = 0; w < 8; ++w) tot += red[w];
        const float inv = 1.0f / sqrtf(tot / (float)p.h + p.eps);
        for (int i = tid; i < p.h; i += 256) out[i] = __ldcg(x + i) * inv * p.w[i];
    } else {
        for (int i = tid; i < p.h; i += 256) out[i] = __ldcg(x + i);
    }
}

}  // namespace dec
