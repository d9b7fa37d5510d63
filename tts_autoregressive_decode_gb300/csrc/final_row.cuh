// final_row.cuh -- the step's output row, shared by k_final (misc.cu) and the persistent step
// kernel (step.cu).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dec {

// Talker: out = x / sqrt(mean(x^2) + eps) * w (the final RMSNorm, RMSNORM_SRC).  Codec: the
// residual stream is the output (Pocket TTS on wgpu: the codec transformer has no final norm),
// or for the FlowLM backbone out = LayerNorm(x; w, b) (mean, then the biased variance of the
// deviations; out_norm) and, with an EOS row, eos = eos_w . out (out_eos, its bias added on
// read-back).  Row r of the residual stream, by the 256 threads of one CTA; red: 8 floats of
// shared memory.  The residual stream is read with ld.global.cg (other CTAs of the same launch
// may have written it).
__device__ __forceinline__ float final_block_sum(float v, float* red) {
    const int tid = threadIdx.x;
    v = warp_sum(v);
    __syncthreads();  // red may still be read by a previous sum
    if ((tid & 31) == 0) red[tid >> 5] = v;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += red[w];
    return tot;
}

__device__ __forceinline__ void final_row(const FinalParams& p, int r, float* red) {
    const int tid = threadIdx.x;
    const float* x = p.x + (size_t)r * p.h;
    float* out = p.out + (size_t)r * p.h;
    float dot = 0.f;
    if (p.w && p.b) {
        float s = 0.f;
        for (int i = tid; i < p.h; i += 256) s += __ldcg(x + i);
        const float mean = final_block_sum(s, red) / (float)p.h;
        float v = 0.f;
        for (int i = tid; i < p.h; i += 256) {
            const float dv = __ldcg(x + i) - mean;
            v += dv * dv;
        }
        const float inv = 1.0f / sqrtf(final_block_sum(v, red) / (float)p.h + p.eps);
        for (int i = tid; i < p.h; i += 256) {
            const float o = (__ldcg(x + i) - mean) * inv * p.w[i] + p.b[i];
            out[i] = o;
            if (p.eos_w) dot += p.eos_w[i] * o;
        }
    } else if (p.w) {
        float ss = 0.f;
        for (int i = tid; i < p.h; i += 256) {
            const float v = __ldcg(x + i);
            ss += v * v;
        }
        const float inv = 1.0f / sqrtf(final_block_sum(ss, red) / (float)p.h + p.eps);
        for (int i = tid; i < p.h; i += 256) {
            const float o = __ldcg(x + i) * inv * p.w[i];
            out[i] = o;
            if (p.eos_w) dot += p.eos_w[i] * o;
        }
    } else {
        for (int i = tid; i < p.h; i += 256) {
            const float o = __ldcg(x + i);
            out[i] = o;
            if (p.eos_w) dot += p.eos_w[i] * o;
        }
    }
    if (p.eos_w) {
        dot = final_block_sum(dot, red);
        if (tid == 0) p.eos[r] = dot;
    }
}

}  // namespace dec
