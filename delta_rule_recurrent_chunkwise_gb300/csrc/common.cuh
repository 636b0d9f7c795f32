// common.cuh -- device helpers shared by the linear-attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

// ---------------------------------------------------------------- I/O types
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// --------------------------------------------------------------- prologue
// beta = sigmoid(x): the write strength of the delta rule.
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// log alpha = -softplus(x) = -(max(x, 0) + log1p(exp(-|x|))): the per-key-
// channel log decay, written so that it neither overflows nor loses digits.
__device__ __forceinline__ float log_decay_f(float x) {
    return -(fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))));
}

// alpha = exp(-softplus(x)) = 1 / (1 + e^x); e^x = inf gives alpha = 0.
__device__ __forceinline__ float decay_f(float x) { return 1.0f / (1.0f + expf(x)); }

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// phi(x) = elu(x) + 1, the positive feature map of ELU+1 linear attention.
__device__ __forceinline__ float elu1_f(float x) { return x > 0.0f ? x + 1.0f : expf(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// d/dx of prep(x) = normalize(silu(x)) (each step optional) for one row held
// by a warp, R values per lane; dy is overwritten by dx.  The norm's floor
// (1e-12) is a constant, so below it the derivative is dy / 1e-12.
template <int R>
__device__ __forceinline__ void prep_backward(const float (&x)[R], float (&dy)[R], bool silu,
                                              bool norm) {
    float s[R], sg[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        sg[r] = silu ? sigmoid_f(x[r]) : 1.0f;
        s[r] = silu ? x[r] * sg[r] : x[r];
    }
    if (norm) {
        float ss = 0.0f;
#pragma unroll
        for (int r = 0; r < R; ++r) ss += s[r] * s[r];
        const float nrm = sqrtf(warp_sum(ss));
        if (nrm > 1e-12f) {
            const float inv = 1.0f / nrm;
            float ydy = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) ydy += s[r] * inv * dy[r];
            ydy = warp_sum(ydy);
#pragma unroll
            for (int r = 0; r < R; ++r) dy[r] = (dy[r] - s[r] * inv * ydy) * inv;
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) dy[r] *= 1e12f;
        }
    }
    if (silu) {
#pragma unroll
        for (int r = 0; r < R; ++r) dy[r] *= sg[r] * (1.0f + x[r] * (1.0f - sg[r]));
    }
}

// Option bits (mirror the public header's LA_* values).
constexpr unsigned kL2NormK = 1u, kL2NormQ = 2u, kSiluQK = 4u, kGateScalar = 8u, kAdditive = 16u;

}  // namespace la
