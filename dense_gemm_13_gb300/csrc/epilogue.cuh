// epilogue.cuh -- the fused epilogue shared by every kernel:
//     y = alpha*acc (+ bias[n]);  y = act(y);  y += beta*R[m,n];  C[m,n] = cast(y)
// applied to four consecutive columns in registers, so C is written once
// ("DeepGEMM", sec. 1.2 and 3.1).  Casts are round-to-nearest-even.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace g13 {

__device__ __forceinline__ float epi_act(int act, float y) {
    if (act == GEMM_ACT_GELU_ERF) return 0.5f * y * (1.0f + erff(y * 0.70710678118654752440f));
    if (act == GEMM_ACT_RELU) return fmaxf(y, 0.0f);
    return y;
}

// Columns [col, col+4) of output row `row` in batch `b`; col is a multiple of 4.
// Rows >= M and columns >= N are skipped.
__device__ __forceinline__ void epi_store4(const EpiParams& e, int64_t b, int64_t row, int64_t col,
                                           float v0, float v1, float v2, float v3) {
    if (row >= e.M || col >= e.N) return;
    const bool full = col + 3 < e.N;
    float y[4] = {v0 * e.alpha, v1 * e.alpha, v2 * e.alpha, v3 * e.alpha};
    if (e.bias) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (full || col + j < e.N) y[j] += __ldg(e.bias + col + j);
    }
    if (e.act != GEMM_ACT_NONE) {
#pragma unroll
        for (int j = 0; j < 4; ++j) y[j] = epi_act(e.act, y[j]);
    }
    if (e.R) {
        const float* r = e.R + b * e.stride_r + row * e.ldr + col;
        if (full && e.r_vec) {
            const float4 rv = __ldg(reinterpret_cast<const float4*>(r));
            y[0] += e.beta * rv.x;
            y[1] += e.beta * rv.y;
            y[2] += e.beta * rv.z;
            y[3] += e.beta * rv.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < e.N) y[j] += e.beta * __ldg(r + j);
        }
    }
    const int64_t off = b * e.stride_c + row * e.ldc + col;
    if (e.out_dtype == GEMM_F32) {
        float* c = static_cast<float*>(e.C) + off;
        if (full && e.c_vec) {
            *reinterpret_cast<float4*>(c) = make_float4(y[0], y[1], y[2], y[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < e.N) c[j] = y[j];
        }
    } else if (e.out_dtype == GEMM_BF16) {
        __nv_bfloat16* c = static_cast<__nv_bfloat16*>(e.C) + off;
        if (full && e.c_vec) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(c) = pk;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < e.N) c[j] = __float2bfloat16_rn(y[j]);
        }
    } else {
        __half* c = static_cast<__half*>(e.C) + off;
        if (full && e.c_vec) {
            __half2 lo = __floats2half2_rn(y[0], y[1]);
            __half2 hi = __floats2half2_rn(y[2], y[3]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(c) = pk;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < e.N) c[j] = __float2half_rn(y[j]);
        }
    }
}

// One output element (for kernels whose columns are not 4-aligned groups).
__device__ __forceinline__ void epi_store1(const EpiParams& e, int64_t b, int64_t row, int64_t col,
                                           float v) {
    if (row >= e.M || col >= e.N) return;
    float y = v * e.alpha;
    if (e.bias) y += __ldg(e.bias + col);
    y = epi_act(e.act, y);
    if (e.R) y += e.beta * __ldg(e.R + b * e.stride_r + row * e.ldr + col);
    const int64_t off = b * e.stride_c + row * e.ldc + col;
    if (e.out_dtype == GEMM_F32)
        static_cast<float*>(e.C)[off] = y;
    else if (e.out_dtype == GEMM_BF16)
        static_cast<__nv_bfloat16*>(e.C)[off] = __float2bfloat16_rn(y);
    else
        static_cast<__half*>(e.C)[off] = __float2half_rn(y);
}

}  // namespace g13
