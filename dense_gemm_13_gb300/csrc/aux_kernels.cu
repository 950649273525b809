// aux_kernels.cu -- operand staging copy and the memory-bound skinny kernel.
//
// Staging: TMA needs 16-byte-aligned base addresses and row strides.  When a
// caller's A or B breaks that (e.g. K = 17 elements of 2 bytes per row), the
// plan copies the operand once per run into its own workspace with rows padded
// to 16 bytes, and the tensor-core / FFMA kernels read the copy.  The copy is
// a plain coalesced row-by-row memcpy (HBM-bound).
//
// Skinny: for M or N at most 64 a 128-row tensor-core tile would be mostly
// padding and the GEMM is bound by reading the large operand once ("DeepGEMM",
// sec. 4.3: a small-block variant for small M or N).  This version gives each
// warp one output element: lanes stride over K, products accumulate in FP32,
// and a fixed shuffle tree reduces them (deterministic), then the epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"

namespace g13 {
namespace {

template <typename T>
__global__ void stage_copy_kernel(const T* __restrict__ src, int64_t rows, int64_t cols, int64_t ld,
                                  int64_t bstride, int64_t batch, T* __restrict__ dst,
                                  int64_t dst_ld) {
    const int64_t total_rows = rows * batch;
    for (int64_t r = blockIdx.x; r < total_rows; r += gridDim.x) {
        const int64_t b = r / rows, i = r - b * rows;
        const T* s = src + b * bstride + i * ld;
        T* d = dst + r * dst_ld;
        for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) d[c] = s[c];
    }
}

template <typename T>
__device__ __forceinline__ float ld_as_float(const T* p);
template <>
__device__ __forceinline__ float ld_as_float<float>(const float* p) {
    return __ldg(p);
}
template <>
__device__ __forceinline__ float ld_as_float<__half>(const __half* p) {
    return __half2float(__ldg(p));
}
template <>
__device__ __forceinline__ float ld_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
}

template <typename T>
__global__ void skinny_dot_kernel(const T* __restrict__ A, const T* __restrict__ B, int64_t lda,
                                  int64_t ldb, int64_t stride_a, int64_t stride_b, int b_nk,
                                  int64_t M, int64_t N, int64_t K, int64_t batch,
                                  const EpiParams e) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t outputs = M * N * batch;
    for (int64_t o = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         o < outputs; o += warps_total) {
        const int64_t b = o / (M * N);
        const int64_t r = o - b * M * N;
        const int64_t m = r / N, n = r - m * N;
        const T* a = A + b * stride_a + m * lda;
        const T* bb = B + b * stride_b;
        float acc = 0.0f;
        if (b_nk) {
            const T* bn = bb + n * ldb;
            for (int64_t k = lane; k < K; k += 32) acc = fmaf(ld_as_float(a + k), ld_as_float(bn + k), acc);
        } else {
            for (int64_t k = lane; k < K; k += 32)
                acc = fmaf(ld_as_float(a + k), ld_as_float(bb + k * ldb + n), acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) epi_store1(e, b, m, n, acc);
    }
}

}  // namespace

cudaError_t launch_stage_copy(const void* src, int64_t rows, int64_t cols, int64_t ld,
                              int64_t bstride, int64_t batch, int esz, void* dst, int64_t dst_ld,
                              cudaStream_t stream) {
    const int64_t total = rows * batch;
    if (total <= 0 || cols <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(total < 65536 ? total : 65536);
    const int threads = cols >= 256 ? 256 : 128;
    if (esz == 2)
        stage_copy_kernel<uint16_t><<<grid, threads, 0, stream>>>(
            static_cast<const uint16_t*>(src), rows, cols, ld, bstride, batch,
            static_cast<uint16_t*>(dst), dst_ld);
    else
        stage_copy_kernel<float><<<grid, threads, 0, stream>>>(static_cast<const float*>(src), rows,
                                                               cols, ld, bstride, batch,
                                                               static_cast<float*>(dst), dst_ld);
    return cudaGetLastError();
}

cudaError_t launch_skinny(const gemm_config_t& cfg, const SkinnyArgs& a, const Shape& s,
                          const EpiParams& e, const LaunchCtx& lc) {
    const int64_t outputs = s.M * s.N * s.batch;
    if (outputs <= 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (outputs + 7) / 8;
    const int64_t cap = static_cast<int64_t>(lc.num_sms > 0 ? lc.num_sms : 148) * 8;
    if (blocks > cap) blocks = cap;
    const unsigned grid = static_cast<unsigned>(blocks);
    const int nk = a.b_layout == GEMM_B_NK;
    (void)cfg;
    switch (a.dtype) {
        case GEMM_F32:
            skinny_dot_kernel<float><<<grid, threads, 0, lc.stream>>>(
                static_cast<const float*>(a.A), static_cast<const float*>(a.B), a.lda, a.ldb,
                a.stride_a, a.stride_b, nk, s.M, s.N, s.K, s.batch, e);
            break;
        case GEMM_F16:
            skinny_dot_kernel<__half><<<grid, threads, 0, lc.stream>>>(
                static_cast<const __half*>(a.A), static_cast<const __half*>(a.B), a.lda, a.ldb,
                a.stride_a, a.stride_b, nk, s.M, s.N, s.K, s.batch, e);
            break;
        default:
            skinny_dot_kernel<__nv_bfloat16><<<grid, threads, 0, lc.stream>>>(
                static_cast<const __nv_bfloat16*>(a.A), static_cast<const __nv_bfloat16*>(a.B),
                a.lda, a.ldb, a.stride_a, a.stride_b, nk, s.M, s.N, s.K, s.batch, e);
            break;
    }
    return cudaGetLastError();
}

}  // namespace g13
