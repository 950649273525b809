// dispatch.h -- problem description, validation and the shape-bucket
// dispatcher with its configuration cache (host only, no CUDA calls).
#pragma once
#include <cstdint>

#include "gemm13.h"

namespace g13 {

// A fully normalised problem (defaults filled in, ldr resolved).
struct Problem {
    int dtype;
    int64_t M, N, K, lda, ldb, ldc;
    gemm_epilogue_t epi;
};

// Fills p from the public arguments; returns GEMM_OK or GEMM_ERR_INVALID_ARG.
int make_problem(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                 int64_t ldc, const gemm_epilogue_t* epi, Problem* p);

// Bytes per element of a gemm_dtype_t (0 for an unknown value).
int dtype_size(int dtype);

// Whether a row stride / batch stride (elements) allows direct TMA loads.
bool stride_tma_ok(int64_t ld, int64_t bstride, int64_t batch, int esz);

// K splits the skinny kernel uses for p (1 = none).
int skinny_splits(const Problem& p, int num_sms);
// Whether p can run the TMA-streamed skinny kernel.
bool skinny_tma_suits(const Problem& p);
// K splits for the tensor-core kernel with BN-wide tiles (1 = none).
int tc_splits(const Problem& p, int num_sms, int bn);

// The dispatcher's heuristic choice for p on a device with num_sms SMs.
int choose_config(const Problem& p, int num_sms, gemm_config_t* out);

// Checks (and completes) a caller-forced configuration for p.
int check_config(const Problem& p, const gemm_config_t& in, gemm_config_t* out);

// Per-process cache of choose_config results, keyed by the whole problem
// shape (sizes, strides, layout, epilogue kind, dtype) and num_sms.
int cached_config(const Problem& p, int num_sms, gemm_config_t* out, bool* hit);
void cache_stats(int64_t* entries, int64_t* hits, int64_t* misses);
void cache_clear();

}  // namespace g13
