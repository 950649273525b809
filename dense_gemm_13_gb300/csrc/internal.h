// internal.h -- declarations shared between the host side (plan, dispatch,
// C ABI) and the kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm13.h"

namespace g13 {

// Everything the fused epilogue needs: y = alpha*acc (+bias[n]) -> act -> (+beta*R) -> cast.
struct EpiParams {
    void* C;
    int64_t ldc, stride_c;
    const float* bias;
    const float* R;
    int64_t ldr, stride_r;
    int64_t M, N;
    float alpha, beta;
    int out_dtype;   // gemm_dtype_t
    int act;         // gemm_act_t
    int c_vec;       // 1: C rows take aligned vector stores at columns that are multiples of 4
    int r_vec;       // 1: R rows take aligned float4 loads at columns that are multiples of 4
};

struct Shape {
    int64_t M, N, K, batch;
    int a_bmul, b_bmul;  // 1, or 0 when that operand is shared by every batch entry
};

struct LaunchCtx {
    unsigned* status;     // per-plan device status word
    uint64_t timeout_ns;  // bound on every mbarrier wait
    uint32_t flags;       // GEMM_FLAG_*
    int num_sms;
    cudaStream_t stream;
    // stream-K (FFMA): partial-sum slots, their tags, grid size, this launch's tag
    float* sk_partials;
    unsigned* sk_tags;
    int64_t sk_grid;
    unsigned sk_epoch;
    // the kernel is launched as a programmatic dependent of the staging copy just
    // before it in the stream (it waits for the copy before its first load)
    int pdl;
};

// TMA descriptors for the tensor-core epilogue: C (box of 32 rows x 128 bytes,
// 128B swizzle) and, when r_tma, the FP32 residual (32 x 32, 128B swizzle).
struct TcEpiMaps {
    CUtensorMap c, r;
    int r_tma;
    int c_bmul, r_bmul;  // batch coordinate multipliers (0: shared across the batch)
    int c_smul;          // split-K: split coordinate multiplier of the C descriptor
    int64_t n_tma;       // columns covered by the C descriptor (N rounded down to 16 bytes)
};

// Tensor-core path: A [batch][M][K] 16-bit via tmA (K innermost); B via tmB:
// NK layout -> dims (K, N, batch), KN layout -> dims (N, K, batch).  With em
// null the epilogue stores C from registers.  Split-K (cfg.split_k > 1): `e`
// describes the FP32 partial slabs [batch][split][M][N] the kernel writes, and
// final_epi the real epilogue a second kernel applies after adding them.
cudaError_t launch_tc(const gemm_config_t& cfg, int dtype, int b_layout, const CUtensorMap& tmA,
                      const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                      const EpiParams& e, const LaunchCtx& lc,
                      const EpiParams* final_epi = nullptr);
// K ranges a tensor-core split-K launch actually uses (<= split_k, none empty).
int tc_effective_splits(int64_t K, int split_k);
// Adds partial slabs [batch][splits][M][N] in split order and applies e.
cudaError_t launch_split_reduce(const float* partial, int64_t M, int64_t N, int64_t batch,
                                int splits, const EpiParams& e, const LaunchCtx& lc);
// Shared memory the TC kernel needs for a config (bytes), or 0 if unsupported.
size_t tc_smem_bytes(const gemm_config_t& cfg);
// FP32 on the tensor cores (3xTF32): A and B come as split buffers
// [batch][hi, lo][rows][K] (B K-major), tmA / tmB over (K, rows, 2 * batch).
cudaError_t launch_tc3(const gemm_config_t& cfg, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const TcEpiMaps* em, const Shape& s, const EpiParams& e,
                       const LaunchCtx& lc);
size_t tc3_smem_bytes(const gemm_config_t& cfg);
// Splits FP32 X[batch][rows][cols] (row stride ld, batch stride bstride,
// any alignment) into out[batch][2][cols or rows][ldo]: hi = X rounded to
// TF32 (nearest), lo = X - hi.  transpose: out rows are X's columns (for B
// in KN layout); columns past the source's are written as zeros up to ldo.
cudaError_t launch_tf32_split(const float* X, int64_t rows, int64_t cols, int64_t ld,
                              int64_t bstride, int64_t batches, bool transpose, float* out,
                              int64_t ldo, cudaStream_t stream);
// TC config variant that runs CTA pairs (tcgen05 cta_group::2, 256-row tiles).
constexpr int TC_VARIANT_PAIR = 2;
// CTA pairs with eight epilogue warps (two per TMEM lane quarter) and 5 stages:
// for C layouts TMA cannot store, whose per-row epilogue outlasts the main loop.
constexpr int TC_VARIANT_PAIR8 = 3;
// Tensor-core kernels by epilogue kind.  TC_EK_ANY runs every epilogue (the
// row softmax; C rows TMA cannot store); the others store C by TMA and hold
// only one kind of epilogue: scale only, bias / ReLU / residual, or GELU (with
// or without bias, no residual).  A kernel whose loop holds only the steps its
// tiles run fetches far fewer instructions per tile.
// TC_EK_ROWS holds only the path for C rows TMA cannot store (any epilogue but
// the row softmax); TC_EK_SOFTMAX only the row softmax with C stored by TMA.
constexpr int TC_EK_ANY = 0, TC_EK_PLAIN = 1, TC_EK_BIAS = 2, TC_EK_GELU = 3, TC_EK_ROWS = 4,
              TC_EK_SOFTMAX = 5;
// The launchers of each part (tc_any_*.cu, tc_spec_*.cu, tc_sk_*.cu); the spec
// ones take the kind, and the spec and stream-K ones the configurations of
// tc_has_spec only.
cudaError_t launch_tc_any_kn(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                             const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe);
cudaError_t launch_tc_any_nk(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                             const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe);
cudaError_t launch_tc_spec_kn(int ek, const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                              const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                              const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe);
cudaError_t launch_tc_spec_nk(int ek, const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                              const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                              const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe);
cudaError_t launch_tc_sk_kn(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                            const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                            const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe);
cudaError_t launch_tc_sk_nk(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                            const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                            const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe);
// Whether cfg has kernels specialised by epilogue kind and stream-K kernels.
bool tc_has_spec(const gemm_config_t& cfg);
cudaError_t tc_preload_sk_kn();
cudaError_t tc_preload_sk_nk();
cudaError_t tc_preload_any_kn();
cudaError_t tc_preload_any_nk();
cudaError_t tc_preload_spec_kn();
cudaError_t tc_preload_spec_nk();
inline bool tc_is_pair(const gemm_config_t& cfg) {
    return cfg.variant == TC_VARIANT_PAIR || cfg.variant == TC_VARIANT_PAIR8;
}
// Rows of a K-major B box: the tile's columns, split between the CTAs of a
// pair, at most 256 (a TMA box dimension's limit; 512-wide tiles take two).
inline int tc_b_box_rows(const gemm_config_t& cfg) {
    const int rows = tc_is_pair(cfg) ? cfg.bn / 2 : cfg.bn;
    return rows < 256 ? rows : 256;
}

// FP32 FFMA config variant for problems with too few 128-row tiles to fill the
// GPU: 32 x 32 tiles from plain loads (any stride or alignment, no TMA, no
// staging, no workspace).
constexpr int FFMA_VARIANT_SMALL = 2;
inline bool ffma_small(const gemm_config_t& c) {
    return c.kernel == GEMM_KERNEL_FFMA && c.variant == FFMA_VARIANT_SMALL;
}
cudaError_t launch_ffma_small(const float* A, const float* B, int64_t lda, int64_t ldb,
                              int64_t stride_a, int64_t stride_b, int b_layout, const Shape& s,
                              const EpiParams& e, cudaStream_t stream);

// FP32 FFMA path: A via tmA (dims K, M, batch), B via tmB (KN: N, K, batch; NK: K, N, batch).
cudaError_t launch_ffma(const gemm_config_t& cfg, int b_layout, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                        const LaunchCtx& lc);
size_t ffma_smem_bytes(const gemm_config_t& cfg);
// Bytes of one stream-K partial-sum slot (one 128 x BN FP32 tile).
size_t ffma_partial_slot_bytes(const gemm_config_t& cfg);
// Whether the FFMA kernel can index this problem's (tile, K-step) units in 32 bits.
bool ffma_units_ok(const Shape& s, int bn);
// Resident CTAs per SM of the FFMA kernel a config selects (0 on error).
int ffma_ctas_per_sm(const gemm_config_t& cfg, int b_layout);

// Memory-bound path for small M or N: plain (unaligned-capable) loads.
struct SkinnyArgs {
    const void* A;
    const void* B;
    int64_t lda, ldb, stride_a, stride_b;
    int dtype;
    int b_layout;
};
// Split partial sums go to lc.sk_partials ([batch][split_k][P][Q] FP32) when
// cfg.split_k > 1; a second kernel reduces them in order and applies the epilogue.
cudaError_t launch_skinny(const gemm_config_t& cfg, const SkinnyArgs& a, const Shape& s,
                          const EpiParams& e, const LaunchCtx& lc);
// Which operand the skinny kernel streams: P = the small dimension, Q = the
// large one; dot = 1 when the streamed operand has K contiguous.
void skinny_geometry(int64_t M, int64_t N, int b_layout, int64_t* P, int64_t* Q, int* dot);

// Skinny config variant that streams the large operand through shared memory
// by TMA (csrc/skinny_tma.cu); the plain-load kernel is variant 0 and also
// runs whenever the large operand's base address is not 16-byte aligned.
constexpr int SKINNY_VARIANT_TMA = 1;
// Host-side geometry of the TMA skinny kernel: K per pipeline stage and rows
// (dot) or columns (axpy) per work block, for a dtype and mode.
int64_t skinny_tma_stage_k(int dtype, int dot);
int64_t skinny_tma_block(int dtype, int dot);
// Whether P small-operand rows of length K fit the kernel's shared memory.
bool skinny_tma_fits(int64_t P, int64_t K, int dtype, int dot);
// Whether this run's large operand can be read by TMA (16-byte aligned base,
// row stride and batch stride).
bool skinny_tma_aligned(const SkinnyArgs& a, const Shape& s);
// Stream-K over the large operand's stages: lc.sk_partials holds the partial
// sums of blocks cut between CTAs (skinny_tma_workspace_bytes(lc.num_sms)),
// lc.sk_tags one zeroed counter per (batch, block) (at most batch * Q).
// num_ctas > 0 caps the grid (one CTA per SM otherwise).
// tm: skinny_tma_encode's descriptor of this run's large operand.
int skinny_tma_encode(const SkinnyArgs& a, const Shape& s, CUtensorMap* tm);
cudaError_t launch_skinny_tma(const SkinnyArgs& a, const Shape& s, const EpiParams& e,
                              const LaunchCtx& lc, int num_ctas, const CUtensorMap& tm);
size_t skinny_tma_workspace_bytes(int num_sms);
// 3-D tiled TMA descriptor without swizzle over [batches][rows][cols] (row
// stride ld, batch stride bstride, in elements), box box_cols x box_rows.
int tmap_encode_3d(CUtensorMap* m, int dtype, const void* base, int64_t cols, int64_t rows,
                   int64_t ld, int64_t batches, int64_t bstride, uint32_t box_cols,
                   uint32_t box_rows);

// Copies [batch][rows][cols] (row stride ld, batch stride bstride, element
// size esz) into a dense [batch][rows][dst_ld] buffer (dst and dst_ld * esz
// multiples of 16 bytes, else cudaErrorInvalidValue).  Padding columns get
// unspecified bytes: the tensor maps over the copy end at column cols.
// One staging copy job: rows x cols elements of esz bytes (row stride ld,
// batch stride bstride, batch batches) into dst with row stride dst_ld.
struct StageJob {
    const void* src;
    int64_t rows, cols, ld, bstride, batch;
    void* dst;
    int64_t dst_ld;
};
// Both operands' staging copies in one launch (njobs 1 or 2).
cudaError_t launch_stage_copies(const StageJob* jobs, int njobs, int esz, cudaStream_t stream);
cudaError_t launch_stage_copy(const void* src, int64_t rows, int64_t cols, int64_t ld,
                              int64_t bstride, int64_t batch, int esz, void* dst,
                              int64_t dst_ld, cudaStream_t stream);

// Load every kernel the allocation-free entry point can launch onto the
// current device (under lazy module loading a kernel is otherwise loaded, and
// its device memory allocated, at its first launch).
cudaError_t tc_preload_kernels();
cudaError_t ffma_preload_kernels();
cudaError_t aux_preload_kernels();

}  // namespace g13
