/*
 * gemm13.h -- C ABI of the GB300 (sm_103a) GEMM library.
 *
 * One operation, in two calls:
 *
 *     C = cast( act( alpha * A.B + bias ) + beta * R )
 *
 * with A, B in FP32, FP16 or BF16, all products accumulated in FP32, and the
 * whole epilogue applied in registers before C is written once.
 *
 * Where the operation is defined:
 *   - "DeepGEMM" (discosf.com), sec. 1.2: FP16/BF16 input, FP32 accumulation,
 *     and a fusion hook so activation, residual add and scaling happen before
 *     the result leaves the kernel; sec. 3.1: K is the outer loop and C is
 *     stored once; sec. 3.4: accumulate in FP32 even for 16-bit inputs;
 *     sec. 2.3 / 4.3: per-shape tile choice with a configuration cache and a
 *     small-block variant for small M or N.
 *   - "CUDA Tile ... GEMM" (pgsm.cn), sec. 4.1: row-major A (M x K), B (K x N),
 *     C (M x N): A[row*K+k], B[k*N+col], C[row*N+col]; sec. 2: the FFN
 *     linear Y = X W^T + b (B given as W[N,K]) and the batched per-head QK^T.
 *   - "SGEMM ... 83% of cuBLAS" (cf-1.com), sec. 2-3: the FP32 SGEMM on CUDA
 *     cores (FFMA), which this library keeps as its FP32 path.
 * Readings where the pages are silent: the epilogue order above, GELU in its
 * erf form, FP32 bias and residual, round-to-nearest-even output casts.
 *
 * Conventions for every call below:
 *   - Pointers to matrices are DEVICE pointers of the current CUDA device;
 *     the caller owns them.  Leading dimensions and batch strides are in
 *     ELEMENTS of the buffer's own type.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every int-returning call returns a gemm_status_t; none of them aborts,
 *     traps or prints (set GEMM_LOG=1 in the environment to print plan
 *     decisions to stderr).
 */
#ifndef GEMM13_H
#define GEMM13_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_F32 = 0, GEMM_F16 = 1, GEMM_BF16 = 2 } gemm_dtype_t;

typedef enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_GELU_ERF = 1, /* 0.5*y*(1+erf(y/sqrt(2))) */
    GEMM_ACT_RELU = 2,     /* max(y, 0) */
    GEMM_ACT_SOFTMAX = 3   /* softmax over each output row: exp(y_ij - max_j y_ij) divided by
                              sum_j exp(y_ij - max_j y_ij), with y = alpha*A.B + bias over all N
                              columns -- the attention step Softmax(QK^T) of "CUDA Tile ...
                              GEMM", sec. 2, fused into the GEMM.  16-bit inputs, N <= 512,
                              K >= 1, no residual (else GEMM_ERR_UNSUPPORTED). */
} gemm_act_t;

typedef enum {
    GEMM_B_KN = 0, /* B[k*ldb + n]: row-major K x N */
    GEMM_B_NK = 1  /* B[n*ldb + k]: row-major N x K ("K-major", e.g. a weight W for X.W^T) */
} gemm_blayout_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,   /* a size, stride, enum or pointer is invalid */
    GEMM_ERR_UNSUPPORTED = -2,   /* valid request this build does not implement */
    GEMM_ERR_MISALIGNED = -3,    /* a base pointer breaks the alignment the plan assumed */
    GEMM_ERR_CUDA = -4,          /* a CUDA runtime/driver call failed */
    GEMM_ERR_DEVICE_TIMEOUT = -5,/* a kernel gave up waiting on a barrier (status word) */
    GEMM_ERR_BAD_PLAN = -6,      /* NULL, destroyed or foreign plan handle */
    GEMM_ERR_NO_DEVICE = -7,     /* no usable CUDA device, or not an sm_103 device */
    GEMM_ERR_OUT_OF_MEMORY = -8, /* plan workspace could not be allocated */
    GEMM_ERR_SCRATCH_LIMIT = -9  /* gemm_run_noalloc: staged operands exceed its fixed scratch */
} gemm_status_t;

/* Plan flags (gemm_epilogue_t.flags). */
#define GEMM_FLAG_FP32_TENSOR 0x1u       /* FP32 inputs: the dispatcher may pick the 3xTF32
                                            tensor-core kernel (GEMM_KERNEL_TF32X3) for large
                                            problems instead of the CUDA-core FFMA kernel; the
                                            result meets the same tolerance */
#define GEMM_FLAG_TEST_STALL 0x80000000u /* test only: the first CTA's producer withholds one
                                            operand tile so its waits run out; with a short
                                            timeout_ms this exercises the timeout path */
#define GEMM_FLAG_TEST_STALL_PEER 0x40000000u /* test only: as GEMM_FLAG_TEST_STALL, for the
                                                 second CTA (tensor-core kernel: the odd CTA of
                                                 the first CTA pair) */

/*
 * Everything about a call besides (dtype, M, N, K, lda, ldb, ldc).  Pass NULL
 * to gemm_plan for plain C = alpha*A.B in FP32 with B in KN layout, batch 1.
 * Start from gemm_epilogue_init() so new fields keep their defaults.
 */
typedef struct {
    gemm_blayout_t b_layout; /* default GEMM_B_KN */
    gemm_dtype_t out_dtype;  /* GEMM_F32 (default), GEMM_BF16 or GEMM_F16; RNE cast */
    int has_bias;            /* 1: bias[N] FP32 added after the alpha scale */
    gemm_act_t act;          /* applied after bias, before the residual (softmax: per row) */
    int has_residual;        /* 1: beta * R[M,N] (FP32, row-major, ldr) added last */
    float beta;              /* residual scale, default 1 */
    int64_t ldr;             /* residual leading dimension; 0 means ldc */
    int64_t batch;           /* number of independent products, default 1 */
    int64_t stride_a;        /* elements between consecutive A matrices (0: shared A) */
    int64_t stride_b;        /* elements between consecutive B matrices (0: shared B) */
    int64_t stride_c;        /* elements between consecutive C matrices; >= M*ldc if batch > 1 */
    int64_t stride_r;        /* elements between consecutive R matrices (0: shared R) */
    uint32_t flags;          /* GEMM_FLAG_* */
    uint32_t timeout_ms;     /* per-wait device timeout; 0 means 2000 ms */
} gemm_epilogue_t;

/* Kernel families a plan can use. */
typedef enum {
    GEMM_KERNEL_AUTO = 0,   /* let the dispatcher choose */
    GEMM_KERNEL_TC = 1,     /* tcgen05 tensor cores, TMA + mbarrier ring, TMEM accumulators (16-bit in) */
    GEMM_KERNEL_FFMA = 2,   /* CUDA-core FP32 FFMA, TMA-fed (FP32 in) */
    GEMM_KERNEL_SKINNY = 3, /* memory-bound streaming kernel for small M or N (any input type;
                               the dispatcher uses it for min(M, N) <= 4 and for K == 0) */
    GEMM_KERNEL_TF32X3 = 4  /* FP32 in on the tensor cores (tcgen05 kind::tf32): each operand
                               is split x = hi + lo into two TF32 numbers by a pre-pass and
                               A.B ~ Ahi.Bhi + Ahi.Blo + Alo.Bhi (the "SGEMM ... 83% of cuBLAS"
                               page, sec. 6, names the TF32 tensor-core path as the next step
                               past FFMA; splitting recovers FP32-level accuracy).  Needs a plan
                               workspace of 2 x (M + N) x K FP32 values per batch entry. */
} gemm_kernel_t;

/* A tile configuration: what the dispatcher chose, or what a caller forces. */
typedef struct {
    gemm_kernel_t kernel;
    int32_t bm, bn, bk;   /* output tile and K step (elements) */
    int32_t stages;       /* shared-memory pipeline depth */
    int32_t split_k;      /* K slices reduced deterministically (1 = none) */
    int32_t raster_group; /* M tiles walked together for L2 reuse */
    int32_t stage_a;      /* 1: A is first copied to an aligned plan workspace */
    int32_t stage_b;      /* 1: B likewise */
    int32_t num_ctas;     /* persistent grid size; 0 = one per SM */
    int32_t variant;      /* family-specific main-loop variant; FFMA: 0 scalar FFMA,
                             1 packed fma.rn.f32x2 (KN layout only), 2 32 x 32 tiles from
                             plain loads for small M x N (bm = bn = bk = 32, any stride or
                             alignment, no stream-K); TC: 0 single CTAs with
                             4 epilogue warps, 1 single CTAs with 8 epilogue warps (short K),
                             2 CTA pairs (cta_group::2, 256 x 256 tiles, no split-K),
                             3 CTA pairs with 8 epilogue warps (bn 256, 5 stages);
                             TF32X3: 0 single CTAs (bn 128), 2 CTA pairs (bn 256) */
    int32_t stream_k;     /* FFMA and TC: 1 = persistent grid with (tile, K-step) units split
                             evenly over the CTAs (CTA pairs); a tile cut between them is
                             finished by the holder of its first K step, which adds the others'
                             partial sums in a fixed order (deterministic).  Needs a plan
                             workspace of grid x 64 KB (FFMA) or grid x 128 x bn x 4 bytes (TC);
                             TC: no split-K, no row softmax. */
} gemm_config_t;

typedef struct gemm_plan_s* gemm_plan_t;

/* Fills *e with the defaults listed above. */
void gemm_epilogue_init(gemm_epilogue_t* e);

/*
 * Validates a problem, picks (or fetches from the per-process cache) a tile
 * configuration, and allocates the plan's device state on the CURRENT device:
 * a status word and, only when a stride or base alignment rules out direct TMA
 * loads, a workspace for aligned operand copies (gemm_plan_info reports its
 * size).  No kernel runs.
 *   M, N, K >= 0 (M or N == 0: runs do nothing; K == 0: C = epilogue(0)).
 *   lda >= K, ldb >= N (KN) or >= K (NK), ldc >= N, ldr >= N.
 * Errors: INVALID_ARG, UNSUPPORTED, NO_DEVICE, OUT_OF_MEMORY, CUDA.
 * On success *out_plan owns its state until gemm_plan_destroy.
 */
int gemm_plan(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc,
              const gemm_epilogue_t* epilogue, gemm_plan_t* out_plan);

/* As gemm_plan, with the configuration forced (cfg->kernel may not be AUTO).
 * Fields a family does not use are ignored; invalid combinations return
 * INVALID_ARG or UNSUPPORTED.  Meant for tests and tuning. */
int gemm_plan_with_config(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc,
                          const gemm_epilogue_t* epilogue, const gemm_config_t* cfg,
                          gemm_plan_t* out_plan);

/*
 * Enqueues the GEMM on `stream` and returns without synchronising.
 *   A: dtype, [batch][M][lda];  B: dtype, [batch][K][ldb] (KN) or [batch][N][ldb] (NK);
 *   C: out_dtype, [batch][M][ldc];  bias: FP32 [N] (must be NULL iff !has_bias);
 *   residual: FP32 [batch][M][ldr] (NULL iff !has_residual).
 * C must not overlap A, B, bias or residual.  Allocates nothing.  Runs of
 * one plan on different streams may overlap on the GPU unless the plan has a
 * staging workspace (gemm_plan_info(...).workspace_bytes > 0): those runs
 * share it and must be ordered.
 * Errors: BAD_PLAN, INVALID_ARG (NULL pointer), MISALIGNED, CUDA (launch failed).
 * A device-side timeout is reported later by gemm_plan_status.
 */
int gemm_run(gemm_plan_t plan, const void* A, const void* B, void* C,
             const void* bias, const void* residual, float alpha, void* stream);

/* Synchronises the device, then reports GEMM_ERR_DEVICE_TIMEOUT if any kernel
 * of this plan gave up on a wait since the plan was made, else GEMM_OK.  The
 * condition is sticky.  Errors: BAD_PLAN, CUDA. */
int gemm_plan_status(gemm_plan_t plan);

/* Information about a plan. */
typedef struct {
    gemm_config_t config;
    int64_t workspace_bytes; /* device bytes owned by the plan besides its status word */
    int32_t num_sms;         /* SMs of the plan's device */
    int32_t device;          /* CUDA ordinal */
    int32_t cache_hit;       /* 1 if gemm_plan found the config in the cache */
    int32_t kernels_per_run; /* kernel launches one gemm_run makes (0 for empty problems) */
} gemm_plan_info_t;

int gemm_plan_info(gemm_plan_t plan, gemm_plan_info_t* out);

/* Releases a plan (NULL is a no-op).  Runs still in flight must finish first. */
void gemm_plan_destroy(gemm_plan_t plan);

/*
 * Host-only: the configuration the dispatcher would choose for this problem
 * on a device with `num_sms` SMs.  Touches no CUDA state and does not use the
 * cache.  Errors: INVALID_ARG, UNSUPPORTED.
 */
int gemm_select_config(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc,
                       const gemm_epilogue_t* epilogue, int32_t num_sms,
                       gemm_config_t* out);

/* Configuration cache: entries, hits and misses since start (or last clear). */
void gemm_cache_stats(int64_t* entries, int64_t* hits, int64_t* misses);
void gemm_cache_clear(void);

/* Static text for a status code ("unknown status" for others). */
const char* gemm_strerror(int status);

/* Library version string. */
const char* gemm_version(void);

/*
 * gemm_run_noalloc -- the same GEMM as gemm_plan + gemm_run in one call that
 * allocates no memory (no cudaMalloc, no plan, no host heap) once its
 * per-device set-up (below) has run.  The
 * pages have no counterpart: this exists for callers that cannot allocate
 * device memory where they run a GEMM -- code inside an allocator or memory-
 * pool callback, code holding a lock the allocator also takes, or programs
 * that reserve all device memory up front.
 *
 * Arguments: as gemm_plan followed by gemm_run (same meaning, layout and
 * validation; epilogue may be NULL).  A, B, C, bias and residual are the
 * caller's device buffers; the call enqueues on `stream` and returns.
 *
 * Scratch: operands that TMA cannot read in place (strides or base addresses
 * not 16-byte aligned) are copied into a fixed 64 MiB device array inside the
 * library, one per GPU, resident from the set-up until process exit.  The
 * array also holds the status word.  If the staged copies need more than
 * that (each staged row padded to 16 bytes, 256 bytes reserved), the call
 * returns GEMM_ERR_SCRATCH_LIMIT and does nothing.
 *
 * Sharing: every call on a device uses the same array and finds the previous
 * call's data in it (it rewrites what it uses).  Calls whose work overlaps on
 * the GPU -- on different streams or from several threads -- race on the
 * array; order them on one stream.
 *
 * Device timeouts: if a kernel gives up on a device-side wait (default limit
 * 2 s per wait), C is left undefined (partly written).  This call cannot
 * report that (there is no plan whose status could be queried); callers that
 * need to know use gemm_plan / gemm_run / gemm_plan_status.
 *
 * Set-up: the first call on each device and CUDA context (with that device
 * current) looks up the array's device address and loads every kernel this
 * entry point can launch.  Under CUDA's lazy module loading both steps make
 * the CUDA driver allocate device memory, so make that first call before the
 * code that must not allocate, and before any stream capture.  A call with
 * M = 0 or N = 0 performs the set-up and nothing else.
 *
 * Errors: INVALID_ARG, UNSUPPORTED, SCRATCH_LIMIT, NO_DEVICE, CUDA.
 */
int gemm_run_noalloc(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, const void* B, int64_t ldb,
                     void* C, int64_t ldc, const gemm_epilogue_t* epilogue,
                     const void* bias, const void* residual, float alpha, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM13_H */
