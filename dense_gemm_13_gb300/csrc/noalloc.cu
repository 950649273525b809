// noalloc.cu -- gemm_run_noalloc: one GEMM call that allocates no memory.
//
// Who needs it: code that must not call cudaMalloc at the point where it runs
// a GEMM -- e.g. a callback running under a memory pool or allocator that
// forbids re-entrant allocation, code holding a lock the allocator may also
// take, or a program that has budgeted every byte of device memory up front.
// gemm_plan is not usable there: it allocates a status word and, for
// operands TMA cannot read directly, a staging workspace.
//
// This entry point runs the same kernels as gemm_plan + gemm_run, but its
// scratch (the status word and the aligned copies of staged operands) lives in
// the file-scope device array g13_noalloc_scratch below, which exists once per
// GPU that loads the library and stays resident until the process exits.
//
// Sharing rules (the array is one buffer per device):
//   * every call uses the same array, and it keeps whatever the previous call
//     left in it; this call rewrites what it reads (status word, staged
//     copies) before use;
//   * calls whose kernels overlap on the GPU (different streams, or several
//     host threads) race on the array: order them on one stream, or use
//     gemm_plan / gemm_run instead;
//   * a device-side wait that runs out (default limit 2 s per wait) makes the
//     kernels give up: C is then undefined (partly written).  The condition is
//     recorded in the shared status word but not reported to the caller
//     (there is no plan to query); use gemm_plan / gemm_run where it matters.
// Set-up: the first call on each device and CUDA context (with that device
// current) looks up the array's device address with cudaGetSymbolAddress and
// loads every kernel this entry point can launch.  Under CUDA's lazy module
// loading both steps allocate device memory inside the CUDA driver, so make
// that first call before the region that must not allocate, and before any
// stream capture; a call with M = 0 or N = 0 does the set-up and nothing else.
// Problems whose staged operands need more than kScratchBytes return
// GEMM_ERR_SCRATCH_LIMIT.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "dispatch.h"
#include "gemm13.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr size_t kStatusBytes = 256;                 // status word, padded to 256 B
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) unsigned char g13_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_setup_mu;
// Per device: the context the set-up ran in and the array's address there.
// A different current context (a non-primary one, or the primary one after a
// device reset) gets its own set-up.
CUcontext g_setup_ctx[kMaxDevices] = {};
void* g_scratch_ptr[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

// Device address of the scratch array in the current device's current
// context; the first call there also loads the kernels this entry point uses.
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return GEMM_ERR_NO_DEVICE;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (!get_ctx) return GEMM_ERR_NO_DEVICE;
    // Null before the runtime has made a context current on this thread.
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return GEMM_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_setup_ctx[dev] != ctx) {
        void* p = nullptr;
        // (binds the device's primary context if none is current)
        if (cudaGetSymbolAddress(&p, g13_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (g13::tc_preload_kernels() != cudaSuccess || g13::ffma_preload_kernels() != cudaSuccess ||
            g13::aux_preload_kernels() != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return GEMM_ERR_NO_DEVICE;
        g_scratch_ptr[dev] = p;
        g_setup_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return GEMM_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn noalloc_encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// 3-D tiled descriptor over [batches][rows][cols] with row stride ld and batch stride bstride.
int noalloc_encode(CUtensorMap* m, int dtype, const void* base, int64_t cols, int64_t rows,
                   int64_t ld, int64_t batches, int64_t bstride, uint32_t box_cols,
                   uint32_t box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = noalloc_encode_fn();
    if (!fn) return GEMM_ERR_NO_DEVICE;
    const int esz = g13::dtype_size(dtype);
    const CUtensorMapDataType t = dtype == GEMM_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dtype == GEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batches)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * esz),
                             static_cast<cuuint64_t>((batches > 1 ? bstride : rows * ld) * esz)};
    if (strides[1] == 0) strides[1] = strides[0];
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, t, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

int status_of(cudaError_t e) {
    if (e == cudaSuccess) return GEMM_OK;
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ||
        e == cudaErrorNoKernelImageForDevice)
        return GEMM_ERR_NO_DEVICE;
    return GEMM_ERR_CUDA;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

}  // namespace

extern "C" int gemm_run_noalloc(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K,
                                const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                                int64_t ldc, const gemm_epilogue_t* epilogue, const void* bias,
                                const void* residual, float alpha, void* stream) {
    using namespace g13;
    Problem p;
    int rc = make_problem(dtype, M, N, K, lda, ldb, ldc, epilogue, &p);
    if (rc != GEMM_OK) return rc;
    const gemm_epilogue_t& ep = p.epi;

    int dev = -1, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;
    // Set-up (first call per device and context), also for empty problems.
    void* scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != GEMM_OK) return rc;

    if (p.M == 0 || p.N == 0) return GEMM_OK;
    if (!C) return GEMM_ERR_INVALID_ARG;
    if (p.K > 0 && (!A || !B)) return GEMM_ERR_INVALID_ARG;
    if ((ep.has_bias != 0) != (bias != nullptr)) return GEMM_ERR_INVALID_ARG;
    if ((ep.has_residual != 0) != (residual != nullptr)) return GEMM_ERR_INVALID_ARG;

    gemm_config_t cfg;
    p.epi.flags &= ~GEMM_FLAG_FP32_TENSOR;  // 3xTF32 needs split buffers: FP32 runs on FFMA
    rc = choose_config(p, sms, &cfg);  // no cache: nothing is allocated, not even on the host
    if (rc != GEMM_OK) return rc;
    cfg.stream_k = 0;  // whole tiles per CTA: stream-K partial slots would need more scratch
    cfg.split_k = 1;   // the skinny kernel runs K unsplit (no partial sums to keep)
    const int esz = dtype_size(p.dtype);
    // Misaligned base pointers are staged too (the scratch is always there).
    if (cfg.kernel != GEMM_KERNEL_SKINNY && !ffma_small(cfg)) {
        if (reinterpret_cast<uintptr_t>(A) % 16 != 0) cfg.stage_a = 1;
        if (reinterpret_cast<uintptr_t>(B) % 16 != 0) cfg.stage_b = 1;
    }

    // Geometry of the operands as [batches][rows][cols].
    const int64_t bt = ep.batch;
    const bool kn = ep.b_layout == GEMM_B_KN;
    const int64_t a_rows = p.M, a_cols = p.K, a_bat = (bt == 1 || ep.stride_a == 0) ? 1 : bt;
    const int64_t b_rows = kn ? p.K : p.N, b_cols = kn ? p.N : p.K;
    const int64_t b_bat = (bt == 1 || ep.stride_b == 0) ? 1 : bt;
    const int64_t pad = 16 / esz;
    const int64_t lda_s = round_up(a_cols > 0 ? a_cols : 1, pad);
    const int64_t ldb_s = round_up(b_cols > 0 ? b_cols : 1, pad);
    const size_t a_bytes = cfg.stage_a ? static_cast<size_t>(round_up(a_bat * a_rows * lda_s * esz, 256)) : 0;
    const size_t b_bytes = cfg.stage_b ? static_cast<size_t>(round_up(b_bat * b_rows * ldb_s * esz, 256)) : 0;
    if (kStatusBytes + a_bytes + b_bytes > kScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned* status = static_cast<unsigned*>(scratch);
    cudaError_t ce = cudaMemsetAsync(status, 0, sizeof(unsigned), st);
    if (ce != cudaSuccess) return status_of(ce);

    const int osz = dtype_size(ep.out_dtype);
    EpiParams e{};
    e.C = C;
    e.ldc = p.ldc;
    e.stride_c = bt > 1 ? ep.stride_c : 0;
    e.bias = static_cast<const float*>(bias);
    e.R = static_cast<const float*>(residual);
    e.ldr = ep.ldr;
    e.stride_r = bt > 1 ? ep.stride_r : 0;
    e.M = p.M;
    e.N = p.N;
    e.alpha = alpha;
    e.beta = ep.beta;
    e.out_dtype = ep.out_dtype;
    e.act = ep.act;
    const uintptr_t cvec = static_cast<uintptr_t>(4 * osz);
    e.c_vec = (reinterpret_cast<uintptr_t>(C) % cvec == 0) && ((p.ldc * osz) % cvec == 0) &&
              (bt == 1 || (e.stride_c * osz) % cvec == 0);
    e.r_vec = residual && (reinterpret_cast<uintptr_t>(residual) % 16 == 0) && (ep.ldr % 4 == 0) &&
              (bt == 1 || e.stride_r % 4 == 0);

    LaunchCtx lc{};
    lc.status = status;
    lc.timeout_ns = static_cast<uint64_t>(ep.timeout_ms) * 1000000ull;
    lc.flags = ep.flags;
    lc.num_sms = sms;
    lc.stream = st;
    Shape s{p.M, p.N, p.K, bt, 1, 1};

    if (cfg.kernel == GEMM_KERNEL_SKINNY) {
        SkinnyArgs a{};
        a.A = A;
        a.B = B;
        a.lda = p.lda;
        a.ldb = p.ldb;
        a.stride_a = bt > 1 ? ep.stride_a : 0;
        a.stride_b = bt > 1 ? ep.stride_b : 0;
        a.dtype = p.dtype;
        a.b_layout = ep.b_layout;
        return status_of(launch_skinny(cfg, a, s, e, lc));
    }
    if (ffma_small(cfg))
        return status_of(launch_ffma_small(static_cast<const float*>(A),
                                           static_cast<const float*>(B), p.lda, p.ldb,
                                           bt > 1 ? ep.stride_a : 0, bt > 1 ? ep.stride_b : 0,
                                           ep.b_layout, s, e, st));

    const void* a_src = A;
    const void* b_src = B;
    int64_t la = p.lda, lb = p.ldb, sa = ep.stride_a, sb = ep.stride_b;
    unsigned char* base = static_cast<unsigned char*>(scratch) + kStatusBytes;
    if (cfg.stage_a) {
        ce = launch_stage_copy(A, a_rows, a_cols, p.lda, ep.stride_a, a_bat, esz, base, lda_s, st);
        if (ce != cudaSuccess) return status_of(ce);
        a_src = base;
        la = lda_s;
        sa = a_rows * lda_s;
    }
    if (cfg.stage_b) {
        void* dst = base + a_bytes;
        ce = launch_stage_copy(B, b_rows, b_cols, p.ldb, ep.stride_b, b_bat, esz, dst, ldb_s, st);
        if (ce != cudaSuccess) return status_of(ce);
        b_src = dst;
        lb = ldb_s;
        sb = b_rows * ldb_s;
    }
    s.a_bmul = a_bat > 1 ? 1 : 0;
    s.b_bmul = b_bat > 1 ? 1 : 0;

    CUtensorMap mA, mB;
    if (cfg.kernel == GEMM_KERNEL_TC) {
        rc = noalloc_encode(&mA, p.dtype, a_src, a_cols, a_rows, la, a_bat, sa, 64, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc == GEMM_OK)
            rc = noalloc_encode(&mB, p.dtype, b_src, b_cols, b_rows, lb, b_bat, sb, 64,
                                kn ? 64u : static_cast<uint32_t>(tc_b_box_rows(cfg)),
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != GEMM_OK) return rc;
        return status_of(launch_tc(cfg, p.dtype, ep.b_layout, mA, mB, nullptr, s, e, lc));
    }
    rc = noalloc_encode(&mA, p.dtype, a_src, a_cols, a_rows, la, a_bat, sa, 32, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == GEMM_OK)
        rc = kn ? noalloc_encode(&mB, p.dtype, b_src, b_cols, b_rows, lb, b_bat, sb,
                                 static_cast<uint32_t>(cfg.bn), 32, CU_TENSOR_MAP_SWIZZLE_NONE)
                : noalloc_encode(&mB, p.dtype, b_src, b_cols, b_rows, lb, b_bat, sb, 32, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != GEMM_OK) return rc;
    return status_of(launch_ffma(cfg, ep.b_layout, mA, mB, s, e, lc));
}
