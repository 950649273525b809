// capi.cpp -- the extern "C" boundary: plans, runs, status, cache queries.
//
// A plan holds the validated problem, its tile configuration, a 4-byte device
// status word (device-side timeouts), an optional staging workspace, and a
// small cache of TMA descriptors keyed by the operand pointers of the last
// run.  gemm_run encodes descriptors only when the pointers change, stages
// misaligned operands, and launches the chosen kernel on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>

#include "dispatch.h"
#include "gemm13.h"
#include "internal.h"

using namespace g13;

namespace {

constexpr uint64_t kPlanMagic = 0x67656d6d31335f70ull;  // "gemm13_p"

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool log_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("GEMM_LOG");
        return v && v[0] && v[0] != '0';
    }();
    return on;
}

}  // namespace

struct gemm_plan_s {
    uint64_t magic = kPlanMagic;
    Problem p{};
    gemm_config_t cfg{};
    int device = 0;
    int num_sms = 0;
    bool cache_hit = false;
    unsigned* d_status = nullptr;
    void* d_ws = nullptr;
    size_t ws_bytes = 0;
    size_t ws_b_off = 0;
    int64_t lda_s = 0, ldb_s = 0;        // leading dims of the staged copies
    int64_t stride_as = 0, stride_bs = 0;
    size_t sk_off = 0, sk_tags_off = 0;   // stream-K / split-K partial slots and tags in d_ws
    size_t sk_ctr_bytes = 0;              // skinny split-K arrival counters
    size_t sk_tag_bytes = 0;              // stream-K tags (zeroed once)
    int64_t sk_grid = 0;
    size_t t3_a_off = 0, t3_b_off = 0;    // 3xTF32 split buffers [batch][hi, lo][rows][t3_ld]
    int64_t t3_ld = 0;
    std::atomic<unsigned> epoch{0};       // tag counter for stream-K launches
    std::mutex mu;                        // guards the descriptor cache
    const void* mapA_src = nullptr;
    const void* mapB_src = nullptr;
    CUtensorMap mapA{}, mapB{};
    const void* mapC_dst = nullptr;       // tensor-core epilogue descriptors (C, residual)
    const void* mapR_src = nullptr;
    bool epi_valid = false;
    TcEpiMaps epi{};
    bool split_map_valid = false;         // split-K partial-slab descriptor (workspace)
    TcEpiMaps split_map{};
};

namespace {

std::mutex g_live_mu;
std::unordered_set<const gemm_plan_s*> g_live;

bool plan_alive(const gemm_plan_s* p) {
    if (!p) return false;
    std::lock_guard<std::mutex> lk(g_live_mu);
    return g_live.count(p) != 0;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Staged copy geometry for one operand: rows x cols per batch entry.
struct OperandGeom {
    int64_t rows, cols, ld, bstride, batches;  // batches = 1 if shared
};

OperandGeom geom_a(const Problem& p) {
    const int64_t bt = p.epi.batch;
    const bool shared = bt == 1 || p.epi.stride_a == 0;
    return {p.M, p.K, p.lda, p.epi.stride_a, shared ? 1 : bt};
}

OperandGeom geom_b(const Problem& p) {
    const int64_t bt = p.epi.batch;
    const bool shared = bt == 1 || p.epi.stride_b == 0;
    const bool kn = p.epi.b_layout == GEMM_B_KN;
    return {kn ? p.K : p.N, kn ? p.N : p.K, p.ldb, p.epi.stride_b, shared ? 1 : bt};
}

int map_cuda_error(cudaError_t e) {
    if (e == cudaSuccess) return GEMM_OK;
    if (e == cudaErrorMemoryAllocation) return GEMM_ERR_OUT_OF_MEMORY;
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ||
        e == cudaErrorNoKernelImageForDevice)
        return GEMM_ERR_NO_DEVICE;
    return GEMM_ERR_CUDA;
}

// Encodes a 3-D tiled descriptor: dims innermost first (cols, rows, batches).
int encode(CUtensorMap* m, int dtype, const void* base, int64_t cols, int64_t rows, int64_t ld,
           int64_t batches, int64_t bstride, uint32_t box_cols, uint32_t box_rows,
           CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return GEMM_ERR_NO_DEVICE;
    const int esz = dtype_size(dtype);
    CUtensorMapDataType t = dtype == GEMM_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                            : dtype == GEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batches)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * esz),
                             static_cast<cuuint64_t>((batches > 1 ? bstride : rows * ld) * esz)};
    if (strides[1] == 0) strides[1] = strides[0];
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, t, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

int g13::tmap_encode_3d(CUtensorMap* m, int dtype, const void* base, int64_t cols, int64_t rows,
                        int64_t ld, int64_t batches, int64_t bstride, uint32_t box_cols,
                        uint32_t box_rows) {
    return encode(m, dtype, base, cols, rows, ld, batches, bstride, box_cols, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

namespace {

bool cfg_is_split_skinny(const gemm_config_t& c) {
    return c.kernel == GEMM_KERNEL_SKINNY && c.split_k > 1;
}

int tc_splits_of(const gemm_plan_s* pl) {
    return pl->cfg.kernel == GEMM_KERNEL_TC ? tc_effective_splits(pl->p.K, pl->cfg.split_k) : 1;
}

int kernels_per_run(const gemm_plan_s* pl) {
    const Problem& p = pl->p;
    if (p.M == 0 || p.N == 0) return 0;
    if (pl->cfg.kernel == GEMM_KERNEL_SKINNY) return 1;
    if (pl->cfg.kernel == GEMM_KERNEL_TF32X3) return 3;  // split A, split B, GEMM
    return 1 + (pl->cfg.stage_a ? 1 : 0) + (pl->cfg.stage_b ? 1 : 0) +
           (tc_splits_of(pl) > 1 ? 1 : 0);
}

int make_plan(const Problem& p, const gemm_config_t* forced, gemm_plan_t* out_plan) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return GEMM_ERR_NO_DEVICE;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;

    gemm_config_t cfg;
    bool hit = false;
    int rc = forced ? check_config(p, *forced, &cfg) : cached_config(p, sms, &cfg, &hit);
    if (rc != GEMM_OK) return rc;
    if (cfg.kernel == GEMM_KERNEL_TC && tc_smem_bytes(cfg) == 0) return GEMM_ERR_UNSUPPORTED;
    if (cfg.kernel == GEMM_KERNEL_TF32X3 && tc3_smem_bytes(cfg) == 0) return GEMM_ERR_UNSUPPORTED;
    if (cfg.kernel == GEMM_KERNEL_FFMA && ffma_smem_bytes(cfg) == 0) return GEMM_ERR_UNSUPPORTED;
    if (cfg.kernel == GEMM_KERNEL_FFMA &&
        !ffma_units_ok(Shape{p.M, p.N, p.K, p.epi.batch, 1, 1}, cfg.bn))
        return GEMM_ERR_UNSUPPORTED;

    gemm_plan_s* pl = new (std::nothrow) gemm_plan_s();
    if (!pl) return GEMM_ERR_OUT_OF_MEMORY;
    pl->p = p;
    pl->cfg = cfg;
    pl->device = dev;
    pl->num_sms = sms;
    pl->cache_hit = hit;

    // Staging workspace: aligned, row-padded copies of misaligned operands.
    const int esz = dtype_size(p.dtype);
    const int64_t pad = 16 / esz;
    size_t ws = 0;
    if (cfg.stage_a) {
        const OperandGeom g = geom_a(p);
        pl->lda_s = round_up(std::max<int64_t>(g.cols, 1), pad);
        pl->stride_as = g.rows * pl->lda_s;
        ws += static_cast<size_t>(round_up(g.batches * pl->stride_as * esz, 256));
    }
    pl->ws_b_off = ws;
    if (cfg.stage_b) {
        const OperandGeom g = geom_b(p);
        pl->ldb_s = round_up(std::max<int64_t>(g.cols, 1), pad);
        pl->stride_bs = g.rows * pl->ldb_s;
        ws += static_cast<size_t>(round_up(g.batches * pl->stride_bs * esz, 256));
    }
    if (cfg.kernel == GEMM_KERNEL_TF32X3) {
        // hi / lo TF32 parts of A ([M][K]) and of B as [N][K], rows padded to 16 bytes
        pl->t3_ld = round_up(std::max<int64_t>(p.K, 1), 4);
        pl->t3_a_off = ws;
        ws += static_cast<size_t>(round_up(geom_a(p).batches * 2 * p.M * pl->t3_ld * 4, 256));
        pl->t3_b_off = ws;
        ws += static_cast<size_t>(round_up(geom_b(p).batches * 2 * p.N * pl->t3_ld * 4, 256));
    }
    if (cfg.kernel == GEMM_KERNEL_TC && tc_effective_splits(p.K, cfg.split_k) > 1) {
        // split-K partial slabs: [batch][splits][M][N] FP32
        pl->sk_off = ws;
        ws += static_cast<size_t>(round_up(
            p.epi.batch * tc_effective_splits(p.K, cfg.split_k) * p.M * p.N * 4, 256));
    }
    if (cfg.kernel == GEMM_KERNEL_SKINNY && cfg.variant == SKINNY_VARIANT_TMA) {
        // TMA skinny kernel: two partial-sum slots per SM for blocks cut between
        // CTAs, then one arrival counter per (batch, block) -- at most batch x Q --
        // zeroed here and reset by the kernel that consumes them
        int64_t P, Q;
        int dot;
        skinny_geometry(p.M, p.N, p.epi.b_layout, &P, &Q, &dot);
        pl->sk_off = ws;
        ws += static_cast<size_t>(round_up(static_cast<int64_t>(skinny_tma_workspace_bytes(sms)), 256));
        pl->sk_tags_off = ws;
        pl->sk_ctr_bytes = static_cast<size_t>(round_up(p.epi.batch * Q * 4, 256));
        ws += pl->sk_ctr_bytes;
    } else if (cfg.kernel == GEMM_KERNEL_SKINNY && cfg.split_k > 1) {
        // split-K partial sums [batch][split_k][P][Q] FP32, then one arrival
        // counter per output group (at most batch x Q), zeroed here and reset
        // by the kernel that consumes them
        int64_t P, Q;
        int dot;
        skinny_geometry(p.M, p.N, p.epi.b_layout, &P, &Q, &dot);
        pl->sk_off = ws;
        ws += static_cast<size_t>(round_up(p.epi.batch * cfg.split_k * P * Q * 4, 256));
        pl->sk_tags_off = ws;
        pl->sk_ctr_bytes = static_cast<size_t>(round_up(p.epi.batch * Q * 4, 256));
        ws += pl->sk_ctr_bytes;
    }
    if (cfg.kernel == GEMM_KERNEL_TC && cfg.stream_k) {
        // Stream-K on the tensor cores: one 128-row x BN partial-sum slot and
        // eight tags (one per epilogue warp) per CTA of the persistent grid.
        int64_t grid = sms;
        if (cfg.num_ctas > 0 && cfg.num_ctas < grid) grid = cfg.num_ctas;
        pl->sk_grid = grid;
        pl->sk_off = ws;
        ws += static_cast<size_t>(grid) * 128 * static_cast<size_t>(cfg.bn) * 4;
        pl->sk_tags_off = ws;
        pl->sk_tag_bytes = static_cast<size_t>(grid) * 8 * 4;
        ws += static_cast<size_t>(round_up(grid * 8 * 4, 256));
    }
    if (cfg.kernel == GEMM_KERNEL_FFMA && cfg.stream_k) {
        // Persistent grid: every CTA the device can hold at once (the launch is
        // cooperative), and one 64 KB partial-sum slot plus a tag per CTA.
        const int per_sm = ffma_ctas_per_sm(cfg, p.epi.b_layout);
        if (per_sm <= 0) {
            delete pl;
            return GEMM_ERR_CUDA;
        }
        int64_t grid = static_cast<int64_t>(per_sm) * sms;
        if (cfg.num_ctas > 0 && cfg.num_ctas < grid) grid = cfg.num_ctas;
        pl->sk_grid = grid;
        pl->sk_off = ws;
        ws += static_cast<size_t>(grid) * ffma_partial_slot_bytes(cfg);
        pl->sk_tags_off = ws;
        pl->sk_tag_bytes = static_cast<size_t>(grid) * 4;
        ws += static_cast<size_t>(round_up(grid * 4, 256));
    }
    ce = cudaMalloc(reinterpret_cast<void**>(&pl->d_status), sizeof(unsigned));
    if (ce == cudaSuccess) ce = cudaMemset(pl->d_status, 0, sizeof(unsigned));
    if (ce == cudaSuccess && ws > 0) ce = cudaMalloc(&pl->d_ws, ws);
    if (ce == cudaSuccess && pl->sk_tag_bytes > 0)
        ce = cudaMemset(static_cast<char*>(pl->d_ws) + pl->sk_tags_off, 0, pl->sk_tag_bytes);
    if (ce == cudaSuccess && pl->sk_ctr_bytes > 0)
        ce = cudaMemset(static_cast<char*>(pl->d_ws) + pl->sk_tags_off, 0, pl->sk_ctr_bytes);
    if (ce != cudaSuccess) {
        if (pl->d_status) cudaFree(pl->d_status);
        delete pl;
        return map_cuda_error(ce);
    }
    pl->ws_bytes = ws;
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        g_live.insert(pl);
    }
    if (log_enabled())
        std::fprintf(stderr,
                     "[gemm13] plan dtype=%d M=%lld N=%lld K=%lld batch=%lld layout=%s -> "
                     "kernel=%d tile=%dx%dx%d stages=%d raster=%d stage_a=%d stage_b=%d "
                     "ws=%zu cache=%s\n",
                     p.dtype, (long long)p.M, (long long)p.N, (long long)p.K,
                     (long long)p.epi.batch, p.epi.b_layout == GEMM_B_KN ? "KN" : "NK", cfg.kernel,
                     cfg.bm, cfg.bn, cfg.bk, cfg.stages, cfg.raster_group, cfg.stage_a, cfg.stage_b,
                     ws, forced ? "forced" : (hit ? "hit" : "miss"));
    *out_plan = pl;
    return GEMM_OK;
}

}  // namespace

extern "C" {

void gemm_epilogue_init(gemm_epilogue_t* e) {
    if (!e) return;
    std::memset(e, 0, sizeof(*e));
    e->b_layout = GEMM_B_KN;
    e->out_dtype = GEMM_F32;
    e->act = GEMM_ACT_NONE;
    e->beta = 1.0f;
    e->batch = 1;
}

int gemm_plan(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              int64_t ldc, const gemm_epilogue_t* epilogue, gemm_plan_t* out_plan) {
    if (!out_plan) return GEMM_ERR_INVALID_ARG;
    *out_plan = nullptr;
    Problem p;
    const int rc = make_problem(dtype, M, N, K, lda, ldb, ldc, epilogue, &p);
    if (rc != GEMM_OK) return rc;
    return make_plan(p, nullptr, out_plan);
}

int gemm_plan_with_config(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K, int64_t lda,
                          int64_t ldb, int64_t ldc, const gemm_epilogue_t* epilogue,
                          const gemm_config_t* cfg, gemm_plan_t* out_plan) {
    if (!out_plan || !cfg) return GEMM_ERR_INVALID_ARG;
    *out_plan = nullptr;
    if (cfg->kernel == GEMM_KERNEL_AUTO) return GEMM_ERR_INVALID_ARG;
    Problem p;
    const int rc = make_problem(dtype, M, N, K, lda, ldb, ldc, epilogue, &p);
    if (rc != GEMM_OK) return rc;
    return make_plan(p, cfg, out_plan);
}

int gemm_run(gemm_plan_t plan, const void* A, const void* B, void* C, const void* bias,
             const void* residual, float alpha, void* stream) {
    if (!plan_alive(plan)) return GEMM_ERR_BAD_PLAN;
    const Problem& p = plan->p;
    const gemm_epilogue_t& ep = p.epi;
    if (p.M == 0 || p.N == 0) return GEMM_OK;
    if (!C) return GEMM_ERR_INVALID_ARG;
    if (p.K > 0 && (!A || !B)) return GEMM_ERR_INVALID_ARG;
    if ((ep.has_bias != 0) != (bias != nullptr)) return GEMM_ERR_INVALID_ARG;
    if ((ep.has_residual != 0) != (residual != nullptr)) return GEMM_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device) return GEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int esz = dtype_size(p.dtype);
    const int osz = dtype_size(ep.out_dtype);

    EpiParams e{};
    e.C = C;
    e.ldc = p.ldc;
    e.stride_c = ep.batch > 1 ? ep.stride_c : 0;
    e.bias = static_cast<const float*>(bias);
    e.R = static_cast<const float*>(residual);
    e.ldr = ep.ldr;
    e.stride_r = ep.batch > 1 ? ep.stride_r : 0;
    e.M = p.M;
    e.N = p.N;
    e.alpha = alpha;
    e.beta = ep.beta;
    e.out_dtype = ep.out_dtype;
    e.act = ep.act;
    const uintptr_t cvec_bytes = static_cast<uintptr_t>(4 * osz);
    e.c_vec = (reinterpret_cast<uintptr_t>(C) % cvec_bytes == 0) && ((p.ldc * osz) % cvec_bytes == 0) &&
              (ep.batch == 1 || (e.stride_c * osz) % cvec_bytes == 0);
    e.r_vec = residual && (reinterpret_cast<uintptr_t>(residual) % 16 == 0) && (ep.ldr % 4 == 0) &&
              (ep.batch == 1 || e.stride_r % 4 == 0);

    LaunchCtx lc{};
    lc.status = plan->d_status;
    lc.timeout_ns = static_cast<uint64_t>(ep.timeout_ms) * 1000000ull;
    lc.flags = ep.flags;
    lc.num_sms = plan->num_sms;
    lc.stream = st;
    const bool skinny_ws = cfg_is_split_skinny(plan->cfg) ||
                           (plan->cfg.kernel == GEMM_KERNEL_SKINNY &&
                            plan->cfg.variant == SKINNY_VARIANT_TMA);
    if (skinny_ws || tc_splits_of(plan) > 1)
        lc.sk_partials = reinterpret_cast<float*>(static_cast<char*>(plan->d_ws) + plan->sk_off);
    if (skinny_ws)
        lc.sk_tags = reinterpret_cast<unsigned*>(static_cast<char*>(plan->d_ws) + plan->sk_tags_off);
    if (plan->sk_grid > 0) {
        lc.sk_partials = reinterpret_cast<float*>(static_cast<char*>(plan->d_ws) + plan->sk_off);
        lc.sk_tags = reinterpret_cast<unsigned*>(static_cast<char*>(plan->d_ws) + plan->sk_tags_off);
        lc.sk_grid = plan->sk_grid;
        unsigned ep_tag = plan->epoch.fetch_add(1) + 1;
        if (ep_tag == 0) ep_tag = plan->epoch.fetch_add(1) + 1;  // 0 marks "never written"
        lc.sk_epoch = ep_tag;
    }

    const gemm_config_t& cfg = plan->cfg;
    Shape s{p.M, p.N, p.K, ep.batch, 1, 1};
    cudaError_t ce;

    if (cfg.kernel == GEMM_KERNEL_SKINNY) {
        SkinnyArgs a{};
        a.A = A;
        a.B = B;
        a.lda = p.lda;
        a.ldb = p.ldb;
        a.stride_a = ep.batch > 1 ? ep.stride_a : 0;
        a.stride_b = ep.batch > 1 ? ep.stride_b : 0;
        a.dtype = p.dtype;
        a.b_layout = ep.b_layout;
        // the TMA-streamed kernel when the large operand allows it on this run
        if (cfg.variant == SKINNY_VARIANT_TMA && skinny_tma_aligned(a, s)) {
            // the large operand's descriptor, re-encoded only when its pointer changes
            const void* L = s.M <= s.N ? B : A;
            std::lock_guard<std::mutex> lk(plan->mu);
            if (plan->mapA_src != L) {
                if (skinny_tma_encode(a, s, &plan->mapA) != GEMM_OK) return GEMM_ERR_CUDA;
                plan->mapA_src = L;
            }
            ce = launch_skinny_tma(a, s, e, lc, cfg.num_ctas, plan->mapA);
        } else {
            ce = launch_skinny(cfg, a, s, e, lc);
        }
        return map_cuda_error(ce);
    }
    if (ffma_small(cfg)) {
        ce = launch_ffma_small(static_cast<const float*>(A), static_cast<const float*>(B), p.lda,
                               p.ldb, ep.batch > 1 ? ep.stride_a : 0, ep.batch > 1 ? ep.stride_b : 0,
                               ep.b_layout, s, e, st);
        return map_cuda_error(ce);
    }

    const OperandGeom ga = geom_a(p), gb = geom_b(p);
    CUtensorMap mA, mB;
    if (cfg.kernel == GEMM_KERNEL_TF32X3) {
        // Split both operands into TF32 hi / lo parts (B transposed to [N][K]
        // when it comes as KN), then the tensor-core kernel reads the parts.
        float* wa = reinterpret_cast<float*>(static_cast<char*>(plan->d_ws) + plan->t3_a_off);
        float* wb = reinterpret_cast<float*>(static_cast<char*>(plan->d_ws) + plan->t3_b_off);
        const int64_t ldt = plan->t3_ld;
        ce = launch_tf32_split(static_cast<const float*>(A), ga.rows, ga.cols, ga.ld, ga.bstride,
                               ga.batches, false, wa, ldt, st);
        if (ce == cudaSuccess)
            ce = launch_tf32_split(static_cast<const float*>(B), gb.rows, gb.cols, gb.ld,
                                   gb.bstride, gb.batches, ep.b_layout == GEMM_B_KN, wb, ldt, st);
        if (ce != cudaSuccess) return map_cuda_error(ce);
        lc.pdl = 1;  // the GEMM starts as a programmatic dependent of the split pass
        s.a_bmul = ga.batches > 1 ? 1 : 0;
        s.b_bmul = gb.batches > 1 ? 1 : 0;
        std::lock_guard<std::mutex> lk(plan->mu);
        if (plan->mapA_src != wa) {
            int rc = encode(&plan->mapA, GEMM_F32, wa, p.K, p.M, ldt, 2 * ga.batches, p.M * ldt,
                            32, 128, CU_TENSOR_MAP_SWIZZLE_128B);
            if (rc == GEMM_OK)
                rc = encode(&plan->mapB, GEMM_F32, wb, p.K, p.N, ldt, 2 * gb.batches, p.N * ldt,
                            32, static_cast<uint32_t>(tc_b_box_rows(cfg)),
                            CU_TENSOR_MAP_SWIZZLE_128B);
            if (rc != GEMM_OK) {
                plan->mapA_src = nullptr;
                return rc;
            }
            plan->mapA_src = wa;
        }
        mA = plan->mapA;
        mB = plan->mapB;
    } else {
    // Effective (possibly staged) operands for the TMA kernels.
    const void* a_src = A;
    const void* b_src = B;
    int64_t lda = p.lda, ldb = p.ldb;
    int64_t sa = ga.bstride, sb = gb.bstride;
    if (reinterpret_cast<uintptr_t>(A) % 16 != 0 && !cfg.stage_a) return GEMM_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(B) % 16 != 0 && !cfg.stage_b) return GEMM_ERR_MISALIGNED;
    // The staging copies of both operands go out as one launch.
    StageJob jobs[2];
    int njobs = 0;
    if (cfg.stage_a) {
        jobs[njobs++] = StageJob{A, ga.rows, ga.cols, ga.ld, ga.bstride, ga.batches, plan->d_ws,
                                 plan->lda_s};
        a_src = plan->d_ws;
        lda = plan->lda_s;
        sa = plan->stride_as;
    }
    if (cfg.stage_b) {
        void* dst = static_cast<char*>(plan->d_ws) + plan->ws_b_off;
        jobs[njobs++] = StageJob{B, gb.rows, gb.cols, gb.ld, gb.bstride, gb.batches, dst, plan->ldb_s};
        b_src = dst;
        ldb = plan->ldb_s;
        sb = plan->stride_bs;
    }
    if (njobs) {
        ce = launch_stage_copies(jobs, njobs, esz, st);
        if (ce != cudaSuccess) return map_cuda_error(ce);
        // the tensor-core kernel may start while the copy finishes (it waits for
        // the copy before its first operand load)
        lc.pdl = cfg.kernel == GEMM_KERNEL_TC ? 1 : 0;
    }
    s.a_bmul = ga.batches > 1 ? 1 : 0;
    s.b_bmul = gb.batches > 1 ? 1 : 0;

    {
        std::lock_guard<std::mutex> lk(plan->mu);
        if (plan->mapA_src != a_src || plan->mapB_src != b_src) {
            const bool kn = ep.b_layout == GEMM_B_KN;
            int rc;
            if (cfg.kernel == GEMM_KERNEL_TC) {
                rc = encode(&plan->mapA, p.dtype, a_src, ga.cols, ga.rows, lda, ga.batches, sa, 64,
                            128, CU_TENSOR_MAP_SWIZZLE_128B);
                if (rc == GEMM_OK)
                    // K-major B boxes hold the tile's columns (half of them per CTA of a pair)
                    rc = encode(&plan->mapB, p.dtype, b_src, gb.cols, gb.rows, ldb, gb.batches, sb,
                                64, kn ? 64 : static_cast<uint32_t>(tc_b_box_rows(cfg)),
                                CU_TENSOR_MAP_SWIZZLE_128B);
            } else {
                rc = encode(&plan->mapA, p.dtype, a_src, ga.cols, ga.rows, lda, ga.batches, sa, 32,
                            128, CU_TENSOR_MAP_SWIZZLE_128B);
                if (rc == GEMM_OK)
                    rc = kn ? encode(&plan->mapB, p.dtype, b_src, gb.cols, gb.rows, ldb, gb.batches,
                                     sb, static_cast<uint32_t>(cfg.bn), 32,
                                     CU_TENSOR_MAP_SWIZZLE_NONE)
                            : encode(&plan->mapB, p.dtype, b_src, gb.cols, gb.rows, ldb, gb.batches,
                                     sb, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B);
            }
            if (rc != GEMM_OK) {
                plan->mapA_src = plan->mapB_src = nullptr;
                return rc;
            }
            plan->mapA_src = a_src;
            plan->mapB_src = b_src;
        }
        mA = plan->mapA;
        mB = plan->mapB;
    }
    }
    if (cfg.kernel == GEMM_KERNEL_FFMA) {
        ce = launch_ffma(cfg, ep.b_layout, mA, mB, s, e, lc);
        return map_cuda_error(ce);
    }
    const int splits = tc_splits_of(plan);
    if (splits > 1) {
        // Split-K: the kernel writes raw FP32 partial slabs [batch][split][M][N]
        // (through TMA when N allows it), a second kernel adds them and applies e.
        EpiParams part{};
        part.C = lc.sk_partials;
        part.ldc = p.N;
        part.stride_c = p.M * p.N;
        part.M = p.M;
        part.N = p.N;
        part.alpha = 1.0f;
        part.beta = 0.0f;
        part.out_dtype = GEMM_F32;
        part.act = GEMM_ACT_NONE;
        part.c_vec = p.N % 4 == 0;
        TcEpiMaps pm{};
        bool use_pm = false;
        const int64_t n_tma = p.N / 4 * 4;
        if (p.N % 4 == 0 && n_tma > 0) {
            std::lock_guard<std::mutex> lk(plan->mu);
            if (!plan->split_map_valid) {
                plan->split_map_valid =
                    encode(&plan->split_map.c, GEMM_F32, part.C, n_tma, p.M, p.N,
                           ep.batch * splits, p.M * p.N, 32u, 32u, CU_TENSOR_MAP_SWIZZLE_128B) ==
                    GEMM_OK;
                plan->split_map.n_tma = n_tma;
                plan->split_map.c_bmul = splits;
                plan->split_map.c_smul = 1;
                plan->split_map.r_tma = 0;
            }
            if (plan->split_map_valid) {
                pm = plan->split_map;
                use_pm = true;
            }
        }
        ce = launch_tc(cfg, p.dtype, ep.b_layout, mA, mB, use_pm ? &pm : nullptr, s, part, lc, &e);
        return map_cuda_error(ce);
    }
    // Tensor-core epilogue through TMA when C (and an FP32 residual) allow it:
    // 16-byte-aligned base, row stride and batch stride.
    TcEpiMaps em;
    bool use_em = false;
    {
        const uintptr_t cp = reinterpret_cast<uintptr_t>(C);
        // TMA stores write whole 16-byte pieces of a row, so the descriptor
        // covers the 16-byte-aligned prefix of each row; the kernel writes
        // the remaining < 16 bytes itself.
        const int64_t n_tma = p.N / (16 / osz) * (16 / osz);
        const bool c_ok = cp % 16 == 0 && (p.ldc * osz) % 16 == 0 && n_tma > 0 &&
                          (ep.batch == 1 || (ep.stride_c * osz) % 16 == 0);
        if (c_ok) {
            std::lock_guard<std::mutex> lk(plan->mu);
            if (!plan->epi_valid || plan->mapC_dst != C || plan->mapR_src != residual) {
                TcEpiMaps m{};
                int rc = encode(&m.c, ep.out_dtype, C, n_tma, p.M, p.ldc, ep.batch,
                                ep.stride_c, osz == 4 ? 32u : 64u, 32u, CU_TENSOR_MAP_SWIZZLE_128B);
                m.n_tma = n_tma;
                const uintptr_t rp = reinterpret_cast<uintptr_t>(residual);
                const bool r_shared = ep.batch > 1 && ep.stride_r == 0;
                m.r_tma = residual && osz == 4 && rp % 16 == 0 && (ep.ldr * 4) % 16 == 0 &&
                          (ep.batch == 1 || r_shared || (ep.stride_r * 4) % 16 == 0);
                if (rc == GEMM_OK && m.r_tma)
                    rc = encode(&m.r, GEMM_F32, residual, p.N, p.M, ep.ldr,
                                r_shared ? 1 : ep.batch, ep.stride_r, 32u, 32u,
                                CU_TENSOR_MAP_SWIZZLE_128B);
                m.c_bmul = ep.batch > 1 ? 1 : 0;
                m.c_smul = 0;
                m.r_bmul = (ep.batch > 1 && !r_shared) ? 1 : 0;
                plan->epi_valid = rc == GEMM_OK;
                plan->epi = m;
                plan->mapC_dst = C;
                plan->mapR_src = residual;
            }
            if (plan->epi_valid) {
                em = plan->epi;
                use_em = true;
            }
        }
    }
    if (cfg.kernel == GEMM_KERNEL_TF32X3)
        ce = launch_tc3(cfg, mA, mB, use_em ? &em : nullptr, s, e, lc);
    else
        ce = launch_tc(cfg, p.dtype, ep.b_layout, mA, mB, use_em ? &em : nullptr, s, e, lc);
    return map_cuda_error(ce);
}

int gemm_plan_status(gemm_plan_t plan) {
    if (!plan_alive(plan)) return GEMM_ERR_BAD_PLAN;
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, plan->d_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return (v & 1u) ? GEMM_ERR_DEVICE_TIMEOUT : GEMM_OK;
}

int gemm_plan_info(gemm_plan_t plan, gemm_plan_info_t* out) {
    if (!plan_alive(plan)) return GEMM_ERR_BAD_PLAN;
    if (!out) return GEMM_ERR_INVALID_ARG;
    out->config = plan->cfg;
    out->workspace_bytes = static_cast<int64_t>(plan->ws_bytes);
    out->num_sms = plan->num_sms;
    out->device = plan->device;
    out->cache_hit = plan->cache_hit ? 1 : 0;
    out->kernels_per_run = kernels_per_run(plan);
    return GEMM_OK;
}

void gemm_plan_destroy(gemm_plan_t plan) {
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        if (!plan || !g_live.erase(plan)) return;
    }
    if (plan->d_status) cudaFree(plan->d_status);
    if (plan->d_ws) cudaFree(plan->d_ws);
    plan->magic = 0;
    delete plan;
}

int gemm_select_config(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldc, const gemm_epilogue_t* epilogue, int32_t num_sms,
                       gemm_config_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    Problem p;
    const int rc = make_problem(dtype, M, N, K, lda, ldb, ldc, epilogue, &p);
    if (rc != GEMM_OK) return rc;
    return choose_config(p, num_sms, out);
}

void gemm_cache_stats(int64_t* entries, int64_t* hits, int64_t* misses) {
    cache_stats(entries, hits, misses);
}

void gemm_cache_clear(void) { cache_clear(); }

const char* gemm_strerror(int status) {
    switch (status) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "unsupported configuration";
        case GEMM_ERR_MISALIGNED: return "operand base pointer not 16-byte aligned for this plan";
        case GEMM_ERR_CUDA: return "CUDA call failed";
        case GEMM_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case GEMM_ERR_BAD_PLAN: return "invalid or destroyed plan";
        case GEMM_ERR_NO_DEVICE: return "no usable sm_103 CUDA device";
        case GEMM_ERR_OUT_OF_MEMORY: return "device allocation failed";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "problem needs more than the 64 MiB fixed scratch of gemm_run_noalloc";
        default: return "unknown status";
    }
}

const char* gemm_version(void) { return "gemm13 0.1.0 (sm_103a)"; }

}  // extern "C"
