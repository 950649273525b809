// sgemm_ffma.cu -- FP32 GEMM on the CUDA cores (FFMA), fed by TMA.
//
// The pages' FP32 SGEMM ("SGEMM ... 83% of cuBLAS", sec. 2.1-3.4; "CUDA Tile
// ... GEMM", sec. 4.2-4.4) tiles C per block, per warp and per thread, stages
// A/B tiles in padded shared memory with cp.async double buffering and keeps
// an 8x8 register tile per thread.  On sm_103a the same three-level tiling is
// kept, but the copy engine changes:
//   * one thread issues TMA box loads into a STAGES-deep ring, completion is
//     tracked by mbarrier transaction counts and stages are released by
//     per-warp arrivals (no __syncthreads in the main loop);
//   * A tiles are 128-byte swizzled by the TMA unit instead of padded, so the
//     float4 fragment loads are bank-conflict free and 16-byte aligned;
//   * out-of-range rows/columns/K arrive as zeros from TMA, so there is no
//     edge code in the main loop; the epilogue masks the stores.
// Block tile 128x128x32, 256 threads = 8 warps as 4 (M) x 2 (N); warp tile
// 32x64; lanes 4 x 8; thread tile 8 rows (stride 4) x 8 columns.
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g13 {
namespace {

constexpr int FBM = 128, FBN = 128, FBK = 32, FTHREADS = 256, FWARPS = 8;
constexpr int F_A_BYTES = FBM * FBK * 4;  // 16 KB: 128 rows of 32 floats, 128-byte swizzle
constexpr int F_B_BYTES = FBK * FBN * 4;  // 16 KB
constexpr int F_STAGE_BYTES = F_A_BYTES + F_B_BYTES;

struct FfmaArgs {
    Shape s;
    int64_t m_tiles, n_tiles, tiles_per_batch;
    int raster;
    int k_tiles;
    EpiParams e;
    unsigned* status;
    uint64_t timeout_ns;
    uint32_t flags;
};

template <int STAGES>
__host__ __device__ constexpr int ffma_bar_off() {
    return STAGES * F_STAGE_BYTES;
}
template <int STAGES>
__host__ __device__ constexpr int ffma_smem_total() {
    return 1024 /* alignment slack */ + ffma_bar_off<STAGES>() + 2 * STAGES * 8 + 16;
}

// Grouped rasterisation: `group` M tiles are walked together for each N tile
// so that concurrently running blocks share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int64_t t, int64_t m_tiles, int64_t n_tiles,
                                            int64_t per_batch, int group, int64_t& b,
                                            int64_t& mt, int64_t& nt) {
    b = t / per_batch;
    const int64_t r = t - b * per_batch;
    const int64_t span = static_cast<int64_t>(group) * n_tiles;
    const int64_t g = r / span;
    const int64_t first = g * group;
    const int64_t gm = min(static_cast<int64_t>(group), m_tiles - first);
    const int64_t w = r - g * span;
    mt = first + w % gm;
    nt = w / gm;
}

// Two FP32 lanes in one 64-bit register pair, for the packed fma.rn.f32x2
// (one instruction issues two FMAs, halving the issue slots the FMAs take).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void ffma2(uint64_t& d, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// Waits for a phase without looking at the abort flag (used to drain copies
// already in flight before a CTA gives up).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return;
}

template <int STAGES, bool B_NK, bool PACKED>
__global__ void __launch_bounds__(FTHREADS, 2)
    ffma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const FfmaArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ffma_bar_off<STAGES>());
    uint64_t* empty = full + STAGES;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + STAGES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t b, mt, nt;
    tile_coords(blockIdx.x, args.m_tiles, args.n_tiles, args.tiles_per_batch, args.raster, b, mt,
                nt);
    const int m0 = static_cast<int>(mt * FBM), n0 = static_cast<int>(nt * FBN);
    const int kt_total = args.k_tiles;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), FWARPS);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    __syncthreads();

    const bool stall = (args.flags & GEMM_FLAG_TEST_STALL) && blockIdx.x == 0;
    // Producer state, kept uniform across warp 0 (lane 0 issues): next K tile to load.
    int next_issue = 0;
    auto issue = [&](int kt) {
        const int s = kt % STAGES;
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t* sa = smem + s * F_STAGE_BYTES;
        uint8_t* sb = sa + F_A_BYTES;
        const int32_t ba = static_cast<int32_t>(b * args.s.a_bmul);
        const int32_t bb = static_cast<int32_t>(b * args.s.b_bmul);
        mbar_arrive_expect_tx(bar, F_STAGE_BYTES);
        tma_load_3d(smem_u32(sa), &tmA, bar, kt * FBK, m0, ba);
        if (B_NK)
            tma_load_3d(smem_u32(sb), &tmB, bar, kt * FBK, n0, bb);
        else
            tma_load_3d(smem_u32(sb), &tmB, bar, n0, kt * FBK, bb);
    };
    if (warp == 0) {
        const int pre = min(STAGES, kt_total);
        if (lane == 0)
            for (int kt = 0; kt < pre; ++kt)
                if (!(stall && kt == 0)) issue(kt);
        next_issue = pre;
    }

    const int wm = warp & 3, wn = warp >> 2;
    const int lr = lane >> 3, lc = lane & 7;
    // acc[i][j] (scalar path) or acc2[i][j/2] holding columns (j, j+1) (packed path)
    float acc[8][8];
    uint64_t acc2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[i][j] = 0.0f;
            if (j < 4) acc2[i][j] = 0ull;
        }

    bool ok = true;
    int kt_done = -1;  // last K tile this thread saw complete
    for (int kt = 0; kt < kt_total; ++kt) {
        const int s = kt % STAGES;
        const uint32_t ph = static_cast<uint32_t>(kt / STAGES) & 1u;
        if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, args.status, args.timeout_ns)) {
            ok = false;
            break;
        }
        kt_done = kt;
        const float* As = reinterpret_cast<const float*>(smem + s * F_STAGE_BYTES);
        const float* Bs = reinterpret_cast<const float*>(smem + s * F_STAGE_BYTES + F_A_BYTES);
        if (!B_NK && PACKED) {
#pragma unroll
            for (int kq = 0; kq < FBK / 4; ++kq) {
                float4 a4[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = wm * 32 + lr + 4 * i;
                    a4[i] = *reinterpret_cast<const float4*>(As + row * FBK +
                                                              ((kq ^ (row & 7)) << 2));
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float* brow = Bs + (kq * 4 + kk) * FBN + wn * 64 + lc * 4;
                    const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(brow);
                    const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(brow + 32);
                    const uint64_t bp[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float a = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
                        const uint64_t ap = pack2(a, a);
#pragma unroll
                        for (int jp = 0; jp < 4; ++jp) ffma2(acc2[i][jp], ap, bp[jp]);
                    }
                }
            }
        } else if (!B_NK) {
#pragma unroll
            for (int kq = 0; kq < FBK / 4; ++kq) {
                float4 a4[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = wm * 32 + lr + 4 * i;
                    a4[i] = *reinterpret_cast<const float4*>(As + row * FBK +
                                                              ((kq ^ (row & 7)) << 2));
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float* brow = Bs + (kq * 4 + kk) * FBN + wn * 64 + lc * 4;
                    const float4 b0 = *reinterpret_cast<const float4*>(brow);
                    const float4 b1 = *reinterpret_cast<const float4*>(brow + 32);
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float a = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a, bv[j], acc[i][j]);
                    }
                }
            }
        } else {
            // B tile is [128 n][32 k], 128-byte swizzled like A; two k at a time.
#pragma unroll
            for (int kp = 0; kp < FBK / 2; ++kp) {
                const int kq = kp >> 1, half = (kp & 1) * 2;
                float2 a2[8], b2[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = wm * 32 + lr + 4 * i;
                    a2[i] = *reinterpret_cast<const float2*>(As + row * FBK +
                                                              ((kq ^ (row & 7)) << 2) + half);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int n = wn * 64 + lc + 8 * j;
                    b2[j] = *reinterpret_cast<const float2*>(Bs + n * FBK + ((kq ^ (n & 7)) << 2) +
                                                              half);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc[i][j] = fmaf(a2[i].x, b2[j].x, acc[i][j]);
                        acc[i][j] = fmaf(a2[i].y, b2[j].y, acc[i][j]);
                    }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (warp == 0 && next_issue < kt_total) {
            // Refill this stage once every warp has released it.  The whole
            // warp waits so that it stays converged for the next tile's FFMAs.
            if (!mbar_wait_bounded(smem_u32(&empty[s]), ph, abort_flag, args.status,
                                   args.timeout_ns)) {
                ok = false;
                break;
            }
            if (lane == 0) issue(next_issue);
            __syncwarp();
            ++next_issue;
        }
    }

    if (!ok) {
        // Give up on this tile, but let copies already in flight land first.
        if (tid == 0) {
            for (int kt = kt_done + 1; kt < next_issue; ++kt) {
                if (stall && kt == 0) continue;
                mbar_drain(smem_u32(&full[kt % STAGES]), static_cast<uint32_t>(kt / STAGES) & 1u,
                           args.timeout_ns);
            }
        }
        return;
    }

    // Fused epilogue; C written once.
    const EpiParams& e = args.e;
    if (PACKED) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) unpack2(acc2[i][jp], acc[i][2 * jp], acc[i][2 * jp + 1]);
    }
    if (!B_NK) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = m0 + wm * 32 + lr + 4 * i;
            const int64_t c0 = n0 + wn * 64 + lc * 4;
            epi_store4(e, b, row, c0, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            epi_store4(e, b, row, c0 + 32, acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = m0 + wm * 32 + lr + 4 * i;
#pragma unroll
            for (int j = 0; j < 8; ++j) epi_store1(e, b, row, n0 + wn * 64 + lc + 8 * j, acc[i][j]);
        }
    }
}

template <int STAGES, bool B_NK, bool PACKED>
cudaError_t launch_ffma_t(const gemm_config_t& cfg, const CUtensorMap& tmA,
                          const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                          const LaunchCtx& lc) {
    FfmaArgs a{};
    a.s = s;
    a.m_tiles = (s.M + FBM - 1) / FBM;
    a.n_tiles = (s.N + FBN - 1) / FBN;
    a.tiles_per_batch = a.m_tiles * a.n_tiles;
    a.raster = cfg.raster_group > 0 ? cfg.raster_group : 8;
    a.k_tiles = static_cast<int>((s.K + FBK - 1) / FBK);
    a.e = e;
    a.status = lc.status;
    a.timeout_ns = lc.timeout_ns;
    a.flags = lc.flags;
    const int smem = ffma_smem_total<STAGES>();
    auto kern = ffma_kernel<STAGES, B_NK, PACKED>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const int64_t grid = a.tiles_per_batch * s.batch;
    kern<<<static_cast<unsigned>(grid), FTHREADS, smem, lc.stream>>>(tmA, tmB, a);
    return cudaGetLastError();
}

}  // namespace

size_t ffma_smem_bytes(const gemm_config_t& cfg) {
    switch (cfg.stages) {
        case 2: return ffma_smem_total<2>();
        case 3: return ffma_smem_total<3>();
        case 4: return ffma_smem_total<4>();
        default: return 0;
    }
}

cudaError_t launch_ffma(const gemm_config_t& cfg, int b_layout, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                        const LaunchCtx& lc) {
    const bool nk = b_layout == GEMM_B_NK;
    const bool packed = cfg.variant == 1 && !nk;  // the packed main loop exists for KN only
#define G13_FFMA_CASE(ST)                                                          \
    case ST:                                                                       \
        if (nk) return launch_ffma_t<ST, true, false>(cfg, tmA, tmB, s, e, lc);    \
        if (packed) return launch_ffma_t<ST, false, true>(cfg, tmA, tmB, s, e, lc); \
        return launch_ffma_t<ST, false, false>(cfg, tmA, tmB, s, e, lc);
    switch (cfg.stages) {
        G13_FFMA_CASE(2)
        G13_FFMA_CASE(3)
        G13_FFMA_CASE(4)
        default: return cudaErrorInvalidValue;
    }
#undef G13_FFMA_CASE
}

}  // namespace g13
