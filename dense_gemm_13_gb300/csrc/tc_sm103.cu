// tc_sm103.cu -- BF16/FP16 GEMM on the 5th-generation tensor cores (tcgen05).
//
// The "DeepGEMM" page (sec. 3.3) moves the inner product from FFMA onto the
// GPU's matrix unit once the operands are laid out the way the unit wants
// them, keeps FP32 accumulation (sec. 3.4) and fuses the epilogue (sec. 1.2).
// On sm_103a that unit is driven by a single thread through tcgen05.mma with
// its accumulator in Tensor Memory, so the kernel is organised around it:
//
//   warp 0      TMA producer: 128-byte-swizzled A / B boxes into a STAGES-deep
//               shared-memory ring; mbarrier full[s] counts the bytes in.
//   warp 1      allocates TMEM (2 x BN columns: double-buffered accumulator),
//               one lane issues tcgen05.mma (128 x BN x 16 per instruction)
//               and tcgen05.commit, which frees ring stages (empty[s]) and
//               hands finished accumulators to the epilogue (tfull[buf]).
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, apply
//               alpha / bias / activation / residual / cast, store C once,
//               release the accumulator buffer (tempty[buf]).
//
// The grid is persistent (one CTA per SM); CTA c walks tiles c, c+grid, ...
// in a grouped raster order.  The double-buffered accumulator lets the
// epilogue of tile t overlap the main loop of tile t+1.  Out-of-range rows,
// columns and K arrive from TMA as zeros, so the main loop has no edge code.
//
// B comes in two layouts: NK ([N,K], K contiguous, "K-major") is loaded like
// A; KN ([K,N], N contiguous, "MN-major") is loaded as BN/64 boxes of
// 64 K-rows x 64 N-columns and described to the MMA as an MN-major operand.
//
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains its own copies
// and MMAs, frees TMEM and exits, and the plan's status word records it.
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g13 {
namespace {

constexpr int TBM = 128, TBK = 64, TTHREADS = 192;
constexpr int T_A_BYTES = TBM * TBK * 2;  // 16 KB: 128 rows x 128 B

template <int BN>
struct TcLayout {
    static constexpr int B_BYTES = BN * TBK * 2;  // BN x 128 B
    static constexpr int STAGE_BYTES = T_A_BYTES + B_BYTES;
};

struct TcArgs {
    int64_t M, N, K, batch;
    int a_bmul, b_bmul;
    int64_t m_tiles, n_tiles, tiles_per_batch, total_tiles;
    int k_blocks;
    int raster;
    uint32_t idesc;
    EpiParams e;
    unsigned* status;
    uint64_t timeout_ns;
    uint32_t flags;
};

template <int BN, int STAGES>
__host__ __device__ constexpr int tc_bar_off() {
    return STAGES * TcLayout<BN>::STAGE_BYTES;
}
template <int BN, int STAGES>
__host__ __device__ constexpr int tc_smem_total() {
    // ring + full/empty per stage + tfull/tempty x2 + drain + tmem slot + abort flag
    return 1024 + tc_bar_off<BN, STAGES>() + (2 * STAGES + 5) * 8 + 16;
}

__device__ __forceinline__ void tc_tile_coords(int64_t t, const TcArgs& a, int64_t& b, int64_t& mt,
                                               int64_t& nt) {
    b = t / a.tiles_per_batch;
    const int64_t r = t - b * a.tiles_per_batch;
    const int64_t span = static_cast<int64_t>(a.raster) * a.n_tiles;
    const int64_t g = r / span;
    const int64_t first = g * a.raster;
    const int64_t gm = min(static_cast<int64_t>(a.raster), a.m_tiles - first);
    const int64_t w = r - g * span;
    mt = first + w % gm;
    nt = w / gm;
}

__device__ __forceinline__ void tc_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return;
}

template <int BN, int STAGES, bool B_KN>
__global__ void __launch_bounds__(TTHREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcArgs args) {
    using L = TcLayout<BN>;
    constexpr uint32_t TMEM_COLS = 2 * BN;  // 256 or 512: powers of two
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + tc_bar_off<BN, STAGES>());
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), 128);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint64_t tmo = args.timeout_ns;
    const int kb_total = args.k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const bool stall = (args.flags & GEMM_FLAG_TEST_STALL) && blockIdx.x == 0;
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;  // per stage: armed and not yet seen consumed
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < args.total_tiles; t += gridDim.x) {
                int64_t b, mt, nt;
                tc_tile_coords(t, args, b, mt, nt);
                const int32_t m0 = static_cast<int32_t>(mt * TBM);
                const int32_t n0 = static_cast<int32_t>(nt * BN);
                for (int kb = 0; kb < kb_total; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, args.status,
                                           tmo)) {
                        ok = false;
                        break;
                    }
                    armed &= ~(1u << s);  // the previous use of this stage was consumed
                    const bool skip = stall && t == blockIdx.x && kb == 0;
                    if (!skip) {
                        const uint32_t bar = smem_u32(&full[s]);
                        uint8_t* sa = smem + s * L::STAGE_BYTES;
                        uint8_t* sb = sa + T_A_BYTES;
                        mbar_arrive_expect_tx(bar, L::STAGE_BYTES);
                        const int32_t ba = static_cast<int32_t>(b * args.a_bmul);
                        const int32_t bb = static_cast<int32_t>(b * args.b_bmul);
                        tma_load_3d(smem_u32(sa), &tmA, bar, kb * TBK, m0, ba);
                        if (B_KN) {
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                tma_load_3d(smem_u32(sb + j * (64 * 128)), &tmB, bar, n0 + 64 * j,
                                            kb * TBK, bb);
                        } else {
                            tma_load_3d(smem_u32(sb), &tmB, bar, kb * TBK, n0, bb);
                        }
                        armed |= 1u << s;
                        armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let our own copies land before the CTA's shared memory goes away.
                for (int i = 0; i < STAGES; ++i)
                    if (armed & (1u << i)) tc_drain(smem_u32(&full[i]), (armed_par >> i) & 1u, tmo);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            bool issued_any = false;
            int lt = 0;
            for (int64_t t = blockIdx.x; ok && t < args.total_tiles; t += gridDim.x, ++lt) {
                const int buf = lt & 1;
                const uint32_t tph = static_cast<uint32_t>(lt >> 1) & 1u;
                if (!mbar_wait_bounded(smem_u32(&tempty[buf]), tph ^ 1u, abort_flag, args.status,
                                       tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                for (int kb = 0; kb < kb_total; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, args.status, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * L::STAGE_BYTES);
                    const uint32_t sb = sa + T_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TBK / 16; ++kk) {
                        // A: K-major, rows of 128 B, 8-row swizzle atoms 1024 B apart;
                        // a K step of 16 elements is 32 B inside the swizzled row.
                        const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                        uint64_t bdesc;
                        if (B_KN) {
                            // MN-major: 64-column panels 8 KB apart (leading offset),
                            // 8-row K groups 1024 B apart (stride offset); a K step of
                            // 16 rows is 2 KB.
                            bdesc = smem_desc_sw128(sb + kk * 2048, 64 * 128, 1024);
                        } else {
                            bdesc = smem_desc_sw128(sb + kk * 32, 16, 1024);
                        }
                        tc_mma_f16(d_tmem, adesc, bdesc, args.idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    tc_commit(smem_u32(&empty[s]));  // stage s is free once these MMAs finish
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(smem_u32(&tfull[buf]));  // accumulator ready for the epilogue
            }
            if (!ok && issued_any) {
                // Wait for every MMA already issued before TMEM is released.
                tc_commit(smem_u32(drain));
                tc_drain(smem_u32(drain), 0u, tmo);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue warps
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        int lt = 0;
        for (int64_t t = blockIdx.x; t < args.total_tiles; t += gridDim.x, ++lt) {
            const int buf = lt & 1;
            const uint32_t tph = static_cast<uint32_t>(lt >> 1) & 1u;
            if (!mbar_wait_bounded(smem_u32(&tfull[buf]), tph, abort_flag, args.status, tmo)) break;
            tc_fence_after();
            int64_t b, mt, nt;
            tc_tile_coords(t, args, b, mt, nt);
            const int64_t row = mt * TBM + q * 32 + lane;
            const int64_t col0 = nt * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(buf * BN + c * 32),
                                   r);
                tmem_ld_wait();
                if (c == BN / 32 - 1) {
                    // All of this buffer is in registers: hand it back to the MMA warp.
                    tc_fence_before();
                    mbar_arrive(smem_u32(&tempty[buf]));
                }
                if (col0 + c * 32 < args.e.N) {
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        epi_store4(args.e, b, row, col0 + c * 32 + 4 * g,
                                   __uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                   __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, int STAGES, bool B_KN>
cudaError_t launch_tc_t(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                        const LaunchCtx& lc) {
    TcArgs a{};
    a.M = s.M;
    a.N = s.N;
    a.K = s.K;
    a.batch = s.batch;
    a.a_bmul = s.a_bmul;
    a.b_bmul = s.b_bmul;
    a.m_tiles = (s.M + TBM - 1) / TBM;
    a.n_tiles = (s.N + BN - 1) / BN;
    a.tiles_per_batch = a.m_tiles * a.n_tiles;
    a.total_tiles = a.tiles_per_batch * s.batch;
    a.k_blocks = static_cast<int>((s.K + TBK - 1) / TBK);
    a.raster = cfg.raster_group > 0 ? cfg.raster_group : 16;
    // Instruction descriptor, kind::f16: D = F32 (bits 4-5 = 1); A and B type
    // (bits 7-9, 10-12) 0 = F16, 1 = BF16; A K-major (bit 15 = 0); B K-major
    // (bit 16 = 0) or MN-major (1); N >> 3 at bits 17-22; M >> 4 at bits 24-28.
    const uint32_t ab = dtype == GEMM_BF16 ? 1u : 0u;
    a.idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((B_KN ? 1u : 0u) << 16) |
              (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(TBM >> 4) << 24);
    a.e = e;
    a.status = lc.status;
    a.timeout_ns = lc.timeout_ns;
    a.flags = lc.flags;
    const int smem = tc_smem_total<BN, STAGES>();
    auto kern = tc_gemm_kernel<BN, STAGES, B_KN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    int64_t grid = cfg.num_ctas > 0 ? cfg.num_ctas : lc.num_sms;
    if (grid > a.total_tiles) grid = a.total_tiles;
    if (grid < 1) grid = 1;
    kern<<<static_cast<unsigned>(grid), TTHREADS, smem, lc.stream>>>(tmA, tmB, a);
    return cudaGetLastError();
}

template <bool B_KN>
cudaError_t launch_tc_layout(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                             const LaunchCtx& lc) {
    if (cfg.bn == 256 && cfg.stages == 4)
        return launch_tc_t<256, 4, B_KN>(cfg, dtype, tmA, tmB, s, e, lc);
    if (cfg.bn == 256 && cfg.stages == 3)
        return launch_tc_t<256, 3, B_KN>(cfg, dtype, tmA, tmB, s, e, lc);
    if (cfg.bn == 128 && cfg.stages == 6)
        return launch_tc_t<128, 6, B_KN>(cfg, dtype, tmA, tmB, s, e, lc);
    if (cfg.bn == 128 && cfg.stages == 4)
        return launch_tc_t<128, 4, B_KN>(cfg, dtype, tmA, tmB, s, e, lc);
    return cudaErrorInvalidValue;
}

}  // namespace

size_t tc_smem_bytes(const gemm_config_t& cfg) {
    if (cfg.bm != TBM || cfg.bk != TBK) return 0;
    if (cfg.bn == 256 && cfg.stages == 4) return tc_smem_total<256, 4>();
    if (cfg.bn == 256 && cfg.stages == 3) return tc_smem_total<256, 3>();
    if (cfg.bn == 128 && cfg.stages == 6) return tc_smem_total<128, 6>();
    if (cfg.bn == 128 && cfg.stages == 4) return tc_smem_total<128, 4>();
    return 0;
}

cudaError_t launch_tc(const gemm_config_t& cfg, int dtype, int b_layout, const CUtensorMap& tmA,
                      const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                      const LaunchCtx& lc) {
    if (b_layout == GEMM_B_KN) return launch_tc_layout<true>(cfg, dtype, tmA, tmB, s, e, lc);
    return launch_tc_layout<false>(cfg, dtype, tmA, tmB, s, e, lc);
}

}  // namespace g13
