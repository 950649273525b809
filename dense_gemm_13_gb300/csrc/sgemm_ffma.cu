// sgemm_ffma.cu -- FP32 GEMM on the CUDA cores (FFMA), fed by TMA.
//
// The pages' FP32 SGEMM ("SGEMM ... 83% of cuBLAS", sec. 2.1-3.4; "CUDA Tile
// ... GEMM", sec. 4.2-4.4) tiles C per block, per warp and per thread, stages
// A/B tiles in padded shared memory with cp.async double buffering and keeps
// an 8x8 register tile per thread.  On sm_103a the same three-level tiling is
// kept, but the copy engine and the schedule change:
//   * one thread issues TMA box loads into a STAGES-deep ring, completion is
//     tracked by mbarrier transaction counts and stages are released by
//     per-warp arrivals (no __syncthreads in the main loop);
//   * A tiles are 128-byte swizzled by the TMA unit instead of padded, so the
//     float4 fragment loads are bank-conflict free and 16-byte aligned;
//   * out-of-range rows/columns/K arrive as zeros from TMA, so there is no
//     edge code in the main loop; the epilogue masks the stores;
//   * the main loop can use Blackwell's packed fma.rn.f32x2 (two FMAs per
//     issue slot), which relieves the issue bottleneck of scalar FFMA;
//   * work is a range of (tile, K-step) units per CTA.  In data-parallel mode
//     each CTA owns one whole tile.  In stream-K mode a persistent grid splits
//     all units evenly, so no wave is left part-empty; a tile cut between CTAs
//     is finished by the CTA holding its first K step, which adds the others'
//     partial sums (left in a per-CTA workspace slot and tagged with this
//     launch's epoch) in CTA order -- the result is deterministic.  Stream-K
//     launches are cooperative, so every CTA it waits for is resident.
// Block tile 128 x BN x 32, 256 threads = 8 warps as 4 (M) x 2 (N); warp tile
// 32 x BN/2; lanes 4 x 8; thread tile 8 rows (stride 4) x BN/16 columns (quads
// of 4 spaced 32 apart).  BN = 128 runs two CTAs per SM; BN = 256 one CTA per
// SM with an 8 x 16 thread tile.  Why the wider tile: a 128-bit shared-memory
// load costs one wavefront per quarter-warp whatever the broadcast, so each
// fragment float a lane loads costs 1/32 of a wavefront; the 8 x 8 tile needs
// 16 fragment floats per 64 FMAs, exactly the shared-memory bandwidth of an SM
// at the FMA rate, while 8 x 16 needs 24 per 128 FMAs (three quarters of it).
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g13 {
namespace {

constexpr int FBM = 128, FBK = 32, FTHREADS = 256, FWARPS = 8;
constexpr int F_A_BYTES = FBM * FBK * 4;  // 16 KB: 128 rows of 32 floats, 128-byte swizzle

template <int BN>
struct FLayout {
    static constexpr int B_BYTES = FBK * BN * 4;  // 16 or 32 KB
    static constexpr int STAGE_BYTES = F_A_BYTES + B_BYTES;
    static constexpr int NQ = BN / 64;            // column quads per thread
};

struct FfmaArgs {
    Shape s;
    int m_tiles, n_tiles, tiles_per_batch;  // the host checks tiles * k_tiles < 2^31
    int raster;
    int k_tiles;
    int units;          // tiles * k_tiles
    int grid;           // CTA c owns units [units*c/grid, units*(c+1)/grid)
    float* partials;    // stream-K: [grid][FBM*BN] partial-sum slots (null otherwise)
    unsigned* tags;     // stream-K: [grid] slot-ready tags
    unsigned epoch;     // tag value of this launch
    EpiParams e;
    unsigned* status;
    uint64_t timeout_ns;
    uint32_t flags;
};

template <int BN, int STAGES>
__host__ __device__ constexpr int ffma_bar_off() {
    return STAGES * FLayout<BN>::STAGE_BYTES;
}
template <int BN, int STAGES>
__host__ __device__ constexpr int ffma_smem_total() {
    return 1024 /* alignment slack */ + ffma_bar_off<BN, STAGES>() + 2 * STAGES * 8 + 16;
}

// Grouped rasterisation: `group` M tiles are walked together for each N tile
// so that concurrently running blocks share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int per_batch,
                                            int group, int& b, int& mt, int& nt) {
    b = t / per_batch;
    const int r = t - b * per_batch;
    const int span = group * n_tiles;
    const int g = r / span;
    const int first = g * group;
    const int gm = min(group, m_tiles - first);
    const int w = r - g * span;
    mt = first + w % gm;
    nt = w / gm;
}

__device__ __forceinline__ int range_begin(const FfmaArgs& a, int c) {
    return static_cast<int>(static_cast<int64_t>(a.units) * c / a.grid);
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

// BN = 128 with row-major B runs two CTAs per SM (128 registers); the K-major
// loop keeps more fragments live and runs one CTA per SM without spilling.
template <int BN, int STAGES, bool B_NK, bool PACKED>
__global__ void __launch_bounds__(FTHREADS, (BN == 128 && !B_NK) ? 2 : 1)
    ffma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const FfmaArgs args) {
    using L = FLayout<BN>;
    constexpr int NQ = L::NQ;
    static_assert(!B_NK || BN == 128, "K-major B is implemented for 128-wide tiles");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ffma_bar_off<BN, STAGES>());
    uint64_t* empty = full + STAGES;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + STAGES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int u_begin = range_begin(args, cta), u_end = range_begin(args, cta + 1);
    const int KT = args.k_tiles;

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

    const bool stall = (args.flags & GEMM_FLAG_TEST_STALL) && cta == 0;
    // Units are handled as offsets r from u_begin.
    const int n_units = u_end - u_begin;
    // TMA loads for unit offset r into stage s (issued by lane 0 of warp 0).
    auto issue = [&](int r, int s) {
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t* sa = smem + s * L::STAGE_BYTES;
        uint8_t* sb = sa + F_A_BYTES;
        const int u = u_begin + r;
        const int tile = u / KT;
        const int k0 = (u - tile * KT) * FBK;
        int b, mt, nt;
        tile_coords(tile, args.m_tiles, args.n_tiles, args.tiles_per_batch, args.raster, b, mt, nt);
        const int m0 = mt * FBM, n0 = nt * BN;
        const int ba = b * args.s.a_bmul, bb = b * args.s.b_bmul;
        mbar_arrive_expect_tx(bar, L::STAGE_BYTES);
        tma_load_3d(smem_u32(sa), &tmA, bar, k0, m0, ba);
        if (B_NK)
            tma_load_3d(smem_u32(sb), &tmB, bar, k0, n0, bb);
        else
            tma_load_3d(smem_u32(sb), &tmB, bar, n0, k0, bb);
    };
    // Producer state, kept uniform across warp 0: offset of the next unit to load.
    int next_issue = min(STAGES, n_units);
    if (warp == 0 && lane == 0)
        for (int r = 0; r < next_issue; ++r)
            if (!(stall && r == 0)) issue(r, r);

    const int wm = warp & 3, wn = warp >> 2;
    const int lr = lane >> 3, lc = lane & 7;
    // acc[i][4q+t]: row i, column quad q (scalar path); acc2[i][2q+h] holds
    // acc[i][4q+2h], acc[i][4q+2h+1] (packed path).
    float acc[8][4 * NQ];
    uint64_t acc2[8][2 * NQ];

    bool ok = true;
    int seen = -1;  // last unit offset whose stage this thread saw arrive
    int stage = 0;
    uint32_t phase = 0;
    int r = 0;
    while (r < n_units) {
        const int tile = (u_begin + r) / KT;
        const int kt0 = u_begin + r - tile * KT;
        const int seg_len = min(n_units - r, KT - kt0);
        const bool first_k = kt0 == 0;               // this segment starts the tile's K loop
        const bool completes = kt0 + seg_len == KT;  // ... and this one ends it
        const int seg_end = r + seg_len;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4 * NQ; ++j) {
                acc[i][j] = 0.0f;
                if (j < 2 * NQ) acc2[i][j] = 0ull;
            }
        for (; r < seg_end; ++r) {
            const int s = stage;
            const uint32_t ph = phase;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if (ok && !mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, args.status,
                                         args.timeout_ns))
                ok = false;
            if (ok) {
                seen = r;
                const float* As = reinterpret_cast<const float*>(smem + s * L::STAGE_BYTES);
                const float* Bs =
                    reinterpret_cast<const float*>(smem + s * L::STAGE_BYTES + F_A_BYTES);
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
                            const float* brow = Bs + (kq * 4 + kk) * BN + wn * (BN / 2) + lc * 4;
                            uint64_t bp[2 * NQ];
#pragma unroll
                            for (int q = 0; q < NQ; ++q) {
                                const ulonglong2 v =
                                    *reinterpret_cast<const ulonglong2*>(brow + 32 * q);
                                bp[2 * q] = v.x;
                                bp[2 * q + 1] = v.y;
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float a = kk == 0   ? a4[i].x
                                                : kk == 1 ? a4[i].y
                                                : kk == 2 ? a4[i].z
                                                          : a4[i].w;
                                const uint64_t ap = pack2(a, a);
#pragma unroll
                                for (int jp = 0; jp < 2 * NQ; ++jp) ffma2(acc2[i][jp], ap, bp[jp]);
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
                            const float* brow = Bs + (kq * 4 + kk) * BN + wn * (BN / 2) + lc * 4;
                            float bv[4 * NQ];
#pragma unroll
                            for (int q = 0; q < NQ; ++q) {
                                const float4 v = *reinterpret_cast<const float4*>(brow + 32 * q);
                                bv[4 * q] = v.x;
                                bv[4 * q + 1] = v.y;
                                bv[4 * q + 2] = v.z;
                                bv[4 * q + 3] = v.w;
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float a = kk == 0   ? a4[i].x
                                                : kk == 1 ? a4[i].y
                                                : kk == 2 ? a4[i].z
                                                          : a4[i].w;
#pragma unroll
                                for (int j = 0; j < 4 * NQ; ++j) acc[i][j] = fmaf(a, bv[j], acc[i][j]);
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
                            a2[i] = *reinterpret_cast<const float2*>(
                                As + row * FBK + ((kq ^ (row & 7)) << 2) + half);
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int n = wn * 64 + lc + 8 * j;
                            b2[j] = *reinterpret_cast<const float2*>(
                                Bs + n * FBK + ((kq ^ (n & 7)) << 2) + half);
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
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (warp == 0 && next_issue < n_units) {
                // Refill this stage (with unit r + STAGES) once every warp has
                // released it.  The whole warp waits so that it stays converged
                // for the next FFMAs.
                if (ok && !mbar_wait_bounded(smem_u32(&empty[s]), ph, abort_flag, args.status,
                                             args.timeout_ns))
                    ok = false;
                if (ok && lane == 0) issue(next_issue, s);
                __syncwarp();
                ++next_issue;
            }
        }
        // Segment end: every thread is here and no wait runs between this
        // barrier and the read of the abort flag, so the decision is uniform.
        __syncthreads();
        if (*abort_flag) {
            ok = false;
            break;
        }
        if (PACKED) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int jp = 0; jp < 2 * NQ; ++jp)
                    unpack2(acc2[i][jp], acc[i][2 * jp], acc[i][2 * jp + 1]);
        }
        // Partial-sum slots hold each thread's 8 * NQ quads at (quad * 256 + tid) * 4.
        if (!first_k) {
            // Contributor: this CTA ran a later K range of a tile that an earlier
            // CTA finishes.  Leave the partial sums in this CTA's slot, tag it.
            float* slot = args.partials + static_cast<int64_t>(cta) * (FBM * BN);
#pragma unroll
            for (int Q = 0; Q < 8 * NQ; ++Q)
                __stcg(reinterpret_cast<float4*>(slot) + Q * FTHREADS + tid,
                       make_float4(acc[Q / NQ][4 * (Q % NQ)], acc[Q / NQ][4 * (Q % NQ) + 1],
                                   acc[Q / NQ][4 * (Q % NQ) + 2], acc[Q / NQ][4 * (Q % NQ) + 3]));
            __threadfence();
            __syncthreads();
            if (tid == 0) st_release_gpu(args.tags + cta, args.epoch);
            continue;
        }
        if (!completes) {
            // Finisher: add the partial sums of the CTAs that ran the rest of
            // this tile's K range, in CTA order.
            const int tile_end = (tile + 1) * KT;
            for (int d = cta + 1; d < args.grid && range_begin(args, d) < tile_end; ++d) {
                if (tid == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(args.tags + d) != args.epoch) {
                        if (*abort_flag) break;
                        if (globaltimer_ns() - t0 > args.timeout_ns) {
                            *abort_flag = 1u;
                            atomicOr(args.status, DEVERR_TIMEOUT);
                            break;
                        }
                    }
                }
                __syncthreads();
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const float* slot = args.partials + static_cast<int64_t>(d) * (FBM * BN);
#pragma unroll
                for (int Q = 0; Q < 8 * NQ; ++Q) {
                    const float4 p =
                        __ldcg(reinterpret_cast<const float4*>(slot) + Q * FTHREADS + tid);
                    acc[Q / NQ][4 * (Q % NQ)] += p.x;
                    acc[Q / NQ][4 * (Q % NQ) + 1] += p.y;
                    acc[Q / NQ][4 * (Q % NQ) + 2] += p.z;
                    acc[Q / NQ][4 * (Q % NQ) + 3] += p.w;
                }
            }
            if (!ok) break;
        }
        // Fused epilogue; C written once.
        int b, mt, nt;
        tile_coords(tile, args.m_tiles, args.n_tiles, args.tiles_per_batch, args.raster, b, mt, nt);
        const int64_t m0 = static_cast<int64_t>(mt) * FBM, n0 = static_cast<int64_t>(nt) * BN;
        const EpiParams& e = args.e;
        // Plain FP32 output of a whole tile (the common case): a compact store
        // sequence.  The general epilogue below is much larger code, and
        // running it once per tile cost ~20 us per tile in instruction fetch
        // (measured per CTA with the global timer), several percent of a 4096^3
        // run.
        const bool plain = !e.bias && e.act == GEMM_ACT_NONE && !e.R &&
                           e.out_dtype == GEMM_F32 && e.c_vec && m0 + FBM <= e.M && n0 + BN <= e.N;
        if (!B_NK && plain) {
            float* cb = static_cast<float*>(e.C) + b * e.stride_c +
                        (m0 + wm * 32 + lr) * e.ldc + n0 + wn * (BN / 2) + lc * 4;
            const int64_t rstep = 4 * e.ldc;
            const float al = e.alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    *reinterpret_cast<float4*>(cb + i * rstep + 32 * q) =
                        make_float4(acc[i][4 * q] * al, acc[i][4 * q + 1] * al,
                                    acc[i][4 * q + 2] * al, acc[i][4 * q + 3] * al);
        } else if (!B_NK) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t row = m0 + wm * 32 + lr + 4 * i;
                const int64_t c0 = n0 + wn * (BN / 2) + lc * 4;
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    epi_store4(e, b, row, c0 + 32 * q, acc[i][4 * q], acc[i][4 * q + 1],
                               acc[i][4 * q + 2], acc[i][4 * q + 3]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t row = m0 + wm * 32 + lr + 4 * i;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    epi_store1(e, b, row, n0 + wn * 64 + lc + 8 * j, acc[i][j]);
            }
        }
    }

    if (!ok && tid == 0) {
        // Give up, but let copies already in flight land first.
        for (int v = seen + 1; v < next_issue; ++v) {
            if (stall && v == 0) continue;
            mbar_drain(smem_u32(&full[v % STAGES]), static_cast<uint32_t>(v / STAGES) & 1u,
                       args.timeout_ns);
        }
    }
}

// Small problems (a few 128-row tiles would leave most SMs idle): 32 x 32
// output tiles, one CTA of 256 threads each, the classic shared-memory tiling
// of the pages ("SGEMM ... 83% of cuBLAS", sec. 3.1-3.4) with a 4-deep ring of
// 32-deep K steps filled by 4-byte cp.async copies three steps ahead (as the
// pages' cp.async double buffering, one step deeper).  The copies land A as
// [k][m] and B as [k][n] (rows padded to 33 floats: conflict-free), each
// thread keeps a 2 x 2 register tile (rows ty, ty + 16; columns tx, tx + 16).
// Any stride and alignment of FP32 data; out-of-range elements arrive as zero.
constexpr int SB = 32;   // tile rows, columns and K step
constexpr int SST = 4;   // K steps in the ring
__global__ void __launch_bounds__(256)
    ffma_small_kernel(const float* __restrict__ A, const float* __restrict__ B, int64_t lda,
                      int64_t ldb, int64_t stride_a, int64_t stride_b, int b_nk, int64_t M,
                      int64_t N, int64_t K, const EpiParams e) {
    __shared__ float As[SST][SB][SB + 1];
    __shared__ float Bs[SST][SB][SB + 1];
    const int tid = threadIdx.x;
    const int64_t bz = blockIdx.z;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * SB, n0 = static_cast<int64_t>(blockIdx.x) * SB;
    const float* Ab = A + bz * stride_a;
    const float* Bb = B + bz * stride_b;
    const int lr = tid >> 3, lc = (tid & 7) * 4;  // copier: row of the tile, 4 consecutive elements
    const int ty = tid >> 4, tx = tid & 15;
    const int64_t nsteps = (K + SB - 1) / SB;
    // copies of K step `step` into ring slot step % SST (zero-filled out of range)
    const auto issue = [&](int64_t step) {
        const int sl = static_cast<int>(step % SST);
        const int64_t k0 = step * SB;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t m = m0 + lr, k = k0 + lc + q;
            const bool in = m < M && k < K;
            cp_async_4(smem_u32(&As[sl][lc + q][lr]), in ? Ab + m * lda + k : A, in);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (!b_nk) {  // B[k][n]: row k0 + lr, columns n0 + lc + q
                const int64_t k = k0 + lr, n = n0 + lc + q;
                const bool in = k < K && n < N;
                cp_async_4(smem_u32(&Bs[sl][lr][lc + q]), in ? Bb + k * ldb + n : B, in);
            } else {      // B[n][k]: row n0 + lr, columns k0 + lc + q
                const int64_t n = n0 + lr, k = k0 + lc + q;
                const bool in = n < N && k < K;
                cp_async_4(smem_u32(&Bs[sl][lc + q][lr]), in ? Bb + n * ldb + k : B, in);
            }
        }
    };
    for (int st = 0; st < SST - 1; ++st) {
        if (st < nsteps) issue(st);
        cp_async_commit();
    }
    float acc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
    for (int64_t step = 0; step < nsteps; ++step) {
        cp_async_wait_group<SST - 2>();  // this thread's copies of `step` have landed
        __syncthreads();                 // everyone's have; everyone is done with step - 1
        const int sl = static_cast<int>(step % SST);
#pragma unroll
        for (int kk = 0; kk < SB; ++kk) {
            const float a0 = As[sl][kk][ty], a1 = As[sl][kk][ty + 16];
            const float b0 = Bs[sl][kk][tx], b1 = Bs[sl][kk][tx + 16];
            acc[0][0] = fmaf(a0, b0, acc[0][0]);
            acc[0][1] = fmaf(a0, b1, acc[0][1]);
            acc[1][0] = fmaf(a1, b0, acc[1][0]);
            acc[1][1] = fmaf(a1, b1, acc[1][1]);
        }
        // refill the slot of step - 1 (every thread passed the barrier above after using it)
        if (step + SST - 1 < nsteps) issue(step + SST - 1);
        cp_async_commit();
    }
    cp_async_wait_all();
    epi_store1(e, bz, m0 + ty, n0 + tx, acc[0][0]);
    epi_store1(e, bz, m0 + ty, n0 + tx + 16, acc[0][1]);
    epi_store1(e, bz, m0 + ty + 16, n0 + tx, acc[1][0]);
    epi_store1(e, bz, m0 + ty + 16, n0 + tx + 16, acc[1][1]);
}

template <int BN, int STAGES, bool B_NK, bool PACKED>
cudaError_t launch_ffma_t(const gemm_config_t& cfg, const CUtensorMap& tmA,
                          const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                          const LaunchCtx& lc) {
    FfmaArgs a{};
    a.s = s;
    const int64_t mt = (s.M + FBM - 1) / FBM, nt = (s.N + BN - 1) / BN;
    const int64_t kt = (s.K + FBK - 1) / FBK;
    const int64_t tiles = mt * nt * s.batch;
    if (tiles * kt >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // see ffma_units_ok
    a.m_tiles = static_cast<int>(mt);
    a.n_tiles = static_cast<int>(nt);
    a.tiles_per_batch = static_cast<int>(mt * nt);
    a.raster = cfg.raster_group > 0 ? cfg.raster_group : 8;
    a.k_tiles = static_cast<int>(kt);
    a.units = static_cast<int>(tiles * kt);
    a.e = e;
    a.status = lc.status;
    a.timeout_ns = lc.timeout_ns;
    a.flags = lc.flags;
    const int smem = ffma_smem_total<BN, STAGES>();
    auto kern = ffma_kernel<BN, STAGES, B_NK, PACKED>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    if (!cfg.stream_k) {
        a.grid = static_cast<int>(tiles);  // one whole tile per CTA
        kern<<<static_cast<unsigned>(tiles), FTHREADS, smem, lc.stream>>>(tmA, tmB, a);
        return cudaGetLastError();
    }
    if (!lc.sk_partials || !lc.sk_tags || lc.sk_grid <= 0) return cudaErrorInvalidValue;
    a.grid = static_cast<int>(lc.sk_grid < a.units ? lc.sk_grid : a.units);
    a.partials = lc.sk_partials;
    a.tags = lc.sk_tags;
    a.epoch = lc.sk_epoch;
    cudaLaunchConfig_t lcfg = {};
    lcfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    lcfg.blockDim = dim3(FTHREADS);
    lcfg.dynamicSmemBytes = smem;
    lcfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    lcfg.attrs = attr;
    lcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&lcfg, kern, tmA, tmB, a);
}

template <int BN, int STAGES, bool B_NK, bool PACKED>
int max_ctas_t() {
    auto kern = ffma_kernel<BN, STAGES, B_NK, PACKED>;
    const int smem = ffma_smem_total<BN, STAGES>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, FTHREADS, smem) != cudaSuccess)
        return 0;
    return per_sm;
}

}  // namespace

cudaError_t launch_ffma_small(const float* A, const float* B, int64_t lda, int64_t ldb,
                              int64_t stride_a, int64_t stride_b, int b_layout, const Shape& s,
                              const EpiParams& e, cudaStream_t stream) {
    if (s.M <= 0 || s.N <= 0) return cudaSuccess;
    const int64_t gx = (s.N + SB - 1) / SB, gy = (s.M + SB - 1) / SB;
    if (gx >= (int64_t(1) << 31) || gy > 65535 || s.batch > 65535) return cudaErrorInvalidValue;
    ffma_small_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                             static_cast<unsigned>(s.batch)),
                        256, 0, stream>>>(A, B, lda, ldb, stride_a, stride_b,
                                          b_layout == GEMM_B_NK ? 1 : 0, s.M, s.N, s.K, e);
    return cudaGetLastError();
}

size_t ffma_smem_bytes(const gemm_config_t& cfg) {
    if (cfg.variant == FFMA_VARIANT_SMALL) return 2 * SST * SB * (SB + 1) * sizeof(float);
    if (cfg.stages < 2 || cfg.stages > 4) return 0;
    if (cfg.bn == 128)
        return cfg.stages == 2   ? ffma_smem_total<128, 2>()
               : cfg.stages == 3 ? ffma_smem_total<128, 3>()
                                 : ffma_smem_total<128, 4>();
    if (cfg.bn == 256)
        return cfg.stages == 2   ? ffma_smem_total<256, 2>()
               : cfg.stages == 3 ? ffma_smem_total<256, 3>()
                                 : ffma_smem_total<256, 4>();
    return 0;
}

size_t ffma_partial_slot_bytes(const gemm_config_t& cfg) {
    return static_cast<size_t>(FBM) * cfg.bn * sizeof(float);
}

bool ffma_units_ok(const Shape& s, int bn) {
    if (bn == SB)  // small-tile variant: grid (N/32, M/32, batch)
        return (s.M + SB - 1) / SB <= 65535 && s.batch <= 65535;
    const int64_t units = ((s.M + FBM - 1) / FBM) * ((s.N + bn - 1) / bn) * s.batch *
                          ((s.K + FBK - 1) / FBK);
    return units < (int64_t(1) << 31);
}

// One switch over the instantiated (BN, STAGES, layout, packed) combinations.
// K-major B exists for BN = 128 only; the packed loop for KN only.
#define G13_FFMA_DISPATCH(CALL)                                                              \
    const bool nk = b_layout == GEMM_B_NK;                                                   \
    const bool packed = cfg.variant == 1 && !nk;                                             \
    if (cfg.bn == 128) {                                                                     \
        switch (cfg.stages) {                                                                \
            case 2:                                                                          \
                if (nk) return CALL(128, 2, true, false);                                    \
                return packed ? CALL(128, 2, false, true) : CALL(128, 2, false, false);      \
            case 3:                                                                          \
                if (nk) return CALL(128, 3, true, false);                                    \
                return packed ? CALL(128, 3, false, true) : CALL(128, 3, false, false);      \
            case 4:                                                                          \
                if (nk) return CALL(128, 4, true, false);                                    \
                return packed ? CALL(128, 4, false, true) : CALL(128, 4, false, false);      \
            default: break;                                                                  \
        }                                                                                    \
    } else if (cfg.bn == 256 && !nk) {                                                       \
        switch (cfg.stages) {                                                                \
            case 2: return packed ? CALL(256, 2, false, true) : CALL(256, 2, false, false);  \
            case 3: return packed ? CALL(256, 3, false, true) : CALL(256, 3, false, false);  \
            case 4: return packed ? CALL(256, 4, false, true) : CALL(256, 4, false, false);  \
            default: break;                                                                  \
        }                                                                                    \
    }

int ffma_ctas_per_sm(const gemm_config_t& cfg, int b_layout) {
#define G13_OCC(BN, ST, NK, PK) max_ctas_t<BN, ST, NK, PK>()
    G13_FFMA_DISPATCH(G13_OCC)
#undef G13_OCC
    return 0;
}

cudaError_t launch_ffma(const gemm_config_t& cfg, int b_layout, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const Shape& s, const EpiParams& e,
                        const LaunchCtx& lc) {
#define G13_LAUNCH(BN, ST, NK, PK) launch_ffma_t<BN, ST, NK, PK>(cfg, tmA, tmB, s, e, lc)
    G13_FFMA_DISPATCH(G13_LAUNCH)
#undef G13_LAUNCH
    return cudaErrorInvalidValue;
}

template <int BN, int ST, bool NK, bool PK>
cudaError_t ffma_attr_t() {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, ffma_kernel<BN, ST, NK, PK>);
}

static cudaError_t ffma_preload_one(const gemm_config_t& cfg, int b_layout) {
#define G13_ATTR(BN, ST, NK, PK) ffma_attr_t<BN, ST, NK, PK>()
    G13_FFMA_DISPATCH(G13_ATTR)
#undef G13_ATTR
    return cudaSuccess;
}

cudaError_t ffma_preload_kernels() {
    // A function-attribute query makes the runtime load a lazily loaded kernel.
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, ffma_small_kernel);
    for (int bn = 128; bn <= 256 && err == cudaSuccess; bn += 128)
        for (int st = 2; st <= 4 && err == cudaSuccess; ++st)
            for (int var = 0; var <= 1 && err == cudaSuccess; ++var)
                for (int lay = GEMM_B_KN; lay <= GEMM_B_NK && err == cudaSuccess; ++lay) {
                    gemm_config_t cfg{};
                    cfg.kernel = GEMM_KERNEL_FFMA;
                    cfg.bn = bn;
                    cfg.stages = st;
                    cfg.variant = var;
                    err = ffma_preload_one(cfg, lay);
                }
    return err;
}

#undef G13_FFMA_DISPATCH

}  // namespace g13
