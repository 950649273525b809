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
//               release the accumulator buffer (tempty[buf]).  Each warp
//               works on 128-byte-wide column chunks of its 32 rows: the
//               values go into a double-buffered 128B-swizzled shared tile
//               that one lane writes out with a TMA store (coalesced,
//               asynchronous, clipped at the matrix edge); an FP32 residual
//               arrives the same way, by a TMA load into that tile first.
//               Layouts TMA cannot address fall back to per-thread stores.
//
// The grid is persistent (one CTA per SM); CTA c walks tiles c, c+grid, ...
// in a grouped raster order.
//
// Pair mode (PAIR): clusters of two CTAs on two SMs share one 256 x BN tile
// through tcgen05 cta_group::2.  Each CTA loads its own 128 rows of A and its
// own BN/2 columns of B, so a CTA moves 32 KB per 64-deep K block instead of
// 48 KB for a 128 x 256 tile; the even CTA's MMA thread issues 256 x BN x 16
// MMAs that read both CTAs' shared memory and write each CTA's 128 rows of the
// accumulator into that CTA's TMEM.  Both CTAs' TMA loads for a stage count
// their bytes on the even CTA's full[s] barrier (cta_group::2 TMA), the even
// CTA's commits are multicast to both CTAs' stage and accumulator barriers,
// and both CTAs' epilogue warps return accumulator buffers to the even CTA.  The double-buffered accumulator lets the
// epilogue of tile t overlap the main loop of tile t+1.  Out-of-range rows,
// columns and K arrive from TMA as zeros, so the main loop has no edge code.
//
// B comes in two layouts: NK ([N,K], K contiguous, "K-major") is loaded like
// A; KN ([K,N], N contiguous, "MN-major") is loaded as BN/64 boxes of
// 64 K-rows x 64 N-columns and described to the MMA as an MN-major operand.
//
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains its own copies
// and MMAs, frees TMEM and exits, and the plan's status word records it.
#include <atomic>
#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g13 {
namespace {

constexpr int kMaxDevices = 64;

// Two FP32 values in one 64-bit register pair, for Blackwell's packed FP32
// arithmetic (mul / fma .rn.f32x2: two IEEE operations per instruction).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// GELU for the tensor-core epilogue, 0.5 y (1 + erf(y / sqrt 2)), two values
// at a time, with erf from Abramowitz & Stegun, Handbook of Mathematical
// Functions, formula 7.1.26 (|error| <= 1.5e-7 on erf): for x >= 0,
//     1 - erf(x) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
//     t = 1 / (1 + p x),  p = 0.3275911,
//     a1..a5 = 0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429.
// With h = 1 - erf(|y| / sqrt 2), GELU(y) = max(y, 0) - 0.5 |y| h for either
// sign of y (erf is odd).  Per pair of values: two MUFU reciprocals, two MUFU
// exp2, and nine packed FP32 operations (the library erff made GELU 44 % of an
// FFN-shaped GEMM's time; scalar arithmetic took twice the instructions).
__device__ __forceinline__ void gelu2_as7126(float& y0, float& y1) {
    const uint64_t ax = f2_pack(fabsf(y0), fabsf(y1));
    // 1 + p |y| / sqrt 2, p = 0.3275911
    const uint64_t u = f2_fma(ax, f2_pack(0.23164189f, 0.23164189f), f2_pack(1.0f, 1.0f));
    float u0, u1;
    f2_unpack(u, u0, u1);
    float t0, t1;  // 1 / u by the MUFU approximation (~1 ulp)
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t0) : "f"(u0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t1) : "f"(u1));
    const uint64_t t = f2_pack(t0, t1);
    uint64_t p = f2_fma(f2_pack(1.061405429f, 1.061405429f), t, f2_pack(-1.453152027f, -1.453152027f));
    p = f2_fma(p, t, f2_pack(1.421413741f, 1.421413741f));
    p = f2_fma(p, t, f2_pack(-0.284496736f, -0.284496736f));
    p = f2_fma(p, t, f2_pack(0.254829592f, 0.254829592f));
    p = f2_mul(p, t);
    const uint64_t y = f2_pack(y0, y1);
    // exponent of exp(-y^2 / 2) in base 2: -y^2 log2(e) / 2
    const uint64_t q = f2_mul(f2_mul(y, f2_pack(-0.72134752044448170f, -0.72134752044448170f)), y);
    float q0, q1;
    f2_unpack(q, q0, q1);
    const uint64_t h = f2_mul(p, f2_pack(ex2_approx(q0), ex2_approx(q1)));
    const uint64_t r = f2_fma(f2_mul(ax, h), f2_pack(-0.5f, -0.5f),
                              f2_pack(fmaxf(y0, 0.0f), fmaxf(y1, 0.0f)));
    f2_unpack(r, y0, y1);
}

constexpr int TBM = 128, TBK = 64;        // rows of A per CTA; K elements per stage (16-bit)
constexpr int TBK3 = 32;                   // K elements per stage for FP32 (3xTF32)
constexpr int T_A_TILE = TBM * 128;        // 16 KB: 128 rows x 128 B (64 x 16-bit or 32 x FP32)
constexpr int EPI_BUF_BYTES = 32 * 128;   // one 32-row x 128-byte output (or residual) chunk

// K3: FP32 inputs as 3xTF32 -- each stage holds the high and the low TF32
// parts of the A and B boxes: [A hi | A lo | B hi | B lo].
template <int BN, bool PAIR, bool K3>
struct TcLayout {
    static constexpr int KE = K3 ? TBK3 : TBK;           // K elements per stage
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;    // B columns this CTA loads
    static constexpr int B_TILE = B_ROWS * 128;          // B_ROWS x 128 B
    static constexpr int A_BYTES = T_A_TILE * (K3 ? 2 : 1);
    static constexpr int B_BYTES = B_TILE * (K3 ? 2 : 1);
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TILE_M = PAIR ? 2 * TBM : TBM;  // rows of a (pair) tile
};

struct TcArgs {
    int64_t M, N, K, batch;
    int a_bmul, b_bmul;
    int epi_tma;    // 1: C is written by TMA stores through shared memory
    int r_tma;      // 1: the FP32 residual is read by TMA loads (implies epi_tma)
    int r_ahead;    // 1: each chunk's residual is requested one chunk ahead (implies r_tma)
    int out16;      // 1: C holds 16-bit values (64 columns per 128-byte chunk)
    int c_bmul, r_bmul;
    int c_smul;     // split-K: C batch coordinate = b * c_bmul + split * c_smul
    int splits;     // split-K: K-block ranges per tile (1 = none)
    int kb_per_split;
    int64_t total_items;  // total_tiles * splits (split-major order)
    int bias_vec;   // 1: bias is 16-byte aligned (float4 loads)
    int epi_plain;  // 1: no bias, activation or residual (C = alpha * acc, cast)
    int64_t n_tma;  // columns [0, n_tma) go out by TMA (a multiple of 16 bytes); the rest,
                    // fewer than 16 bytes per row, from registers
    int64_t m_tiles, n_tiles, tiles_per_batch, total_tiles;
    int k_blocks;
    int raster;
    uint32_t idesc;
    EpiParams e;
    unsigned* status;
    uint64_t timeout_ns;
    uint32_t flags;
};

// EW epilogue warps: 4 (one per TMEM lane quarter) or 8 (two per quarter,
// each taking half of the columns).
template <int EW>
__host__ __device__ constexpr int tc_threads() {
    return 64 + 32 * EW;
}
template <int BN, int STAGES, bool PAIR, bool K3>
__host__ __device__ constexpr int tc_epi_off() {
    return STAGES * TcLayout<BN, PAIR, K3>::STAGE_BYTES;
}
template <int BN, int STAGES, int EW, bool PAIR, bool K3>
__host__ __device__ constexpr int tc_bar_off() {
    return tc_epi_off<BN, STAGES, PAIR, K3>() + EW * 2 * EPI_BUF_BYTES;
}
template <int BN, int STAGES, int EW, bool PAIR, bool K3>
__host__ __device__ constexpr int tc_smem_total() {
    // ring + epilogue tiles + full/empty per stage + tfull/tempty x2 + drain
    // + residual barriers (2 per epilogue warp) + softmax exchange barriers (4)
    // + pair exit barriers (2) + per-stage copy counts (8) + tmem slot + abort
    // flag + softmax exchange values [2][EW][32] floats (single CTAs only: the
    // row softmax never runs on CTA pairs)
    return 1024 + tc_bar_off<BN, STAGES, EW, PAIR, K3>() + (2 * STAGES + 11 + 2 * EW) * 8 + 32 +
           16 + (PAIR ? 0 : 2 * EW * 32 * 4);
}

// 32-bit arithmetic: the host keeps the tile count below 2^31.
__device__ __forceinline__ void tc_tile_coords(int64_t t, const TcArgs& a, int64_t& b, int64_t& mt,
                                               int64_t& nt) {
    const uint32_t tu = static_cast<uint32_t>(t);
    const uint32_t tpb = static_cast<uint32_t>(a.tiles_per_batch);
    const uint32_t bu = tu / tpb;
    const uint32_t r = tu - bu * tpb;
    const uint32_t span = static_cast<uint32_t>(a.raster) * static_cast<uint32_t>(a.n_tiles);
    const uint32_t g = r / span;
    const uint32_t first = g * static_cast<uint32_t>(a.raster);
    const uint32_t gm =
        min(static_cast<uint32_t>(a.raster), static_cast<uint32_t>(a.m_tiles) - first);
    const uint32_t w = r - g * span;
    b = bu;
    mt = first + w % gm;
    nt = w / gm;
}

__device__ __forceinline__ void tc_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return;
}

// Pair exit: waits, with acquire at cluster scope, for a phase of a local
// barrier that the peer CTA arrives on; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_peer(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}
// 32-bit load from the shared memory of a CTA of the cluster (a mapa address).
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}
// Counts `bytes` as arrived on a local barrier's current phase without a copy.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

template <int BN, int STAGES, bool B_KN, int EW, bool PAIR, bool K3>
__global__ void __launch_bounds__(tc_threads<EW>(), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                   const TcArgs args) {
    using L = TcLayout<BN, PAIR, K3>;
    static_assert(!(K3 && B_KN), "3xTF32 reads B K-major (the split pass transposes KN)");
    static_assert(STAGES <= 8, "per-stage copy counts hold 8 stages");
    // Accumulator buffers in TMEM: two of BN columns, or one for 512-wide
    // tiles (the row softmax), which fill all 512 columns.
    constexpr int NBUF = BN > 256 ? 1 : 2;
    constexpr uint32_t TMEM_COLS = NBUF * BN <= 256 ? 256u : 512u;  // allocations: powers of two
    constexpr int NHALF = BN > 256 ? 2 : 1;    // MMAs per K step (N <= 256 per MMA)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + tc_bar_off<BN, STAGES, EW, PAIR, K3>());
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* rbar = drain + 1;  // [EW][2] residual-chunk barriers
    uint64_t* xbar = rbar + 2 * EW;  // [4] softmax: the two warps of a lane quarter meet
    uint64_t* oreport = xbar + 4;    // pair exit: the odd CTA's copy counts are ready (even CTA's)
    uint64_t* pdone = oreport + 1;   // pair exit: the even CTA saw them all land (odd CTA's)
    uint32_t* uses = reinterpret_cast<uint32_t*>(pdone + 1);  // [8] copies issued per stage
    uint32_t* tmem_slot = uses + 8;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(tmem_slot + 1);
    float* xch = reinterpret_cast<float*>(tmem_slot + 4);  // [2][EW][32] softmax partials

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Pair mode: rank 0 / 1 in the CTA pair; the pair walks tiles together.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int64_t first_item = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
    const int64_t item_stride = PAIR ? (gridDim.x >> 1) : gridDim.x;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            // pair mode: lane 0 of every epilogue warp of both CTAs; else every epilogue thread
            mbar_init(smem_u32(&tempty[i]), PAIR ? 2 * EW : 32 * EW);
        }
        mbar_init(smem_u32(drain), 1);
        for (int i = 0; i < 2 * EW; ++i) mbar_init(smem_u32(&rbar[i]), 1);
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&xbar[i]), 64);
        mbar_init(smem_u32(oreport), 1);
        mbar_init(smem_u32(pdone), 1);
        for (int i = 0; i < 8; ++i) uses[i] = 0u;
        *abort_flag = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if (PAIR)
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        else
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint64_t tmo = args.timeout_ns;
    const int kb_total = args.k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const bool stall = ((args.flags & GEMM_FLAG_TEST_STALL) && blockIdx.x == 0) ||
                               ((args.flags & GEMM_FLAG_TEST_STALL_PEER) && blockIdx.x == 1);
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;  // per stage: armed and not yet seen consumed
            bool ok = true;
            for (int64_t t = first_item; ok && t < args.total_items; t += item_stride) {
                const int split = static_cast<int>(t / args.total_tiles);
                int64_t b, mt, nt;
                tc_tile_coords(t - split * args.total_tiles, args, b, mt, nt);
                // this CTA's rows of A and columns of B
                const int32_t m0 = static_cast<int32_t>(mt * L::TILE_M + rank * TBM);
                const int32_t n0 = static_cast<int32_t>(nt * BN + rank * L::B_ROWS);
                const int kb_lo = split * args.kb_per_split;
                const int kb_hi = min(kb_total, kb_lo + args.kb_per_split);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, args.status,
                                           tmo)) {
                        ok = false;
                        break;
                    }
                    armed &= ~(1u << s);  // the previous use of this stage was consumed
                    const bool skip = stall && t == first_item && kb == kb_lo;
                    if (!skip) {
                        uint8_t* sa = smem + s * L::STAGE_BYTES;
                        uint8_t* sb = sa + L::A_BYTES;
                        // 3xTF32: the split buffers hold [batch][hi, lo][rows][K]
                        const int32_t ba = static_cast<int32_t>(b * args.a_bmul) * (K3 ? 2 : 1);
                        const int32_t bb = static_cast<int32_t>(b * args.b_bmul) * (K3 ? 2 : 1);
                        // In a pair, both CTAs' boxes for stage s land on the even
                        // CTA's full[s], which expects both CTAs' bytes.
                        const uint32_t bar =
                            PAIR ? mapa_shared(smem_u32(&full[s]), 0) : smem_u32(&full[s]);
                        if (rank == 0)
                            mbar_arrive_expect_tx(smem_u32(&full[s]),
                                                  (PAIR ? 2 : 1) * L::STAGE_BYTES);
                        const auto load = [&](uint32_t dst, const CUtensorMap* m, int32_t c0,
                                              int32_t c1, int32_t c2) {
                            if (PAIR)
                                tma_load_3d_pair(dst, m, bar, c0, c1, c2);
                            else
                                tma_load_3d(dst, m, bar, c0, c1, c2);
                        };
                        load(smem_u32(sa), &tmA, kb * L::KE, m0, ba);
                        if (K3) {
                            load(smem_u32(sa + T_A_TILE), &tmA, kb * L::KE, m0, ba + 1);
                            load(smem_u32(sb), &tmB, kb * L::KE, n0, bb);
                            load(smem_u32(sb + L::B_TILE), &tmB, kb * L::KE, n0, bb + 1);
                        } else if (B_KN) {
#pragma unroll
                            for (int j = 0; j < L::B_ROWS / 64; ++j)
                                load(smem_u32(sb + j * (64 * 128)), &tmB, n0 + 64 * j, kb * L::KE, bb);
                        } else {
                            // K-major boxes of at most 256 rows (a TMA box limit)
                            constexpr int BOXR = L::B_ROWS < 256 ? L::B_ROWS : 256;
#pragma unroll
                            for (int h = 0; h < L::B_ROWS / BOXR; ++h)
                                load(smem_u32(sb + h * BOXR * 128), &tmB, kb * L::KE, n0 + h * BOXR,
                                     bb);
                        }
                        armed |= 1u << s;
                        armed_par = (armed_par & ~(1u << s)) | (ph << s);
                        if (PAIR) uses[s] += 1u;
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (PAIR) {
                // Every copy of a pair counts on the even CTA's full[] barriers, so
                // the even producer sees each copy either CTA issued land before the
                // pair may leave (normal end or abort).  The odd producer reports its
                // per-stage copy counts; a stage's copies all belong to its last
                // phase (a producer issues use u + 1 of a stage only after use u was
                // consumed), and the even producer makes that phase completable by
                // counting the share that will never come -- the odd CTA's, by
                // complete_tx, or its own, by arming the phase for the odd share
                // alone -- then waits for it and acknowledges.  Both CTAs then stay
                // resident until the exit cluster barrier.
                const uint64_t lim = 3 * tmo + 1000000ull;
                if (rank == 1) {
                    mbar_arrive_cluster(mapa_shared(smem_u32(oreport), 0));
                    if (!mbar_wait_peer(smem_u32(pdone), 0u, lim) && armed) {
                        // no acknowledgement: give our copies a fixed 200 us
                        const uint64_t t0 = globaltimer_ns();
                        while (globaltimer_ns() - t0 < 200000ull) {
                        }
                    }
                } else {
                    const bool got = mbar_wait_peer(smem_u32(oreport), 0u, lim);
                    for (int i = 0; i < STAGES; ++i) {
                        if (!got) {  // no report: our own armed phases only
                            if (!ok && (armed & (1u << i)))
                                tc_drain(smem_u32(&full[i]), (armed_par >> i) & 1u, tmo);
                            continue;
                        }
                        const uint32_t ne = uses[i];
                        const uint32_t no = ld_peer_u32(mapa_shared(smem_u32(&uses[i]), 1));
                        const uint32_t n = ne > no ? ne : no;
                        if (n == 0) continue;
                        if (ne == no + 1)
                            mbar_complete_tx(smem_u32(&full[i]), L::STAGE_BYTES);
                        else if (no == ne + 1)
                            mbar_arrive_expect_tx(smem_u32(&full[i]), L::STAGE_BYTES);
                        else if (ne != no)
                            continue;
                        tc_drain(smem_u32(&full[i]), (n - 1) & 1u, tmo);
                    }
                    if (got) mbar_arrive_cluster(mapa_shared(smem_u32(pdone), 1));
                }
            } else if (!ok) {
                // Let our own copies land before the CTA's shared memory goes away.
                for (int i = 0; i < STAGES; ++i)
                    if (armed & (1u << i))
                        tc_drain(smem_u32(&full[i]), (armed_par >> i) & 1u, tmo);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer
            // (in a pair, only the even CTA's thread issues; the odd CTA's
            // warp 1 only holds its half of the TMEM allocation)
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            bool issued_any = false;
            int lt = 0;
            for (int64_t t = first_item; ok && t < args.total_items; t += item_stride, ++lt) {
                const int buf = NBUF == 1 ? 0 : (lt & 1);
                const uint32_t tph = static_cast<uint32_t>(NBUF == 1 ? lt : (lt >> 1)) & 1u;
                if (!mbar_wait_bounded(smem_u32(&tempty[buf]), tph ^ 1u, abort_flag, args.status,
                                       tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                const int kb_lo = static_cast<int>(t / args.total_tiles) * args.kb_per_split;
                const int kb_hi = min(kb_total, kb_lo + args.kb_per_split);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, args.status, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * L::STAGE_BYTES);
                    const uint32_t sb = sa + L::A_BYTES;
                    if (K3) {
                        // 3xTF32: per 8-deep K step, A.B ~ Alo.Bhi + Ahi.Blo + Ahi.Bhi
                        // (the small terms first); a K step of 8 FP32 is 32 B
                        // inside the swizzled 128-byte row, as for 16-bit inputs.
#pragma unroll
                        for (int kk = 0; kk < L::KE / 8; ++kk) {
                            const uint64_t ah = smem_desc_sw128(sa + kk * 32, 16, 1024);
                            const uint64_t al = smem_desc_sw128(sa + T_A_TILE + kk * 32, 16, 1024);
                            const uint64_t bh = smem_desc_sw128(sb + kk * 32, 16, 1024);
                            const uint64_t bl = smem_desc_sw128(sb + L::B_TILE + kk * 32, 16, 1024);
                            const uint32_t acc = ((kb - kb_lo) | kk) != 0 ? 1u : 0u;
                            if (PAIR) {
                                tc_mma_tf32_pair(d_tmem, al, bh, args.idesc, acc);
                                tc_mma_tf32_pair(d_tmem, ah, bl, args.idesc, 1u);
                                tc_mma_tf32_pair(d_tmem, ah, bh, args.idesc, 1u);
                            } else {
                                tc_mma_tf32(d_tmem, al, bh, args.idesc, acc);
                                tc_mma_tf32(d_tmem, ah, bl, args.idesc, 1u);
                                tc_mma_tf32(d_tmem, ah, bh, args.idesc, 1u);
                            }
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < (K3 ? 0 : TBK / 16); ++kk) {
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
                        const uint32_t acc = ((kb - kb_lo) | kk) != 0 ? 1u : 0u;
                        if (PAIR) {
                            tc_mma_f16_pair(d_tmem, adesc, bdesc, args.idesc, acc);
                        } else {
                            // 512-wide tiles: two N = 256 MMAs, the second on B rows
                            // (KN: panels) 256.. at +32 KB and accumulator columns 256..
#pragma unroll
                            for (int h = 0; h < NHALF; ++h)
                                tc_mma_f16(d_tmem + h * 256, adesc, bdesc + h * (32768 >> 4),
                                           args.idesc, acc);
                        }
                    }
                    issued_any = true;
                    // stage s (in both CTAs of a pair) is free once these MMAs finish
                    if (PAIR)
                        tc_commit_pair(smem_u32(&empty[s]), 0x3);
                    else
                        tc_commit(smem_u32(&empty[s]));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                // accumulator ready for the epilogue (of both CTAs of a pair)
                if (PAIR)
                    tc_commit_pair(smem_u32(&tfull[buf]), 0x3);
                else
                    tc_commit(smem_u32(&tfull[buf]));
            }
            if (!ok && issued_any) {
                // Wait for every MMA already issued before TMEM is released.
                if (PAIR)
                    tc_commit_pair(smem_u32(drain), 0x1);
                else
                    tc_commit(smem_u32(drain));
                tc_drain(smem_u32(drain), 0u, tmo);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue warps
        const int ew = warp - 2;  // 0 .. EW-1
        const int q = warp & 3;   // TMEM lane quarter this warp may access
        // Warps sharing a quarter split the tile's columns into EW/4 slices.
        constexpr int SLICE = BN / (EW / 4);
        const int c_lo = (ew >> 2) * SLICE;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* etile = smem + tc_epi_off<BN, STAGES, PAIR, K3>() + ew * 2 * EPI_BUF_BYTES;
        // Hand an accumulator buffer back to the MMA thread (the even CTA's in a pair).
        const auto release = [&](int buf) {
            tc_fence_before();
            if (PAIR) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
            } else {
                mbar_arrive(smem_u32(&tempty[buf]));
            }
        };
        uint64_t* rb = rbar + 2 * ew;
        const EpiParams& e = args.e;
        uint32_t rph = 0;  // bit i: phase parity of rb[i]
        int nchunk = 0;    // chunks this warp has staged (selects the buffer)
        // Residual by TMA, when the host asks for it (args.r_ahead: short K or one
        // tile per CTA, where the epilogue is not hidden behind a next main loop):
        // the tile of chunk k + 1 is requested while chunk k is being worked on,
        // so its load overlaps a whole chunk (the first one overlaps the first
        // main loop).  r_ahead = index of the chunk whose residual is already in
        // flight (-1: none).
        int r_ahead = -1;
        // TMA coordinates are 32-bit: (column, row, batch coordinate).
        const auto r_issue = [&](int sel, int32_t cg, int32_t r0, int32_t bc) {
            mbar_arrive_expect_tx(smem_u32(&rb[sel]), EPI_BUF_BYTES);
            tma_load_3d(smem_u32(etile + sel * EPI_BUF_BYTES), &tmR, smem_u32(&rb[sel]), cg, r0,
                        bc);
        };
        // First chunk of work item t for this warp: its column, row and residual
        // batch coordinate; false when the item has no columns for this warp.
        // (The residual is never read under split-K, so work items are tiles.)
        const auto first_chunk = [&](int64_t t, int32_t& cg, int32_t& r0, int32_t& bc) {
            int64_t bidx, mt2, nt2;
            tc_tile_coords(t, args, bidx, mt2, nt2);
            cg = static_cast<int32_t>(nt2) * BN + c_lo;
            r0 = static_cast<int32_t>(mt2) * L::TILE_M + static_cast<int32_t>(rank * TBM + q * 32);
            bc = static_cast<int32_t>(bidx) * args.r_bmul;
            return cg < e.N;
        };
        if (args.r_ahead && first_item < args.total_items) {
            int32_t cg, r0, bidx;
            if (first_chunk(first_item, cg, r0, bidx)) {
                if (lane == 0) r_issue(0, cg, r0, bidx);
                r_ahead = 0;
            }
        }
        bool ok = true;
        int lt = 0;
        for (int64_t t = first_item; ok && t < args.total_items; t += item_stride, ++lt) {
            const int buf = NBUF == 1 ? 0 : (lt & 1);
            const uint32_t tph = static_cast<uint32_t>(NBUF == 1 ? lt : (lt >> 1)) & 1u;
            if (!mbar_wait_bounded(smem_u32(&tfull[buf]), tph, abort_flag, args.status, tmo)) break;
            tc_fence_after();
            const int split = static_cast<int>(t / args.total_tiles);
            int64_t bt, mt, nt;
            tc_tile_coords(t - split * args.total_tiles, args, bt, mt, nt);
            // output batch index: the partial-sum slab (batch, split) under split-K
            const int64_t b = args.splits > 1 ? bt * args.splits + split : bt;
            const int32_t row0 = static_cast<int32_t>(mt * L::TILE_M + rank * TBM + q * 32);
            const int64_t row = row0 + lane;
            const int64_t col0 = nt * BN;
            const uint32_t tbase = tmem_base + lane_base + static_cast<uint32_t>(buf * BN);
            // Row softmax: this thread's row is all in TMEM (one tile spans N);
            // with 8 epilogue warps the row's columns are split between the
            // two warps of a lane quarter, which trade their partial maximum
            // and sum through shared memory (both arrive on xbar[q], bounded
            // wait; two phases per tile, so exchange k waits on parity k).
            // Work in the base-2 domain, u = t * log2(e) with t = alpha*acc +
            // bias: pass 1 finds the maximum m of u over the row; pass 2
            // overwrites each accumulator with 2^(u - m) (ex2.approx, one MUFU
            // op) and sums them; the store loop below writes each value
            // divided by the sum.  Columns past N are skipped (only the last
            // chunk checks).
            float sinv = 0.0f;
            bool xok = true;
            const auto exchange = [&](int k, float val) {
                if (EW != 8) return val;
                float* xb = xch + k * EW * 32;
                xb[ew * 32 + lane] = val;
                mbar_arrive(smem_u32(&xbar[q]));
                if (!mbar_wait_bounded(smem_u32(&xbar[q]), static_cast<uint32_t>(k), abort_flag,
                                       args.status, tmo)) {
                    xok = false;
                    return val;
                }
                return xb[(ew ^ 4) * 32 + lane];
            };
            if (e.act == GEMM_ACT_SOFTMAX) {
                constexpr float LOG2E = 1.4426950408889634f;
                const float a2 = e.alpha * LOG2E;
                // valid columns in this warp's slice (int32: at most SLICE)
                const int nrow = static_cast<int>(
                    max(static_cast<int64_t>(0),
                        min(static_cast<int64_t>(SLICE), e.N - (col0 + c_lo))));
                const float* bias = e.bias ? e.bias + col0 + c_lo : nullptr;
                float mu = -INFINITY;  // max over the slice of u
#pragma unroll 1
                for (int c = 0; c < nrow; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c_lo + c, v);
                    tmem_ld_wait();
                    const int nv = min(32, nrow - c);
                    float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    if (nv == 32 && !bias) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            mc[i & 3] = fmaxf(mc[i & 3], __uint_as_float(v[i]) * a2);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < nv) {
                                const float ub = bias ? __ldg(bias + c + i) * LOG2E : 0.0f;
                                mc[i & 3] = fmaxf(mc[i & 3], fmaf(__uint_as_float(v[i]), a2, ub));
                            }
                    }
                    mu = fmaxf(mu, fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])));
                }
                mu = fmaxf(mu, exchange(0, mu));
                float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
                for (int c = 0; c < nrow; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c_lo + c, v);
                    tmem_ld_wait();
                    const int nv = min(32, nrow - c);
                    if (nv == 32 && !bias) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float ex = ex2_approx(fmaf(__uint_as_float(v[i]), a2, -mu));
                            z[i & 3] += ex;
                            v[i] = __float_as_uint(ex);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float ex = 0.0f;
                            if (i < nv) {
                                const float ub = bias ? fmaf(__ldg(bias + c + i), LOG2E, -mu) : -mu;
                                ex = ex2_approx(fmaf(__uint_as_float(v[i]), a2, ub));
                            }
                            z[i & 3] += ex;
                            v[i] = __float_as_uint(ex);
                        }
                    }
                    tmem_st_32x32b_x32(tbase + c_lo + c, v);
                }
                tmem_st_wait();
                const float zh = (z[0] + z[1]) + (z[2] + z[3]);
                const float zp = exchange(1, zh);
                // the same order in both warps: lower column half first
                sinv = 1.0f / (EW == 8 ? (ew < 4 ? zh + zp : zp + zh) : zh);
                if (!xok) {
                    ok = false;
                    break;
                }
            }
            if (args.epi_tma) {
                // The chunk loop, compiled for each chunk width (W columns = 128
                // bytes: 32 FP32 or 64 16-bit) so its arrays are exactly W long
                // (a runtime width kept 64 of each live and spilled).  Returns
                // false when a residual wait gave up.
                const auto chunk_loop = [&](auto w_tag) -> bool {
                constexpr int W = decltype(w_tag)::value;
#pragma unroll 1
                for (int c = c_lo; c < c_lo + SLICE; c += W) {
                    uint32_t v[W];
                    tmem_ld_32x32b_x32(tbase + c, *reinterpret_cast<uint32_t(*)[32]>(v));
                    if constexpr (W == 64)
                        tmem_ld_32x32b_x32(tbase + c + 32,
                                           *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                    tmem_ld_wait();
                    if (c + W >= c_lo + SLICE) {
                        // This warp's part of the accumulator is in registers: release it.
                        release(buf);
                    }
                    const int64_t cg = col0 + c;  // first global column of the chunk
                    if (cg >= e.N) continue;
                    const int k = nchunk;
                    const int sel = k & 1;
                    ++nchunk;
                    uint8_t* sb = etile + sel * EPI_BUF_BYTES;
                    if (!args.r_tma) {
                        // The TMA store issued from this buffer two chunks ago must
                        // have finished reading it.
                        if (lane == 0) bulk_wait_read<1>();
                    } else {
                        if (r_ahead != k && lane == 0) {
                            bulk_wait_read<1>();
                            r_issue(sel, static_cast<int32_t>(cg), row0,
                                    static_cast<int32_t>(bt) * args.r_bmul);
                        }
                        // Next chunk: the rest of this tile, else the first chunk of
                        // this warp's next work item.
                        int32_t cn = static_cast<int32_t>(cg) + W, rn = row0,
                                bn = static_cast<int32_t>(bt) * args.r_bmul;
                        bool has_next = args.r_ahead && c + W < c_lo + SLICE && cn < e.N;
                        if (args.r_ahead && !has_next && t + item_stride < args.total_items)
                            has_next = first_chunk(t + item_stride, cn, rn, bn);
                        if (has_next) {
                            // its buffer was read by the store of the previous chunk
                            if (lane == 0) {
                                bulk_wait_read<0>();
                                r_issue(sel ^ 1, cn, rn, bn);
                            }
                            r_ahead = k + 1;
                        }
                    }
                    __syncwarp();
                    float y[W];
                    const bool smx = e.act == GEMM_ACT_SOFTMAX;  // v holds exp(t - max)
                    // 16-byte chunk j of this thread's row sits at position j ^ (row & 7).
                    uint8_t* rowp = sb + lane * 128;
                    // The plain case (scale only) first and compact: the general
                    // steps below are large unrolled blocks that it jumps over once.
                    if (args.epi_plain || smx) {
                        const float sc = smx ? sinv : e.alpha;
#pragma unroll
                        for (int i = 0; i < W; ++i)
                            if (i < W) y[i] = __uint_as_float(v[i]) * sc;
                    } else if (e.bias && args.bias_vec && cg + W <= e.N) {
                        // alpha * acc + bias for pairs of columns: one packed FMA each
                        const float* bp = e.bias + cg;
                        const uint64_t a2 = f2_pack(e.alpha, e.alpha);
#pragma unroll
                        for (int i = 0; i < W; i += 4)
                            if (i < W) {
                                const float4 bv = __ldg(reinterpret_cast<const float4*>(bp + i));
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                                 a2, f2_pack(bv.x, bv.y)),
                                          y[i], y[i + 1]);
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])),
                                                 a2, f2_pack(bv.z, bv.w)),
                                          y[i + 2], y[i + 3]);
                            }
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i)
                            if (i < W) y[i] = __uint_as_float(v[i]) * e.alpha;
                        if (e.bias) {
                            const float* bp = e.bias + cg;
#pragma unroll
                            for (int i = 0; i < W; ++i)
                                if (i < W && cg + i < e.N) y[i] += __ldg(bp + i);
                        }
                    }
                    if (!(args.epi_plain || smx)) {
                        if (e.act == GEMM_ACT_GELU_ERF) {
#pragma unroll
                            for (int i = 0; i < W; i += 2) gelu2_as7126(y[i], y[i + 1]);
                        } else if (e.act == GEMM_ACT_RELU) {
#pragma unroll
                            for (int i = 0; i < W; ++i)
                                if (i < W) y[i] = fmaxf(y[i], 0.0f);
                        }
                        if (e.R) {
                            if (args.r_tma) {
                                if (!mbar_wait_bounded(smem_u32(&rb[sel]), (rph >> sel) & 1u, abort_flag,
                                                       args.status, tmo)) {
                                    tc_drain(smem_u32(&rb[sel]), (rph >> sel) & 1u, tmo);
                                    return false;
                                }
                                rph ^= 1u << sel;
                                const uint64_t b2 = f2_pack(e.beta, e.beta);
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 r4 =
                                        *reinterpret_cast<const float4*>(rowp + ((j ^ (lane & 7)) << 4));
                                    f2_unpack(f2_fma(f2_pack(r4.x, r4.y), b2, f2_pack(y[4 * j], y[4 * j + 1])),
                                              y[4 * j], y[4 * j + 1]);
                                    f2_unpack(f2_fma(f2_pack(r4.z, r4.w), b2, f2_pack(y[4 * j + 2], y[4 * j + 3])),
                                              y[4 * j + 2], y[4 * j + 3]);
                                }
                            } else if (row < e.M) {
                                const float* rp = e.R + bt * e.stride_r + row * e.ldr + cg;
#pragma unroll
                                for (int i = 0; i < W; ++i)
                                    if (i < W && cg + i < e.N) y[i] += e.beta * __ldg(rp + i);
                            }
                        }
                    }  // general epilogue
                    if constexpr (W == 32) {  // FP32 out
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                                make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint32_t w4[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float lo = y[8 * j + 2 * h], hi = y[8 * j + 2 * h + 1];
                                if (e.out_dtype == GEMM_BF16) {
                                    __nv_bfloat162 p2 = __floats2bfloat162_rn(lo, hi);
                                    w4[h] = *reinterpret_cast<uint32_t*>(&p2);
                                } else {
                                    __half2 p2 = __floats2half2_rn(lo, hi);
                                    w4[h] = *reinterpret_cast<uint32_t*>(&p2);
                                }
                            }
                            *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                                make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && cg < args.n_tma) {
                        tma_store_3d(&tmC, smem_u32(sb), static_cast<int32_t>(cg), row0,
                                     static_cast<int32_t>(bt * args.c_bmul + split * args.c_smul));
                        bulk_commit();
                    }
                    if (cg + W > args.n_tma && row < e.M) {
                        // Ragged right edge: TMA stores whole 16-byte pieces, so the
                        // last < 16 bytes of each row (columns n_tma .. N-1, all in
                        // one 16-byte piece of this chunk) are copied from the
                        // shared tile by the row's own thread.
                        const int jt = static_cast<int>((args.n_tma - cg) * (args.out16 ? 2 : 4) / 16);
                        const uint4 piece =
                            *reinterpret_cast<const uint4*>(rowp + ((jt ^ (lane & 7)) << 4));
                        const int64_t base = b * e.stride_c + row * e.ldc + args.n_tma;
                        const int nrest = static_cast<int>(e.N - args.n_tma);
                        if (!args.out16) {
                            const float f[4] = {__uint_as_float(piece.x), __uint_as_float(piece.y),
                                                __uint_as_float(piece.z), __uint_as_float(piece.w)};
#pragma unroll
                            for (int t = 0; t < 3; ++t)
                                if (t < nrest) static_cast<float*>(e.C)[base + t] = f[t];
                        } else {
                            const uint32_t w[4] = {piece.x, piece.y, piece.z, piece.w};
#pragma unroll
                            for (int t = 0; t < 7; ++t)
                                if (t < nrest)
                                    static_cast<uint16_t*>(e.C)[base + t] =
                                        static_cast<uint16_t>(w[t >> 1] >> (16 * (t & 1)));
                        }
                    }
                }
                return true;
                };
                const bool cok = args.out16 ? chunk_loop(std::integral_constant<int, 64>{})
                                            : chunk_loop(std::integral_constant<int, 32>{});
                if (!cok) {
                    ok = false;
                    break;
                }
            } else {
                // C rows TMA cannot address (row stride, batch stride or base not a
                // multiple of 16 bytes, e.g. N odd).  Each thread holds one row of a
                // 32-row x 32-column chunk; the warp turns the chunk around in its
                // staging buffer so that every store (and every residual load)
                // covers 32 consecutive columns of one row instead of one column of
                // 32 rows.  The buffer has the layout of the TMA path: 16-byte piece
                // j of row r at r * 128 + ((j ^ (r & 7)) << 4), so row-wise
                // (16-byte) and column-wise (4-byte) accesses are both free of bank
                // conflicts.
                const uint32_t colx = ((lane >> 2) << 4) | ((lane & 3) << 2);  // column `lane`
                const int rows_here =
                    static_cast<int>(max(int64_t(0), min(int64_t(32), e.M - row0)));
                const bool smx = e.act == GEMM_ACT_SOFTMAX;  // v holds exp(t - max)
                const bool any_r = !smx && !args.epi_plain && e.R != nullptr;
                // The residual of a chunk goes out as asynchronous copies straight into
                // the chunk's buffer (lane = column: 32 coalesced row segments, no
                // registers held), one chunk ahead: chunk k uses buffer k & 1, and the
                // copies for chunk k + 1 are issued when chunk k starts.
                const auto r_copy = [&](uint8_t* dstb, int64_t bidx, int64_t r0, int64_t cgc,
                                        int rows, int cols) {
                    const float* rp = e.R + bidx * e.stride_r + r0 * e.ldr + cgc + lane;
#pragma unroll
                    for (int r = 0; r < 32; ++r) {
                        const bool in = r < rows && lane < cols;
                        cp_async_4(smem_u32(dstb + r * 128 + (colx ^ ((r & 7) << 4))),
                                   in ? rp + r * e.ldr : e.R, in);
                    }
                    cp_async_commit();
                };
#pragma unroll 1
                for (int c = c_lo; c < c_lo + SLICE; c += 32) {
                    const int64_t cg = col0 + c;
                    const int ncol = static_cast<int>(max(int64_t(0), min(int64_t(32), e.N - cg)));
                    const bool with_r = ncol > 0 && any_r;
                    const int k = nchunk;
                    uint8_t* sb = etile + (k & 1) * EPI_BUF_BYTES;
                    uint8_t* rowp = sb + lane * 128;
                    __syncwarp();  // the previous chunks' reads of both buffers are done
                    bool ahead = false;
                    if (with_r) {
                        if (r_ahead != k) r_copy(sb, bt, row0, cg, rows_here, ncol);
                        // next chunk: the rest of this tile, else this warp's first
                        // chunk of its next work item (never split-K: no residual there)
                        int64_t cn = cg + 32, rn = row0, bn = bt;
                        bool has_next = c + 32 < c_lo + SLICE && cn < e.N;
                        if (!has_next && t + item_stride < args.total_items) {
                            int64_t mt2, nt2;
                            tc_tile_coords(t + item_stride, args, bn, mt2, nt2);
                            cn = nt2 * BN + c_lo;
                            rn = mt2 * L::TILE_M + rank * TBM + q * 32;
                            has_next = cn < e.N;
                        }
                        if (has_next) {
                            r_copy(etile + ((k + 1) & 1) * EPI_BUF_BYTES, bn, rn, cn,
                                   static_cast<int>(max(int64_t(0), min(int64_t(32), e.M - rn))),
                                   static_cast<int>(min(int64_t(32), e.N - cn)));
                            r_ahead = k + 1;
                            ahead = true;
                        }
                    }
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), v);
                    tmem_ld_wait();
                    if (c + 32 >= c_lo + SLICE) {
                        // All of this buffer is in registers: hand it back to the MMA warp.
                        release(buf);
                    }
                    if (ncol == 0) continue;
                    ++nchunk;
                    if (with_r) {
                        // this chunk's copies (all but the newest group when one is ahead)
                        if (ahead)
                            cp_async_wait_group<1>();
                        else
                            cp_async_wait_all();
                        __syncwarp();
                    }
                    float y[32];
                    const float sc = smx ? sinv : e.alpha;
#pragma unroll
                    for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(v[i]) * sc;
                    if (!smx && !args.epi_plain) {
                        if (e.bias) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i < ncol) y[i] += __ldg(e.bias + cg + i);
                        }
                        if (e.act == GEMM_ACT_GELU_ERF) {
#pragma unroll
                            for (int i = 0; i < 32; i += 2) gelu2_as7126(y[i], y[i + 1]);
                        } else if (e.act == GEMM_ACT_RELU) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) y[i] = fmaxf(y[i], 0.0f);
                        }
                        if (with_r) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 r4 =
                                    *reinterpret_cast<const float4*>(rowp + ((j ^ (lane & 7)) << 4));
                                y[4 * j] += e.beta * r4.x;
                                y[4 * j + 1] += e.beta * r4.y;
                                y[4 * j + 2] += e.beta * r4.z;
                                y[4 * j + 3] += e.beta * r4.w;
                            }
                        }
                    }
                    // this thread's row into the buffer, then the buffer out by rows
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                            make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
                    __syncwarp();
                    if (lane < ncol) {
                        const int64_t off =
                            b * e.stride_c + static_cast<int64_t>(row0) * e.ldc + cg + lane;
                        const auto at = [&](int r) {
                            return *reinterpret_cast<const float*>(sb + r * 128 +
                                                                   (colx ^ ((r & 7) << 4)));
                        };
                        if (e.out_dtype == GEMM_F32) {
                            float* cp = static_cast<float*>(e.C) + off;
#pragma unroll 8
                            for (int r = 0; r < rows_here; ++r) cp[r * e.ldc] = at(r);
                        } else if (e.out_dtype == GEMM_BF16) {
                            __nv_bfloat16* cp = static_cast<__nv_bfloat16*>(e.C) + off;
#pragma unroll 8
                            for (int r = 0; r < rows_here; ++r) cp[r * e.ldc] = __float2bfloat16_rn(at(r));
                        } else {
                            __half* cp = static_cast<__half*>(e.C) + off;
#pragma unroll 8
                            for (int r = 0; r < rows_here; ++r) cp[r * e.ldc] = __float2half_rn(at(r));
                        }
                    }
                }
            }
        }
        // A residual load for a chunk that was never reached (the loop gave up)
        // must land before the CTA's shared memory goes away.
        if (args.epi_tma && r_ahead >= nchunk && lane == 0)
            tc_drain(smem_u32(&rb[r_ahead & 1]), (rph >> (r_ahead & 1)) & 1u, tmo);
        cp_async_wait_all();
        // Shared memory must outlive the TMA stores that read it.
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // A pair's CTAs stay resident until neither will touch the other's shared memory.
    if (PAIR) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, int STAGES, bool B_KN, int EW, bool PAIR, bool K3>
cudaError_t launch_tc_t(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                        const EpiParams& e, const LaunchCtx& lc, const EpiParams* final_epi) {
    using L = TcLayout<BN, PAIR, K3>;
    TcArgs a{};
    a.M = s.M;
    a.N = s.N;
    a.K = s.K;
    a.batch = s.batch;
    a.a_bmul = s.a_bmul;
    a.b_bmul = s.b_bmul;
    static const CUtensorMap unused_map{};
    a.epi_tma = em != nullptr;
    a.r_tma = em != nullptr && em->r_tma;
    a.r_ahead = 0;  // set below, once the grid is known
    a.out16 = e.out_dtype != GEMM_F32;
    a.c_bmul = em ? em->c_bmul : 0;
    a.c_smul = em ? em->c_smul : 0;
    a.r_bmul = em ? em->r_bmul : 0;
    a.bias_vec = e.bias && (reinterpret_cast<uintptr_t>(e.bias) % 16 == 0);
    a.epi_plain = !e.bias && e.act == GEMM_ACT_NONE && !e.R;
    a.n_tma = em ? em->n_tma : 0;
    a.m_tiles = (s.M + L::TILE_M - 1) / L::TILE_M;
    a.n_tiles = (s.N + BN - 1) / BN;
    a.tiles_per_batch = a.m_tiles * a.n_tiles;
    a.total_tiles = a.tiles_per_batch * s.batch;
    a.k_blocks = static_cast<int>((s.K + L::KE - 1) / L::KE);
    a.splits = (PAIR || K3) ? 1 : tc_effective_splits(s.K, cfg.split_k);
    a.kb_per_split = (a.k_blocks + a.splits - 1) / a.splits;
    a.total_items = a.total_tiles * a.splits;
    if (a.total_items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // 32-bit tile coordinates
    a.raster = cfg.raster_group > 0 ? cfg.raster_group : 16;
    // Instruction descriptor, kind::f16 / kind::tf32: D = F32 (bits 4-5 = 1);
    // A and B type (bits 7-9, 10-12) 0 = F16, 1 = BF16, 2 = TF32; A K-major
    // (bit 15 = 0); B K-major (bit 16 = 0) or MN-major (1); N >> 3 at bits
    // 17-22; M >> 4 at bits 24-28.
    const uint32_t ab = K3 ? 2u : dtype == GEMM_BF16 ? 1u : 0u;
    a.idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((B_KN ? 1u : 0u) << 16) |
              (static_cast<uint32_t>((BN > 256 ? 256 : BN) >> 3) << 17) |
              (static_cast<uint32_t>(L::TILE_M >> 4) << 24);
    a.e = e;
    a.status = lc.status;
    a.timeout_ns = lc.timeout_ns;
    a.flags = lc.flags;
    const int smem = tc_smem_total<BN, STAGES, EW, PAIR, K3>();
    auto kern = tc_gemm_kernel<BN, STAGES, B_KN, EW, PAIR, K3>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const CUtensorMap& mc = em ? em->c : unused_map;
    const CUtensorMap& mr = (em && em->r_tma) ? em->r : unused_map;
    cudaError_t err2;
    if (PAIR) {
        // clusters of two CTAs, as many pairs as can be resident at once
        cudaLaunchConfig_t lcfg = {};
        lcfg.blockDim = dim3(tc_threads<EW>());
        lcfg.dynamicSmemBytes = smem;
        lcfg.stream = lc.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lcfg.attrs = attr;
        lcfg.numAttrs = 1;
        int64_t pairs = cfg.num_ctas > 0 ? cfg.num_ctas / 2 : lc.num_sms / 2;
        lcfg.gridDim = dim3(static_cast<unsigned>(2 * (pairs > 0 ? pairs : 1)));
        // resident pairs per device, looked up once per instantiation and device
        static std::atomic<int> resident[kMaxDevices];
        int dev = 0;
        err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        int max_pairs = dev >= 0 && dev < kMaxDevices ? resident[dev].load() : 0;
        if (max_pairs == 0) {
            err = cudaOccupancyMaxActiveClusters(&max_pairs, kern, &lcfg);
            if (err != cudaSuccess) return err;
            if (dev >= 0 && dev < kMaxDevices) resident[dev].store(max_pairs);
        }
        if (max_pairs < 1) return cudaErrorInvalidConfiguration;
        if (pairs > max_pairs) pairs = max_pairs;
        if (pairs > a.total_items) pairs = a.total_items;
        if (pairs < 1) pairs = 1;
        lcfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
        a.r_ahead = a.r_tma && (a.k_blocks <= 8 || a.total_items <= pairs);
        err2 = cudaLaunchKernelEx(&lcfg, kern, tmA, tmB, mc, mr, a);
        return err2;
    }
    int64_t grid = cfg.num_ctas > 0 ? cfg.num_ctas : lc.num_sms;
    if (grid > a.total_items) grid = a.total_items;
    if (grid < 1) grid = 1;
    a.r_ahead = a.r_tma && (a.k_blocks <= 8 || a.total_items <= grid);
    kern<<<static_cast<unsigned>(grid), tc_threads<EW>(), smem, lc.stream>>>(tmA, tmB, mc, mr, a);
    err2 = cudaGetLastError();
    if (err2 != cudaSuccess || a.splits == 1) return err2;
    // split-K: add the partial slabs in split order and apply the real epilogue
    return launch_split_reduce(static_cast<const float*>(e.C), s.M, s.N, s.batch, a.splits,
                               *final_epi, lc);
}

// Instantiated configurations: (BN, STAGES, epilogue warps, variant, pair).
// Eight epilogue warps (variant 1) take 64 KB of staging tiles, so they pair
// with fewer stages; variant 2 is the CTA-pair kernel (32 KB stages).
#define G13_TC_CONFIGS(X)    \
    X(256, 4, 4, 0, false)   \
    X(256, 3, 4, 0, false)   \
    X(128, 6, 4, 0, false)   \
    X(128, 4, 4, 0, false)   \
    X(256, 3, 8, 1, false)   \
    X(128, 4, 8, 1, false)   \
    X(512, 1, 8, 1, false)   \
    X(256, 6, 4, 2, true)    \
    X(256, 4, 4, 2, true)    \
    X(256, 5, 8, 3, true)

template <bool B_KN>
cudaError_t launch_tc_layout(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                             const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe) {
#define G13_TC_LAUNCH(BN, ST, EW, VAR, PAIR)                                             \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR)                          \
        return launch_tc_t<BN, ST, B_KN, EW, PAIR, false>(cfg, dtype, tmA, tmB, em, s, e, lc, fe);
    G13_TC_CONFIGS(G13_TC_LAUNCH)
#undef G13_TC_LAUNCH
    return cudaErrorInvalidValue;
}

// 3xTF32 configurations: (BN, STAGES, epilogue warps, variant, pair); 64 KB stages.
#define G13_TC3_CONFIGS(X)   \
    X(256, 3, 4, 2, true)    \
    X(128, 3, 4, 0, false)

}  // namespace

cudaError_t launch_tc3(const gemm_config_t& cfg, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const TcEpiMaps* em, const Shape& s, const EpiParams& e,
                       const LaunchCtx& lc) {
#define G13_TC3_LAUNCH(BN, ST, EW, VAR, PAIR)                                              \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR)                            \
        return launch_tc_t<BN, ST, false, EW, PAIR, true>(cfg, GEMM_F32, tmA, tmB, em, s, e, lc, \
                                                          nullptr);
    G13_TC3_CONFIGS(G13_TC3_LAUNCH)
#undef G13_TC3_LAUNCH
    return cudaErrorInvalidValue;
}

size_t tc3_smem_bytes(const gemm_config_t& cfg) {
#define G13_TC3_SMEM(BN, ST, EW, VAR, PAIR)                     \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR) \
        return tc_smem_total<BN, ST, EW, PAIR, true>();
    G13_TC3_CONFIGS(G13_TC3_SMEM)
#undef G13_TC3_SMEM
    return 0;
}

size_t tc_smem_bytes(const gemm_config_t& cfg) {
    if (cfg.bm != TBM || cfg.bk != TBK) return 0;
#define G13_TC_SMEM(BN, ST, EW, VAR, PAIR)                      \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR) \
        return tc_smem_total<BN, ST, EW, PAIR, false>();
    G13_TC_CONFIGS(G13_TC_SMEM)
#undef G13_TC_SMEM
    return 0;
}

int tc_effective_splits(int64_t K, int split_k) {
    const int64_t kb = (K + TBK - 1) / TBK;
    if (split_k <= 1 || kb <= 1) return 1;
    const int64_t per = (kb + split_k - 1) / split_k;
    return static_cast<int>((kb + per - 1) / per);
}

cudaError_t launch_tc(const gemm_config_t& cfg, int dtype, int b_layout, const CUtensorMap& tmA,
                      const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                      const EpiParams& e, const LaunchCtx& lc, const EpiParams* final_epi) {
    if (tc_effective_splits(s.K, cfg.split_k) > 1 && !final_epi) return cudaErrorInvalidValue;
    if (b_layout == GEMM_B_KN)
        return launch_tc_layout<true>(cfg, dtype, tmA, tmB, em, s, e, lc, final_epi);
    return launch_tc_layout<false>(cfg, dtype, tmA, tmB, em, s, e, lc, final_epi);
}

cudaError_t tc_preload_kernels() {
    // A function-attribute query makes the runtime load a lazily loaded kernel.
    cudaFuncAttributes fa;
    cudaError_t err = cudaSuccess;
#define G13_TC_PRELOAD(BN, ST, EW, VAR, PAIR)                                                   \
    if (err == cudaSuccess)                                                                     \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, true, EW, PAIR, false>);        \
    if (err == cudaSuccess)                                                                     \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, false, EW, PAIR, false>);
    G13_TC_CONFIGS(G13_TC_PRELOAD)
#undef G13_TC_PRELOAD
    return err;
}

#undef G13_TC_CONFIGS
#undef G13_TC3_CONFIGS

}  // namespace g13
