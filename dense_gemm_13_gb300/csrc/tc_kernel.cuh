// tc_kernel.cuh -- BF16/FP16 GEMM on the 5th-generation tensor cores (tcgen05):
// the kernel template and its launcher, instantiated by the tc_*.cu files.
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
#pragma once
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
    // Stream-K: the first sk_dp_tiles tiles go to the holders (CTAs or pairs)
    // whole, in waves, as without it; the rest, sk_units = tiles x k_blocks
    // (tile, K block) units in tile-major order, are cut into sk_holders equal
    // ranges, one per holder, after its whole tiles.  A tile cut between
    // holders is finished by the holder of its first K block, which adds the
    // partial sums the later holders leave in their slots, in holder order.
    int sk;
    int sk_holders;
    int64_t sk_dp_tiles;
    int64_t sk_units;
    float* sk_partials;  // [CTA][TBM x BN] FP32: a CTA's partial sums of its first, cut tile
    unsigned* sk_tags;   // [CTA][8]: per epilogue warp, the epoch once its part is in place
    unsigned sk_epoch;
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
__host__ __device__ constexpr int tc_tail_end() {
    // ring + epilogue tiles + full/empty per stage + tfull/tempty x2 + drain
    // + residual barriers (2 per epilogue warp) + softmax exchange barriers (4)
    // + pair exit barriers (2) + per-stage copy counts (8) + tmem slot + abort
    // flag + softmax exchange values [2][EW][32] floats (single CTAs only: the
    // row softmax never runs on CTA pairs)
    return tc_bar_off<BN, STAGES, EW, PAIR, K3>() + (2 * STAGES + 11 + 2 * EW) * 8 + 32 + 16 +
           (PAIR ? 0 : 2 * EW * 32 * 4);
}
// Bias slices: each epilogue warp keeps its columns' bias for two tiles
// ([EW][2][SLICE] floats = 32 * BN bytes), loaded one tile ahead, where the
// configuration leaves room for them (otherwise the bias is read from global
// memory chunk by chunk).
template <int BN, int STAGES, int EW, bool PAIR, bool K3>
__host__ __device__ constexpr int tc_bias_off() {
    return (tc_tail_end<BN, STAGES, EW, PAIR, K3>() + 15) & ~15;
}
constexpr int kMaxDynSmem = 232448;  // 227 KB per block on sm_103
// Stream-K finishers bring a holder's partial sums (128 rows x BN FP32) into
// the idle stage ring.
template <int BN, int STAGES, bool PAIR, bool K3>
__host__ __device__ constexpr bool tc_sk_ring_ok() {
    return STAGES * TcLayout<BN, PAIR, K3>::STAGE_BYTES >= TBM * BN * 4;
}
template <int BN, int STAGES, int EW, bool PAIR, bool K3>
__host__ __device__ constexpr bool tc_bias_smem() {
    return 1024 + tc_bias_off<BN, STAGES, EW, PAIR, K3>() + 32 * BN <= kMaxDynSmem;
}
template <int BN, int STAGES, int EW, bool PAIR, bool K3>
__host__ __device__ constexpr int tc_smem_total() {
    return 1024 + (tc_bias_smem<BN, STAGES, EW, PAIR, K3>()
                       ? tc_bias_off<BN, STAGES, EW, PAIR, K3>() + 32 * BN
                       : tc_tail_end<BN, STAGES, EW, PAIR, K3>());
}

// A CTA's (pair's) work item at cursor `cur`: a tile (split-K: a tile and a
// split) and its K-block range, and the cursor of the CTA's next item.  Data
// parallel and split-K: cursors are item indices, stepping by the number of
// holders (CTAs or pairs).  Stream-K: cursors are unit indices; a whole tile
// steps by the number of holders, then jumps to the holder's stream-K range,
// where an item runs to the end of its tile or of the range.
struct TcItem {
    int64_t tile;
    int split, kb_lo, kb_hi;
    int64_t next;
};
__device__ __forceinline__ int64_t tc_sk_lo(const TcArgs& a, int64_t holder) {
    return holder * a.sk_units / a.sk_holders;
}
template <bool SK>
__device__ __forceinline__ TcItem tc_item(const TcArgs& a, int64_t cur, int64_t stride, int64_t end,
                                          int64_t holder) {
    TcItem it;
    if constexpr (SK) {
        const int64_t kb = a.k_blocks;
        const int64_t dp_units = a.sk_dp_tiles * kb;
        it.tile = cur / kb;
        it.split = 0;
        if (cur < dp_units) {  // a whole tile
            it.kb_lo = 0;
            it.kb_hi = a.k_blocks;
            it.next = it.tile + stride < a.sk_dp_tiles ? (it.tile + stride) * kb
                                                        : dp_units + tc_sk_lo(a, holder);
        } else {
            it.kb_lo = static_cast<int>(cur - it.tile * kb);
            const int64_t hi = min(end, (it.tile + 1) * kb);
            it.kb_hi = static_cast<int>(hi - it.tile * kb);
            it.next = hi;
        }
    } else {
        it.split = static_cast<int>(cur / a.total_tiles);
        it.tile = cur - it.split * a.total_tiles;
        it.kb_lo = it.split * a.kb_per_split;
        it.kb_hi = min(a.k_blocks, it.kb_lo + a.kb_per_split);
        it.next = cur + stride;
    }
    return it;
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

template <int BN, int STAGES, bool B_KN, int EW, bool PAIR, bool K3, int EK, bool SK>
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
    const int64_t holder = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
    const int64_t n_holders = PAIR ? (gridDim.x >> 1) : gridDim.x;
    // This CTA's (pair's) work: cursors w_begin .. w_end (see tc_item).
    const int64_t sk_base = args.sk_dp_tiles * args.k_blocks;  // first stream-K unit
    const int64_t w_begin = !SK ? holder
                            : holder < args.sk_dp_tiles ? holder * args.k_blocks
                                                        : sk_base + tc_sk_lo(args, holder);
    const int64_t w_end = SK ? sk_base + tc_sk_lo(args, holder + 1) : args.total_items;
    const int64_t w_stride = n_holders;

    if (warp == 0 && lane == 0) {
        // a kernel launched after this one as its programmatic dependent (the
        // split-K reduction) may start; it waits for this grid before its reads
        griddep_launch();
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

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const bool stall = ((args.flags & GEMM_FLAG_TEST_STALL) && blockIdx.x == 0) ||
                               ((args.flags & GEMM_FLAG_TEST_STALL_PEER) && blockIdx.x == 1);
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;  // per stage: armed and not yet seen consumed
            bool ok = true;
            // A staging copy launched just before this kernel (programmatic
            // dependent launch) must have finished before the first operand load.
            griddep_wait();
            for (int64_t cur = w_begin; ok && cur < w_end;) {
                const bool first_it = cur == w_begin;
                const TcItem it = tc_item<SK>(args, cur, w_stride, w_end, holder);
                cur = it.next;
                int64_t b, mt, nt;
                tc_tile_coords(it.tile, args, b, mt, nt);
                // this CTA's rows of A and columns of B
                const int32_t m0 = static_cast<int32_t>(mt * L::TILE_M + rank * TBM);
                const int32_t n0 = static_cast<int32_t>(nt * BN + rank * L::B_ROWS);
                const int kb_lo = it.kb_lo;
                const int kb_hi = it.kb_hi;
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, args.status,
                                           tmo)) {
                        ok = false;
                        break;
                    }
                    armed &= ~(1u << s);  // the previous use of this stage was consumed
                    const bool skip = stall && first_it && kb == kb_lo;
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
            for (int64_t cur = w_begin; ok && cur < w_end; ++lt) {
                const TcItem it = tc_item<SK>(args, cur, w_stride, w_end, holder);
                cur = it.next;
                const int buf = NBUF == 1 ? 0 : (lt & 1);
                const uint32_t tph = static_cast<uint32_t>(NBUF == 1 ? lt : (lt >> 1)) & 1u;
                if (!mbar_wait_bounded(smem_u32(&tempty[buf]), tph ^ 1u, abort_flag, args.status,
                                       tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                const int kb_lo = it.kb_lo;
                const int kb_hi = it.kb_hi;
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
        // First chunk of `tile` for this warp: its column, row and residual batch
        // coordinate; false when the tile has no columns for this warp.
        const auto first_chunk = [&](int64_t tile, int32_t& cg, int32_t& r0, int32_t& bc) {
            int64_t bidx, mt2, nt2;
            tc_tile_coords(tile, args, bidx, mt2, nt2);
            cg = static_cast<int32_t>(nt2) * BN + c_lo;
            r0 = static_cast<int32_t>(mt2) * L::TILE_M + static_cast<int32_t>(rank * TBM + q * 32);
            bc = static_cast<int32_t>(bidx) * args.r_bmul;
            return cg < e.N;
        };
        // The first item that runs the chunk loop and its position (under
        // stream-K the first item can be a later K range of a cut tile, whose
        // partial sums go to the slot instead).
        int64_t epi0_tile = -1;
        int epi0_lt = 0;
        if (w_begin < w_end) {
            const TcItem i0 = tc_item<SK>(args, w_begin, w_stride, w_end, holder);
            if (!(SK && i0.kb_lo > 0)) {
                epi0_tile = i0.tile;
            } else if (i0.next < w_end) {
                epi0_tile = tc_item<SK>(args, i0.next, w_stride, w_end, holder).tile;
                epi0_lt = 1;
            }
        }
        // C rows TMA cannot address: the four-byte residual copies of the per-row
        // path wait on DRAM one chunk at a time, so with a short main loop (K of
        // at most 8 blocks: the epilogue is the kernel's work) the warp asks L2
        // for its rows of a work item's residual an item ahead (the first item's
        // at the start).  With longer K the requests compete with the operand
        // loads and cost more than they save.
        const bool r_pf = (EK == TC_EK_ANY || EK == TC_EK_ROWS) && !args.epi_tma &&
                          args.k_blocks <= 8 && e.R != nullptr && !args.epi_plain &&
                          e.act != GEMM_ACT_SOFTMAX;
        const auto r_prefetch = [&](int64_t tile) {
            int64_t bidx, mt2, nt2;
            tc_tile_coords(tile, args, bidx, mt2, nt2);
            const int64_t r = mt2 * L::TILE_M + rank * TBM + q * 32 + lane;
            const int64_t c0 = nt2 * BN + c_lo;
            if (r >= e.M || c0 >= e.N) return;
            const int64_t n = min(int64_t(SLICE), e.N - c0);
            const float* p = e.R + bidx * e.stride_r + r * e.ldr + c0;
            // one element per 128-byte line of the row segment, and its last
            for (int64_t i = 0; i < n; i += 32) prefetch_l2(p + i);
            prefetch_l2(p + n - 1);
        };
        if (r_pf && epi0_tile >= 0) r_prefetch(epi0_tile);
        if (args.r_ahead && epi0_tile >= 0) {
            int32_t cg, r0, bidx;
            if (first_chunk(epi0_tile, cg, r0, bidx)) {
                if (lane == 0) r_issue(0, cg, r0, bidx);
                r_ahead = 0;
            }
        }
        // Bias in shared memory (TMA epilogue, where the configuration has room):
        // the warp copies its columns' bias for its next work item while it
        // works on the current one, by asynchronous copies into the other half
        // of its two-item area; the copies of one item form one cp.async group.
        constexpr bool BSM = tc_bias_smem<BN, STAGES, EW, PAIR, K3>();
        const bool bias_pf =
            BSM && args.epi_tma && e.bias != nullptr && e.act != GEMM_ACT_SOFTMAX;
        float* bias_sm = reinterpret_cast<float*>(smem + tc_bias_off<BN, STAGES, EW, PAIR, K3>()) +
                         ew * 2 * SLICE;
        const auto b_issue = [&](int64_t tile, int sel) {
            int64_t bidx, mt2, nt2;
            tc_tile_coords(tile, args, bidx, mt2, nt2);
            const int64_t c0 = nt2 * BN + c_lo;
            float* dst = bias_sm + sel * SLICE;
            for (int i = 4 * lane; i < SLICE; i += 128) {
                const int64_t gc = c0 + i;
                if (args.bias_vec) {
                    const int64_t nv = min(max(e.N - gc, int64_t(0)), int64_t(4));
                    cp_async_16z(smem_u32(dst + i), nv > 0 ? e.bias + gc : e.bias,
                                 static_cast<uint32_t>(4 * nv));
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const bool in = gc + u < e.N;
                        cp_async_4(smem_u32(dst + i + u), in ? e.bias + gc + u : e.bias, in);
                    }
                }
            }
            cp_async_commit();
        };
        if (bias_pf && epi0_tile >= 0) b_issue(epi0_tile, epi0_lt & 1);
        bool ok = true;
        int lt = 0;
        for (int64_t cur = w_begin; ok && cur < w_end; ++lt) {
            const TcItem it = tc_item<SK>(args, cur, w_stride, w_end, holder);
            cur = it.next;
            const bool has_nx = cur < w_end;  // another item follows
            // The tile of the next item that runs the chunk loop (under stream-K a
            // cut tile's later K range can come between: its sums go to the slot).
            const auto next_epi_tile = [&](int64_t& tile) -> bool {
                for (int64_t c = cur; c < w_end;) {
                    const TcItem ni = tc_item<SK>(args, c, w_stride, w_end, holder);
                    if (!(SK && ni.kb_lo > 0)) {
                        tile = ni.tile;
                        return true;
                    }
                    c = ni.next;
                }
                return false;
            };
            if (r_pf) {
                int64_t ntile;
                if (next_epi_tile(ntile)) r_prefetch(ntile);
            }
            const int buf = NBUF == 1 ? 0 : (lt & 1);
            const uint32_t tph = static_cast<uint32_t>(NBUF == 1 ? lt : (lt >> 1)) & 1u;
            const bool b_next = bias_pf && has_nx && lt + 1 > epi0_lt;
            if (b_next) {
                __syncwarp();  // every lane is done with the area's other half (item lt - 1)
                b_issue(tc_item<SK>(args, cur, w_stride, w_end, holder).tile, (lt + 1) & 1);
            }
            if (!mbar_wait_bounded(smem_u32(&tfull[buf]), tph, abort_flag, args.status, tmo)) break;
            tc_fence_after();
            const int split = it.split;
            int64_t bt, mt, nt;
            tc_tile_coords(it.tile, args, bt, mt, nt);
            // output batch index: the partial-sum slab (batch, split) under split-K
            const int64_t b = args.splits > 1 ? bt * args.splits + split : bt;
            const int32_t row0 = static_cast<int32_t>(mt * L::TILE_M + rank * TBM + q * 32);
            const int64_t row = row0 + lane;
            const int64_t col0 = nt * BN;
            const uint32_t tbase = tmem_base + lane_base + static_cast<uint32_t>(buf * BN);
            if (SK && it.kb_lo > 0) {
                // A later K range of a tile that an earlier holder finishes: this
                // warp's 32 rows x SLICE columns of partial sums go to the CTA's
                // slot as [group][16-byte piece][lane] (each store instruction of
                // the warp covers 512 contiguous bytes), then the warp's tag
                // takes this launch's epoch.
                float4* wp = reinterpret_cast<float4*>(args.sk_partials +
                                                       static_cast<int64_t>(blockIdx.x) * (TBM * BN)) +
                             ew * 8 * SLICE;
#pragma unroll 1
                for (int g = 0; g < SLICE / 32; ++g) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c_lo + 32 * g, v);
                    tmem_ld_wait();
                    if (g == SLICE / 32 - 1) release(buf);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(wp + g * 256 + j * 32 + lane,
                               make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                           __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                }
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    st_release_gpu(args.sk_tags + static_cast<int64_t>(blockIdx.x) * 8 + ew, args.sk_epoch);
                continue;
            }
            // The first K range of a cut tile: the partial sums of its later K
            // ranges are in the slots of the holders after this one up to d_end
            // (those with non-empty ranges), added to this CTA's in holder order
            // (deterministic).  Lane 0 waits (bounded) for their tags.
            int64_t d_end = holder + 1;
            if (SK && it.kb_hi < args.k_blocks) {
                const int64_t tile_end = (it.tile + 1) * args.k_blocks;
                while (d_end < args.sk_holders && sk_base + tc_sk_lo(args, d_end) < tile_end) ++d_end;
            }
            // holder d's CTA (this CTA's rank in a pair); -1: d's range is empty
            const auto contrib_cta = [&](int64_t d) -> int64_t {
                if (tc_sk_lo(args, d) == tc_sk_lo(args, d + 1)) return -1;
                return PAIR ? 2 * d + rank : d;
            };
            int nd = static_cast<int>(d_end - holder - 1);  // 0: nothing to add
            if (nd) {
                int tok = 1;
                if (lane == 0) {
                    for (int64_t d = holder + 1; d < d_end && tok; ++d) {
                        const int64_t cta = contrib_cta(d);
                        if (cta < 0) continue;
                        const unsigned* tg = args.sk_tags + cta * 8 + ew;
                        const uint64_t t0 = globaltimer_ns();
                        while (ld_acquire_gpu(tg) != args.sk_epoch) {
                            if (*abort_flag) {
                                tok = 0;
                                break;
                            }
                            if (globaltimer_ns() - t0 > tmo) {
                                *abort_flag = 1u;
                                atomicOr(args.status, DEVERR_TIMEOUT);
                                tok = 0;
                                break;
                            }
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, tok, 0)) {
                    ok = false;
                    break;
                }
            }
            // The CTA's last item, so its stage ring is idle (every MMA of the
            // item has completed): each holder's partial sums for this warp come
            // into the warp's share of the ring by asynchronous copies.  The
            // first holder's stay there and are added as the chunk loops read
            // the accumulator (ring_add); any further holders' are added to the
            // accumulator in TMEM beforehand, group by group (a fixed order:
            // deterministic).
            const float4* rs = reinterpret_cast<const float4*>(smem) + ew * (8 * SLICE);
            bool ring_add = false;
            if (nd && !has_nx) {
                float4* rw = reinterpret_cast<float4*>(smem) + ew * (8 * SLICE);
                const auto fetch = [&](int64_t cta) {
                    const float4* src =
                        reinterpret_cast<const float4*>(args.sk_partials + cta * (TBM * BN)) +
                        ew * 8 * SLICE;
                    for (int k = lane; k < 8 * SLICE; k += 32) cp_async_16z(smem_u32(rw + k), src + k, 16);
                    cp_async_commit();
                    cp_async_wait_all();
                    __syncwarp();
                };
                int64_t first = -1;
#pragma unroll 1
                for (int64_t d = holder + 1; d < d_end; ++d) {
                    const int64_t cta = contrib_cta(d);
                    if (cta < 0) continue;
                    if (first < 0) {
                        first = cta;
                        continue;
                    }
                    fetch(cta);
#pragma unroll 1
                    for (int g = 0; g < SLICE / 32; ++g) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tbase + c_lo + 32 * g, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 pv = rw[g * 256 + j * 32 + lane];
                            v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + pv.x);
                            v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + pv.y);
                            v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + pv.z);
                            v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + pv.w);
                        }
                        tmem_st_32x32b_x32(tbase + c_lo + 32 * g, v);
                    }
                    tmem_st_wait();
                    __syncwarp();  // every lane is done with the ring before the next copies
                }
                if (first >= 0) {
                    fetch(first);
                    ring_add = true;
                }
                nd = 0;
            }
            // Adds the first holder's partial sums of 32-column group g (in the ring) to v.
            const auto add_ring = [&](uint32_t (&v)[32], int g) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 pv = rs[g * 256 + j * 32 + lane];
                    v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + pv.x);
                    v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + pv.y);
                    v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + pv.z);
                    v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + pv.w);
                }
            };
            // Adds the later K ranges' partial sums of 32-column group g of this
            // warp's slice to v, from global memory (an item with another item
            // after it, whose loads use the ring).
            const auto add_partials = [&](uint32_t (&v)[32], int g) {
#pragma unroll 1
                for (int64_t d = holder + 1; d < d_end; ++d) {
                    const int64_t cta = contrib_cta(d);
                    if (cta < 0) continue;
                    const float4* pp = reinterpret_cast<const float4*>(args.sk_partials + cta * (TBM * BN)) +
                                       ew * 8 * SLICE + g * 256 + lane;
                    float4 pv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) pv[j] = __ldcg(pp + j * 32);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + pv[j].x);
                        v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + pv[j].y);
                        v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + pv[j].z);
                        v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + pv[j].w);
                    }
                }
            };
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
            if ((EK == TC_EK_ANY || EK == TC_EK_SOFTMAX) && e.act == GEMM_ACT_SOFTMAX) {
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
            if (EK != TC_EK_ROWS && (EK != TC_EK_ANY || args.epi_tma)) {
            if constexpr (EK != TC_EK_ROWS) {
                if (bias_pf) {
                    // this item's bias slice (the group issued one item ago)
                    if (b_next)
                        cp_async_wait_group<1>();
                    else
                        cp_async_wait_all();
                    __syncwarp();
                }
                const float* bsm = bias_sm + (lt & 1) * SLICE;
                // The warp walks its slice in 32-column groups: the TMEM load of
                // group g + 1 is in flight while group g is computed (two
                // register sets, taken in turn).  An output
                // chunk is W columns = 128 bytes of a row (W = 32 FP32 or 64
                // 16-bit, compiled per width so the arrays are exactly sized):
                // its groups go into one 128B-swizzled staging buffer, which one
                // lane writes out with a TMA store.  Returns false when a
                // residual wait gave up.
                const auto chunk_loop = [&](auto w_tag, auto k_tag) -> bool {
                constexpr int W = decltype(w_tag)::value;
                // Epilogue steps compiled in: 0 scale only; 1 bias, ReLU and / or
                // residual; 3 GELU with or without bias, no residual; 4 any of
                // them chosen at run time (also the row softmax's final scaling).
                constexpr int KIND = decltype(k_tag)::value;
                constexpr int G = W / 32;       // groups per chunk
                constexpr int NG = SLICE / 32;  // groups in the slice
                static_assert(NG % 2 == 0, "groups are taken in pairs");
                uint32_t va[32], vb[32];
                tmem_ld_32x32b_x32(tbase + c_lo, va);
                bool live = false;  // the current chunk has columns inside the matrix
                int sel = 0;
                uint8_t* sb = etile;
                uint8_t* rowp = etile;
                // Group g from v (loaded by the previous step); starts the load of
                // group g + 1 into vn.
                const auto group = [&](int g, uint32_t (&v)[32], uint32_t (&vn)[32]) -> bool {
                    tmem_ld_wait_regs(v);
                    if (g + 1 < NG)
                        tmem_ld_32x32b_x32(tbase + c_lo + 32 * (g + 1), vn);
                    else
                        release(buf);  // this warp's part of the accumulator is in registers
                    if (ring_add)
                        add_ring(v, g);
                    else if (nd)
                        add_partials(v, g);
                    const int h = g % G;                       // group within its chunk
                    const int64_t cq = col0 + c_lo + 32 * g;   // first column of the group
                    const int64_t cg = cq - 32 * h;            // first column of the chunk
                    if (h == 0) {
                        live = cg < e.N;
                        if (!live) return true;
                        const int k = nchunk;
                        sel = k & 1;
                        ++nchunk;
                        sb = etile + sel * EPI_BUF_BYTES;
                        rowp = sb + lane * 128;
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
                            bool has_next = args.r_ahead && g + G < NG && cn < e.N;
                            int64_t ntile;
                            if (args.r_ahead && !has_next && next_epi_tile(ntile))
                                has_next = first_chunk(ntile, cn, rn, bn);
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
                    } else if (!live) {
                        return true;
                    }
                    float y[32];
                    const bool smx = (KIND == 4 || EK == TC_EK_SOFTMAX) && e.act == GEMM_ACT_SOFTMAX;  // v: exp(t - max)
                    if (KIND == 0 || (KIND == 4 && (args.epi_plain || smx))) {
                        const float sc = smx ? sinv : e.alpha;
#pragma unroll
                        for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(v[i]) * sc;
                    } else {
                        if (bias_pf || (e.bias && args.bias_vec && cq + 32 <= e.N)) {
                            // alpha * acc + bias for pairs of columns: one packed FMA each
                            const uint64_t a2 = f2_pack(e.alpha, e.alpha);
                            const float* bp = bias_pf ? bsm + 32 * g : e.bias + cq;
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                const float4 bv = bias_pf ? *reinterpret_cast<const float4*>(bp + i)
                                                          : __ldg(reinterpret_cast<const float4*>(bp + i));
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                                 a2, f2_pack(bv.x, bv.y)),
                                          y[i], y[i + 1]);
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])),
                                                 a2, f2_pack(bv.z, bv.w)),
                                          y[i + 2], y[i + 3]);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(v[i]) * e.alpha;
                            if (e.bias) {
                                const float* bp = e.bias + cq;
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (cq + i < e.N) y[i] += __ldg(bp + i);
                            }
                        }
                        if (KIND == 3 || (KIND == 4 && e.act == GEMM_ACT_GELU_ERF)) {
#pragma unroll
                            for (int i = 0; i < 32; i += 2) gelu2_as7126(y[i], y[i + 1]);
                        } else if (KIND != 3 && e.act == GEMM_ACT_RELU) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) y[i] = fmaxf(y[i], 0.0f);
                        }
                        if (KIND != 3 && e.R) {
                            if (args.r_tma) {  // FP32 out: one group per chunk
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
                                const float* rp = e.R + bt * e.stride_r + row * e.ldr + cq;
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (cq + i < e.N) y[i] += e.beta * __ldg(rp + i);
                            }
                        }
                    }
                    // 16-byte piece j of this thread's row sits at position j ^ (row & 7).
                    if constexpr (W == 32) {  // FP32 out
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                                make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t w4[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float lo = y[8 * j + 2 * u], hi = y[8 * j + 2 * u + 1];
                                if (e.out_dtype == GEMM_BF16) {
                                    __nv_bfloat162 p2 = __floats2bfloat162_rn(lo, hi);
                                    w4[u] = *reinterpret_cast<uint32_t*>(&p2);
                                } else {
                                    __half2 p2 = __floats2half2_rn(lo, hi);
                                    w4[u] = *reinterpret_cast<uint32_t*>(&p2);
                                }
                            }
                            *reinterpret_cast<uint4*>(rowp + (((4 * h + j) ^ (lane & 7)) << 4)) =
                                make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    if (h != G - 1) return true;
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
                            for (int u = 0; u < 3; ++u)
                                if (u < nrest) static_cast<float*>(e.C)[base + u] = f[u];
                        } else {
                            const uint32_t w[4] = {piece.x, piece.y, piece.z, piece.w};
#pragma unroll
                            for (int u = 0; u < 7; ++u)
                                if (u < nrest)
                                    static_cast<uint16_t*>(e.C)[base + u] =
                                        static_cast<uint16_t>(w[u >> 1] >> (16 * (u & 1)));
                        }
                    }
                    return true;
                };
#pragma unroll 1
                for (int g = 0; g < NG; g += 2) {
                    if (!group(g, va, vb) || !group(g + 1, vb, va)) {
                        tmem_ld_wait();  // no load left in flight
                        return false;
                    }
                }
                return true;
                };
                const auto run_kind = [&](auto w_tag) -> bool {
                    constexpr int KIND = EK == TC_EK_PLAIN || EK == TC_EK_SOFTMAX ? 0 : EK == TC_EK_BIAS ? 1
                                         : EK == TC_EK_GELU ? 3 : 4;
                    return chunk_loop(w_tag, std::integral_constant<int, KIND>{});
                };
                const bool cok = args.out16 ? run_kind(std::integral_constant<int, 64>{})
                                            : run_kind(std::integral_constant<int, 32>{});
                if (!cok) {
                    ok = false;
                    break;
                }
            }
            } else if constexpr (EK == TC_EK_ANY || EK == TC_EK_ROWS) {
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
                        int64_t ntile;
                        if (!has_next && next_epi_tile(ntile)) {
                            int64_t mt2, nt2;
                            tc_tile_coords(ntile, args, bn, mt2, nt2);
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
                    if (ring_add)
                        add_ring(v, (c - c_lo) >> 5);
                    else if (nd)
                        add_partials(v, (c - c_lo) >> 5);
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

// Splits the tiles between whole-tile waves and the stream-K part for
// `holders` CTAs (pairs): the remainder of the last wave goes to stream-K, with
// one more whole wave when the remainder is under half a wave (so that every
// holder's stream-K range is at least one tile long).
inline void tc_sk_split(TcArgs& a, int64_t holders) {
    const int64_t T = a.total_tiles, P = holders > 0 ? holders : 1;
    const int64_t r = T % P;
    int64_t t_sk = r == 0 ? 0 : (T >= P + r && 2 * r < P ? P + r : r);
    if (T < P) t_sk = T;
    a.sk_dp_tiles = T - t_sk;
    a.sk_units = t_sk * a.k_blocks;
    a.sk_holders = static_cast<int>(P);
}

template <int BN, int STAGES, bool B_KN, int EW, bool PAIR, bool K3, int EK, bool SK>
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
    a.sk = SK ? 1 : 0;
    if ((cfg.stream_k != 0) != SK) return cudaErrorInvalidValue;
    if (SK) {
        // stream-K: whole tiles' epilogues only (no split-K slabs, no row softmax)
        if (a.splits != 1 || e.act == GEMM_ACT_SOFTMAX || !lc.sk_partials || !lc.sk_tags ||
            lc.sk_grid < (PAIR ? 2 : 1))
            return cudaErrorInvalidValue;
        if (!tc_sk_ring_ok<BN, STAGES, PAIR, K3>()) return cudaErrorInvalidValue;
        a.sk_partials = lc.sk_partials;
        a.sk_tags = lc.sk_tags;
        a.sk_epoch = lc.sk_epoch;
    }
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
    static_assert(tc_smem_total<BN, STAGES, EW, PAIR, K3>() <= kMaxDynSmem, "shared memory");
    const int smem = tc_smem_total<BN, STAGES, EW, PAIR, K3>();
    auto kern = tc_gemm_kernel<BN, STAGES, B_KN, EW, PAIR, K3, EK, SK>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const CUtensorMap& mc = em ? em->c : unused_map;
    const CUtensorMap& mr = (em && em->r_tma) ? em->r : unused_map;
    cudaError_t err2;
    // Stream-K launches are cooperative: every CTA a finisher waits for is resident.
    cudaLaunchAttribute coop;
    coop.id = cudaLaunchAttributeCooperative;
    coop.val.cooperative = 1;
    if (PAIR) {
        // clusters of two CTAs, as many pairs as can be resident at once
        cudaLaunchConfig_t lcfg = {};
        lcfg.blockDim = dim3(tc_threads<EW>());
        lcfg.dynamicSmemBytes = smem;
        lcfg.stream = lc.stream;
        cudaLaunchAttribute attr[2];
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
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
        if (a.sk) {
            if (pairs > lc.sk_grid / 2) pairs = lc.sk_grid / 2;  // partial-sum slots
            if (pairs > a.total_tiles * a.k_blocks) pairs = a.total_tiles * a.k_blocks;
            tc_sk_split(a, pairs);
            attr[1] = coop;
            lcfg.numAttrs = 2;
        } else {
            if (pairs > a.total_items) pairs = a.total_items;
            if (lc.pdl) lcfg.numAttrs = 2;  // programmatic dependent of the staging copy
        }
        if (pairs < 1) pairs = 1;
        lcfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
        // residual lookahead: short K, or at most about one tile per pair
        a.r_ahead = a.r_tma && (a.k_blocks <= 8 || (a.sk ? a.sk_units <= 2 * a.k_blocks * pairs
                                                          : a.total_items <= pairs));
        err2 = cudaLaunchKernelEx(&lcfg, kern, tmA, tmB, mc, mr, a);
        return err2;
    }
    int64_t grid = cfg.num_ctas > 0 ? cfg.num_ctas : lc.num_sms;
    if (a.sk) {
        if (grid > lc.sk_grid) grid = lc.sk_grid;
        if (grid > a.total_tiles * a.k_blocks) grid = a.total_tiles * a.k_blocks;
        tc_sk_split(a, grid);
    } else if (grid > a.total_items) {
        grid = a.total_items;
    }
    if (grid < 1) grid = 1;
    a.r_ahead = a.r_tma && (a.k_blocks <= 8 || (a.sk ? a.sk_units <= 2 * a.k_blocks * grid
                                                      : a.total_items <= grid));
    if (a.sk) {
        cudaLaunchConfig_t lcfg = {};
        lcfg.gridDim = dim3(static_cast<unsigned>(grid));
        lcfg.blockDim = dim3(tc_threads<EW>());
        lcfg.dynamicSmemBytes = smem;
        lcfg.stream = lc.stream;
        lcfg.attrs = &coop;
        lcfg.numAttrs = 1;
        return cudaLaunchKernelEx(&lcfg, kern, tmA, tmB, mc, mr, a);
    }
    if (lc.pdl) {
        // a programmatic dependent of the staging copy just before it
        cudaLaunchConfig_t lcfg = {};
        lcfg.gridDim = dim3(static_cast<unsigned>(grid));
        lcfg.blockDim = dim3(tc_threads<EW>());
        lcfg.dynamicSmemBytes = smem;
        lcfg.stream = lc.stream;
        cudaLaunchAttribute pdl;
        pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl.val.programmaticStreamSerializationAllowed = 1;
        lcfg.attrs = &pdl;
        lcfg.numAttrs = 1;
        err2 = cudaLaunchKernelEx(&lcfg, kern, tmA, tmB, mc, mr, a);
    } else {
        kern<<<static_cast<unsigned>(grid), tc_threads<EW>(), smem, lc.stream>>>(tmA, tmB, mc, mr, a);
        err2 = cudaGetLastError();
    }
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

// The configurations the dispatcher picks, which also come as kernels
// specialised to one epilogue kind (TC_EK_PLAIN / BIAS / GELU) and as
// stream-K kernels (any epilogue).
#define G13_TC_SPEC_CONFIGS(X) \
    X(256, 4, 4, 0, false)     \
    X(128, 6, 4, 0, false)     \
    X(256, 3, 8, 1, false)     \
    X(128, 4, 8, 1, false)     \
    X(256, 6, 4, 2, true)      \
    X(256, 5, 8, 3, true)

// The configurations the dispatcher picks for the row softmax, which also come
// as kernels holding only the softmax epilogue (TC_EK_SOFTMAX).
#define G13_TC_SOFTMAX_CONFIGS(X) \
    X(256, 3, 8, 1, false)        \
    X(512, 1, 8, 1, false)

// 3xTF32 configurations: (BN, STAGES, epilogue warps, variant, pair); 64 KB stages.
#define G13_TC3_CONFIGS(X)   \
    X(256, 3, 4, 2, true)    \
    X(128, 3, 4, 0, false)

}  // namespace
}  // namespace g13
