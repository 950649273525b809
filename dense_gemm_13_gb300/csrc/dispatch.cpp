// dispatch.cpp -- validation, shape buckets and the configuration cache.
//
// "DeepGEMM", sec. 2.3 and 4.3: choose tile parameters per problem size,
// hit a cached configuration when the same shape comes back, and switch to a
// small-block kernel when M or N is small.  Buckets here:
//   * empty problems (M or N = 0) and K = 0, and M or N <= kSkinnyMax:
//     the memory-bound skinny kernel, with K split over CTAs when the large
//     operand alone would not fill the GPU;
//   * FP32 inputs: the FFMA kernel, 128x128x32 tiles;
//   * FP16/BF16 inputs: the tcgen05 kernel, 128 x BN x 64 tiles, BN chosen
//     between 128 and 256 by the number of waves the tile count needs on
//     the device's SMs (each wave costs time proportional to BN).
// Operands whose strides rule out TMA are staged into an aligned copy.
#include "dispatch.h"

#include <algorithm>
#include "internal.h"
#include <array>
#include <map>
#include <mutex>

namespace g13 {

namespace {
// Up to 4 small-operand rows the skinny kernel streams the large operand at
// HBM speed; beyond that its FMAs per loaded element make it CUDA-core bound
// (16 rows: 199 us for 16 x 6144 x 6144 BF16) and the tensor cores (with
// split-K) are faster (17 rows: 39 us).
constexpr int64_t kSkinnyMax = 4;

std::mutex g_cache_mu;
std::map<std::array<int64_t, 20>, gemm_config_t> g_cache;
int64_t g_hits = 0, g_misses = 0;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

int dtype_size(int dtype) {
    switch (dtype) {
        case GEMM_F32: return 4;
        case GEMM_F16:
        case GEMM_BF16: return 2;
        default: return 0;
    }
}

int make_problem(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                 int64_t ldc, const gemm_epilogue_t* epi, Problem* p) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    gemm_epilogue_t e;
    gemm_epilogue_init(&e);
    if (epi) e = *epi;
    if (dtype_size(dtype) == 0) return GEMM_ERR_INVALID_ARG;
    if (e.out_dtype != GEMM_F32 && e.out_dtype != GEMM_BF16 && e.out_dtype != GEMM_F16)
        return GEMM_ERR_INVALID_ARG;
    if (e.b_layout != GEMM_B_KN && e.b_layout != GEMM_B_NK) return GEMM_ERR_INVALID_ARG;
    if (e.act != GEMM_ACT_NONE && e.act != GEMM_ACT_GELU_ERF && e.act != GEMM_ACT_RELU &&
        e.act != GEMM_ACT_SOFTMAX)
        return GEMM_ERR_INVALID_ARG;
    if (e.has_bias != 0 && e.has_bias != 1) return GEMM_ERR_INVALID_ARG;
    if (e.has_residual != 0 && e.has_residual != 1) return GEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    // Sizes must fit the 32-bit coordinates of TMA boxes.
    if (M > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 31) - 256 ||
        K > (int64_t(1) << 31) - 256)
        return GEMM_ERR_UNSUPPORTED;
    if (e.batch == 0) e.batch = 1;
    if (e.batch < 0 || e.batch > (int64_t(1) << 31) - 1) return GEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(K, 1)) return GEMM_ERR_INVALID_ARG;
    const int64_t ldb_min = e.b_layout == GEMM_B_KN ? N : K;
    if (ldb < std::max<int64_t>(ldb_min, 1)) return GEMM_ERR_INVALID_ARG;
    if (ldc < std::max<int64_t>(N, 1)) return GEMM_ERR_INVALID_ARG;
    if (e.ldr == 0) e.ldr = ldc;
    if (e.has_residual && e.ldr < std::max<int64_t>(N, 1)) return GEMM_ERR_INVALID_ARG;
    if (e.stride_a < 0 || e.stride_b < 0 || e.stride_c < 0 || e.stride_r < 0)
        return GEMM_ERR_INVALID_ARG;
    if (e.batch > 1 && M > 0 && N > 0 && e.stride_c < M * ldc) return GEMM_ERR_INVALID_ARG;
    if (e.timeout_ms == 0) e.timeout_ms = 2000;
    // The row softmax runs in the tensor-core epilogue with a whole row (up to
    // 512 FP32 accumulator columns) in one CTA's TMEM.
    if (e.act == GEMM_ACT_SOFTMAX &&
        (dtype == GEMM_F32 || N > 512 || (K == 0 && M > 0 && N > 0) || e.has_residual))
        return GEMM_ERR_UNSUPPORTED;
    p->dtype = dtype;
    p->M = M;
    p->N = N;
    p->K = K;
    p->lda = lda;
    p->ldb = ldb;
    p->ldc = ldc;
    p->epi = e;
    return GEMM_OK;
}

bool stride_tma_ok(int64_t ld, int64_t bstride, int64_t batch, int esz) {
    if ((ld * esz) % 16 != 0) return false;
    if (batch > 1 && bstride != 0 && (bstride * esz) % 16 != 0) return false;
    return true;
}

static void set_staging(const Problem& p, gemm_config_t* c) {
    const int esz = dtype_size(p.dtype);
    const int64_t bt = p.epi.batch;
    if (!stride_tma_ok(p.lda, p.epi.stride_a, bt, esz)) c->stage_a = 1;
    if (!stride_tma_ok(p.ldb, p.epi.stride_b, bt, esz)) c->stage_b = 1;
}

int skinny_splits(const Problem& p, int num_sms) {
    if (p.M == 0 || p.N == 0 || p.K == 0) return 1;
    int64_t P, Q;
    int dot;
    skinny_geometry(p.M, p.N, p.epi.b_layout, &P, &Q, &dot);
    const int64_t bt = p.epi.batch;
    int64_t splits;
    if (dot) {
        // one warp per streamed row: aim for ~24 rows in flight per SM, >= 512 K per split
        splits = cdiv(static_cast<int64_t>(num_sms) * 24, bt * Q);
        splits = std::min(splits, std::max<int64_t>(1, p.K / 512));
    } else {
        // a CTA covers 32 x 16 bytes of columns with 8 warps along K: aim for a full
        // wave at the kernel's occupancy (3 CTAs per SM for one row, else 2) and
        // at least two row groups per warp
        const int64_t vw = p.dtype == GEMM_F32 ? 4 : 8;
        const int64_t ctas = cdiv(Q, 32 * vw) * bt;
        splits = cdiv(static_cast<int64_t>(num_sms) * (P == 1 ? 3 : 2), ctas);
        splits = std::min(splits, std::max<int64_t>(1, p.K / (16 * vw)));
    }
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(splits, 1024)));
}

// The TMA-streamed skinny kernel can run p: large operand rows (and batch
// stride) 16-byte aligned for TMA, and the small operand (P <= 4 rows of K, as
// FP32) fits shared memory beside the ring.
bool skinny_tma_suits(const Problem& p) {
    if (p.M == 0 || p.N == 0 || p.K == 0) return false;
    int64_t P, Q;
    int dot;
    skinny_geometry(p.M, p.N, p.epi.b_layout, &P, &Q, &dot);
    if (P > kSkinnyMax) return false;
    const bool l_is_b = p.M <= p.N;
    const int64_t ldl = l_is_b ? p.ldb : p.lda;
    const int64_t sl = l_is_b ? p.epi.stride_b : p.epi.stride_a;
    if (!stride_tma_ok(ldl, sl, p.epi.batch, dtype_size(p.dtype))) return false;
    return skinny_tma_fits(P, p.K, p.dtype, dot);
}

// Split-K for the tensor-core kernel when its tiles cannot fill the GPU (small
// M and N, long K): a rough time model -- waves of (tile, split) items, each
// limited by its MMA work or by the HBM share its SM gets -- plus the partial
// slabs' write + read and the reduction launch.  Returns 1 when splitting does
// not pay by at least 10 %.
int tc_splits(const Problem& p, int num_sms, int bn) {
    const int64_t M = p.M, N = p.N, K = p.K, bt = p.epi.batch;
    const int64_t tiles = bt * cdiv(M, 128) * cdiv(N, bn);
    const int64_t kb = cdiv(K, 64);
    if (tiles * 2 > num_sms || kb < 4) return 1;
    const double esz = dtype_size(p.dtype);
    // rows/columns a tile really reads (TMA zero-fills past the edge without traffic)
    const double rows = static_cast<double>(std::min<int64_t>(M, 128));
    const double cols = static_cast<double>(std::min<int64_t>(N, bn));
    auto model = [&](int64_t s) {
        const int64_t items = tiles * s;
        const double kpart = static_cast<double>(cdiv(kb, s)) * 64.0;
        const double t_mma = 128.0 * bn * kpart * 2.0 / 15e12;  // ~15 TFLOP/s per SM
        // one SM streams ~80 GB/s; all of them share ~6 TB/s of HBM
        const double share =
            std::min(80e9, 6e12 / static_cast<double>(std::min<int64_t>(items, num_sms)));
        const double t_mem = (rows + cols) * kpart * esz / share;
        const double waves = static_cast<double>(cdiv(items, num_sms));
        double t = waves * std::max(t_mma, t_mem);
        // the reduction pass: its slab traffic and ~2 us (its launch overlaps the
        // GEMM's tail as a programmatic dependent)
        if (s > 1) t += static_cast<double>(s) * M * N * bt * 8.0 / 6e12 + 2e-6;
        return t;
    };
    int best = 1;
    double best_t = model(1);
    for (int64_t s = 2; s <= 64 && s <= kb / 2; ++s) {
        const double t = model(s);
        if (t < best_t * 0.9) {
            best_t = t;
            best = static_cast<int>(s);
        }
    }
    return best;
}

int choose_config(const Problem& p, int num_sms, gemm_config_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    if (num_sms <= 0) num_sms = 1;
    gemm_config_t c{};
    c.split_k = 1;
    c.num_ctas = 0;
    const int64_t M = p.M, N = p.N, K = p.K, bt = p.epi.batch;
    if (p.epi.act == GEMM_ACT_SOFTMAX && M > 0 && N > 0) {
        // one tile spans the whole row: 256 columns (double-buffered TMEM) or
        // 512 (single-buffered, one 80 KB stage); 8 epilogue warps, two per
        // TMEM lane quarter, each thread half a row
        c.kernel = GEMM_KERNEL_TC;
        c.bm = 128;
        c.bk = 64;
        c.bn = N <= 256 ? 256 : 512;
        c.stages = N <= 256 ? 3 : 1;
        c.variant = 1;
        c.raster_group = static_cast<int32_t>(std::min<int64_t>(16, cdiv(M, 128)));
        set_staging(p, &c);
        *out = c;
        return GEMM_OK;
    }
    if (M == 0 || N == 0 || K == 0 || std::min(M, N) <= kSkinnyMax) {
        c.kernel = GEMM_KERNEL_SKINNY;
        c.bm = 1;
        c.bn = 1;
        c.bk = 32;
        c.stages = 1;
        c.raster_group = 1;
        c.split_k = skinny_splits(p, num_sms);
        // Dot mode (the large operand's rows hold K) streams through the TMA
        // ring once the large operand has 2^20 elements or more: GB300, BF16,
        // L2 flushed: 1 x 6144 x 6144 NK 31 vs 38 us, 6144 x 1 x 6144 31 vs 40,
        // 6144 x 4 x 6144 (a strided small operand) 44 vs 300.  Axpy mode keeps the
        // plain-load kernel, whose many CTAs spread over SMs of unequal memory
        // bandwidth better than one CTA per SM does (1 x 6144 x 6144 KN 25 vs 33 us).
        int64_t P, Q;
        int dot;
        skinny_geometry(M, N, p.epi.b_layout, &P, &Q, &dot);
        if (dot && skinny_tma_suits(p) && bt * Q * K >= (int64_t(1) << 20)) {
            c.variant = SKINNY_VARIANT_TMA;
            c.split_k = 1;  // stream-K over the stages instead of fixed K slices
        }
        *out = c;
        return GEMM_OK;
    }
    if (p.dtype == GEMM_F32 && (p.epi.flags & GEMM_FLAG_FP32_TENSOR) && K >= 256 &&
        bt * M * N >= (int64_t(1) << 20)) {
        // 3xTF32 on the tensor cores: three TF32 MMAs per K step at half the
        // BF16 rate, after an HBM-bound split pass over A and B.
        c.kernel = GEMM_KERNEL_TF32X3;
        c.bm = 128;
        c.bk = 32;
        c.stages = 3;
        const bool pair = M > 128 && N > 128 && num_sms >= 2;
        c.bn = pair ? 256 : 128;
        c.variant = pair ? TC_VARIANT_PAIR : 0;
        c.raster_group = static_cast<int32_t>(std::min<int64_t>(16, cdiv(M, pair ? 256 : 128)));
        *out = c;
        return GEMM_OK;
    }
    if (p.dtype == GEMM_F32) {
        c.kernel = GEMM_KERNEL_FFMA;
        c.bm = 128;
        c.bk = 32;
        const bool kn = p.epi.b_layout == GEMM_B_KN;
        // packed fma.rn.f32x2 main loop (KN layout): +17 % over scalar FFMA at 4096^3
        c.variant = kn ? 1 : 0;
        // Large KN problems: 128 x 256 tiles (8 x 16 per thread, one CTA per SM),
        // which need a quarter less shared-memory bandwidth per FMA than 128 x 128
        // (two CTAs per SM); 55.4 vs 51.7 TFLOPS at 4096^3 on GB300.
        const bool wide = kn && bt * M * N >= (int64_t(1) << 22);
        c.bn = wide ? 256 : 128;
        c.stages = wide ? 4 : 3;
        c.raster_group = wide ? 4 : 8;
        // When whole-tile waves would leave more than a tenth of the CTA slots
        // idle (4096^2 with 128 x 256 tiles: 512 tiles on 152 slots = 3.37
        // waves), split (tile, K-step) units evenly over a persistent grid.
        const int64_t slots = (wide ? 1 : 2) * static_cast<int64_t>(num_sms);
        const int64_t tiles = bt * cdiv(M, 128) * cdiv(N, c.bn);
        const int64_t waves = cdiv(tiles, slots);
        c.stream_k = (tiles * 10 < waves * slots * 9) ? 1 : 0;
        // A few 128 x 128 tiles (at most one per eight SMs, e.g. 256^3 or 512^2)
        // and K <= 512: split over stream-K, each tile's fix-up chain of partial
        // sums costs more than the FMAs; 32 x 32 tiles from plain loads spread the
        // work instead (GB300: 256^3 13.0 vs 25.3 us, 512^3 31.5 vs 47.6 us; with
        // longer K stream-K's split of K wins: 512 x 512 x 1024 49.9 vs 58.0 us).
        if (!wide && K <= 512 && bt * cdiv(M, 128) * cdiv(N, 128) * 8 <= num_sms &&
            cdiv(M, 32) <= 65535 && bt <= 65535) {
            c.variant = FFMA_VARIANT_SMALL;
            c.bm = c.bn = c.bk = 32;
            c.stages = 2;
            c.raster_group = 1;
            c.stream_k = 0;
            *out = c;
            return GEMM_OK;
        }
    } else {
        c.kernel = GEMM_KERNEL_TC;
        c.bm = 128;
        c.bk = 64;
        const int64_t mt = cdiv(M, 128);
        const int64_t waves256 = cdiv(bt * mt * cdiv(N, 256), num_sms);
        const int64_t waves128 = cdiv(bt * mt * cdiv(N, 128), num_sms);
        // Time per wave ~ BN / efficiency.  A 128x128x16 MMA reads 8 KB of
        // shared memory per 64 tensor-core clocks (the whole 128 B/clk), a
        // 128x256x16 one 12 KB per 128 clocks, so 128-wide tiles run at
        // roughly 4/5 of the 256-wide rate.
        if (waves128 * 128 * 5 < waves256 * 256 * 4) {
            c.bn = 128;
            c.stages = 6;
        } else {
            c.bn = 256;
            c.stages = 4;
        }
        // Short K: the epilogue (per output) weighs as much as the main loop
        // (per output, per K step), so give it eight warps -- two per TMEM lane
        // quarter -- at the cost of one or two pipeline stages.
        if (K <= 1024) {
            c.variant = 1;
            c.stages = c.bn == 256 ? 3 : 4;
        }
        c.raster_group = static_cast<int32_t>(std::min<int64_t>(16, mt));
        c.split_k = tc_splits(p, num_sms, c.bn);
        // CTA pairs (cta_group::2, 256 x 256 tiles, 6 stages) move a third less
        // operand data per SM for the same MMA work: 1876 vs 1602 TFLOPS at
        // 8192^3 and 1521 vs 1242 at 4096^3 on GB300.  A pair tile costs one SM
        // wave like a 128 x 256 tile but runs ~15 % faster; with short K the
        // 8-warp epilogue of the single-CTA kernel wins instead.
        if (c.split_k == 1 && K > 1024 && num_sms >= 2) {
            const int64_t pair_waves = cdiv(bt * cdiv(M, 256) * cdiv(N, 256), num_sms / 2);
            const int64_t cost_single =
                (c.bn == 128 ? waves128 * 128 * 5 : waves256 * 256 * 4) * 100;
            const int64_t cost_pair = pair_waves * 256 * 4 * 85;
            if (cost_pair < cost_single) {
                c.bn = 256;
                c.stages = 6;
                c.variant = TC_VARIANT_PAIR;
                c.raster_group = static_cast<int32_t>(std::min<int64_t>(16, cdiv(M, 256)));
                // C rows TMA cannot store (e.g. N odd): the per-row epilogue of a pair
                // tile outlasts its main loop with four epilogue warps, so use eight
                const int osz = dtype_size(p.epi.out_dtype);
                if ((p.ldc * osz) % 16 != 0 || (bt > 1 && (p.epi.stride_c * osz) % 16 != 0)) {
                    c.variant = TC_VARIANT_PAIR8;
                    c.stages = 5;
                }
            }
        }
        // Short K with C rows TMA can store: when a tile's main loop outlasts its
        // epilogue, CTA pairs with eight epilogue warps (5 stages) run the main
        // loop ~17 % faster than single CTAs and keep the 8-warp epilogue.  Clock64
        // traces on GB300: a 128 x 256 x 64 block takes ~700 cycles on a single
        // CTA; the epilogue of a 128 x 256 tile ~4.5 K cycles plain, ~9 K with
        // bias + GELU, ~8 K with an FP32 residual.  Measured (L2 flushed, us,
        // single -> pairs): 4096^2 x 768 BF16 out 33.3 -> 30.4, 8192^2 x 1024
        // 111.3 -> 92.3, 4096^2 x 1024 bias + GELU 42.1 -> 39.6, 6144^2 x 1000
        // + FP32 residual 99.6 -> 88.1; FFN1 (4096 x 3072 x 768, bias + GELU)
        // stays single: 29.4 vs 32.0 with pairs.
        const int osz = dtype_size(p.epi.out_dtype);
        const bool c_tma = (p.ldc * osz) % 16 == 0 && (bt == 1 || (p.epi.stride_c * osz) % 16 == 0);
        if (c.split_k == 1 && K <= 1024 && num_sms >= 2 && c_tma) {
            int64_t epi_cycles = 4500;
            if (p.epi.act == GEMM_ACT_GELU_ERF) epi_cycles += 4500;
            if (p.epi.has_residual) epi_cycles += 3500;
            if (cdiv(K, 64) * 700 > epi_cycles) {
                const int64_t pair_waves = cdiv(bt * cdiv(M, 256) * cdiv(N, 256), num_sms / 2);
                const int64_t cost_single =
                    (c.bn == 128 ? waves128 * 128 * 5 : waves256 * 256 * 4) * 100;
                const int64_t cost_pair = pair_waves * 256 * 4 * 85;
                if (cost_pair < cost_single) {
                    c.bn = 256;
                    c.stages = 5;
                    c.variant = TC_VARIANT_PAIR8;
                    c.raster_group = static_cast<int32_t>(std::min<int64_t>(16, cdiv(M, 256)));
                }
            }
        }
    }
    set_staging(p, &c);
    *out = c;
    return GEMM_OK;
}

int check_config(const Problem& p, const gemm_config_t& in, gemm_config_t* out) {
    gemm_config_t c = in;
    if (c.split_k == 0) c.split_k = 1;
    if (c.split_k < 1 || (c.split_k != 1 && c.kernel == GEMM_KERNEL_FFMA) || c.split_k > 1024)
        return GEMM_ERR_UNSUPPORTED;
    if (c.num_ctas < 0 || c.raster_group < 0) return GEMM_ERR_INVALID_ARG;
    if (p.epi.act == GEMM_ACT_SOFTMAX && c.kernel != GEMM_KERNEL_TC && p.M > 0 && p.N > 0)
        return GEMM_ERR_UNSUPPORTED;
    switch (c.kernel) {
        case GEMM_KERNEL_SKINNY:
            c.stage_a = c.stage_b = 0;
            if (c.stream_k != 0) return GEMM_ERR_UNSUPPORTED;
            if (c.variant != 0 && c.variant != SKINNY_VARIANT_TMA) return GEMM_ERR_UNSUPPORTED;
            if (c.variant == SKINNY_VARIANT_TMA) {
                if (!skinny_tma_suits(p)) return GEMM_ERR_UNSUPPORTED;
                c.split_k = 1;  // the TMA kernel balances by stream-K, num_ctas caps its grid
            }
            break;
        case GEMM_KERNEL_FFMA:
            if (p.dtype != GEMM_F32 || p.K == 0) return GEMM_ERR_UNSUPPORTED;
            if (c.variant == FFMA_VARIANT_SMALL) {
                // 32 x 32 tiles from plain loads: no stream-K, no staging
                if (c.bm != 32 || c.bn != 32 || c.bk != 32 || c.stream_k != 0)
                    return GEMM_ERR_UNSUPPORTED;
                c.stages = 2;
                c.stage_a = c.stage_b = 0;
                if (c.raster_group == 0) c.raster_group = 1;
                *out = c;
                return GEMM_OK;
            }
            if (c.variant < 0 || c.variant > 1) return GEMM_ERR_UNSUPPORTED;
            if (c.stream_k < 0 || c.stream_k > 1) return GEMM_ERR_UNSUPPORTED;
            if (c.bm != 128 || c.bk != 32) return GEMM_ERR_UNSUPPORTED;
            if (c.bn != 128 && !(c.bn == 256 && p.epi.b_layout == GEMM_B_KN))
                return GEMM_ERR_UNSUPPORTED;
            if (c.stages < 2 || c.stages > 4) return GEMM_ERR_UNSUPPORTED;
            if (c.raster_group == 0) c.raster_group = 8;
            break;
        case GEMM_KERNEL_TF32X3:
            // (BN, variant): (256, 2) CTA pairs or (128, 0) single CTAs, 3 stages
            if (p.dtype != GEMM_F32 || p.K == 0) return GEMM_ERR_UNSUPPORTED;
            if (c.stream_k != 0 || c.split_k > 1) return GEMM_ERR_UNSUPPORTED;
            if (c.bm != 128 || c.bk != 32 || c.stages != 3) return GEMM_ERR_UNSUPPORTED;
            if (!((c.bn == 256 && c.variant == TC_VARIANT_PAIR) || (c.bn == 128 && c.variant == 0)))
                return GEMM_ERR_UNSUPPORTED;
            c.stage_a = c.stage_b = 0;  // the split pass reads any stride and alignment
            if (c.raster_group == 0) c.raster_group = 16;
            *out = c;
            return GEMM_OK;
        case GEMM_KERNEL_TC:
            if (p.dtype == GEMM_F32 || p.K == 0) return GEMM_ERR_UNSUPPORTED;
            // stream-K: whole-tile epilogues only (no split-K, no row softmax)
            if (c.stream_k < 0 || c.stream_k > 1) return GEMM_ERR_UNSUPPORTED;
            if (c.stream_k && (c.split_k > 1 || p.epi.act == GEMM_ACT_SOFTMAX || !tc_has_spec(c)))
                return GEMM_ERR_UNSUPPORTED;
            if (c.bm != 128 || c.bk != 64) return GEMM_ERR_UNSUPPORTED;
            // (BN, stages) pairs with 4 epilogue warps (variant 0) or 8 (variant 1);
            // variant 2: CTA pairs on 256 x 256 tiles, no split-K
            if (!((c.variant == 0 && ((c.bn == 256 && (c.stages == 4 || c.stages == 3)) ||
                                      (c.bn == 128 && (c.stages == 6 || c.stages == 4)))) ||
                  (c.variant == 1 && ((c.bn == 256 && c.stages == 3) ||
                                      (c.bn == 128 && c.stages == 4) ||
                                      (c.bn == 512 && c.stages == 1))) ||
                  (c.variant == TC_VARIANT_PAIR && c.bn == 256 && (c.stages == 6 || c.stages == 4)) ||
                  (c.variant == TC_VARIANT_PAIR8 && c.bn == 256 && c.stages == 5)))
                return GEMM_ERR_UNSUPPORTED;

            if (tc_is_pair(c) && c.split_k > 1) return GEMM_ERR_UNSUPPORTED;
            // 512-wide tiles exist for the row softmax; the softmax needs the whole
            // row in one tile with one epilogue thread per row
            if (c.bn == 512 && p.epi.act != GEMM_ACT_SOFTMAX) return GEMM_ERR_UNSUPPORTED;
            if (p.epi.act == GEMM_ACT_SOFTMAX &&
                (tc_is_pair(c) || c.split_k > 1 || c.bn < p.N))
                return GEMM_ERR_UNSUPPORTED;
            if (c.raster_group == 0) c.raster_group = 16;
            break;
        default:
            return GEMM_ERR_INVALID_ARG;
    }
    if (c.kernel != GEMM_KERNEL_SKINNY) {
        gemm_config_t need = c;
        need.stage_a = need.stage_b = 0;
        set_staging(p, &need);
        c.stage_a = (c.stage_a || need.stage_a) ? 1 : 0;
        c.stage_b = (c.stage_b || need.stage_b) ? 1 : 0;
    }
    *out = c;
    return GEMM_OK;
}

int cached_config(const Problem& p, int num_sms, gemm_config_t* out, bool* hit) {
    const gemm_epilogue_t& e = p.epi;
    const std::array<int64_t, 20> key = {
        p.dtype,   p.M,        p.N,        p.K,        p.lda,        p.ldb,   p.ldc,
        e.b_layout, e.out_dtype, e.has_bias, e.act,    e.has_residual, e.ldr, e.batch,
        e.stride_a, e.stride_b, e.stride_c, e.stride_r, num_sms,
        static_cast<int64_t>(e.flags & GEMM_FLAG_FP32_TENSOR)};
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            ++g_hits;
            *out = it->second;
            if (hit) *hit = true;
            return GEMM_OK;
        }
    }
    gemm_config_t c;
    const int rc = choose_config(p, num_sms, &c);
    if (rc != GEMM_OK) return rc;
    std::lock_guard<std::mutex> lk(g_cache_mu);
    ++g_misses;
    g_cache.emplace(key, c);
    *out = c;
    if (hit) *hit = false;
    return GEMM_OK;
}

void cache_stats(int64_t* entries, int64_t* hits, int64_t* misses) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    if (entries) *entries = static_cast<int64_t>(g_cache.size());
    if (hits) *hits = g_hits;
    if (misses) *misses = g_misses;
}

void cache_clear() {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    g_cache.clear();
    g_hits = g_misses = 0;
}

}  // namespace g13
