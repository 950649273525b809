// aux_kernels.cu -- operand staging copy and the memory-bound skinny kernel.
//
// Staging: TMA needs 16-byte-aligned base addresses and row strides.  When a
// caller's A or B breaks that (e.g. K = 17 elements of 2 bytes per row), the
// plan copies the operand once per run into its own workspace with rows padded
// to 16 bytes, and the tensor-core / FFMA kernels read the copy.  The copy is
// a plain coalesced row-by-row memcpy (HBM-bound).
//
// Skinny: when M or N is tiny a 128-row tensor-core tile would be mostly
// padding and the GEMM is bound by reading the large operand once ("DeepGEMM",
// sec. 4.3: a small-block variant for small M or N).  The small operand S
// (P <= 16 rows per pass) is read through L1; the large one, L, is streamed
// with 16-byte loads in one of two modes:
//   dot   L is [Q][K] with K contiguous (A when N is small; B in NK layout
//         when M is small): a warp walks one row q, lanes split K, and a
//         shuffle tree reduces the P partial dot products;
//   axpy  L is [K][Q] with Q contiguous (B in KN layout when M is small): each
//         thread owns 8 (16-bit) or 4 (FP32) consecutive columns q and walks K.
// K may be split over several CTAs: each writes FP32 partial sums to the plan
// workspace and counts its arrival on an atomic counter per output group; the
// CTA (or warp) that arrives last adds the partials in split order
// (deterministic), applies the epilogue and resets the counter -- no second
// launch and no waiting.  Unaligned operands take scalar loads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g13 {
namespace {

// Bytes [sh, sh + 16) of the 32-byte window lo:hi (sh even).  The shift is
// the same for every lane of a warp here, so the switch does not diverge.
__device__ __forceinline__ uint4 window16(const uint4& lo, const uint4& hi, int sh) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t sel = 0x3210u + static_cast<uint32_t>(sh & 3) * 0x1111u;
    switch (sh >> 2) {
        case 0:
            return make_uint4(__byte_perm(w[0], w[1], sel), __byte_perm(w[1], w[2], sel),
                              __byte_perm(w[2], w[3], sel), __byte_perm(w[3], w[4], sel));
        case 1:
            return make_uint4(__byte_perm(w[1], w[2], sel), __byte_perm(w[2], w[3], sel),
                              __byte_perm(w[3], w[4], sel), __byte_perm(w[4], w[5], sel));
        case 2:
            return make_uint4(__byte_perm(w[2], w[3], sel), __byte_perm(w[3], w[4], sel),
                              __byte_perm(w[4], w[5], sel), __byte_perm(w[5], w[6], sel));
        default:
            return make_uint4(__byte_perm(w[3], w[4], sel), __byte_perm(w[4], w[5], sel),
                              __byte_perm(w[5], w[6], sel), __byte_perm(w[6], w[7], sel));
    }
}

// Work unit = (row, 128 consecutive 16-byte pieces of the padded destination
// row); a warp's lane takes pieces lane, lane + 32, lane + 64, lane + 96 and
// issues all their loads before the stores, so a warp keeps up to 8 KB of
// reads in flight.  Piece j comes from the one or two aligned 16-byte source
// pieces that hold its bytes, shifted by the row's misalignment.  A source
// piece is read only when it holds a wanted byte, so nothing outside the
// operand's pages is touched.  Destination bytes past the row's end (padding
// up to dst_ld) get whatever the last source piece holds there; the GEMM's
// tensor maps end at the row's last column and never read them.
constexpr int STAGE_PIECES = 4;  // per lane per unit
struct StageArgs {
    const uint8_t* src;
    int64_t rows, row_bytes, ld_bytes, bstride_bytes, batch;
    uint8_t* dst;
    int64_t dst_ld_bytes;
    int64_t units;  // work units of this job
};
// Up to two jobs (both operands of a GEMM) in one launch: units of job 0, then of job 1.
__global__ void stage_copy_kernel(const StageArgs j0, const StageArgs j1, int njobs) {
    // the GEMM launched after this copy may start its set-up now; it waits for
    // this grid to finish before reading the copies
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t units = j0.units + (njobs > 1 ? j1.units : 0);
    for (int64_t uu = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         uu < units; uu += warps) {
        const bool second = uu >= j0.units;
        const StageArgs& J = second ? j1 : j0;
        const int64_t u = second ? uu - j0.units : uu;
        const int64_t npiece = (J.row_bytes + 15) / 16;
        const int64_t per_row = (npiece + 32 * STAGE_PIECES - 1) / (32 * STAGE_PIECES);
        const int64_t r = u / per_row;
        const int64_t j0p = (u - r * per_row) * (32 * STAGE_PIECES) + lane;
        const int64_t b = r / J.rows, i = r - b * J.rows;
        const uintptr_t a = reinterpret_cast<uintptr_t>(J.src + b * J.bstride_bytes + i * J.ld_bytes);
        const int sh = static_cast<int>(a & 15);
        const uint4* base = reinterpret_cast<const uint4*>(a - sh);
        uint4* d = reinterpret_cast<uint4*>(J.dst + r * J.dst_ld_bytes);
        uint4 lo[STAGE_PIECES], hi[STAGE_PIECES];
#pragma unroll
        for (int q = 0; q < STAGE_PIECES; ++q) {
            const int64_t j = j0p + 32 * q;
            const int64_t left = J.row_bytes - 16 * j;  // wanted bytes from piece j on
            lo[q] = j < npiece ? __ldg(base + j) : make_uint4(0, 0, 0, 0);
            hi[q] = j < npiece && sh + (left < 16 ? left : 16) > 16 ? __ldg(base + j + 1)
                                                                   : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < STAGE_PIECES; ++q) {
            const int64_t j = j0p + 32 * q;
            if (j < npiece) d[j] = window16(lo[q], hi[q], sh);
        }
    }
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
    return v;
}
template <>
__device__ __forceinline__ float to_f<__half>(__half v) {
    return __half2float(v);
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ float ldf(const T* p) {
    return to_f<T>(__ldg(p));
}

// VW elements at an unaligned (or short) position p, in two steps so that the
// loads of several positions are in flight before any is used: load_pair
// fetches the 16-byte-aligned chunk holding the first element and, only when
// the wanted bytes reach into it, the next one (both hold at least one wanted
// element, so nothing outside the operand's pages is touched); pair_shift then
// shifts by the misalignment with selects and funnel shifts (no branches) and
// zero-fills past n_valid.
struct RawPair {
    uint4 lo, hi;
};
template <typename T, int VW>
__device__ __forceinline__ RawPair load_pair(const T* p, int n_valid) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint4* base = reinterpret_cast<const uint4*>(a & ~static_cast<uintptr_t>(15));
    const int sh = static_cast<int>(a & 15);  // bytes, a multiple of sizeof(T)
    RawPair r;
    r.lo = n_valid > 0 ? __ldg(base) : make_uint4(0, 0, 0, 0);
    r.hi = n_valid > 0 && sh + n_valid * static_cast<int>(sizeof(T)) > 16 ? __ldg(base + 1)
                                                                          : make_uint4(0, 0, 0, 0);
    return r;
}
template <typename T, int VW>
__device__ __forceinline__ uint4 pair_shift(const RawPair& c, const T* p, int n_valid) {
    const int sh = static_cast<int>(reinterpret_cast<uintptr_t>(p) & 15);
    const int wo = sh >> 2;
    const uint32_t w[8] = {c.lo.x, c.lo.y, c.lo.z, c.lo.w, c.hi.x, c.hi.y, c.hi.z, c.hi.w};
    uint32_t sw[5];  // words wo .. wo + 4
#pragma unroll
    for (int j = 0; j < 5; ++j) {
        const uint32_t a0 = w[j], a1 = w[j + 1], a2 = w[j + 2], a3 = j + 3 < 8 ? w[j + 3] : 0u;
        sw[j] = wo == 0 ? a0 : wo == 1 ? a1 : wo == 2 ? a2 : a3;
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = (sh & 2) ? __funnelshift_r(sw[j], sw[j + 1], 16) : sw[j];
    uint4 r = make_uint4(o[0], o[1], o[2], o[3]);
    if (n_valid < VW) {  // elements past n_valid read as zero
        T* e = reinterpret_cast<T*>(&r);
#pragma unroll
        for (int i = 0; i < VW; ++i)
            if (i >= n_valid) e[i] = T(0.0f);
    }
    return r;
}
template <typename T, int VW>
__device__ __forceinline__ uint4 load_raw_unaligned(const T* p, int n_valid) {
    if (n_valid <= 0) return make_uint4(0, 0, 0, 0);
    return pair_shift<T, VW>(load_pair<T, VW>(p, n_valid), p, n_valid);
}

// 16 raw bytes (VW elements of T): one 16-byte load when `vec` (aligned, all in
// range); otherwise, with UA (the operand's rows are not 16-byte aligned), the
// two-chunk shifted load above, and without it (only a short tail can miss
// `vec`) up to n_valid element loads.  Zero-filled past n_valid.  Kept raw so
// that several loads can be in flight before any conversion.
template <typename T, int VW, bool UA>
__device__ __forceinline__ uint4 load_raw(const T* p, bool vec, int n_valid) {
    if (vec) return __ldg(reinterpret_cast<const uint4*>(p));
    if constexpr (UA) {
        if (n_valid <= 0) return make_uint4(0, 0, 0, 0);
        return load_raw_unaligned<T, VW>(p, n_valid);
    } else {
        uint4 r = make_uint4(0, 0, 0, 0);
        T* e = reinterpret_cast<T*>(&r);
#pragma unroll
        for (int i = 0; i < VW; ++i)
            if (i < n_valid) e[i] = __ldg(p + i);
        return r;
    }
}

template <typename T, int VW>
__device__ __forceinline__ void raw_to_f(const uint4& r, float (&out)[VW]) {
    const T* e = reinterpret_cast<const T*>(&r);
#pragma unroll
    for (int i = 0; i < VW; ++i) out[i] = to_f<T>(e[i]);
}

// VW consecutive elements (16 bytes) of T as floats; `vec` selects one 16-byte
// load (aligned, all in range) over scalar loads guarded by `n_valid`.
template <typename T, int VW>
__device__ __forceinline__ void load_vec(const T* p, bool vec, int n_valid, float (&out)[VW]) {
    if (vec) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
        const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int i = 0; i < VW; ++i) out[i] = to_f<T>(e[i]);
    } else {
#pragma unroll
        for (int i = 0; i < VW; ++i) out[i] = i < n_valid ? ldf(p + i) : 0.0f;
    }
}

struct SkinnyParams {
    const void* L;          // large operand
    int64_t ldl, stride_l;  // row stride ([Q][K] rows in dot mode, [K][Q] rows in axpy mode)
    const void* S;          // small operand: element (p, k) at S[p*s_sp + k*s_sk]
    int64_t s_sp, s_sk, stride_s;
    int64_t P, Q, K, batch;
    int p_is_m;             // 1: C[p][q];  0: C[q][p]
    int splits;
    int64_t kslice;         // K range per split (a multiple of 8)
    int l_vec, s_vec;       // 16-byte loads allowed for L / S rows
    float* partial;         // [batch][splits][P][Q] when splits > 1
    unsigned* arrive;       // split arrival counters (zero between launches)
    EpiParams e;
};

// Sum of the split partials of output (p, q) in split order.
__device__ __forceinline__ float split_sum(const SkinnyParams& sp, int64_t b, int64_t p,
                                           int64_t q) {
    const int64_t slab = sp.P * sp.Q;
    const float* src = sp.partial + b * sp.splits * slab + p * sp.Q + q;
    float y = 0.0f;
    int s = 0;
    for (; s + 4 <= sp.splits; s += 4) {  // four loads in flight, added in order
        const float x0 = __ldcg(src + s * slab), x1 = __ldcg(src + (s + 1) * slab);
        const float x2 = __ldcg(src + (s + 2) * slab), x3 = __ldcg(src + (s + 3) * slab);
        y += x0;
        y += x1;
        y += x2;
        y += x3;
    }
    for (; s < sp.splits; ++s) y += __ldcg(src + s * slab);
    return y;
}

__device__ __forceinline__ void skinny_final(const SkinnyParams& sp, int64_t b, int64_t p,
                                             int64_t q, float v) {
    if (sp.p_is_m)
        epi_store1(sp.e, b, p, q, v);
    else
        epi_store1(sp.e, b, q, p, v);
}

__device__ __forceinline__ void skinny_out(const SkinnyParams& sp, int64_t b, int split, int64_t p,
                                           int64_t q, float v) {
    if (sp.splits > 1) {
        sp.partial[((b * sp.splits + split) * sp.P + p) * sp.Q + q] = v;
    } else if (sp.p_is_m) {
        epi_store1(sp.e, b, p, q, v);
    } else {
        epi_store1(sp.e, b, q, p, v);
    }
}

// One warp per (batch, row q, split); lanes split the K range in 16-byte steps.
// PMAX small-operand rows per pass (1, 4 or 16); UA: the streamed rows are not
// 16-byte aligned (a separate instantiation, so the aligned one keeps its
// registers).
template <typename T, int PMAX, bool UA>
__global__ void __launch_bounds__(256, PMAX == 1 && !UA ? 3 : 2) skinny_dot_kernel(const SkinnyParams sp) {
    constexpr int VW = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t items = sp.batch * sp.Q * sp.splits;
    const T* Lbase = static_cast<const T*>(sp.L);
    const T* Sbase = static_cast<const T*>(sp.S);
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         it < items; it += warps) {
        const int split = static_cast<int>(it % sp.splits);
        const int64_t bq = it / sp.splits;
        const int64_t b = bq / sp.Q, q = bq - b * sp.Q;
        const int64_t k0 = split * sp.kslice;
        const int64_t k1 = min(sp.K, k0 + sp.kslice);
        const T* lrow = Lbase + b * sp.stride_l + q * sp.ldl;
        const T* sb = Sbase + b * sp.stride_s;
        // U 16-byte loads of the streamed row in flight per lane (fewer when P is large)
        constexpr int U = PMAX == 1 ? (UA ? 6 : 8) : PMAX == 4 ? 4 : 2;
        for (int64_t p0 = 0; p0 < sp.P; p0 += PMAX) {
            float acc[PMAX];
#pragma unroll
            for (int i = 0; i < PMAX; ++i) acc[i] = 0.0f;
            for (int64_t kb = k0 + lane * VW; kb < k1; kb += 32 * VW * U) {
                uint4 raw[U];
                if constexpr (UA) {
                    // every chunk load of the U positions first, then the shifts
                    RawPair pr[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int64_t k = kb + u * 32 * VW;
                        const int nv = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(VW), k1 - k)));
                        pr[u] = load_pair<T, VW>(lrow + k, nv);
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int64_t k = kb + u * 32 * VW;
                        const int nv = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(VW), k1 - k)));
                        raw[u] = pair_shift<T, VW>(pr[u], lrow + k, nv);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int64_t k = kb + u * 32 * VW;
                        const int nv = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(VW), k1 - k)));
                        raw[u] = load_raw<T, VW, UA>(lrow + k, sp.l_vec && nv == VW, nv);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t k = kb + u * 32 * VW;
                    const int nv = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(VW), k1 - k)));
                    if (nv == 0) break;
                    float lvu[VW];
                    raw_to_f<T, VW>(raw[u], lvu);
#pragma unroll
                    for (int i = 0; i < PMAX; ++i) {
                        if (p0 + i >= sp.P) break;
                        const T* srow = sb + (p0 + i) * sp.s_sp;
                        float sv[VW];
                        if (sp.s_sk == 1) {
                            load_vec<T, VW>(srow + k, sp.s_vec && nv == VW, nv, sv);
                        } else {
#pragma unroll
                            for (int j = 0; j < VW; ++j)
                                sv[j] = j < nv ? ldf(srow + (k + j) * sp.s_sk) : 0.0f;
                        }
#pragma unroll
                        for (int j = 0; j < VW; ++j) acc[i] = fmaf(lvu[j], sv[j], acc[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < PMAX; ++i) {
                if (p0 + i >= sp.P) break;
                float v = acc[i];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == i) skinny_out(sp, b, split, p0 + i, q, v);
            }
        }
        if (sp.splits > 1) {
            // The warp that finishes row (b, q) last adds all splits' partials.
            __threadfence();
            __syncwarp();
            unsigned last = 0;
            if (lane == 0) last = atomicAdd(sp.arrive + b * sp.Q + q, 1u) == static_cast<unsigned>(sp.splits - 1);
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                for (int64_t p = lane; p < sp.P; p += 32) skinny_final(sp, b, p, q, split_sum(sp, b, p, q));
                if (lane == 0) sp.arrive[b * sp.Q + q] = 0u;
            }
        }
    }
}

// Each CTA owns CW = 32 x VW consecutive columns q of L = [K][Q] (lane l the VW
// columns at q0 + l*VW, loaded as one 16-byte vector per row); its 8 warps take
// interleaved groups of G = VW rows of the split's K range, so every warp reads
// whole 512-byte row segments, and their sums are added in warp order through
// shared memory (deterministic).
template <typename T, int PMAX, bool UA>
__global__ void __launch_bounds__(256, PMAX == 1 ? (UA ? 2 : 3) : PMAX == 4 && !UA ? 2 : 1)
    skinny_axpy_kernel(const SkinnyParams sp) {
    constexpr int VW = 16 / sizeof(T);
    constexpr int CW = 32 * VW;
    constexpr int G = VW;
    __shared__ float red[8][CW];
    __shared__ unsigned s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t qb = static_cast<int64_t>(blockIdx.x) * CW;
    const int64_t q0 = qb + lane * VW;
    const int split = blockIdx.y;
    const int64_t b = blockIdx.z;
    const bool active = q0 < sp.Q;
    const int nv = active ? static_cast<int>(min(static_cast<int64_t>(VW), sp.Q - q0)) : 0;
    const bool vec = sp.l_vec && nv == VW;
    const int64_t k0 = split * sp.kslice;
    const int64_t k1 = min(sp.K, k0 + sp.kslice);
    const T* lcol = static_cast<const T*>(sp.L) + b * sp.stride_l + q0;
    const T* sb = static_cast<const T*>(sp.S) + b * sp.stride_s;
    const bool s_vec = sp.s_vec && sp.s_sk == 1;
    for (int64_t p0 = 0; p0 < sp.P; p0 += PMAX) {
        float acc[PMAX][VW];
#pragma unroll
        for (int i = 0; i < PMAX; ++i)
#pragma unroll
            for (int j = 0; j < VW; ++j) acc[i][j] = 0.0f;
        // A group's G streamed rows are in flight together before any
        // conversion; one 16-byte load of each small-operand row covers the
        // group when K is contiguous there.
        for (int64_t kb = k0 + warp * G; active && kb < k1; kb += 8 * G) {
            const int gn = static_cast<int>(min(static_cast<int64_t>(G), k1 - kb));
            uint4 raw[G];
            if constexpr (UA) {
                // Rows not 16-byte aligned: every row's chunk loads first (two per
                // row), then the shifts, so that the loads are in flight together.
                RawPair pr[G];
#pragma unroll
                for (int u = 0; u < G; ++u) {
                    if (u < gn)
                        pr[u] = load_pair<T, VW>(lcol + (kb + u) * sp.ldl, nv);
                    else
                        pr[u].lo = pr[u].hi = make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < G; ++u)
                    if (u < gn) raw[u] = pair_shift<T, VW>(pr[u], lcol + (kb + u) * sp.ldl, nv);
            } else {
#pragma unroll
                for (int u = 0; u < G; ++u)
                    if (u < gn) raw[u] = load_raw<T, VW, false>(lcol + (kb + u) * sp.ldl, vec, nv);
            }
#pragma unroll
            for (int i = 0; i < PMAX; ++i) {
                if (p0 + i >= sp.P) break;
                const T* srow = sb + (p0 + i) * sp.s_sp;
                float a[G];
                if (s_vec && gn == G && (kb & (G - 1)) == 0) {
                    raw_to_f<T, VW>(__ldg(reinterpret_cast<const uint4*>(srow + kb)), a);
                } else {
#pragma unroll
                    for (int u = 0; u < G; ++u) a[u] = u < gn ? ldf(srow + (kb + u) * sp.s_sk) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < G; ++u) {
                    if (u >= gn) break;
                    float lv[VW];
                    raw_to_f<T, VW>(raw[u], lv);
#pragma unroll
                    for (int j = 0; j < VW; ++j) acc[i][j] = fmaf(a[u], lv[j], acc[i][j]);
                }
            }
        }
        // add the 8 warps' sums column by column, in warp order
#pragma unroll
        for (int i = 0; i < PMAX; ++i) {
            if (p0 + i >= sp.P) break;
            __syncthreads();
#pragma unroll
            for (int j = 0; j < VW; ++j) red[warp][lane * VW + j] = acc[i][j];
            __syncthreads();
            for (int c = threadIdx.x; c < CW; c += 256) {
                if (qb + c >= sp.Q) break;
                float v = red[0][c];
#pragma unroll
                for (int w = 1; w < 8; ++w) v += red[w][c];
                skinny_out(sp, b, split, p0 + i, qb + c, v);
            }
        }
    }
    if (sp.splits > 1) {
        // The CTA that finishes this column block last adds all splits' partials.
        __threadfence();
        __syncthreads();
        unsigned* ctr = sp.arrive + b * gridDim.x + blockIdx.x;
        if (threadIdx.x == 0) s_last = atomicAdd(ctr, 1u) == static_cast<unsigned>(sp.splits - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            for (int64_t p = 0; p < sp.P; ++p)
                for (int c = threadIdx.x; c < CW; c += 256) {
                    if (qb + c >= sp.Q) break;
                    skinny_final(sp, b, p, qb + c, split_sum(sp, b, p, qb + c));
                }
            if (threadIdx.x == 0) *ctr = 0u;
        }
    }
}

// Split-K reduction for the tensor-core kernel: the partial slabs
// [batch][split][M][N] (FP32, N contiguous) are added in split order and the
// real epilogue is applied.  A thread owns four consecutive columns of one
// row: 16-byte loads from each slab when N allows, 32-bit index arithmetic
// when the quad count fits, and the vectorised four-column epilogue.
__global__ void __launch_bounds__(256) split_reduce_kernel(const float* __restrict__ partial,
                                                           int64_t M, int64_t N, int64_t batch,
                                                           int splits, int vec, EpiParams e) {
    griddep_wait();  // launched as a programmatic dependent of the GEMM writing the partials
    const int64_t nq = (N + 3) / 4;
    const int64_t total = batch * M * nq;
    const int64_t slab = M * N;
    const bool small = total < (int64_t(1) << 31);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t r, qd;
        if (small) {
            const uint32_t iu = static_cast<uint32_t>(i), nqu = static_cast<uint32_t>(nq);
            r = iu / nqu;
            qd = iu - static_cast<uint32_t>(r) * nqu;
        } else {
            r = i / nq;
            qd = i - r * nq;
        }
        const int64_t b = r / M, row = r - b * M, col = qd * 4;
        const float* src = partial + (b * splits) * slab + row * N + col;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        if (vec && col + 4 <= N) {
            int s = 0;
            for (; s + 2 <= splits; s += 2) {  // two slabs in flight, added in order
                const float4 p = __ldcg(reinterpret_cast<const float4*>(src + s * slab));
                const float4 q = __ldcg(reinterpret_cast<const float4*>(src + (s + 1) * slab));
                a0 += p.x;
                a1 += p.y;
                a2 += p.z;
                a3 += p.w;
                a0 += q.x;
                a1 += q.y;
                a2 += q.z;
                a3 += q.w;
            }
            if (s < splits) {
                const float4 p = __ldcg(reinterpret_cast<const float4*>(src + s * slab));
                a0 += p.x;
                a1 += p.y;
                a2 += p.z;
                a3 += p.w;
            }
        } else {
            for (int s = 0; s < splits; ++s) {
                const float* ps = src + s * slab;
                a0 += __ldcg(ps);
                if (col + 1 < N) a1 += __ldcg(ps + 1);
                if (col + 2 < N) a2 += __ldcg(ps + 2);
                if (col + 3 < N) a3 += __ldcg(ps + 3);
            }
        }
        epi_store4(e, b, row, col, a0, a1, a2, a3);
    }
}


}  // namespace

namespace {
template <typename T, int PM>
cudaError_t skinny_attr_t() {
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, skinny_dot_kernel<T, PM, false>);
    if (err == cudaSuccess) err = cudaFuncGetAttributes(&fa, skinny_dot_kernel<T, PM, true>);
    if (err == cudaSuccess) err = cudaFuncGetAttributes(&fa, skinny_axpy_kernel<T, PM, false>);
    if (err == cudaSuccess) err = cudaFuncGetAttributes(&fa, skinny_axpy_kernel<T, PM, true>);
    return err;
}
template <typename T>
cudaError_t skinny_attr_pm() {
    cudaError_t err = skinny_attr_t<T, 1>();
    if (err == cudaSuccess) err = skinny_attr_t<T, 4>();
    if (err == cudaSuccess) err = skinny_attr_t<T, 16>();
    return err;
}
// SMs of the launch's device: the plan's count, else the current device's.
int launch_sms(const LaunchCtx& lc) {
    if (lc.num_sms > 0) return lc.num_sms;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
        return sms;
    return 1;
}

}  // namespace

cudaError_t aux_preload_kernels() {
    // A function-attribute query makes the runtime load a lazily loaded kernel.
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, stage_copy_kernel);
    if (err == cudaSuccess) err = skinny_attr_pm<float>();
    if (err == cudaSuccess) err = skinny_attr_pm<__half>();
    if (err == cudaSuccess) err = skinny_attr_pm<__nv_bfloat16>();
    return err;
}

cudaError_t launch_stage_copies(const StageJob* jobs, int njobs, int esz, cudaStream_t stream) {
    StageArgs a[2] = {};
    int n = 0;
    for (int k = 0; k < njobs && k < 2; ++k) {
        const StageJob& J = jobs[k];
        const int64_t total = J.rows * J.batch;
        if (total <= 0 || J.cols <= 0) continue;
        if (reinterpret_cast<uintptr_t>(J.dst) % 16 != 0 || (J.dst_ld * esz) % 16 != 0)
            return cudaErrorInvalidValue;
        const int64_t npiece = (J.cols * esz + 15) / 16;
        a[n].src = static_cast<const uint8_t*>(J.src);
        a[n].rows = J.rows;
        a[n].row_bytes = J.cols * esz;
        a[n].ld_bytes = J.ld * esz;
        a[n].bstride_bytes = J.bstride * esz;
        a[n].batch = J.batch;
        a[n].dst = static_cast<uint8_t*>(J.dst);
        a[n].dst_ld_bytes = J.dst_ld * esz;
        a[n].units = total * ((npiece + 127) / 128);
        ++n;
    }
    if (n == 0) return cudaSuccess;
    // 8 warps per block, at most 8 blocks per SM's worth of work units
    const int64_t units = a[0].units + (n > 1 ? a[1].units : 0);
    const int64_t blocks = (units + 7) / 8;
    const unsigned grid = static_cast<unsigned>(blocks < 152 * 8 ? blocks : 152 * 8);
    stage_copy_kernel<<<grid, 256, 0, stream>>>(a[0], a[1], n);
    return cudaGetLastError();
}

cudaError_t launch_stage_copy(const void* src, int64_t rows, int64_t cols, int64_t ld,
                              int64_t bstride, int64_t batch, int esz, void* dst, int64_t dst_ld,
                              cudaStream_t stream) {
    const StageJob j{src, rows, cols, ld, bstride, batch, dst, dst_ld};
    return launch_stage_copies(&j, 1, esz, stream);
}

void skinny_geometry(int64_t M, int64_t N, int b_layout, int64_t* P, int64_t* Q, int* dot) {
    if (M <= N) {
        *P = M;
        *Q = N;
        *dot = b_layout == GEMM_B_NK;
    } else {
        *P = N;
        *Q = M;
        *dot = 1;
    }
}

cudaError_t launch_skinny(const gemm_config_t& cfg, const SkinnyArgs& a, const Shape& s,
                          const EpiParams& e, const LaunchCtx& lc) {
    if (s.M <= 0 || s.N <= 0) return cudaSuccess;
    SkinnyParams sp{};
    int dot = 0;
    skinny_geometry(s.M, s.N, a.b_layout, &sp.P, &sp.Q, &dot);
    const int esz = a.dtype == GEMM_F32 ? 4 : 2;
    if (s.M <= s.N) {
        // small operand A (rows p = m, K contiguous); large operand B
        sp.S = a.A;
        sp.s_sp = a.lda;
        sp.s_sk = 1;
        sp.stride_s = a.stride_a;
        sp.L = a.B;
        sp.ldl = a.ldb;
        sp.stride_l = a.stride_b;
        sp.p_is_m = 1;
    } else {
        // small operand B^ (rows p = n); large operand A (rows q = m, K contiguous)
        sp.S = a.B;
        const bool kn = a.b_layout == GEMM_B_KN;
        sp.s_sp = kn ? 1 : a.ldb;
        sp.s_sk = kn ? a.ldb : 1;
        sp.stride_s = a.stride_b;
        sp.L = a.A;
        sp.ldl = a.lda;
        sp.stride_l = a.stride_a;
        sp.p_is_m = 0;
    }
    sp.K = s.K;
    sp.batch = s.batch;
    sp.splits = cfg.split_k > 1 ? cfg.split_k : 1;
    sp.kslice = ((s.K + sp.splits - 1) / sp.splits + 7) / 8 * 8;
    if (sp.kslice == 0) sp.kslice = 8;
    sp.partial = sp.splits > 1 ? lc.sk_partials : nullptr;
    sp.arrive = sp.splits > 1 ? lc.sk_tags : nullptr;
    if (sp.splits > 1 && (!sp.partial || !sp.arrive)) return cudaErrorInvalidValue;
    const auto al16 = [](const void* p, int64_t ld, int64_t bs, int64_t batch, int es) {
        return reinterpret_cast<uintptr_t>(p) % 16 == 0 && (ld * es) % 16 == 0 &&
               (batch == 1 || (bs * es) % 16 == 0);
    };
    sp.l_vec = al16(sp.L, sp.ldl, sp.stride_l, s.batch, esz) ? 1 : 0;
    // (the stride between small-operand rows matters only when there are several)
    sp.s_vec = (sp.s_sk == 1 && al16(sp.S, sp.P > 1 ? sp.s_sp : 8, sp.stride_s, s.batch, esz)) ? 1 : 0;
    sp.e = e;
    const int sms = launch_sms(lc);
    const int pm = sp.P == 1 ? 1 : sp.P <= 4 ? 4 : 16;
    if (dot) {
        const int64_t items = s.batch * sp.Q * sp.splits;
        int64_t blocks = (items + 7) / 8;
        if (blocks > static_cast<int64_t>(sms) * 16) blocks = static_cast<int64_t>(sms) * 16;
        const unsigned grid = static_cast<unsigned>(blocks > 0 ? blocks : 1);
#define G13_DOT(T, PM)                                                      \
    do {                                                                    \
        if (sp.l_vec) skinny_dot_kernel<T, PM, false><<<grid, 256, 0, lc.stream>>>(sp); \
        else skinny_dot_kernel<T, PM, true><<<grid, 256, 0, lc.stream>>>(sp);           \
    } while (0)
#define G13_DOT_PM(T) \
    if (pm == 1) G13_DOT(T, 1); else if (pm == 4) G13_DOT(T, 4); else G13_DOT(T, 16)
        if (a.dtype == GEMM_F32) {
            G13_DOT_PM(float);
        } else if (a.dtype == GEMM_F16) {
            G13_DOT_PM(__half);
        } else {
            G13_DOT_PM(__nv_bfloat16);
        }
#undef G13_DOT_PM
#undef G13_DOT
    } else {
        const int vw = 16 / esz;
        const dim3 grid(static_cast<unsigned>((sp.Q + 32 * vw - 1) / (32 * vw)),
                        static_cast<unsigned>(sp.splits), static_cast<unsigned>(s.batch));
#define G13_AXPY(T, PM)                                                             \
    do {                                                                            \
        if (sp.l_vec) skinny_axpy_kernel<T, PM, false><<<grid, 256, 0, lc.stream>>>(sp); \
        else skinny_axpy_kernel<T, PM, true><<<grid, 256, 0, lc.stream>>>(sp);           \
    } while (0)
#define G13_AXPY_PM(T) \
    if (pm == 1) G13_AXPY(T, 1); else if (pm == 4) G13_AXPY(T, 4); else G13_AXPY(T, 16)
        if (a.dtype == GEMM_F32) {
            G13_AXPY_PM(float);
        } else if (a.dtype == GEMM_F16) {
            G13_AXPY_PM(__half);
        } else {
            G13_AXPY_PM(__nv_bfloat16);
        }
#undef G13_AXPY_PM
#undef G13_AXPY
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------ 3xTF32 split
// x = hi + lo with hi = x rounded to TF32 (10 explicit mantissa bits, nearest,
// ties away) and lo = x - hi, which is exact in FP32 (x and hi are within half
// a TF32 ulp).  The tensor core reads lo as TF32 too, so A.B ~ Ah.Bh + Ah.Bl +
// Al.Bh keeps about 21 bits of each operand.
__device__ __forceinline__ void tf32_split(float x, float& hi, float& lo) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
    float h = __uint_as_float(u);
    if (isinf(h) && !isinf(x)) h = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);  // no overflow
    hi = h;
    lo = isfinite(x) ? x - h : 0.0f;
}

// out[b][0 / 1][r][c] = hi / lo of X[b][r][c]; columns cols .. ldo-1 are zero.
__global__ void __launch_bounds__(256) tf32_split_rows_kernel(const float* __restrict__ X,
                                                              int64_t rows, int64_t cols,
                                                              int64_t ld, int64_t bstride,
                                                              int64_t batches, int vec,
                                                              float* __restrict__ out,
                                                              int64_t ldo) {
    griddep_launch();  // the tensor-core GEMM after this pass may start its set-up
    const int64_t q = ldo / 4;  // 4-column groups per output row
    const int64_t total = batches * rows * q;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t g = i % q, br = i / q;
        const int64_t r = br % rows, b = br / rows;
        const int64_t c0 = 4 * g;
        const float* src = X + b * bstride + r * ld + c0;
        float v[4];
        if (vec && c0 + 4 <= cols) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(src));
            v[0] = t.x;
            v[1] = t.y;
            v[2] = t.z;
            v[3] = t.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = c0 + j < cols ? __ldg(src + j) : 0.0f;
        }
        float h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) tf32_split(v[j], h[j], l[j]);
        float* dh = out + ((2 * b) * rows + r) * ldo + c0;
        float* dl = out + ((2 * b + 1) * rows + r) * ldo + c0;
        *reinterpret_cast<float4*>(dh) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(dl) = make_float4(l[0], l[1], l[2], l[3]);
    }
}

// out[b][0 / 1][c][r] = hi / lo of X[b][r][c] (transposed through a 32 x 32
// shared tile so both the loads and the stores are coalesced); columns
// rows .. ldo-1 of out are zero.
__global__ void __launch_bounds__(256) tf32_split_transpose_kernel(
    const float* __restrict__ X, int64_t rows, int64_t cols, int64_t ld, int64_t bstride,
    int64_t batches, float* __restrict__ out, int64_t ldo) {
    __shared__ float t[32][33];
    griddep_launch();  // the tensor-core GEMM after this pass may start its set-up
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32;
    for (int64_t b = blockIdx.z; b < batches; b += gridDim.z) {
        const float* src = X + b * bstride;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            const int64_t r = r0 + ty + j, c = c0 + tx;
            t[ty + j][tx] = (r < rows && c < cols) ? __ldg(src + r * ld + c) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            const int64_t c = c0 + ty + j, r = r0 + tx;  // output row c, column r
            if (c < cols && r < ldo) {
                float h, l;
                tf32_split(t[tx][ty + j], h, l);
                out[((2 * b) * cols + c) * ldo + r] = h;
                out[((2 * b + 1) * cols + c) * ldo + r] = l;
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_tf32_split(const float* X, int64_t rows, int64_t cols, int64_t ld,
                              int64_t bstride, int64_t batches, bool transpose, float* out,
                              int64_t ldo, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0 || batches <= 0) return cudaSuccess;
    if (ldo % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 16 != 0) return cudaErrorInvalidValue;
    if (!transpose) {
        const int vec = reinterpret_cast<uintptr_t>(X) % 16 == 0 && ld % 4 == 0 &&
                        (batches == 1 || bstride % 4 == 0);
        const int64_t total = batches * rows * (ldo / 4);
        int64_t blocks = (total + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        tf32_split_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            X, rows, cols, ld, bstride, batches, vec, out, ldo);
    } else {
        const int64_t gx = (cols + 31) / 32, gy = (ldo + 31) / 32;
        if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidValue;
        const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                        static_cast<unsigned>(batches < 65535 ? batches : 65535));
        tf32_split_transpose_kernel<<<grid, 256, 0, stream>>>(X, rows, cols, ld, bstride, batches,
                                                              out, ldo);
    }
    return cudaGetLastError();
}

// The same reduction when there are many splits and few outputs: a block
// takes 32 consecutive outputs and its 8 warps sum interleaved splits (warp w:
// splits w, w+8, ...), combined through shared memory in warp order, so the
// slab loads are spread over warps instead of one chain per output.
__global__ void __launch_bounds__(256) split_reduce_wide_kernel(const float* __restrict__ partial,
                                                                int64_t M, int64_t N,
                                                                int64_t batch, int splits,
                                                                EpiParams e) {
    __shared__ float part[8][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t slab = M * N, total = batch * slab;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * 32; base < total;
         base += static_cast<int64_t>(gridDim.x) * 32) {
        const int64_t i = base + lane;
        float v = 0.0f;
        int64_t b = 0, rc = 0;
        if (i < total) {
            b = i / slab;
            rc = i - b * slab;
            const float* src = partial + (b * splits) * slab + rc;
            for (int s = w; s < splits; s += 8) v += __ldcg(src + s * slab);
        }
        part[w][lane] = v;
        __syncthreads();
        if (w == 0 && i < total) {
            float y = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) y += part[k][lane];
            const int64_t row = rc / N, col = rc - row * N;
            epi_store1(e, b, row, col, y);
        }
        __syncthreads();
    }
}

cudaError_t launch_split_reduce(const float* partial, int64_t M, int64_t N, int64_t batch,
                                int splits, const EpiParams& e, const LaunchCtx& lc) {
    const int64_t quads = batch * M * ((N + 3) / 4);
    if (quads <= 0) return cudaSuccess;
    const int sms = launch_sms(lc);
    if (splits > 8 && quads < static_cast<int64_t>(sms) * 64) {
        const int64_t outs = batch * M * N;
        int64_t rb = (outs + 31) / 32;
        if (rb > static_cast<int64_t>(sms) * 8) rb = static_cast<int64_t>(sms) * 8;
        split_reduce_wide_kernel<<<static_cast<unsigned>(rb), 256, 0, lc.stream>>>(partial, M, N,
                                                                                batch, splits, e);
        return cudaGetLastError();
    }
    int64_t rb = (quads + 255) / 256;
    if (rb > static_cast<int64_t>(sms) * 16) rb = static_cast<int64_t>(sms) * 16;
    const int vec = (N % 4 == 0 && reinterpret_cast<uintptr_t>(partial) % 16 == 0) ? 1 : 0;
    // a programmatic dependent of the GEMM that writes the partials (it waits for
    // that grid before reading them), so its launch overlaps the GEMM's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rb));
    cfg.blockDim = dim3(256);
    cfg.stream = lc.stream;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_reduce_kernel, partial, M, N, batch, splits, vec, e);
}

}  // namespace g13
