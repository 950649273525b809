// skinny_tma.cu -- the memory-bound skinny GEMM (M or N <= 4) with the large
// operand streamed through shared memory by TMA.
//
// When M or N is tiny the product is bound by reading the large operand L once
// ("DeepGEMM", sec. 4.3: a small-block variant for small M or N).  The
// plain-load skinny kernel keeps only a few 16-byte loads per lane in flight,
// so its warps spend most cycles waiting on memory and it reaches a third to a
// half of HBM bandwidth.  Here one producer warp keeps a ring of 16 KB TMA
// boxes (512 bytes x 32 rows) in flight per SM and eight consumer warps only
// read shared memory:
//   dot   L is [Q][K] (K contiguous): a stage holds 32 rows x 512 bytes of K;
//         warp w takes rows 4w..4w+3, lane l the 16 bytes at 16 l of each row,
//         and a shuffle tree adds the lanes' partial dot products;
//   axpy  L is [K][Q] (Q contiguous): a stage holds 32 rows of K x 512 bytes
//         of Q; lane l owns the 16 bytes of columns at 16 l, warp w the rows
//         w, w + 8, w + 16, w + 24, and the warps' sums are added in warp
//         order through shared memory.
// The small operand S (P <= 4 rows of K, any strides) is converted to FP32
// once into shared memory as [P][K].
//
// Work is split stream-K style: a block (32 rows for dot, 512 bytes of
// columns for axpy) needs ceil(K / stage K) stages, the grid's CTAs take equal
// contiguous ranges of the blocks' stages in block order, and a block cut
// between CTAs is finished by the CTA that arrives last on its counter, which
// adds the contributors' partial sums in CTA order (deterministic) and applies
// the epilogue.  Each CTA leaves at most two partial blocks (its first and its
// last), in two slots of the plan workspace.
//
// Every wait is bounded: on a timeout the plan's status word records it, the
// consumers run through the rest of their stages without data (so the named
// barriers stay matched), and the producer lets its own copies land.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g13 {
namespace {

constexpr int SKT_MAX_STAGES = 6;                // ring depth (fewer when S needs the room)
constexpr int SKT_STAGE_BYTES = 16384;           // one 512-byte x 32-row box
constexpr int SKT_ROWS = 32;                     // rows of a box
constexpr int SKT_CONSUMERS = 256;               // 8 consumer warps
constexpr int SKT_THREADS = SKT_CONSUMERS + 32;  // + one producer warp
constexpr int SKT_SLOT_FLOATS = 256 * 4;         // one partial block: <= 256 outputs x 4 rows of S

struct SkinnyTmaParams {
    const void* S;
    int64_t s_sp, s_sk, stride_s;  // S element (p, k) of batch b at S[b*stride_s + p*s_sp + k*s_sk]
    int64_t P, Q, K, batch;
    int l_bmul;        // 1: L has a batch coordinate; 0: shared by every batch entry
    int s_batched;     // 1: S differs between batch entries
    int p_is_m;        // 1: C[p][q]; 0: C[q][p]
    int64_t nblk;      // blocks per batch entry
    int64_t sblk;      // stages per block
    int64_t total;     // batch * nblk * sblk stages
    float* slots;      // [2 * grid][SKT_SLOT_FLOATS] partial sums of cut blocks
    unsigned* arrive;  // one counter per (batch, block), zero between launches
    EpiParams e;
    unsigned* status;
    uint64_t timeout_ns;
    int stages;        // ring depth
};

template <typename T>
__device__ __forceinline__ float sk_to_f(T v);
template <>
__device__ __forceinline__ float sk_to_f<float>(float v) {
    return v;
}
template <>
__device__ __forceinline__ float sk_to_f<__half>(__half v) {
    return __half2float(v);
}
template <>
__device__ __forceinline__ float sk_to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

// The 16 bytes at p (shared memory) as VW floats.
template <typename T, int VW>
__device__ __forceinline__ void lds16_to_f(const uint8_t* p, float (&out)[VW]) {
    const uint4 raw = *reinterpret_cast<const uint4*>(p);
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < VW; ++i) out[i] = sk_to_f<T>(e[i]);
}

// Position of S element k in its shared-memory row (dot mode; the row length
// is a multiple of 256).  For 16-bit L a dot lane reads 8 consecutive K values
// per stage; they are kept as two float4 halves 128 floats apart (per
// 256-element block) so that each of the lane's two float4 loads covers 128
// contiguous bytes per quarter-warp (no bank conflicts).
template <int VW>
__device__ __forceinline__ int64_t s_index(int64_t k) {
    if (VW == 8) return (k & ~int64_t(255)) + ((k & 7) >> 2) * 128 + ((k & 255) >> 3) * 4 + (k & 3);
    return k;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(SKT_CONSUMERS) : "memory");
}

// Stream-K ranges: CTA c owns stages [first(c), first(c + 1)).
__device__ __forceinline__ int64_t range_first(int64_t total, int64_t grid, int64_t c) {
    return total * c / grid;
}
// The CTA whose range holds stage x.
__device__ __forceinline__ int64_t cta_of(int64_t total, int64_t grid, int64_t x) {
    int64_t c = x * grid / total;
    while (c + 1 < grid && range_first(total, grid, c + 1) <= x) ++c;
    while (c > 0 && range_first(total, grid, c) > x) --c;
    return c;
}
// Slot of CTA c's partial sums for the block with stages [bs, be) that c's
// range cuts: slot 1 when the block is c's last segment but not its first,
// else slot 0.
__device__ __forceinline__ int64_t slot_of(int64_t total, int64_t grid, int64_t c, int64_t bs,
                                           int64_t be) {
    const int64_t f = range_first(total, grid, c), l = range_first(total, grid, c + 1);
    const bool first_seg = f >= bs;  // c's first stage lies in this block
    const bool last_seg = l <= be;   // c's last stage lies in this block
    return 2 * c + ((last_seg && !first_seg) ? 1 : 0);
}

template <typename T, int PMAX, bool DOT>
__global__ void __launch_bounds__(SKT_THREADS, 1)
    skinny_tma_kernel(const __grid_constant__ CUtensorMap tmL, const SkinnyTmaParams sp) {
    constexpr int VW = 16 / sizeof(T);         // elements per 16 bytes
    constexpr int BOXE = 512 / sizeof(T);      // elements per 512-byte box row
    constexpr int KE = DOT ? BOXE : SKT_ROWS;  // K per stage
    constexpr int QE = DOT ? SKT_ROWS : BOXE;  // rows (dot) / columns (axpy) per block
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int nst = sp.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + nst * SKT_STAGE_BYTES);
    uint64_t* empty = full + SKT_MAX_STAGES;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + SKT_MAX_STAGES);
    unsigned* s_last = reinterpret_cast<unsigned*>(empty + SKT_MAX_STAGES) + 1;
    float* red = reinterpret_cast<float*>(smem + nst * SKT_STAGE_BYTES + 1024);
    // axpy: [8 warps][32 lanes][VW] partial sums ahead of S
    float* s_sm = DOT ? red : red + 8 * 32 * VW;
    const int64_t kpad = (sp.K + 255) / 256 * 256;  // S row length in shared memory, zero past K

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), SKT_CONSUMERS / 32);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tmL);
    }
    __syncthreads();

    const int64_t grid = gridDim.x, cta = blockIdx.x;
    const int64_t xb = range_first(sp.total, grid, cta), xe = range_first(sp.total, grid, cta + 1);
    if (warp == SKT_CONSUMERS / 32) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;
            for (int64_t x = xb; x < xe; ++x) {
                if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, sp.status,
                                       sp.timeout_ns))
                    break;
                const int64_t gb = x / sp.sblk;  // block over the batch
                const int64_t ks = x - gb * sp.sblk;
                const int64_t b = gb / sp.nblk, blk = gb - b * sp.nblk;
                const int32_t bc = static_cast<int32_t>(b * sp.l_bmul);
                const uint32_t bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(bar, SKT_STAGE_BYTES);
                if (DOT)
                    tma_load_3d(smem_u32(smem + s * SKT_STAGE_BYTES), &tmL, bar,
                                static_cast<int32_t>(ks * KE), static_cast<int32_t>(blk * QE), bc);
                else
                    tma_load_3d(smem_u32(smem + s * SKT_STAGE_BYTES), &tmL, bar,
                                static_cast<int32_t>(blk * QE), static_cast<int32_t>(ks * KE), bc);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (ph << s);
                if (++s == nst) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // After an abort, let our own copies land before the shared memory goes away.
            if (*abort_flag)
                for (int i = 0; i < nst; ++i)
                    if (armed & (1u << i)) {
                        const uint64_t t0 = globaltimer_ns();
                        while (!mbar_try_wait(smem_u32(&full[i]), (armed_par >> i) & 1u))
                            if (globaltimer_ns() - t0 > sp.timeout_ns) break;
                    }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const T* Sg = static_cast<const T*>(sp.S);
    int64_t staged_b = -1;
    bool ok = true;
    int s = 0;
    uint32_t ph = 0;
    int64_t x = xb;
    while (x < xe) {
        // one segment: the stages of block gb that this CTA owns
        const int64_t gb = x / sp.sblk;
        const int64_t bs = gb * sp.sblk, be = bs + sp.sblk;  // the block's stages
        const int64_t seg_end = min(xe, be);
        const int64_t b = gb / sp.nblk, blk = gb - b * sp.nblk;
        const int64_t sb = sp.s_batched ? b : 0;
        if (sb != staged_b) {
            // S for this batch entry as FP32 [P][kpad], zero past K: each thread
            // converts runs of 8 consecutive K values, all loads of a run in
            // flight together (one 16-byte load per run when S rows are
            // contiguous and aligned)
            consumer_sync();
            const T* src = Sg + sb * sp.stride_s;
            const int64_t runs = kpad / 8;
            constexpr int RB = 4;  // runs per thread with their loads in flight together
            for (int64_t r0 = tid; r0 < PMAX * runs; r0 += RB * SKT_CONSUMERS) {
                float v[RB][8];
#pragma unroll
                for (int u = 0; u < RB; ++u) {
                    const int64_t r8 = r0 + u * SKT_CONSUMERS;
                    const int64_t p = r8 / runs, k0 = (r8 - p * runs) * 8;
                    const bool live = r8 < PMAX * runs && p < sp.P;
                    const T* rp = src + (live ? p * sp.s_sp + k0 * sp.s_sk : 0);
                    if (live && sp.s_sk == 1 && k0 + 8 <= sp.K &&
                        reinterpret_cast<uintptr_t>(rp) % 16 == 0) {
#pragma unroll
                        for (int h = 0; h < 8; h += VW) {
                            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(rp + h));
                            const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
                            for (int j = 0; j < VW; ++j) v[u][h + j] = sk_to_f<T>(e[j]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            v[u][j] = (live && k0 + j < sp.K) ? sk_to_f<T>(rp[j * sp.s_sk]) : 0.0f;
                    }
                }
#pragma unroll
                for (int u = 0; u < RB; ++u) {
                    const int64_t r8 = r0 + u * SKT_CONSUMERS;
                    if (r8 >= PMAX * runs) break;
                    const int64_t p = r8 / runs, k0 = (r8 - p * runs) * 8;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        s_sm[p * kpad + (DOT ? s_index<VW>(k0 + j) : k0 + j)] = v[u][j];
                }
            }
            consumer_sync();
            staged_b = sb;
        }
        // accumulate the segment: dot acc[row i][p], axpy acc[p][column j]
        float acc[DOT ? 4 : PMAX][DOT ? PMAX : VW];
#pragma unroll
        for (int i = 0; i < (DOT ? 4 : PMAX); ++i)
#pragma unroll
            for (int j = 0; j < (DOT ? PMAX : VW); ++j) acc[i][j] = 0.0f;
        for (; x < seg_end; ++x) {
            const int64_t k = (x - bs) * KE;
            if (ok && !mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, sp.status, sp.timeout_ns))
                ok = false;
            if (ok) {
                const uint8_t* base = smem + s * SKT_STAGE_BYTES + lane * 16;
                if constexpr (DOT) {
                    // S for K values k + lane * VW .. + VW - 1
                    float sv[PMAX][VW];
#pragma unroll
                    for (int p = 0; p < PMAX; ++p) {
                        const float* srow = s_sm + p * kpad + k;
#pragma unroll
                        for (int j = 0; j < VW; j += 4) {
                            const float4 v =
                                *reinterpret_cast<const float4*>(srow + j / 4 * 128 + lane * 4);
                            sv[p][j] = v.x;
                            sv[p][j + 1] = v.y;
                            sv[p][j + 2] = v.z;
                            sv[p][j + 3] = v.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float lv[VW];
                        lds16_to_f<T, VW>(base + (warp * 4 + i) * 512, lv);
#pragma unroll
                        for (int p = 0; p < PMAX; ++p)
#pragma unroll
                            for (int j = 0; j < VW; ++j) acc[i][p] = fmaf(lv[j], sv[p][j], acc[i][p]);
                    }
                } else {
#pragma unroll
                    for (int jr = 0; jr < SKT_ROWS / 8; ++jr) {
                        const int row = warp + 8 * jr;
                        float lv[VW];
                        lds16_to_f<T, VW>(base + row * 512, lv);
#pragma unroll
                        for (int p = 0; p < PMAX; ++p) {
                            const float a = s_sm[p * kpad + k + row];  // warp-uniform
#pragma unroll
                            for (int c = 0; c < VW; ++c) acc[p][c] = fmaf(a, lv[c], acc[p][c]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (++s == nst) {
                s = 0;
                ph ^= 1u;
            }
        }
        // The segment's sums, one output (o, p) per thread: dot o = row
        // warp * 4 + (lane & 3), p = lane >> 2 (lanes < 4 * PMAX); axpy o = tid
        // (tid < 32 * VW), every p.
        float outv[PMAX];
        int o = -1;
        if constexpr (DOT) {
            float mine = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int p = 0; p < PMAX; ++p) {
                    float v = acc[i][p];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == p * 4 + i) mine = v;
                }
#pragma unroll
            for (int p = 0; p < PMAX; ++p) outv[p] = mine;  // only outv[lane >> 2] is used
            if (lane < 4 * PMAX) o = warp * 4 + (lane & 3);
        } else {
#pragma unroll
            for (int p = 0; p < PMAX; ++p) {
                consumer_sync();
#pragma unroll
                for (int c = 0; c < VW; ++c) red[(warp * 32 + lane) * VW + c] = acc[p][c];
                consumer_sync();
                float y = 0.0f;
                if (tid < 32 * VW) {
                    const int l = tid / VW, c = tid % VW;
#pragma unroll
                    for (int w = 0; w < 8; ++w) y += red[(w * 32 + l) * VW + c];
                }
                outv[p] = y;
            }
            if (tid < 32 * VW) o = tid;
        }
        const int p_lo = DOT ? (lane >> 2) : 0;
        const int p_hi = DOT ? p_lo + 1 : PMAX;
        const int64_t q = blk * QE + o;
        const bool has_out = o >= 0 && q < sp.Q;
        if (bs >= xb && be <= xe) {
            // the whole block is this CTA's: C directly
            if (ok && has_out)
#pragma unroll
                for (int p = 0; p < PMAX; ++p)
                    if (p >= p_lo && p < p_hi && p < sp.P)
                        epi_store1(sp.e, b, sp.p_is_m ? p : q, sp.p_is_m ? q : p, outv[p]);
            continue;
        }
        // A cut block: partial sums to this CTA's slot, then the last contributor
        // adds every contributor's slot in CTA order.
        float* slot = sp.slots + slot_of(sp.total, grid, cta, bs, be) * SKT_SLOT_FLOATS;
        if (has_out)
#pragma unroll
            for (int p = 0; p < PMAX; ++p)
                if (p >= p_lo && p < p_hi) slot[o * PMAX + p] = outv[p];
        __threadfence();
        consumer_sync();
        const int64_t c0 = cta_of(sp.total, grid, bs), c1 = cta_of(sp.total, grid, be - 1);
        if (tid == 0)
            *s_last = atomicAdd(sp.arrive + gb, 1u) == static_cast<unsigned>(c1 - c0);
        consumer_sync();
        if (*s_last) {
            __threadfence();
            for (int i = tid; i < QE * PMAX; i += SKT_CONSUMERS) {
                const int oo = i / PMAX, p = i - oo * PMAX;
                const int64_t qq = blk * QE + oo;
                if (qq >= sp.Q || p >= sp.P) continue;
                float y = 0.0f;
                for (int64_t c = c0; c <= c1; ++c)
                    y += __ldcg(sp.slots + slot_of(sp.total, grid, c, bs, be) * SKT_SLOT_FLOATS + i);
                if (ok) epi_store1(sp.e, b, sp.p_is_m ? p : qq, sp.p_is_m ? qq : p, y);
            }
            if (tid == 0) sp.arrive[gb] = 0u;
        }
    }
}

constexpr int kMaxDevices = 64;

template <typename T, int PMAX, bool DOT>
cudaError_t launch_t(const CUtensorMap& tm, const SkinnyTmaParams& sp, size_t smem, int grid,
                     cudaStream_t stream) {
    auto kern = skinny_tma_kernel<T, PMAX, DOT>;
    // the shared-memory limit is raised once per device and size, not per launch
    static std::atomic<int> raised[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (!cached || raised[dev].load() < static_cast<int>(smem)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        if (cached) {
            int cur = raised[dev].load();
            while (cur < static_cast<int>(smem) &&
                   !raised[dev].compare_exchange_weak(cur, static_cast<int>(smem))) {
            }
        }
    }
    kern<<<static_cast<unsigned>(grid), SKT_THREADS, smem, stream>>>(tm, sp);
    return cudaGetLastError();
}

template <typename T, bool DOT>
cudaError_t launch_p(int64_t P, const CUtensorMap& tm, const SkinnyTmaParams& sp, size_t smem,
                     int grid, cudaStream_t stream) {
    if (P == 1) return launch_t<T, 1, DOT>(tm, sp, smem, grid, stream);
    if (P == 2) return launch_t<T, 2, DOT>(tm, sp, smem, grid, stream);
    return launch_t<T, 4, DOT>(tm, sp, smem, grid, stream);
}

int pmax_of(int64_t P) { return P == 1 ? 1 : P == 2 ? 2 : 4; }

constexpr size_t kMaxSmem = 232448;  // dynamic shared memory per CTA

size_t smem_bytes(int64_t P, int64_t K, int dtype, int dot, int stages) {
    const int esz = dtype == GEMM_F32 ? 4 : 2;
    const int64_t kpad = (K + 255) / 256 * 256;
    const size_t red = dot ? 0 : static_cast<size_t>(8 * 32 * (16 / esz)) * sizeof(float);
    return 1024 + static_cast<size_t>(stages) * SKT_STAGE_BYTES + 1024 + red +
           static_cast<size_t>(pmax_of(P)) * static_cast<size_t>(kpad) * sizeof(float);
}

// Ring depth: 6 stages (96 KB in flight) when they fit beside the small
// operand, else as many as fit, at least 4.
int ring_stages(int64_t P, int64_t K, int dtype, int dot) {
    int st = SKT_MAX_STAGES;
    while (st > 4 && smem_bytes(P, K, dtype, dot, st) > kMaxSmem) --st;
    return st;
}

// The large operand of the skinny geometry: pointer, row stride, batch stride.
void large_operand(const SkinnyArgs& a, const Shape& s, const void** L, int64_t* ldl,
                   int64_t* stride_l) {
    if (s.M <= s.N) {
        *L = a.B;
        *ldl = a.ldb;
        *stride_l = a.stride_b;
    } else {
        *L = a.A;
        *ldl = a.lda;
        *stride_l = a.stride_a;
    }
}

}  // namespace

int64_t skinny_tma_stage_k(int dtype, int dot) {
    const int esz = dtype == GEMM_F32 ? 4 : 2;
    return dot ? 512 / esz : SKT_ROWS;
}

int64_t skinny_tma_block(int dtype, int dot) {
    const int esz = dtype == GEMM_F32 ? 4 : 2;
    return dot ? SKT_ROWS : 512 / esz;
}

bool skinny_tma_fits(int64_t P, int64_t K, int dtype, int dot) {
    return P >= 1 && P <= 4 && K >= 1 && smem_bytes(P, K, dtype, dot, 4) <= kMaxSmem;
}

size_t skinny_tma_workspace_bytes(int num_sms) {
    return static_cast<size_t>(2) * static_cast<size_t>(num_sms > 0 ? num_sms : 1) *
           SKT_SLOT_FLOATS * sizeof(float);
}

bool skinny_tma_aligned(const SkinnyArgs& a, const Shape& s) {
    const void* L;
    int64_t ldl, stride_l;
    large_operand(a, s, &L, &ldl, &stride_l);
    const int esz = a.dtype == GEMM_F32 ? 4 : 2;
    const bool batched = s.batch > 1 && stride_l != 0;
    return reinterpret_cast<uintptr_t>(L) % 16 == 0 && (ldl * esz) % 16 == 0 &&
           (!batched || (stride_l * esz) % 16 == 0);
}

int skinny_tma_encode(const SkinnyArgs& a, const Shape& s, CUtensorMap* tm) {
    int64_t P, Q;
    int dot = 0;
    skinny_geometry(s.M, s.N, a.b_layout, &P, &Q, &dot);
    const void* L;
    int64_t ldl, stride_l;
    large_operand(a, s, &L, &ldl, &stride_l);
    const int esz = a.dtype == GEMM_F32 ? 4 : 2;
    const int64_t l_batches = (s.batch > 1 && stride_l != 0) ? s.batch : 1;
    // L as a 3-D tensor -- dot (K, Q, batch), axpy (Q, K, batch) -- read in boxes
    // of 512 bytes x 32 rows.
    const int64_t cols = dot ? s.K : Q, rows = dot ? Q : s.K;
    return tmap_encode_3d(tm, a.dtype, L, cols, rows, ldl, l_batches, stride_l,
                          static_cast<uint32_t>(512 / esz), SKT_ROWS);
}

cudaError_t launch_skinny_tma(const SkinnyArgs& a, const Shape& s, const EpiParams& e,
                              const LaunchCtx& lc, int num_ctas, const CUtensorMap& tm) {
    if (s.M <= 0 || s.N <= 0) return cudaSuccess;
    int64_t P, Q;
    int dot = 0;
    skinny_geometry(s.M, s.N, a.b_layout, &P, &Q, &dot);
    if (!skinny_tma_fits(P, s.K, a.dtype, dot) || !skinny_tma_aligned(a, s))
        return cudaErrorInvalidValue;
    if (!lc.sk_partials || !lc.sk_tags || lc.num_sms <= 0) return cudaErrorInvalidValue;
    SkinnyTmaParams sp{};
    const void* L;
    int64_t ldl, stride_l;
    large_operand(a, s, &L, &ldl, &stride_l);
    if (s.M <= s.N) {
        sp.S = a.A;
        sp.s_sp = a.lda;
        sp.s_sk = 1;
        sp.stride_s = a.stride_a;
        sp.p_is_m = 1;
    } else {
        sp.S = a.B;
        const bool kn = a.b_layout == GEMM_B_KN;
        sp.s_sp = kn ? 1 : a.ldb;
        sp.s_sk = kn ? a.ldb : 1;
        sp.stride_s = a.stride_b;
        sp.p_is_m = 0;
    }
    const int64_t bt = s.batch;
    const int64_t l_batches = (bt > 1 && stride_l != 0) ? bt : 1;
    sp.P = P;
    sp.Q = Q;
    sp.K = s.K;
    sp.batch = bt;
    sp.l_bmul = l_batches > 1 ? 1 : 0;
    sp.s_batched = (bt > 1 && sp.stride_s != 0) ? 1 : 0;
    const int64_t ke = skinny_tma_stage_k(a.dtype, dot);
    const int64_t qe = skinny_tma_block(a.dtype, dot);
    sp.nblk = (Q + qe - 1) / qe;
    sp.sblk = (s.K + ke - 1) / ke;
    sp.total = bt * sp.nblk * sp.sblk;
    sp.slots = lc.sk_partials;
    sp.arrive = lc.sk_tags;
    sp.e = e;
    sp.status = lc.status;
    sp.timeout_ns = lc.timeout_ns;
    sp.stages = ring_stages(P, s.K, a.dtype, dot);

    // one CTA per SM (the workspace holds two slots per SM), or fewer when asked
    int64_t grid = lc.num_sms;
    if (num_ctas > 0 && num_ctas < grid) grid = num_ctas;
    if (grid > sp.total) grid = sp.total;
    const size_t smem = smem_bytes(P, s.K, a.dtype, dot, sp.stages);
    if (a.dtype == GEMM_F32)
        return dot ? launch_p<float, true>(P, tm, sp, smem, static_cast<int>(grid), lc.stream)
                   : launch_p<float, false>(P, tm, sp, smem, static_cast<int>(grid), lc.stream);
    if (a.dtype == GEMM_F16)
        return dot ? launch_p<__half, true>(P, tm, sp, smem, static_cast<int>(grid), lc.stream)
                   : launch_p<__half, false>(P, tm, sp, smem, static_cast<int>(grid), lc.stream);
    return dot ? launch_p<__nv_bfloat16, true>(P, tm, sp, smem, static_cast<int>(grid), lc.stream)
               : launch_p<__nv_bfloat16, false>(P, tm, sp, smem, static_cast<int>(grid), lc.stream);
}

}  // namespace g13
