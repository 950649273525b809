// tc_sm103.cu -- dispatch of the tensor-core GEMM (tc_kernel.cuh) to its
// kernels: one that runs any epilogue, or, for the configurations the
// dispatcher picks and C stored by TMA, one compiled for the epilogue kind at
// hand; stream-K runs have kernels of their own.  The kernels are
// instantiated by tc_any_*.cu, tc_spec_*.cu and tc_sk_*.cu (compiled in
// parallel).
#include "tc_kernel.cuh"

namespace g13 {

bool tc_has_spec(const gemm_config_t& cfg) {
    if (cfg.bm != TBM || cfg.bk != TBK) return false;
#define G13_TC_HAS(BN, ST, EW, VAR, PAIR) \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR) return true;
    G13_TC_SPEC_CONFIGS(G13_TC_HAS)
#undef G13_TC_HAS
    return false;
}

namespace {

bool tc_has_softmax(const gemm_config_t& cfg) {
#define G13_TC_HAS(BN, ST, EW, VAR, PAIR) \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR) return true;
    G13_TC_SOFTMAX_CONFIGS(G13_TC_HAS)
#undef G13_TC_HAS
    return false;
}

// The epilogue kind of a run: em (TMA store maps) is null when C's rows cannot
// be stored by TMA.
int tc_pick_ek(const EpiParams& e, const TcEpiMaps* em) {
    if (e.act == GEMM_ACT_SOFTMAX) return em ? TC_EK_SOFTMAX : TC_EK_ANY;
    if (!em) return TC_EK_ROWS;
    if (!e.bias && e.act == GEMM_ACT_NONE && !e.R) return TC_EK_PLAIN;
    if (e.act == GEMM_ACT_GELU_ERF) return e.R ? TC_EK_ANY : TC_EK_GELU;
    return TC_EK_BIAS;
}

}  // namespace

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
    const bool kn = b_layout == GEMM_B_KN;
    if (cfg.stream_k) {
        if (!tc_has_spec(cfg)) return cudaErrorInvalidValue;
        return kn ? launch_tc_sk_kn(cfg, dtype, tmA, tmB, em, s, e, lc, final_epi)
                  : launch_tc_sk_nk(cfg, dtype, tmA, tmB, em, s, e, lc, final_epi);
    }
    const int ek = tc_pick_ek(e, em);
    if (ek == TC_EK_SOFTMAX && tc_has_softmax(cfg))
        return kn ? launch_tc_spec_kn(ek, cfg, dtype, tmA, tmB, em, s, e, lc, final_epi)
                  : launch_tc_spec_nk(ek, cfg, dtype, tmA, tmB, em, s, e, lc, final_epi);
    if (ek != TC_EK_ANY && ek != TC_EK_SOFTMAX && tc_has_spec(cfg))
        return kn ? launch_tc_spec_kn(ek, cfg, dtype, tmA, tmB, em, s, e, lc, final_epi)
                  : launch_tc_spec_nk(ek, cfg, dtype, tmA, tmB, em, s, e, lc, final_epi);
    return kn ? launch_tc_any_kn(cfg, dtype, tmA, tmB, em, s, e, lc, final_epi)
              : launch_tc_any_nk(cfg, dtype, tmA, tmB, em, s, e, lc, final_epi);
}

cudaError_t tc_preload_kernels() {
    cudaError_t err = tc_preload_any_kn();
    if (err == cudaSuccess) err = tc_preload_any_nk();
    if (err == cudaSuccess) err = tc_preload_spec_kn();
    if (err == cudaSuccess) err = tc_preload_spec_nk();
    if (err == cudaSuccess) err = tc_preload_sk_kn();
    if (err == cudaSuccess) err = tc_preload_sk_nk();
    return err;
}

}  // namespace g13
