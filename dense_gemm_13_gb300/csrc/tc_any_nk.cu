// tc_any_nk.cu -- the tensor-core kernels that run any epilogue, K-major ([N, K]), and the 3xTF32 kernels B.
#include "tc_kernel.cuh"

namespace g13 {

cudaError_t launch_tc_any_nk(const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                             const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe) {
#define G13_TC_LAUNCH(BN, ST, EW, VAR, PAIR)                                                  \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR)                               \
        return launch_tc_t<BN, ST, false, EW, PAIR, false, TC_EK_ANY, false>(cfg, dtype, tmA, tmB, em, s, e, \
                                                                     lc, fe);
    G13_TC_CONFIGS(G13_TC_LAUNCH)
#undef G13_TC_LAUNCH
    return cudaErrorInvalidValue;
}

cudaError_t tc_preload_any_nk() {
    // A function-attribute query makes the runtime load a lazily loaded kernel.
    cudaFuncAttributes fa;
    cudaError_t err = cudaSuccess;
#define G13_TC_PRELOAD(BN, ST, EW, VAR, PAIR)                                                  \
    if (err == cudaSuccess)                                                                    \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, false, EW, PAIR, false, TC_EK_ANY, false>);
    G13_TC_CONFIGS(G13_TC_PRELOAD)
#undef G13_TC_PRELOAD
#define G13_TC3_PRELOAD(BN, ST, EW, VAR, PAIR)                                                 \
    if (err == cudaSuccess)                                                                    \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, false, EW, PAIR, true, TC_EK_ANY, false>);
    G13_TC3_CONFIGS(G13_TC3_PRELOAD)
#undef G13_TC3_PRELOAD
    return err;
}

cudaError_t launch_tc3(const gemm_config_t& cfg, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const TcEpiMaps* em, const Shape& s, const EpiParams& e,
                       const LaunchCtx& lc) {
#define G13_TC3_LAUNCH(BN, ST, EW, VAR, PAIR)                                                 \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR)                               \
        return launch_tc_t<BN, ST, false, EW, PAIR, true, TC_EK_ANY, false>(cfg, GEMM_F32, tmA, tmB, em, s, \
                                                                     e, lc, nullptr);
    G13_TC3_CONFIGS(G13_TC3_LAUNCH)
#undef G13_TC3_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace g13
