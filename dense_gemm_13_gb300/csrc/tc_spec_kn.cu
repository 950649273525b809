// tc_spec_kn.cu -- the tensor-core kernels specialised to one epilogue kind, row-major ([K, N]) B.
#include "tc_kernel.cuh"

namespace g13 {

cudaError_t launch_tc_spec_kn(int ek, const gemm_config_t& cfg, int dtype, const CUtensorMap& tmA,
                              const CUtensorMap& tmB, const TcEpiMaps* em, const Shape& s,
                              const EpiParams& e, const LaunchCtx& lc, const EpiParams* fe) {
#define G13_TC_LAUNCH(BN, ST, EW, VAR, PAIR)                                                    \
    if (cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR) {                              \
        if (ek == TC_EK_PLAIN)                                                                  \
            return launch_tc_t<BN, ST, true, EW, PAIR, false, TC_EK_PLAIN, false>(cfg, dtype, tmA, tmB, em, \
                                                                           s, e, lc, fe);       \
        if (ek == TC_EK_BIAS)                                                                   \
            return launch_tc_t<BN, ST, true, EW, PAIR, false, TC_EK_BIAS, false>(cfg, dtype, tmA, tmB, em,  \
                                                                          s, e, lc, fe);        \
        if (ek == TC_EK_GELU)                                                                   \
            return launch_tc_t<BN, ST, true, EW, PAIR, false, TC_EK_GELU, false>(cfg, dtype, tmA, tmB, em,  \
                                                                          s, e, lc, fe);        \
        if (ek == TC_EK_ROWS)                                                                   \
            return launch_tc_t<BN, ST, true, EW, PAIR, false, TC_EK_ROWS, false>(cfg, dtype, tmA, tmB, em,  \
                                                                          s, e, lc, fe);        \
    }
    G13_TC_SPEC_CONFIGS(G13_TC_LAUNCH)
#undef G13_TC_LAUNCH
#define G13_TC_LAUNCH_SMX(BN, ST, EW, VAR, PAIR)                                                \
    if (ek == TC_EK_SOFTMAX && cfg.bn == BN && cfg.stages == ST && cfg.variant == VAR)         \
        return launch_tc_t<BN, ST, true, EW, PAIR, false, TC_EK_SOFTMAX, false>(cfg, dtype, tmA, tmB,  \
                                                                            em, s, e, lc, fe);
    G13_TC_SOFTMAX_CONFIGS(G13_TC_LAUNCH_SMX)
#undef G13_TC_LAUNCH_SMX
    return cudaErrorInvalidValue;
}

cudaError_t tc_preload_spec_kn() {
    cudaFuncAttributes fa;
    cudaError_t err = cudaSuccess;
#define G13_TC_PRELOAD(BN, ST, EW, VAR, PAIR)                                                      \
    if (err == cudaSuccess)                                                                        \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, true, EW, PAIR, false, TC_EK_PLAIN, false>); \
    if (err == cudaSuccess)                                                                        \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, true, EW, PAIR, false, TC_EK_BIAS, false>);  \
    if (err == cudaSuccess)                                                                        \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, true, EW, PAIR, false, TC_EK_GELU, false>); \
    if (err == cudaSuccess)                                                                        \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, true, EW, PAIR, false, TC_EK_ROWS, false>);
    G13_TC_SPEC_CONFIGS(G13_TC_PRELOAD)
#undef G13_TC_PRELOAD
#define G13_TC_PRELOAD_SMX(BN, ST, EW, VAR, PAIR)                                                   \
    if (err == cudaSuccess)                                                                         \
        err = cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, ST, true, EW, PAIR, false, TC_EK_SOFTMAX, false>);
    G13_TC_SOFTMAX_CONFIGS(G13_TC_PRELOAD_SMX)
#undef G13_TC_PRELOAD_SMX
    return err;
}

}  // namespace g13
