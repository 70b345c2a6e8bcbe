// Backward kernel instances for shared key/value heads, for packed
// variable-length sequences, for the sliding window, for block-sparse
// attention and for rectangular attention (bf16 gradients).
#include "bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_gqa(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                const BwdParams& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                      : bwd::launch<C128, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
    return causal ? bwd::launch<C64, true, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
}

cudaError_t launch_bwd_main_varlen(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                   const BwdParams& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                      : bwd::launch<C128, false, false, true, true>(tq, tk, tv, tdo, tdq, p, grid, s);
    return causal ? bwd::launch<C64, true, false, true, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, true>(tq, tk, tv, tdo, tdq, p, grid, s);
}

cudaError_t launch_bwd_main_varlen_window(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                          const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsWin& p,
                                          int grid, cudaStream_t s) {
    if (d == 128) return bwd::launch<bwd::Cfg<128>, false, false, true, true, true>(tq, tk, tv, tdo, tdq, p, grid, s);
    return bwd::launch<bwd::Cfg<64>, false, false, true, true, true>(tq, tk, tv, tdo, tdq, p, grid, s);
}

cudaError_t launch_bwd_main_window(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsWin& p, int grid,
                                   cudaStream_t s) {
    if (d == 128) return bwd::launch<bwd::Cfg<128>, false, false, true, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
    return bwd::launch<bwd::Cfg<64>, false, false, true, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
}

cudaError_t launch_bwd_main_sparse(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                   const BwdParamsSparse& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                      : bwd::launch<C128, false, false, true, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
    return causal ? bwd::launch<C64, true, false, true, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
}

cudaError_t launch_bwd_main_rect(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsRect& p, int grid,
                                 cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                      : bwd::launch<C128, false, false, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
    return causal ? bwd::launch<C64, true, false, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s);
}

}  // namespace fa
