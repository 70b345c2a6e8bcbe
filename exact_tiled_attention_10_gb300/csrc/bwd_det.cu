// Deterministic backward kernel instances (bf16 gradients; plain, shared
// key/value heads, sliding window, block lists, rectangular, packed
// sequences): dQ tiles
// take their key blocks' contributions in a fixed order, so repeated runs give
// bitwise-identical dQ, dK and dV.
#include "bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_det(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                const BwdParamsDet& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, false, false, false, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                               grid, s)
                      : bwd::launch<C128, false, false, true, false, false, false, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                                grid, s);
    return causal ? bwd::launch<C64, true, false, true, false, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, false, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid,
                                                                                           s);
}

cudaError_t launch_bwd_main_det_window(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdDet<BwdParamsWin>& p,
                                       int grid, cudaStream_t s) {
    if (d == 128)
        return bwd::launch<bwd::Cfg<128>, false, false, true, false, true, false, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                               grid, s);
    return bwd::launch<bwd::Cfg<64>, false, false, true, false, true, false, false, true>(tq, tk, tv, tdo, tdq, p, grid,
                                                                                          s);
}

cudaError_t launch_bwd_main_det_rect(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                     const BwdDet<BwdParamsRect>& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, false, false, false, true, true>(tq, tk, tv, tdo, tdq, p,
                                                                                              grid, s)
                      : bwd::launch<C128, false, false, true, false, false, false, true, true>(tq, tk, tv, tdo, tdq, p,
                                                                                               grid, s);
    return causal ? bwd::launch<C64, true, false, true, false, false, false, true, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, false, false, false, true, true>(tq, tk, tv, tdo, tdq, p, grid,
                                                                                          s);
}

cudaError_t launch_bwd_main_det_sparse(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                       const BwdDet<BwdParamsSparse>& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, false, false, true, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                              grid, s)
                      : bwd::launch<C128, false, false, true, false, false, true, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                               grid, s);
    return causal ? bwd::launch<C64, true, false, true, false, false, true, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, false, false, true, false, true>(tq, tk, tv, tdo, tdq, p, grid,
                                                                                          s);
}

cudaError_t launch_bwd_main_det_varlen_window(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                                              const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                              const BwdDet<BwdParamsWin>& p, int grid, cudaStream_t s) {
    if (d == 128)
        return bwd::launch<bwd::Cfg<128>, false, false, true, true, true, false, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                              grid, s);
    return bwd::launch<bwd::Cfg<64>, false, false, true, true, true, false, false, true>(tq, tk, tv, tdo, tdq, p, grid,
                                                                                         s);
}

cudaError_t launch_bwd_main_det_varlen(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                       const BwdParamsDet& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128)
        return causal ? bwd::launch<C128, true, false, true, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                              grid, s)
                      : bwd::launch<C128, false, false, true, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p,
                                                                                               grid, s);
    return causal ? bwd::launch<C64, true, false, true, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                  : bwd::launch<C64, false, false, true, true, false, false, false, true>(tq, tk, tv, tdo, tdq, p, grid,
                                                                                          s);
}

}  // namespace fa
