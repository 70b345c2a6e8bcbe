// Backward main kernel instantiations (head dim 64 and 128, causal or not,
// bf16 or float32 gradient output).
#include "bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main(int d, bool causal, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdParams& p, int grid, cudaStream_t s) {
    using C128 = bwd::Cfg<128>;
    using C64 = bwd::Cfg<64>;
    if (d == 128) {
        if (causal) return out_f32 ? bwd::launch<C128, true, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                                   : bwd::launch<C128, true, false>(tq, tk, tv, tdo, tdq, p, grid, s);
        return out_f32 ? bwd::launch<C128, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                       : bwd::launch<C128, false, false>(tq, tk, tv, tdo, tdq, p, grid, s);
    }
    if (causal) return out_f32 ? bwd::launch<C64, true, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                               : bwd::launch<C64, true, false>(tq, tk, tv, tdo, tdq, p, grid, s);
    return out_f32 ? bwd::launch<C64, false, true>(tq, tk, tv, tdo, tdq, p, grid, s)
                   : bwd::launch<C64, false, false>(tq, tk, tv, tdo, tdq, p, grid, s);
}

}  // namespace fa
