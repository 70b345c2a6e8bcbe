// bf16 forward instantiations, head dim 128.
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_bf16_d128(int block_c, bool causal, bool out_f32, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                                 int grid, cudaStream_t s) {
    using C128 = fwd::Cfg<128, 128, false>;
    using C64 = fwd::Cfg<128, 64, false>;
    if (block_c == 64) {
        if (causal) return out_f32 ? fwd::launch<C64, true, true>(tq, tk, tv, p, grid, s)
                                   : fwd::launch<C64, true, false>(tq, tk, tv, p, grid, s);
        return out_f32 ? fwd::launch<C64, false, true>(tq, tk, tv, p, grid, s)
                       : fwd::launch<C64, false, false>(tq, tk, tv, p, grid, s);
    }
    if (causal) return out_f32 ? fwd::launch<C128, true, true>(tq, tk, tv, p, grid, s)
                               : fwd::launch<C128, true, false>(tq, tk, tv, p, grid, s);
    return out_f32 ? fwd::launch<C128, false, true>(tq, tk, tv, p, grid, s)
                   : fwd::launch<C128, false, false>(tq, tk, tv, p, grid, s);
}

}  // namespace fa
