// FP8 E4M3 forward instantiations (head dim 128, 128-key blocks, bf16 output).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_fp8_d128(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s) {
    using C = fwd::Cfg<128, 128, true>;
    return causal ? fwd::launch<C, true, false>(tq, tk, tv, p, grid, s)
                  : fwd::launch<C, false, false>(tq, tk, tv, p, grid, s);
}

}  // namespace fa
