// FP8 E4M3 forward instantiations (head dim 128, 128-key blocks, bf16 output).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_fp8_d128(bool causal, const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
    using C = fwd::Cfg<128, 128, true>;
    return causal ? fwd::launch<C, true, false>(m, p, grid, s) : fwd::launch<C, false, false>(m, p, grid, s);
}

}  // namespace fa
