// bf16 forward instantiations, head dim 128 (plus the split-bf16 variant used
// for float32 inputs, which needs 64-key blocks to fit shared memory).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_bf16_d128(int block_c, bool causal, bool out_f32, bool split, const FwdMaps& m,
                                 const FwdParams& p, int grid, cudaStream_t s) {
    if (split) {
        if (block_c != 64 || !out_f32) return cudaErrorInvalidValue;
        using CS = fwd::Cfg<128, 64, false, true>;
        return causal ? fwd::launch<CS, true, true>(m, p, grid, s) : fwd::launch<CS, false, true>(m, p, grid, s);
    }
    if (block_c == 64) return fwd::launch_any<fwd::Cfg<128, 64, false>>(causal, out_f32, m, p, grid, s);
    return fwd::launch_any<fwd::Cfg<128, 128, false>>(causal, out_f32, m, p, grid, s);
}

}  // namespace fa
