// bf16 forward instantiations, head dim 64 (plus the split-bf16 variants used
// for float32 inputs).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_bf16_d64(int block_c, bool causal, bool out_f32, bool split, const FwdMaps& m,
                                const FwdParams& p, int grid, cudaStream_t s) {
    if (split) {
        if (!out_f32) return cudaErrorInvalidValue;
        if (block_c == 64) {
            using CS = fwd::Cfg<64, 64, false, true>;
            return causal ? fwd::launch<CS, true, true>(m, p, grid, s) : fwd::launch<CS, false, true>(m, p, grid, s);
        }
        using CS = fwd::Cfg<64, 128, false, true>;
        return causal ? fwd::launch<CS, true, true>(m, p, grid, s) : fwd::launch<CS, false, true>(m, p, grid, s);
    }
    if (block_c == 64) return fwd::launch_any<fwd::Cfg<64, 64, false>>(causal, out_f32, m, p, grid, s);
    return fwd::launch_any<fwd::Cfg<64, 128, false>>(causal, out_f32, m, p, grid, s);
}

}  // namespace fa
