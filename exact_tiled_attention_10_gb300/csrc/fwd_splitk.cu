// Split-key instances of the forward kernel (128-key blocks, bf16 output):
// bf16 with d = 128 and d = 64, and FP8 with d = 128.
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_splitk(int d, bool fp8, bool causal, const FwdMaps& m, const FwdParams& p, int grid,
                              cudaStream_t s) {
    if (fp8) return fwd::launch_splitk<fwd::Cfg<128, 128, true>>(causal, m, p, grid, s);
    if (d == 128) return fwd::launch_splitk<fwd::Cfg<128, 128, false>>(causal, m, p, grid, s);
    return fwd::launch_splitk<fwd::Cfg<64, 128, false>>(causal, m, p, grid, s);
}

}  // namespace fa
