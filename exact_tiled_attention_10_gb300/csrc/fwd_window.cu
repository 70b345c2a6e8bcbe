// Forward kernel instances for the sliding-window mask (bf16, 128-key blocks).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_window(int d, const FwdMaps& m, const FwdParamsWin& p, int grid, cudaStream_t s) {
    if (d == 128) return fwd::launch_window<fwd::Cfg<128, 128, false>>(m, p, grid, s);
    return fwd::launch_window<fwd::Cfg<64, 128, false>>(m, p, grid, s);
}

}  // namespace fa
