// Forward kernel instances for packed variable-length sequences (bf16, 128-key blocks).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_varlen(int d, bool causal, const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
    if (d == 128) return fwd::launch_varlen<fwd::Cfg<128, 128, false>>(causal, m, p, grid, s);
    return fwd::launch_varlen<fwd::Cfg<64, 128, false>>(causal, m, p, grid, s);
}

cudaError_t launch_fwd_varlen_window(int d, const FwdMaps& m, const FwdParamsWin& p, int grid, cudaStream_t s) {
    if (d == 128) return fwd::launch_varlen_window<fwd::Cfg<128, 128, false>>(m, p, grid, s);
    return fwd::launch_varlen_window<fwd::Cfg<64, 128, false>>(m, p, grid, s);
}

}  // namespace fa
