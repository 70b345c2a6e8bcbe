// Forward kernel instances for block-sparse attention (bf16, 128 x 128 blocks).
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_sparse(int d, bool causal, const FwdMaps& m, const FwdParamsSparse& p, int grid,
                              cudaStream_t s) {
    if (d == 128) return fwd::launch_sparse<fwd::Cfg<128, 128, false>>(causal, m, p, grid, s);
    return fwd::launch_sparse<fwd::Cfg<64, 128, false>>(causal, m, p, grid, s);
}

}  // namespace fa
