// Forward kernel instances for rectangular attention (Nq != Nk: decoding
// against a key/value cache, cross-attention), split-key form, bf16.
#include "fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_rect(int d, bool causal, const FwdMaps& m, const FwdParamsRect& p, int grid, cudaStream_t s) {
    if (d == 128) return fwd::launch_rect<fwd::Cfg<128, 128, false>>(causal, m, p, grid, s);
    return fwd::launch_rect<fwd::Cfg<64, 128, false>>(causal, m, p, grid, s);
}

}  // namespace fa
