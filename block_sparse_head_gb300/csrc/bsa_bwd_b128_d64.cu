// Backward kernel instances (dQ and dK/dV) for block 128, head dim 64.
#include "bsa_bwd_kernel.cuh"

namespace bsa {

cudaError_t launch_bwd_b128_d64(bool kv, const BwdParams& p, const CUtensorMap& a, const CUtensorMap& b,
    const CUtensorMap& x, const CUtensorMap& y, int grid, cudaStream_t stream) {
  return kv ? launch_bwd<128, 64, true>(p, a, b, x, y, grid, stream)
            : launch_bwd<128, 64, false>(p, a, b, x, y, grid, stream);
}

}  // namespace bsa
