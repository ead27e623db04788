// Backward kernel instances (dQ and dK/dV) for block 64, head dim 128.
#include "bsa_bwd_kernel.cuh"

namespace bsa {

cudaError_t launch_bwd_b64_d128(bool kv, const BwdParams& p, const CUtensorMap& a, const CUtensorMap& b,
    const CUtensorMap& x, const CUtensorMap& y, int grid, cudaStream_t stream) {
  return kv ? launch_bwd<64, 128, true>(p, a, b, x, y, grid, stream)
            : launch_bwd<64, 128, false>(p, a, b, x, y, grid, stream);
}

}  // namespace bsa
