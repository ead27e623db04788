// Forward kernel instance for block 64, head dim 64.
#include "bsa_fwd_kernel.cuh"

namespace bsa {

cudaError_t launch_fwd_b64_d64(const FwdParams& p, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, int grid, cudaStream_t stream) {
  return launch_fwd<64, 64>(p, q, k, v, grid, stream);
}

}  // namespace bsa
