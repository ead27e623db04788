// Forward kernel instance for block 128, head dim 64.
#include "bsa_fwd_kernel.cuh"

namespace bsa {

cudaError_t launch_fwd_b128_d64(const FwdParams& p, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, int grid, cudaStream_t stream) {
  return launch_fwd<128, 64>(p, q, k, v, grid, stream);
}

}  // namespace bsa
