// Forward kernel instance for block 64, head dim 128.
#include "bsa_fwd_kernel.cuh"

namespace bsa {

cudaError_t launch_fwd_b64_d128(const FwdParams& p, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, int grid, cudaStream_t stream) {
  return launch_fwd<64, 128>(p, q, k, v, grid, stream);
}

}  // namespace bsa
