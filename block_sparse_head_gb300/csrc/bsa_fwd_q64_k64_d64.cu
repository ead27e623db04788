// Forward kernel instances (plain and extended) for query block 64, key block 64, head dim 64.
#include "bsa_fwd_kernel.cuh"

namespace bsa {

cudaError_t launch_fwd_q64_k64_d64(bool ext, const FwdParams& p, const CUtensorMap& q,
    const CUtensorMap& k, const CUtensorMap& v, int grid, cudaStream_t stream) {
  return ext ? launch_fwd<64, 64, 64, true>(p, q, k, v, grid, stream)
             : launch_fwd<64, 64, 64, false>(p, q, k, v, grid, stream);
}

}  // namespace bsa
