// Forward kernel instances (extended) for query block 128, key block 64, head dim 64.
#include "bsa_fwd_kernel.cuh"

namespace bsa {

cudaError_t launch_fwd_q128_k64_d64(bool ext, const FwdParams& p, const CUtensorMap& q,
    const CUtensorMap& k, const CUtensorMap& v, int grid, cudaStream_t stream) {
  if (!ext) return cudaErrorInvalidValue;  // unequal blocks: extended kernel only
  return launch_fwd<128, 64, 64, true>(p, q, k, v, grid, stream);
}

}  // namespace bsa
