// Forward kernel instances (extended) for query block 64, key block 128, head dim 128.
#include "bsa_fwd_kernel.cuh"

namespace bsa {

cudaError_t launch_fwd_q64_k128_d128(bool ext, const FwdParams& p, const CUtensorMap& q,
    const CUtensorMap& k, const CUtensorMap& v, int grid, cudaStream_t stream) {
  if (!ext) return cudaErrorInvalidValue;  // unequal blocks: extended kernel only
  return launch_fwd<64, 128, 128, true>(p, q, k, v, grid, stream);
}

}  // namespace bsa
