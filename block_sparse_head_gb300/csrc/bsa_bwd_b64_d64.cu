// Backward kernel instances (dQ and dK/dV) for block 64, head dim 64.
#include "bsa_bwd_kernel.cuh"

namespace bsa {

cudaError_t launch_bwd_b64_d64(bool kv, const BwdParams& p, const CUtensorMap& a, const CUtensorMap& b,
    const CUtensorMap& x, const CUtensorMap& y, int grid, cudaStream_t stream) {
  return kv ? launch_bwd<64, 64, true>(p, a, b, x, y, grid, stream)
            : launch_bwd<64, 64, false>(p, a, b, x, y, grid, stream);
}

cudaError_t launch_bwd_delta(const void* out, const void* dout, float* delta, int64_t rows, int d,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int64_t threads = rows * (d / 8);
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  const auto* o = static_cast<const __nv_bfloat16*>(out);
  const auto* g = static_cast<const __nv_bfloat16*>(dout);
  if (d == 128)
    bsa_bwd_delta_kernel<128><<<grid, 256, 0, stream>>>(o, g, delta, static_cast<int>(rows));
  else
    bsa_bwd_delta_kernel<64><<<grid, 256, 0, stream>>>(o, g, delta, static_cast<int>(rows));
  return cudaGetLastError();
}

}  // namespace bsa
