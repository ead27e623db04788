// bsa_topk.cu -- bsa_topk_forward: top-k token-gather attention with an attention sink
// (kernel in bsa_topk_kernel.cuh; contract in include/bsa.h).
#include "../../include/bsa.h"

#include <cmath>

#include <cudaTypedefs.h>

#include "bsa_topk_kernel.cuh"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 topk_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

extern "C" int bsa_topk_forward(const void* q, const void* kv, const float* sink,
                                const int32_t* idx, void* out, float* lse, int32_t* status, int B,
                                int M, int N, int H, int D, int K, float scale, void* stream) {
  using C = bsa::TopkCfg;
  if (q == nullptr || kv == nullptr || sink == nullptr || idx == nullptr || out == nullptr ||
      lse == nullptr || status == nullptr)
    return BSA_ERR_NULL;
  if (H != C::kH || D != C::kD) return BSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return BSA_ERR_UNSUPPORTED;
  if (B < 1 || M < 1 || N < 1 || K < 1) return BSA_ERR_SHAPE;
  const int64_t npos = static_cast<int64_t>(B) * M;
  if (npos * H > 0x7fffffffLL || static_cast<int64_t>(B) * N > 0x7fffffffLL ||
      npos * K > 0x7fffffffLL)
    return BSA_ERR_SHAPE;
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!a16(q) || !a16(kv) || !a16(out) || !a16(lse) || !a16(sink) || !a16(idx) ||
      (reinterpret_cast<uintptr_t>(status) & 3u) != 0)
    return BSA_ERR_ALIGN;
  auto fn = topk_encode_fn();
  if (fn == nullptr) return BSA_ERR_CUDA;
  // Q as [64 columns, B*M*H rows, D/64 chunks]: one box is one position's 64 heads, all
  // chunks.  (The listed kv rows are gathered by the kernel's own copies.)
  CUtensorMap tq;
  {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(npos * H), static_cast<cuuint64_t>(D / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(H), static_cast<cuuint32_t>(D / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return BSA_ERR_CUDA;
  }
  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return BSA_ERR_CUDA;
  bsa::TopkParams p{};
  p.kv = kv;
  p.idx = idx;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.M = M;
  p.N = N;
  p.K = K;
  p.npos = static_cast<int>(npos);
  p.wait_limit_ns = 10000000000ull;
  p.expire_site = 0;
  p.status = status;
  static int attr_done[64] = {0};
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    if (cudaFuncSetAttribute(bsa::bsa_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return BSA_ERR_CUDA;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  const int grid = static_cast<int>(npos < sms ? npos : sms);
  bsa::bsa_topk_kernel<<<grid, C::kThreads, C::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(
      tq, p);
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}
