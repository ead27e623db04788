// bsa_noalloc.cu -- bsa_forward_noalloc: the forward for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a host
// callback or a driver/plugin hook where allocation would deadlock or is forbidden,
// under a memory manager that owns the whole device heap, or in a process that must
// not grow its footprint after start-up.  Such callers can still build a LUT on the
// host (bsa_build_lut allocates only host memory) and hand over their own q/k/v/out/
// lse buffers; the device copies of the LUT that bsa_lut_upload would allocate live
// here instead, in one fixed array that is part of the library image.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes (4 MiB).  Every
// GPU that loads the library holds those 4 MiB until the process exits.  All calls
// share it, and each call overwrites it (status word cleared, LUT copied in) before
// its kernel runs: two calls whose kernels overlap on the GPU (different streams, or
// host threads racing) corrupt each other's LUT.  Serialize them on one stream.
#include "../../include/bsa.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include <cudaTypedefs.h>

#include "bsa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;
constexpr size_t kNoAllocScratchWords = kNoAllocScratchBytes / 4;
// Room reserved for the per-CTA starts: grids up to this many CTAs.
constexpr int kMaxGrid = 1023;

// Layout, in int32 words, each part starting on a 16-byte boundary:
//   [0, 4)           status word (+ padding)
//   [4, 4 + 4n)      work list regrouped per CTA, n device records of 4 words
//   then the per-CTA starts (grid + 1 words) and col_idx (nnz words)
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchWords];

size_t round4(size_t words) { return (words + 3) & ~static_cast<size_t>(3); }

bool encode_rows_noalloc(CUtensorMap* map, const void* base, int64_t rows, int d, int box_rows,
                         int box_halves) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  // Same three-dimensional view as bsa_forward's maps: 64 columns, rows, d/64 halves.
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(d / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_halves)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int bsa_forward_noalloc(const void* q, const void* k, const void* v, const bsa_lut* lut,
                                   void* out, float* lse, int B, int H, int L, int d, float scale,
                                   int block, int causal_diag, void* stream, int sync_status) {
  if (q == nullptr || k == nullptr || v == nullptr || lut == nullptr || out == nullptr ||
      lse == nullptr)
    return BSA_ERR_NULL;
  if ((block != 64 && block != 128) || (d != 64 && d != 128)) return BSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return BSA_ERR_UNSUPPORTED;
  if (B != lut->batch || H != lut->H || L <= 0 || lut->nbk != lut->nb ||
      static_cast<int64_t>(lut->nb) * block != L)
    return BSA_ERR_SHAPE;
  const int64_t rows = static_cast<int64_t>(B) * H * L;
  if (rows > 0x7fffffffLL - 128) return BSA_ERR_SHAPE;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out) || !a16(lse)) return BSA_ERR_ALIGN;

  const size_t off_items = 4;
  const size_t off_start = off_items + round4(static_cast<size_t>(lut->n_items) * 4);
  const size_t off_colidx = off_start + round4(static_cast<size_t>(kMaxGrid) + 1);
  const size_t total = off_colidx + round4(lut->col_idx.size());
  if (total > kNoAllocScratchWords) return BSA_ERR_TOO_LARGE;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BSA_ERR_CUDA;
  // Looked up on every call (it allocates nothing): a cached address would go stale if
  // the device's context were reset and the module loaded again.
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr)
    return BSA_ERR_CUDA;
  int32_t* base = static_cast<int32_t*>(scratch);
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return BSA_ERR_CUDA;
  const int grid = std::max(1, std::min({lut->n_items, sms, kMaxGrid}));
  // The schedule made at upload serves when it was made for this grid; otherwise it is
  // built here (host memory only).
  const int o = bsa::schedule_by_head(lut->sched_policy, B, H, L, d, dev) ? 1 : 0;
  std::vector<int32_t> own_items, own_start, own_records;
  const std::vector<int32_t>* sched_items = &lut->sched_records[o];
  const std::vector<int32_t>* sched_start = &lut->sched_start[o];
  if (lut->sched_grid != grid || lut->sched_start[o].empty()) {
    try {
      bsa::build_schedule(*lut, grid, o == 1, own_items, own_start);
      bsa::device_records(*lut, own_items, own_records);
    } catch (const std::bad_alloc&) {
      return BSA_ERR_ALLOC;
    }
    sched_items = &own_records;
    sched_start = &own_start;
  }

  CUtensorMap tq, tk, tv;
  if (!encode_rows_noalloc(&tq, q, rows, d, block, d / 64) ||
      !encode_rows_noalloc(&tk, k, rows, d, block, d / 64) ||
      !encode_rows_noalloc(&tv, v, rows, d, block, d / 64))
    return BSA_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word must start at zero; the LUT parts are overwritten in full.
  if (cudaMemsetAsync(base, 0, 16, st) != cudaSuccess ||
      (!sched_items->empty() &&
       cudaMemcpyAsync(base + off_items, sched_items->data(), sched_items->size() * 4,
                       cudaMemcpyHostToDevice, st) != cudaSuccess) ||
      cudaMemcpyAsync(base + off_start, sched_start->data(), sched_start->size() * 4,
                      cudaMemcpyHostToDevice, st) != cudaSuccess ||
      (!lut->col_idx.empty() &&
       cudaMemcpyAsync(base + off_colidx, lut->col_idx.data(), lut->col_idx.size() * 4,
                       cudaMemcpyHostToDevice, st) != cudaSuccess))
    return BSA_ERR_CUDA;

  bsa::FwdParams p{};
  p.items = reinterpret_cast<const int4*>(base + off_items);
  p.cta_start = base + off_start;
  p.col_idx = base + off_colidx;
  p.out = out;
  p.lse = lse;
  p.status = base;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.causal_diag = causal_diag != 0;
  p.wait_limit_ns = lut->wait_limit_ns;
  p.expire_site = lut->expire_site;
  p.Lq = p.Lk = L;
  p.H = H;
  p.window_left = p.window_right = -1;
  const cudaError_t e = bsa::launch_fwd_variant(block, block, d, false, p, tq, tk, tv, grid, st);
  if (e != cudaSuccess) return BSA_ERR_CUDA;
  if (!sync_status) return BSA_OK;
  int32_t word = 0;
  if (cudaMemcpyAsync(&word, base, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return BSA_ERR_CUDA;
  return word == 0 ? BSA_OK : BSA_ERR_DEVICE_TIMEOUT;
}
