// bsa_host.cpp -- host side of libbsa: LUT construction (CSR + work list), argument
// validation, TMA descriptor encoding and kernel launch.  See include/bsa.h for the
// contract of every exported function.
#include "../../include/bsa.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <new>

#include <cudaTypedefs.h>

#include "bsa_internal.h"

namespace {

constexpr int64_t kInt32Max = std::numeric_limits<int32_t>::max();

// ------------------------------------------------------------- LUT building

// Work-list keys.  Items are generated in (b, h, i) order, so a stable sort on the
// remaining key fields yields the documented total orders.
bool less_global(const int32_t* a, const int32_t* b) { return a[3] > b[3]; }

bool less_grouped(const int32_t* a, const int32_t* b) {
  if (a[0] != b[0]) return a[0] < b[0];
  if (a[1] != b[1]) return a[1] < b[1];
  return a[3] > b[3];
}

// ------------------------------------------------------------ TMA encoding

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [rows, d] bf16 view of a [B,H,L,d] tensor as three dimensions: 64 columns, rows,
// d/64 column halves (the halves 128 bytes apart, rows d*2 bytes apart).  The box is 64
// columns x `box_rows` rows x `box_halves` halves with the 128-byte swizzle: one copy
// lands the halves one after the other, each a swizzled [box_rows][64] region, which is
// the kernel's shared-memory operand layout.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, int d, int box_rows,
                 int box_halves) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(d / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_halves)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count(int dev) {
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Longest-processing-time-first assignment of the work list to `grid` CTAs.  Items are
// taken in work-list order (descending block count) and each goes to the CTA with the
// least work so far (ties: lowest index); an item costs 4 per active block plus 2 for
// its fixed per-item work (Q load, output write), so empty items spread out too.  Each
// CTA then walks its own items in the order it received them.  Round-robin assignment
// of the same list left the busiest CTA 4 % above the mean on the window workload.
// by_head takes the items (batch, head) by (batch, head) instead, keeping the list order
// within each pair: the CTAs then work on a few pairs at a time, whose K and V stay in L2.
void bsa::build_schedule(const bsa_lut& lut, int grid, bool by_head, std::vector<int32_t>& items,
                         std::vector<int32_t>& start) {
  build_schedule_list(lut.items, grid, by_head, items, start);
}

void bsa::build_schedule_list(const std::vector<int32_t>& list, int grid, bool by_head,
                              std::vector<int32_t>& items, std::vector<int32_t>& start) {
  const int n = static_cast<int>(list.size() / 4);
  std::vector<int32_t> order(static_cast<size_t>(n));
  for (int k = 0; k < n; ++k) order[static_cast<size_t>(k)] = k;
  if (by_head) {
    const int32_t* it = list.data();
    std::stable_sort(order.begin(), order.end(), [it](int32_t a, int32_t b) {
      const int32_t* x = it + 4 * static_cast<size_t>(a);
      const int32_t* y = it + 4 * static_cast<size_t>(b);
      return x[0] != y[0] ? x[0] < y[0] : x[1] < y[1];
    });
  }
  std::vector<int32_t> owner(static_cast<size_t>(n));
  std::vector<int32_t> count(static_cast<size_t>(grid), 0);
  // min-heap of (load, cta)
  using Load = std::pair<int64_t, int32_t>;
  std::vector<Load> heap;
  heap.reserve(static_cast<size_t>(grid));
  for (int c = 0; c < grid; ++c) heap.emplace_back(0, c);
  auto cmp = [](const Load& a, const Load& b) {
    return a.first != b.first ? a.first > b.first : a.second > b.second;
  };
  std::make_heap(heap.begin(), heap.end(), cmp);
  for (int k = 0; k < n; ++k) {
    std::pop_heap(heap.begin(), heap.end(), cmp);
    Load& top = heap.back();
    owner[static_cast<size_t>(k)] = top.second;
    ++count[static_cast<size_t>(top.second)];
    top.first += 4 * static_cast<int64_t>(list[static_cast<size_t>(order[static_cast<size_t>(k)]) * 4 + 3]) + 2;
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  start.assign(static_cast<size_t>(grid) + 1, 0);
  for (int c = 0; c < grid; ++c)
    start[static_cast<size_t>(c) + 1] = start[static_cast<size_t>(c)] + count[static_cast<size_t>(c)];
  std::vector<int32_t> fill(start.begin(), start.end() - 1);
  items.assign(static_cast<size_t>(n) * 4, 0);
  for (int k = 0; k < n; ++k) {
    const int32_t pos = fill[static_cast<size_t>(owner[static_cast<size_t>(k)])]++;
    std::memcpy(&items[static_cast<size_t>(pos) * 4],
                &list[static_cast<size_t>(order[static_cast<size_t>(k)]) * 4], 16);
  }
}

void bsa::device_records(const bsa_lut& lut, const std::vector<int32_t>& items,
                         std::vector<int32_t>& records) {
  records.resize(items.size());
  for (size_t k = 0; k + 3 < items.size(); k += 4) {
    const int32_t b = items[k], h = items[k + 1], i = items[k + 2], nnz = items[k + 3];
    const int32_t row = h * lut.nb + i;
    records[k] = b * lut.H + h;
    records[k + 1] = i;
    records[k + 2] = lut.row_ptr[static_cast<size_t>(row)];
    records[k + 3] = nnz | ((lut.diag_pos[static_cast<size_t>(row)] + 1) << 16);
  }
}

namespace {

// Device records of a regrouped column work list ({b, h, j, count} items):
// {b*H + h, j, first row_idx entry of the column, count | (dpos + 1) << 16}.
void csc_records(const bsa_lut& lut, const std::vector<int32_t>& items,
                 std::vector<int32_t>& records) {
  records.resize(items.size());
  for (size_t k = 0; k + 3 < items.size(); k += 4) {
    const int32_t b = items[k], h = items[k + 1], j = items[k + 2], cnt = items[k + 3];
    const int32_t col = h * lut.nb + j;
    records[k] = b * lut.H + h;
    records[k + 1] = j;
    records[k + 2] = lut.col_ptr[static_cast<size_t>(col)];
    records[k + 3] = cnt | ((lut.diag_pos_t[static_cast<size_t>(col)] + 1) << 16);
  }
}

}  // namespace

cudaError_t bsa::launch_bwd_variant(int block, int d, bool kv, const BwdParams& p,
                                    const CUtensorMap& a, const CUtensorMap& b,
                                    const CUtensorMap& x, const CUtensorMap& y, int grid,
                                    cudaStream_t stream) {
  if (block == 128)
    return d == 128 ? launch_bwd_b128_d128(kv, p, a, b, x, y, grid, stream)
                    : launch_bwd_b128_d64(kv, p, a, b, x, y, grid, stream);
  return d == 128 ? launch_bwd_b64_d128(kv, p, a, b, x, y, grid, stream)
                  : launch_bwd_b64_d64(kv, p, a, b, x, y, grid, stream);
}

cudaError_t bsa::launch_fwd_variant(int q_block, int kv_block, int d, bool ext,
                                    const FwdParams& p, const CUtensorMap& q, const CUtensorMap& k,
                                    const CUtensorMap& v, int grid, cudaStream_t stream) {
  const bool d128 = d == 128;
  if (q_block == 64 && kv_block == 64)
    return d128 ? launch_fwd_q64_k64_d128(ext, p, q, k, v, grid, stream)
                : launch_fwd_q64_k64_d64(ext, p, q, k, v, grid, stream);
  if (q_block == 128 && kv_block == 128)
    return d128 ? launch_fwd_q128_k128_d128(ext, p, q, k, v, grid, stream)
                : launch_fwd_q128_k128_d64(ext, p, q, k, v, grid, stream);
  if (q_block == 64 && kv_block == 128)
    return d128 ? launch_fwd_q64_k128_d128(ext, p, q, k, v, grid, stream)
                : launch_fwd_q64_k128_d64(ext, p, q, k, v, grid, stream);
  return d128 ? launch_fwd_q128_k64_d128(ext, p, q, k, v, grid, stream)
              : launch_fwd_q128_k64_d64(ext, p, q, k, v, grid, stream);
}

bool bsa::schedule_by_head(int policy, int64_t B, int64_t H, int64_t L, int64_t d, int dev) {
  if (policy == BSA_SCHEDULE_LIST) return false;
  if (policy == BSA_SCHEDULE_BY_HEAD) return true;
  static int cache[64] = {0};
  int l2 = (dev >= 0 && dev < 64) ? cache[dev] : 0;
  if (l2 <= 0) {
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0)
      return false;
    if (dev >= 0 && dev < 64) cache[dev] = l2;
  }
  return B * H * L * d * 4 > static_cast<int64_t>(l2);
}

namespace {

void free_device(bsa_lut* lut) {
  if (lut->d_row_idx) cudaFree(lut->d_row_idx);
  lut->d_row_idx = nullptr;
  for (int o = 0; o < 2; ++o) {
    if (lut->d_items_t[o]) cudaFree(lut->d_items_t[o]);
    if (lut->d_sched_start_t[o]) cudaFree(lut->d_sched_start_t[o]);
    lut->d_items_t[o] = lut->d_sched_start_t[o] = nullptr;
  }
  if (lut->d_col_idx) cudaFree(lut->d_col_idx);
  if (lut->d_items) cudaFree(lut->d_items);
  if (lut->d_status) cudaFree(lut->d_status);
  if (lut->d_sched_start) cudaFree(lut->d_sched_start);
  if (lut->d_items_g) cudaFree(lut->d_items_g);
  if (lut->d_sched_start_g) cudaFree(lut->d_sched_start_g);
  lut->d_items_g = lut->d_sched_start_g = nullptr;
  lut->d_col_idx = lut->d_items = lut->d_status = nullptr;
  lut->d_sched_start = nullptr;
  lut->device = -1;
}

}  // namespace

extern "C" {

int bsa_build_lut(const int32_t* layout, int H, int nb, int batch, int order, bsa_lut** out) {
  return bsa_build_lut_rect(layout, H, nb, nb, batch, order, out);
}

int bsa_build_lut_rect(const int32_t* layout, int H, int nb, int nbk, int batch, int order,
                       bsa_lut** out) {
  if (out == nullptr) return BSA_ERR_NULL;
  *out = nullptr;
  if (layout == nullptr) return BSA_ERR_NULL;
  // nb, nbk < 2^15: the device work-list record packs a row's count and diagonal
  // position into 16 bits each.
  if (H < 1 || nb < 1 || nb > 32767 || nbk < 1 || nbk > 32767 || batch < 1) return BSA_ERR_SHAPE;
  const int64_t cells = static_cast<int64_t>(H) * nb * nbk;
  const int64_t n_items = static_cast<int64_t>(batch) * H * nb;
  if (cells > kInt32Max || n_items > kInt32Max) return BSA_ERR_SHAPE;
  if (order != BSA_ORDER_GLOBAL && order != BSA_ORDER_GROUPED) return BSA_ERR_UNSUPPORTED;
  for (int64_t e = 0; e < cells; ++e)
    if (layout[e] != 0 && layout[e] != 1) return BSA_ERR_LAYOUT_VALUE;

  bsa_lut* lut = new (std::nothrow) bsa_lut();
  if (lut == nullptr) return BSA_ERR_ALLOC;
  try {
    lut->H = H;
    lut->nb = nb;
    lut->nbk = nbk;
    lut->batch = batch;
    lut->order = order;
    const int rows = H * nb;
    lut->row_ptr.assign(rows + 1, 0);
    for (int r = 0; r < rows; ++r) {
      const int32_t* lr = layout + static_cast<int64_t>(r) * nbk;
      int cnt = 0;
      for (int j = 0; j < nbk; ++j) cnt += lr[j];
      lut->row_ptr[r + 1] = lut->row_ptr[r] + cnt;
    }
    lut->nnz_total = lut->row_ptr[rows];
    lut->col_idx.resize(lut->nnz_total);
    for (int r = 0; r < rows; ++r) {
      const int32_t* lr = layout + static_cast<int64_t>(r) * nbk;
      int32_t* dst = lut->col_idx.data() + lut->row_ptr[r];
      for (int j = 0; j < nbk; ++j)
        if (lr[j]) *dst++ = j;
    }
    // Position of the diagonal block (j == i) inside each row, for the causal mask of the
    // plain kernels (equal block sizes).
    lut->diag_pos.assign(rows, -1);
    for (int r = 0; r < rows; ++r) {
      const int i = r % nb;
      for (int e = lut->row_ptr[r]; e < lut->row_ptr[r + 1]; ++e)
        if (lut->col_idx[e] == i) lut->diag_pos[r] = e - lut->row_ptr[r];
    }
    // Column view for the backward's key-side walk (square layouts).
    if (nb == nbk) {
      lut->has_csc = true;
      lut->col_ptr.assign(rows + 1, 0);
      for (int h = 0; h < H; ++h)
        for (int j = 0; j < nb; ++j) {
          int cnt = 0;
          for (int i = 0; i < nb; ++i) cnt += layout[(static_cast<int64_t>(h) * nb + i) * nb + j];
          lut->col_ptr[h * nb + j + 1] = lut->col_ptr[h * nb + j] + cnt;
        }
      lut->row_idx.resize(lut->nnz_total);
      lut->diag_pos_t.assign(rows, -1);
      for (int h = 0; h < H; ++h)
        for (int j = 0; j < nb; ++j) {
          int32_t* dst = lut->row_idx.data() + lut->col_ptr[h * nb + j];
          int e = 0;
          for (int i = 0; i < nb; ++i)
            if (layout[(static_cast<int64_t>(h) * nb + i) * nb + j]) {
              if (i == j) lut->diag_pos_t[h * nb + j] = e;
              dst[e++] = i;
            }
        }
      lut->items_t.resize(static_cast<size_t>(n_items) * 4);
      std::vector<int32_t> rawt(static_cast<size_t>(n_items) * 4);
      size_t wt = 0;
      for (int b = 0; b < batch; ++b)
        for (int h = 0; h < H; ++h)
          for (int j = 0; j < nb; ++j) {
            rawt[wt++] = b;
            rawt[wt++] = h;
            rawt[wt++] = j;
            rawt[wt++] = lut->col_ptr[h * nb + j + 1] - lut->col_ptr[h * nb + j];
          }
      std::vector<const int32_t*> idt(static_cast<size_t>(n_items));
      for (size_t e = 0; e < idt.size(); ++e) idt[e] = rawt.data() + 4 * e;
      std::stable_sort(idt.begin(), idt.end(), less_global);
      for (size_t e = 0; e < idt.size(); ++e) std::memcpy(&lut->items_t[4 * e], idt[e], 16);
    }
    lut->n_items = static_cast<int>(n_items);
    std::vector<int32_t> raw(static_cast<size_t>(n_items) * 4);
    size_t w = 0;
    for (int b = 0; b < batch; ++b)
      for (int h = 0; h < H; ++h)
        for (int i = 0; i < nb; ++i) {
          const int r = h * nb + i;
          raw[w++] = b;
          raw[w++] = h;
          raw[w++] = i;
          raw[w++] = lut->row_ptr[r + 1] - lut->row_ptr[r];
        }
    std::vector<const int32_t*> idx(static_cast<size_t>(n_items));
    for (size_t e = 0; e < idx.size(); ++e) idx[e] = raw.data() + 4 * e;
    std::stable_sort(idx.begin(), idx.end(),
                     order == BSA_ORDER_GLOBAL ? less_global : less_grouped);
    lut->items.resize(raw.size());
    for (size_t e = 0; e < idx.size(); ++e) std::memcpy(&lut->items[4 * e], idx[e], 16);
  } catch (const std::bad_alloc&) {
    delete lut;
    return BSA_ERR_ALLOC;
  }
  *out = lut;
  return BSA_OK;
}

int bsa_lut_info(const bsa_lut* lut, int* H, int* nb, int* batch, int* nnz_total, int* n_items) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (H) *H = lut->H;
  if (nb) *nb = lut->nb;
  if (batch) *batch = lut->batch;
  if (nnz_total) *nnz_total = lut->nnz_total;
  if (n_items) *n_items = lut->n_items;
  return BSA_OK;
}

int bsa_lut_kv_blocks(const bsa_lut* lut, int* nbk) {
  if (lut == nullptr || nbk == nullptr) return BSA_ERR_NULL;
  *nbk = lut->nbk;
  return BSA_OK;
}

int bsa_lut_export(const bsa_lut* lut, int32_t* row_ptr, int32_t* col_idx, int32_t* items) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (row_ptr) std::memcpy(row_ptr, lut->row_ptr.data(), lut->row_ptr.size() * 4);
  if (col_idx && !lut->col_idx.empty())
    std::memcpy(col_idx, lut->col_idx.data(), lut->col_idx.size() * 4);
  if (items) std::memcpy(items, lut->items.data(), lut->items.size() * 4);
  return BSA_OK;
}

int bsa_lut_schedule(const bsa_lut* lut, int grid, int by_head, int32_t* items,
                     int32_t* cta_start) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (grid < 1 || grid > std::max(1, lut->n_items)) return BSA_ERR_SHAPE;
  std::vector<int32_t> it, st;
  try {
    bsa::build_schedule(*lut, grid, by_head != 0, it, st);
  } catch (const std::bad_alloc&) {
    return BSA_ERR_ALLOC;
  }
  if (items && !it.empty()) std::memcpy(items, it.data(), it.size() * 4);
  if (cta_start) std::memcpy(cta_start, st.data(), st.size() * 4);
  return BSA_OK;
}

int bsa_lut_upload(bsa_lut* lut, void* stream) {
  if (lut == nullptr) return BSA_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  free_device(lut);
  const int sms = sm_count(dev);
  if (sms <= 0) return BSA_ERR_CUDA;
  lut->sched_grid = std::max(1, std::min(lut->n_items, sms));
  std::vector<int32_t>* rec = lut->sched_records;  // device records of both schedules
  try {
    for (int o = 0; o < 2; ++o) {
      bsa::build_schedule(*lut, lut->sched_grid, o == 1, lut->sched_items[o], lut->sched_start[o]);
      bsa::device_records(*lut, lut->sched_items[o], rec[o]);
    }
  } catch (const std::bad_alloc&) {
    lut->sched_grid = 0;
    return BSA_ERR_ALLOC;
  }
  const size_t nc = std::max<size_t>(lut->col_idx.size(), 1) * 4;
  const size_t ni = std::max<size_t>(lut->items.size(), 4) * 4;
  const size_t ns = lut->sched_start[0].size() * 4;
  if (cudaMalloc(&lut->d_col_idx, nc) != cudaSuccess || cudaMalloc(&lut->d_items, ni) != cudaSuccess ||
      cudaMalloc(&lut->d_status, 16) != cudaSuccess ||
      cudaMalloc(&lut->d_sched_start, ns) != cudaSuccess ||
      cudaMalloc(&lut->d_items_g, ni) != cudaSuccess ||
      cudaMalloc(&lut->d_sched_start_g, ns) != cudaSuccess) {
    free_device(lut);
    cudaGetLastError();
    return BSA_ERR_ALLOC;
  }
  bool ok = (lut->col_idx.empty() ||
             cudaMemcpyAsync(lut->d_col_idx, lut->col_idx.data(), lut->col_idx.size() * 4,
                             cudaMemcpyHostToDevice, st) == cudaSuccess) &&
            (rec[0].empty() ||
             (cudaMemcpyAsync(lut->d_items, rec[0].data(), rec[0].size() * 4,
                              cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(lut->d_items_g, rec[1].data(), rec[1].size() * 4,
                              cudaMemcpyHostToDevice, st) == cudaSuccess)) &&
            cudaMemcpyAsync(lut->d_sched_start, lut->sched_start[0].data(), ns,
                            cudaMemcpyHostToDevice, st) == cudaSuccess &&
            cudaMemcpyAsync(lut->d_sched_start_g, lut->sched_start[1].data(), ns,
                            cudaMemcpyHostToDevice, st) == cudaSuccess &&
            cudaMemsetAsync(lut->d_status, 0, 16, st) == cudaSuccess &&
            cudaStreamSynchronize(st) == cudaSuccess;
  if (ok && lut->has_csc) {
    try {
      for (int o = 0; o < 2; ++o) {
        std::vector<int32_t> it;
        bsa::build_schedule_list(lut->items_t, lut->sched_grid, o == 1, it, lut->sched_start_t[o]);
        csc_records(*lut, it, lut->sched_records_t[o]);
      }
    } catch (const std::bad_alloc&) {
      free_device(lut);
      return BSA_ERR_ALLOC;
    }
    const size_t nr = std::max<size_t>(lut->row_idx.size(), 1) * 4;
    if (cudaMalloc(&lut->d_row_idx, nr) != cudaSuccess ||
        cudaMalloc(&lut->d_items_t[0], ni) != cudaSuccess ||
        cudaMalloc(&lut->d_items_t[1], ni) != cudaSuccess ||
        cudaMalloc(&lut->d_sched_start_t[0], ns) != cudaSuccess ||
        cudaMalloc(&lut->d_sched_start_t[1], ns) != cudaSuccess) {
      free_device(lut);
      cudaGetLastError();
      return BSA_ERR_ALLOC;
    }
    ok = lut->row_idx.empty() ||
         cudaMemcpyAsync(lut->d_row_idx, lut->row_idx.data(), lut->row_idx.size() * 4,
                         cudaMemcpyHostToDevice, st) == cudaSuccess;
    for (int o = 0; o < 2 && ok; ++o)
      ok = (lut->sched_records_t[o].empty() ||
            cudaMemcpyAsync(lut->d_items_t[o], lut->sched_records_t[o].data(),
                            lut->sched_records_t[o].size() * 4, cudaMemcpyHostToDevice,
                            st) == cudaSuccess) &&
           cudaMemcpyAsync(lut->d_sched_start_t[o], lut->sched_start_t[o].data(), ns,
                           cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
  }
  if (!ok) {
    free_device(lut);
    return BSA_ERR_CUDA;
  }
  lut->device = dev;
  return BSA_OK;
}

void bsa_lut_free(bsa_lut* lut) {
  if (lut == nullptr) return;
  free_device(lut);
  delete lut;
}

int bsa_forward(const void* q, const void* k, const void* v, const bsa_lut* lut, void* out,
                float* lse, int B, int H, int L, int d, float scale, int block, int causal_diag,
                void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || lut == nullptr || out == nullptr ||
      lse == nullptr)
    return BSA_ERR_NULL;
  if ((block != 64 && block != 128) || (d != 64 && d != 128)) return BSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return BSA_ERR_UNSUPPORTED;
  if (B != lut->batch || H != lut->H || L <= 0 || lut->nbk != lut->nb ||
      static_cast<int64_t>(lut->nb) * block != L)
    return BSA_ERR_SHAPE;
  const int64_t rows = static_cast<int64_t>(B) * H * L;
  if (rows > kInt32Max - 128) return BSA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return BSA_ERR_ALIGN;
  if (lut->d_items == nullptr) return BSA_ERR_STATE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  if (dev != lut->device) return BSA_ERR_STATE;

  CUtensorMap tq, tk, tv;
  if (!encode_rows(&tq, q, rows, d, block, d / 64) || !encode_rows(&tk, k, rows, d, block, d / 64) ||
      !encode_rows(&tv, v, rows, d, block, d / 64))
    return BSA_ERR_CUDA;

  bsa::FwdParams p{};
  const bool by_head = bsa::schedule_by_head(lut->sched_policy, B, H, L, d, dev);
  p.items = reinterpret_cast<const int4*>(by_head ? lut->d_items_g : lut->d_items);
  p.cta_start = by_head ? lut->d_sched_start_g : lut->d_sched_start;
  p.col_idx = lut->d_col_idx;
  p.out = out;
  p.lse = lse;
  p.status = lut->d_status;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.causal_diag = causal_diag != 0;
  p.wait_limit_ns = lut->wait_limit_ns;
  p.expire_site = lut->expire_site;
  p.Lq = p.Lk = L;
  p.H = H;
  p.window_left = p.window_right = -1;

  const int grid = lut->sched_grid;  // the schedule uploaded with the LUT
  if (grid <= 0) return BSA_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = bsa::launch_fwd_variant(block, block, d, false, p, tq, tk, tv, grid, st);
  return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

int bsa_forward_ext(const void* q, const void* k, const void* v, const bsa_lut* lut, void* out,
                    float* lse, int B, int H, int Lq, int Lk, int d, float scale, int q_block,
                    int kv_block, int causal_diag, const bsa_ext_args* ext, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || lut == nullptr || out == nullptr ||
      lse == nullptr)
    return BSA_ERR_NULL;
  bsa_ext_args x{-1, -1, 0.f, nullptr, nullptr, nullptr};
  if (ext != nullptr) x = *ext;
  if ((x.q_segment_ids == nullptr) != (x.kv_segment_ids == nullptr)) return BSA_ERR_NULL;
  if ((q_block != 64 && q_block != 128) || (kv_block != 64 && kv_block != 128) ||
      (d != 64 && d != 128))
    return BSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !std::isfinite(x.softcap) || x.softcap < 0.f)
    return BSA_ERR_UNSUPPORTED;
  if (B != lut->batch || H != lut->H || Lq <= 0 || Lk <= 0 ||
      lut->nb != (Lq + q_block - 1) / q_block || lut->nbk != (Lk + kv_block - 1) / kv_block)
    return BSA_ERR_SHAPE;
  const int64_t rows_q = static_cast<int64_t>(B) * H * Lq;
  const int64_t rows_k = static_cast<int64_t>(B) * H * Lk;
  if (rows_q > kInt32Max - 128 || rows_k > kInt32Max - 128) return BSA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return BSA_ERR_ALIGN;
  auto aligned4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
  if (!aligned4(x.sinks) || !aligned4(x.q_segment_ids) || !aligned4(x.kv_segment_ids))
    return BSA_ERR_ALIGN;
  const bool plain = q_block == kv_block && Lq == Lk && Lq % q_block == 0 && x.window_left < 0 &&
                     x.window_right < 0 && x.softcap == 0.f && x.sinks == nullptr &&
                     x.q_segment_ids == nullptr;
  if (plain)  // nothing beyond the plain operation: the plain kernel
    return bsa_forward(q, k, v, lut, out, lse, B, H, Lq, d, scale, q_block, causal_diag, stream);
  if (lut->d_items == nullptr) return BSA_ERR_STATE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  if (dev != lut->device) return BSA_ERR_STATE;

  CUtensorMap tq, tk, tv;
  if (!encode_rows(&tq, q, rows_q, d, q_block, d / 64) ||
      !encode_rows(&tk, k, rows_k, d, kv_block, d / 64) ||
      !encode_rows(&tv, v, rows_k, d, kv_block, d / 64))
    return BSA_ERR_CUDA;
  bsa::FwdParams p{};
  const bool by_head = bsa::schedule_by_head(lut->sched_policy, B, H, Lk, d, dev);
  p.items = reinterpret_cast<const int4*>(by_head ? lut->d_items_g : lut->d_items);
  p.cta_start = by_head ? lut->d_sched_start_g : lut->d_sched_start;
  p.col_idx = lut->d_col_idx;
  p.out = out;
  p.lse = lse;
  p.status = lut->d_status;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.causal_diag = causal_diag != 0;
  p.wait_limit_ns = lut->wait_limit_ns;
  p.expire_site = lut->expire_site;
  p.Lq = Lq;
  p.Lk = Lk;
  p.H = H;
  p.window_left = x.window_left < 0 ? -1 : x.window_left;
  p.window_right = x.window_right < 0 ? -1 : x.window_right;
  if (x.softcap > 0.f) {
    p.softcap_log2 = static_cast<float>(static_cast<double>(x.softcap) * 1.4426950408889634);
    p.softcap_inv = static_cast<float>(static_cast<double>(scale) / x.softcap);
  }
  p.sinks = x.sinks;
  p.q_seg = x.q_segment_ids;
  p.kv_seg = x.kv_segment_ids;
  const int grid = lut->sched_grid;
  if (grid <= 0) return BSA_ERR_STATE;
  const cudaError_t e = bsa::launch_fwd_variant(q_block, kv_block, d, true, p, tq, tk, tv, grid,
                                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

int bsa_lut_export_csc(const bsa_lut* lut, int32_t* col_ptr, int32_t* row_idx, int32_t* items) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (!lut->has_csc) return BSA_ERR_SHAPE;
  if (col_ptr) std::memcpy(col_ptr, lut->col_ptr.data(), lut->col_ptr.size() * 4);
  if (row_idx && !lut->row_idx.empty())
    std::memcpy(row_idx, lut->row_idx.data(), lut->row_idx.size() * 4);
  if (items) std::memcpy(items, lut->items_t.data(), lut->items_t.size() * 4);
  return BSA_OK;
}

int bsa_backward(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout, const bsa_lut* lut, void* dq, void* dk, void* dv, float* delta,
                 int B, int H, int L, int d, float scale, int block, int causal_diag,
                 void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || lse == nullptr ||
      dout == nullptr || lut == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
      delta == nullptr)
    return BSA_ERR_NULL;
  if ((block != 64 && block != 128) || (d != 64 && d != 128)) return BSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return BSA_ERR_UNSUPPORTED;
  if (!lut->has_csc || B != lut->batch || H != lut->H || L <= 0 ||
      static_cast<int64_t>(lut->nb) * block != L)
    return BSA_ERR_SHAPE;
  const int64_t rows = static_cast<int64_t>(B) * H * L;
  if (rows > kInt32Max - 128) return BSA_ERR_SHAPE;
  for (const void* ptr : {q, k, v, out, static_cast<const void*>(lse), dout,
                          static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv), static_cast<const void*>(delta)})
    if (!aligned16(ptr)) return BSA_ERR_ALIGN;
  if (lut->d_items_t[0] == nullptr) return BSA_ERR_STATE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  if (dev != lut->device) return BSA_ERR_STATE;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_rows(&tq, q, rows, d, block, d / 64) || !encode_rows(&tk, k, rows, d, block, d / 64) ||
      !encode_rows(&tv, v, rows, d, block, d / 64) ||
      !encode_rows(&tdo, dout, rows, d, block, d / 64))
    return BSA_ERR_CUDA;
  const int grid = lut->sched_grid;
  if (grid <= 0) return BSA_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int o = bsa::schedule_by_head(lut->sched_policy, B, H, L, d, dev) ? 1 : 0;
  bsa::BwdParams p{};
  p.lse = lse;
  p.delta = delta;
  p.status = lut->d_status;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.scale = scale;
  p.causal_diag = causal_diag != 0;
  p.L = L;
  p.wait_limit_ns = lut->wait_limit_ns;
  p.expire_site = lut->expire_site;
  // delta = rowsum(dO * O), then dQ over the rows, then dK and dV over the columns.
  if (bsa::launch_bwd_delta(out, dout, delta, rows, d, st) != cudaSuccess) return BSA_ERR_CUDA;
  p.items = reinterpret_cast<const int4*>(o ? lut->d_items_g : lut->d_items);
  p.cta_start = o ? lut->d_sched_start_g : lut->d_sched_start;
  p.col_idx = lut->d_col_idx;
  p.out1 = dq;
  if (bsa::launch_bwd_variant(block, d, false, p, tq, tdo, tk, tv, grid, st) != cudaSuccess)
    return BSA_ERR_CUDA;
  p.items = reinterpret_cast<const int4*>(lut->d_items_t[o]);
  p.cta_start = lut->d_sched_start_t[o];
  p.col_idx = lut->d_row_idx;
  p.out1 = dv;
  p.out2 = dk;
  if (bsa::launch_bwd_variant(block, d, true, p, tk, tv, tq, tdo, grid, st) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

int bsa_device_status(const bsa_lut* lut, void* stream, int32_t* detail) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (lut->d_status == nullptr) return BSA_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpyAsync(&word, lut->d_status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(lut->d_status, 0, 4, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (detail) *detail = word;
  return word == 0 ? BSA_OK : BSA_ERR_DEVICE_TIMEOUT;
}

int bsa_set_schedule(bsa_lut* lut, int policy) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (policy != BSA_SCHEDULE_AUTO && policy != BSA_SCHEDULE_LIST && policy != BSA_SCHEDULE_BY_HEAD)
    return BSA_ERR_UNSUPPORTED;
  lut->sched_policy = policy;
  return BSA_OK;
}

int bsa_set_wait_limit(bsa_lut* lut, uint64_t ns) {
  if (lut == nullptr) return BSA_ERR_NULL;
  lut->wait_limit_ns = ns == 0 ? 10000000000ull : ns;
  return BSA_OK;
}

int bsa_debug_expire_wait(bsa_lut* lut, int site) {
  if (lut == nullptr) return BSA_ERR_NULL;
  if (site < 0 || site > 0xFFFF) return BSA_ERR_UNSUPPORTED;
  lut->expire_site = site;
  return BSA_OK;
}

int bsa_wait_selftest(uint64_t limit_ns, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* d = nullptr;
  if (cudaMalloc(&d, 4) != cudaSuccess) return BSA_ERR_ALLOC;
  int32_t word = 0;
  bool ok = cudaMemsetAsync(d, 0, 4, st) == cudaSuccess &&
            bsa::launch_wait_selftest(d, limit_ns, st) == cudaSuccess &&
            cudaMemcpyAsync(&word, d, 4, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
            cudaStreamSynchronize(st) == cudaSuccess;
  cudaFree(d);
  if (!ok) return BSA_ERR_CUDA;
  return word == (bsa::kSiteSelftest | 0x10000) ? BSA_ERR_DEVICE_TIMEOUT : BSA_OK;
}

const char* bsa_status_string(int status) {
  switch (status) {
    case BSA_OK: return "ok";
    case BSA_ERR_NULL: return "null pointer argument";
    case BSA_ERR_SHAPE: return "inconsistent sizes";
    case BSA_ERR_LAYOUT_VALUE: return "layout value not 0 or 1";
    case BSA_ERR_DTYPE: return "unsupported element type";
    case BSA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case BSA_ERR_UNSUPPORTED: return "unsupported block/head-dim/order/scale";
    case BSA_ERR_CUDA: return "CUDA call failed";
    case BSA_ERR_DEVICE_TIMEOUT: return "bounded wait timed out on the device";
    case BSA_ERR_STATE: return "LUT not uploaded to the current device";
    case BSA_ERR_ALLOC: return "allocation failed";
    case BSA_ERR_TOO_LARGE: return "LUT too large for the fixed 4 MiB no-allocation scratch";
    default: return "unknown status";
  }
}

const char* bsa_version(void) { return "0.1.0"; }

}  // extern "C"
