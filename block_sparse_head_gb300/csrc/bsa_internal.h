// bsa_internal.h -- types shared by the host library and the kernel translation units.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

// The look-up table behind the opaque bsa_lut handle of bsa.h.
struct bsa_lut {
  int H = 0, nb = 0, batch = 0, order = 0;
  int nbk = 0;  // key blocks per row (nb for a square layout)
  int nnz_total = 0, n_items = 0;
  std::vector<int32_t> row_ptr;  // [H*nb + 1]
  std::vector<int32_t> col_idx;  // [nnz_total]
  std::vector<int32_t> items;    // [n_items][4] = {b, h, i, nnz}
  std::vector<int32_t> diag_pos; // [H*nb]: index of block j == i in row (h, i), or -1
  // Device schedules for `sched_grid` CTAs (built at upload): the work list regrouped
  // so that CTA c takes sched_items[o][sched_start[o][c] .. sched_start[o][c+1]).  o = 0
  // hands items out in work-list order, o = 1 (batch, head) by (batch, head).
  int sched_grid = 0;
  int sched_policy = 0;  // BSA_SCHEDULE_*
  std::vector<int32_t> sched_items[2];  // [n_items][4]
  std::vector<int32_t> sched_start[2];  // [sched_grid + 1]
  std::vector<int32_t> sched_records[2];  // device records of sched_items (device_records)
  // Column view (square layouts only; the backward's key-side walk): col_ptr over
  // columns h*nb + j, row_idx the active query blocks i ascending, items_t one
  // {b, h, j, count} per (batch, head, key block) sorted by (-count, b, h, j), diag_pos_t
  // the position of i == j in each column (-1: none); and its two per-CTA schedules.
  bool has_csc = false;
  std::vector<int32_t> col_ptr, row_idx, items_t, diag_pos_t;
  std::vector<int32_t> sched_records_t[2];
  std::vector<int32_t> sched_start_t[2];
  // device copies (valid after bsa_lut_upload)
  int device = -1;
  int32_t* d_col_idx = nullptr;
  int32_t* d_items = nullptr;
  int32_t* d_status = nullptr;
  int32_t* d_sched_start = nullptr;  // device copy of sched_start[0] (d_items: records of sched_items[0])
  int32_t* d_items_g = nullptr;        // records of sched_items[1]
  int32_t* d_sched_start_g = nullptr;  // sched_start[1]
  int32_t* d_row_idx = nullptr;        // column view: row_idx
  int32_t* d_items_t[2] = {nullptr, nullptr};        // records of both column schedules
  int32_t* d_sched_start_t[2] = {nullptr, nullptr};
  uint64_t wait_limit_ns = 10000000000ull;
  int expire_site = 0;  // bsa_debug_expire_wait
};

namespace bsa {

// Kernel arguments besides the three tensor maps.
struct FwdParams {
  const int4* items;        // work list regrouped per CTA, as device records (kernel header)
  const int32_t* cta_start; // CTA c takes items[cta_start[c] .. cta_start[c+1])
  const int32_t* col_idx;   // active column blocks, ascending per row
  void* out;                // bf16 [B,H,L,d]
  float* lse;               // fp32 [B,H,L]
  int32_t* status;          // device status word (0 = fine)
  float scale_log2;         // scale * log2(e)
  int causal_diag;
  unsigned long long wait_limit_ns;
  int expire_site;          // wait site that gives up at once (0: none; bsa_debug_expire_wait)
  int Lq, Lk;               // rows per (batch, head) of Q/O and of K/V
  // Extended kernels only:
  int H;                    // heads: a record's bh = b * H + h
  int window_left, window_right;  // keys c < r - left / c > r + right masked (< 0: no bound)
  float softcap_log2;       // cap * log2(e); 0: no soft-cap
  float softcap_inv;        // scale / cap
  const float* sinks;       // [H] sink logits (natural log units) or null
  const int32_t* q_seg;     // [B, Lq] or null
  const int32_t* kv_seg;    // [B, Lk] or null (null exactly when q_seg is)
};

// Wait-site ids recorded in the status word's low bits.
enum WaitSite : int {
  kSiteProdKEmpty = 1,
  kSiteProdVEmpty = 2,
  kSiteMmaStage = 6,
  kSiteMmaPFull = 7,
  kSiteMmaPvDone = 8,
  kSiteSoftSFull = 9,
  kSiteMmaORead = 10,
  kSiteSoftPvDone = 11,
  kSiteSoftItemDone = 12,
  kSiteEpiStats = 13,
  kSiteSoftStatsFree = 14,
  kSiteSelftest = 15,
};

// Regroups lut's work list for `grid` CTAs: CTA c takes items[start[c] .. start[c+1]).
// by_head: hand the items out (batch, head) by (batch, head) instead of in list order.
void build_schedule(const bsa_lut& lut, int grid, bool by_head, std::vector<int32_t>& items,
                    std::vector<int32_t>& start);
// The same for any work list `list` of {b, h, block, count} items.
void build_schedule_list(const std::vector<int32_t>& list, int grid, bool by_head,
                         std::vector<int32_t>& items, std::vector<int32_t>& start);

// Device records of a regrouped work list `items` ({b, h, i, nnz} each):
// {b*H + h, i, first col_idx entry of the row, nnz | (dpos + 1) << 16} with dpos the
// position of block j == i in row (h, i) (-1 if absent), so the kernel needs no other
// table to start an item.
void device_records(const bsa_lut& lut, const std::vector<int32_t>& items,
                    std::vector<int32_t>& records);

// Whether a forward over [B,H,L,d] should use the (batch, head) schedule: as `policy`
// says, or (BSA_SCHEDULE_AUTO) when its K and V (B*H*L*d*4 bytes) exceed the L2 of
// device `dev`.
bool schedule_by_head(int policy, int64_t B, int64_t H, int64_t L, int64_t d, int dev);

// Launches the forward kernel for (q_block, kv_block, head_dim, ext); the instances live
// in their own translation units (bsa_fwd_q*_k*_d*.cu) so they compile in parallel.  The
// plain kernels (ext = false) exist for q_block == kv_block only.
cudaError_t launch_fwd_variant(int q_block, int kv_block, int d, bool ext, const FwdParams& p,
                               const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               int grid, cudaStream_t stream);
cudaError_t launch_fwd_q64_k64_d64(bool ext, const FwdParams& p, const CUtensorMap& q,
                                  const CUtensorMap& k, const CUtensorMap& v, int grid,
                                  cudaStream_t stream);
cudaError_t launch_fwd_q64_k64_d128(bool ext, const FwdParams& p, const CUtensorMap& q,
                                   const CUtensorMap& k, const CUtensorMap& v, int grid,
                                   cudaStream_t stream);
cudaError_t launch_fwd_q128_k128_d64(bool ext, const FwdParams& p, const CUtensorMap& q,
                                    const CUtensorMap& k, const CUtensorMap& v, int grid,
                                    cudaStream_t stream);
cudaError_t launch_fwd_q128_k128_d128(bool ext, const FwdParams& p, const CUtensorMap& q,
                                     const CUtensorMap& k, const CUtensorMap& v, int grid,
                                     cudaStream_t stream);
cudaError_t launch_fwd_q64_k128_d64(bool ext, const FwdParams& p, const CUtensorMap& q,
                                   const CUtensorMap& k, const CUtensorMap& v, int grid,
                                   cudaStream_t stream);
cudaError_t launch_fwd_q64_k128_d128(bool ext, const FwdParams& p, const CUtensorMap& q,
                                    const CUtensorMap& k, const CUtensorMap& v, int grid,
                                    cudaStream_t stream);
cudaError_t launch_fwd_q128_k64_d64(bool ext, const FwdParams& p, const CUtensorMap& q,
                                   const CUtensorMap& k, const CUtensorMap& v, int grid,
                                   cudaStream_t stream);
cudaError_t launch_fwd_q128_k64_d128(bool ext, const FwdParams& p, const CUtensorMap& q,
                                    const CUtensorMap& k, const CUtensorMap& v, int grid,
                                    cudaStream_t stream);

// Backward kernel arguments besides the four tensor maps (item tiles A, B; step tiles X, Y).
struct BwdParams {
  const int4* items;         // work list regrouped per CTA (records as in the forward)
  const int32_t* cta_start;  // CTA c takes items[cta_start[c] .. cta_start[c+1])
  const int32_t* col_idx;    // dQ: key blocks of each row; dK/dV: query blocks of each column
  const float* lse;          // [B,H,L] from the forward
  const float* delta;        // [B,H,L] = rowsum(dO * O)
  void* out1;                // dQ mode: dq; dK/dV mode: dv   (bf16 [B,H,L,d])
  void* out2;                // dK/dV mode: dk
  int32_t* status;
  float scale_log2;          // scale * log2(e)
  float scale;
  int causal_diag;
  int L;
  unsigned long long wait_limit_ns;
  int expire_site;
};

// Backward kernels for (block, head_dim); kv selects the dK/dV walk over the columns
// (else dQ over the rows).  Each (block, head_dim) pair lives in its own translation unit.
cudaError_t launch_bwd_variant(int block, int d, bool kv, const BwdParams& p, const CUtensorMap& a,
                               const CUtensorMap& b, const CUtensorMap& x, const CUtensorMap& y,
                               int grid, cudaStream_t stream);
cudaError_t launch_bwd_b64_d64(bool kv, const BwdParams& p, const CUtensorMap& a,
                               const CUtensorMap& b, const CUtensorMap& x, const CUtensorMap& y,
                               int grid, cudaStream_t stream);
cudaError_t launch_bwd_b64_d128(bool kv, const BwdParams& p, const CUtensorMap& a,
                                const CUtensorMap& b, const CUtensorMap& x, const CUtensorMap& y,
                                int grid, cudaStream_t stream);
cudaError_t launch_bwd_b128_d64(bool kv, const BwdParams& p, const CUtensorMap& a,
                                const CUtensorMap& b, const CUtensorMap& x, const CUtensorMap& y,
                                int grid, cudaStream_t stream);
cudaError_t launch_bwd_b128_d128(bool kv, const BwdParams& p, const CUtensorMap& a,
                                 const CUtensorMap& b, const CUtensorMap& x, const CUtensorMap& y,
                                 int grid, cudaStream_t stream);
// delta[r] = sum_x dout[r,x] out[r,x] over `rows` rows of d bf16 (fp32 result).
cudaError_t launch_bwd_delta(const void* out, const void* dout, float* delta, int64_t rows, int d,
                             cudaStream_t stream);

// One-CTA kernel whose only wait never completes; it must give up after limit_ns.
cudaError_t launch_wait_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace bsa
