/*
 * bsa.h -- C ABI of libbsa: layout-driven block-sparse multi-head attention forward
 * on GB300 (sm_103a).
 *
 * The operation.  A per-head int32 block layout [H x nb x nb] (nb = L / block) marks
 * which block x block tiles of the attention matrix are computed: 1 = compute,
 * 0 = skip (layout of the "Implementation:Deepspeedai DeepSpeed Sparse Attention
 * Utils" page, "I/O Contract").  For batch b, head h and query row r the output is
 * masked softmax attention over exactly the active keys
 *
 *     A(r)   = { c : layout[h][r/block][c/block] == 1,
 *                    and not (causal_diag && r/block == c/block && c > r) }
 *     s_c    = scale * <q[b,h,r,:], k[b,h,c,:]>
 *     lse[r] = ln sum_{c in A(r)} exp(s_c)                (-inf when A(r) is empty)
 *     O[r,:] = sum_{c in A(r)} exp(s_c - lse[r]) v[b,h,c,:]  (0 when A(r) is empty)
 *
 * i.e. dense attention (page "Block Sparse Attention Techniques", section 1,
 * "Scaled Dot-Product Attention") under the elementwise mask that the block layout
 * expands to (page "Block-Sparse Attention", section "Block Structure"; the masked
 * scores are -inf as in the Longformer case-study equation of "Block Sparse
 * Attention Techniques", section 2).  The online-softmax evaluation and the all-zero
 * output of an empty row follow the sparse_attn kernel of the DeepSeek-V4.1
 * "Sparse attention / Weighted row sum" page.
 *
 * Conventions shared by every call:
 *   - Return value: BSA_OK (0) or a negative bsa_status.  No call aborts, throws or
 *     prints.  Arguments are validated before any device work is queued.
 *   - Tensors are dense, row-major, C-contiguous; "[B,H,L,d]" means element
 *     (b,h,l,x) sits at ((b*H + h)*L + l)*d + x.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Device pointers must belong to the device that is current when the call is
 *     made, the same device the LUT was uploaded to.
 */
#ifndef BSA_H_
#define BSA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bsa_status {
  BSA_OK = 0,
  BSA_ERR_NULL = -1,           /* a required pointer is NULL                           */
  BSA_ERR_SHAPE = -2,          /* sizes inconsistent (L != nb*block, H/B vs the LUT...) */
  BSA_ERR_LAYOUT_VALUE = -3,   /* a layout entry is neither 0 nor 1                    */
  BSA_ERR_DTYPE = -4,          /* reserved for bindings that see element types          */
  BSA_ERR_ALIGN = -5,          /* a tensor pointer is not 16-byte aligned              */
  BSA_ERR_UNSUPPORTED = -6,    /* (block, d) pair or order flag not supported          */
  BSA_ERR_CUDA = -7,           /* a CUDA runtime/driver call failed                    */
  BSA_ERR_DEVICE_TIMEOUT = -8, /* a bounded wait inside the kernel ran out             */
  BSA_ERR_STATE = -9,          /* the LUT has not been uploaded to a device            */
  BSA_ERR_ALLOC = -10,         /* host or device allocation failed                     */
  BSA_ERR_TOO_LARGE = -11      /* LUT does not fit the fixed scratch of
                                  bsa_forward_noalloc                                   */
} bsa_status;

/* Work-list orders accepted by bsa_build_lut. */
enum {
  BSA_ORDER_GLOBAL = 0,  /* items sorted by (-nnz, b, h, i): longest rows first           */
  BSA_ORDER_GROUPED = 1  /* items sorted by (b, h, -nnz, i): one (b,h) at a time, K/V
                            tiles stay hot in L2                                          */
};

/* Opaque look-up table: host CSR + work list, plus device copies after upload.
 * Owned by the library; released by bsa_lut_free. */
typedef struct bsa_lut bsa_lut;

/*
 * bsa_build_lut -- turn a block layout into a CSR of active column blocks and a
 * load-balanced work list (host only; needs no GPU).
 *
 * CSR storage of the non-zero blocks follows "Block Sparse Attention Techniques",
 * section 3.2, "Implementation with Sparse Matrix Formats".
 *
 *   layout  host, int32 [H, nb, nb], values 0/1, row-major; read only, not retained.
 *   H, nb   heads and blocks per side (both >= 1, nb < 2^15, H*nb*nb < 2^31).
 *   batch   batch size B the work list is built for (>= 1).
 *   order   BSA_ORDER_GLOBAL or BSA_ORDER_GROUPED.
 *   out     receives the new LUT (set to NULL on error).
 *
 * Contents (see bsa_lut_export): row_ptr int32[H*nb + 1] over rows r = h*nb + i,
 * col_idx int32[nnz] with the active j of each row ascending, and items
 * int32[B*H*nb][4] = {b, h, i, nnz of row (h,i)}, every (b,h,i) present once
 * (zero-count items included), sorted stably by the order's key.
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_LAYOUT_VALUE, BSA_ERR_UNSUPPORTED
 * (bad order), BSA_ERR_ALLOC.
 */
int bsa_build_lut(const int32_t* layout, int H, int nb, int batch, int order, bsa_lut** out);

/*
 * bsa_build_lut_rect -- bsa_build_lut for a rectangular layout int32 [H, nb, nbk]: nb
 * query blocks by nbk key blocks per head, as bsa_forward_ext takes when the query and
 * key block sizes differ or the lengths are not multiples of them (nb = ceil(Lq /
 * q_block), nbk = ceil(Lk / kv_block); the last block of a ragged sequence is clipped
 * at its end, as the mask builder of the "Block-Sparse Attention" page, section "Block
 * Structure", clips it).  Rows are the nb query blocks; col_idx holds key-block
 * indices in [0, nbk).  1 <= nb, nbk < 2^15.  Errors as bsa_build_lut.
 */
int bsa_build_lut_rect(const int32_t* layout, int H, int nb, int nbk, int batch, int order,
                       bsa_lut** out);

/* bsa_lut_kv_blocks -- key blocks per row (nbk) of a LUT; nb for a square one. */
int bsa_lut_kv_blocks(const bsa_lut* lut, int* nbk);

/*
 * bsa_lut_info -- sizes of a LUT.  Any output pointer may be NULL.
 * nnz_total = sum of the layout = length of col_idx; n_items = batch*H*nb.
 */
int bsa_lut_info(const bsa_lut* lut, int* H, int* nb, int* batch, int* nnz_total, int* n_items);

/*
 * bsa_lut_export -- copy the host CSR and work list into caller buffers of
 * H*nb+1, nnz_total and 4*n_items int32 (any may be NULL to skip it).
 */
int bsa_lut_export(const bsa_lut* lut, int32_t* row_ptr, int32_t* col_idx, int32_t* items);

/*
 * bsa_lut_schedule -- a per-CTA schedule the kernel runs for a grid of `grid` CTAs
 * (host only; needs no GPU).  Items are handed out one at a time, each to the CTA with
 * the least work so far (ties: lowest index), an item costing 4*nnz + 2; CTA c then runs
 * items[4*cta_start[c] .. 4*cta_start[c+1]) in the order it received them.  by_head = 0
 * hands them out in work-list order; nonzero, (batch, head) by (batch, head) (ascending),
 * in work-list order within each pair.  items: 4*n_items int32, cta_start: grid+1 int32
 * (either may be NULL).  bsa_lut_upload uploads both schedules for grid = min(n_items,
 * SM count); bsa_forward runs the (batch, head) one when the K and V of the call
 * (B*H*L*d*4 bytes) exceed the device's L2, so that the CTAs share a few pairs' K and V
 * at a time, and the other one otherwise (bsa_set_schedule overrides the choice).
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE (grid < 1 or grid > max(1, n_items)),
 * BSA_ERR_ALLOC.
 */
int bsa_lut_schedule(const bsa_lut* lut, int grid, int by_head, int32_t* items,
                     int32_t* cta_start);

/*
 * bsa_lut_upload -- allocate device copies of col_idx and the work list (plus a
 * device status word) on the current device and copy them there on
 * `stream`, then synchronize `stream`.  The device work lists are the two schedules of
 * bsa_lut_schedule for a grid of min(n_items, SM count of the device); the exported
 * list keeps its own order.  Call once before the first bsa_forward;
 * calling again re-uploads to the now-current device.  Errors: BSA_ERR_NULL,
 * BSA_ERR_ALLOC, BSA_ERR_CUDA.
 */
int bsa_lut_upload(bsa_lut* lut, void* stream);

/* bsa_lut_free -- release host and device memory of a LUT (NULL is a no-op).  The
 * caller makes sure no forward that uses it is still running. */
void bsa_lut_free(bsa_lut* lut);

/*
 * bsa_forward -- O and lse of block-sparse attention (the operation above).
 *
 *   q, k, v  device, bf16 [B,H,L,d], 16-byte aligned, read only.
 *   lut      uploaded LUT built for this (H, nb = L/block, batch = B).
 *   out      device, bf16 [B,H,L,d], 16-byte aligned; every element written.
 *   lse      device, fp32 [B,H,L], 16-byte aligned; natural-log log-sum-exp of the
 *            scaled scores, -inf on rows without an active key.
 *   scale    multiplies q.k before the softmax (any finite value, 0 included).
 *   block    64 or 128; d (head dim) 64 or 128.  L must equal nb * block.
 *   causal_diag  nonzero: inside diagonal blocks (row block == column block) key
 *            c > query r is masked; other active blocks are not masked.
 *   stream   cudaStream_t (void*) the kernel is queued on.
 *
 * Asynchronous: returns after queuing one kernel launch; allocates nothing and
 * does not synchronize.  One forward per LUT may run at a time (the device status
 * word is per LUT).  Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_ALIGN,
 * BSA_ERR_UNSUPPORTED, BSA_ERR_STATE, BSA_ERR_CUDA (launch failure).
 */
int bsa_forward(const void* q, const void* k, const void* v, const bsa_lut* lut, void* out,
                float* lse, int B, int H, int L, int d, float scale, int block, int causal_diag,
                void* stream);

/*
 * Per-element predicates and extra terms of bsa_forward_ext.  They follow the argument
 * list of ejkernel's blocksparse_attention ("sliding_window" as a (left, right) pair,
 * "logits_soft_cap", "softmax_aux" for attention sinks, query / key-value segment ids)
 * and the sink term of the DeepSeek-V4.1 sparse_attn kernel ("Sparse attention /
 * Weighted row sum").  A zeroed struct with both window sides set to -1 (or a NULL
 * pointer) means none of them.
 */
typedef struct bsa_ext_args {
  int window_left;               /* key c masked when c < r - window_left; < 0: no bound  */
  int window_right;              /* key c masked when c > r + window_right; < 0: no bound */
  float softcap;                 /* > 0: each scaled score s becomes softcap*tanh(s /
                                    softcap); 0: off                                       */
  const float* sinks;            /* device fp32 [H] or NULL: head h's sink logit t_h adds
                                    exp(t_h) to the softmax normaliser (no value row), so
                                    lse includes it and an empty row gets lse = t_h        */
  const int32_t* q_segment_ids;  /* device int32 [B, Lq] or NULL                          */
  const int32_t* kv_segment_ids; /* device int32 [B, Lk] or NULL (both or neither): key c
                                    is masked for query r when their ids differ            */
} bsa_ext_args;

/*
 * bsa_forward_ext -- bsa_forward with ragged lengths, different query and key block
 * sizes, and the predicates of bsa_ext_args.  For batch b, head h, query row r in
 * [0, Lq):
 *
 *   A(r) = { c in [0, Lk) : layout[h][r/q_block][c/kv_block] == 1, not masked by the
 *            window or the segment ids, and not (causal_diag && c > r && key block
 *            c/kv_block overlaps the rows of query block r/q_block) }
 *   s_c  = scale * <q[b,h,r,:], k[b,h,c,:]>, then softcap*tanh(s_c/softcap) if set
 *   lse[r] = ln( sum_{c in A(r)} exp(s_c) + exp(sinks[h]) if sinks )  (-inf if empty)
 *   O[r,:] = sum_{c in A(r)} exp(s_c - lse[r]) v[b,h,c,:]            (0 if A(r) empty)
 *
 * The diagonal mask reads "diagonal block" as every key block whose key range overlaps
 * the query block's rows (the block j == i when the sizes are equal).
 *
 *   q, out   device bf16 [B,H,Lq,d];  k, v  device bf16 [B,H,Lk,d]  (16-byte aligned).
 *   lse      device fp32 [B,H,Lq].
 *   lut      uploaded LUT of layout [H, ceil(Lq/q_block), ceil(Lk/kv_block)]
 *            (bsa_build_lut_rect; bsa_build_lut when both are nb).
 *   q_block, kv_block  64 or 128 each;  d 64 or 128.
 *   ext      predicates (NULL: none); its device arrays 4-byte aligned.
 *
 * With equal blocks, Lq == Lk a multiple of the block and no predicate this is exactly
 * bsa_forward (the same kernel).  Asynchronous, no allocation, one kernel launch.
 * Errors: BSA_ERR_NULL (also: exactly one segment array given), BSA_ERR_SHAPE,
 * BSA_ERR_ALIGN, BSA_ERR_UNSUPPORTED (block or head dim, non-finite scale, negative or
 * non-finite softcap), BSA_ERR_STATE, BSA_ERR_CUDA.
 */
int bsa_forward_ext(const void* q, const void* k, const void* v, const bsa_lut* lut, void* out,
                    float* lse, int B, int H, int Lq, int Lk, int d, float scale, int q_block,
                    int kv_block, int causal_diag, const bsa_ext_args* ext, void* stream);

/*
 * bsa_lut_export_csc -- the column view the backward walks (square layouts only):
 * col_ptr int32[H*nb + 1] over columns h*nb + j, row_idx int32[nnz] with the active query
 * blocks i of each column ascending, items int32[B*H*nb][4] = {b, h, j, count}, sorted
 * stably by (-count, b, h, j).  Any pointer may be NULL.  Errors: BSA_ERR_NULL,
 * BSA_ERR_SHAPE (rectangular layout).
 */
int bsa_lut_export_csc(const bsa_lut* lut, int32_t* col_ptr, int32_t* row_idx, int32_t* items);

/*
 * bsa_backward -- gradients of the forward (the operation above) with respect to q, k
 * and v, given the forward's out and lse and the upstream gradient dout.  Gradients flow
 * through the active blocks only ("Block Sparse Attention Techniques", section 2,
 * "Gradient Propagation in Block Sparse Attention"); with P the masked softmax:
 *
 *   delta[r] = sum_x dout[r,x] out[r,x]
 *   dS = P * (dout V^T - delta),   dq = scale dS K,   dk = scale dS^T Q,   dv = P^T dout
 *
 * P is recomputed from q, k and lse (P = exp(scale q.k - lse) on the active entries).
 *
 *   q, k, v, out, dout   device bf16 [B,H,L,d] (out, lse: the bsa_forward results for
 *                        these q, k, v and arguments).
 *   lse                  device fp32 [B,H,L].
 *   lut                  uploaded LUT of a square layout (bsa_build_lut).
 *   dq, dk, dv           device bf16 [B,H,L,d]; every element written (rows and keys with
 *                        no active entry get 0).
 *   delta                device fp32 [B,H,L], caller-owned workspace; overwritten.
 *   B .. causal_diag     as bsa_forward.
 *
 * All pointers 16-byte aligned.  Asynchronous: queues three kernels on `stream` (delta,
 * then dq over the layout's rows, then dk and dv over its columns); allocates nothing.
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_ALIGN, BSA_ERR_UNSUPPORTED, BSA_ERR_STATE,
 * BSA_ERR_CUDA.  Device timeouts are reported by bsa_device_status as for the forward.
 */
int bsa_backward(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout, const bsa_lut* lut, void* dq, void* dk, void* dv, float* delta,
                 int B, int H, int L, int d, float scale, int block, int causal_diag,
                 void* stream);

/*
 * bsa_topk_forward -- top-k token-gather attention with an attention sink, the second
 * sparsity granularity of the pages: the sparse_attn kernel of the DeepSeek-V4.1
 * "Sparse attention / Weighted row sum" page.  Every query position lists K rows of its
 * batch's key-value matrix; a row is both key and value and is shared by all H heads;
 * each head's sink logit adds one term to the softmax denominator.  For batch b,
 * position m, head h, with J the list entries whose index lies in [0, N) (-1 marks an
 * unused slot; any other index outside [0, N) is treated the same; a row listed twice
 * counts twice):
 *
 *   s_j = scale * <q[b,m,h,:], kv[b, idx[b,m,j], :]>
 *   Z   = sum_{j in J} exp(s_j) + exp(sink[h])
 *   out[b,m,h,:] = sum_{j in J} exp(s_j) / Z * kv[b, idx[b,m,j], :],   lse[b,m,h] = ln Z
 *
 * (a position with no valid entry gets out = 0 and lse = sink[h], the page's all-zero
 * convention).
 *
 *   q       device bf16 [B, M, H, D];  kv  device bf16 [B, N, D];  out  bf16 [B, M, H, D].
 *   sink    device fp32 [H];  idx  device int32 [B, M, K];  lse  device fp32 [B, M, H].
 *   status  device int32, caller-owned, zero before the call: a bounded wait that gives
 *           up in the kernel writes 0x10000 | site there (and the outputs are undefined).
 *   H must be 64 and D 512 (the page's shape); K >= 1 (the list runs in steps of 128).
 *
 * All pointers 16-byte aligned (status 4-byte).  Asynchronous, one kernel launch,
 * allocates nothing.  Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_ALIGN,
 * BSA_ERR_UNSUPPORTED (H, D, or non-finite scale), BSA_ERR_CUDA.
 */
int bsa_topk_forward(const void* q, const void* kv, const float* sink, const int32_t* idx,
                     void* out, float* lse, int32_t* status, int B, int M, int N, int H, int D,
                     int K, float scale, void* stream);

/*
 * bsa_forward_noalloc -- the same forward as bsa_forward for callers that cannot
 * allocate device memory.  The pages have no counterpart of this call.
 *
 * Some callers may not call cudaMalloc at all: code running inside a host callback
 * or a plugin hook where allocating could deadlock or is forbidden, code under a
 * memory manager that owns the whole device heap, or a process that must not grow
 * its device footprint after start-up.  They build the LUT on the host with
 * bsa_build_lut (host memory only; no bsa_lut_upload needed) and pass their own q,
 * k, v, out and lse buffers, exactly as for bsa_forward.  The LUT's device copy and
 * the device status word go into one fixed 4 MiB array that is part of the library
 * image (every GPU that loads the library holds it until the process exits); this
 * call calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments q ... stream: as bsa_forward (`lut` need not be uploaded).
 *   sync_status  0: asynchronous.  A bounded wait that gives up in the kernel is then
 *                reported to no one (the status word lives in the shared array, not in
 *                the LUT, so bsa_device_status cannot see it, and the next call clears
 *                it), and the outputs of that call are undefined.  Nonzero: the call
 *                synchronizes `stream` after the kernel and returns
 *                BSA_ERR_DEVICE_TIMEOUT if a bounded wait in the kernel gave up.
 *
 * Limit: 4 + 4*n_items + 1024 + nnz int32 words (each part rounded up to 4 words) must
 * fit in 1 Mi words; larger LUTs return BSA_ERR_TOO_LARGE before
 * any device work.  The per-CTA schedule comes from bsa_lut_upload when the LUT was
 * uploaded on this device; otherwise the call builds it in host memory.  Each call
 * looks up the array's device address (cudaGetSymbolAddress, which allocates nothing)
 * on the current device.  All calls share the array and each call overwrites it: calls
 * whose kernels overlap on the GPU (other streams, other host threads) race, so
 * serialize them on one stream.  Other errors: as bsa_forward.
 */
int bsa_forward_noalloc(const void* q, const void* k, const void* v, const bsa_lut* lut,
                        void* out, float* lse, int B, int H, int L, int d, float scale, int block,
                        int causal_diag, void* stream, int sync_status);

/*
 * bsa_device_status -- synchronize `stream`, read and clear the LUT's device status
 * word.  Returns BSA_OK, or BSA_ERR_DEVICE_TIMEOUT if a bounded wait inside a
 * kernel gave up since the last check (the kernel then skipped the remaining work
 * and its outputs are undefined), or BSA_ERR_CUDA.  `detail` (may be NULL)
 * receives the raw status word: wait-site id in the low 16 bits.
 */
int bsa_device_status(const bsa_lut* lut, void* stream, int32_t* detail);

/* Device schedule policies (bsa_set_schedule). */
enum {
  BSA_SCHEDULE_AUTO = 0,    /* (batch, head) schedule when the call's K and V exceed L2 */
  BSA_SCHEDULE_LIST = 1,    /* items handed out in work-list order */
  BSA_SCHEDULE_BY_HEAD = 2  /* items handed out (batch, head) by (batch, head) */
};

/*
 * bsa_set_schedule -- which of the two uploaded per-CTA schedules (bsa_lut_schedule)
 * forwards queued after this call run: BSA_SCHEDULE_AUTO (default) picks the (batch,
 * head) one when B*H*L*d*4 bytes of K and V exceed the device L2.  The schedule changes
 * only the order in which CTAs take items; results are bitwise the same.  Errors:
 * BSA_ERR_NULL, BSA_ERR_UNSUPPORTED (unknown policy).
 */
int bsa_set_schedule(bsa_lut* lut, int policy);

/*
 * bsa_set_wait_limit -- per-wait time limit, in nanoseconds, that kernels queued
 * after this call use for every barrier wait (default 1e10 = 10 s; 0 restores the
 * default).  A wait that runs out records BSA_ERR_DEVICE_TIMEOUT in the status word
 * and the kernel returns instead of hanging.
 */
int bsa_set_wait_limit(bsa_lut* lut, uint64_t ns);

/*
 * bsa_debug_expire_wait -- test knob for the device-side failure path.  Kernels
 * queued after this call treat every wait at wait site `site` as a wait that ran
 * out: the waiting role records BSA_ERR_DEVICE_TIMEOUT with that site id in the
 * status word, raises its CTA's abort flag, and every role of the CTA leaves its
 * loop, waits for its own copies and MMAs in flight, frees TMEM and returns -- the
 * same path a real timeout takes, without waiting for one.  The outputs of such a
 * forward are undefined; bsa_device_status reports it.  site 0 turns the knob off.
 * Site ids (low 16 bits of the status word): 1 producer, K slot free; 2 producer, V
 * slot free; 6 MMA issuers, K or V landed; 7 PV issuer, P written; 8 S issuer, S
 * buffer free; 9 softmax, S computed; 10 PV issuer, the previous item's O read out;
 * 11 softmax, O free for a rescale; 12 the item's last PV done (forward: epilogue at
 * block 128, softmax at block 64; backward: softmax); 13 epilogue, the rows'
 * statistics written; 14 softmax, the previous rows' statistics read (sites 10, 13
 * and 14: the forward at block 128 only).  The backward's kernels use the same ids for
 * their counterparts: 1 and 2 the producer's item and step slots free, 6 tiles landed,
 * 7 the elementwise warps' operands written (or the accumulators read out), 8 a TMEM
 * region free, 9 the elementwise warps waiting for a product, 12 an item's last
 * products done.  Errors: BSA_ERR_NULL, BSA_ERR_UNSUPPORTED (site outside [0, 65535]).
 */
int bsa_debug_expire_wait(bsa_lut* lut, int site);

/*
 * bsa_wait_selftest -- launch a one-CTA kernel that waits on a shared-memory
 * barrier nothing ever signals, bounded by `limit_ns`, and report what the
 * kernel recorded: BSA_ERR_DEVICE_TIMEOUT when the bounded wait fired as
 * designed (the expected result), BSA_OK if it did not.  Synchronizes `stream`.
 * This exercises the timeout path of every wait in the forward kernel without a
 * fault or a hang.
 */
int bsa_wait_selftest(uint64_t limit_ns, void* stream);

/* bsa_status_string -- static English text for a status code. */
const char* bsa_status_string(int status);

/* bsa_version -- library version string ("major.minor.patch"). */
const char* bsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
