// bsa_fwd_kernel.cuh -- persistent block-sparse attention forward kernel for sm_103a.
//
// Method: for each work item (batch b, head h, query block i) the kernel streams the
// key/value blocks listed in the CSR row (h, i) and runs the online softmax over them
// (running max and running sum, the accumulator rescaled when the max grows), as the
// sparse_attn kernel of the DeepSeek-V4.1 "Sparse attention / Weighted row sum" page
// does for gathered rows; the block layout and its CSR follow "Block Sparse Attention
// Techniques" (sections 3.2 and 4) and the DeepSpeed sparse-attention utils page.
// Scores outside the active blocks are never formed: their exp() would be 0.
//
// Keys are consumed in steps of 128 rows: one block when b = 128, the next two active
// blocks of the row when b = 64 (the last step of a row with an odd count holds one).
//
// GB300 mapping.  One CTA per SM, 384 threads, two work items in flight per CTA
// ("slots" 0 and 1, each with its own Q tile, TMEM S/P and O, and softmax warpgroup),
// so the tensor core runs one slot's MMAs while the other slot's softmax runs:
//   warp 0        TMA producer: Q tile of each item into its slot's Q buffer (and an
//                 L2 prefetch of the slot's next Q), K and V step tiles into one ring
//                 of kRing slots, in exactly the order the MMA warp consumes them.
//   warp 1        tcgen05 issuer (one thread) and TMEM owner.  Per slot, alternating:
//                   O += P V   (M = b, N = d, K = keys; A = P read from TMEM)
//                   S = Q K^T  (M = b, N = keys, K = d; into the slot's TMEM S, which
//                              P overwrites in place once the softmax has read S)
//   warps 4..7    softmax warpgroup of slot 0; warps 8..11 that of slot 1: TMEM ->
//                 registers, causal mask on diagonal blocks, base-2 online softmax
//                 (exp2(s*c - m) with c = scale*log2(e) in one FFMA, tree reductions),
//                 lazy rescale (the running max moves only when it grows by more than
//                 2^8; O is rescaled in TMEM, which is safe because S(j) completing
//                 implies PV(j-1) completed), P -> TMEM as bf16, and the epilogue
//                 (O / l -> bf16, lse = ln 2 * (m + log2 l)); an item with no active
//                 block writes O = 0 and lse = -inf.
//   warps 2..3    idle.
// b = 128 uses M = 128 MMAs (row r of S/P/O in TMEM lane r, one thread per row);
// b = 64 uses M = 64 MMAs, whose rows sit in lanes 0-15 of each 32-lane quadrant:
// lanes t and t+16 of a warp share a row, each holding one of the step's two key
// blocks (16x32bx2 TMEM loads and stores).
//
// Every barrier wait is bounded (WaitCtl): a wait that runs out records a timeout in
// the status word, and all roles leave their loops, drain in-flight copies and MMAs,
// free TMEM and return.
#pragma once

#include <cuda_bf16.h>

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

template <int BLK, int D>
struct FwdCfg {
  static_assert(BLK == 64 || BLK == 128, "block must be 64 or 128");
  static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
  static constexpr int kThreads = 384;
  static constexpr int kKR = 128;                 // key rows per step
  static constexpr int kG = kKR / BLK;            // blocks per step (1 or 2)
  static constexpr int kQTile = BLK * D * 2;      // bytes of one Q tile
  static constexpr int kKVTile = kKR * D * 2;     // bytes of one K or V step tile
  static constexpr int kQRegion = BLK * 128;      // one 64-column swizzled box of BLK rows
  static constexpr int kKVRegion = kKR * 128;     // one 64-column box of a step tile
  static constexpr int kSlotCols = 256;           // TMEM columns per slot: S/P then O
  static constexpr int kOCol = 128;               // O offset inside a slot
  static constexpr int kTmemCols = 512;
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + 2 * kQTile;
  static constexpr int kBarBytes = 512;
  static constexpr int kRingFit = (232448 - 1024 - kBarBytes - kOffRing) / kKVTile;
  static constexpr int kRing = kRingFit < 8 ? kRingFit : 8;
  static constexpr int kOffBar = kOffRing + kRing * kKVTile;
  // barrier indices
  static constexpr int kBarQF = 0;                // [2] per slot
  static constexpr int kBarQE = 2;                // [2]
  static constexpr int kBarSF = 4;                // [2]
  static constexpr int kBarPF = 6;                // [2]
  static constexpr int kBarOF = 8;                // [2]
  static constexpr int kBarDrain = 10;
  static constexpr int kBarRF = 11;               // [kRing] ring full
  static constexpr int kBarRE = kBarRF + kRing;   // [kRing] ring empty
  static constexpr int kNumBars = kBarRE + kRing;
  static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + align slack
  static_assert(kRing >= 4, "ring too small");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // instruction descriptors: S over a full step (N = 128) or a single 64-key block
  static constexpr uint32_t kIdescS = idesc_bf16_f32(BLK, kKR, false, false);
  static constexpr uint32_t kIdescS1 = idesc_bf16_f32(BLK, BLK, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BLK, D, false, true);
};

// Bounded wait that ignores the abort flag and never records a status: used only
// to drain work already in flight before the CTA releases its resources.  Its limit
// is fixed and independent of the (possibly tiny) per-wait limit of the main loop.
constexpr uint64_t kDrainLimitNs = 4000000000ull;

__device__ __forceinline__ void mbar_drain_wait(uint32_t bar, uint32_t parity,
                                                uint64_t limit_ns = kDrainLimitNs) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Blocks in step s of a row with nnz active blocks.
template <int G>
__device__ __forceinline__ int step_blocks(int nnz, int s) {
  const int rem = nnz - s * G;
  return rem < G ? rem : G;
}

// Slot X of a CTA owns positions k = X, X+2, X+4, ... of the CTA's round-robin share
// of the work list (item blockIdx.x + k * gridDim.x).  Advances k to the next
// non-empty item at or after k; false when the share is exhausted.
__device__ __forceinline__ bool seek_item(const FwdParams& p, int& k, int4& item) {
  for (;; k += 2) {
    const int t = blockIdx.x + k * gridDim.x;
    if (t >= p.n_items) return false;
    item = p.items[t];
    if (item.w > 0) return true;
  }
}

// The consumption schedule shared by the producer and the MMA warp.  Slots take
// turns; a turn of slot X is: PV of X's pending step (if any), then S of X's next
// step (the next item's step 0 when the current item is exhausted).  Each action
// uses one ring tile (V for PV, K for S), so both warps see the same ring order.
// on_pv(X, item, step, nblk, last_step) / on_s(X, item, step, nblk, k) return false
// to stop early.
template <int G, class OnPV, class OnS>
__device__ __forceinline__ void walk_schedule(const FwdParams& p, OnPV&& on_pv, OnS&& on_s) {
  int k[2] = {0, 1};
  int4 it[2];
  int nsteps[2], s_next[2] = {0, 0}, pend[2] = {-1, -1};
  bool done[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    done[x] = !seek_item(p, k[x], it[x]);
    nsteps[x] = done[x] ? 0 : (it[x].w + G - 1) / G;
  }
  while (!(done[0] && done[1])) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (done[x]) continue;
      if (pend[x] >= 0) {
        if (!on_pv(x, it[x], pend[x], step_blocks<G>(it[x].w, pend[x]), pend[x] == nsteps[x] - 1))
          return;
        pend[x] = -1;
      }
      if (s_next[x] >= nsteps[x]) {
        k[x] += 2;
        if (!seek_item(p, k[x], it[x])) {
          done[x] = true;
          continue;
        }
        nsteps[x] = (it[x].w + G - 1) / G;
        s_next[x] = 0;
      }
      const int s = s_next[x]++;
      if (!on_s(x, it[x], s, step_blocks<G>(it[x].w, s), k[x])) return;
      pend[x] = s;
    }
  }
}

// ----------------------------------------------------------------- producer

template <int BLK, int D>
__device__ __forceinline__ void fwd_producer(const FwdParams& p, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             uint32_t sbase, const WaitCtl& ctl) {
  using C = FwdCfg<BLK, D>;
  constexpr int R = C::kRing;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  int qc[2] = {0, 0};
  int rc = 0;

  // Loads the K or V rows of one step into the next ring tile.
  auto load_step = [&](const CUtensorMap* tm, const int4& it, int step, int nblk) -> bool {
    const int r = rc % R;
    if (!mbar_wait(bar(C::kBarRE + r), ((rc / R) & 1) ^ 1, ctl, kSiteProdRingEmpty)) return false;
    const int rowbase = (it.x * p.H + it.y) * p.L;
    const int* cols = p.col_idx + p.row_ptr[it.y * p.nb + it.z] + step * G;
    mbar_arrive_expect_tx(bar(C::kBarRF + r), nblk * BLK * D * 2);
    for (int g = 0; g < nblk; ++g) {
      const int krow = rowbase + cols[g] * BLK;
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sbase + C::kOffRing + r * C::kKVTile + c * C::kKVRegion + g * BLK * 128, tm,
                    bar(C::kBarRF + r), c * 64, krow);
    }
    ++rc;
    return true;
  };

  walk_schedule<G>(
      p,
      [&](int x, const int4& it, int step, int nblk, bool) { return load_step(tm_v, it, step, nblk); },
      [&](int x, const int4& it, int step, int nblk, int k) {
        if (step == 0) {
          if (!mbar_wait(bar(C::kBarQE + x), (qc[x] & 1) ^ 1, ctl, kSiteProdQEmpty)) return false;
          mbar_arrive_expect_tx(bar(C::kBarQF + x), C::kQTile);
          const int qrow = (it.x * p.H + it.y) * p.L + it.z * BLK;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sbase + C::kOffQ + x * C::kQTile + c * C::kQRegion, tm_q,
                        bar(C::kBarQF + x), c * 64, qrow);
          ++qc[x];
          // Warm L2 with the slot's next Q tile.
          int k2 = k + 2;
          int4 nxt;
          if (seek_item(p, k2, nxt)) {
            const int nrow = (nxt.x * p.H + nxt.y) * p.L + nxt.z * BLK;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_2d(tm_q, c * 64, nrow);
          }
        }
        return load_step(tm_k, it, step, nblk);
      });

  // Wait until every copy this thread issued has landed (immediate on the normal path).
  for (int x = 0; x < 2; ++x)
    if (qc[x] > 0) mbar_drain_wait(bar(C::kBarQF + x), (qc[x] - 1) & 1);
  for (int r = 0; r < R; ++r)
    if (rc > r) {
      const int f = r + R * ((rc - 1 - r) / R);
      mbar_drain_wait(bar(C::kBarRF + r), (f / R) & 1);
    }
}

// --------------------------------------------------------------- MMA issuer

template <int BLK, int D>
__device__ __forceinline__ void fwd_mma(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                        const WaitCtl& ctl) {
  using C = FwdCfg<BLK, D>;
  constexpr int R = C::kRing;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  int qc[2] = {0, 0}, pc[2] = {0, 0};
  int rc = 0;
  // Descriptors are built once; per MMA only the low word (start address >> 4) moves.
  const uint64_t kdesc0 = sdesc_sw128(sbase + C::kOffRing, 16, 1024);          // K-major
  const uint64_t vdesc0 = sdesc_sw128(sbase + C::kOffRing, C::kKVRegion, 1024);  // MN-major
  const uint32_t desc_hi = static_cast<uint32_t>(kdesc0 >> 32);  // same for Q, K and V
  const uint32_t k_lo0 = static_cast<uint32_t>(kdesc0);
  const uint32_t v_lo0 = static_cast<uint32_t>(vdesc0);
  const uint32_t q_lo0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffQ, 16, 1024));
  constexpr uint32_t kTileStep = C::kKVTile >> 4;  // descriptor units per ring tile

  walk_schedule<G>(
      p,
      // O_x (+)= P_x V : P from the slot's TMEM S columns, V from the ring.
      [&](int x, const int4&, int step, int nblk, bool last) -> bool {
        if (!mbar_wait(bar(C::kBarPF + x), pc[x] & 1, ctl, kSiteMmaPFull)) return false;
        ++pc[x];
        const int r = rc % R;
        if (!mbar_wait(bar(C::kBarRF + r), (rc / R) & 1, ctl, kSiteMmaRingFull)) return false;
        tc_fence_after();
        const uint32_t ts = tmem + x * C::kSlotCols;
        const uint32_t vlo = v_lo0 + r * kTileStep;
        tc_mma_ts_lh(ts + C::kOCol, ts, vlo, desc_hi, C::kIdescPV, step > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < C::kKR / 16; ++kk) {
          if (kk < nblk * BLK / 16)
            tc_mma_ts_lh(ts + C::kOCol, ts + kk * 8, vlo + kk * ((16 * 128) >> 4), desc_hi,
                         C::kIdescPV, 1u);
        }
        tc_commit(bar(C::kBarRE + r));
        if (last) tc_commit(bar(C::kBarOF + x));
        ++rc;
        return true;
      },
      // S_x = Q_x K^T into the slot's TMEM S columns.
      [&](int x, const int4& it, int step, int nblk, int) -> bool {
        if (step == 0) {
          if (!mbar_wait(bar(C::kBarQF + x), qc[x] & 1, ctl, kSiteMmaQFull)) return false;
          ++qc[x];
        }
        const int r = rc % R;
        if (!mbar_wait(bar(C::kBarRF + r), (rc / R) & 1, ctl, kSiteMmaRingFull)) return false;
        tc_fence_after();
        const uint32_t qlo = q_lo0 + x * (C::kQTile >> 4);
        const uint32_t klo = k_lo0 + r * kTileStep;
        const uint32_t idesc = (nblk == G) ? C::kIdescS : C::kIdescS1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss_lh(tmem + x * C::kSlotCols,
                       qlo + (((kk >> 2) * C::kQRegion + (kk & 3) * 32) >> 4), desc_hi,
                       klo + (((kk >> 2) * C::kKVRegion + (kk & 3) * 32) >> 4), desc_hi, idesc,
                       kk > 0 ? 1u : 0u);
        tc_commit(bar(C::kBarRE + r));
        tc_commit(bar(C::kBarSF + x));
        if (step == (it.w + G - 1) / G - 1) tc_commit(bar(C::kBarQE + x));
        ++rc;
        return true;
      });

  // Let every MMA issued so far finish before TMEM is released.
  tc_commit(bar(C::kBarDrain));
  mbar_drain_wait(bar(C::kBarDrain), 0);
}

// ------------------------------------------------------------ softmax group

// Loads this thread's NC score columns of the slot's S into x[].
template <int BLK, int NC>
__device__ __forceinline__ void load_s(uint32_t ts, float (&x)[NC]) {
  if constexpr (BLK == 128) {
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld_32x32b_x32(ts + 0, r0);
    tmem_ld_32x32b_x32(ts + 32, r1);
    tmem_ld_32x32b_x32(ts + 64, r2);
    tmem_ld_32x32b_x32(ts + 96, r3);
    tmem_ld_wait(r0);
    tmem_ld_wait(r1);
    tmem_ld_wait(r2);
    tmem_ld_wait(r3);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      x[i] = __uint_as_float(r0[i]);
      x[32 + i] = __uint_as_float(r1[i]);
      x[64 + i] = __uint_as_float(r2[i]);
      x[96 + i] = __uint_as_float(r3[i]);
    }
  } else {
    // lanes 0-15 get columns [0, 64) of their row, lanes 16-31 columns [64, 128)
    uint32_t r0[32], r1[32];
    tmem_ld_16x32bx2_x32<64>(ts + 0, r0);
    tmem_ld_16x32bx2_x32<64>(ts + 32, r1);
    tmem_ld_wait(r0);
    tmem_ld_wait(r1);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      x[i] = __uint_as_float(r0[i]);
      x[32 + i] = __uint_as_float(r1[i]);
    }
  }
}

template <int BLK, int D>
__device__ __forceinline__ void fwd_softmax(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                            int slot, const WaitCtl& ctl) {
  using C = FwdCfg<BLK, D>;
  constexpr int G = C::kG;
  constexpr int NC = (BLK == 128) ? 128 : 64;   // S columns held per thread
  constexpr int OC = (BLK == 128) ? D : D / 2;  // O columns held per thread
  constexpr int NA = 8;                         // independent reduction chains
  constexpr float kLn2 = 0.6931471805599453f;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int wq = (threadIdx.x >> 5) & 3;  // TMEM lane quadrant of this warp
  const int lane = threadIdx.x & 31;
  const int row = (BLK == 128) ? (wq * 32 + lane) : (wq * 16 + (lane & 15));
  const int half = (BLK == 128) ? 0 : (lane >> 4);  // which block of the step (b = 64)
  const uint32_t ts = tmem + (static_cast<uint32_t>(wq * 32) << 16) + slot * C::kSlotCols;
  const uint32_t to = ts + C::kOCol;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  // scale > 0: the row max of the raw scores gives the max of the scaled ones and the
  // exponent is one FFMA.  Otherwise the scores are scaled first (c = 1 afterwards).
  const bool pos_scale = p.scale_log2 > 0.f;
  const float cs = pos_scale ? p.scale_log2 : 1.f;
  int sc = 0, oc = 0;
  bool ok = true;

  for (int k = slot;; k += 2) {
    const int t = blockIdx.x + k * gridDim.x;
    if (t >= p.n_items || !ok) break;
    const int4 it = p.items[t];
    const int nnz = it.w;
    const int qrow = (it.x * p.H + it.y) * p.L + it.z * BLK + row;  // global query row
    uint4* orow = reinterpret_cast<uint4*>(outp + static_cast<size_t>(qrow) * D + half * OC);
    if (nnz == 0) {
#pragma unroll
      for (int c = 0; c < OC / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      if (half == 0) p.lse[qrow] = -INFINITY;
      continue;
    }
    // Position of the diagonal block inside the row (-1: none, or no causal mask).
    const int dpos = p.causal_diag ? p.diag_pos[it.y * p.nb + it.z] : -1;
    const int nsteps = (nnz + G - 1) / G;
    float m_used = -INFINITY;
    float l = 0.f;
    for (int s = 0; s < nsteps; ++s) {
      const int nblk = step_blocks<G>(nnz, s);
      const bool valid = half < nblk;
      const bool diag = valid && (s * G + half == dpos);
      ok = mbar_wait(bar(C::kBarSF + slot), sc & 1, ctl, kSiteSoftSFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++sc;
      tc_fence_after();
      float x[NC];
      load_s<BLK, NC>(ts, x);

      if (!pos_scale) {
#pragma unroll
        for (int c = 0; c < NC; ++c) x[c] *= p.scale_log2;
      }
      if (!valid) {
#pragma unroll
        for (int c = 0; c < NC; ++c) x[c] = -INFINITY;
      } else if (diag) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (c > row) x[c] = -INFINITY;
      }
      // Row max: NA chains of three-input maxima over columns c = a (mod NA).
      float mr[NA];
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        mr[a] = x[a];
#pragma unroll
        for (int c = a + NA; c < NC; c += 2 * NA)
          mr[a] = (c + NA < NC) ? fmax3(mr[a], x[c], x[c + NA]) : fmaxf(mr[a], x[c]);
      }
#pragma unroll
      for (int w = NA / 2; w >= 1; w /= 2)
#pragma unroll
        for (int a = 0; a < w; ++a) mr[a] = fmaxf(mr[a], mr[a + w]);
      float mx = mr[0] * cs;  // -inf stays -inf (cs > 0)
      if constexpr (BLK == 64) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      float alpha = 1.f;
      const float m_new = fmaxf(m_used, mx);
      if (s == 0) {
        m_used = m_new;
      } else if (m_new > m_used + 8.f) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;

      // exp2(x*c - m) on pairs (packed f32x2 FFMA, MUFU ex2).  Row sums in NS packed
      // accumulators, P (bf16 pairs) -> TMEM over the S columns, 32 columns at a time.
      constexpr int NS = 4;
      uint64_t sr2[NS];
#pragma unroll
      for (int a = 0; a < NS; ++a) sr2[a] = 0ull;
      const uint64_t c2 = f2_pack(cs, cs), m2 = f2_pack(neg_m, neg_m);
#pragma unroll
      for (int cc = 0; cc < NC / 64; ++cc) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint64_t y = f2_fma(f2_pack(x[cc * 64 + 2 * i], x[cc * 64 + 2 * i + 1]), c2, m2);
          const uint64_t e = f2_pack(ex2_approx(f2_lo(y)), ex2_approx(f2_hi(y)));
          sr2[i % NS] = f2_add(sr2[i % NS], e);
          pk[i] = pack_bf16x2(f2_lo(e), f2_hi(e));
        }
        if constexpr (BLK == 128) {
          tmem_st_32x32b_x32(ts + cc * 32, pk);
        } else {
          tmem_st_16x32bx2_x32<32>(ts, pk);
        }
      }
      sr2[0] = f2_add(f2_add(sr2[0], sr2[1]), f2_add(sr2[2], sr2[3]));
      float rs = f2_lo(sr2[0]) + f2_hi(sr2[0]);
      if constexpr (BLK == 64) rs += __shfl_xor_sync(0xffffffffu, rs, 16);
      l = l * alpha + rs;
      // O rescale: S(s) complete implies PV(s-1) complete; PV(s) waits for P below.
      if (s > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < OC / 32; ++c) {
          uint32_t r[32];
          if constexpr (BLK == 128) {
            tmem_ld_32x32b_x32(to + c * 32, r);
          } else {
            tmem_ld_16x32bx2_x32<D / 2>(to + c * 32, r);
          }
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          if constexpr (BLK == 128) {
            tmem_st_32x32b_x32(to + c * 32, r);
          } else {
            tmem_st_16x32bx2_x32<D / 2>(to + c * 32, r);
          }
        }
      }

      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPF + slot));
    }
    if (!ok) break;

    // epilogue: wait for the item's last PV, then O / l -> bf16 and lse.
    ok = mbar_wait(bar(C::kBarOF + slot), oc & 1, ctl, kSiteSoftOFull);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    ++oc;
    tc_fence_after();
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < OC / 32; ++c) {
      uint32_t r[32];
      if constexpr (BLK == 128) {
        tmem_ld_32x32b_x32(to + c * 32, r);
      } else {
        tmem_ld_16x32bx2_x32<D / 2>(to + c * 32, r);
      }
      tmem_ld_wait(r);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        orow[c * 4 + q] = make_uint4(
            pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv, __uint_as_float(r[8 * q + 1]) * inv),
            pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv),
            pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv),
            pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv));
      }
    }
    if (half == 0) p.lse[qrow] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
    tc_fence_before();
  }
}

// ------------------------------------------------------------------- kernel

template <int BLK, int D>
__global__ void __launch_bounds__(384, 1)
    bsa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<BLK, D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::kBarQF + x), 1);
      mbar_init(bar(C::kBarQE + x), 1);
      mbar_init(bar(C::kBarSF + x), 1);
      mbar_init(bar(C::kBarPF + x), 128);
      mbar_init(bar(C::kBarOF + x), 1);
    }
    mbar_init(bar(C::kBarDrain), 1);
    for (int r = 0; r < C::kRing; ++r) {
      mbar_init(bar(C::kBarRF + r), 1);
      mbar_init(bar(C::kBarRE + r), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) fwd_producer<BLK, D>(p, &tm_q, &tm_k, &tm_v, sbase, ctl);
  } else if (warp == 1) {
    if (lane == 0) fwd_mma<BLK, D>(p, sbase, tmem, ctl);
  } else if (warp >= 4) {
    fwd_softmax<BLK, D>(p, sbase, tmem, (warp - 4) >> 2, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BLK, int D>
cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, int grid, cudaStream_t stream) {
  using C = FwdCfg<BLK, D>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(bsa_fwd_kernel<BLK, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  bsa_fwd_kernel<BLK, D><<<grid, C::kThreads, C::kSmemBytes, stream>>>(q, k, v, p);
  return cudaGetLastError();
}

}  // namespace bsa
