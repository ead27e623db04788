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
// Query blocks have QB rows and key blocks KB keys (64 or 128 each; equal in the plain
// kernels).  Keys are consumed in steps of 128: one block when KB = 128, the next two
// active blocks of the row when KB = 64 (the last step of a row with an odd count holds
// one).
// A CTA walks its own range of the work list, regrouped per CTA on the host (each item to
// the least-loaded CTA), as one continuous stream of steps g = 0, 1, ...
//
// GB300 mapping.  One CTA per SM, warp-specialised:
//   warp 0      TMA producer.  For step t it loads K(t) (plus the Q tile when t opens an
//               item) on one barrier and V(t-2) on another; one 3-D copy per tile or
//               block brings all of its column halves.
//   warp 1      S issuer (one thread) and TMEM owner.  TMEM holds three S buffers and one
//               O accumulator.  Step t: S(t) = Q K(t)^T into S[t % 3] once K(t) landed
//               and PV(t-3), the last reader of that buffer, completed.
//   warp 2      PV issuer (one thread).  Step g: O += P(g) V(g), reading P from S[g % 3],
//               once the softmax wrote P(g) and V(g) landed (an item's first PV also
//               once the epilogue read the previous item's O out).
//               Two issuing threads keep the tensor pipe fed: it takes only a couple of
//               MMAs ahead of issue, so a lone issuer idles it at every barrier check;
//               the two streams order themselves through completion barriers only.
//   warp 3      idle (completes the first warpgroup).
//   softmax     warps 4-7 (and 8-11).
//               b = 128: two warpgroups; each warp owns 16 TMEM lanes (rows) of its
//               quadrant, lane t and t+16 holding the two 64-key halves of one row.
//               b = 64 (M = 64 MMAs, rows in lanes 0-15 of each quadrant): one warpgroup,
//               lane t and t+16 holding the step's two key blocks.  Per step: TMEM ->
//               registers (the S barrier of the next step is probed during this one),
//               causal mask on diagonal blocks, base-2 online softmax (row max
//               by three-input maxima and one shuffle, exp2(s*c - m) with the scale c =
//               scale*log2(e) folded into a packed f32x2 FFMA), lazy rescale (the
//               running max moves only when it grows by more than 2^8), P -> TMEM as bf16
//               pairs over the S columns.  When an item ends (b = 128), each row's
//               (m, l) goes to the epilogue through shared memory and the softmax moves
//               straight on; at b = 64 the softmax itself reads the item's O out at the
//               next item's first step and stores it.
//   epilogue    b = 128: the last warpgroup.  Per item: waits for the row statistics and
//               the item's last PV, reads O out of TMEM (32x32b: one row per thread),
//               releases the accumulator to the PV issuer, then stores O / l as bf16
//               (32-byte stores spaced apart) and lse = ln 2 * (m + log2 l).
//   An item with no active block gets O = 0 and lse = -inf (or the sink, EXT).
//   At b = 128 the 16 warps are launched at 128 registers each and re-split per
//   warpgroup with setmaxnreg (control 72, softmax 160, epilogue 120); b = 64 runs the
//   control warpgroup and one softmax warpgroup.
// Work-list records (which carry each item's block indices, CSR row start and diagonal
// position) are fetched two items ahead and column indices one step ahead of use, so no
// role waits on a global load in its steady state.
//
// The extended kernels (EXT) add per-element predicates on the same path, following the
// ejkernel blocksparse_attention arguments: a key past the end of a ragged sequence, a
// key outside the sliding window (left, right) of its query, a key of another segment
// (packed sequences), and the diagonal mask in every key block that overlaps the query
// block's rows, are all masked to -inf; the scores may be soft-capped
// (cap * tanh(s / cap)); and a per-head sink logit joins the softmax normaliser (the
// DeepSeek-V4.1 sparse_attn kernel's attn_sink) without a value row.  Rows past the end
// of a ragged query sequence are computed but not stored.
//
// Every barrier wait is bounded (WaitCtl): a wait that runs out records a timeout in
// the status word, and all roles leave their loops, drain in-flight copies and MMAs,
// free TMEM and return.
#pragma once

#include <cuda_bf16.h>

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

template <int QB, int KB, int D>
struct FwdCfg {
  static_assert(QB == 64 || QB == 128, "query block must be 64 or 128");
  static_assert(KB == 64 || KB == 128, "key block must be 64 or 128");
  static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
  static constexpr int kNumWG = (QB == 128) ? 2 : 1;  // softmax warpgroups
  // QB = 128: an epilogue warpgroup reads O out and stores it.  QB = 64 (one softmax
  // warpgroup, items of many steps): the softmax does it at the next item's first step.
  static constexpr bool kEpi = (QB == 128);
  static constexpr int kSoftWarp = 4;                  // first softmax warp
  static constexpr int kEpiWarp = 4 + 4 * kNumWG;      // first epilogue warp
  static constexpr int kThreads = 32 * (kEpiWarp + (kEpi ? 4 : 0));
  // The epilogue spaces its 32-byte stores of a row this far apart: a burst of an item's
  // 32 KB of stores stalls the softmax warps' next step by about a thousand cycles.
  static constexpr unsigned kStoreGapNs = 150;
  // Registers per thread after the split (b = 128): the launch gives every thread
  // 65536 / 512 = 128; the control and epilogue warpgroups hand 56 and 8 to each
  // softmax thread.
  static constexpr bool kSplitRegs = (QB == 128);
  static constexpr int kLaunchRegs = 128;
  static constexpr int kRegCtl = 72, kRegSoft = 160, kRegEpi = 120;
  static_assert(!kSplitRegs || kRegCtl + kNumWG * kRegSoft + kRegEpi == 4 * kLaunchRegs,
                "register split must add up to the launch's registers");
  static constexpr int kKR = 128;                 // key rows per step
  static constexpr int kG = kKR / KB;             // blocks per step (1 or 2)
  static constexpr int kNS = 3;                   // S buffers = stage barriers in flight
  static constexpr int kNK = 3;                   // K tiles in shared memory
  static constexpr int kQTileB = QB * D * 2;      // (bytes of one Q tile, for the budget below)
  static constexpr int kKVTileB = 128 * D * 2;
  // Two Q tiles, so the next item's Q loads while the current item's last S runs; V gets
  // three tiles when they fit beside them, else two (b = 128, d = 128).
  static constexpr int kNV = (2 * kQTileB + 6 * kKVTileB + 1216 <= 232448) ? 3 : 2;  // V tiles
  static constexpr int kQTile = QB * D * 2;       // bytes of one Q tile
  static constexpr int kKVTile = kKR * D * 2;     // bytes of one K or V step tile
  static constexpr int kNQ = 2;                   // Q tiles
  static constexpr int kQRegion = QB * 128;       // one 64-column swizzled box of QB rows
  // A K or V step tile holds its blocks one after another, each as d/64 swizzled
  // [KB][64] column halves (the layout one 3-D TMA copy of a block lands in).
  static constexpr int kHalfB = KB * 128;         // one 64-column half of one block
  static constexpr int kBlkB = KB * D * 2;        // one block
  static constexpr int kOCol = kNS * 128;         // O after the S buffers
  static constexpr int kTmemCols = 512;
  static_assert(kOCol + D <= kTmemCols, "TMEM budget");
  static constexpr int kOffQ = 0;                 // kNQ Q tiles
  static constexpr int kOffK = kOffQ + kNQ * kQTile;
  static constexpr int kOffV = kOffK + kNK * kKVTile;
  static constexpr int kOffBar = kOffV + kNV * kKVTile;
  // barrier indices
  static constexpr int kBarSF = 0;                // [3] S(g) computed
  static constexpr int kBarPVD = 3;               // [3] PV(g) complete
  static constexpr int kBarKF = 6;                // [3] K(t) (+Q) landed
  static constexpr int kBarVF = 9;                // [3] V(g) landed
  static constexpr int kBarPF = 12;               // [3] P(g) written, O free (one arrive per softmax warp)
  static constexpr int kBarDrainS = 15;
  static constexpr int kBarDrainP = 16;
  static constexpr int kBarOFree = 17;            // O read out (one arrive per epilogue warp)
  static constexpr int kBarStFull = 18;           // row statistics written (per softmax warp)
  static constexpr int kBarStFree = 19;           // row statistics read (per epilogue warp)
  static constexpr int kNumBars = 20;
  static constexpr int kBarBytes = 192;           // barriers, TMEM slot, abort flag
  static_assert(kNumBars * 8 + 8 <= kBarBytes, "barrier area");
  static constexpr int kOffStats = kOffBar + kBarBytes;  // float2 (m, l) per row
  static constexpr int kSmemBytes = kOffStats + QB * 8 + 1024;  // + align slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // Launch request: more than half of the SM's shared memory, so that two CTAs never
  // share an SM (each allocates all 512 TMEM columns; a second one would stall in
  // tcgen05.alloc until the first, persistent, CTA finished).
  static constexpr int kLaunchSmem = kSmemBytes > 120 * 1024 ? kSmemBytes : 120 * 1024;
  // instruction descriptors: S over a full step (N = 128) or a single 64-key block
  static constexpr uint32_t kIdescS = idesc_bf16_f32(QB, kKR, false, false);
  static constexpr uint32_t kIdescS1 = idesc_bf16_f32(QB, KB, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(QB, D, false, true);
};

// Bounded wait: with the slow path inline where registers are re-split per warpgroup
// (no calls there), out of line elsewhere (smaller code).
template <bool kInline>
__device__ __forceinline__ bool fwd_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                         int site) {
  if constexpr (kInline) return mbar_wait_inl(bar, parity, ctl, site);
  else return mbar_wait(bar, parity, ctl, site);
}

// Blocks in step s of a row with nnz active blocks.
template <int G>
__device__ __forceinline__ int step_blocks(int nnz, int s) {
  const int rem = nnz - s * G;
  return rem < G ? rem : G;
}

// The CTA's share of the work list: items[cta_start[c] .. cta_start[c+1]) for CTA c, as
// device records {bh, i, rs, nnz | (dpos + 1) << 16}: the item's (batch, head) pair
// bh = b * H + h and query block i (its rows start at row bh * Lq + i * QB of Q and O;
// key block j of the pair at row bh * Lk + j * KB of K and V), its row's first col_idx
// entry, its active block count and the position of block i in its row (-1: none).
// w = 0 marks an empty item, w = -1 the end.  Records are fetched two items ahead of use.
struct ItemStream {
  int t;                 // work-list index of the current item
  int end;               // one past the CTA's last item
  int n;                 // index of the current item among the non-empty ones
  int4 cur;
  int4 nx1;
  int4 nx2;

  // P: any kernel-argument struct with `items` and `cta_start` (forward or backward).
  template <class P>
  __device__ __forceinline__ int4 fetch(const P& p, int u) const {
    return u < end ? p.items[u] : make_int4(0, 0, 0, -1);
  }
  // Moves to the next item (kSkipEmpty: the next one with active blocks).
  template <bool kSkipEmpty, class P>
  __device__ __forceinline__ void next(const P& p) {
    for (;;) {
      ++t;
      cur = nx1;
      nx1 = nx2;
      nx2 = fetch(p, t + 2);
      if (cur.w > 0) ++n;
      if (!kSkipEmpty || cur.w != 0) return;
    }
  }
  template <bool kSkipEmpty, class P>
  __device__ __forceinline__ void init(const P& p) {
    t = p.cta_start[blockIdx.x] - 1;
    end = p.cta_start[blockIdx.x + 1];
    n = -1;
    nx1 = fetch(p, t + 1);
    nx2 = fetch(p, t + 2);
    next<kSkipEmpty>(p);
  }
  __device__ __forceinline__ bool done() const { return cur.w < 0; }
  __device__ __forceinline__ int nnz() const { return cur.w & 0xFFFF; }
  __device__ __forceinline__ int dpos() const { return (cur.w >> 16) - 1; }
};

// Steps of the non-empty items, in order.
template <int G>
struct StepCursor {
  ItemStream is;
  int s, nsteps;
  template <class P>
  __device__ __forceinline__ void init(const P& p) {
    is.init<true>(p);
    s = 0;
    nsteps = is.done() ? 0 : (is.nnz() + G - 1) / G;
  }
  template <class P>
  __device__ __forceinline__ void advance(const P& p) {
    if (++s >= nsteps) {
      is.next<true>(p);
      s = 0;
      nsteps = is.done() ? 0 : (is.nnz() + G - 1) / G;
    }
  }
  __device__ __forceinline__ bool valid() const { return !is.done(); }
  __device__ __forceinline__ int nblk() const { return step_blocks<G>(is.nnz(), s); }
};

// ----------------------------------------------------------------- producer

template <int QB, int KB, int D>
__device__ __forceinline__ void fwd_producer(const FwdParams& p, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             uint32_t sbase, const WaitCtl& ctl) {
  using C = FwdCfg<QB, KB, D>;
  constexpr int G = C::kG;
  static_assert(C::kNK == 3, "K slot reuse is tied to the three S buffers");
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  // Global row of each block of a step (nblk = 0: no step).
  struct StepRows {
    int krow[G];
    int nblk;
  };

  StepCursor<G> c;
  c.init(p);
  int colv[G];  // column blocks of the cursor's step, loaded one step ahead
  auto fetch_cols = [&]() {
    if (!c.valid()) return;
    const int nb = c.nblk();
    const int* cols = p.col_idx + c.is.cur.z + c.s * G;
#pragma unroll
    for (int g = 0; g < G; ++g) colv[g] = (g < nb) ? cols[g] : 0;
  };
  fetch_cols();

  StepRows h1{}, h2{};  // steps t-1, t-2
  h1.nblk = h2.nblk = 0;
  int nsteps = -1;  // known once the cursor runs out
  int nk = 0, nv = 0;  // K and V loads armed
  for (int t = 0;; ++t) {
    StepRows r0{};
    r0.nblk = 0;
    bool first = false;
    int qrow = 0, qb = 0;
    if (c.valid()) {
      r0.nblk = c.nblk();
      const int kv0 = c.is.cur.x * p.Lk;  // first K/V row of the item's (batch, head)
#pragma unroll
      for (int g = 0; g < G; ++g) r0.krow[g] = kv0 + colv[g] * KB;
      first = (c.s == 0);
      qrow = c.is.cur.x * p.Lq + c.is.cur.y * QB;
      qb = c.is.n % C::kNQ;
      if (first && c.is.nx1.w > 0) {
        // Warm L2 with the following item's Q.
        const int nrow = c.is.nx1.x * p.Lq + c.is.nx1.y * QB;
        tma_prefetch_l2_3d(tm_q, 0, nrow, 0);
      }
      c.advance(p);
      fetch_cols();  // the next step's columns, consumed one iteration later
    } else {
      if (nsteps < 0) nsteps = t;
      if (nsteps == 0 || t >= nsteps + 2) break;
    }
    if (r0.nblk > 0) {
      // K slot t % 3 held K(t-3), read by S(t-3); S(t-3) completing also shows that the S
      // issuer took that K barrier phase.  A step that opens an item needs its Q buffer
      // back: with one Q buffer the previous item's last S, S(t-1), must be complete;
      // with two, the last S of the item before that, S(t-2) or earlier.  S completes in
      // issue order, so one wait covers all of it.
      int j = (t >= 3) ? t - 3 : -1;
      if (first) j = max(j, t - (C::kNQ == 1 ? 1 : 2));
      if (j >= 0 && !fwd_wait<C::kSplitRegs>(bar(C::kBarSF + j % 3), (j / 3) & 1, ctl, kSiteProdKEmpty)) break;
      const uint32_t fb = bar(C::kBarKF + t % 3);
      mbar_arrive_expect_tx(fb, (first ? C::kQTile : 0) + r0.nblk * C::kBlkB);
      ++nk;
      // One copy per tile or block, all column halves at once.
      if (first) tma_load_3d(sbase + C::kOffQ + qb * C::kQTile, tm_q, fb, 0, qrow, 0);
      const uint32_t kdst = sbase + C::kOffK + (t % 3) * C::kKVTile;
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < r0.nblk) tma_load_3d(kdst + g * C::kBlkB, tm_k, fb, 0, r0.krow[g], 0);
    }
    const StepRows rv = h2;
    if (rv.nblk > 0) {
      // V slot g % kNV (g = t-2) held V(g-kNV), read by PV(g-kNV), which the PV issuer
      // issued after taking that V barrier phase.
      const int g = t - 2;
      const int gv = g - C::kNV;
      if (gv >= 0 && !fwd_wait<C::kSplitRegs>(bar(C::kBarPVD + gv % 3), (gv / 3) & 1, ctl, kSiteProdVEmpty))
        break;
      const uint32_t fb = bar(C::kBarVF + g % 3);
      mbar_arrive_expect_tx(fb, rv.nblk * C::kBlkB);
      ++nv;
      const uint32_t vdst = sbase + C::kOffV + (g % C::kNV) * C::kKVTile;
#pragma unroll
      for (int b = 0; b < G; ++b)
        if (b < rv.nblk) tma_load_3d(vdst + b * C::kBlkB, tm_v, fb, 0, rv.krow[b], 0);
    }
    h2 = h1;
    h1 = r0;
  }

  // Wait until every copy this thread issued has landed (immediate on the normal path).
  for (int j = (nk > 3 ? nk - 3 : 0); j < nk; ++j)
    mbar_drain_wait(bar(C::kBarKF + j % 3), (j / 3) & 1);
  for (int j = (nv > 3 ? nv - 3 : 0); j < nv; ++j)
    mbar_drain_wait(bar(C::kBarVF + j % 3), (j / 3) & 1);
}

// --------------------------------------------------------------- MMA issuers

// Shared-memory descriptors are built once; per MMA only the low word (start address >> 4)
// moves.  K and Q are K-major, V is MN-major; all three share the high word.
template <int QB, int KB, int D>
struct MmaDescs {
  using C = FwdCfg<QB, KB, D>;
  uint32_t hi, k0, v0, q0;
  __device__ __forceinline__ explicit MmaDescs(uint32_t sbase) {
    const uint64_t kdesc0 = sdesc_sw128(sbase + C::kOffK, 16, 1024);
    hi = static_cast<uint32_t>(kdesc0 >> 32);
    k0 = static_cast<uint32_t>(kdesc0);
    v0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffV, C::kHalfB, 1024));
    q0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffQ, 16, 1024));
  }
};

// S(t) = Q K(t)^T into S[t % 3].
template <int QB, int KB, int D>
__device__ __forceinline__ void fwd_mma_s(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                          const WaitCtl& ctl) {
  using C = FwdCfg<QB, KB, D>;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const MmaDescs<QB, KB, D> md(sbase);
  constexpr uint32_t kTileStep = C::kKVTile >> 4;  // descriptor units per K/V tile
  StepCursor<G> c;
  c.init(p);
  for (int t = 0; c.valid(); ++t) {
    const int nblk = c.nblk();
    const int qb = c.is.n % C::kNQ;
    c.advance(p);
    if (!fwd_wait<C::kSplitRegs>(bar(C::kBarKF + t % 3), (t / 3) & 1, ctl, kSiteMmaStage)) break;
    // S[t % 3] was last read by PV(t-3).
    if (t >= 3 && !fwd_wait<C::kSplitRegs>(bar(C::kBarPVD + t % 3), ((t - 3) / 3) & 1, ctl, kSiteMmaPvDone)) break;
    tc_fence_after();
    const uint32_t sb = tmem + (t % 3) * 128;
    const uint32_t qlo = md.q0 + qb * (C::kQTile >> 4);
    const uint32_t klo = md.k0 + (t % 3) * kTileStep;
    // KB = 128: one N = 128 MMA per 16 columns of d.  KB = 64: one N = 64 MMA per block
    // (the blocks' rows are not contiguous), into S columns [64g, 64g + 64), the two
    // blocks' MMAs alternating.  The block count is tested once, not between MMAs (a
    // branch between two MMAs slows their issue).
    auto s_mmas = [&](int nb) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qa = qlo + (((kk >> 2) * C::kQRegion + (kk & 3) * 32) >> 4);
        const uint32_t kb = klo + (((kk >> 2) * C::kHalfB + (kk & 3) * 32) >> 4);
        if (KB == 128) {
          tc_mma_ss_lh(sb, qa, md.hi, kb, md.hi, C::kIdescS, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int g = 0; g < nb; ++g)
            tc_mma_ss_lh(sb + g * KB, qa, md.hi, kb + ((g * C::kBlkB) >> 4), md.hi, C::kIdescS1,
                         kk > 0 ? 1u : 0u);
        }
      }
    };
    if (KB == 64 && nblk > 1)
      s_mmas(2);
    else
      s_mmas(1);
    tc_commit(bar(C::kBarSF + t % 3));
  }
  // Let every MMA this thread issued finish before TMEM is released.
  tc_commit(bar(C::kBarDrainS));
  mbar_drain_wait(bar(C::kBarDrainS), 0);
}

// O += P(g) V(g), P read from S[g % 3].
template <int QB, int KB, int D>
__device__ __forceinline__ void fwd_mma_pv(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                           const WaitCtl& ctl) {
  using C = FwdCfg<QB, KB, D>;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const MmaDescs<QB, KB, D> md(sbase);
  constexpr uint32_t kTileStep = C::kKVTile >> 4;
  StepCursor<G> c;
  c.init(p);
  for (int g = 0; c.valid(); ++g) {
    const int nblk = c.nblk();
    const bool first = (c.s == 0);
    const int item = c.is.n;  // among the non-empty items
    c.advance(p);
    // P(g) written, V(g) landed; on an item's first step, the previous item's O read out
    // (the epilogue releases O once per item, after this thread issued that item's PVs,
    // so its barrier cannot be a phase ahead; without an epilogue the softmax reads O
    // out before it hands that step's P over).
    if (!fwd_wait<C::kSplitRegs>(bar(C::kBarPF + g % 3), (g / 3) & 1, ctl, kSiteMmaPFull)) break;
    if (!fwd_wait<C::kSplitRegs>(bar(C::kBarVF + g % 3), (g / 3) & 1, ctl, kSiteMmaStage)) break;
    if (C::kEpi && first && item > 0 &&
        !fwd_wait<C::kSplitRegs>(bar(C::kBarOFree), (item - 1) & 1, ctl, kSiteMmaORead))
      break;
    tc_fence_after();
    const uint32_t ps = tmem + (g % 3) * 128;
    const uint32_t od = tmem + C::kOCol;
    const uint32_t vlo = md.v0 + (g % C::kNV) * kTileStep;
    // K = 16 keys per MMA: eight for a step of one 128-key block or two 64-key blocks, four
    // for a lone 64-key block.  The second block's four go in under one branch (a branch
    // between two MMAs slows their issue).
    auto pv = [&](int kk) {
      tc_mma_ts_lh(od, ps + kk * 8,
                   vlo + ((((kk * 16) / KB) * C::kBlkB + ((kk * 16) % KB) * 128) >> 4), md.hi,
                   C::kIdescPV, (kk == 0 && first) ? 0u : 1u);
    };
    static_assert(C::kKR == 128, "a step is 128 keys");
#pragma unroll
    for (int kk = 0; kk < (KB == 128 ? 8 : 4); ++kk) pv(kk);
    if (KB == 64 && nblk > 1) {
#pragma unroll
      for (int kk = 4; kk < 8; ++kk) pv(kk);
    }
    tc_commit(bar(C::kBarPVD + g % 3));
  }
  tc_commit(bar(C::kBarDrainP));
  mbar_drain_wait(bar(C::kBarDrainP), 0);
}

// ------------------------------------------------------------ softmax group

// Group c of this thread's O columns: lanes 0-15 hold columns [64c, 64c + 32), lanes
// 16-31 columns [64c + 32, 64c + 64) of the same rows.  The two lanes of a row thus hold
// the two halves of one 128-byte line of the bf16 output, which their stores fill together.
__device__ __forceinline__ void load_o32(uint32_t to, int c, uint32_t (&r)[32]) {
  tmem_ld_16x32bx2_x32<32>(to + c * 64, r);
}
__device__ __forceinline__ void store_o32(uint32_t to, int c, const uint32_t (&r)[32]) {
  tmem_st_16x32bx2_x32<32>(to + c * 64, r);
}

// Reads this thread's half row of O (the load_o32 groups), scales it by inv and packs it
// to bf16 pairs.
template <int D>
__device__ __forceinline__ void read_o(uint32_t to, float inv, uint32_t (&pk)[D / 4]) {
  constexpr int OC = D / 2;
  uint32_t r[OC / 32][32];
#pragma unroll
  for (int c = 0; c < OC / 32; ++c) load_o32(to, c, r[c]);
#pragma unroll
  for (int c = 0; c < OC / 32; ++c) tmem_ld_wait(r[c]);
#pragma unroll
  for (int c = 0; c < OC / 32; ++c)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[c * 16 + i] =
          pack_bf16x2(__uint_as_float(r[c][2 * i]) * inv, __uint_as_float(r[c][2 * i + 1]) * inv);
}

// Stores this thread's packed O columns (the load_o32 groups) and, from half 0, the lse.
// 32-byte stores (whole sectors) when the output base allows it, else 16-byte ones.
template <int D>
__device__ __forceinline__ void store_o(const FwdParams& p, int qrow, int half,
                                        const uint32_t (&pk)[D / 4], float m, float l) {
  constexpr int OC = D / 2;
  constexpr float kLn2 = 0.6931471805599453f;
  __nv_bfloat16* row = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(qrow) * D + half * 32;
  if ((reinterpret_cast<uintptr_t>(p.out) & 31) == 0) {
#pragma unroll
    for (int q = 0; q < OC / 16; ++q)  // 16 columns per store; group q / 2
      st_global_v8(row + (q >> 1) * 64 + (q & 1) * 16, pk[8 * q], pk[8 * q + 1], pk[8 * q + 2],
                   pk[8 * q + 3], pk[8 * q + 4], pk[8 * q + 5], pk[8 * q + 6], pk[8 * q + 7]);
  } else {
#pragma unroll
    for (int q = 0; q < OC / 8; ++q)  // 8 columns per store; group q / 4
      *reinterpret_cast<uint4*>(row + (q >> 2) * 64 + (q & 3) * 8) =
          make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
  if (half == 0) p.lse[qrow] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// tanh(z) = 1 - 2 / (1 + e^(2z)); e^(2z) from ex2 gives the exact limits +-1 for large
// |z| (the quotient goes to 0 or 2).
__device__ __forceinline__ float tanh_via_ex2(float z) {
  return 1.f - __fdividef(2.f, 1.f + ex2_approx(z * 2.8853900817779268f));
}

// The final (m, l) of a row and the factor its O accumulator is scaled by.  With a sink
// logit t (log2 units; -inf when there is none) the normaliser gains the term 2^t:
// m' = max(m, t), l' = l 2^(m - m') + 2^(t - m'), O / l' scaled by 2^(m - m').
__device__ __forceinline__ float finish_row(float& m, float& l, float t) {
  if (t == -INFINITY) return (l > 0.f) ? 1.f / l : 0.f;
  const float mf = fmaxf(m, t);
  const float a = (m == -INFINITY) ? 0.f : ex2_approx(m - mf);
  l = l * a + ex2_approx(t - mf);
  m = mf;
  return a / l;
}

template <int QB, int KB, int D, bool EXT>
__device__ __forceinline__ void fwd_softmax(const FwdParams& p, uint32_t sbase, uint8_t* smem,
                                            uint32_t tmem, const WaitCtl& ctl) {
  using C = FwdCfg<QB, KB, D>;
  constexpr int G = C::kG;
  constexpr int NC = 64;      // score columns per thread
  constexpr int OC = D / 2;   // O columns per thread
  constexpr int NA = 8;       // independent max chains
  constexpr int NS = 4;       // packed sum accumulators
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int wg = ((threadIdx.x >> 5) - C::kSoftWarp) >> 2;  // softmax group (warps 4-7, 8-11)
  const int wq = (threadIdx.x >> 5) & 3;         // TMEM lane quadrant of this warp
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  // Row of the query block held by this lane pair, and the TMEM lane base of the warp.
  const int row = (QB == 128) ? (wq * 32 + wg * 16 + (lane & 15)) : (wq * 16 + (lane & 15));
  const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32 + (QB == 128 ? wg * 16 : 0)) << 16);
  const uint32_t to = tl + C::kOCol;
  // This half holds keys [64*half, 64*half + 64) of the step: half of the block when
  // KB = 128, block `half` of the step (all of its 64 keys) when KB = 64.
  const int kbase = (KB == 128) ? 64 * half : 0;
  float2* stats = reinterpret_cast<float2*>(smem + C::kOffStats);
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  constexpr float kLog2e = 1.4426950408889634f;
  // scale > 0: the row max of the raw scores gives the max of the scaled ones and the
  // exponent is one FFMA.  Otherwise (and always in the extended kernels, which transform
  // the scores first) the scores are scaled first (c = 1 afterwards).
  const bool pos_scale = !EXT && p.scale_log2 > 0.f;
  const float cs = pos_scale ? p.scale_log2 : 1.f;
  int g = 0;
  bool ok = true;
  // Without an epilogue: the previous item's row, O read out at this item's first step.
  bool have_pending = false;
  int pend_row = 0;
  float pend_m = 0.f, pend_l = 0.f;
  bool pend_ok = true;            // (EXT) the pending row lies inside the sequence
  float pend_t = -INFINITY;       // (EXT) the pending row's sink logit, log2 units
  // S(g+1) already complete, as seen by a probe issued during step g (its latency then
  // overlaps the end of step g instead of opening step g+1).
  bool s_next = false;

  // Every thread of a warp has finished its TMEM traffic: one arrive per warp.
  auto warp_arrive = [&](int b) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(b));
  };
  // Waits (bounded, warp-uniform result) for phase `parity` of barrier b.
  auto wait_bar = [&](int b, int parity, int site) -> bool {
    bool w = fwd_wait<C::kSplitRegs>(bar(b), parity, ctl, site);
    w = __all_sync(0xffffffffu, w);
    if (w) tc_fence_after();
    return w;
  };

  // With an epilogue, items with no active block are the epilogue's alone.
  ItemStream is;
  for (is.init<C::kEpi>(p); ok && !is.done(); is.next<C::kEpi>(p)) {
    const int nnz = is.nnz();
    const int qrow = is.cur.x * p.Lq + is.cur.y * QB + row;  // global query row
    // (EXT) the row's position in its sequence, batch, segment and sink
    int qpos = 0, qseg = 0;
    bool row_ok = true;
    float sink_t = -INFINITY;
    const int32_t* kvseg = nullptr;
    if constexpr (EXT) {
      qpos = is.cur.y * QB + row;
      row_ok = qpos < p.Lq;
      const int bi = is.cur.x / p.H;
      if (!C::kEpi && p.sinks != nullptr) sink_t = p.sinks[is.cur.x - bi * p.H] * kLog2e;
      if (p.kv_seg != nullptr) {
        kvseg = p.kv_seg + static_cast<size_t>(bi) * p.Lk;
        qseg = row_ok ? p.q_seg[static_cast<size_t>(bi) * p.Lq + qpos] : 0;
      }
    }
    if (!C::kEpi && nnz == 0) {
      if (row_ok) {
        uint4* orow = reinterpret_cast<uint4*>(outp + static_cast<size_t>(qrow) * D + half * OC);
#pragma unroll
        for (int c = 0; c < OC / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
        if (half == 0) p.lse[qrow] = (sink_t == -INFINITY) ? -INFINITY : sink_t / kLog2e;
      }
      continue;
    }
    const int dpos = (!EXT && p.causal_diag) ? is.dpos() : -1;  // position of block i in the row
    const int nsteps = (nnz + G - 1) / G;
    float m_used = -INFINITY;
    float l = 0.f;
    for (int s = 0; s < nsteps; ++s, ++g) {
      const int nblk = step_blocks<G>(nnz, s);
      const bool valid = (KB == 128) || (half < nblk);
      const bool diag = !EXT && valid && (((KB == 128) ? s : s * 2 + half) == dpos);
      const uint32_t ts = tl + (g % 3) * 128;
      // (EXT) key block of this half's keys; the load overlaps the S wait
      int colh = 0;
      if constexpr (EXT) {
        if (valid) colh = p.col_idx[is.cur.z + s * G + (KB == 64 ? half : 0)];
      }
      if (__all_sync(0xffffffffu, s_next)) {
        tc_fence_after();
      } else {
        ok = wait_bar(C::kBarSF + g % 3, (g / 3) & 1, kSiteSoftSFull);
        if (!ok) break;
      }
      float x[NC];
      {
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
      if constexpr (EXT) {
        // Scores in log2 units: soft-capped (cap * log2e * tanh(s / cap)) or scaled.
        if (p.softcap_log2 > 0.f) {
#pragma unroll
          for (int c = 0; c < NC; ++c) x[c] = p.softcap_log2 * tanh_via_ex2(x[c] * p.softcap_inv);
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c) x[c] *= p.scale_log2;
        }
        // Keys kpos0 + c allowed for c in [lo, hi]: inside the sequence, the window, and
        // (in a key block overlapping the query block's rows, with causal_diag) not after
        // the query.
        const int kpos0 = colh * KB + kbase;
        int lo = 0;
        int hi = min(NC - 1, p.Lk - 1 - kpos0);
        if (!row_ok || !valid) hi = -1;
        if (p.window_left >= 0) lo = max(lo, qpos - p.window_left - kpos0);
        if (p.window_right >= 0) hi = min(hi, qpos + p.window_right - kpos0);
        if (p.causal_diag) {
          const int k0 = colh * KB;
          if (k0 < (is.cur.y + 1) * QB && k0 + KB > is.cur.y * QB) hi = min(hi, qpos - kpos0);
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) x[c] = mask_outside(x[c], c, lo, hi);
        if (kvseg != nullptr && hi >= lo) {
          // Keys of another segment; only keys inside [lo, hi] (so inside the sequence)
          // are read.
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const bool in = (c >= lo) && (c <= hi);
            const int sg = in ? __ldg(kvseg + kpos0 + c) : qseg;
            if (sg != qseg) x[c] = -INFINITY;
          }
        }
      } else {
        if (!pos_scale) {
#pragma unroll
          for (int c = 0; c < NC; ++c) x[c] *= p.scale_log2;
        }
        if (!valid) {
#pragma unroll
          for (int c = 0; c < NC; ++c) x[c] = -INFINITY;
        } else if (diag) {
          // Key kbase + c is masked when it lies after the query row.  Predicated selects:
          // written as branches, the per-lane bounds made this step twice as slow.
          const int qin = row - kbase;
#pragma unroll
          for (int c = 0; c < NC; ++c) x[c] = mask_gt(x[c], c, qin);
        }
      }
      // Row max: NA chains of three-input maxima over columns c = a (mod NA), then the
      // other half of the row (lane ^ 16).
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
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      float alpha = 1.f;
      const float m_new = fmaxf(m_used, mx);
      if (s == 0) {
        m_used = m_new;
      } else if (m_new > m_used + 8.f) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;

      // exp2(x*c - m) on pairs (packed f32x2 FFMA, MUFU ex2); packed row sums; P (bf16
      // pairs) written over the S columns just read.
      uint64_t sr2[NS];
#pragma unroll
      for (int a = 0; a < NS; ++a) sr2[a] = 0ull;
      const uint64_t c2 = f2_pack(cs, cs), m2 = f2_pack(neg_m, neg_m);
      {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint64_t y = f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), c2, m2);
          const uint64_t e = f2_pack(ex2_approx(f2_lo(y)), ex2_approx(f2_hi(y)));
          sr2[i % NS] = f2_add(sr2[i % NS], e);
          pk[i] = pack_bf16x2(f2_lo(e), f2_hi(e));
        }
        tmem_st_16x32bx2_x32<32>(ts, pk);
      }
      // S(g+4) needs this step's P, so the barrier of S(g+1) cannot be a phase ahead.
      s_next = mbar_test_wait(bar(C::kBarSF + (g + 1) % 3), ((g + 1) / 3) & 1);
      sr2[0] = f2_add(f2_add(sr2[0], sr2[1]), f2_add(sr2[2], sr2[3]));
      float rs = f2_lo(sr2[0]) + f2_hi(sr2[0]);
      rs += __shfl_xor_sync(0xffffffffu, rs, 16);
      l = l * alpha + rs;

      // O rescale (rare): PV(g-1) must be complete first.  Its barrier cannot have moved
      // on to PV(g+2), which needs this step's P.
      if (s > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = wait_bar(C::kBarPVD + (g - 1) % 3, ((g - 1) / 3) & 1, kSiteSoftPvDone);
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < OC / 32; ++c) {
          uint32_t r[32];
          load_o32(to, c, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          store_o32(to, c, r);
        }
      }
      // Without an epilogue, at an item's first step: the previous item's O (its last
      // PV is g-1) is read out before this P is handed over, since the next PV
      // overwrites O.
      uint32_t opk[D / 4];
      if (!C::kEpi && s == 0 && have_pending) {
        ok = wait_bar(C::kBarPVD + (g - 1) % 3, ((g - 1) / 3) & 1, kSiteSoftItemDone);
        if (!ok) break;
        const float inv = EXT ? finish_row(pend_m, pend_l, pend_t)
                              : ((pend_l > 0.f) ? 1.f / pend_l : 0.f);
        read_o<D>(to, inv, opk);
      }
      tmem_st_wait();
      warp_arrive(C::kBarPF + g % 3);
      if (!C::kEpi && s == 0 && have_pending) {
        if (pend_ok) store_o<D>(p, pend_row, half, opk, pend_m, pend_l);
        have_pending = false;
      }
    }
    if (!ok) break;
    if constexpr (C::kEpi) {
      // Row statistics to the epilogue, once it has read the previous item's (both
      // barriers complete once per item, so neither can be a phase ahead of its waiter).
      if (is.n > 0) {
        ok = wait_bar(C::kBarStFree, (is.n - 1) & 1, kSiteSoftStatsFree);
        if (!ok) break;
      }
      if (half == 0) stats[row] = make_float2(m_used, l);
      __threadfence_block();
      warp_arrive(C::kBarStFull);
    } else {
      pend_row = qrow;
      pend_m = m_used;
      pend_l = l;
      pend_ok = row_ok;
      pend_t = sink_t;
      have_pending = true;
    }
  }
  if (!C::kEpi && ok && have_pending &&
      wait_bar(C::kBarPVD + (g - 1) % 3, ((g - 1) / 3) & 1, kSiteSoftItemDone)) {
    uint32_t opk[D / 4];
    const float inv = EXT ? finish_row(pend_m, pend_l, pend_t)
                          : ((pend_l > 0.f) ? 1.f / pend_l : 0.f);
    read_o<D>(to, inv, opk);
    if (pend_ok) store_o<D>(p, pend_row, half, opk, pend_m, pend_l);
  }
}

// ----------------------------------------------------------------- epilogue

// Per item: the rows' (m, l) from the softmax, O out of TMEM once the item's last PV is
// done (one row per thread, 32x32b; at QB = 64 the rows sit in lanes 0-15 of each
// quadrant), O released to the PV issuer, then O / l stored as bf16 and the lse.
template <int QB, int KB, int D, bool EXT>
__device__ __forceinline__ void fwd_epilogue(const FwdParams& p, uint32_t sbase, const uint8_t* smem,
                                             uint32_t tmem, const WaitCtl& ctl) {
  using C = FwdCfg<QB, KB, D>;
  constexpr int G = C::kG;
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.6931471805599453f;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int wq = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const bool lane_row = (QB == 128) || lane < 16;
  const int row = (QB == 128) ? wq * 32 + lane : wq * 16 + (lane & 15);
  const uint32_t to = tmem + (static_cast<uint32_t>(wq * 32) << 16) + C::kOCol;
  const float2* stats = reinterpret_cast<const float2*>(smem + C::kOffStats);
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  const bool v8 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
  auto wait_bar = [&](int b, int parity, int site) -> bool {
    bool w = fwd_wait<C::kSplitRegs>(bar(b), parity, ctl, site);
    w = __all_sync(0xffffffffu, w);
    if (w) tc_fence_after();
    return w;
  };
  auto warp_arrive = [&](int b) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(b));
  };

  int g = 0;  // first step of the current item
  ItemStream is;
  for (is.init<false>(p); !is.done(); is.next<false>(p)) {
    const int nnz = is.nnz();
    const int qrow = is.cur.x * p.Lq + is.cur.y * QB + row;  // global query row
    bool row_ok = lane_row;
    float sink_t = -INFINITY;  // (EXT) sink logit, log2 units
    if constexpr (EXT) {
      row_ok = row_ok && (is.cur.y * QB + row < p.Lq);
      if (p.sinks != nullptr) sink_t = p.sinks[is.cur.x % p.H] * kLog2e;
    }
    __nv_bfloat16* orow = outp + static_cast<size_t>(qrow) * D;
    if (nnz == 0) {
      if (row_ok) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
        p.lse[qrow] = (sink_t == -INFINITY) ? -INFINITY : sink_t / kLog2e;
      }
      continue;
    }
    const int gl = g + (nnz + G - 1) / G - 1;  // the item's last step
    g = gl + 1;
    if (!wait_bar(C::kBarStFull, is.n & 1, kSiteEpiStats)) break;
    const float2 ml = stats[row];
    warp_arrive(C::kBarStFree);
    // PV(gl)'s barrier cannot move on to PV(gl+3): the next item's first PV waits for
    // the O release below.
    if (!wait_bar(C::kBarPVD + gl % 3, (gl / 3) & 1, kSiteSoftItemDone)) break;
    float m = ml.x, l = ml.y;
    const float inv = EXT ? finish_row(m, l, sink_t) : ((l > 0.f) ? 1.f / l : 0.f);
    uint32_t pk[D / 2];
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(to + h * 64, r0);
      tmem_ld_32x32b_x32(to + h * 64 + 32, r1);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      if (h == D / 64 - 1) warp_arrive(C::kBarOFree);  // O may be overwritten now
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        pk[h * 32 + i] = pack_bf16x2(__uint_as_float(r0[2 * i]) * inv,
                                     __uint_as_float(r0[2 * i + 1]) * inv);
        pk[h * 32 + 16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]) * inv,
                                          __uint_as_float(r1[2 * i + 1]) * inv);
      }
    }
    if (row_ok) {
      if (v8) {
#pragma unroll
        for (int q = 0; q < D / 16; ++q) {
          if (q > 0) __nanosleep(C::kStoreGapNs);
          st_global_v8(orow + q * 16, pk[8 * q], pk[8 * q + 1], pk[8 * q + 2], pk[8 * q + 3],
                       pk[8 * q + 4], pk[8 * q + 5], pk[8 * q + 6], pk[8 * q + 7]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < D / 8; ++q)
          reinterpret_cast<uint4*>(orow)[q] =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      p.lse[qrow] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }
}

// ------------------------------------------------------------------- kernel

template <int QB, int KB, int D, bool EXT>
__global__ void __launch_bounds__(FwdCfg<QB, KB, D>::kThreads, 1)
    bsa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<QB, KB, D>;
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
    for (int x = 0; x < 3; ++x) {
      mbar_init(bar(C::kBarSF + x), 1);
      mbar_init(bar(C::kBarPVD + x), 1);
      mbar_init(bar(C::kBarKF + x), 1);
      mbar_init(bar(C::kBarVF + x), 1);
      mbar_init(bar(C::kBarPF + x), 4 * C::kNumWG);
    }
    mbar_init(bar(C::kBarDrainS), 1);
    mbar_init(bar(C::kBarDrainP), 1);
    mbar_init(bar(C::kBarOFree), 4);
    mbar_init(bar(C::kBarStFull), 4 * C::kNumWG);
    mbar_init(bar(C::kBarStFree), 4);
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
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns, p.expire_site};

  if (warp < C::kSoftWarp) {
    if constexpr (C::kSplitRegs) setmaxnreg_dec<C::kRegCtl>();
    if (warp == 0) {
      if (lane == 0) fwd_producer<QB, KB, D>(p, &tm_q, &tm_k, &tm_v, sbase, ctl);
    } else if (warp == 1) {
      if (lane == 0) fwd_mma_s<QB, KB, D>(p, sbase, tmem, ctl);
    } else if (warp == 2) {
      if (lane == 0) fwd_mma_pv<QB, KB, D>(p, sbase, tmem, ctl);
    }
  } else if (warp < C::kEpiWarp) {
    if constexpr (C::kSplitRegs) setmaxnreg_inc<C::kRegSoft>();
    fwd_softmax<QB, KB, D, EXT>(p, sbase, smem, tmem, ctl);
  } else if constexpr (C::kEpi) {
    if constexpr (C::kSplitRegs) setmaxnreg_dec<C::kRegEpi>();
    fwd_epilogue<QB, KB, D, EXT>(p, sbase, smem, tmem, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int QB, int KB, int D, bool EXT>
cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, int grid, cudaStream_t stream) {
  using C = FwdCfg<QB, KB, D>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(bsa_fwd_kernel<QB, KB, D, EXT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kLaunchSmem);
    if (e != cudaSuccess) return e;
    if (C::kSplitRegs) {
      // setmaxnreg.inc waits for registers that the other warpgroups gave back: the
      // shares only add up when the kernel is launched at exactly kLaunchRegs.
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, bsa_fwd_kernel<QB, KB, D, EXT>);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  bsa_fwd_kernel<QB, KB, D, EXT><<<grid, C::kThreads, C::kLaunchSmem, stream>>>(q, k, v, p);
  return cudaGetLastError();
}

}  // namespace bsa
