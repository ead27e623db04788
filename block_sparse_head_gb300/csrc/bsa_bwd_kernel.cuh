// bsa_bwd_kernel.cuh -- block-sparse attention backward for sm_103a: dQ over the layout's
// rows, dK and dV over its columns.
//
// Method.  With P the masked softmax of the forward (recomputed from Q, K and the
// forward's lse, so P = exp(scale * q.k - lse) on active entries and 0 elsewhere) and
// delta[r] = sum_x dO[r,x] O[r,x]:
//     dP = dO V^T,  dS = P * (dP - delta),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// Masked entries have P = 0, so only the active blocks pass gradient ("Block Sparse
// Attention Techniques", section 2, "Gradient Propagation in Block Sparse Attention").
//
// One kernel template, two modes over the same pipeline:
//   dQ mode (KV = false): a work item is a query block i of one (batch, head) and walks
//     the key blocks j of its CSR row.  Item tiles A = Q_i, B = dO_i; step tiles X = K_j,
//     Y = V_j.  T1 = A X^T = S, T2 = B Y^T = dP; E1 = dS;  acc1 += E1 X = dQ / scale.
//   dK/dV mode (KV = true): a work item is a key block j and walks the query blocks i of
//     its CSC column.  Item tiles A = K_j, B = V_j; step tiles X = Q_i, Y = dO_i (plus
//     the lse and delta of those query rows).  T1 = A X^T = S^T, T2 = B Y^T = dP^T;
//     E1 = P^T, E2 = dS^T;  acc1 += E1 Y = dV,  acc2 += E2 X = dK / scale.
// A step covers 128 columns: one block when b = 128, two when b = 64.
//
// GB300 mapping.  One CTA per SM, persistent over its share of the work list (the same
// longest-first per-CTA schedule as the forward):
//   warp 0      TMA producer: item tiles (one 3-D copy each) and step tiles; in dK/dV mode
//               X and Y in two stages plus the step's lse and delta (bulk copies), in dQ
//               mode X (= K) in a ring of three and Y (= V) in a ring of two.
//   warp 1      MMA issuer (one thread) and TMEM owner: MMA1 and MMA2.  A second issuing
//               warp after the elementwise ones issues MMA3 (and MMA4).
//   warps 2..   elementwise warpgroups (two at b = 128, one at b = 64), laid out as the
//               forward's softmax: per step they read T1 and T2, form P and dS, and write
//               the bf16 operands for the second MMAs into TMEM.  At an item's end they
//               read the accumulators, scale and store them as bf16.
// dK/dV mode: T1 and T2 (128 columns each) and acc1 and acc2 (d each) fill the 512
// columns.  E1 and E2 (bf16, 64 columns each) both go over T1, so T2 is free as soon as
// the warps have loaded it and takes the next step's T1: the regions swap every step.
// MMA1 of step t+1 then runs while the warps form E2 of step t, and MMA2 of step t+1 (into
// the region E1/E2 of step t leave) follows MMA3/MMA4 of step t.  The item tile B gets a
// barrier of its own, so that A reloads once the item's last MMA1 is done.
// dQ mode: T1 alternates between two 128-column regions (steps of even and odd index)
// beside T2 and acc1.  MMA1 of step t goes in as soon as MMA3 of step t-2 has read its
// region, so it runs while the elementwise warps work on step t-1; MMA3 of step t-1, from
// the second issuing thread, goes in once dS of step t-1 is written.  An item's
// accumulator is read out at the next item's first step, after that step's operands are
// handed over.
// Every wait is bounded (WaitCtl), as in the forward.
#pragma once

#include "bsa_fwd_kernel.cuh"

namespace bsa {

template <int BLK, int D, bool KV>
struct BwdCfg {
  static_assert(BLK == 64 || BLK == 128, "block must be 64 or 128");
  static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
  static constexpr int kNumWG = (BLK == 128) ? 2 : 1;  // elementwise warpgroups
  static constexpr int kEwWarps = 4 * kNumWG;
  // A second MMA-issuing warp after the elementwise ones (the products with an operand
  // in TMEM: dQ, or dV and dK).
  static constexpr int kMma2Warp = 2 + kEwWarps;
  static constexpr int kThreads = 32 * (3 + kEwWarps);
  static constexpr int kG = 128 / BLK;           // column blocks per step
  static constexpr int kItemTile = BLK * D * 2;  // one item tile (A or B)
  static constexpr int kStepTile = 128 * D * 2;  // one step tile (X or Y), kG blocks
  static constexpr int kBlkB = BLK * D * 2;      // one block of a step tile
  static constexpr int kHalf = BLK * 128;        // one 64-column half of one block
  static constexpr int kNX = KV ? 2 : 3;  // X slots (dQ mode: K, held until MMA3 one step on)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kItemTile;
  static constexpr int kOffX = 2 * kItemTile;              // [kNX] slots
  static constexpr int kOffY = kOffX + kNX * kStepTile;    // [2] slots
  // dK/dV mode, per stage: lse of the step's 128 query rows, then delta, fp32, each as two
  // 64-row chunks 272 bytes apart (256 + 16), so that the two half-warps, which read
  // different chunks with the same index, hit different banks.
  static constexpr int kVecChunk = 272, kVecDelta = 2 * kVecChunk, kVecStage = 4 * kVecChunk;
  static constexpr int kOffVec = kOffY + 2 * kStepTile;    // [2] stages
  static constexpr int kVecBytes = KV ? 2 * kVecStage : 0;
  static constexpr int kOffBar = kOffVec + kVecBytes;
  // barriers
  static constexpr int kBarIF = 0;    // item tiles landed
  static constexpr int kBarIE = 1;    // item tiles free (the item's last MMA1/MMA2 done)
  static constexpr int kBarXF = 2;    // [kNX] X landed (dK/dV mode: X, Y and the vectors)
  static constexpr int kBarXE = 5;    // [kNX] X free (its step's MMA3 (and MMA4) done)
  static constexpr int kBarYF = 8;    // [2] dQ mode: Y landed
  static constexpr int kBarYE = 10;   // [2] dQ mode: Y free (its step's MMA2 done)
  static constexpr int kBarTF = 12;   // T1, T2 computed (dK/dV mode: T1 = S^T only)
  static constexpr int kBarEF = 13;   // E1 (E2) written (one arrive per elementwise warp)
  static constexpr int kBarAD = 14;   // [2] a step's MMA3/MMA4 done (dQ mode: by T1 region)
  static constexpr int kBarAR = 16;   // accumulators read out (one arrive per elementwise warp)
  static constexpr int kBarDrain = 17;
  static constexpr int kBarEF1 = 18;  // dK/dV mode: E1 (P^T) written (per elementwise warp)
  static constexpr int kBarDF = 19;   // dK/dV mode: T2 (dP^T) computed
  static constexpr int kBarDL = 20;   // dK/dV mode: T2 loaded by every elementwise warp
  static constexpr int kBarIFV = 21;  // dK/dV mode: item tile B (V) landed; kBarIF is A's
  static constexpr int kBarIEV = 22;  // dK/dV mode: item tile B free; kBarIE is A's
  static constexpr int kBarVI = 23;   // dK/dV mode: MMA3 (dV) of a step issued
  static constexpr int kBarDrain2 = 24;
  static constexpr int kBarQI = 25;   // dQ mode: MMA3 (dQ) of a step issued
  static constexpr int kNumBars = 26;
  static constexpr int kBarBytes = 256;  // barriers, TMEM slot, abort flag
  static_assert(kNumBars * 8 + 8 <= kBarBytes, "barrier area");
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr int kLaunchSmem = kSmemBytes > 120 * 1024 ? kSmemBytes : 120 * 1024;
  // TMEM columns.  dQ mode: T1 at 0 (even steps) or 256 (odd steps), T2 at 128, acc1 at
  // 384.  dK/dV mode: T1 and T2 swap between the regions at 0 and 128 from one step to
  // the next (T1 at 0 on even steps), E1 and E2 (bf16) share T1's region; acc1 at 256,
  // acc2 after it.
  static constexpr int kT1 = 0, kT2 = 128, kT1b = 256;
  static constexpr int kAcc1 = KV ? 256 : 384, kAcc2 = 256 + D;
  static_assert(KV ? (kAcc2 + D <= 512) : (kAcc1 + D <= 512), "TMEM budget");
  static constexpr uint32_t kIdesc1 = idesc_bf16_f32(BLK, 128, false, false);  // N = 128
  static constexpr uint32_t kIdesc1b = idesc_bf16_f32(BLK, BLK, false, false); // one block
  static constexpr uint32_t kIdesc3 = idesc_bf16_f32(BLK, D, false, true);     // B MN-major
};

// Stores this thread's packed columns of one row (the read_o layout) as bf16.
template <int D>
__device__ __forceinline__ void store_row_bf16(void* base, int row, int half,
                                               const uint32_t (&pk)[D / 4]) {
  constexpr int OC = D / 2;
  __nv_bfloat16* r = static_cast<__nv_bfloat16*>(base) + static_cast<size_t>(row) * D + half * 32;
#pragma unroll
  for (int q = 0; q < OC / 8; ++q)  // 8 columns per store; group q / 4
    *reinterpret_cast<uint4*>(r + (q >> 2) * 64 + (q & 3) * 8) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

template <int D>
__device__ __forceinline__ void zero_row_bf16(void* base, int row, int half) {
  constexpr int OC = D / 2;
  uint4* r = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) +
                                      static_cast<size_t>(row) * D + half * OC);
#pragma unroll
  for (int c = 0; c < OC / 8; ++c) r[c] = make_uint4(0, 0, 0, 0);
}

// ----------------------------------------------------------------- producer

template <int BLK, int D, bool KV>
__device__ __forceinline__ void bwd_producer(const BwdParams& p, const CUtensorMap* tm_a,
                                             const CUtensorMap* tm_b, const CUtensorMap* tm_x,
                                             const CUtensorMap* tm_y, uint32_t sbase,
                                             const WaitCtl& ctl) {
  using C = BwdCfg<BLK, D, KV>;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  StepCursor<G> c;
  c.init(p);
  int n = -1, t = 0;
  int nx = 0, ny = 0;  // dQ mode: steps whose X (Y) copies were armed
  int nv = 0;          // dK/dV mode: items whose B was armed
  bool ok = true;
  for (; c.valid(); ++t) {
    const int nblk = c.nblk();
    const int bh = c.is.cur.x;
    int cols[G];
#pragma unroll
    for (int g = 0; g < G; ++g) cols[g] = (g < nblk) ? p.col_idx[c.is.cur.z + c.s * G + g] : 0;
    const bool item_first = c.s == 0;
    const int irow = bh * p.L + c.is.cur.y * BLK;  // the item's first row
    if (item_first) {
      // Item tiles: one buffer each.  A is free once the previous item's last MMA1
      // completed; dQ mode loads B with it (free once that item's last MMA2 completed).
      // n counts the items whose A was armed.
      if (n >= 0 && !mbar_wait(bar(C::kBarIE), n & 1, ctl, kSiteProdKEmpty)) {
        ok = false;
        break;
      }
      const uint32_t fb = bar(C::kBarIF);
      mbar_arrive_expect_tx(fb, (KV ? 1 : 2) * C::kItemTile);
      ++n;
      tma_load_3d(sbase + C::kOffA, tm_a, fb, 0, irow, 0);
      if constexpr (!KV) tma_load_3d(sbase + C::kOffB, tm_b, fb, 0, irow, 0);
    }
    c.advance(p);
    if constexpr (KV) {
      // Step stage t % 2 held step t-2, read by its MMA3/MMA4.
      if (t >= 2 && !mbar_wait(bar(C::kBarXE + t % 2), ((t - 2) / 2) & 1, ctl, kSiteProdVEmpty)) {
        ok = false;
        break;
      }
      const uint32_t fb = bar(C::kBarXF + t % 2);
      mbar_arrive_expect_tx(fb, nblk * (2 * C::kBlkB + 2 * BLK * 4));
      const uint32_t xd = sbase + C::kOffX + (t % 2) * C::kStepTile;
      const uint32_t yd = sbase + C::kOffY + (t % 2) * C::kStepTile;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (g < nblk) {
          const int row = bh * p.L + cols[g] * BLK;
          tma_load_3d(xd + g * C::kBlkB, tm_x, fb, 0, row, 0);
          tma_load_3d(yd + g * C::kBlkB, tm_y, fb, 0, row, 0);
#pragma unroll
          for (int h = 0; h < BLK / 64; ++h) {
            const uint32_t vd = sbase + C::kOffVec + (t % 2) * C::kVecStage +
                                (g * (BLK / 64) + h) * C::kVecChunk;
            bulk_load(vd, p.lse + row + 64 * h, 256, fb);
            bulk_load(vd + C::kVecDelta, p.delta + row + 64 * h, 256, fb);
          }
        }
      }
      if (item_first) {
        // B (V) after the step's tiles: the previous item's last MMA2, which frees its
        // slot, goes in after that item's last MMA1 and completes later.
        if (nv > 0 && !mbar_wait(bar(C::kBarIEV), (nv - 1) & 1, ctl, kSiteProdKEmpty)) {
          ok = false;
          break;
        }
        const uint32_t fv = bar(C::kBarIFV);
        mbar_arrive_expect_tx(fv, C::kItemTile);
        tma_load_3d(sbase + C::kOffB, tm_b, fv, 0, irow, 0);
        ++nv;
      }
    } else {
      // X slot t % 3 held K(t-3), read by MMA3(t-3); Y slot t % 2 held V(t-2), read by
      // MMA2(t-2).
      if (t >= 3 && !mbar_wait(bar(C::kBarXE + t % 3), ((t - 3) / 3) & 1, ctl, kSiteProdKEmpty)) {
        ok = false;
        break;
      }
      const uint32_t fx = bar(C::kBarXF + t % 3);
      mbar_arrive_expect_tx(fx, nblk * C::kBlkB);
      const uint32_t xd = sbase + C::kOffX + (t % 3) * C::kStepTile;
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < nblk) tma_load_3d(xd + g * C::kBlkB, tm_x, fx, 0, bh * p.L + cols[g] * BLK, 0);
      ++nx;
      if (t >= 2 && !mbar_wait(bar(C::kBarYE + t % 2), ((t - 2) / 2) & 1, ctl, kSiteProdVEmpty)) {
        ok = false;
        break;
      }
      const uint32_t fy = bar(C::kBarYF + t % 2);
      mbar_arrive_expect_tx(fy, nblk * C::kBlkB);
      const uint32_t yd = sbase + C::kOffY + (t % 2) * C::kStepTile;
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < nblk) tma_load_3d(yd + g * C::kBlkB, tm_y, fy, 0, bh * p.L + cols[g] * BLK, 0);
      ++ny;
    }
  }
  // Wait for every copy this thread issued (immediate on the normal path).
  if constexpr (KV) {
    for (int j = (t > 2 ? t - 2 : 0); j < t; ++j) mbar_drain_wait(bar(C::kBarXF + j % 2), (j / 2) & 1);
  } else {
    for (int j = (nx > 3 ? nx - 3 : 0); j < nx; ++j) mbar_drain_wait(bar(C::kBarXF + j % 3), (j / 3) & 1);
    for (int j = (ny > 2 ? ny - 2 : 0); j < ny; ++j) mbar_drain_wait(bar(C::kBarYF + j % 2), (j / 2) & 1);
  }
  (void)ok;
  if (n >= 0) mbar_drain_wait(bar(C::kBarIF), n & 1);
  if (KV && nv > 0) mbar_drain_wait(bar(C::kBarIFV), (nv - 1) & 1);
}

// ---------------------------------------------------------------- MMA issuer

template <int BLK, int D, bool KV>
__device__ __forceinline__ void bwd_mma(const BwdParams& p, uint32_t sbase, uint32_t tmem,
                                        const WaitCtl& ctl) {
  using C = BwdCfg<BLK, D, KV>;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  // Descriptor low words (start address >> 4 and the leading offset); the high word
  // (stride 1024, version, 128-byte swizzle) is shared.  K-major operands.
  const uint64_t a_desc = sdesc_sw128(sbase + C::kOffA, 16, 1024);
  const uint32_t hi = static_cast<uint32_t>(a_desc >> 32);
  const uint32_t a0 = static_cast<uint32_t>(a_desc);
  const uint32_t b0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffB, 16, 1024));
  const uint32_t x0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffX, 16, 1024));
  const uint32_t y0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffY, 16, 1024));
  constexpr uint32_t kStage = C::kStepTile >> 4;
  const uint32_t t2 = tmem + C::kT2;
  // T = item tile (A or B) x step tile^T over d: one N = 128 MMA per 16 columns of d, or
  // one N = 64 MMA per block at b = 64.
  // A branch between two MMAs slows their issue, so the block count of a step is tested
  // once, not between MMAs.
  auto issue_first = [&](uint32_t td, uint32_t it, uint32_t st, int nblk) {
    auto mmas = [&](int nb) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ia = ((kk >> 2) * (BLK * 128) + (kk & 3) * 32) >> 4;  // item tile offset
        const uint32_t is = ((kk >> 2) * C::kHalf + (kk & 3) * 32) >> 4;     // step block offset
        if (BLK == 128) {
          tc_mma_ss_lh(td, it + ia, hi, st + is, hi, C::kIdesc1, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int g = 0; g < nb; ++g)
            tc_mma_ss_lh(td + g * BLK, it + ia, hi, st + is + ((g * C::kBlkB) >> 4), hi,
                         C::kIdesc1b, kk > 0 ? 1u : 0u);
        }
      }
    };
    if (BLK == 64 && nblk > 1)
      mmas(2);
    else
      mmas(1);
  };
  StepCursor<G> c;
  c.init(p);
  int n = -1;
  if constexpr (KV) {
    // T1(t) (S^T, then E1 = P^T in its first 64 columns and E2 = dS^T in the next 64) is
    // the region at 0 on even steps and at 128 on odd ones; T2(t) (dP^T) is the other.
    // Two issuing threads: this one puts in MMA1 and MMA2 (both operands in shared
    // memory), the other (bwd_mma_kv2) MMA3 and MMA4.  Per step t, here:
    //   MMA2(t) into T2(t) = T1(t-1), once MMA3/MMA4(t-1) have read E1/E2 there;
    //   MMA1(t+1) into T1(t+1) = T2(t), once every elementwise warp has loaded dP^T(t)
    //   and MMA3(t) has been issued (so that E1 of step t+1, which needs this MMA1,
    //   cannot complete before the other thread has waited for E1 of step t).
    auto reg1 = [&](int t) { return tmem + ((t & 1) ? C::kT2 : C::kT1); };
    auto reg2 = [&](int t) { return tmem + ((t & 1) ? C::kT1 : C::kT2); };
    if (c.valid()) {
      int nblk = c.nblk();
      bool first = true;
      bool last = c.s == c.nsteps - 1;
      c.advance(p);
      n = 0;
      bool ok = mbar_wait(bar(C::kBarIF), 0, ctl, kSiteMmaStage) &&
                mbar_wait(bar(C::kBarXF), 0, ctl, kSiteMmaStage);
      if (ok) {
        tc_fence_after();
        issue_first(reg1(0), a0, x0, nblk);  // S^T = K Q^T
        tc_commit(bar(C::kBarTF));
        if (last) tc_commit(bar(C::kBarIE));
      }
      for (int t = 0; ok; ++t) {
        if (t > 0 && !mbar_wait(bar(C::kBarAD), (t - 1) & 1, ctl, kSiteMmaPvDone)) break;
        if (first && !mbar_wait(bar(C::kBarIFV), n & 1, ctl, kSiteMmaStage)) break;
        tc_fence_after();
        issue_first(reg2(t), b0, y0 + (t % 2) * kStage, nblk);  // dP^T = V dO^T
        tc_commit(bar(C::kBarDF));
        if (last) tc_commit(bar(C::kBarIEV));
        if (!c.valid()) break;
        nblk = c.nblk();
        first = c.s == 0;
        last = c.s == c.nsteps - 1;
        c.advance(p);
        if (!mbar_wait(bar(C::kBarDL), t & 1, ctl, kSiteMmaPFull)) break;
        if (!mbar_wait(bar(C::kBarVI), t & 1, ctl, kSiteMmaPFull)) break;
        if (first && !mbar_wait(bar(C::kBarIF), (n + 1) & 1, ctl, kSiteMmaStage)) break;
        if (!mbar_wait(bar(C::kBarXF + (t + 1) % 2), ((t + 1) / 2) & 1, ctl, kSiteMmaStage)) break;
        tc_fence_after();
        issue_first(reg1(t + 1), a0, x0 + ((t + 1) % 2) * kStage, nblk);
        tc_commit(bar(C::kBarTF));
        if (last) tc_commit(bar(C::kBarIE));
        if (first) ++n;
      }
    }
  } else {
    // This thread issues MMA1 and MMA2; the other (bwd_mma_dq2) MMA3 (dQ += dS K).
    auto t1_of = [&](int u) { return tmem + ((u & 1) ? C::kT1b : C::kT1); };
    for (int t = 0; c.valid(); ++t) {
      const int nblk = c.nblk();
      const bool first = c.s == 0;
      const bool last = c.s == c.nsteps - 1;
      c.advance(p);
      if (first) {
        ++n;
        if (!mbar_wait(bar(C::kBarIF), n & 1, ctl, kSiteMmaStage)) break;
      }
      if (!mbar_wait(bar(C::kBarXF + t % 3), (t / 3) & 1, ctl, kSiteMmaStage)) break;
      // This T1 region held step t-2, whose MMA3 read E1 from it (AD of that region cannot
      // be a phase ahead: its next phase is step t's own MMA3).
      if (t >= 2 && !mbar_wait(bar(C::kBarAD + (t & 1)), ((t - 2) / 2) & 1, ctl, kSiteMmaPvDone))
        break;
      tc_fence_after();
      issue_first(t1_of(t), a0, x0 + (t % 3) * kStage, nblk);  // S = Q K^T
      // T2 is free once the elementwise warps finished step t-1.
      if (t >= 1 && !mbar_wait(bar(C::kBarEF), (t - 1) & 1, ctl, kSiteMmaPFull)) break;
      if (!mbar_wait(bar(C::kBarYF + t % 2), (t / 2) & 1, ctl, kSiteMmaStage)) break;
      tc_fence_after();
      issue_first(t2, b0, y0 + (t % 2) * kStage, nblk);  // dP = dO V^T
      tc_commit(bar(C::kBarTF));
      tc_commit(bar(C::kBarYE + t % 2));
      if (last) tc_commit(bar(C::kBarIE));
    }
  }
  tc_commit(bar(C::kBarDrain));
  mbar_drain_wait(bar(C::kBarDrain), 0);
}

// acc += E (bf16 in TMEM, 128 columns of the step) x step tile (MN-major: columns d
// contiguous, halves kHalf apart); K = 16 rows of the step per MMA.  A branch between two
// MMAs slows their issue, so the block count is tested once.
template <int BLK, int D, bool KV>
__device__ __forceinline__ void bwd_issue_second(uint32_t acc, uint32_t te, uint32_t sm,
                                                 uint32_t hi, int nblk, bool first) {
  using C = BwdCfg<BLK, D, KV>;
  auto one = [&](int kk) {
    const uint32_t bo = ((((kk * 16) / BLK) * C::kBlkB + ((kk * 16) % BLK) * 128) >> 4);
    tc_mma_ts_lh(acc, te + kk * 8, sm + bo, hi, C::kIdesc3, (first && kk == 0) ? 0u : 1u);
  };
#pragma unroll
  for (int kk = 0; kk < (BLK == 128 ? 8 : 4); ++kk) one(kk);
  if (BLK == 64 && nblk > 1) {
#pragma unroll
    for (int kk = 4; kk < 8; ++kk) one(kk);
  }
}

// dQ mode, second issuing thread: per step u, MMA3(u) (dQ += dS K, dS over T1 of step u)
// once the warps have written dS; its completion frees that T1 region and the step's K
// slot.  Each MMA3 issued is marked on a barrier that the warps wait for before they hand
// over the next step's dS, so this thread cannot fall two phases behind the dS barrier.
template <int BLK, int D>
__device__ __forceinline__ void bwd_mma_dq2(const BwdParams& p, uint32_t sbase, uint32_t tmem,
                                            const WaitCtl& ctl) {
  using C = BwdCfg<BLK, D, false>;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const uint64_t x_desc = sdesc_sw128(sbase + C::kOffX, C::kHalf, 1024);
  const uint32_t hi = static_cast<uint32_t>(x_desc >> 32);
  const uint32_t xm0 = static_cast<uint32_t>(x_desc);
  constexpr uint32_t kStage = C::kStepTile >> 4;
  const uint32_t acc1 = tmem + C::kAcc1;
  StepCursor<G> c;
  c.init(p);
  int n = -1;
  for (int u = 0; c.valid(); ++u) {
    const int nblk = c.nblk();
    const bool first = c.s == 0;
    c.advance(p);
    if (first) ++n;
    if (!mbar_wait(bar(C::kBarEF), u & 1, ctl, kSiteMmaPFull)) break;
    // An item's first accumulation overwrites acc1: the previous item's must have been
    // read out.
    if (first && n > 0 && !mbar_wait(bar(C::kBarAR), (n - 1) & 1, ctl, kSiteMmaPFull)) break;
    tc_fence_after();
    bwd_issue_second<BLK, D, false>(acc1, tmem + ((u & 1) ? C::kT1b : C::kT1),
                                    xm0 + (u % 3) * kStage, hi, nblk, first);
    tc_commit(bar(C::kBarAD + (u & 1)));
    tc_commit(bar(C::kBarXE + u % 3));
    mbar_arrive(bar(C::kBarQI));
  }
  tc_commit(bar(C::kBarDrain2));
  mbar_drain_wait(bar(C::kBarDrain2), 0);
}

// dK/dV mode, second issuing thread: per step t, MMA3(t) (dV += P^T dO) once E1 is written
// and MMA4(t) (dK += dS^T Q) once E2 is; their completion frees T1(t) and the step's
// tiles.  An item's first accumulation overwrites the accumulators, so it waits until
// the previous item's have been read out.
template <int BLK, int D>
__device__ __forceinline__ void bwd_mma_kv2(const BwdParams& p, uint32_t sbase, uint32_t tmem,
                                            const WaitCtl& ctl) {
  using C = BwdCfg<BLK, D, true>;
  constexpr int G = C::kG;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const uint64_t x_desc = sdesc_sw128(sbase + C::kOffX, C::kHalf, 1024);
  const uint32_t hi = static_cast<uint32_t>(x_desc >> 32);
  const uint32_t xm0 = static_cast<uint32_t>(x_desc);
  const uint32_t ym0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffY, C::kHalf, 1024));
  constexpr uint32_t kStage = C::kStepTile >> 4;
  const uint32_t acc1 = tmem + C::kAcc1, acc2 = tmem + C::kAcc2;
  StepCursor<G> c;
  c.init(p);
  int n = -1;
  for (int t = 0; c.valid(); ++t) {
    const int nblk = c.nblk();
    const bool first = c.s == 0;
    c.advance(p);
    if (first) ++n;
    const uint32_t t1 = tmem + ((t & 1) ? C::kT2 : C::kT1);
    const uint32_t st = (t % 2) * kStage;
    if (!mbar_wait(bar(C::kBarEF1), t & 1, ctl, kSiteMmaPFull)) break;
    if (first && n > 0 && !mbar_wait(bar(C::kBarAR), (n - 1) & 1, ctl, kSiteMmaPFull)) break;
    tc_fence_after();
    bwd_issue_second<BLK, D, true>(acc1, t1, ym0 + st, hi, nblk, first);  // dV += P^T dO
    mbar_arrive(bar(C::kBarVI));
    if (!mbar_wait(bar(C::kBarEF), t & 1, ctl, kSiteMmaPFull)) break;
    tc_fence_after();
    bwd_issue_second<BLK, D, true>(acc2, t1 + 64, xm0 + st, hi, nblk, first);  // dK += dS^T Q
    tc_commit(bar(C::kBarAD));
    tc_commit(bar(C::kBarXE + t % 2));
  }
  tc_commit(bar(C::kBarDrain2));
  mbar_drain_wait(bar(C::kBarDrain2), 0);
}

// ----------------------------------------------------------- elementwise warps

template <int BLK, int D, bool KV>
__device__ __forceinline__ void bwd_elementwise(const BwdParams& p, uint32_t sbase,
                                                const uint8_t* smem, uint32_t tmem,
                                                const WaitCtl& ctl) {
  using C = BwdCfg<BLK, D, KV>;
  constexpr int G = C::kG;
  constexpr float kLog2e = 1.4426950408889634f;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int wg = ((threadIdx.x >> 5) - 2) >> 2;
  const int wq = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int row = (BLK == 128) ? (wq * 32 + wg * 16 + (lane & 15)) : (wq * 16 + (lane & 15));
  const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32 + (BLK == 128 ? wg * 16 : 0)) << 16);
  const int kbase = (BLK == 128) ? 64 * half : 0;  // first column of this half in its block
  const float* vec = reinterpret_cast<const float*>(smem + C::kOffVec);  // KV: lse and delta

  auto warp_arrive = [&](int b) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(b));
  };
  auto wait_bar = [&](int b, int parity, int site) -> bool {
    bool w = mbar_wait(bar(b), parity, ctl, site);
    w = __all_sync(0xffffffffu, w);
    if (w) tc_fence_after();
    return w;
  };

  // dQ mode: the accumulator of the previous item, read out at the next item's first
  // step once that step's E1 is handed over (its last MMA3 goes in only after that
  // step's MMA2).
  bool pending = false;
  int prow = 0, pg = 0;  // its output row and last step
  auto read_pending = [&]() -> bool {
    if (!wait_bar(C::kBarAD + (pg & 1), (pg / 2) & 1, kSiteSoftItemDone)) return false;
    uint32_t pk[D / 4];
    read_o<D>(tl + C::kAcc1, p.scale, pk);
    warp_arrive(C::kBarAR);
    store_row_bf16<D>(p.out1, prow, half, pk);
    pending = false;
    return true;
  };

  int g = 0;
  bool ok = true;
  ItemStream is;
  for (is.init<false>(p); ok && !is.done(); is.next<false>(p)) {
    const int cnt = is.nnz();
    const int orow = is.cur.x * p.L + is.cur.y * BLK + row;  // this thread's output row
    if (cnt == 0) {
      zero_row_bf16<D>(p.out1, orow, half);
      if (KV) zero_row_bf16<D>(p.out2, orow, half);
      continue;
    }
    float lr = 0.f, dr = 0.f;  // dQ mode: this row's lse (log2 units) and delta
    if constexpr (!KV) {
      lr = p.lse[orow] * kLog2e;
      dr = p.delta[orow];
    }
    const int dpos = p.causal_diag ? is.dpos() : -1;
    const int nsteps = (cnt + G - 1) / G;
    for (int s = 0; s < nsteps; ++s, ++g) {
      const int nblk = step_blocks<G>(cnt, s);
      const bool valid = (BLK == 128) || (half < nblk);
      const bool diag = valid && (((BLK == 128) ? s : s * 2 + half) == dpos);
      if constexpr (KV) {
        // T1 (S^T, then P^T | dS^T) and T2 (dP^T) swap regions every step.
        const uint32_t t1 = tl + ((g & 1) ? C::kT2 : C::kT1);
        const uint32_t t2 = tl + ((g & 1) ? C::kT1 : C::kT2);
        const int lo = diag ? row - kbase : -(1 << 30);  // query before the key: masked
        const float* vl = vec + ((g % 2) * C::kVecStage + half * C::kVecChunk) / 4;  // lse ...
        const float* vd = vl + C::kVecDelta / 4;                                    // ... delta
        if (!wait_bar(C::kBarTF, g & 1, kSiteSoftSFull)) {
          ok = false;
          break;
        }
        uint32_t rs[64];
        tmem_ld_16x32bx2_x32<64>(t1, *reinterpret_cast<uint32_t(*)[32]>(rs));
        tmem_ld_16x32bx2_x32<64>(t1 + 32, *reinterpret_cast<uint32_t(*)[32]>(rs + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rs));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rs + 32));
        // P^T over the first 64 columns of T1, handed over on its own so that dV's MMAs
        // run while dS^T is formed; rs keeps P^T (fp32) for dS^T.
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float e[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cc = 2 * i + u;
            // masked after scaling, so that a negative scale cannot turn -inf into +inf
            const float y = mask_outside(__uint_as_float(rs[cc]) * p.scale_log2 - vl[cc] * kLog2e,
                                         cc, lo, 1 << 30);
            e[u] = valid ? ex2_approx(y) : 0.f;
            rs[cc] = __float_as_uint(e[u]);
          }
          pk[i] = pack_bf16x2(e[0], e[1]);
        }
        tmem_st_16x32bx2_x32<32>(t1, pk);
        tmem_st_wait();
        warp_arrive(C::kBarEF1);
        if (!wait_bar(C::kBarDF, g & 1, kSiteSoftSFull)) {
          ok = false;
          break;
        }
        uint32_t rp[64];
        tmem_ld_16x32bx2_x32<64>(t2, *reinterpret_cast<uint32_t(*)[32]>(rp));
        tmem_ld_16x32bx2_x32<64>(t2 + 32, *reinterpret_cast<uint32_t(*)[32]>(rp + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rp));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rp + 32));
        warp_arrive(C::kBarDL);  // T2 may now take the next step's S^T
        // dS^T over the next 64 columns of T1.
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c0 = 2 * i, c1 = 2 * i + 1;
          const float d0 = __uint_as_float(rs[c0]) * (__uint_as_float(rp[c0]) - vd[c0]);
          const float d1 = __uint_as_float(rs[c1]) * (__uint_as_float(rp[c1]) - vd[c1]);
          pk[i] = valid ? pack_bf16x2(d0, d1) : 0u;
        }
        tmem_st_16x32bx2_x32<32>(t1 + 64, pk);
        tmem_st_wait();
        warp_arrive(C::kBarEF);
      } else {
        if (!wait_bar(C::kBarTF, g & 1, kSiteSoftSFull)) {
          ok = false;
          break;
        }
        const uint32_t t1 = tl + ((g & 1) ? C::kT1b : C::kT1);
        uint32_t rs[64], rp[64];
        tmem_ld_16x32bx2_x32<64>(t1, *reinterpret_cast<uint32_t(*)[32]>(rs));
        tmem_ld_16x32bx2_x32<64>(t1 + 32, *reinterpret_cast<uint32_t(*)[32]>(rs + 32));
        tmem_ld_16x32bx2_x32<64>(tl + C::kT2, *reinterpret_cast<uint32_t(*)[32]>(rp));
        tmem_ld_16x32bx2_x32<64>(tl + C::kT2 + 32, *reinterpret_cast<uint32_t(*)[32]>(rp + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rs));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rs + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rp));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(rp + 32));
        // Masked columns: the diagonal block's entries above the diagonal (key after the
        // query).
        const int hi = diag ? row - kbase : (1 << 30);
        uint32_t pk1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float ds[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cc = 2 * i + u;
            // masked after scaling, so that a negative scale cannot turn -inf into +inf
            const float y = mask_outside(__uint_as_float(rs[cc]) * p.scale_log2 - lr, cc, -(1 << 30), hi);
            const float pe = valid ? ex2_approx(y) : 0.f;
            ds[u] = valid ? pe * (__uint_as_float(rp[cc]) - dr) : 0.f;
          }
          pk1[i] = pack_bf16x2(ds[0], ds[1]);
        }
        tmem_st_16x32bx2_x32<32>(t1, pk1);
        tmem_st_wait();
        // The previous step's dQ product issued (see bwd_mma_dq2).
        if (g >= 1 && !wait_bar(C::kBarQI, (g - 1) & 1, kSiteSoftSFull)) {
          ok = false;
          break;
        }
        warp_arrive(C::kBarEF);
        if (s == 0 && pending && !read_pending()) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) break;
    if constexpr (KV) {
      // The item's accumulators are complete once its last step's MMA3/MMA4 are.
      if (!wait_bar(C::kBarAD, (g - 1) & 1, kSiteSoftItemDone)) break;
      uint32_t pk[D / 4], pk2[D / 4];
      read_o<D>(tl + C::kAcc1, 1.f, pk);
      read_o<D>(tl + C::kAcc2, p.scale, pk2);
      warp_arrive(C::kBarAR);
      store_row_bf16<D>(p.out1, orow, half, pk);
      store_row_bf16<D>(p.out2, orow, half, pk2);
    } else {
      pending = true;
      prow = orow;
      pg = g - 1;
    }
  }
  if (!KV && ok && pending) read_pending();
}

// ------------------------------------------------------------------- kernel

template <int BLK, int D, bool KV>
__global__ void __launch_bounds__(BwdCfg<BLK, D, KV>::kThreads, 1)
    bsa_bwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                   const BwdParams p) {
  using C = BwdCfg<BLK, D, KV>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, by pointer arithmetic on the shared array itself, so that the
  // compiler keeps shared-memory loads for it.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
    for (int i = 0; i < C::kNumBars; ++i)
      mbar_init(bar(i), (i == C::kBarEF || i == C::kBarAR || i == C::kBarEF1 || i == C::kBarDL)
                           ? C::kEwWarps
                           : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns, p.expire_site};
  if (warp == 0) {
    if (lane == 0) bwd_producer<BLK, D, KV>(p, &tm_a, &tm_b, &tm_x, &tm_y, sbase, ctl);
  } else if (warp == 1) {
    if (lane == 0) bwd_mma<BLK, D, KV>(p, sbase, tmem, ctl);
  } else if (warp == C::kMma2Warp) {
    if (lane == 0) {
      if constexpr (KV)
        bwd_mma_kv2<BLK, D>(p, sbase, tmem, ctl);
      else
        bwd_mma_dq2<BLK, D>(p, sbase, tmem, ctl);
    }
  } else {
    bwd_elementwise<BLK, D, KV>(p, sbase, smem, tmem, ctl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int BLK, int D, bool KV>
cudaError_t launch_bwd(const BwdParams& p, const CUtensorMap& a, const CUtensorMap& b,
                       const CUtensorMap& x, const CUtensorMap& y, int grid, cudaStream_t stream) {
  using C = BwdCfg<BLK, D, KV>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(bsa_bwd_kernel<BLK, D, KV>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kLaunchSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  bsa_bwd_kernel<BLK, D, KV><<<grid, C::kThreads, C::kLaunchSmem, stream>>>(a, b, x, y, p);
  return cudaGetLastError();
}

// delta[r] = sum_x dO[r,x] O[r,x] (fp32), D/8 lanes per row, 16-byte loads.
template <int D>
__global__ void __launch_bounds__(256) bsa_bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                            const __nv_bfloat16* __restrict__ dout,
                                                            float* __restrict__ delta, int rows) {
  constexpr int R = D / 8;  // lanes per row
  const int lane = threadIdx.x & 31;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) / R;
  float acc = 0.f;
  if (r < rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + r * D + (lane % R) * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + r * D + (lane % R) * 8);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa = __bfloat1622float2(a2[i]);
      const float2 fb = __bfloat1622float2(b2[i]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int w = R / 2; w >= 1; w /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (r < rows && lane % R == 0) delta[r] = acc;
}

}  // namespace bsa
