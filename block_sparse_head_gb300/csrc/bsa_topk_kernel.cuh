// bsa_topk_kernel.cuh -- top-k token-gather attention with an attention sink, sm_103a.
//
// Method (DeepSeek-V4.1 "Sparse attention / Weighted row sum", the sparse_attn kernel):
// every query position m lists K rows of its batch's key-value matrix kv (one row is
// both key and value, shared by all H heads; -1 marks an unused slot).  Each head
// scores the listed rows, the softmax over them gets one more denominator term
// exp(sink[h]), and the output is the softmax-weighted sum of the same rows.  The
// online softmax runs over the list in steps of 128 rows.
//
// GB300 mapping.  H = 64 heads of D = 512 give M = 64 in the direct form (Q K^T), which
// keeps the tensor pipe half idle, and an accumulator of 512 fp32 columns, all of TMEM.
// So both products are taken transposed, with the gathered rows as M = 128:
//     S^T (128 rows x 64 heads)  = KV_sel (128 x 512) . Q^T       (K = 512)
//     O^T (512 x 64 heads)      += KV_sel^T (512 x 128) . P^T     (four M = 128 pieces)
// S^T uses 64 TMEM columns and O^T 256.  The softmax then runs down the TMEM lanes (one
// lane per gathered row): its per-head maximum and sum are reductions across the 128
// lanes (a shuffle reduce-scatter within each warp, then shared memory across the four
// warps).  The running maximum moves lazily, so past a position's first step a CTA-wide
// vote first decides whether any head's maximum moves at all, and only then is it
// reduced.  P^T goes to shared memory as bf16, the B operand of the second product.
// One CTA per SM walks positions m = blockIdx.x, blockIdx.x + gridDim.x, ...:
//   warp 0      producer: the position's Q (one 3-D TMA copy, 64 KB).
//   warp 1      MMA issuer (one thread) and TMEM owner.
//   warps 2-5   softmax, one per TMEM lane quadrant (row 32*(warp % 4) + lane of the
//               step), then the epilogue: O^T / l per head, bf16 out[m, h, :] and lse.
//               They also gather the next step's 128 listed rows (16-byte cp.async
//               copies into the 128-byte-swizzled operand layout, each warp instruction
//               reading 512 contiguous bytes) while the tensor core runs this step's
//               O^T product: the tile is refilled quarter by quarter (128 columns of D)
//               as soon as the product's piece that reads the quarter completed.  (TMA
//               gather4 moves four 128-byte row pieces per copy; 256 of them per step
//               kept the tensor core waiting.)
// Every wait is bounded (WaitCtl), as in the other kernels.
#pragma once

#include <cuda_bf16.h>

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

struct TopkCfg {
  static constexpr int kH = 64, kD = 512;
  static constexpr int kRows = 128;                  // listed rows per step
  static constexpr int kChunks = kD / 64;             // 64-column chunks of a row
  static constexpr int kThreads = 6 * 32;
  static constexpr int kQBytes = kH * kD * 2;         // [chunk][64 heads][64] swizzled
  static constexpr int kKVBytes = kRows * kD * 2;     // [chunk][128 rows][64] swizzled
  static constexpr int kChunkKV = kRows * 128;        // one chunk of the gathered tile
  static constexpr int kChunkQ = kH * 128;            // one chunk of Q
  static constexpr int kPBytes = kRows * kH * 2;      // P^T [128 rows][64 heads] swizzled
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffP = kOffKV + kKVBytes;
  static constexpr int kOffRed = kOffP + kPBytes;     // [4][64] partials, m[64], alpha[64],
  static constexpr int kRedBytes = 2048;              // inv[64], flag, vote
  static constexpr int kVoteWord = 4 * 64 + 3 * 64 + 1;  // int index of the vote counter
  static constexpr int kOffBar = kOffRed + kRedBytes;
  static constexpr int kBarQF = 0, kBarQE = 1, kBarKF = 2 /* [4] */, kBarKE = 6 /* [4] */,
                       kBarSF = 10, kBarPF = 11, kBarPVD = 12, kBarOR = 13, kBarDrain = 14,
                       kBarG0 = 15, kBarG1 = 16;  // softmax-group syncs (one arrive per warp)
  static constexpr int kNumBars = 17;
  static constexpr int kBarBytes = 192;
  static_assert(kNumBars * 8 + 8 <= kBarBytes, "barrier area");
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr int kST = 0, kOT = 64;            // TMEM columns: S^T, O^T (4 x 64)
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, kH, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kH, true, true);
};

struct TopkParams {
  const void* kv;       // bf16 [B][N][D]
  const int32_t* idx;   // [B*M][K]
  const float* sink;    // [H]
  void* out;            // bf16 [B*M][H][D]
  float* lse;           // fp32 [B*M][H]
  int32_t* status;
  float scale_log2;     // scale * log2(e)
  int M, N, K, npos;    // positions per batch, kv rows per batch, list length, B*M
  unsigned long long wait_limit_ns;
  int expire_site;
};

// ------------------------------------------------------------------ producer (warp 0)

__device__ __forceinline__ void topk_producer(const TopkParams& p, const CUtensorMap* tm_q,
                                              uint32_t sbase, const WaitCtl& ctl) {
  using C = TopkCfg;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  int item = 0;
  for (int pos = blockIdx.x; pos < p.npos; pos += gridDim.x, ++item) {
    // Q: one buffer, free once the previous position's last S^T completed.
    if (item > 0 && !mbar_wait(bar(C::kBarQE), (item - 1) & 1, ctl, kSiteProdKEmpty)) break;
    mbar_arrive_expect_tx(bar(C::kBarQF), C::kQBytes);
    tma_load_3d(sbase + C::kOffQ, tm_q, bar(C::kBarQF), 0, pos * C::kH, 0);
  }
  // Wait for the last copy issued (immediate on the normal path).
  if (item > 0) mbar_drain_wait(bar(C::kBarQF), (item - 1) & 1, 100000000ull);
}

// ----------------------------------------------------------------- MMA issuer (warp 1)

__device__ __forceinline__ void topk_mma(const TopkParams& p, uint32_t sbase, uint32_t tmem,
                                         const WaitCtl& ctl) {
  using C = TopkCfg;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int nsteps = (p.K + C::kRows - 1) / C::kRows;
  // K-major descriptors (S^T = KV Q^T) and MN-major ones (O^T = KV^T P^T): the gathered
  // tile as A both times, Q and P^T as B.
  const uint64_t kv_k = sdesc_sw128(sbase + C::kOffKV, 16, 1024);
  const uint32_t hi = static_cast<uint32_t>(kv_k >> 32);
  const uint32_t kv0 = static_cast<uint32_t>(kv_k);
  const uint32_t q0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffQ, 16, 1024));
  const uint32_t kvm0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffKV, C::kChunkKV, 1024));
  const uint32_t pm0 = static_cast<uint32_t>(sdesc_sw128(sbase + C::kOffP, C::kChunkKV, 1024));
  int item = 0, t = 0;
  bool ok = true;
  for (int pos = blockIdx.x; ok && pos < p.npos; pos += gridDim.x, ++item) {
    for (int s = 0; s < nsteps; ++s, ++t) {
      if (s == 0 && !mbar_wait(bar(C::kBarQF), item & 1, ctl, kSiteMmaStage)) { ok = false; break; }
#pragma unroll 1
      for (int qq = 0; qq < 4; ++qq) {
        if (!mbar_wait(bar(C::kBarKF + qq), t & 1, ctl, kSiteMmaStage)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {  // K = 16 columns of D each; chunk 2qq + k4 / 4
          const int kk = 8 * qq + k4;
          const uint32_t off_kv = ((kk >> 2) * C::kChunkKV + (kk & 3) * 32) >> 4;
          const uint32_t off_q = ((kk >> 2) * C::kChunkQ + (kk & 3) * 32) >> 4;
          tc_mma_ss_lh(tmem + C::kST, kv0 + off_kv, hi, q0 + off_q, hi, C::kIdescS, kk > 0 ? 1u : 0u);
        }
      }
      if (!ok) break;
      tc_commit(bar(C::kBarSF));
      if (s == nsteps - 1) tc_commit(bar(C::kBarQE));
      if (!mbar_wait(bar(C::kBarPF), t & 1, ctl, kSiteMmaPFull)) { ok = false; break; }
      // A position's first O^T product overwrites the accumulator: the previous
      // position's must have been read out.
      if (s == 0 && item > 0 && !mbar_wait(bar(C::kBarOR), (item - 1) & 1, ctl, kSiteMmaPFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16) {  // K = 16 rows each
          const uint32_t off = (k16 * 16 * 128) >> 4;
          tc_mma_ss_lh(tmem + C::kOT + 64 * qq, kvm0 + ((2 * qq * C::kChunkKV) >> 4) + off, hi,
                       pm0 + off, hi, C::kIdescPV, (s == 0 && k16 == 0) ? 0u : 1u);
        }
        tc_commit(bar(C::kBarKE + qq));
      }
      tc_commit(bar(C::kBarPVD));
    }
  }
  tc_commit(bar(C::kBarDrain));
  mbar_drain_wait(bar(C::kBarDrain), 0);
}

// ------------------------------------------------------------ softmax (warps 2-5)

// Reduce-scatter across the warp: v[0..63] (one value per column) -> the lane's two
// columns 2*lane, 2*lane + 1 combined over the 32 lanes.  Round w keeps the upper half of
// the remaining columns when lane & w, so the columns left are 32b4 + 16b3 + ... + 2b0.
template <bool kMax>
__device__ __forceinline__ float2 warp_reduce_scatter64(float (&v)[64]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16, n = 64; w >= 1; w >>= 1, n >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? v[i + n / 2] : v[i];
      const float send = up ? v[i] : v[i + n / 2];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return make_float2(v[0], v[1]);
}

__device__ __forceinline__ void topk_softmax(const TopkParams& p, uint32_t sbase, uint8_t* smem,
                                             uint32_t tmem, const WaitCtl& ctl) {
  using C = TopkCfg;
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.6931471805599453f;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qd = warp & 3;              // TMEM lane quadrant
  const int row = 32 * qd + lane;       // gathered row of the step (and O^T lane)
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);  // [4][64]
  float* smax = red + 256;                                   // [64] running max (log2)
  float* salpha = smax + 64;                                 // [64] rescale factors
  float* sinv = salpha + 64;                                 // [64] 1 / normaliser
  int* sflag = reinterpret_cast<int*>(sinv + 64);
  int* svote = reinterpret_cast<int*>(red) + C::kVoteWord;  // latest step + 1 whose vote said
                                                            // a max moves
  uint8_t* pt = smem + C::kOffP;
  const int nsteps = (p.K + C::kRows - 1) / C::kRows;
  auto wait = [&](int b, int parity, int site) {
    bool w = mbar_wait(bar(b), parity, ctl, site);
    w = __all_sync(0xffffffffu, w);
    if (w) tc_fence_after();
    return w;
  };
  auto warp_arrive = [&](int b) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(b));
  };
  // The four softmax warps meet on an mbarrier (G0 or G1, alternately) rather than a
  // named barrier, so that the meeting is a bounded wait: a warp that gives up on a
  // wait cannot leave the others stuck.  n_sync counts the meetings (same in every warp).
  int n_sync = 0;
  auto group_sync = [&]() -> bool {
    const int b = (n_sync & 1) ? C::kBarG1 : C::kBarG0;
    const int parity = (n_sync >> 1) & 1;
    ++n_sync;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(b));
    bool w = mbar_wait(bar(b), parity, ctl, kSiteSoftSFull);
    return __all_sync(0xffffffffu, w);
  };
  // Gathers step s of position pos (the CTA's step t) into the tile: thread u of the 128
  // copies, for each quarter qq (columns 128qq .. 128qq + 127 of D), 16 bytes (column piece
  // jj = 16qq + u % 16) of rows u / 16 + 8k, k < 16 -- two rows of 256 contiguous bytes per
  // warp instruction -- into the swizzled chunk 2qq + jj / 8.  A quarter is refilled once
  // the previous step's O^T piece that reads it completed; each warp arrives on the
  // quarter's barrier when its copies landed.  Unused or invalid slots copy row 0 (finite
  // data; their scores are masked).
  const int u = 32 * ((warp - 2) & 3) + lane;
  auto gather = [&](int gpos, int gs, int gt) -> bool {
    const int32_t* gl = p.idx + static_cast<size_t>(gpos) * p.K;
    const int bi = gpos / p.M;
    const __nv_bfloat16* base = static_cast<const __nv_bfloat16*>(p.kv) + static_cast<size_t>(bi) * p.N * C::kD;
    const int jj = u & 15;
    const __nv_bfloat16* src[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int j = gs * C::kRows + (u >> 4) + 8 * k;
      const int v = (j < p.K) ? gl[j] : -1;
      src[k] = base + static_cast<size_t>((v >= 0 && v < p.N) ? v : 0) * C::kD + 8 * jj;
    }
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      if (gt > 0 && !wait(C::kBarKE + qq, (gt - 1) & 1, kSiteProdVEmpty)) {
        cp_async_wait<0>();  // nothing of this thread's may still be landing on exit
        return false;
      }
      const uint32_t chunk = sbase + C::kOffKV + (2 * qq + (jj >> 3)) * C::kChunkKV;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int r = (u >> 4) + 8 * k;
        cp_async16(chunk + r * 128 + (((jj & 7) ^ (r & 7)) << 4), src[k] + 128 * qq);
      }
      cp_async_commit();
    }
    // Quarter qq is complete when at most 3 - qq later groups are still in flight.
    auto land = [&](int qq) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBarKF + qq));
    };
    cp_async_wait<3>();
    land(0);
    cp_async_wait<2>();
    land(1);
    cp_async_wait<1>();
    land(2);
    cp_async_wait<0>();
    land(3);
    return true;
  };
  // This row's list entry for step gs of position gpos (fetched a step ahead of use).
  auto entry = [&](int gpos, int gs) -> int {
    const int j = gs * C::kRows + row;
    return (gpos < p.npos && j < p.K) ? p.idx[static_cast<size_t>(gpos) * p.K + j] : -1;
  };
  int item = 0, t = 0;
  bool ok = p.npos > static_cast<int>(blockIdx.x) ? gather(blockIdx.x, 0, 0) : true;
  int v_next = entry(blockIdx.x, 0);
  for (int pos = blockIdx.x; ok && pos < p.npos; pos += gridDim.x, ++item) {
    float lp[64];  // this row's share of each head's normaliser
#pragma unroll
    for (int c = 0; c < 64; ++c) lp[c] = 0.f;
    for (int s = 0; s < nsteps; ++s, ++t) {
      const int v = v_next;
      v_next = (s + 1 < nsteps) ? entry(pos, s + 1) : entry(pos + gridDim.x, 0);
      const bool valid = v >= 0 && v < p.N;
      if (!wait(C::kBarSF, t & 1, kSiteSoftSFull)) { ok = false; break; }
      float x[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tl + C::kST, r0);
        tmem_ld_32x32b_x32(tl + C::kST + 32, r1);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = valid ? __uint_as_float(r0[c]) * p.scale_log2 : -INFINITY;
          x[32 + c] = valid ? __uint_as_float(r1[c]) * p.scale_log2 : -INFINITY;
        }
      }
      // A head's running max moves only on a position's first step or when one of the
      // step's scores exceeds it by more than 2^8 (log2 units).  Past the first step,
      // whether any score does is a CTA-wide vote (one meeting); only then are the
      // per-head maxima reduced (two more).  Every warp reads the vote before it
      // gathers the next step's rows, and no warp votes on the next step before that
      // step's S^T, which needs those rows: so the counter cannot have moved on when read.
      bool full = (s == 0);
      if (!full) {
        bool need = false;
#pragma unroll
        for (int c = 0; c < 64; ++c) need |= x[c] > smax[c] + 8.f;
        if (__any_sync(0xffffffffu, need) && lane == 0) atomicMax(svote, t + 1);
        if (!group_sync()) { ok = false; break; }
        full = *reinterpret_cast<volatile int*>(svote) >= t + 1;
      }
      bool moved = false;
      if (full) {
        // Per-head maximum over the step's 128 rows.
        {
          float v2[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) v2[c] = x[c];
          const float2 m2 = warp_reduce_scatter64<true>(v2);
          reinterpret_cast<float2*>(red + 64 * qd)[lane] = m2;
        }
        if (!group_sync()) { ok = false; break; }
        if (qd == 0) {
          // Lazy update: a head's running max moves only when it grows by more than 2^8
          // (or on the position's first step); alpha rescales what was summed before.
          bool mv = false;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 2 * lane + u;
            const float cm = fmaxf(fmaxf(red[c], red[64 + c]), fmaxf(red[128 + c], red[192 + c]));
            const float old = smax[c];
            float nw = old, a = 1.f;
            if (s == 0) {
              nw = cm;
            } else if (cm > old + 8.f) {
              nw = cm;
              a = ex2_approx(old - cm);  // old = -inf gives 0
              mv = true;
            }
            smax[c] = nw;
            salpha[c] = a;
          }
          mv = __any_sync(0xffffffffu, mv);
          if (lane == 0) *sflag = mv ? 1 : 0;
        }
        if (!group_sync()) { ok = false; break; }
        moved = *reinterpret_cast<volatile int*>(sflag) != 0;
      }
      // P^T row (bf16, this row's 64 heads) into shared memory, 128-byte swizzle.
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float m0 = smax[c], m1 = smax[c + 1];
        const float e0 = ex2_approx(x[c] - (m0 == -INFINITY ? 0.f : m0));
        const float e1 = ex2_approx(x[c + 1] - (m1 == -INFINITY ? 0.f : m1));
        if (moved) {
          lp[c] *= salpha[c];
          lp[c + 1] *= salpha[c + 1];
        }
        lp[c] += e0;
        lp[c + 1] += e1;
        pk[c / 2] = pack_bf16x2(e0, e1);
      }
      uint8_t* prow = pt + row * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      fence_proxy_async_smem();
      // A moved max rescales O^T (this thread's lane of each of the four pieces) before
      // this step's product adds to it; the previous step's product must be complete.
      if (moved && s > 0) {
        if (!wait(C::kBarPVD, (t - 1) & 1, kSiteSoftPvDone)) { ok = false; break; }
#pragma unroll 1
        for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t r[32];
            const uint32_t ta = tl + C::kOT + 64 * qq + 32 * h2;
            tmem_ld_32x32b_x32(ta, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              r[c] = __float_as_uint(__uint_as_float(r[c]) * salpha[32 * h2 + c]);
            tmem_st_32x32b_x32(ta, r);
          }
        }
        tmem_st_wait();
      }
      warp_arrive(C::kBarPF);
      // The next step's rows (of this position, or of the CTA's next one).
      const int npos2 = (s + 1 < nsteps) ? pos : pos + static_cast<int>(gridDim.x);
      if (npos2 < p.npos && !gather(npos2, (s + 1 < nsteps) ? s + 1 : 0, t + 1)) {
        ok = false;
        break;
      }
    }
    if (!ok) break;
    // Position done: the normaliser of each head is the sum of lp over the 128 rows (and
    // the sink); O^T is complete once the last step's product is.
    {
      float v2[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) v2[c] = lp[c];
      const float2 l2 = warp_reduce_scatter64<false>(v2);
      reinterpret_cast<float2*>(red + 64 * qd)[lane] = l2;
    }
    if (!group_sync()) break;
    if (qd == 0) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = 2 * lane + u;
        const float l = (red[c] + red[64 + c]) + (red[128 + c] + red[192 + c]);
        const float m = smax[c];
        const float tt = p.sink[c] * kLog2e;
        const float mf = fmaxf(m, tt);
        const float a = (m == -INFINITY) ? 0.f : ex2_approx(m - mf);
        const float lf = l * a + ex2_approx(tt - mf);
        sinv[c] = a / lf;
        p.lse[static_cast<size_t>(pos) * C::kH + c] = (mf + log2f(lf)) * kLn2;
      }
    }
    if (!group_sync()) break;
    if (!wait(C::kBarPVD, (t - 1) & 1, kSiteSoftItemDone)) break;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(pos) * C::kH * C::kD;
#pragma unroll 1
    for (int qq = 0; qq < 4; ++qq) {
      const int dcol = 128 * qq + row;  // this thread's column of D
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tl + C::kOT + 64 * qq + 32 * h2, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int h = 32 * h2 + c;
          orow[static_cast<size_t>(h) * C::kD + dcol] = __float2bfloat16_rn(__uint_as_float(r[c]) * sinv[h]);
        }
      }
    }
    warp_arrive(C::kBarOR);
  }
}

// ------------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(TopkCfg::kThreads, 1)
    bsa_topk_kernel(const __grid_constant__ CUtensorMap tm_q, const TopkParams p) {
  using C = TopkCfg;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, by pointer arithmetic on the shared array itself, so that the
  // compiler keeps shared-memory loads and stores (not generic ones) for it.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
    for (int i = 0; i < C::kNumBars; ++i)
      mbar_init(bar(i), (i == C::kBarPF || i == C::kBarOR || i == C::kBarG0 || i == C::kBarG1 ||
                       (i >= C::kBarKF && i < C::kBarKF + 4)) ? 4 : 1);
    *abort_flag = 0;
    reinterpret_cast<int*>(smem + C::kOffRed)[C::kVoteWord] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm_q);
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
    if (lane == 0) topk_producer(p, &tm_q, sbase, ctl);
  } else if (warp == 1) {
    if (lane == 0) topk_mma(p, sbase, tmem, ctl);
  } else {
    topk_softmax(p, sbase, smem, tmem, ctl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace bsa
