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
// GB300 mapping (one CTA per SM, 256 threads, warp-specialised):
//   warp 0       TMA producer: Q tile once per item, K and V tiles of each active
//                block into two rings of kStages slots (128-byte swizzled boxes).
//   warp 1       tcgen05 issuer (one thread) and TMEM owner:
//                  S = Q K^T   (M = block, N = block, K = d) into one of two TMEM
//                              S buffers, so S(j+1) runs while softmax works on S(j);
//                  O += P V    (M = block, N = d, K = block) into the TMEM O tile,
//                              P from shared memory, V as an MN-major operand.
//   warps 4..7   softmax warpgroup: TMEM -> registers, causal mask on the diagonal
//                block, base-2 online softmax with a lazy rescale (the running max is
//                only moved when it grows by more than 2^8), P -> shared memory as
//                bf16, O rescale in TMEM when needed, and the epilogue (O / l -> bf16,
//                lse = ln 2 * (m + log2 l)).  An item with no active block writes
//                O = 0 and lse = -inf.
//   warps 2..3   idle.
// Block 128 uses M = 128 MMAs (row r of S/O in TMEM lane r, one thread per row);
// block 64 uses M = 64 MMAs, whose rows sit in lanes 0-15 of each 32-lane quadrant,
// and each row is split between lanes t and t+16 of a warp (16x32bx2 TMEM loads).
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
  static constexpr int kThreads = 256;
  static constexpr int kTile = BLK * D * 2;  // bytes of one Q, K or V tile
  static constexpr int kStages = kTile >= 32768 ? 2 : (kTile >= 16384 ? 3 : 4);
  static constexpr int kPBytes = BLK * BLK * 2;
  static constexpr int kRegion = BLK * 128;  // one 64-column swizzled box of BLK rows
  static constexpr int kSCols = BLK;         // TMEM columns of one S buffer
  static constexpr int kOCol = 2 * kSCols;   // TMEM column of the O tile
  static constexpr int kTmemCols = (2 * kSCols + D) <= 256 ? 256 : 512;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTile;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffP = kOffV + kStages * kTile;
  static constexpr int kOffBar = kOffP + kPBytes;
  // barrier indices
  static constexpr int kBarQF = 0, kBarQE = 1;
  static constexpr int kBarKF = 2;
  static constexpr int kBarKE = kBarKF + kStages;
  static constexpr int kBarVF = kBarKE + kStages;
  static constexpr int kBarVE = kBarVF + kStages;
  static constexpr int kBarSF = kBarVE + kStages;
  static constexpr int kBarSE = kBarSF + 2;
  static constexpr int kBarPF = kBarSE + 2;
  static constexpr int kBarOF = kBarPF + 1;
  static constexpr int kBarDrain = kBarOF + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + align slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // instruction descriptors
  static constexpr uint32_t kIdescS = idesc_bf16_f32(BLK, BLK, false, false);
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ----------------------------------------------------------------- producer

template <int BLK, int D>
__device__ __forceinline__ void fwd_producer(const FwdParams& p, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             uint32_t sbase, const WaitCtl& ctl) {
  using C = FwdCfg<BLK, D>;
  constexpr int S = C::kStages;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  int qc = 0, kc = 0, vc = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
    const int4 it = p.items[t];
    const int nnz = it.w;
    if (nnz == 0) continue;
    const int rowbase = (it.x * p.H + it.y) * p.L;
    const int start = p.row_ptr[it.y * p.nb + it.z];
    ok = mbar_wait(bar(C::kBarQE), (qc & 1) ^ 1, ctl, kSiteProdQEmpty);
    if (!ok) break;
    mbar_arrive_expect_tx(bar(C::kBarQF), C::kTile);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_2d(sbase + C::kOffQ + c * C::kRegion, tm_q, bar(C::kBarQF), c * 64,
                  rowbase + it.z * BLK);
    ++qc;
    for (int j = 0; j < nnz; ++j) {
      const int krow = rowbase + p.col_idx[start + j] * BLK;
      const int ks = kc % S;
      ok = mbar_wait(bar(C::kBarKE + ks), ((kc / S) & 1) ^ 1, ctl, kSiteProdKEmpty);
      if (!ok) break;
      mbar_arrive_expect_tx(bar(C::kBarKF + ks), C::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sbase + C::kOffK + ks * C::kTile + c * C::kRegion, tm_k, bar(C::kBarKF + ks),
                    c * 64, krow);
      ++kc;
      const int vs = vc % S;
      ok = mbar_wait(bar(C::kBarVE + vs), ((vc / S) & 1) ^ 1, ctl, kSiteProdVEmpty);
      if (!ok) break;
      mbar_arrive_expect_tx(bar(C::kBarVF + vs), C::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sbase + C::kOffV + vs * C::kTile + c * C::kRegion, tm_v, bar(C::kBarVF + vs),
                    c * 64, krow);
      ++vc;
    }
  }
  // Wait until every copy this thread issued has landed (immediate on the normal path).
  if (qc > 0) mbar_drain_wait(bar(C::kBarQF), (qc - 1) & 1);
  for (int s = 0; s < S; ++s) {
    if (kc > s) {
      const int f = s + S * ((kc - 1 - s) / S);
      mbar_drain_wait(bar(C::kBarKF + s), (f / S) & 1);
    }
    if (vc > s) {
      const int f = s + S * ((vc - 1 - s) / S);
      mbar_drain_wait(bar(C::kBarVF + s), (f / S) & 1);
    }
  }
}

// --------------------------------------------------------------- MMA issuer

template <int BLK, int D>
__device__ __forceinline__ void fwd_mma(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                        const WaitCtl& ctl) {
  using C = FwdCfg<BLK, D>;
  constexpr int S = C::kStages;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  int qc = 0, kc = 0, vc = 0, sc = 0, pc = 0;
  bool ok = true;

  // S(sc) = Q K(kc)^T into TMEM buffer sc & 1.
  auto issue_s = [&]() -> bool {
    const int sb = sc & 1;
    if (!mbar_wait(bar(C::kBarSE + sb), ((sc >> 1) & 1) ^ 1, ctl, kSiteMmaSEmpty)) return false;
    const int ks = kc % S;
    if (!mbar_wait(bar(C::kBarKF + ks), (kc / S) & 1, ctl, kSiteMmaKFull)) return false;
    tc_fence_after();
    const uint32_t qa = sbase + C::kOffQ;
    const uint32_t ka = sbase + C::kOffK + ks * C::kTile;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * C::kRegion + (kk & 3) * 32;
      tc_mma_ss(tmem + sb * C::kSCols, sdesc_sw128(qa + off, 16, 1024),
                sdesc_sw128(ka + off, 16, 1024), C::kIdescS, kk > 0);
    }
    tc_commit(bar(C::kBarKE + ks));
    tc_commit(bar(C::kBarSF + sb));
    ++kc;
    ++sc;
    return true;
  };

  for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
    const int nnz = p.items[t].w;
    if (nnz == 0) continue;
    ok = mbar_wait(bar(C::kBarQF), qc & 1, ctl, kSiteMmaQFull);
    if (!ok) break;
    ++qc;
    tc_fence_after();
    ok = issue_s();
    if (!ok) break;
    if (nnz == 1) tc_commit(bar(C::kBarQE));
    for (int j = 0; j < nnz; ++j) {
      if (j + 1 < nnz) {
        ok = issue_s();
        if (!ok) break;
        if (j + 2 == nnz) tc_commit(bar(C::kBarQE));  // last S of the item issued
      }
      ok = mbar_wait(bar(C::kBarPF), pc & 1, ctl, kSiteMmaPFull);
      if (!ok) break;
      const int vs = vc % S;
      ok = mbar_wait(bar(C::kBarVF + vs), (vc / S) & 1, ctl, kSiteMmaVFull);
      if (!ok) break;
      tc_fence_after();
      const uint32_t pa = sbase + C::kOffP;
      const uint32_t va = sbase + C::kOffV + vs * C::kTile;
#pragma unroll
      for (int kk = 0; kk < BLK / 16; ++kk) {
        const uint32_t aoff = (kk >> 2) * C::kRegion + (kk & 3) * 32;
        tc_mma_ss(tmem + C::kOCol, sdesc_sw128(pa + aoff, 16, 1024),
                  sdesc_sw128(va + kk * 16 * 128, C::kRegion, 1024), C::kIdescPV,
                  (j > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(bar(C::kBarVE + vs));
      tc_commit(bar(C::kBarOF));
      ++vc;
      ++pc;
    }
  }
  // Let every MMA issued so far finish before TMEM is released.
  tc_commit(bar(C::kBarDrain));
  mbar_drain_wait(bar(C::kBarDrain), 0);
}

// ------------------------------------------------------------ softmax group

template <int BLK, int D>
__device__ __forceinline__ void fwd_softmax(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                            const WaitCtl& ctl) {
  using C = FwdCfg<BLK, D>;
  constexpr int NC = (BLK == 128) ? 128 : 32;  // S columns held per thread
  constexpr int OC = (BLK == 128) ? D : D / 2;  // O columns held per thread
  constexpr float kLn2 = 0.6931471805599453f;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };
  const int wq = (threadIdx.x >> 5) & 3;  // TMEM lane quadrant of this warp
  const int lane = threadIdx.x & 31;
  const int row = (BLK == 128) ? (wq * 32 + lane) : (wq * 16 + (lane & 15));
  const int half = (BLK == 128) ? 0 : (lane >> 4);
  const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t p_tile = sbase + C::kOffP;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  int sc = 0, oc = 0;
  bool ok = true;

  for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
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
    const int start = p.row_ptr[it.y * p.nb + it.z];
    float m_used = -INFINITY;
    float l = 0.f;
    for (int j = 0; j < nnz; ++j) {
      const bool diag = p.causal_diag && (p.col_idx[start + j] == it.z);
      const int sb = sc & 1;
      ok = mbar_wait(bar(C::kBarSF + sb), (sc >> 1) & 1, ctl, kSiteSoftSFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float x[NC];
      if constexpr (BLK == 128) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tl + sb * C::kSCols + c * 32, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[i]);
        }
      } else {
        uint32_t r[32];
        tmem_ld_16x32bx2_x32<32>(tl + sb * C::kSCols, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::kBarSE + sb));
      ++sc;

      // scores in log2 units, causal mask inside the diagonal block
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int key = half * 32 + c;
        float v = x[c] * p.scale_log2;
        if (diag && key > row) v = -INFINITY;
        x[c] = v;
        mx = fmaxf(mx, v);
      }
      if constexpr (BLK == 64) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      float alpha = 1.f;
      const float m_new = fmaxf(m_used, mx);
      if (j == 0) {
        m_used = m_new;
      } else if (m_new > m_used + 8.f) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      const float msub = (m_used == -INFINITY) ? 0.f : m_used;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        x[c] = ex2_approx(x[c] - msub);
        rs += x[c];
      }
      if constexpr (BLK == 64) rs += __shfl_xor_sync(0xffffffffu, rs, 16);
      l = l * alpha + rs;

      if (j > 0) {
        // PV(j-1) must be complete before O is rescaled and P is overwritten.
        ok = mbar_wait(bar(C::kBarOF), oc & 1, ctl, kSiteSoftOFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++oc;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < OC / 32; ++c) {
            uint32_t r[32];
            if constexpr (BLK == 128) {
              tmem_ld_32x32b_x32(tl + C::kOCol + c * 32, r);
            } else {
              tmem_ld_16x32bx2_x32<D / 2>(tl + C::kOCol + c * 32, r);
            }
            tmem_ld_wait(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            if constexpr (BLK == 128) {
              tmem_st_32x32b_x32(tl + C::kOCol + c * 32, r);
            } else {
              tmem_st_16x32bx2_x32<D / 2>(tl + C::kOCol + c * 32, r);
            }
          }
          tmem_st_wait();
        }
      }
      // P -> shared memory, bf16, K-major 128-byte-swizzled (8 keys per 16-byte chunk).
#pragma unroll
      for (int q = 0; q < NC / 8; ++q) {
        const int ch = half * 4 + q;  // chunk index along the keys of this row
        const int region = ch >> 3;
        const int phys = (ch & 7) ^ (row & 7);
        const uint32_t addr = p_tile + region * C::kRegion + row * 128 + phys * 16;
        st_shared_v4(addr, pack_bf16x2(x[8 * q + 0], x[8 * q + 1]),
                     pack_bf16x2(x[8 * q + 2], x[8 * q + 3]), pack_bf16x2(x[8 * q + 4], x[8 * q + 5]),
                     pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPF));
    }
    if (!ok) break;

    // epilogue: wait for the last PV, then O / l -> bf16 and lse.
    ok = mbar_wait(bar(C::kBarOF), oc & 1, ctl, kSiteSoftOFull);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    ++oc;
    tc_fence_after();
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < OC / 32; ++c) {
      uint32_t r[32];
      if constexpr (BLK == 128) {
        tmem_ld_32x32b_x32(tl + C::kOCol + c * 32, r);
      } else {
        tmem_ld_16x32bx2_x32<D / 2>(tl + C::kOCol + c * 32, r);
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
__global__ void __launch_bounds__(256, 1)
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
    mbar_init(bar(C::kBarQF), 1);
    mbar_init(bar(C::kBarQE), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarKF + s), 1);
      mbar_init(bar(C::kBarKE + s), 1);
      mbar_init(bar(C::kBarVF + s), 1);
      mbar_init(bar(C::kBarVE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kBarSF + s), 1);
      mbar_init(bar(C::kBarSE + s), 128);
    }
    mbar_init(bar(C::kBarPF), 128);
    mbar_init(bar(C::kBarOF), 1);
    mbar_init(bar(C::kBarDrain), 1);
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
    fwd_softmax<BLK, D>(p, sbase, tmem, ctl);
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
