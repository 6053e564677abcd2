// mha_bwd_kernel.cuh - attention backward for sm_103a (GB300).
//
// What it computes: the gradients of L = sum(dO * O) with respect to Q, K and
// V for the forward pass of mha_fwd_kernel.cuh (same scale, same square
// top-left causal mask).  The pages give no attention backward; this is the
// derivative of the forward definition (chain rule through the row softmax),
// organised the FlashAttention-2 way: P is recomputed from the saved
// log-sum-exp instead of being stored.  Per head, with P_ij =
// exp(scale q_i.k_j - LSE_i) on the visible keys:
//
//   D_i   = sum_c dO_ic O_ic                       (bwd_rowdot_kernel)
//   dV_j  = sum_i P_ij dO_i                        (bwd_tile_kernel, DKDV)
//   dS_ij = P_ij (dO_i.v_j - D_i)
//   dK_j  = scale sum_i dS_ij q_i                  (bwd_tile_kernel, DKDV)
//   dQ_i  = scale sum_j dS_ij k_j                  (bwd_tile_kernel, !DKDV)
//
// dK/dV and dQ come from two instantiations of one tile kernel that each
// recompute the scores they need (S^T and dP^T per key tile in one, S and dP
// per query tile in the other), so no partial sum goes through global
// atomics.
//
// Both kernels share the forward kernel's shape.  Warp 0 loads the CTA's
// fixed pair of tiles and feeds ring A (the score product's operand: Q_i for
// dK/dV, K_j for dQ) with TMA; warp 3 feeds ring B (the second product's
// operand: dO_i, V_j), each ring a set of mbarrier-guarded shared-memory
// slots.  Warp 1 allocates TMEM and runs the tcgen05.mma issue loop (whole
// warp, one elected lane issues).  Warps 4-11 do the elementwise work, two
// threads per row of the tile (one TMEM lane): warps 4-7 take columns 0-63
// and warps 8-11 columns 64-127.  The recomputed P needs no row-wise
// reduction (it comes from the saved LSE), so the two halves never exchange
// anything.  Warp 2 only keeps warps 4-11 on TMEM lane quarters.  P^T is written back to TMEM as
// bf16 over S^T, and dS (dS^T) over dP (dP^T), each packed into columns
// 32-95 of its 128: every warp then overwrites only score columns it has
// already read itself.  Each is the A operand of a later MMA straight from
// TMEM.
//
// Every mbarrier wait is bounded (see mha_wait.cuh); a wait that runs out
// records a status bit, raises the CTA's abort flag, and the CTA drains its
// own copies and MMAs before freeing TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "mha_wait.cuh"
#include "sm103_ptx.cuh"

namespace mha {

struct BwdParams {
  const float* lse;        // [BH, N] natural log, from the forward pass
  const float* dsum;       // [BH, N] D_i (workspace, written by bwd_rowdot_kernel)
  __nv_bfloat16* dq;       // [BH, N, D]
  __nv_bfloat16* dk;       // [BH, N, D]
  __nv_bfloat16* dv;       // [BH, N, D]
  unsigned* status;        // device status word
  long long wait_limit;    // SM cycles per wait
  int N;
  int n_tiles;             // ceil(N / 128)
  int tiles_fastest;       // grid is (n_tiles, BH) instead of (BH, n_tiles)
  float scale;             // score multiplier
  float scale_log2;        // scale * log2(e)
};

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int kBlock = 128;             // rows per tile (queries or keys)
  static constexpr int kHalves = D / 64;         // 128-byte swizzle atoms across d
  static constexpr int kHalfBytes = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kRing = (D == 128) ? 2 : 3;  // the rings' space, in tile pairs
  // The other side's tiles come through two rings: ring A carries the
  // score product's operand (Q_i for dK/dV, K_j for dQ), ring B the second
  // product's (dO_i, V_j).  B's tile is free once the products that read
  // it are done (dP^T and dV += P^T dO; dP), A's only after the last one
  // (dK += dS^T Q; dQ += dS K), so A gets the deeper ring.
  static constexpr int kARing = (D == 128) ? 3 : 4, kBRing = 2 * kRing - kARing;
  // fixed pair (K,V for dK/dV; Q,dO for dQ), then ring A, then ring B
  static constexpr int kOffFixed = 0;
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffRowBuf = kOffRing + kRing * 2 * kTileBytes;  // float [8 warps][2][64]
  static constexpr int kOffBar = kOffRowBuf + 4 * 128 * 8;
  // barriers: fixed_full ring_full[2R] ring_empty[2R] s_full dp_full[2]
  //           p_ready ds_ready[2] acc_full drain
  // ring_*[0, kARing) serve ring A and ring_*[kARing, 2R) ring B; dK/dV
  // uses dp_full[0] and ds_ready[0], dQ one of each per dP buffer
  static constexpr int kBarFixed = 0, kBarRingFull = 1, kBarRingEmpty = 1 + 2 * kRing;
  static constexpr int kBarSFull = 1 + 4 * kRing, kBarDpFull = kBarSFull + 1;
  // p_ready: P^T written back (dK/dV), or S read into registers (dQ)
  static constexpr int kBarPReady = kBarDpFull + 2, kBarDsReady = kBarPReady + 1;
  static constexpr int kBarAcc = kBarDsReady + 2, kBarDrain = kBarAcc + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kOffBar % 8 == 0 && kOffRing % 1024 == 0, "mbarrier / swizzle-atom alignment");
  static constexpr int kThreads = 384;
  static constexpr uint32_t kTmemCols = 512;
  // scores [0,128), second product [128,256), accumulators from 256; the
  // bf16 P^T and dS are packed into columns 32-95 of the first two.  The dQ
  // kernel has one accumulator, so it double-buffers the second product
  // ([128,256) and [256,384)) and keeps dQ at [384, 384 + D).
  static constexpr uint32_t kColS = 0, kColP2 = 128, kColAcc = 256, kPackOff = 32;
  static constexpr uint32_t kColP2b = 256, kColAccQ = 384;
};

// D_i = sum_c dO_ic O_ic in fp32 over rows [0, rows).  A thread reads 16
// bytes (8 elements) of each, so D/8 lanes cover a row and a 256-thread
// block covers kRowsPerBlock rows.
template <int D>
struct RowdotCfg {
  static constexpr int kLanesPerRow = D / 8;
  static constexpr int kRowsPerBlock = 256 / kLanesPerRow;
};

template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         float* __restrict__ dsum,
                                                         long long rows) {
  constexpr int kL = RowdotCfg<D>::kLanesPerRow;
  const long long row = static_cast<long long>(blockIdx.x) * RowdotCfg<D>::kRowsPerBlock + threadIdx.x / kL;
  const int sub = threadIdx.x % kL;
  float acc = 0.f;
  if (row < rows) {
    const uint4 ua = *reinterpret_cast<const uint4*>(o + row * D + sub * 8);
    const uint4 ub = *reinterpret_cast<const uint4*>(dout + row * D + sub * 8);
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
  }
  // every lane takes part in the shuffles (rows past the end add zeros)
#pragma unroll
  for (int off = kL / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) dsum[row] = acc;
}

// Shared skeleton of the two tile kernels.  DKDV = true: one CTA per
// (batch*head, 128-key tile); the fixed pair is (K, V) and the ring carries
// (Q_i, dO_i) for every query tile that sees these keys.  DKDV = false: one
// CTA per (batch*head, 128-query tile); the fixed pair is (Q, dO) and the
// ring carries (K_j, V_j).
template <int D, bool CAUSAL, bool DKDV>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    bwd_tile_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Long sequences put a head's tiles next to each other in the launch
  // order, so the CTAs of one head run together and share its tiles in L2;
  // short ones keep heads fastest, which spreads the causal load better.
  const int bh = p.tiles_fastest ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.x);
  const int tpos = p.tiles_fastest ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.y);
  const int N = p.N;
  // this CTA's own tile (keys for dK/dV, queries for dQ), heaviest first
  // under the causal mask
  const int tile = (CAUSAL && !DKDV) ? (p.n_tiles - 1 - tpos) : tpos;
  const int r0 = tile * C::kBlock;
  // the other side's tiles this CTA walks: [t_begin, t_end)
  const int t_begin = (CAUSAL && DKDV) ? tile : 0;
  const int t_end = (CAUSAL && !DKDV) ? tile + 1 : p.n_tiles;
  const int n_steps = t_end - t_begin;

  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  const uint32_t fixed_full = bar(C::kBarFixed);
  auto ring_full = [&](int i) { return bar(C::kBarRingFull + i); };
  auto ring_empty = [&](int i) { return bar(C::kBarRingEmpty + i); };
  const uint32_t s_full = bar(C::kBarSFull);    // scores in TMEM
  // dO.V products in TMEM, per buffer (dK/dV: one buffer; dQ: step t uses t & 1)
  auto dp_full = [&](int b) { return bar(C::kBarDpFull + b); };
  // dK/dV: P^T written back over S^T; dQ: S read into registers
  const uint32_t p_ready = bar(C::kBarPReady);
  // dS (dS^T) written back over dP (dP^T), per buffer like dp_full
  auto ds_ready = [&](int b) { return bar(C::kBarDsReady + b); };
  // the buffer and the phase parity of step t's second product
  auto p2_buf = [](int t) { return DKDV ? 0 : (t & 1); };
  auto p2_par = [](int t) { return static_cast<uint32_t>(DKDV ? (t & 1) : ((t >> 1) & 1)); };
  auto p2_col = [&](int t) -> uint32_t { return p2_buf(t) ? C::kColP2b : C::kColP2; };
  constexpr uint32_t kColAccK = DKDV ? C::kColAcc : C::kColAccQ;
  // step t's ring-A tile sits in slot t % kARing, its ring-B tile in slot
  // t % kBRing
  auto sA = [&](int t) -> uint32_t { return sbase + C::kOffRing + (t % C::kARing) * C::kTileBytes; };
  auto sB = [&](int t) -> uint32_t {
    return sbase + C::kOffRing + (C::kARing + t % C::kBRing) * C::kTileBytes;
  };
  auto a_full = [&](int t) { return ring_full(t % C::kARing); };
  auto a_empty = [&](int t) { return ring_empty(t % C::kARing); };
  auto b_full = [&](int t) { return ring_full(C::kARing + t % C::kBRing); };
  auto b_empty = [&](int t) { return ring_empty(C::kARing + t % C::kBRing); };
  const uint32_t acc_full = bar(C::kBarAcc);
  const uint32_t drain_bar = bar(C::kBarDrain);
  // fixed pair: [0] K or Q, [1] V or dO; ring slot i: [0] Q or K, [1] dO or V
  auto sFixed = [&](int w) -> uint32_t { return sbase + C::kOffFixed + w * C::kTileBytes; };

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit};

  if (threadIdx.x == 0) {
    ptx::mbar_init(fixed_full, 1);
    for (int i = 0; i < 2 * C::kRing; ++i) {
      ptx::mbar_init(ring_full(i), 1);
      ptx::mbar_init(ring_empty(i), 1);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(p_ready, 8);  // one elected arrive per elementwise warp
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(dp_full(b), 1);
      ptx::mbar_init(ds_ready(b), 8);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmQ);
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
    ptx::prefetch_tensormap(&tmDO);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const CUtensorMap* fixed0 = DKDV ? &tmK : &tmQ;
  const CUtensorMap* fixed1 = DKDV ? &tmV : &tmDO;
  const CUtensorMap* ringA = DKDV ? &tmQ : &tmK;
  const CUtensorMap* ringB = DKDV ? &tmDO : &tmV;

  if (warp == 0 || warp == 3) {
    // ----------------------------------------------------------- producers
    // Warp 0 loads the fixed pair, then ring A; warp 3 loads ring B.  Each
    // runs at its own pace.
    if (lane == 0 && n_steps > 0) {
      if (warp == 0) {
        ptx::mbar_arrive_expect_tx(fixed_full, 2 * C::kTileBytes);
        for (int h = 0; h < C::kHalves; ++h) {
          ptx::tma_load_3d(sFixed(0) + h * C::kHalfBytes, fixed0, fixed_full, h * 64, r0, bh);
          ptx::tma_load_3d(sFixed(1) + h * C::kHalfBytes, fixed1, fixed_full, h * 64, r0, bh);
        }
      }
      const bool is_b = warp == 3;
      const int depth = is_b ? C::kBRing : C::kARing;
      const CUtensorMap* map = is_b ? ringB : ringA;
      auto full_of = [&](int t) { return is_b ? b_full(t) : a_full(t); };
      int t = 0;
      bool ok = true;
      for (; t < n_steps; ++t) {
        const int use = t / depth;
        if (use > 0 && !wait_one(is_b ? b_empty(t) : a_empty(t), (use - 1) & 1, ctl, kSiteProducerEmpty)) {
          ok = false;
          break;
        }
        const int y = (t_begin + t) * C::kBlock;
        const uint32_t dst = is_b ? sB(t) : sA(t);
        ptx::mbar_arrive_expect_tx(full_of(t), C::kTileBytes);
        for (int h = 0; h < C::kHalves; ++h)
          ptx::tma_load_3d(dst + h * C::kHalfBytes, map, full_of(t), h * 64, y, bh);
        // warm L2 one ring's depth ahead (two steps for a one-slot ring)
        const int ahead = t + max(depth, 2);
        if (ahead < n_steps) {
          const int y2 = (t_begin + ahead) * C::kBlock;
          for (int h = 0; h < C::kHalves; ++h) ptx::tma_prefetch_3d(map, h * 64, y2, bh);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA goes away
        if (warp == 0) drain_wait(fixed_full, 0, ctl);
        for (int u = max(0, t - depth); u < t; ++u) drain_wait(full_of(u), (u / depth) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // Every lane runs the loop with the same values; an elected lane issues.
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t kIdescAcc = ptx::idesc_bf16_f32(128, D, 0, 1);
    const uint32_t tS = tmem + C::kColS;
    const uint32_t tAcc0 = tmem + kColAccK, tAcc1 = tmem + kColAccK + D;
    // K-major views (rows x d, 128-byte swizzle, 8-row groups 1 KiB apart)
    // and MN-major views (d contiguous, d-halves 16 KiB apart) of a tile
    auto kmaj = [](uint32_t a) { return ptx::desc_sw128(a, 16, 1024); };
    auto mnmaj = [](uint32_t a) { return ptx::desc_sw128(a, C::kHalfBytes, 1024); };
    // dst[128 x 128] = a_tile . b_tile^T over d
    auto issue_scores = [&](uint32_t dst, uint32_t a_tile, uint32_t b_tile) {
      const uint64_t da = kmaj(a_tile), db = kmaj(b_tile);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t koff =
              static_cast<uint64_t>(((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4);
          ptx::mma_ss(dst, da + koff, db + koff, kIdescS, kk > 0 ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    // acc[128 x D] (+)= A . b_tile, A (128 x 128, bf16) read from TMEM at a_cols
    auto issue_acc = [&](uint32_t acc, uint32_t a_cols, uint32_t b_tile, bool first) {
      const uint64_t db = mnmaj(b_tile);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < C::kBlock / 16; ++kk)
          ptx::mma_ts(acc, a_cols + kk * 8, db + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                      kIdescAcc, (!first || kk > 0) ? 1u : 0u);
      }
      __syncwarp();
    };
    auto commit = [&](uint32_t b) {
      if (ptx::elect_one()) ptx::mma_commit(b);
      __syncwarp();
    };
    bool ok = n_steps > 0 && wait_warp(fixed_full, 0, ctl, kSiteMmaQ);
    // The scores of the next tile are computed while this tile's dS is being
    // made, and (dK/dV) the next dO.V product while its P is: per tile the
    // tensor core sees
    //   dK/dV: dV += P^T dO_t | S^T_{t+1} | dK += dS^T Q_t | dP^T_{t+1}
    //   dQ:    S_{t+1} | dP_{t+1} | dQ += dS K_t
    // dQ double-buffers dP, so dP_{t+1} need not wait for dS_t: the
    // elementwise warps make dS_{t+1} while the tensor core still works on
    // dQ_t.  Each product overwrites TMEM that an earlier one in this order
    // reads (P^T over S^T, dS over dP, dP_{t+1} over dS_{t-1}), which the
    // tensor pipe's in-order execution makes safe; the elementwise side has
    // read those columns before it signals.  No barrier can complete two
    // phases ahead of its waiter: each next-but-one phase needs an action
    // that follows the waiter's observation of the current one.
    auto a_wait = [&](int t) {
      const bool r = wait_warp(a_full(t), (t / C::kARing) & 1, ctl, kSiteMmaKV);
      if (r) ptx::tc_fence_after();
      return r;
    };
    auto b_wait = [&](int t) {
      const bool r = wait_warp(b_full(t), (t / C::kBRing) & 1, ctl, kSiteMmaKV);
      if (r) ptx::tc_fence_after();
      return r;
    };
    // prologue: step 0's scores and second product
    if (ok && (ok = a_wait(0))) {
      issue_scores(tS, sFixed(0), sA(0));  // S^T = K Q_0^T  |  S = Q K_0^T
      commit(s_full);
    }
    if (ok && (ok = b_wait(0))) {
      issue_scores(tmem + p2_col(0), sFixed(1), sB(0));  // dP^T = V dO_0^T  |  dP = dO V_0^T
      commit(dp_full(0));
      if constexpr (!DKDV) commit(b_empty(0));  // V_0 is read by dP_0 alone
    }
    for (int t = 0; t < n_steps && ok; ++t) {
      const bool more = t + 1 < n_steps;
      if (!(ok = wait_warp(p_ready, t & 1, ctl, kSiteMmaP))) break;
      ptx::tc_fence_after();
      if constexpr (DKDV) {
        issue_acc(tAcc0, tS + C::kPackOff, sB(t), t == 0);  // dV += P^T dO_t
        commit(b_empty(t));  // dO_t: read by dP^T_t and dV_t, both issued
        if (more) {
          if (!(ok = a_wait(t + 1))) break;
          issue_scores(tS, sFixed(0), sA(t + 1));  // S^T_{t+1}
          commit(s_full);
        }
        if (!(ok = wait_warp(ds_ready(0), t & 1, ctl, kSiteMmaP))) break;
        ptx::tc_fence_after();
        issue_acc(tAcc1, tmem + C::kColP2 + C::kPackOff, sA(t), t == 0);  // dK += dS^T Q_t
        commit(a_empty(t));
        if (more) {
          if (!(ok = b_wait(t + 1))) break;
          issue_scores(tmem + C::kColP2, sFixed(1), sB(t + 1));  // dP^T_{t+1}
          commit(dp_full(0));
        }
      } else {
        if (more) {
          const int u = t + 1;
          if (!(ok = a_wait(u))) break;
          issue_scores(tS, sFixed(0), sA(u));  // S_{t+1}
          commit(s_full);
          if (!(ok = b_wait(u))) break;
          issue_scores(tmem + p2_col(u), sFixed(1), sB(u));  // dP_{t+1}
          commit(dp_full(p2_buf(u)));
          commit(b_empty(u));
        }
        if (!(ok = wait_warp(ds_ready(p2_buf(t)), p2_par(t), ctl, kSiteMmaP))) break;
        ptx::tc_fence_after();
        issue_acc(tAcc0, tmem + p2_col(t) + C::kPackOff, sA(t), t == 0);  // dQ += dS K_t
        commit(a_empty(t));
      }
    }
    if (ok) commit(acc_full);
    // every MMA this warp issued completes before TMEM is released
    commit(drain_bar);
    if (lane == 0) drain_wait(drain_bar, 0, ctl);
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ elementwise rows
    const int wq = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 4) >> 2;   // columns [64 * half, 64 * half + 64)
    const int cbase = 64 * half;
    const int row = wq * 32 + lane;
    const int my = r0 + row;  // this thread's key (dK/dV) or query (dQ)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS + cbase;  // this warp's score columns
    // where its 64 bf16 results go: 32 packed columns inside the 64 it reads
    const uint32_t tSPack = tmem + lane_off + C::kColS + C::kPackOff + 32 * half;
    const float sl2 = p.scale_log2;
    constexpr float kLog2e = 1.4426950408889634f;
    const size_t base = static_cast<size_t>(bh) * N;
    // per-warp copy of its 64 columns' LSE * log2 e and D (dK/dV), as two
    // float[64] arrays so one 16-byte load covers four columns
    float* lse_buf = reinterpret_cast<float*>(smem + C::kOffRowBuf) + (warp - 4) * 128;
    float* d_buf = lse_buf + 64;
    // this row's own (LSE * log2 e, D) (dQ); rows past N see no key
    float my_lse2 = INFINITY, my_d = 0.f;
    if (!DKDV && my < N) {
      my_lse2 = p.lse[base + my] * kLog2e;
      my_d = p.dsum[base + my];
    }
    bool ok = true;
    for (int t = 0; t < n_steps && ok; ++t) {
      const int y0 = (t_begin + t) * C::kBlock;  // first column's query (dK/dV) or key (dQ)
      if constexpr (DKDV) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int c = lane + 32 * m;
          const int qi = y0 + cbase + c;
          // a query past N has LSE = +inf here, so its P and dS are 0
          lse_buf[c] = qi < N ? p.lse[base + qi] * kLog2e : INFINITY;
          d_buf[c] = qi < N ? p.dsum[base + qi] : 0.f;
        }
        __syncwarp();
      }
      // only a tile on the causal diagonal, or (dQ) one holding keys past
      // N, needs a per-element mask; queries past N (dK/dV) get P = 0 from
      // their LSE of +inf
      const bool edge = DKDV ? (CAUSAL && y0 < r0 + C::kBlock)
                             : (y0 + C::kBlock > N || (CAUSAL && y0 + C::kBlock - 1 > r0));
      if (!wait_warp(s_full, t & 1, ctl, kSiteSoftmaxS)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      // P over this thread's 64 columns, kept in registers for dS.  All 64
      // scores are read before any P goes back over them.
      float pr[64];
      {
        uint32_t sr[64];
        ptx::tmem_ld_x64(tS, sr);
#pragma unroll
        for (int i4 = 0; i4 < 16; ++i4) {
          const int c = 4 * i4;
          const float4 l4 = DKDV ? *reinterpret_cast<const float4*>(lse_buf + c)
                                 : make_float4(my_lse2, my_lse2, my_lse2, my_lse2);
          pr[c] = ptx::ex2(__uint_as_float(sr[c]) * sl2 - l4.x);
          pr[c + 1] = ptx::ex2(__uint_as_float(sr[c + 1]) * sl2 - l4.y);
          pr[c + 2] = ptx::ex2(__uint_as_float(sr[c + 2]) * sl2 - l4.z);
          pr[c + 3] = ptx::ex2(__uint_as_float(sr[c + 3]) * sl2 - l4.w);
        }
      }
      if (edge) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          bool vis;
          if constexpr (DKDV) {
            vis = !CAUSAL || my <= y0 + cbase + c;  // key my, query y0 + cbase + c
          } else {
            const int key = y0 + cbase + c;
            vis = key < N && (!CAUSAL || key <= my);
          }
          pr[c] = vis ? pr[c] : 0.f;
        }
      }
      if constexpr (DKDV) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16x2(pr[32 * k + 2 * i], pr[32 * k + 2 * i + 1]);
          ptx::tmem_st_x16(tSPack + 16 * k, pk);  // P^T over S^T
        }
        ptx::tmem_wait_st();
      }
      // dK/dV: P^T is in TMEM; dQ: S has been read.  Either way the issuer
      // may go on (dV += P^T dO, or the next tile's scores over S).
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(p_ready);
      if (!wait_warp(dp_full(p2_buf(t)), p2_par(t), ctl, kSiteSoftmaxS)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      // this step's second-product columns, and the packed dS over them
      const uint32_t tP2 = tmem + lane_off + p2_col(t) + cbase;
      const uint32_t tP2Pack = tmem + lane_off + p2_col(t) + C::kPackOff + 32 * half;
      {
        uint32_t dr[64];
        ptx::tmem_ld_x64(tP2, dr);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t pk[16];
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const int c = 32 * k + 4 * i4;
            const float4 d4 = DKDV ? *reinterpret_cast<const float4*>(d_buf + c)
                                   : make_float4(my_d, my_d, my_d, my_d);
            pk[2 * i4] = ptx::pack_bf16x2(pr[c] * (__uint_as_float(dr[c]) - d4.x),
                                          pr[c + 1] * (__uint_as_float(dr[c + 1]) - d4.y));
            pk[2 * i4 + 1] = ptx::pack_bf16x2(pr[c + 2] * (__uint_as_float(dr[c + 2]) - d4.z),
                                              pr[c + 3] * (__uint_as_float(dr[c + 3]) - d4.w));
          }
          // dS^T over dP^T (dK/dV) or dS over dP (dQ)
          ptx::tmem_st_x16(tP2Pack + 16 * k, pk);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ds_ready(p2_buf(t)));
    }
    if (ok && n_steps > 0 && wait_warp(acc_full, 0, ctl, kSiteSoftmaxO)) {
      ptx::tc_fence_after();
      const bool valid = my < N;
      // epilogue: accumulators -> bf16 rows (dK and dQ carry the scale);
      // each half of the warps writes half of every row
#pragma unroll 1
      for (int which = 0; which < (DKDV ? 2 : 1); ++which) {
        __nv_bfloat16* out = DKDV ? (which == 0 ? p.dv : p.dk) : p.dq;
        const float mul = (DKDV && which == 0) ? 1.f : p.scale;
        const uint32_t tacc = tmem + lane_off + kColAccK + which * D;
        __nv_bfloat16* orow = out + (base + (valid ? my : 0)) * D;
#pragma unroll
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
          uint32_t av[32];
          ptx::tmem_ld_x32(tacc + c * 32, av);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = ptx::pack_bf16x2(__uint_as_float(av[2 * i]) * mul,
                                     __uint_as_float(av[2 * i + 1]) * mul);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace mha
