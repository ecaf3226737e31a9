// Backward of replay attention, split in two passes.
//
// dQ pass (attn_bwd_dq_kernel): one CTA = 128 packed query rows of one
// kv-head group against one partial (a prompt shard or the response keys).
// Per key tile: S = Q K^T and dP = dO V^T on the tensor cores, then
// P = exp(S*scale - lse), dS = P * (dP - D) in registers (one thread per
// row), dS (bf16) back to TMEM and dQ += dS K with dS as the TMEM-resident
// A operand.  Each partial writes its own dQ slice; a reduction kernel adds
// the slices into dQ in a fixed order.  Prompt keys are read only.
//
// dK/dV pass (attn_bwd_dkdv_kernel): one CTA = 128 response keys of one kv
// head; it walks the query tiles that see those keys and accumulates
// dV += P^T dO and dK += dS^T Q in TMEM, then adds them (+=) into the
// response gradient pages.  No prompt key is ever given a gradient: the
// prompt is stop-gradient resident state (LongStraw explainer, "The move:
// change the graph boundary"), and K/V gradient pages exist only for keys a
// response backward touches (explainer, "Two incompatible architectures,
// same transaction", Qwen bullet).
#include <cmath>
#include <climits>
#include "attn_common.cuh"
#include "internal.h"

namespace lsr {

// =========================================================== dQ pass
// K tiles are needed by S = Q K^T and, late, by dQ += dS K; V tiles only by
// dP = dO V^T.  The two live in separate rings so that a V stage is freed
// as soon as dP has been computed and the K ring can run three tiles ahead.
template <int D, int BN>
struct DqCfg {
  static constexpr int KST = 3;
  static constexpr int VST = (D == 128 && BN == 128) ? 2 : 3;
  static constexpr int Q_BYTES = kTileRows * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr uint32_t TM_DP = 2 * BN;
  static constexpr uint32_t TM_DQ = 3 * BN;
  static constexpr uint32_t TMEM_COLS = (3 * BN + D <= 256) ? 256 : 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, BN, false, false);
  static constexpr uint32_t ID_DQ = idesc_bf16(128, D, false, true);
};

template <int D, int BN>
struct __align__(1024) DqSmem {
  __nv_bfloat16 q[kTileRows * D];
  __nv_bfloat16 dO[kTileRows * D];
  __nv_bfloat16 k[DqCfg<D, BN>::KST][BN * D];
  __nv_bfloat16 v[DqCfg<D, BN>::VST][BN * D];
  uint64_t qd_full;
  uint64_t k_full[DqCfg<D, BN>::KST];  // K_j and V_j (one barrier per step)
  uint64_t k_empty[DqCfg<D, BN>::KST];
  uint64_t v_empty[DqCfg<D, BN>::VST];
  uint64_t sdp_full, ds_full[2], dp_free, dq_ready, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D, int BN>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mq,
                       const __grid_constant__ CUtensorMap mdo,
                       const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv,
                       const AttnParams p) {
  using C = DqCfg<D, BN>;
  constexpr int KST = C::KST, VST = C::VST;
  extern __shared__ uint8_t smem_raw[];
  DqSmem<D, BN>& s = *reinterpret_cast<DqSmem<D, BN>*>(align1024(smem_raw));
  const int warp = warp_id(), lane = lane_id();

  int u = blockIdx.x;
  const int qt = u % p.n_qtiles;
  u /= p.n_qtiles;
  const int g = u % p.Hkv;
  const int part = u / p.Hkv;
  const int r0 = qt * p.rows_per_tile;
  const int k_resp = resp_of_row(p, r0);
  const KeyRange kr = key_range(p, part, k_resp, r0, p.rows_per_tile);
  const int n_tiles = (kr.nkeys + BN - 1) / BN;
  const bool rev = walk_reversed(p, kr);

  if (threadIdx.x == 0) {
    mbar_init(&s.qd_full, 1);
    for (int i = 0; i < KST; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) mbar_init(&s.v_empty[i], 1);
    for (int i = 0; i < 2; ++i) mbar_init(&s.ds_full[i], 128);
    mbar_init(&s.sdp_full, 1);
    mbar_init(&s.dp_free, 128);
    mbar_init(&s.dq_ready, 1);
    mbar_init(&s.mma_done, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (n_tiles > 0) {  // the whole warp: one elected lane issues
      if (lane == 0) {
        prefetch_tmap(&mq);
        prefetch_tmap(&mdo);
        prefetch_tmap(&mk);
        prefetch_tmap(&mv);
      }
      __syncwarp();
      mbar_expect_tx_e(&s.qd_full, 2 * C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d_e(s.q + c * kTileRows * 64, &mq, &s.qd_full, c * 64,
                      g * p.G, r0);
        tma_load_3d_e(s.dO + c * kTileRows * 64, &mdo, &s.qd_full, c * 64,
                      g * p.G, r0);
      }
      int k_issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int row = pool_row(p, kr.page0, (rev ? n_tiles - 1 - j : j) * BN, g);
        const int ks = j % KST, vs = j % VST;
        if (j >= KST &&
            !warp_wait(&s.k_empty[ks], ((j / KST) & 1) ^ 1, &s.abort_flag, p.wait_ns))
          break;
        if (j >= VST &&
            !warp_wait(&s.v_empty[vs], ((j / VST) & 1) ^ 1, &s.abort_flag, p.wait_ns))
          break;
        // K_j and V_j land on one barrier
        mbar_expect_tx_e(&s.k_full[ks], 2 * C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d_e(s.k[ks] + c * BN * 64, &mk, &s.k_full[ks], c * 64, row);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d_e(s.v[vs] + c * BN * 64, &mv, &s.k_full[ks], c * 64, row);
        k_issued = j + 1;
      }
      // every copy lands before the CTA can exit (see the forward kernel)
      mbar_wait_drain(&s.qd_full, 0);
      for (int t = max(0, k_issued - KST); t < k_issued; ++t)
        mbar_wait_drain(&s.k_full[t % KST], (t / KST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Order: S_0, dP_0; then per step j: S_j+1, dP_j+1, dQ_j.  Every commit
    // and every wait of this warp costs the tensor pipe time, so there are
    // two commits per step (one after S_j+1 and dP_j+1, which the dS warps
    // wait for; one after dQ_j, which releases K_j's ring slot) and three
    // waits (K_j+1 and V_j+1 on one barrier, dP's buffer, dS_j).  The dS
    // warps release V's slots.
    if (n_tiles > 0) {  // the whole warp: one elected lane issues
      bool ok = warp_wait(&s.qd_full, 0, &s.abort_flag, p.wait_ns);
      // descriptors: one per operand tile, k-steps added as constants
      const uint64_t qd = sdesc(smem_u32(s.q), 16, 1024);
      const uint64_t dd = sdesc(smem_u32(s.dO), 16, 1024);
      // S_i = Q K_i^T into S buffer i & 1, dP_i = dO V_i^T
      auto issue_s_dp = [&](int i) -> bool {
        const int ks = i % KST, vs = i % VST;
        if (!warp_wait(&s.k_full[ks], (i / KST) & 1, &s.abort_flag, p.wait_ns))
          return false;
        tc_fence_after();
        const uint64_t kd = sdesc(smem_u32(s.k[ks]), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_e(tm + (i & 1) * BN, qd + kmaj_step<kTileRows>(k),
                   kd + kmaj_step<BN>(k), C::ID_S, k > 0);
        // dP has one buffer: the dS warps have loaded dP_{i-1}
        if (i >= 1 &&
            !warp_wait(&s.dp_free, (i - 1) & 1, &s.abort_flag, p.wait_ns))
          return false;
        tc_fence_after();
        const uint64_t vd = sdesc(smem_u32(s.v[vs]), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_e(tm + C::TM_DP, dd + kmaj_step<kTileRows>(k),
                   vd + kmaj_step<BN>(k), C::ID_S, k > 0);
        mma_commit_e(&s.sdp_full);
        return true;
      };
      if (ok) ok = issue_s_dp(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles && !issue_s_dp(j + 1)) break;
        const int ks = j % KST, b = j & 1;
        if (!warp_wait(&s.ds_full[b], (j >> 1) & 1, &s.abort_flag, p.wait_ns))
          break;
        tc_fence_after();
        // K as the MN-major B operand: 16 key rows of 128 bytes per step
        const uint64_t kd = sdesc(smem_u32(s.k[ks]), BN * 128, 1024);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts_e(tm + C::TM_DQ, tm + b * BN + k * 8, kd + (uint64_t)k * 128,
                   C::ID_DQ, (j > 0 || k > 0) ? 1u : 0u);
        mma_commit_e(&s.k_empty[ks]);
      }
      mma_commit_e(&s.dq_ready);
      mma_commit_e(&s.mma_done);
      mbar_wait_drain(&s.mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ dS warps
    const int quarter = warp & 3;
    const int mrow = quarter * 32 + lane;
    const int r = r0 + mrow / p.G;
    const int h = g * p.G + mrow % p.G;
    const RowInfo ri = row_info(p, k_resp, r);
    const bool valid = ri.valid;
    const int qpos = (valid && kr.causal) ? ri.qpos : INT_MAX;
    const uint32_t lane_base = tm + ((uint32_t)(quarter * 32) << 16);
    const float lse2 = valid ? p.lse[(size_t)h * p.R_b + r] * kLog2e : 0.f;
    const float Dv = valid ? p.Dvec[(size_t)h * p.R_b + r] : 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      // S_j and dP_j are complete
      if (!warp_wait(&s.sdp_full, j & 1, &s.abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dP_j has read V_j: its ring slot is free
      if (threadIdx.x == 64) mbar_arrive(&s.v_empty[j % VST]);
      // all of dP first, so the next dP product can start right away
      uint32_t dp[BN];
#pragma unroll
      for (int c = 0; c < BN; c += 32) tmem_ld32(lane_base + C::TM_DP + c, dp + c);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.dp_free);
      const int kbase = (rev ? n_tiles - 1 - j : j) * BN;
      const bool need_mask = kbase + BN - 1 > qpos;
#pragma unroll
      for (int c = 0; c < BN; c += 32) {
        uint32_t sv[32], ds[16];
        tmem_ld32(lane_base + b * BN + c, sv);
        tmem_ld_wait();
        if (need_mask)
          dq_chunk<true>(sv, dp + c, ds, p.scale_log2, lse2, Dv, kbase + c,
                         qpos);
        else
          dq_chunk<false>(sv, dp + c, ds, p.scale_log2, lse2, Dv, kbase + c,
                          qpos);
        tmem_st16(lane_base + b * BN + c / 2, ds);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.ds_full[b]);
    }
    float* drow = p.o + (((size_t)part * p.R_b + r) * p.Hq + h) * D;
    // the dQ slice row lies inside the workspace's num_shards + 1 slices
    const bool inb = valid && LSR_IN_BOUNDS(p, part <= p.num_shards &&
                                                   r < p.R_b && h < p.Hq);
    if (ok && n_tiles > 0) {
      ok = warp_wait(&s.dq_ready, 0, &s.abort_flag, p.wait_ns);
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::TM_DQ + c, o);
          tmem_ld_wait();
          if (inb) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 f = make_float4(__uint_as_float(o[i]) * p.scale,
                                     __uint_as_float(o[i + 1]) * p.scale,
                                     __uint_as_float(o[i + 2]) * p.scale,
                                     __uint_as_float(o[i + 3]) * p.scale);
              *reinterpret_cast<float4*>(drow + c + i) = f;
            }
          }
        }
      }
    } else if (n_tiles == 0 && inb) {
      for (int c = 0; c < D; c += 4)
        *reinterpret_cast<float4*>(drow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && s.abort_flag) atomicOr(p.status, LSR_DEV_WAIT_TIMEOUT);
}

// =========================================================== dK/dV pass
// Key tile is always 128 response keys (M = 128 MMAs); it is loaded as
// 128/KL sub-tiles of KL = min(page_size, 128) rows, one page each.
template <int D>
struct DkvCfg {
  static constexpr int STAGES = 2;
  static constexpr int QT_BYTES = kTileRows * D * 2;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256,
                            TM_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t ID_T = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t ID_ACC = idesc_bf16(128, D, false, true);
};

template <int D>
struct __align__(1024) DkvSmem {
  __nv_bfloat16 k[128 * D];
  __nv_bfloat16 v[128 * D];
  __nv_bfloat16 q[DkvCfg<D>::STAGES][kTileRows * D];
  __nv_bfloat16 dO[DkvCfg<D>::STAGES][kTileRows * D];
  float lse2[DkvCfg<D>::STAGES][kTileRows];
  float dvec[DkvCfg<D>::STAGES][kTileRows];
  int qpos[DkvCfg<D>::STAGES][kTileRows];
  uint64_t kv_full;
  uint64_t q_full[DkvCfg<D>::STAGES];
  uint64_t q_empty[DkvCfg<D>::STAGES];
  uint64_t s_full, p_full, acc_ready, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mq,
                         const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv,
                         const AttnParams p, int KL) {
  using C = DkvCfg<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  DkvSmem<D>& s = *reinterpret_cast<DkvSmem<D>*>(align1024(smem_raw));
  const int warp = warp_id(), lane = lane_id();

  const int e = blockIdx.x / p.Hkv;
  const int g = blockIdx.x % p.Hkv;
  int k_resp = 0;
  while (k_resp + 1 < p.resp.n && e >= p.resp.kt0[k_resp + 1]) ++k_resp;
  const int key0 = (e - p.resp.kt0[k_resp]) * 128;  // response key index
  // keys visible to the response's rows in this call
  const int nk_vis = p.resp.pos0[k_resp] + p.resp.rows[k_resp];
  const int rmin = key0 - p.resp.pos0[k_resp];  // first local row seeing key0
  const int qt_first = p.resp.row0[k_resp] / p.rows_per_tile;
  const int qt0 = qt_first + (rmin > 0 ? rmin / p.rows_per_tile : 0);
  const int n_q =
      qt_first +
      (p.resp.rows[k_resp] + p.rows_per_tile - 1) / p.rows_per_tile - qt0;
  const int nsub = (min(128, nk_vis - key0) + KL - 1) / KL;

  if (threadIdx.x == 0) {
    mbar_init(&s.kv_full, 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&s.q_full[i], 33);
      mbar_init(&s.q_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_full, 128);
    mbar_init(&s.acc_ready, 1);
    mbar_init(&s.mma_done, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s.tmem_base;

  if (warp == 0) {
    int issued = 0;
    if (lane == 0) {
      prefetch_tmap(&mq);
      prefetch_tmap(&mdo);
      prefetch_tmap(&mk);
      prefetch_tmap(&mv);
      mbar_expect_tx(&s.kv_full, 2 * nsub * KL * D * 2);
      for (int sub = 0; sub < nsub; ++sub) {
        const int row = pool_row(p, p.resp.page0[k_resp], key0 + sub * KL, g);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(s.k + c * 128 * 64 + sub * KL * 64, &mk, &s.kv_full,
                      c * 64, row);
          tma_load_2d(s.v + c * 128 * 64 + sub * KL * 64, &mv, &s.kv_full,
                      c * 64, row);
        }
      }
    }
    for (int i = 0; i < n_q; ++i) {
      const int st = i % ST;
      if (i >= ST &&
          !warp_wait(&s.q_empty[st], ((i / ST) & 1) ^ 1, &s.abort_flag, p.wait_ns))
        break;
      const int qt = qt0 + i;
      const int r0 = qt * p.rows_per_tile;
      if (lane == 0) {
        mbar_expect_tx(&s.q_full[st], 2 * C::QT_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(s.q[st] + c * kTileRows * 64, &mq, &s.q_full[st],
                      c * 64, g * p.G, r0);
          tma_load_3d(s.dO[st] + c * kTileRows * 64, &mdo, &s.q_full[st],
                      c * 64, g * p.G, r0);
        }
      }
      for (int m = lane; m < kTileRows; m += 32) {
        const int r = r0 + m / p.G;
        const int h = g * p.G + m % p.G;
        const RowInfo ri = row_info(p, k_resp, r);
        s.lse2[st][m] =
            ri.valid ? p.lse[(size_t)h * p.R_b + r] * kLog2e : INFINITY;
        s.dvec[st][m] = ri.valid ? p.Dvec[(size_t)h * p.R_b + r] : 0.f;
        s.qpos[st][m] = ri.valid ? ri.qpos : -1;
      }
      mbar_arrive(&s.q_full[st]);
      issued = i + 1;
    }
    if (lane == 0) {  // every copy lands before the CTA can exit
      mbar_wait_drain(&s.kv_full, 0);
      for (int t = max(0, issued - ST); t < issued; ++t)
        mbar_wait_drain(&s.q_full[t % ST], (t / ST) & 1);
    }
  } else if (warp == 1) {
    {  // the whole warp: one elected lane issues
      bool ok = warp_wait(&s.kv_full, 0, &s.abort_flag, p.wait_ns);
      const uint32_t ka = smem_u32(s.k), va = smem_u32(s.v);
      for (int i = 0; ok && i < n_q; ++i) {
        const int st = i % ST;
        if (!warp_wait(&s.q_full[st], (i / ST) & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t qa = smem_u32(s.q[st]), da = smem_u32(s.dO[st]);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          mma_ss_e(tm + C::TM_S, sdesc(ka, 16, 1024) + kmaj_step<128>(k),
                   sdesc(qa, 16, 1024) + kmaj_step<128>(k), C::ID_T, k > 0);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          mma_ss_e(tm + C::TM_DP, sdesc(va, 16, 1024) + kmaj_step<128>(k),
                   sdesc(da, 16, 1024) + kmaj_step<128>(k), C::ID_T, k > 0);
        }
        mma_commit_e(&s.s_full);
        if (!warp_wait(&s.p_full, i & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k) {
          mma_ts_e(tm + C::TM_DV, tm + C::TM_S + k * 8,
                   sdesc(da, kTileRows * 128, 1024) + (uint64_t)k * 128,
                   C::ID_ACC, (i > 0 || k > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k) {
          mma_ts_e(tm + C::TM_DK, tm + C::TM_DP + k * 8,
                   sdesc(qa, kTileRows * 128, 1024) + (uint64_t)k * 128,
                   C::ID_ACC, (i > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit_e(&s.q_empty[st]);
      }
      mma_commit_e(&s.acc_ready);
      mma_commit_e(&s.mma_done);
      mbar_wait_drain(&s.mma_done, 0);
    }
  } else {
    const int quarter = warp & 3;
    const int krow = quarter * 32 + lane;
    const int kj = key0 + krow;
    const uint32_t lane_base = tm + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      const int st = i % ST;
      if (!warp_wait(&s.s_full, i & 1, &s.abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        uint32_t sv[32], dp[32], pp[16], ds[16];
        tmem_ld32(lane_base + C::TM_S + c, sv);
        tmem_ld32(lane_base + C::TM_DP + c, dp);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int m0 = c + e, m1 = c + e + 1;
          const bool v0 = kj <= s.qpos[st][m0], v1 = kj <= s.qpos[st][m1];
          const float p0 =
              v0 ? ex2_approx(__uint_as_float(sv[e]) * p.scale_log2 -
                              s.lse2[st][m0])
                 : 0.f;
          const float p1 =
              v1 ? ex2_approx(__uint_as_float(sv[e + 1]) * p.scale_log2 -
                              s.lse2[st][m1])
                 : 0.f;
          const float d0 = v0 ? p0 * (__uint_as_float(dp[e]) - s.dvec[st][m0]) : 0.f;
          const float d1 =
              v1 ? p1 * (__uint_as_float(dp[e + 1]) - s.dvec[st][m1]) : 0.f;
          pp[e / 2] = pack_bf16x2(p0, p1);
          ds[e / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(lane_base + C::TM_S + c / 2, pp);
        tmem_st16(lane_base + C::TM_DP + c / 2, ds);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full);
    }
    if (ok) {
      ok = warp_wait(&s.acc_ready, 0, &s.abort_flag, p.wait_ns);
      tc_fence_after();
    }
    if (ok && n_q > 0) {
      // the key's gradient page is one of the pages the call writes
      const bool live =
          kj < nk_vis &&
          LSR_IN_BOUNDS(p, p.resp.gpage0[k_resp] + kj / p.ps < p.grad_pages &&
                               g < p.Hkv);
      const size_t base =
          (((size_t)(p.resp.gpage0[k_resp] + kj / p.ps) * p.Hkv + g) * p.ps +
           kj % p.ps) * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t a[32], b[32];
        tmem_ld32(lane_base + C::TM_DV + c, a);
        tmem_ld32(lane_base + C::TM_DK + c, b);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4* pv = reinterpret_cast<float4*>(p.dv + base + c + i);
            float4* pk = reinterpret_cast<float4*>(p.dk + base + c + i);
            float4 x = *pv, y = *pk;
            x.x += __uint_as_float(a[i]);
            x.y += __uint_as_float(a[i + 1]);
            x.z += __uint_as_float(a[i + 2]);
            x.w += __uint_as_float(a[i + 3]);
            y.x += __uint_as_float(b[i]) * p.scale;
            y.y += __uint_as_float(b[i + 1]) * p.scale;
            y.z += __uint_as_float(b[i + 2]) * p.scale;
            y.w += __uint_as_float(b[i + 3]) * p.scale;
            *pv = x;
            *pk = y;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && s.abort_flag) atomicOr(p.status, LSR_DEV_WAIT_TIMEOUT);
}

// =========================================================== launchers

template <int D, int BN>
static cudaError_t launch_dq_t(const AttnParams& p, int grid,
                               const CUtensorMap& mq, const CUtensorMap& mdo,
                               const CUtensorMap& mk, const CUtensorMap& mv,
                               cudaStream_t stream) {
  const size_t smem = sizeof(DqSmem<D, BN>) + 1024;
  cudaError_t e =
      set_smem_limit(reinterpret_cast<const void*>(attn_bwd_dq_kernel<D, BN>),
                     smem);
  if (e != cudaSuccess) return e;
  attn_bwd_dq_kernel<D, BN><<<grid, 192, smem, stream>>>(mq, mdo, mk, mv, p);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const Pool& pl, const BlockGeom& g,
                               const CUtensorMap& mq, const CUtensorMap& mdo,
                               const CUtensorMap& mk, const CUtensorMap& mv,
                               const int32_t* table, const float* lse,
                               const float* D, float* dq_part,
                               cudaStream_t s) {
  AttnParams p = make_params(pl, g, table, lse, D);
  p.o = dq_part;
  const int grid = g.n_qtiles * g.Hkv * (g.num_shards + 1);
  if (g.d == 128 && g.BN == 128) return launch_dq_t<128, 128>(p, grid, mq, mdo, mk, mv, s);
  if (g.d == 128 && g.BN == 64) return launch_dq_t<128, 64>(p, grid, mq, mdo, mk, mv, s);
  if (g.d == 64 && g.BN == 128) return launch_dq_t<64, 128>(p, grid, mq, mdo, mk, mv, s);
  if (g.d == 64 && g.BN == 64) return launch_dq_t<64, 64>(p, grid, mq, mdo, mk, mv, s);
  return cudaErrorInvalidValue;
}

template <int D>
static cudaError_t launch_dkdv_t(const AttnParams& p, int grid, int KL,
                                 const CUtensorMap& mq, const CUtensorMap& mdo,
                                 const CUtensorMap& mk, const CUtensorMap& mv,
                                 cudaStream_t stream) {
  const size_t smem = sizeof(DkvSmem<D>) + 1024;
  cudaError_t e = set_smem_limit(
      reinterpret_cast<const void*>(attn_bwd_dkdv_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<D><<<grid, 192, smem, stream>>>(mq, mdo, mk, mv, p, KL);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dkdv(const Pool& pl, const BlockGeom& g,
                                 const CUtensorMap& mq, const CUtensorMap& mdo,
                                 const CUtensorMap& mk, const CUtensorMap& mv,
                                 const int32_t* table, const float* lse,
                                 const float* D, float* dk, float* dv,
                                 cudaStream_t s) {
  AttnParams p = make_params(pl, g, table, lse, D);
  p.dk = dk;
  p.dv = dv;
  const int grid = g.resp.kt0[g.resp.n] * g.Hkv;
  if (g.d == 128) return launch_dkdv_t<128>(p, grid, g.BN, mq, mdo, mk, mv, s);
  if (g.d == 64) return launch_dkdv_t<64>(p, grid, g.BN, mq, mdo, mk, mv, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsr
