// Backward of replay attention over latent pages (MLA-style resident state,
// the GLM bullet of the LongStraw explainer's "Two incompatible
// architectures, same transaction").  Every query head attends to the same
// latent rows L = [c, r]: keys are L (DL = 192 columns), values are c (the
// first DC = 128 columns).  Queries q~ and their gradient are DL wide; O~
// and dO~ are DC wide.
//
// dq~ pass (latent_bwd_dq_kernel): one CTA = one packed tile of 128 query
// rows (128/Hq positions x Hq heads) against one partial.  Per key tile:
// S = q~ L^T, dP = dO~ c^T, P = exp(S*scale - lse), dS = P * (dP - D), and
// dq~ += dS L.  A 192-column dq~ accumulator leaves no room in the 512 TMEM
// columns for a second S buffer:
//   TMEM: S [0,128), dP [128,256), dq~ [256,448), dS (bf16 pairs) [448,512)
//   - two dS warpgroups, each taking half of a tile's keys, first load all
//     of their S_j and dP_j into registers, which frees both buffers at
//     once;
//   - the MMA order is the K/V dQ pass's: S_{j+1} and dP_{j+1} under one
//     commit, then dq~ += dS_j L_j under another, so dS_j has the time of
//     dq~_{j-1}, S_{j+1} and dP_{j+1} to be ready;
//   - the dS warps write dS_j once the commit after dq~_{j-1} shows that
//     product has read dS_{j-1}.
// The key tile in shared memory serves S, dP (its first two 64-column
// boxes are c) and dq~; it is freed after the dq~ product.
//
// Latent-row gradient pass (latent_bwd_dlat_kernel): one CTA = 128 response
// keys; it walks the query tiles that see them.  S^T = L q~^T and
// dP^T = c dO~^T go to TMEM, P^T and scale*dS^T are written back over them
// as bf16, and one 192-column accumulator takes dS^T q~ (all columns) plus
// P^T dO~ (the first DC columns): dL = dK + [dV, 0].  The softmax scale is
// folded into dS^T before rounding so that both products share the
// accumulator.  No prompt latent row is written: the prompt is
// stop-gradient resident state.
#include <cmath>
#include <climits>
#include "attn_common.cuh"
#include "internal.h"

namespace lsr {

namespace {
constexpr int kDL = 192;  // latent row width (keys, queries, dq~)
constexpr int kDC = 128;  // value width (O~, dO~)
}  // namespace

// =========================================================== dq~ pass
template <int BN>
struct LdqCfg {
  static constexpr int KST = 3;
  static constexpr int Q_BYTES = kTileRows * kDL * 2;
  static constexpr int DO_BYTES = kTileRows * kDC * 2;
  static constexpr int K_BYTES = BN * kDL * 2;
  static constexpr uint32_t TM_S = 0, TM_DP = BN, TM_DQ = 2 * BN,
                            TM_DS = 2 * BN + kDL;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, BN, false, false);
  static constexpr uint32_t ID_DQ = idesc_bf16(128, kDL, false, true);
  static_assert(BN == 128, "key tiles of 128");
  static_assert(TM_DS + BN / 2 <= TMEM_COLS, "TMEM columns");
};

template <int BN>
struct __align__(1024) LdqSmem {
  __nv_bfloat16 q[kTileRows * kDL];
  __nv_bfloat16 dO[kTileRows * kDC];
  __nv_bfloat16 k[LdqCfg<BN>::KST][BN * kDL];
  uint64_t qd_full;
  uint64_t k_full[LdqCfg<BN>::KST];
  uint64_t k_empty[LdqCfg<BN>::KST];
  uint64_t sdp_full, sdp_free, ds_full, dq_ready, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int BN>
__global__ void __launch_bounds__(320, 1)
    latent_bwd_dq_kernel(const __grid_constant__ CUtensorMap mq,
                         const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ CUtensorMap mk,
                         const AttnParams p) {
  using C = LdqCfg<BN>;
  constexpr int KST = C::KST;
  extern __shared__ uint8_t smem_raw[];
  LdqSmem<BN>& s = *reinterpret_cast<LdqSmem<BN>*>(align1024(smem_raw));
  const int warp = warp_id(), lane = lane_id();

  const int qt = blockIdx.x % p.n_qtiles;
  const int part = blockIdx.x / p.n_qtiles;
  const int g = 0;  // one latent head
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
    mbar_init(&s.sdp_full, 1);
    mbar_init(&s.sdp_free, 256);
    mbar_init(&s.ds_full, 256);
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
      }
      __syncwarp();
      mbar_expect_tx_e(&s.qd_full, C::Q_BYTES + C::DO_BYTES);
#pragma unroll
      for (int c = 0; c < kDL / 64; ++c)
        tma_load_3d_e(s.q + c * kTileRows * 64, &mq, &s.qd_full, c * 64, 0, r0);
#pragma unroll
      for (int c = 0; c < kDC / 64; ++c)
        tma_load_3d_e(s.dO + c * kTileRows * 64, &mdo, &s.qd_full, c * 64, 0,
                      r0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int row =
            pool_row(p, kr.page0, (rev ? n_tiles - 1 - j : j) * BN, g);
        const int ks = j % KST;
        if (j >= KST &&
            !warp_wait(&s.k_empty[ks], ((j / KST) & 1) ^ 1, &s.abort_flag, p.wait_ns))
          break;
        mbar_expect_tx_e(&s.k_full[ks], C::K_BYTES);
#pragma unroll
        for (int c = 0; c < kDL / 64; ++c)
          tma_load_2d_e(s.k[ks] + c * BN * 64, &mk, &s.k_full[ks], c * 64, row);
        issued = j + 1;
      }
      // every copy lands before the CTA can exit
      mbar_wait_drain(&s.qd_full, 0);
      for (int t = max(0, issued - KST); t < issued; ++t)
        mbar_wait_drain(&s.k_full[t % KST], (t / KST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n_tiles > 0) {  // the whole warp: one elected lane issues
      bool ok = warp_wait(&s.qd_full, 0, &s.abort_flag, p.wait_ns);
      const uint32_t qa = smem_u32(s.q), da = smem_u32(s.dO);
      // Order: S_0, dP_0; then per step j: S_{j+1} and dP_{j+1} (one commit,
      // which the dS warps wait for), dq~_j (one commit, which releases
      // K_j's ring slot and tells the dS warps that dS_j has been read).
      // The dS warps take S_j and dP_j into registers at once, so S_{j+1}
      // and dP_{j+1} follow without waiting for dS_j, and dS_j has the
      // time of dq~_{j-1}, S_{j+1} and dP_{j+1} to be ready.
      auto issue_s_dp = [&](int i) -> bool {
        const int ks = i % KST;
        if (!warp_wait(&s.k_full[ks], (i / KST) & 1, &s.abort_flag, p.wait_ns))
          return false;
        // the dS warps hold S_{i-1} and dP_{i-1} in registers
        if (i >= 1 &&
            !warp_wait(&s.sdp_free, (i - 1) & 1, &s.abort_flag, p.wait_ns))
          return false;
        tc_fence_after();
        const uint32_t ka = smem_u32(s.k[ks]);
#pragma unroll
        for (int k = 0; k < kDL / 16; ++k)
          mma_ss_e(tm + C::TM_S, sdesc(qa, 16, 1024) + kmaj_step<kTileRows>(k),
                   sdesc(ka, 16, 1024) + kmaj_step<BN>(k), C::ID_S, k > 0);
        // dP = dO~ c^T: c is the first kDC columns of the key tile
#pragma unroll
        for (int k = 0; k < kDC / 16; ++k)
          mma_ss_e(tm + C::TM_DP, sdesc(da, 16, 1024) + kmaj_step<kTileRows>(k),
                   sdesc(ka, 16, 1024) + kmaj_step<BN>(k), C::ID_S, k > 0);
        mma_commit_e(&s.sdp_full);
        return true;
      };
      if (ok) ok = issue_s_dp(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles && !issue_s_dp(j + 1)) break;
        // dq~ += dS_j L_j
        const int ks = j % KST;
        if (!warp_wait(&s.ds_full, j & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t ka = smem_u32(s.k[ks]);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts_e(tm + C::TM_DQ, tm + C::TM_DS + k * 8,
                   sdesc(ka, BN * 128, 1024) + (uint64_t)k * 128, C::ID_DQ,
                   (j > 0 || k > 0) ? 1u : 0u);
        mma_commit_e(&s.k_empty[ks]);
      }
      mma_commit_e(&s.dq_ready);
      mma_commit_e(&s.mma_done);
      mbar_wait_drain(&s.mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ dS warps
    // Two warpgroups: a row's keys are split between warps w and w + 4
    // (both own TMEM lanes 32*(w%4) .. +31), half of every key tile each.
    // dS is elementwise in the keys, so the halves never exchange data.
    // Each thread holds its half of S_j and dP_j (64 + 64 registers).
    constexpr int HK = BN / 2;
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int mrow = quarter * 32 + lane;
    const int r = r0 + mrow / p.G;
    const int h = mrow % p.G;
    const RowInfo ri = row_info(p, k_resp, r);
    const bool valid = ri.valid;
    const int qpos = (valid && kr.causal) ? ri.qpos : INT_MAX;
    const uint32_t lane_base = tm + ((uint32_t)(quarter * 32) << 16);
    const float lse2 = valid ? p.lse[(size_t)h * p.R_b + r] * kLog2e : 0.f;
    const float Dv = valid ? p.Dvec[(size_t)h * p.R_b + r] : 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      // S_j and dP_j are complete
      if (!warp_wait(&s.sdp_full, j & 1, &s.abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[HK], dp[HK];
#pragma unroll
      for (int c = 0; c < HK; c += 32) {
        tmem_ld32(lane_base + C::TM_S + hf * HK + c, sv + c);
        tmem_ld32(lane_base + C::TM_DP + hf * HK + c, dp + c);
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.sdp_free);
      const int kbase = (rev ? n_tiles - 1 - j : j) * BN + hf * HK;
      const bool need_mask = kbase + HK - 1 > qpos;
      uint32_t ds[HK / 2];
#pragma unroll
      for (int c = 0; c < HK; c += 32) {
        if (need_mask)
          dq_chunk<true>(sv + c, dp + c, ds + c / 2, p.scale_log2, lse2, Dv,
                         kbase + c, qpos);
        else
          dq_chunk<false>(sv + c, dp + c, ds + c / 2, p.scale_log2, lse2, Dv,
                          kbase + c, qpos);
      }
      // dq~_{j-1} has read dS_{j-1}: its commit also released K_{j-1}
      if (j >= 1 && !warp_wait(&s.k_empty[(j - 1) % KST], ((j - 1) / KST) & 1,
                               &s.abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < HK / 2; c += 16)
        tmem_st16(lane_base + C::TM_DS + hf * (HK / 2) + c, ds + c);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.ds_full);
    }
    // each half writes its kDL / 2 columns of the row
    constexpr int HW = kDL / 2;
    float* drow = p.o + (((size_t)part * p.R_b + r) * p.Hq + h) * kDL + hf * HW;
    // the dq~ slice row lies inside the workspace's num_shards + 1 slices
    const bool inb = valid && LSR_IN_BOUNDS(p, part <= p.num_shards &&
                                                   r < p.R_b && h < p.Hq);
    if (ok && n_tiles > 0) {
      ok = warp_wait(&s.dq_ready, 0, &s.abort_flag, p.wait_ns);
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int c = 0; c < HW; c += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::TM_DQ + hf * HW + c, o);
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
      for (int c = 0; c < HW; c += 4)
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

// =========================================================== dL pass
struct LdlCfg {
  static constexpr int STAGES = 2;
  static constexpr int QT_BYTES = kTileRows * kDL * 2;
  static constexpr int DOT_BYTES = kTileRows * kDC * 2;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_ACC = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t ID_T = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t ID_ACC_L = idesc_bf16(128, kDL, false, true);
  static constexpr uint32_t ID_ACC_C = idesc_bf16(128, kDC, false, true);
};

struct __align__(1024) LdlSmem {
  __nv_bfloat16 k[128 * kDL];
  __nv_bfloat16 q[LdlCfg::STAGES][kTileRows * kDL];
  __nv_bfloat16 dO[LdlCfg::STAGES][kTileRows * kDC];
  float lse2[LdlCfg::STAGES][kTileRows];
  float dvec[LdlCfg::STAGES][kTileRows];
  int qpos[LdlCfg::STAGES][kTileRows];
  uint64_t kv_full;
  uint64_t q_full[LdlCfg::STAGES];
  uint64_t q_empty[LdlCfg::STAGES];
  uint64_t s_full, p_full, acc_ready, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(192, 1)
    latent_bwd_dlat_kernel(const __grid_constant__ CUtensorMap mq,
                           const __grid_constant__ CUtensorMap mdo,
                           const __grid_constant__ CUtensorMap mk,
                           const AttnParams p, int KL) {
  using C = LdlCfg;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  LdlSmem& s = *reinterpret_cast<LdlSmem*>(align1024(smem_raw));
  const int warp = warp_id(), lane = lane_id();

  const int e = blockIdx.x;
  int k_resp = 0;
  while (k_resp + 1 < p.resp.n && e >= p.resp.kt0[k_resp + 1]) ++k_resp;
  const int key0 = (e - p.resp.kt0[k_resp]) * 128;  // response key index
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
      mbar_expect_tx(&s.kv_full, nsub * KL * kDL * 2);
      for (int sub = 0; sub < nsub; ++sub) {
        const int row = pool_row(p, p.resp.page0[k_resp], key0 + sub * KL, 0);
#pragma unroll
        for (int c = 0; c < kDL / 64; ++c)
          tma_load_2d(s.k + c * 128 * 64 + sub * KL * 64, &mk, &s.kv_full,
                      c * 64, row);
      }
    }
    for (int i = 0; i < n_q; ++i) {
      const int st = i % ST;
      if (i >= ST &&
          !warp_wait(&s.q_empty[st], ((i / ST) & 1) ^ 1, &s.abort_flag, p.wait_ns))
        break;
      const int r0 = (qt0 + i) * p.rows_per_tile;
      if (lane == 0) {
        mbar_expect_tx(&s.q_full[st], C::QT_BYTES + C::DOT_BYTES);
#pragma unroll
        for (int c = 0; c < kDL / 64; ++c)
          tma_load_3d(s.q[st] + c * kTileRows * 64, &mq, &s.q_full[st],
                      c * 64, 0, r0);
#pragma unroll
        for (int c = 0; c < kDC / 64; ++c)
          tma_load_3d(s.dO[st] + c * kTileRows * 64, &mdo, &s.q_full[st],
                      c * 64, 0, r0);
      }
      for (int m = lane; m < kTileRows; m += 32) {
        const int r = r0 + m / p.G;
        const int h = m % p.G;
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
      const uint32_t ka = smem_u32(s.k);
      for (int i = 0; ok && i < n_q; ++i) {
        const int st = i % ST;
        if (!warp_wait(&s.q_full[st], (i / ST) & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t qa = smem_u32(s.q[st]), da = smem_u32(s.dO[st]);
        // S^T = L q~^T (keys on the lanes, query rows as N)
#pragma unroll
        for (int k = 0; k < kDL / 16; ++k) {
          mma_ss_e(tm + C::TM_S, sdesc(ka, 16, 1024) + kmaj_step<128>(k),
                   sdesc(qa, 16, 1024) + kmaj_step<128>(k), C::ID_T, k > 0);
        }
        // dP^T = c dO~^T
#pragma unroll
        for (int k = 0; k < kDC / 16; ++k) {
          mma_ss_e(tm + C::TM_DP, sdesc(ka, 16, 1024) + kmaj_step<128>(k),
                   sdesc(da, 16, 1024) + kmaj_step<128>(k), C::ID_T, k > 0);
        }
        mma_commit_e(&s.s_full);
        if (!warp_wait(&s.p_full, i & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
        // dL += (scale dS^T) q~ over all kDL columns (first product
        // initialises the accumulator) ...
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k)
          mma_ts_e(tm + C::TM_ACC, tm + C::TM_DP + k * 8,
                   sdesc(qa, kTileRows * 128, 1024) + (uint64_t)k * 128,
                   C::ID_ACC_L, (i > 0 || k > 0) ? 1u : 0u);
        // ... and dL[:, :kDC] += P^T dO~
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k)
          mma_ts_e(tm + C::TM_ACC, tm + C::TM_S + k * 8,
                   sdesc(da, kTileRows * 128, 1024) + (uint64_t)k * 128,
                   C::ID_ACC_C, 1u);
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
        for (int e2 = 0; e2 < 32; e2 += 2) {
          const int m0 = c + e2, m1 = c + e2 + 1;
          const bool v0 = kj <= s.qpos[st][m0], v1 = kj <= s.qpos[st][m1];
          const float p0 =
              v0 ? ex2_approx(__uint_as_float(sv[e2]) * p.scale_log2 -
                              s.lse2[st][m0])
                 : 0.f;
          const float p1 =
              v1 ? ex2_approx(__uint_as_float(sv[e2 + 1]) * p.scale_log2 -
                              s.lse2[st][m1])
                 : 0.f;
          const float d0 =
              v0 ? p0 * (__uint_as_float(dp[e2]) - s.dvec[st][m0]) * p.scale
                 : 0.f;
          const float d1 =
              v1 ? p1 * (__uint_as_float(dp[e2 + 1]) - s.dvec[st][m1]) *
                       p.scale
                 : 0.f;
          pp[e2 / 2] = pack_bf16x2(p0, p1);
          ds[e2 / 2] = pack_bf16x2(d0, d1);
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
      // the row's gradient page is one of the pages the call writes
      const bool live =
          kj < nk_vis &&
          LSR_IN_BOUNDS(p, p.resp.gpage0[k_resp] + kj / p.ps < p.grad_pages);
      const size_t base =
          ((size_t)(p.resp.gpage0[k_resp] + kj / p.ps) * p.ps + kj % p.ps) *
          kDL;
#pragma unroll
      for (int c = 0; c < kDL; c += 32) {
        uint32_t a[32];
        tmem_ld32(lane_base + C::TM_ACC + c, a);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4* pd = reinterpret_cast<float4*>(p.dk + base + c + i);
            float4 x = *pd;
            x.x += __uint_as_float(a[i]);
            x.y += __uint_as_float(a[i + 1]);
            x.z += __uint_as_float(a[i + 2]);
            x.w += __uint_as_float(a[i + 3]);
            *pd = x;
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
cudaError_t launch_latent_bwd_dq(const Pool& pl, const BlockGeom& g,
                                 const CUtensorMap& mq, const CUtensorMap& mdo,
                                 const CUtensorMap& mk, const int32_t* table,
                                 const float* lse, const float* D,
                                 float* dq_part, cudaStream_t s) {
  if (!pl.latent || g.d != kDL || g.dv != kDC || g.BN != 128 || g.Hkv != 1)
    return cudaErrorInvalidValue;
  AttnParams p = make_params(pl, g, table, lse, D);
  p.o = dq_part;
  const size_t smem = sizeof(LdqSmem<128>) + 1024;
  static_assert(sizeof(LdqSmem<128>) + 1024 <= 232448,
                "shared memory of one CTA");
  cudaError_t e = set_smem_limit(
      reinterpret_cast<const void*>(latent_bwd_dq_kernel<128>), smem);
  if (e != cudaSuccess) return e;
  const int grid = g.n_qtiles * (g.num_shards + 1);
  latent_bwd_dq_kernel<128><<<grid, 320, smem, s>>>(mq, mdo, mk, p);
  return cudaGetLastError();
}

cudaError_t launch_latent_bwd_dlat(const Pool& pl, const BlockGeom& g,
                                   const CUtensorMap& mq,
                                   const CUtensorMap& mdo,
                                   const CUtensorMap& mk, const int32_t* table,
                                   const float* lse, const float* D,
                                   float* dlat, cudaStream_t s) {
  if (!pl.latent || g.d != kDL || g.dv != kDC || g.Hkv != 1 ||
      g.ps % 128 != 0)
    return cudaErrorInvalidValue;
  AttnParams p = make_params(pl, g, table, lse, D);
  p.dk = dlat;
  const size_t smem = sizeof(LdlSmem) + 1024;
  static_assert(sizeof(LdlSmem) + 1024 <= 232448, "shared memory of one CTA");
  cudaError_t e = set_smem_limit(
      reinterpret_cast<const void*>(latent_bwd_dlat_kernel), smem);
  if (e != cudaSuccess) return e;
  const int grid = g.resp.kt0[g.resp.n];
  if (grid == 0) return cudaSuccess;
  latent_bwd_dlat_kernel<<<grid, 192, smem, s>>>(mq, mdo, mk, p, 128);
  return cudaGetLastError();
}

}  // namespace lsr
