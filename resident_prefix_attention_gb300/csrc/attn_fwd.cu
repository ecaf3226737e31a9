// Forward partials of replay attention.  One CTA = two tiles of 128 packed
// query rows (the G query heads of one kv head times 128/G positions each)
// against one partial: a prompt shard or the response keys.  For every key
// tile j and query tile t: S_t = Q_t K_j^T on the tensor cores into TMEM,
// online softmax in registers (one thread per row), P_t (bf16) written back
// over the second half of S_t's columns in TMEM, and O_t += P_t V_j with P_t
// as the TMEM-resident A operand.  The result is the partial's
// (m, l, O / l) -- the rank-local softmax statistics that the LongStraw
// explainer ("Two incompatible architectures, same transaction", Qwen
// bullet) composes into the exact output.
//
// Warp roles (384 threads, three warpgroups): warp 0 issues TMA loads (both
// Q tiles once, then K and V pages through the page table into one ring, in
// the order K_0, V_0, K_1, ...), warp 1 allocates TMEM and issues
// tcgen05.mma (the whole warp runs the issue loop, an elected lane issues),
// warps 2-3 idle; warps 4-7 and 8-11 are the softmax warpgroups of query
// tiles 0 and 1 (warp w owns TMEM lanes 32*(w%4) .. +31).  The first
// warpgroup hands registers to the softmax warpgroups (setmaxnreg), which
// hold a whole 128-key row of S in registers.  The MMA order S0_j, S1_j, PV0_j, S0_j+1, PV1_j, S1_j+1,
// ... keeps one tile's products queued while the other tile's softmax runs,
// and each K/V tile in shared memory serves both query tiles.
//
// Latent pages (LAT = true): one latent row [c, r] per position is both the
// key (all DQK columns) and, through its first DV columns, the value, for
// every query head (MLA-style resident state, the GLM bullet of the same
// section).  No V tile is loaded: the key tile's c part feeds the PV
// products.  It sits in the ring until both PV products have read it,
// while the r part sits in a ring of its own that frees as soon as both S
// products have run.
#include <cmath>
#include <climits>
#include "attn_common.cuh"
#include "internal.h"

namespace lsr {

// DQK: width of queries and keys; DV: width of values and outputs.
template <int DQK, int DV, int BN, bool LAT>
struct FwdCfg {
  static constexpr bool kStd128 = DQK == 128 && BN == 128;
  // One ring of key-tile slots.  K/V pages: K_j and V_j are ring tiles 2j
  // and 2j+1 (DQK == DV, so both fit a slot), loaded and released in that
  // order, so both kinds of tile get the same lead over their use.  Latent
  // pages: ring tile j holds the first DV columns of key tile j (c, which
  // is also V_j); its last DQK - DV columns (r) go to a second ring of NSR
  // slots.  The r part is free once both S products have run, the c part
  // only after both PV products, so the split gives the c part a third
  // slot of lead in the same shared memory.
  static constexpr int NS = LAT ? 3 : (kStd128 ? 5 : 8);
  static constexpr int NSR = 2;
  static constexpr int RING_COLS = LAT ? DV : DQK;  // columns of a ring slot
  static constexpr int R_COLS = LAT ? DQK - DV : 64;  // of an r slot
  static constexpr int Q_BYTES = kTileRows * DQK * 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr uint32_t TM_O = 2 * BN;  // O_t at TM_O + t * DV
  static constexpr uint32_t TMEM_COLS = (2 * BN + 2 * DV <= 256) ? 256 : 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, BN, false, false);
  static constexpr uint32_t ID_PV = idesc_bf16(128, DV, false, true);
  static constexpr int THREADS = 384;
  // Registers per thread: the block launches at kLaunchRegs (the cap for
  // 384 threads); the first warpgroup drops to kRegsIssue and the two
  // softmax warpgroups rise to kRegsSoftmax, which adds up to the launch
  // total exactly.
  static constexpr int kLaunchRegs = 168;
  static constexpr int kRegsIssue = 120;
  static constexpr int kRegsSoftmax = 192;
  static_assert(128 * kRegsIssue + 256 * kRegsSoftmax <=
                    THREADS * kLaunchRegs,
                "register shares exceed the block's launch total");
  static_assert(2 * BN + 2 * DV <= 512, "TMEM holds two S and two O tiles");
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= DQK, "box widths");
  static_assert(LAT || DV == DQK, "K and V tiles share the ring slots");
};

// Ring tile of K_j and of V_j.
template <bool LAT>
__device__ __forceinline__ int ring_k(int j) { return LAT ? j : 2 * j; }
template <bool LAT>
__device__ __forceinline__ int ring_v(int j) { return LAT ? j : 2 * j + 1; }

template <int DQK, int DV, int BN, bool LAT>
struct __align__(1024) FwdSmem {
  using C = FwdCfg<DQK, DV, BN, LAT>;
  __nv_bfloat16 q[2][kTileRows * DQK];
  __nv_bfloat16 ring[C::NS][BN * C::RING_COLS];
  __nv_bfloat16 rring[LAT ? C::NSR : 1][LAT ? BN * C::R_COLS : 64];
  uint64_t q_full;
  uint64_t empty[C::NS];
  uint64_t r_empty[C::NSR];  // latent pages: the r slots
  // K/V pages: group 0 is K_0, group g > 0 is V_{g-1} and K_g (the ring
  // tiles between two S products); group g lands on step_full[g % 3].
  // Latent pages: both parts of key tile g land on step_full[g % 3].
  uint64_t step_full[3];
  uint64_t s_full[2], p_full[2], o_final, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// S = Q K^T over DQK/16 k-steps; qd, kd: descriptors of the two tiles.
// The key tile's first KC columns are at kd, the rest (latent pages: the r
// part, in its own ring) at kd2.
template <int DQK, int KC, int BN, uint32_t ID>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t qd,
                                        uint64_t kd, uint64_t kd2) {
#pragma unroll
  for (int k = 0; k < DQK / 16; ++k)
    mma_ss_e(d_tmem, qd + kmaj_step<kTileRows>(k),
             k < KC / 16 ? kd + kmaj_step<BN>(k)
                         : kd2 + kmaj_step<BN>(k - KC / 16),
             ID, k > 0);
}

// O += P V with V the first DV columns of a [BN][.] tile stored as 64-column
// boxes (the ring slot of V_j, or of a latent key tile): vd describes it as
// an MN-major B operand (16 key rows of 128 bytes per k-step).
template <int BN, uint32_t ID>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem,
                                         uint64_t vd, bool first) {
#pragma unroll
  for (int k = 0; k < BN / 16; ++k)
    mma_ts_e(o_tmem, p_tmem + k * 8, vd + (uint64_t)k * 128, ID,
             (!first || k > 0) ? 1u : 0u);
}

// One pass of the softmax over a row of S (x: the raw logits, masked keys at
// -inf): P = 2^(x * scale_log2 - mu) in packed pairs, written as bf16 into
// the BN/2 TMEM columns that start at tmem_s, with the sum of P as computed
// (s_exact, for lse) and of the bf16 P the product sees (s_rnd, for
// normalising O).  Per pair of keys the pass issues one packed FMA, two
// exponentials, one packed conversion, one packed add and two adds of a
// bf16 half into fp32.
template <int BN>
__device__ __forceinline__ void p_pass(const float (&x)[BN], float scale_log2,
                                       float mu, uint32_t tmem_s,
                                       float& s_exact, float& s_rnd) {
  const uint64_t sc2 = f32x2(scale_log2, scale_log2);
  const uint64_t nm2 = f32x2(-mu, -mu);
  // P goes out every 16 packed columns; two partial sums of each kind keep
  // the add chains short
  uint64_t r2[2] = {0ull, 0ull};
  float qa[2] = {0.f, 0.f}, qb[2] = {0.f, 0.f};
#pragma unroll
  for (int qq = 0; qq < BN / 32; ++qq) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const int cc = qq * 32 + c;
      float t0, t1;
      f32x2_split(fma_f32x2(f32x2(x[cc], x[cc + 1]), sc2, nm2), t0, t1);
      const float p0 = ex2_approx(t0);
      const float p1 = ex2_approx(t1);
      const uint32_t pr = pack_bf16x2(p0, p1);
      const int a = (c >> 1) & 1;
      r2[a] = add_f32x2(r2[a], f32x2(p0, p1));
      qa[a] = add_bf16_lo(pr, qa[a]);
      qb[a] = add_bf16_hi(pr, qb[a]);
      pk[c / 2] = pr;
    }
    tmem_st16(tmem_s + qq * 16, pk);
  }
  float s0, s1;
  f32x2_split(add_f32x2(r2[0], r2[1]), s0, s1);
  s_exact = s0 + s1;
  s_rnd = (qa[0] + qb[0]) + (qa[1] + qb[1]);
}

// Largest raw logit of a row of S, in independent three-input chains.
template <int BN>
__device__ __forceinline__ float row_max(const float (&x)[BN]) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < BN; c += 2)
    m4[(c >> 1) & 3] = max3f(m4[(c >> 1) & 3], x[c], x[c + 1]);
  return fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
}

template <int DQK, int DV, int BN, bool LAT>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq,
                    const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv,
                    const AttnParams p) {
  using C = FwdCfg<DQK, DV, BN, LAT>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<DQK, DV, BN, LAT>& s =
      *reinterpret_cast<FwdSmem<DQK, DV, BN, LAT>*>(align1024(smem_raw));
  const int warp = warp_id(), lane = lane_id();

  const int n_pairs = (p.n_qtiles + 1) >> 1;
  int u = blockIdx.x;
  const int pair = u % n_pairs;
  u /= n_pairs;
  const int g = u % p.Hkv;
  const int part = u / p.Hkv;
  const int r0 = pair * 2 * p.rows_per_tile;
  const int k_resp = resp_of_row(p, r0);
  const KeyRange kr = key_range(p, part, k_resp, r0, 2 * p.rows_per_tile);
  const int n_tiles = (kr.nkeys + BN - 1) / BN;
  const bool rev = walk_reversed(p, kr);

  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < NS; ++i) mbar_init(&s.empty[i], 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s.s_full[t], 1);
      mbar_init(&s.p_full[t], 128);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&s.step_full[i], 1);
    for (int i = 0; i < C::NSR; ++i) mbar_init(&s.r_empty[i], 1);
    mbar_init(&s.o_final, 1);
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
    regs_dec<C::kRegsIssue>();
    if (n_tiles > 0) {  // the whole warp: one elected lane issues
      if (lane == 0) {
        prefetch_tmap(&mq);
        prefetch_tmap(&mk);
        if (!LAT) prefetch_tmap(&mv);
      }
      __syncwarp();
      mbar_expect_tx_e(&s.q_full, 2 * C::Q_BYTES);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_3d_e(s.q[t] + c * kTileRows * 64, &mq, &s.q_full, c * 64,
                        g * p.G, r0 + t * p.rows_per_tile);
      int issued = 0;  // ring tiles issued (latent) or key tiles (K/V)
      for (int j = 0; j < n_tiles; ++j) {
        const int row = pool_row(p, kr.page0, (rev ? n_tiles - 1 - j : j) * BN, g);
        const int tk = ring_k<LAT>(j), sk = tk % NS;
        if (tk >= NS &&
            !warp_wait(&s.empty[sk], ((tk / NS) & 1) ^ 1, &s.abort_flag, p.wait_ns))
          break;
        if (LAT) {
          // c part into ring slot sk, r part into r slot j % NSR
          const int sr = j % C::NSR;
          if (j >= C::NSR &&
              !warp_wait(&s.r_empty[sr], ((j / C::NSR) & 1) ^ 1, &s.abort_flag,
                         p.wait_ns))
            break;
          uint64_t* bar = &s.step_full[j % 3];
          mbar_expect_tx_e(bar, C::K_BYTES);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_2d_e(s.ring[sk] + c * BN * 64, &mk, bar, c * 64, row);
#pragma unroll
          for (int c = 0; c < C::R_COLS / 64; ++c)
            tma_load_2d_e(s.rring[sr] + c * BN * 64, &mk, bar, DV + c * 64,
                          row);
          issued = j + 1;
          continue;
        }
        // group j: V_{j-1} (issued with it) and K_j
        uint64_t* bar = &s.step_full[j % 3];
        if (j > 0) {
          const int tv = ring_v<LAT>(j - 1), sv = tv % NS;
          if (tv >= NS &&
              !warp_wait(&s.empty[sv], ((tv / NS) & 1) ^ 1, &s.abort_flag, p.wait_ns))
            break;
        }
        mbar_expect_tx_e(bar, C::K_BYTES + (j > 0 ? C::V_BYTES : 0));
        if (j > 0) {
          const int sv = ring_v<LAT>(j - 1) % NS;
          const int rowv = pool_row(p, kr.page0, (rev ? n_tiles - j : j - 1) * BN, g);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_2d_e(s.ring[sv] + c * BN * 64, &mv, bar, c * 64, rowv);
        }
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_2d_e(s.ring[sk] + c * BN * 64, &mk, bar, c * 64, row);
        issued = j + 1;
      }
      // the last group: V_{n-1} alone
      if (!LAT && issued == n_tiles && n_tiles > 0) {
        const int j = n_tiles;
        const int tv = ring_v<LAT>(j - 1), sv = tv % NS;
        if (tv < NS ||
            warp_wait(&s.empty[sv], ((tv / NS) & 1) ^ 1, &s.abort_flag, p.wait_ns)) {
          uint64_t* bar = &s.step_full[j % 3];
          mbar_expect_tx_e(bar, C::V_BYTES);
          const int rowv = pool_row(p, kr.page0, (rev ? 0 : j - 1) * BN, g);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_2d_e(s.ring[sv] + c * BN * 64, &mv, bar, c * 64, rowv);
          issued = j + 1;
        }
      }
      // Every copy lands before the CTA can exit.  After a normal run the
      // consumers have already waited for all of them; after an abort
      // (any role's wait ran out) this keeps late copies out of the shared
      // memory of whatever CTA runs next on the SM.
      mbar_wait_drain(&s.q_full, 0);
      for (int t = max(0, issued - 3); t < issued; ++t)
        mbar_wait_drain(&s.step_full[t % 3], (t / 3) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    regs_dec<C::kRegsIssue>();
    if (n_tiles > 0) {  // the whole warp: one elected lane issues
      const uint64_t qd0 = sdesc(smem_u32(s.q[0]), 16, 1024);
      const uint64_t qd1 = sdesc(smem_u32(s.q[1]), 16, 1024);
      // latent: key tile j has landed; K/V pages: group j (V_{j-1}, K_j)
      auto tile_wait = [&](int j) -> bool {
        return warp_wait(&s.step_full[j % 3], (j / 3) & 1, &s.abort_flag,
                         p.wait_ns);
      };
      // descriptors of key tile j's parts (the r slot only for latent pages)
      auto kdesc = [&](int j) {
        return sdesc(smem_u32(s.ring[ring_k<LAT>(j) % NS]), 16, 1024);
      };
      auto rdesc = [&](int j) {
        return sdesc(smem_u32(s.rring[LAT ? j % C::NSR : 0]), 16, 1024);
      };
      constexpr int KC = C::RING_COLS;
      bool ok = warp_wait(&s.q_full, 0, &s.abort_flag, p.wait_ns) &&
                tile_wait(0);
      if (ok) {
        tc_fence_after();
        const uint64_t kd = kdesc(0), kd2 = rdesc(0);
        issue_s<DQK, KC, BN, C::ID_S>(tm, qd0, kd, kd2);
        mma_commit_e(&s.s_full[0]);
        issue_s<DQK, KC, BN, C::ID_S>(tm + BN, qd1, kd, kd2);
        mma_commit_e(&s.s_full[1]);
      }
      // Two commits per key tile, one per query tile's S.  The softmax
      // warps learn from them that the products issued earlier have run
      // too: the previous PV of their tile (before an O rescale) and, for
      // the second tile, every product that read K_j and V_{j-1} (they
      // release those ring slots).
      for (int j = 0; ok && j < n_tiles; ++j) {
        const bool more = j + 1 < n_tiles;
        const int tv = ring_v<LAT>(j), sv = tv % NS;
        // V_j and K_{j+1} have landed (waited for before P0, so that PV0 and
        // S0 go out back to back: a wait between the products of a group
        // leaves the tensor pipe idle)
        if (!LAT && !tile_wait(j + 1)) break;
        // O0 += P0 V_j, then S0 of the next key tile over P0's columns
        if (!warp_wait(&s.p_full[0], j & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint64_t vd = sdesc(smem_u32(s.ring[sv]), BN * 128, 1024);
        issue_pv<BN, C::ID_PV>(tm + C::TM_O, tm + BN / 2, vd, j == 0);
        if (more) {
          if (LAT) {
            if (!tile_wait(j + 1)) break;
            tc_fence_after();
          }
          issue_s<DQK, KC, BN, C::ID_S>(tm, qd0, kdesc(j + 1), rdesc(j + 1));
          mma_commit_e(&s.s_full[0]);
        }
        // O1 += P1 V_j, then S1 of the next key tile
        if (!warp_wait(&s.p_full[1], j & 1, &s.abort_flag, p.wait_ns)) break;
        tc_fence_after();
        issue_pv<BN, C::ID_PV>(tm + C::TM_O + DV, tm + BN + BN / 2, vd,
                               j == 0);
        // a latent key tile is also V_j: both PV products have read it
        if (LAT) mma_commit_e(&s.empty[sv]);
        if (more) {
          issue_s<DQK, KC, BN, C::ID_S>(tm + BN, qd1, kdesc(j + 1),
                                        rdesc(j + 1));
          mma_commit_e(&s.s_full[1]);
        }
      }
      // A single-phase barrier for the epilogue (the per-tile barriers are
      // reused every key tile).
      mma_commit_e(&s.o_final);
      mma_commit_e(&s.mma_done);
      mbar_wait_drain(&s.mma_done, 0);
    }
  } else if (warp < 4) {
    regs_dec<C::kRegsIssue>();  // idle warps of the first warpgroup
  } else {
    // ------------------------------------------------------------ softmax
    regs_inc<C::kRegsSoftmax>();
    const int t = (warp - 4) >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;
    const int mrow = quarter * 32 + lane;
    const int r = r0 + t * p.rows_per_tile + mrow / p.G;
    const int h = g * p.G + mrow % p.G;
    const RowInfo ri = row_info(p, k_resp, r);
    const bool valid = ri.valid;
    const int qpos = (valid && kr.causal) ? ri.qpos : INT_MAX;
    const uint32_t lane_base = tm + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = t * BN, o_col = C::TM_O + t * DV;
    // mu: the reference (log2 units) that P, lsum and O are taken against:
    // the scaled logit of the largest key seen when it was last set, rounded
    // up to an integer.  A tile whose sum of P exceeds 2^8 (which every tile
    // with a key more than 2^8 times the reference's weight does, and the
    // first tile, where mu = -inf, does through inf) sets it again from the
    // tile's max and computes P a second time; otherwise mu stays, so mu
    // lies at most 8 below the row max (and at most 1 above it) and every P
    // is at most 2^8.  lsum: sum of P as computed (gives
    // lse); lrnd: sum of the bf16 P the product uses (normalises O, so every
    // key weighs the same in the numerator and the denominator, and a row
    // dominated by one key returns that key's V whatever its P rounds to).
    float mu = -INFINITY, lsum = 0.f, lrnd = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(&s.s_full[t], j & 1, &s.abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (LAT && t == 1 && threadIdx.x == 256) {
        // S1_j has run, and with it S0_j: both have read key tile j's r part
        mbar_arrive(&s.r_empty[j % C::NSR]);
      }
      if (!LAT && t == 1 && threadIdx.x == 256) {
        // S1_j has run, and with it every product issued before it: both
        // S products of K_j and both PV products of V_{j-1}
        mbar_arrive(&s.empty[ring_k<LAT>(j) % NS]);
        if (j > 0) mbar_arrive(&s.empty[ring_v<LAT>(j - 1) % NS]);
      }
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN; c += 32)
        tmem_ld32(lane_base + s_col + c, reinterpret_cast<uint32_t*>(x) + c);
      tmem_ld_wait();
      const int kbase = (rev ? n_tiles - 1 - j : j) * BN;
      if (kbase + BN - 1 > qpos) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (kbase + c > qpos) x[c] = -INFINITY;
      }
      // P against the current reference.  P goes over the second half of
      // S's columns (the PV product reads it there), so S of the first BN/2
      // keys survives for a second pass.
      float ls_t, lr_t;
      p_pass<BN>(x, p.scale_log2, mu, lane_base + s_col + BN / 2, ls_t,
                 lr_t);
      const bool rescale = __any_sync(0xffffffffu, !(ls_t <= 256.f));
      float alpha = 1.f;
      if (rescale) {
        tmem_st_wait();  // the first pass's stores land before the second's
        float y[BN];
#pragma unroll
        for (int c = 0; c < BN / 2; c += 32)
          tmem_ld32(lane_base + s_col + c, reinterpret_cast<uint32_t*>(y) + c);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < BN / 2; ++c)
          if (kbase + c > qpos) y[c] = -INFINITY;
#pragma unroll
        for (int c = BN / 2; c < BN; ++c) y[c] = x[c];
        // an integer reference: rescales are exact powers of two, and P's
        // mantissa does not depend on when the reference was raised (so the
        // result does not depend on the order the key tiles are walked in)
        const float mu_new = fmaxf(mu, ceilf(row_max<BN>(y) * p.scale_log2));
        if (mu_new != mu) {
          alpha = ex2_approx(mu - mu_new);
          mu = mu_new;
          lsum *= alpha;
          lrnd *= alpha;
        }
        p_pass<BN>(y, p.scale_log2, mu, lane_base + s_col + BN / 2, ls_t,
                   lr_t);
      }
      lsum += ls_t;
      lrnd += lr_t;
      if (j > 0 && rescale) {
        // S_t of this tile was issued after PV_t of the previous one, so
        // the s_full wait above has seen that product complete
#pragma unroll
        for (int c = 0; c < DV; c += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + o_col + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + o_col + c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[t]);
    }
    tmem_st_wait();  // an aborted tile's stores complete before TMEM is freed
    if (ok && n_tiles > 0) {
      ok = warp_wait(&s.o_final, 0, &s.abort_flag, p.wait_ns);
      tc_fence_after();
      if (ok) {
        const float inv = 1.f / lrnd;
        const bool inb =
            valid && LSR_IN_BOUNDS(p, part <= p.num_shards && r < p.R_b &&
                                          h < p.Hq);
        float* orow = p.o + (((size_t)part * p.R_b + r) * p.Hq + h) * DV;
#pragma unroll
        for (int c = 0; c < DV; c += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + o_col + c, o);
          tmem_ld_wait();
          if (inb) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 f = make_float4(__uint_as_float(o[i]) * inv,
                                     __uint_as_float(o[i + 1]) * inv,
                                     __uint_as_float(o[i + 2]) * inv,
                                     __uint_as_float(o[i + 3]) * inv);
              *reinterpret_cast<float4*>(orow + c + i) = f;
            }
          }
        }
        if (inb) {
          // (m, l): the reference in natural-log units and the sum of
          // exp(logit - m) against it
          const size_t si = ((size_t)part * p.Hq + h) * p.R_b + r;
          p.m[si] = mu * kLn2;
          p.l[si] = lsum;
        }
      }
    } else if (n_tiles == 0 && valid &&
               LSR_IN_BOUNDS(p, part <= p.num_shards && r < p.R_b &&
                                    h < p.Hq)) {
      float* orow = p.o + (((size_t)part * p.R_b + r) * p.Hq + h) * DV;
      for (int c = 0; c < DV; c += 4)
        *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      const size_t si = ((size_t)part * p.Hq + h) * p.R_b + r;
      p.m[si] = -INFINITY;
      p.l[si] = 0.f;
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

template <int DQK, int DV, int BN, bool LAT>
static cudaError_t launch_fwd_t(const AttnParams& p, int grid,
                                const CUtensorMap& mq, const CUtensorMap& mk,
                                const CUtensorMap& mv, cudaStream_t stream) {
  const size_t smem = sizeof(FwdSmem<DQK, DV, BN, LAT>) + 1024;
  static_assert(sizeof(FwdSmem<DQK, DV, BN, LAT>) + 1024 <= 232448,
                "shared memory of one CTA");
  cudaError_t e = set_smem_limit(
      reinterpret_cast<const void*>(attn_fwd_kernel<DQK, DV, BN, LAT>), smem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<DQK, DV, BN, LAT>
      <<<grid, FwdCfg<DQK, DV, BN, LAT>::THREADS, smem, stream>>>(mq, mk, mv,
                                                                  p);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const Pool& pl, const BlockGeom& g,
                            const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const int32_t* table,
                            float* m, float* l, float* o, cudaStream_t s) {
  AttnParams p{};
  p.table = table;
  p.status = pl.dev_status;
  p.m = m;
  p.l = l;
  p.o = o;
  p.R_b = g.R_b;
  p.Hq = g.Hq;
  p.Hkv = g.Hkv;
  p.G = g.G;
  p.rows_per_tile = g.rows_per_tile;
  p.n_qtiles = g.n_qtiles;
  p.ps = g.ps;
  p.num_pages = pl.num_pages;
  p.prompt_pages = g.prompt_pages;
  p.num_shards = g.num_shards;
  p.resp = g.resp;
  p.scale = g.scale;
  p.scale_log2 = g.scale * kLog2e;
  p.num_sms = num_sms();
  p.wait_ns = pl.wait_ns;
  const int n_pairs = (g.n_qtiles + 1) / 2;
  const int grid = n_pairs * g.Hkv * (g.num_shards + 1);
  if (pl.latent) {
    if (g.d == 192 && g.dv == 128 && g.BN == 128)
      return launch_fwd_t<192, 128, 128, true>(p, grid, mq, mk, mv, s);
    return cudaErrorInvalidValue;
  }
  if (g.d == 128 && g.BN == 128)
    return launch_fwd_t<128, 128, 128, false>(p, grid, mq, mk, mv, s);
  if (g.d == 128 && g.BN == 64)
    return launch_fwd_t<128, 128, 64, false>(p, grid, mq, mk, mv, s);
  if (g.d == 64 && g.BN == 128)
    return launch_fwd_t<64, 64, 128, false>(p, grid, mq, mk, mv, s);
  if (g.d == 64 && g.BN == 64)
    return launch_fwd_t<64, 64, 64, false>(p, grid, mq, mk, mv, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsr
