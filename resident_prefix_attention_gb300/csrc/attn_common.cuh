// Device-side pieces shared by the attention kernels.
#pragma once
#include <cstdint>
#include "sm103.cuh"
#include "../../include/lsr.h"
#include "internal.h"

namespace lsr {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  const int32_t* table;  // logical -> physical page
  int* status;           // device status word (LSR_DEV_* bits)
  const float* lse;      // [Hq][R_b] (backward)
  const float* Dvec;     // [Hq][R_b] rowsum(dO * O) (backward)
  float* m;              // forward partial stats [parts][Hq][R_b]
  float* l;
  float* o;              // forward partial outputs / backward dQ partials
  float* dk;             // backward response gradient pages
  float* dv;
  int R_b, Hq, Hkv, G, rows_per_tile, n_qtiles;   // R_b: rows of q in total
  int ps, num_pages, prompt_pages, num_shards;
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  int num_sms;           // CTAs resident at once (one per SM)
  uint64_t wait_ns;      // limit of every pipeline wait (drains excepted)
  int grad_pages;        // gradient pages the call writes (bounds checks)
  RespTable resp;        // which response each row of q belongs to
};

// Bounds checks of the debug build (compiled with -DLSR_DEBUG): a failed
// check sets LSR_DEV_BOUNDS in the status word and the access is skipped.
// In the release build every check is the constant true.
#ifdef LSR_DEBUG
#define LSR_IN_BOUNDS(p, cond) \
  ((cond) ? true : (atomicOr((p).status, LSR_DEV_BOUNDS), false))
#else
#define LSR_IN_BOUNDS(p, cond) true
#endif

// Response owning row r of q (rows never straddle two responses in a CTA).
__device__ __forceinline__ int resp_of_row(const AttnParams& p, int r) {
  int k = 0;
  while (k + 1 < p.resp.n && r >= p.resp.row0[k + 1]) ++k;
  return k;
}

// Real (non-padding) rows of q and their response positions.
struct RowInfo {
  bool valid;
  int qpos;  // response position of the row
};
__device__ __forceinline__ RowInfo row_info(const AttnParams& p, int k, int r) {
  const int local = r - p.resp.row0[k];
  RowInfo ri;
  ri.valid = local >= 0 && local < p.resp.rows[k] && r < p.R_b;
  ri.qpos = p.resp.pos0[k] + local;
  return ri;
}

// Aligns the dynamic shared memory window to 1024 bytes (128-byte swizzle
// atoms must start on a 1024-byte boundary).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                    ~uintptr_t(1023));
}

// Keys of partial `part` for the query tile starting at position r0:
// prompt shards are contiguous logical-page ranges, the last partial holds
// the response keys visible to the tile's last row.
struct KeyRange {
  int page0;   // first logical page
  int nkeys;   // number of keys (multiple of page size for prompt shards)
  bool causal;
};
// `rows` is the number of rows of q the CTA covers from r0, all of them in
// response k.
__device__ __forceinline__ KeyRange key_range(const AttnParams& p, int part,
                                              int k, int r0, int rows) {
  KeyRange kr;
  if (part < p.num_shards) {
    const int a = (int)((long long)part * p.prompt_pages / p.num_shards);
    const int b = (int)((long long)(part + 1) * p.prompt_pages / p.num_shards);
    kr.page0 = a;
    kr.nkeys = (b - a) * p.ps;
    kr.causal = false;
  } else {
    const int end = min(r0 + rows, p.resp.row0[k] + p.resp.rows[k]);
    const int local_last = max(end - 1 - p.resp.row0[k], -1);
    kr.page0 = p.resp.page0[k];
    kr.nkeys = p.resp.pos0[k] + local_last + 1;
    kr.causal = true;
  }
  return kr;
}

// Order of the key tiles a CTA walks.  CTAs sharing one prompt shard run
// side by side, but a group of them can straddle two waves of CTAs; the
// later CTAs of such a group would find the start of the shard evicted
// from L2 by then.  CTAs of odd waves therefore walk prompt shards from
// the end, where the earlier CTAs finished.  The causal response partial
// keeps the forward order (its first tile always holds a visible key).
__device__ __forceinline__ bool walk_reversed(const AttnParams& p,
                                              const KeyRange& kr) {
  return !kr.causal && ((blockIdx.x / max(p.num_sms, 1)) & 1);
}

// Row coordinate of key `key` (relative to the range start) of kv head g in
// the pool viewed as [num_pages * Hkv * ps] rows.  An out-of-range page id
// sets LSR_DEV_BAD_PAGE and is replaced by a row past the end of the pool,
// which the TMA unit fills with zeros.
__device__ __forceinline__ int pool_row(const AttnParams& p, int page0,
                                        int key, int g) {
  const int lp = page0 + key / p.ps;
  int phys = __ldg(p.table + lp);
  if (phys < 0 || phys >= p.num_pages) {
    atomicOr(p.status, LSR_DEV_BAD_PAGE);
    phys = p.num_pages;
  }
  return (phys * p.Hkv + g) * p.ps + key % p.ps;
}

// Wait for a phase without giving up on the shared abort flag (used to
// drain in-flight copies and MMAs before the CTA exits).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar,
                                                uint32_t parity) {
  int never = 0;
  return mbar_wait(bar, parity, &never, 1000000000ull);
}

// Warp-uniform bounded wait: every lane waits, the warp agrees on success.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          uint64_t limit_ns) {
  bool ok = mbar_wait(bar, parity, abort_flag, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// dS = P * (dP - D) for one 32-column chunk, packed to bf16 pairs.
// MASK drops keys after the row's position (response keys only).  The
// arithmetic runs on packed fp32 pairs (the f32x2 forms round each element
// as the scalar forms do), so the pass issues about three instructions per
// element instead of four and a half.
template <bool MASK>
__device__ __forceinline__ void dq_chunk(const uint32_t* sv, const uint32_t* dp,
                                         uint32_t* ds, float scale_log2,
                                         float lse2, float Dv, int key0,
                                         int qpos) {
  const uint64_t sc2 = f32x2(scale_log2, scale_log2);
  const uint64_t nl2 = f32x2(-lse2, -lse2);
  const uint64_t nd2 = f32x2(-Dv, -Dv);
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float t0, t1;
    f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[e]),
                                __uint_as_float(sv[e + 1])),
                          sc2, nl2),
                t0, t1);
    const uint64_t g2 = add_f32x2(
        f32x2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2);
    float d0, d1;
    f32x2_split(mul_f32x2(f32x2(ex2_approx(t0), ex2_approx(t1)), g2), d0, d1);
    if (MASK) {
      if (key0 + e > qpos) d0 = 0.f;
      if (key0 + e + 1 > qpos) d1 = 0.f;
    }
    ds[e / 2] = pack_bf16x2(d0, d1);
  }
}


// Kernel parameters of a validated backward launch.
inline AttnParams make_params(const Pool& pl, const BlockGeom& g,
                              const int32_t* table, const float* lse,
                              const float* D) {
  AttnParams p{};
  p.table = table;
  p.status = pl.dev_status;
  p.lse = lse;
  p.Dvec = D;
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
  // pages of the response gradient the call writes: every response's
  // visible keys, from its first gradient page
  p.grad_pages = 0;
  for (int k = 0; k < g.resp.n; ++k) {
    const int end =
        g.resp.gpage0[k] + (g.resp.pos0[k] + g.resp.rows[k] + g.ps - 1) / g.ps;
    if (end > p.grad_pages) p.grad_pages = end;
  }
  return p;
}

}  // namespace lsr
