// Host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lsr {

// One attention CTA handles 128 packed query rows: 128/G response positions
// times the G query heads that share one kv head.
constexpr int kTileRows = 128;

// Default limit of an in-kernel pipeline wait: 4 s.
constexpr uint64_t kDefaultWaitNs = 4000000000ull;

// A K/V pool holds [num_pages][Hkv][page_size][head_dim] K and V pages.  A
// latent pool holds one row [c, r] of width head_dim per position
// ([num_pages][1][page_size][head_dim]); it is the key, and its first v_dim
// columns are the value (k_pages == v_pages).
struct Pool {
  int num_pages, page_size, num_kv_heads, head_dim;
  void* k_pages;
  void* v_pages;
  int* dev_status;
  int v_dim;    // value width: head_dim for K/V pools, d_c for latent pools
  bool latent;
  // limit of the attention kernels' pipeline waits (lsr_pool_set_wait_limit)
  uint64_t wait_ns = kDefaultWaitNs;
};

// Query blocks of one or more responses stacked along the rows of q.
// Response k owns rows [row0[k], row0[k+1]); the first rows[k] are real and
// the rest pad to a whole pair of query tiles, so no CTA mixes responses.
// Its row row0[k]+i sits at response position pos0[k]+i, its key j at
// logical page page0[k] + j/page_size, and its dK/dV at gradient page
// gpage0[k] + j/page_size.  kt0 is the prefix count of 128-key tiles
// (pos0[k] + rows[k] visible keys) for the dK/dV grid.
constexpr int kMaxResp = 32;
struct RespTable {
  int n;
  int row0[kMaxResp + 1];
  int rows[kMaxResp];
  int pos0[kMaxResp];
  int page0[kMaxResp];
  int gpage0[kMaxResp];
  int kt0[kMaxResp + 1];
};

// Geometry of one replay launch, validated by the API layer.
struct BlockGeom {
  int Hq, Hkv, G;          // G = Hq / Hkv query heads per kv head
  int d, ps, BN;           // query/key width, page size, key-tile rows
  int dv;                  // value (and output) width
  int R_b, resp_pos0;
  int prompt_pages;        // P / page_size
  int num_shards;
  int rows_per_tile;       // 128 / G response positions per query tile
  int n_qtiles;            // ceil(R_b / rows_per_tile)
  float scale;
  RespTable resp;          // responses stacked in q (one for a plain block)
};

// Builds a 2D bf16 tensor map {inner, rows} with box {64, box_rows},
// 128-byte swizzle.  Returns false (and sets the error text) on failure.
bool make_map_2d(CUtensorMap* map, const void* base, uint64_t inner,
                 uint64_t rows, uint32_t box_rows);
// 3D bf16 map {d, Hq, R} with box {64, G, 128/G} for packed GQA rows.
bool make_map_q(CUtensorMap* map, const void* base, int d, int Hq, int R,
                int G);

void set_error(const char* fmt, ...);

// Streaming multiprocessors of the current device (cached).
int num_sms();

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device).  Thread-safe.
cudaError_t set_smem_limit(const void* kernel, size_t bytes);

// Counts a launch of kernel `kernel` (an LSR_K_* id) and, while profiling
// is enabled, brackets it with CUDA events recorded on `s`.
class ProfScope {
 public:
  ProfScope(int kernel, cudaStream_t s);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  int k_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace lsr

#include "../../include/lsr.h"

namespace lsr {

// Validates a block replay call on a pool of the expected kind (K/V pages
// when latent is false, latent pages when true) and fills the geometry.
lsr_status block_geom(const struct ::lsr_pool* pool, int Hq, int R_b, int P,
                      int resp_pos0, int table_len, int num_shards,
                      float scale, bool latent, BlockGeom* g);

// The dQ passes split every prompt shard of the forward in kBwdSplit
// contiguous halves.  A (kv head, shard) key stream is read by all the
// query tiles of a kv head, and a wave of CTAs spans about one stream; at
// 2M positions a forward shard's K/V (134 MB per kv head) is larger than
// L2, a half fits.  The dQ slices are internal workspace, so the split
// changes no output, only the summation order of dQ.
constexpr int kBwdSplit = 2;
inline int bwd_shards(int num_shards) { return kBwdSplit * num_shards; }

// Launch sequences shared by the entry points (arguments validated).
// bwd_ws_bytes: the dQ slices (bwd_shards(num_shards) + 1 partials of
// R_b x Hq x d fp32) and the row dots D.
size_t bwd_ws_bytes(int num_shards, int Hq, int R_b, int d);
lsr_status run_fwd(const struct ::lsr_pool* pool, const BlockGeom& g,
                   const void* q, const int32_t* table, float* m, float* l,
                   float* o_part, cudaStream_t s);
lsr_status run_bwd(const struct ::lsr_pool* pool, const BlockGeom& g,
                   const void* q, const float* o, const void* dO,
                   const float* lse, const int32_t* table, float* dq,
                   float* dk, float* dv, void* workspace, cudaStream_t s);
// Latent pages: preprocess (width 128), dq~ pass, dq~ reduction and the
// response latent-row gradient; q is 192 wide, o and dO 128 wide.
lsr_status run_latent_bwd(const struct ::lsr_pool* pool, const BlockGeom& g,
                          const void* q, const float* o, const void* dO,
                          const float* lse, const int32_t* table, float* dq,
                          float* dlat, void* workspace, cudaStream_t s);

// Launchers (return a CUDA error code; 0 = launched).
cudaError_t launch_write_pages(const Pool& p, const void* k, const void* v,
                               int T, int pos0, const int32_t* table,
                               int table_len, cudaStream_t s);
cudaError_t launch_lse_merge(const float* m, const float* l, const float* o,
                             int parts, int Hq, int R_b, int d, float* out,
                             float* lse, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const float* o, const void* dO, int Hq,
                                  int R_b, int d, float* D, cudaStream_t s);
cudaError_t launch_dq_reduce(const float* parts, int nparts, size_t n,
                             float* dq, cudaStream_t s);
cudaError_t launch_attn_fwd(const Pool& p, const BlockGeom& g,
                            const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const int32_t* table,
                            float* m, float* l, float* o, cudaStream_t s);
cudaError_t launch_attn_bwd_dq(const Pool& p, const BlockGeom& g,
                               const CUtensorMap& mq, const CUtensorMap& mdo,
                               const CUtensorMap& mk, const CUtensorMap& mv,
                               const int32_t* table, const float* lse,
                               const float* D, float* dq_part,
                               cudaStream_t s);
cudaError_t launch_attn_bwd_dkdv(const Pool& p, const BlockGeom& g,
                                 const CUtensorMap& mq, const CUtensorMap& mdo,
                                 const CUtensorMap& mk, const CUtensorMap& mv,
                                 const int32_t* table, const float* lse,
                                 const float* D, float* dk, float* dv,
                                 cudaStream_t s);
// Latent pages: dq~ partials and the response latent-row gradients.
cudaError_t launch_latent_bwd_dq(const Pool& p, const BlockGeom& g,
                                 const CUtensorMap& mq, const CUtensorMap& mdo,
                                 const CUtensorMap& mk, const int32_t* table,
                                 const float* lse, const float* D,
                                 float* dq_part, cudaStream_t s);
cudaError_t launch_latent_bwd_dlat(const Pool& p, const BlockGeom& g,
                                   const CUtensorMap& mq,
                                   const CUtensorMap& mdo,
                                   const CUtensorMap& mk, const int32_t* table,
                                   const float* lse, const float* D,
                                   float* dlat, cudaStream_t s);

}  // namespace lsr

// Host handle behind lsr_pool_t: the pool geometry and its K/V tensor maps.
struct lsr_pool {
  lsr::Pool p;
  CUtensorMap mk, mv;
  int BN;  // key-tile rows: 128 when page_size % 128 == 0, else 64
  uint64_t version = 0;  // model version the resident state belongs to
};
