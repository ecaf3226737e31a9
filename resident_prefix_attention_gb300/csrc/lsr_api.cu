// C ABI of the replay-attention library: argument validation, tensor-map
// encoding, workspace layout and kernel launch order.  Every entry point
// validates on the host and returns a status before launching anything.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <cudaTypedefs.h>
#include "../../include/lsr.h"
#include "internal.h"

namespace lsr {

static thread_local std::string g_err;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once (thread-safe static initialisation); null if the driver
  // does not provide it
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000)f;
    return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
  }();
  return fn;
}

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t inner,
                 uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (2D) failed with %d", (int)r);
    return false;
  }
  return true;
}

bool make_map_q(CUtensorMap* map, const void* base, int d, int Hq, int R,
                int G) {
  auto enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)Hq * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kTileRows / G)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (3D) failed with %d", (int)r);
    return false;
  }
  return true;
}

}  // namespace lsr

using namespace lsr;

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

#define LSR_REQUIRE(cond, ...)   \
  do {                           \
    if (!(cond)) {               \
      set_error(__VA_ARGS__);    \
      return LSR_ERR_INVALID_ARG; \
    }                            \
  } while (0)

lsr_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return LSR_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return LSR_ERR_CUDA;
}

}  // namespace

namespace lsr {

lsr_status block_geom(const lsr_pool* pool, int Hq, int R_b, int P,
                      int resp_pos0, int table_len, int num_shards,
                      float scale, bool latent, BlockGeom* g) {
  LSR_REQUIRE(pool != nullptr, "pool is NULL");
  const Pool& pl = pool->p;
  LSR_REQUIRE(pl.latent == latent,
              latent ? "this entry point needs a latent pool "
                       "(lsr_latent_pool_create)"
                     : "this entry point needs a K/V pool; latent pools use "
                       "the lsr_latent_* entry points");
  LSR_REQUIRE(Hq >= 1 && Hq % pl.num_kv_heads == 0,
              "Hq (%d) must be a positive multiple of Hkv (%d)", Hq,
              pl.num_kv_heads);
  const int G = Hq / pl.num_kv_heads;
  LSR_REQUIRE(G <= kTileRows && kTileRows % G == 0,
              "Hq/Hkv (%d) must divide %d", G, kTileRows);
  LSR_REQUIRE(R_b >= 1, "R_b (%d) must be >= 1", R_b);
  LSR_REQUIRE(P >= 0 && P % pl.page_size == 0,
              "P (%d) must be a non-negative multiple of page_size (%d)", P,
              pl.page_size);
  LSR_REQUIRE(resp_pos0 >= 0, "resp_pos0 (%d) must be >= 0", resp_pos0);
  LSR_REQUIRE(num_shards >= 1, "num_shards (%d) must be >= 1", num_shards);
  LSR_REQUIRE(std::isfinite(scale) && scale > 0.f,
              "scale must be finite and > 0");
  const long long need = (long long)P + resp_pos0 + R_b;
  LSR_REQUIRE(need <= (long long)table_len * pl.page_size,
              "page table (%d entries of %d) does not cover %lld keys",
              table_len, pl.page_size, need);
  LSR_REQUIRE((long long)R_b * Hq * pl.head_dim < (1ll << 31),
              "block too large");
  g->Hq = Hq;
  g->Hkv = pl.num_kv_heads;
  g->G = G;
  g->d = pl.head_dim;
  g->dv = pl.v_dim;
  g->ps = pl.page_size;
  g->BN = pool->BN;
  g->R_b = R_b;
  g->resp_pos0 = resp_pos0;
  g->prompt_pages = P / pl.page_size;
  g->num_shards = num_shards;
  g->rows_per_tile = kTileRows / G;
  g->n_qtiles = (R_b + g->rows_per_tile - 1) / g->rows_per_tile;
  g->scale = scale;
  // a plain block is a one-response table
  RespTable& t = g->resp;
  t.n = 1;
  t.row0[0] = 0;
  t.row0[1] = R_b;
  t.rows[0] = R_b;
  t.pos0[0] = resp_pos0;
  t.page0[0] = g->prompt_pages;
  t.gpage0[0] = 0;
  t.kt0[0] = 0;
  t.kt0[1] = (resp_pos0 + R_b + 127) / 128;
  return LSR_OK;
}

size_t bwd_ws_bytes(int num_shards, int Hq, int R_b, int d) {
  return round_up((size_t)(bwd_shards(num_shards) + 1) * R_b * Hq * d *
                  sizeof(float)) +
         round_up((size_t)Hq * R_b * sizeof(float));
}

lsr_status run_fwd(const lsr_pool* pool, const BlockGeom& g, const void* q,
                   const int32_t* table, float* m, float* l, float* o_part,
                   cudaStream_t s) {
  CUtensorMap mq;
  if (!make_map_q(&mq, q, g.d, g.Hq, g.R_b, g.G)) return LSR_ERR_CUDA;
  ProfScope ps(LSR_K_ATTN_FWD, s);
  return cuda_status(launch_attn_fwd(pool->p, g, mq, pool->mk, pool->mv, table,
                                     m, l, o_part, s),
                     "attn_fwd launch");
}

lsr_status run_bwd(const lsr_pool* pool, const BlockGeom& g, const void* q,
                   const float* o, const void* dO, const float* lse,
                   const int32_t* table, float* dq, float* dk, float* dv,
                   void* workspace, cudaStream_t s) {
  const int R_b = g.R_b, Hq = g.Hq;
  BlockGeom gb = g;  // the dQ pass over split prompt shards
  gb.num_shards = bwd_shards(g.num_shards);
  float* dq_part = reinterpret_cast<float*>(workspace);
  float* Dvec = reinterpret_cast<float*>(
      reinterpret_cast<char*>(workspace) +
      round_up((size_t)(gb.num_shards + 1) * R_b * Hq * g.d * sizeof(float)));
  CUtensorMap mq, mdo;
  if (!make_map_q(&mq, q, g.d, Hq, R_b, g.G) ||
      !make_map_q(&mdo, dO, g.d, Hq, R_b, g.G))
    return LSR_ERR_CUDA;
  lsr_status r;
  {
    ProfScope ps(LSR_K_BWD_PREPROCESS, s);
    r = cuda_status(launch_bwd_preprocess(o, dO, Hq, R_b, g.dv, Dvec, s),
                    "preprocess");
  }
  if (r != LSR_OK) return r;
  {
    ProfScope ps(LSR_K_ATTN_BWD_DQ, s);
    r = cuda_status(launch_attn_bwd_dq(pool->p, gb, mq, mdo, pool->mk,
                                       pool->mv, table, lse, Dvec, dq_part, s),
                    "attn_bwd_dq launch");
  }
  if (r != LSR_OK) return r;
  {
    ProfScope ps(LSR_K_DQ_REDUCE, s);
    r = cuda_status(launch_dq_reduce(dq_part, gb.num_shards + 1,
                                     (size_t)R_b * Hq * g.d, dq, s),
                    "dq_reduce launch");
  }
  if (r != LSR_OK) return r;
  ProfScope ps(LSR_K_ATTN_BWD_DKDV, s);
  return cuda_status(launch_attn_bwd_dkdv(pool->p, g, mq, mdo, pool->mk,
                                          pool->mv, table, lse, Dvec, dk, dv,
                                          s),
                     "attn_bwd_dkdv launch");
}

}  // namespace lsr

extern "C" {

const char* lsr_last_error(void) { return g_err.c_str(); }

lsr_status lsr_page_pool_create(int num_pages, int page_size, int num_kv_heads,
                                int head_dim, void* k_pages, void* v_pages,
                                int* dev_status, lsr_pool_t* out) {
  LSR_REQUIRE(out != nullptr, "out is NULL");
  *out = nullptr;
  LSR_REQUIRE(num_pages >= 1, "num_pages (%d) must be >= 1", num_pages);
  LSR_REQUIRE(page_size >= 64 && page_size % 64 == 0,
              "page_size (%d) must be a positive multiple of 64", page_size);
  LSR_REQUIRE(num_kv_heads >= 1, "num_kv_heads (%d) must be >= 1",
              num_kv_heads);
  if (head_dim != 64 && head_dim != 128) {
    set_error("head_dim %d is not built (64 or 128)", head_dim);
    return LSR_ERR_UNSUPPORTED;
  }
  LSR_REQUIRE(k_pages && v_pages && dev_status,
              "k_pages, v_pages and dev_status must be non-NULL");
  LSR_REQUIRE(aligned16(k_pages) && aligned16(v_pages) && aligned16(dev_status),
              "pool pointers must be 16-byte aligned");
  LSR_REQUIRE((long long)(num_pages + 1) * num_kv_heads * page_size <
                  (1ll << 31),
              "pool too large: (num_pages+1)*Hkv*page_size must be < 2^31");
  lsr_pool* pool = new (std::nothrow) lsr_pool();
  if (!pool) {
    set_error("host allocation of the pool handle failed");
    return LSR_ERR_INVALID_ARG;
  }
  pool->p = Pool{num_pages, page_size, num_kv_heads, head_dim,
                 k_pages,   v_pages,   dev_status, head_dim, false};
  pool->BN = (page_size % 128 == 0) ? 128 : 64;
  const uint64_t rows = (uint64_t)num_pages * num_kv_heads * page_size;
  if (!make_map_2d(&pool->mk, k_pages, head_dim, rows, pool->BN) ||
      !make_map_2d(&pool->mv, v_pages, head_dim, rows, pool->BN)) {
    delete pool;
    return LSR_ERR_CUDA;
  }
  *out = pool;
  return LSR_OK;
}

lsr_status lsr_pool_set_wait_limit(lsr_pool_t pool, int limit_us) {
  LSR_REQUIRE(pool != nullptr, "pool is NULL");
  LSR_REQUIRE(limit_us >= 0 && limit_us <= 4000000,
              "limit_us (%d) must be 0 (default) or 1 .. 4000000", limit_us);
  pool->p.wait_ns =
      limit_us == 0 ? kDefaultWaitNs : (uint64_t)limit_us * 1000ull;
  return LSR_OK;
}

lsr_status lsr_page_pool_destroy(lsr_pool_t pool) {
  delete pool;
  return LSR_OK;
}

lsr_status lsr_write_prefix_pages(lsr_pool_t pool, const void* k,
                                  const void* v, int T, int pos0,
                                  const int32_t* page_table, int table_len,
                                  void* stream) {
  LSR_REQUIRE(pool != nullptr, "pool is NULL");
  LSR_REQUIRE(!pool->p.latent,
              "latent pools are written with lsr_latent_write_pages");
  LSR_REQUIRE(T >= 0 && pos0 >= 0, "T and pos0 must be >= 0");
  if (T == 0) return LSR_OK;
  LSR_REQUIRE(k && v && page_table, "k, v and page_table must be non-NULL");
  LSR_REQUIRE(aligned16(k) && aligned16(v), "k and v must be 16-byte aligned");
  LSR_REQUIRE((long long)pos0 + T <=
                  (long long)table_len * pool->p.page_size,
              "page table (%d entries) does not cover positions up to %lld",
              table_len, (long long)pos0 + T);
  ProfScope ps(LSR_K_WRITE_PAGES, (cudaStream_t)stream);
  return cuda_status(launch_write_pages(pool->p, k, v, T, pos0, page_table,
                                        table_len, (cudaStream_t)stream),
                     "write_pages launch");
}

lsr_status lsr_replay_attn_fwd(lsr_pool_t pool, const void* q, int Hq, int R_b,
                               int P, int resp_pos0, const int32_t* page_table,
                               int table_len, int num_shards, float scale,
                               float* m, float* l, float* o_part,
                               void* stream) {
  BlockGeom g;
  lsr_status st = block_geom(pool, Hq, R_b, P, resp_pos0, table_len,
                             num_shards, scale, false, &g);
  if (st != LSR_OK) return st;
  LSR_REQUIRE(q && page_table && m && l && o_part,
              "q, page_table, m, l and o_part must be non-NULL");
  LSR_REQUIRE(aligned16(q) && aligned16(m) && aligned16(l) && aligned16(o_part),
              "q, m, l and o_part must be 16-byte aligned");
  return run_fwd(pool, g, q, page_table, m, l, o_part, (cudaStream_t)stream);
}

lsr_status lsr_lse_merge(const float* m, const float* l, const float* o_part,
                         int num_parts, int Hq, int R_b, int head_dim, float* o,
                         float* lse, void* stream) {
  LSR_REQUIRE(num_parts >= 1 && Hq >= 1 && R_b >= 1,
              "num_parts, Hq and R_b must be >= 1");
  if (head_dim != 64 && head_dim != 128) {
    set_error("head_dim %d is not built (64 or 128)", head_dim);
    return LSR_ERR_UNSUPPORTED;
  }
  LSR_REQUIRE(m && l && o_part && o && lse, "NULL pointer argument");
  LSR_REQUIRE(aligned16(o_part) && aligned16(o),
              "o_part and o must be 16-byte aligned");
  ProfScope ps(LSR_K_LSE_MERGE, (cudaStream_t)stream);
  return cuda_status(launch_lse_merge(m, l, o_part, num_parts, Hq, R_b,
                                      head_dim, o, lse, (cudaStream_t)stream),
                     "lse_merge launch");
}

lsr_status lsr_bwd_workspace_size(int num_shards, int Hq, int R_b,
                                  int head_dim, size_t* bytes) {
  LSR_REQUIRE(bytes != nullptr, "bytes is NULL");
  LSR_REQUIRE(num_shards >= 1 && Hq >= 1 && R_b >= 1 && head_dim >= 1,
              "sizes must be >= 1");
  *bytes = bwd_ws_bytes(num_shards, Hq, R_b, head_dim);
  return LSR_OK;
}

lsr_status lsr_replay_attn_bwd(lsr_pool_t pool, const void* q, const float* o,
                               const void* dO, const float* lse, int Hq,
                               int R_b, int P, int resp_pos0,
                               const int32_t* page_table, int table_len,
                               int num_shards, float scale, float* dq,
                               float* dk_resp, float* dv_resp,
                               void* workspace, size_t workspace_bytes,
                               void* stream) {
  BlockGeom g;
  lsr_status st = block_geom(pool, Hq, R_b, P, resp_pos0, table_len,
                             num_shards, scale, false, &g);
  if (st != LSR_OK) return st;
  LSR_REQUIRE(q && o && dO && lse && page_table && dq && dk_resp && dv_resp &&
                  workspace,
              "NULL pointer argument");
  LSR_REQUIRE(aligned16(q) && aligned16(o) && aligned16(dO) && aligned16(dq) &&
                  aligned16(dk_resp) && aligned16(dv_resp) &&
                  aligned16(workspace),
              "q, o, dO, dq, dk_resp, dv_resp and workspace must be 16-byte "
              "aligned");
  const size_t need = bwd_ws_bytes(num_shards, Hq, R_b, g.d);
  LSR_REQUIRE(workspace_bytes >= need,
              "workspace too small: %zu bytes given, %zu needed",
              workspace_bytes, need);
  return run_bwd(pool, g, q, o, dO, lse, page_table, dq, dk_resp, dv_resp,
                 workspace, (cudaStream_t)stream);
}

static int max_block_rows(int R, int num_blocks) {
  const int base = R / num_blocks;
  return R - base * (num_blocks - 1);
}

static size_t replay_ws_bytes(int num_shards, int Hq, int R, int num_blocks,
                              int d) {
  const int Rb = max_block_rows(R, num_blocks);
  const size_t parts = (size_t)(num_shards + 1);
  return 2 * round_up(parts * Hq * Rb * sizeof(float)) +
         round_up(parts * Rb * Hq * d * sizeof(float)) +
         round_up((size_t)Hq * Rb * sizeof(float)) +
         bwd_ws_bytes(num_shards, Hq, Rb, d);
}

lsr_status lsr_replay_workspace_size(int num_shards, int Hq, int R,
                                     int num_blocks, int head_dim,
                                     size_t* bytes) {
  LSR_REQUIRE(bytes != nullptr, "bytes is NULL");
  LSR_REQUIRE(num_shards >= 1 && Hq >= 1 && R >= 1 && head_dim >= 1,
              "sizes must be >= 1");
  LSR_REQUIRE(num_blocks >= 1 && num_blocks <= R,
              "num_blocks (%d) must be in [1, R]", num_blocks);
  *bytes = replay_ws_bytes(num_shards, Hq, R, num_blocks, head_dim);
  return LSR_OK;
}

lsr_status lsr_replay_response(lsr_pool_t pool, const void* q, const void* dO,
                               int Hq, int R, int num_blocks, int P,
                               const int32_t* page_table, int table_len,
                               int num_shards, float scale, float* o,
                               float* lse, float* dq, float* dk_resp,
                               float* dv_resp, void* workspace,
                               size_t workspace_bytes, void* stream) {
  LSR_REQUIRE(pool != nullptr, "pool is NULL");
  LSR_REQUIRE(R >= 1 && num_blocks >= 1 && num_blocks <= R,
              "need R >= 1 and 1 <= num_blocks <= R");
  BlockGeom g;
  lsr_status st = block_geom(pool, Hq, R, P, 0, table_len, num_shards, scale,
                             false, &g);
  if (st != LSR_OK) return st;
  LSR_REQUIRE(q && dO && o && lse && dq && dk_resp && dv_resp && workspace,
              "NULL pointer argument");
  LSR_REQUIRE(aligned16(workspace), "workspace must be 16-byte aligned");
  const size_t need = replay_ws_bytes(num_shards, Hq, R, num_blocks, g.d);
  LSR_REQUIRE(workspace_bytes >= need,
              "workspace too small: %zu bytes given, %zu needed",
              workspace_bytes, need);
  const int d = g.d;
  const int Rb_max = max_block_rows(R, num_blocks);
  const size_t parts = (size_t)(num_shards + 1);
  char* w = reinterpret_cast<char*>(workspace);
  float* m = reinterpret_cast<float*>(w);
  w += round_up(parts * Hq * Rb_max * sizeof(float));
  float* l = reinterpret_cast<float*>(w);
  w += round_up(parts * Hq * Rb_max * sizeof(float));
  float* op = reinterpret_cast<float*>(w);
  w += round_up(parts * Rb_max * Hq * d * sizeof(float));
  float* lse_b = reinterpret_cast<float*>(w);
  w += round_up((size_t)Hq * Rb_max * sizeof(float));
  void* bws = w;
  const size_t bws_bytes = bwd_ws_bytes(num_shards, Hq, Rb_max, d);
  cudaStream_t s = (cudaStream_t)stream;
  const int base = R / num_blocks;
  const size_t row_elems = (size_t)Hq * d;
  for (int b = num_blocks - 1; b >= 0; --b) {
    const int pos0 = b * base;
    const int n = (b == num_blocks - 1) ? R - pos0 : base;
    const char* qb = reinterpret_cast<const char*>(q) + pos0 * row_elems * 2;
    const char* dob = reinterpret_cast<const char*>(dO) + pos0 * row_elems * 2;
    float* ob = o + pos0 * row_elems;
    st = lsr_replay_attn_fwd(pool, qb, Hq, n, P, pos0, page_table, table_len,
                             num_shards, scale, m, l, op, stream);
    if (st != LSR_OK) return st;
    st = lsr_lse_merge(m, l, op, num_shards + 1, Hq, n, d, ob, lse_b, stream);
    if (st != LSR_OK) return st;
    st = cuda_status(cudaMemcpy2DAsync(lse + pos0, (size_t)R * sizeof(float),
                                       lse_b, (size_t)n * sizeof(float),
                                       (size_t)n * sizeof(float), Hq,
                                       cudaMemcpyDeviceToDevice, s),
                     "lse copy");
    if (st != LSR_OK) return st;
    st = lsr_replay_attn_bwd(pool, qb, ob, dob, lse_b, Hq, n, P, pos0,
                             page_table, table_len, num_shards, scale,
                             dq + pos0 * row_elems, dk_resp, dv_resp, bws,
                             bws_bytes, stream);
    if (st != LSR_OK) return st;
  }
  return LSR_OK;
}

lsr_status lsr_pool_device_status(lsr_pool_t pool, int* out, void* stream) {
  LSR_REQUIRE(pool != nullptr && out != nullptr, "pool and out must be set");
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, pool->p.dev_status, sizeof(int),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e, "device status read");
  *out = v;
  if (v != 0) {
    set_error("device status word is 0x%x", v);
    return LSR_ERR_DEVICE;
  }
  return LSR_OK;
}

}  // extern "C"
