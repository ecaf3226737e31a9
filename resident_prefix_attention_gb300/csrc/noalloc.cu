// Response-only backward that allocates nothing.
//
// lsr_replay_attn_bwd needs a scratch workspace (per-shard dQ slices and
// the row dots D = rowsum(dO * O)) that the caller allocates.  Some callers
// cannot do that at the point where they run the backward: code that must
// not call cudaMalloc/cudaFree (for instance while it holds a memory budget
// enforced by a custom allocator, or from a context where an allocation
// could block or fail unpredictably), or a caller written against a plain
// C interface with no device allocator of its own.  This entry point serves
// them: its scratch is a fixed array in the library's own device memory,
// which every GPU that loads the library holds until the process exits.
#include <mutex>
#include "../../include/lsr.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device, looked up once
// per device (the array's host-side name is not a device address).
lsr_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    lsr::set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return LSR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    lsr::set_error("device %d is beyond the %d devices this entry point "
                   "supports",
                   dev, kMaxDevices);
    return LSR_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      lsr::set_error("cudaGetSymbolAddress of the backward scratch: %s",
                     cudaGetErrorString(e));
      return LSR_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LSR_OK;
}

}  // namespace

extern "C" lsr_status lsr_replay_attn_bwd_noalloc(
    lsr_pool_t pool, const void* q, const float* o, const void* dO,
    const float* lse, int Hq, int R_b, int P, int resp_pos0,
    const int32_t* page_table, int table_len, int num_shards, float scale,
    float* dq, float* dk_resp, float* dv_resp, void* stream) {
  // The block's geometry is checked first, as lsr_replay_attn_bwd checks
  // it, so that a bad argument is reported as itself and not as a scratch
  // size problem.
  lsr::BlockGeom g;
  lsr_status st = lsr::block_geom(pool, Hq, R_b, P, resp_pos0, table_len,
                                  num_shards, scale, false, &g);
  if (st != LSR_OK) return st;
  size_t need = 0;
  st = lsr_bwd_workspace_size(num_shards, Hq, R_b, g.d, &need);
  if (st != LSR_OK) return st;
  if (need > kScratchBytes) {
    lsr::set_error(
        "lsr_replay_attn_bwd_noalloc: this block needs %zu bytes of scratch "
        "but the built-in scratch holds %zu bytes (64 MiB); replay smaller "
        "blocks or pass your own workspace to lsr_replay_attn_bwd",
        need, kScratchBytes);
    return LSR_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != LSR_OK) return st;
  // Nothing in the scratch has to start at zero: every dQ slice and every D
  // entry the backward reads is written earlier in the same call.
  return lsr_replay_attn_bwd(pool, q, o, dO, lse, Hq, R_b, P, resp_pos0,
                             page_table, table_len, num_shards, scale, dq,
                             dk_resp, dv_resp, scratch, kScratchBytes, stream);
}
