// Bandwidth-bound kernels of the replay path: page scatter (prompt capture
// and response pages), exact LSE merge of partial statistics, the backward
// row dot D = rowsum(dO * O), and the dQ partial reduction.  All use 16-byte
// (or 8-byte) vector accesses and grid-stride loops sized to the SM count.
#include <atomic>
#include <mutex>
#include <set>
#include <utility>
#include <cmath>
#include "attn_common.cuh"
#include "internal.h"

namespace lsr {

int num_sms() {
  // per device; a failed query gives 1, which only narrows the grids of
  // the bandwidth-bound kernels
  constexpr int kDevices = 64;
  static std::atomic<int> cache[kDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices)
    dev = 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        v <= 0)
      v = 1;
    n = v;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t set_smem_limit(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

namespace {
int grid_for(size_t n, int threads, int per_sm = 8) {
  size_t blocks = (n + threads - 1) / threads;
  size_t cap = (size_t)num_sms() * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}
}  // namespace

// --------------------------------------------------------------- page write
// Token t of kv head g goes to row (pos0+t) % ps of page table[(pos0+t)/ps].
// One thread moves one 16-byte vector; rows after the end in the last page
// are zeroed.
__global__ void write_pages_kernel(const uint4* __restrict__ k,
                                   const uint4* __restrict__ v,
                                   uint4* __restrict__ kpool,
                                   uint4* __restrict__ vpool,
                                   const int32_t* __restrict__ table, int T,
                                   int pos0, int Hkv, int ps, int vpr,
                                   int num_pages, int* status) {
  const size_t n_main = (size_t)T * Hkv * vpr;
  const int end = pos0 + T;
  const int tail = (end % ps) ? ps - end % ps : 0;
  const size_t n_tail = (size_t)tail * Hkv * vpr;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
       i < n_main + n_tail; i += stride) {
    int pos, g, vec;
    bool is_tail = i >= n_main;
    size_t j = is_tail ? i - n_main : i;
    vec = (int)(j % vpr);
    j /= vpr;
    g = (int)(j % Hkv);
    const int t = (int)(j / Hkv);
    pos = is_tail ? end + t : pos0 + t;
    const int phys = __ldg(table + pos / ps);
    if (phys < 0 || phys >= num_pages) {
      atomicOr(status, LSR_DEV_BAD_PAGE);
      continue;
    }
    const size_t dst = (((size_t)phys * Hkv + g) * ps + pos % ps) * vpr + vec;
    // vpool is NULL for a latent pool (one row is both key and value)
    if (is_tail) {
      kpool[dst] = make_uint4(0, 0, 0, 0);
      if (vpool) vpool[dst] = make_uint4(0, 0, 0, 0);
    } else {
      const size_t src = ((size_t)t * Hkv + g) * vpr + vec;
      kpool[dst] = __ldg(k + src);
      if (vpool) vpool[dst] = __ldg(v + src);
    }
  }
}

cudaError_t launch_write_pages(const Pool& p, const void* k, const void* v,
                               int T, int pos0, const int32_t* table,
                               int table_len, cudaStream_t s) {
  (void)table_len;
  const int vpr = p.head_dim * 2 / 16;
  const int end = pos0 + T;
  const int tail = (end % p.page_size) ? p.page_size - end % p.page_size : 0;
  const size_t n = ((size_t)T + tail) * p.num_kv_heads * vpr;
  if (n == 0) return cudaSuccess;
  write_pages_kernel<<<grid_for(n, 256), 256, 0, s>>>(
      (const uint4*)k, (const uint4*)v, (uint4*)p.k_pages,
      p.latent ? nullptr : (uint4*)p.v_pages,
      table, T, pos0, p.num_kv_heads, p.page_size, vpr, p.num_pages,
      p.dev_status);
  return cudaGetLastError();
}

// --------------------------------------------------------------- LSE merge
// One warp per (row r, head h), at most 32 partials: lane s loads partial
// s's (m, l), the warp reduces the max of t_s = m_s + ln l_s and the total
// weight, and the O rows of all partials are then read independently with
// the weights broadcast from their lanes.  Each lane holds VEC = d/32
// output columns.
template <int VEC>
__global__ void lse_merge_warp_kernel(const float* __restrict__ m,
                                      const float* __restrict__ l,
                                      const float* __restrict__ o, int parts,
                                      int Hq, int R_b, float* __restrict__ out,
                                      float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const size_t nrows = (size_t)R_b * Hq;
  const size_t wstride = (size_t)gridDim.x * (blockDim.x >> 5);
  constexpr int D = VEC * 32;
  for (size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < nrows; row += wstride) {
    const int r = (int)(row / Hq), h = (int)(row % Hq);
    float t = -INFINITY;
    if (lane < parts) {
      const size_t si = ((size_t)lane * Hq + h) * R_b + r;
      const float ls = __ldg(l + si);
      if (ls > 0.f) t = __ldg(m + si) + logf(ls);
    }
    float tmax = t;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float w = (tmax > -INFINITY && t > -INFINITY) ? expf(t - tmax) : 0.f;
    float tot = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      tot += __shfl_xor_sync(0xffffffffu, tot, off);
    float acc[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
    const float* src = o + ((size_t)r * Hq + h) * D + lane * VEC;
    const size_t part_stride = (size_t)R_b * Hq * D;
#pragma unroll 4
    for (int s = 0; s < parts; ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      if (ws == 0.f) continue;
      const float* p = src + (size_t)s * part_stride;
      if constexpr (VEC == 4) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p));
        acc[0] += ws * f.x; acc[1] += ws * f.y; acc[2] += ws * f.z; acc[3] += ws * f.w;
      } else {
        const float2 f = __ldg(reinterpret_cast<const float2*>(p));
        acc[0] += ws * f.x; acc[1] += ws * f.y;
      }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    float* dst = out + ((size_t)r * Hq + h) * D + lane * VEC;
    if constexpr (VEC == 4) {
      *reinterpret_cast<float4*>(dst) =
          make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0)
      lse[(size_t)h * R_b + r] = tot > 0.f ? tmax + logf(tot) : -INFINITY;
  }
}

// The general form for more than 32 partials: two passes over the
// partials, one warp per (row r, head h).
template <int VEC>
__global__ void lse_merge_kernel(const float* __restrict__ m,
                                 const float* __restrict__ l,
                                 const float* __restrict__ o, int parts,
                                 int Hq, int R_b, float* __restrict__ out,
                                 float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const size_t nrows = (size_t)R_b * Hq;
  const size_t wstride = (size_t)gridDim.x * (blockDim.x >> 5);
  constexpr int D = VEC * 32;
  for (size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < nrows; row += wstride) {
    const int r = (int)(row / Hq), h = (int)(row % Hq);
    float tmax = -INFINITY;
    for (int s = 0; s < parts; ++s) {
      const size_t si = ((size_t)s * Hq + h) * R_b + r;
      const float ls = __ldg(l + si);
      if (ls > 0.f) tmax = fmaxf(tmax, __ldg(m + si) + logf(ls));
    }
    float acc[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
    float tot = 0.f;
    if (tmax > -INFINITY) {
      for (int s = 0; s < parts; ++s) {
        const size_t si = ((size_t)s * Hq + h) * R_b + r;
        const float ls = __ldg(l + si);
        if (!(ls > 0.f)) continue;
        const float w = expf(__ldg(m + si) + logf(ls) - tmax);
        tot += w;
        const float* src = o + (((size_t)s * R_b + r) * Hq + h) * D + lane * VEC;
        if constexpr (VEC == 4) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(src));
          acc[0] += w * f.x; acc[1] += w * f.y; acc[2] += w * f.z; acc[3] += w * f.w;
        } else {
          const float2 f = __ldg(reinterpret_cast<const float2*>(src));
          acc[0] += w * f.x; acc[1] += w * f.y;
        }
      }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    float* dst = out + ((size_t)r * Hq + h) * D + lane * VEC;
    if constexpr (VEC == 4) {
      *reinterpret_cast<float4*>(dst) =
          make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0)
      lse[(size_t)h * R_b + r] = tot > 0.f ? tmax + logf(tot) : -INFINITY;
  }
}

// The same merge for few (row, head) pairs and many partials (scoring a
// handful of rows, where the shard count is raised to fill the GPU): one
// 256-thread block per (row, head); the eight warps take every eighth
// partial and combine their sums through shared memory.
template <int VEC>
__global__ void __launch_bounds__(256)
    lse_merge_split_kernel(const float* __restrict__ m,
                           const float* __restrict__ l,
                           const float* __restrict__ o, int parts, int Hq,
                           int R_b, float* __restrict__ out,
                           float* __restrict__ lse) {
  constexpr int W = 8, D = VEC * 32;
  __shared__ float s_max[W], s_tot[W];
  __shared__ float s_acc[W][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (int)(blockIdx.x / Hq), h = (int)(blockIdx.x % Hq);
  float tmax = -INFINITY;
  for (int s = threadIdx.x; s < parts; s += W * 32) {
    const size_t si = ((size_t)s * Hq + h) * R_b + r;
    const float ls = __ldg(l + si);
    if (ls > 0.f) tmax = fmaxf(tmax, __ldg(m + si) + logf(ls));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
  if (lane == 0) s_max[warp] = tmax;
  __syncthreads();
  tmax = s_max[0];
#pragma unroll
  for (int w = 1; w < W; ++w) tmax = fmaxf(tmax, s_max[w]);
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  float tot = 0.f;
  if (tmax > -INFINITY) {
    for (int s = warp; s < parts; s += W) {
      const size_t si = ((size_t)s * Hq + h) * R_b + r;
      const float ls = __ldg(l + si);
      if (!(ls > 0.f)) continue;
      const float wt = expf(__ldg(m + si) + logf(ls) - tmax);
      tot += wt;
      const float* src = o + (((size_t)s * R_b + r) * Hq + h) * D + lane * VEC;
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[i] += wt * __ldg(src + i);
    }
  }
#pragma unroll
  for (int i = 0; i < VEC; ++i) s_acc[warp][lane * VEC + i] = acc[i];
  if (lane == 0) s_tot[warp] = tot;
  __syncthreads();
  if (warp != 0) return;
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < W; ++w) t += s_tot[w];
  const float inv = t > 0.f ? 1.f / t : 0.f;
  float* dst = out + ((size_t)r * Hq + h) * D + lane * VEC;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) a += s_acc[w][lane * VEC + i];
    dst[i] = a * inv;
  }
  if (lane == 0)
    lse[(size_t)h * R_b + r] = t > 0.f ? tmax + logf(t) : -INFINITY;
}

cudaError_t launch_lse_merge(const float* m, const float* l, const float* o,
                             int parts, int Hq, int R_b, int d, float* out,
                             float* lse, cudaStream_t s) {
  const size_t rows = (size_t)R_b * Hq;
  if (parts >= 32 && rows <= (size_t)4 * num_sms()) {
    if (d == 128)
      lse_merge_split_kernel<4><<<(unsigned)rows, 256, 0, s>>>(
          m, l, o, parts, Hq, R_b, out, lse);
    else
      lse_merge_split_kernel<2><<<(unsigned)rows, 256, 0, s>>>(
          m, l, o, parts, Hq, R_b, out, lse);
    return cudaGetLastError();
  }
  const int grid = grid_for(rows * 32, 256);
  if (parts <= 32) {
    if (d == 128)
      lse_merge_warp_kernel<4><<<grid, 256, 0, s>>>(m, l, o, parts, Hq, R_b,
                                                    out, lse);
    else
      lse_merge_warp_kernel<2><<<grid, 256, 0, s>>>(m, l, o, parts, Hq, R_b,
                                                    out, lse);
    return cudaGetLastError();
  }
  if (d == 128)
    lse_merge_kernel<4><<<grid, 256, 0, s>>>(m, l, o, parts, Hq, R_b, out,
                                             lse);
  else
    lse_merge_kernel<2><<<grid, 256, 0, s>>>(m, l, o, parts, Hq, R_b, out,
                                             lse);
  return cudaGetLastError();
}

// --------------------------------------------------------- bwd preprocess
// D[h][r] = sum_c dO[r][h][c] * O[r][h][c] in fp32; one warp per row.
template <int VEC>
__global__ void bwd_preprocess_kernel(const float* __restrict__ o,
                                      const __nv_bfloat16* __restrict__ dO,
                                      int Hq, int R_b, float* __restrict__ D) {
  const int lane = threadIdx.x & 31;
  const size_t nrows = (size_t)R_b * Hq;
  const size_t wstride = (size_t)gridDim.x * (blockDim.x >> 5);
  // RPW rows per warp at a time: their loads are all in flight before the
  // first reduction
  constexpr int RPW = 4;
  for (size_t row0 =
           ((size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;
       row0 < nrows; row0 += wstride * RPW) {
    float acc[RPW];
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      acc[k] = 0.f;
      const size_t row = row0 + k;
      if (row >= nrows) continue;
      const size_t base = row * (VEC * 32) + lane * VEC;
      if constexpr (VEC == 4) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(o + base));
        const uint2 b = __ldg(reinterpret_cast<const uint2*>(dO + base));
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
        const float2 f0 = __bfloat1622float2(pb[0]);
        const float2 f1 = __bfloat1622float2(pb[1]);
        acc[k] = a.x * f0.x + a.y * f0.y + a.z * f1.x + a.w * f1.y;
      } else {
        const float2 a = __ldg(reinterpret_cast<const float2*>(o + base));
        const __nv_bfloat162 b =
            *reinterpret_cast<const __nv_bfloat162*>(dO + base);
        const float2 fb = __bfloat1622float2(b);
        acc[k] = a.x * fb.x + a.y * fb.y;
      }
    }
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
    }
    if (lane < RPW && row0 + lane < nrows) {
      float a = acc[0];
#pragma unroll
      for (int k = 1; k < RPW; ++k)
        if (lane == k) a = acc[k];
      const size_t row = row0 + lane;
      const int r = (int)(row / Hq), h = (int)(row % Hq);
      D[(size_t)h * R_b + r] = a;
    }
  }
}

cudaError_t launch_bwd_preprocess(const float* o, const void* dO, int Hq,
                                  int R_b, int d, float* D, cudaStream_t s) {
  const size_t rows = (size_t)R_b * Hq;
  const int grid = grid_for((rows + 3) / 4 * 32, 256);  // four rows per warp
  if (d == 128)
    bwd_preprocess_kernel<4><<<grid, 256, 0, s>>>(
        o, (const __nv_bfloat16*)dO, Hq, R_b, D);
  else
    bwd_preprocess_kernel<2><<<grid, 256, 0, s>>>(
        o, (const __nv_bfloat16*)dO, Hq, R_b, D);
  return cudaGetLastError();
}

// --------------------------------------------------------- dQ reduction
// dq[i] += sum_s parts[s][i], float4 per thread, fixed summation order.
__global__ void dq_reduce_kernel(const float4* __restrict__ parts, int nparts,
                                 size_t n4, float4* __restrict__ dq) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    float4 acc = dq[i];
    for (int s = 0; s < nparts; ++s) {
      const float4 f = __ldg(parts + (size_t)s * n4 + i);
      acc.x += f.x; acc.y += f.y; acc.z += f.z; acc.w += f.w;
    }
    dq[i] = acc;
  }
}

cudaError_t launch_dq_reduce(const float* parts, int nparts, size_t n,
                             float* dq, cudaStream_t s) {
  const size_t n4 = n / 4;
  dq_reduce_kernel<<<grid_for(n4, 256), 256, 0, s>>>(
      (const float4*)parts, nparts, n4, (float4*)dq);
  return cudaGetLastError();
}

}  // namespace lsr
