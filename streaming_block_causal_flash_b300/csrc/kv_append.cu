// kv_append.cu -- append one unit's K/V slice to the full-history cache.
//
// The performer appends each KV slice it receives to its own full-history
// cache ("全双工语音模型精读⑫：Wan-Streamer" (alwayszhang.cn), 四、推理, step 3).
// Slice layout [n][H][row] (token-major, as a projection emits it); cache
// layout [H][capacity][row].  Pure data movement: every thread moves 16-byte
// chunks, K and V in one launch, several independent loads in flight before
// the matching stores.
#include "ws_internal.h"

namespace ws {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Chunk index c runs over [2][n][H][CH]: tensor (K, V), token, head, 16-byte
// column.  Reads are contiguous in c; each cache row of CH chunks is written
// contiguously.
__global__ void __launch_bounds__(kThreads)
kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int64_t cache_len,
                 int64_t n_new, int64_t capacity, int heads, int CH) {
  const int64_t per_tensor = n_new * heads * CH;
  const int64_t total = 2 * per_tensor;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; base < total;
       base += stride * kUnroll) {
    uint4 val[kUnroll];
    uint4* dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * stride;
      dst[u] = nullptr;
      if (c < total) {
        const bool is_v = c >= per_tensor;
        const int64_t i = is_v ? c - per_tensor : c;
        const int64_t col = i % CH;
        const int64_t th = i / CH;
        const int64_t h = th % heads;
        const int64_t t = th / heads;
        val[u] = ld_stream((is_v ? v_new : k_new) + i);
        dst[u] = (is_v ? v_cache : k_cache) + ((h * capacity + cache_len + t) * CH + col);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u]) *dst[u] = val[u];
  }
}

}  // namespace

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             int64_t cache_len, int64_t n_new, int64_t capacity, int heads,
                             int row_bytes, int num_sms, cudaStream_t s) {
  const int CH = row_bytes / 16;
  const int64_t total = 2 * n_new * heads * CH;
  if (total == 0) return cudaSuccess;
  const int64_t per_block = static_cast<int64_t>(kThreads) * kUnroll;
  int64_t blocks = (total + per_block - 1) / per_block;
  const int64_t cap_blocks = static_cast<int64_t>(num_sms) * 8;   // 8 x 256 threads per SM
  if (blocks > cap_blocks) blocks = cap_blocks;
  kv_append_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), cache_len, n_new, capacity,
      heads, CH);
  return cudaGetLastError();
}

}  // namespace ws
