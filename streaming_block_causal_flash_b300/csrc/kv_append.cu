// kv_append.cu -- append one unit's K/V slice to the full-history cache.
//
// The performer appends each KV slice it receives to its own full-history
// cache ("全双工语音模型精读⑫：Wan-Streamer" (alwayszhang.cn), 四、推理, step 3).
// Slice layout [n][H][row] (token-major, as a projection emits it); cache
// layout [H][capacity][row].  Pure data movement: every thread moves 16-byte
// chunks, K and V in one launch (grid.y), several independent loads in
// flight before the matching stores.
#include "ws_debug.cuh"
#include "ws_internal.h"

namespace ws {
namespace {

// Device error word of this file's kernels: [0] code (0 clean, 2 device-
// resident sizes out of range, 3 a debug-build bounds check failed), [1] info
// (code 2: 1 n_new out of range, 2 the unit does not fit the capacity;
// code 3: (check site << 16) | block).
__device__ unsigned int g_unit_error[2];

constexpr int kThreads = 128;
constexpr int kMaxPerThread = 8;   // 16-byte chunks per thread held in flight

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One block per (tensor, token): it moves that token's [H][row] slice
// (heads * CH 16-byte chunks, contiguous in the source) into row
// cache_len + token of every head.  Chunk c of the slice belongs to head
// c / CH, column c % CH.  All loads of a thread are issued before its stores.
__global__ void __launch_bounds__(kThreads)
kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int64_t cache_len,
                 int64_t capacity, int heads, int CH) {
  const int64_t t = blockIdx.x;
  const bool is_v = blockIdx.y != 0;
  const int per_token = heads * CH;
  const uint4* src = (is_v ? v_new : k_new) + t * per_token;
  uint4* dst = (is_v ? v_cache : k_cache) + (cache_len + t) * CH;
  const int64_t head_stride = capacity * CH;
  for (int base = threadIdx.x; base < per_token; base += kThreads * kMaxPerThread) {
    uint4 val[kMaxPerThread];
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = base + u * kThreads;
      if (c < per_token &&
          WS_BOUND(g_unit_error, t * per_token + c, static_cast<int64_t>(gridDim.x) * per_token, 31))
        val[u] = ld_stream(src + c);
    }
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = base + u * kThreads;
      if (c < per_token) {
        const int h = c / CH;
        const int64_t at = h * head_stride + (c - h * CH);
        if (WS_BOUND(g_unit_error, (cache_len + t) * CH + at, heads * head_stride, 32))
          dst[at] = val[u];
      }
    }
  }
}

__device__ __forceinline__ void unit_error(unsigned info) {
  if (atomicCAS(&g_unit_error[0], 0u, 2u) == 0u) g_unit_error[1] = info;
}

// kv_append_kernel with the sizes read at run time from the device-resident
// unit state {cache_len, n_new}: the grid covers n_max tokens; blocks past
// n_new return.  A state out of range writes nothing and sets the error word.
__global__ void __launch_bounds__(kThreads)
kv_append_dev_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     const long long* __restrict__ state, int64_t n_max, int64_t capacity,
                     int heads, int CH) {
  const long long cache_len = state[0];
  const long long n_new = state[1];
  if (n_new < 0 || n_new > n_max) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) unit_error(1u);
    return;
  }
  if (cache_len < 0 || cache_len > capacity - n_new) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) unit_error(2u);
    return;
  }
  const int64_t t = blockIdx.x;
  if (t >= n_new) return;
  const bool is_v = blockIdx.y != 0;
  const int per_token = heads * CH;
  const uint4* src = (is_v ? v_new : k_new) + t * per_token;
  uint4* dst = (is_v ? v_cache : k_cache) + (cache_len + t) * CH;
  const int64_t head_stride = capacity * CH;
  for (int base = threadIdx.x; base < per_token; base += kThreads * kMaxPerThread) {
    uint4 val[kMaxPerThread];
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = base + u * kThreads;
      if (c < per_token &&
          WS_BOUND(g_unit_error, t * per_token + c, static_cast<int64_t>(gridDim.x) * per_token, 31))
        val[u] = ld_stream(src + c);
    }
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = base + u * kThreads;
      if (c < per_token) {
        const int h = c / CH;
        const int64_t at = h * head_stride + (c - h * CH);
        if (WS_BOUND(g_unit_error, (cache_len + t) * CH + at, heads * head_stride, 32))
          dst[at] = val[u];
      }
    }
  }
}

// Moves the device-resident unit state to the next unit: the current unit
// joins the history (cache_len += n_new), and n_new becomes the size of unit
// `unit + 1` in the caller's list (0 past its end).
__global__ void unit_state_advance_kernel(long long* state, const int32_t* __restrict__ sizes,
                                          int64_t n_sizes) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  state[0] += state[1];
  const long long next = state[2] + 1;
  state[2] = next;
  state[1] = (next >= 0 && next < n_sizes) ? static_cast<long long>(sizes[next]) : 0;
}

}  // namespace

cudaError_t launch_kv_append_dev(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const long long* state, int64_t n_max,
                                 int64_t capacity, int heads, int row_bytes, cudaStream_t s) {
  const int CH = row_bytes / 16;
  if (n_max <= 0) return cudaSuccess;
  if (n_max > 0x7FFFFFFF) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(n_max), 2);
  kv_append_dev_kernel<<<grid, kThreads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), state, n_max, capacity, heads,
      CH);
  return cudaGetLastError();
}

cudaError_t launch_unit_state_advance(long long* state, const int32_t* sizes, int64_t n_sizes,
                                      cudaStream_t s) {
  unit_state_advance_kernel<<<1, 32, 0, s>>>(state, sizes, n_sizes);
  return cudaGetLastError();
}

cudaError_t read_unit_device_error(int* code, int* info) {
  unsigned int h[2] = {0u, 0u};
  cudaError_t err = cudaMemcpyFromSymbol(h, g_unit_error, sizeof(h));
  if (err != cudaSuccess) return err;
  *code = static_cast<int>(h[0]);
  *info = static_cast<int>(h[1]);
  return cudaSuccess;
}

cudaError_t clear_unit_device_error() {
  const unsigned int z[2] = {0u, 0u};
  return cudaMemcpyToSymbol(g_unit_error, z, sizeof(z));
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             int64_t cache_len, int64_t n_new, int64_t capacity, int heads,
                             int row_bytes, int num_sms, cudaStream_t s) {
  (void)num_sms;
  const int CH = row_bytes / 16;
  if (n_new == 0) return cudaSuccess;
  if (n_new > 0x7FFFFFFF) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(n_new), 2);
  kv_append_kernel<<<grid, kThreads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), cache_len, capacity, heads, CH);
  return cudaGetLastError();
}

}  // namespace ws
