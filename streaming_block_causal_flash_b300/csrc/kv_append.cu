// kv_append.cu -- append one unit's K/V slice to the full-history cache.
//
// The performer appends each KV slice it receives to its own full-history
// cache ("全双工语音模型精读⑫：Wan-Streamer" (alwayszhang.cn), 四、推理, step 3).
// Slice layout [n][H][row] (token-major, as a projection emits it); cache
// layout [H][capacity][row].  Pure data movement: every thread moves 16-byte
// chunks, K and V in one launch (grid.y), several independent loads in
// flight before the matching stores.
#include <mutex>

#include "ws_debug.cuh"
#include "ws_internal.h"

namespace ws {
namespace {

// Device error word of this file's kernels: [0] code (0 clean, 1 a bounded
// wait gave up, 2 device-resident sizes out of range, 3 a debug-build bounds
// check failed), [1] info (code 1 and 3: (site << 16) | block; code 2: 1 n_new
// out of range, 2 the unit does not fit the capacity).
__device__ unsigned int g_unit_error[2];

__device__ __forceinline__ void unit_error(unsigned info) {
  if (atomicCAS(&g_unit_error[0], 0u, 2u) == 0u) g_unit_error[1] = info;
}

constexpr int kThreads = 128;
constexpr int kMaxPerThread = 8;   // 16-byte chunks per thread held in flight

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The TMA copy: one CTA per (tensor, token) of a warp whose lane 0 does all
// the work.  A bulk copy brings the token's [H][row] slice (contiguous) into
// shared memory; one 3-D tensor store then writes it to row cache_len + t of
// every head.  The tensor map views the cache as (row elements, head, cache
// row) with strides (2 B, capacity * row, row), so the store's box
// {row, H, 1} has exactly the slice's layout in shared memory.  The DMA
// engine does the scatter over the heads.  A plain device-to-device copy of
// the same bytes is slower (the copy roofline at this size).  With
// device-resident sizes (state != null), cache_len and n_new are read from
// state = {cache_len, n_new}, and the launch covers n_max tokens.  Every wait
// is bounded; a copy that never lands sets the error word (code 1) after its
// bytes have been waited for once more, so the CTA never exits with a copy in
// flight into its shared memory.
__global__ void __launch_bounds__(32)
kv_append_tma_kernel(const uint8_t* __restrict__ k_new, const uint8_t* __restrict__ v_new,
                     const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                     int64_t cache_len_host, const long long* __restrict__ state, int64_t n_max,
                     int64_t capacity, int per_token) {
  extern __shared__ __align__(128) uint8_t slab_raw[];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  long long cache_len = cache_len_host;
  const int64_t t = blockIdx.x;
  if (state != nullptr) {
    cache_len = state[0];
    const long long n_new = state[1];
    if (n_new < 0 || n_new > n_max) {
      if (blockIdx.x == 0 && blockIdx.y == 0) unit_error(1u);
      return;
    }
    if (cache_len < 0 || cache_len > capacity - n_new) {
      if (blockIdx.x == 0 && blockIdx.y == 0) unit_error(2u);
      return;
    }
    if (t >= n_new) return;
  }
  if (!WS_BOUND(g_unit_error, t * per_token, static_cast<int64_t>(gridDim.x) * per_token, 31) ||
      !WS_BOUND(g_unit_error, cache_len + t, capacity, 32))
    return;
  const bool is_v = blockIdx.y != 0;
  uint8_t* slab = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(slab_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const uint32_t b = smem_u32(&bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(per_token)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(slab)),
      "l"((is_v ? v_new : k_new) + t * per_token), "r"(per_token), "r"(b)
      : "memory");
  bool landed = false;
  for (int round = 0; round < 2 && !landed; ++round) {
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t it = 0;; ++it) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(b)
          : "memory");
      if (ok) { landed = true; break; }
      uint64_t now;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
      if (now - t0 > 2000000000ull) break;   // 2 s
    }
    if (!landed && round == 0 && atomicCAS(&g_unit_error[0], 0u, 1u) == 0u)
      g_unit_error[1] = (15u << 16) | (blockIdx.x & 0xFFFFu);   // wait site 15
  }
  if (!landed) return;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const CUtensorMap* map = is_v ? &map_v : &map_k;
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(0), "r"(0), "r"(static_cast<int>(cache_len + t)), "r"(smem_u32(slab))
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

// The TMA append's shared memory: the slice of one token plus alignment slack.
int tma_append_smem(int per_token) { return per_token + 128; }

cudaError_t launch_tma_append(const void* k_new, const void* v_new, const AppendMaps& maps,
                              int64_t cache_len, const long long* state, int64_t n_tokens,
                              int64_t capacity, int per_token, cudaStream_t s) {
  static std::mutex mu;
  static int smem_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int smem = tma_append_smem(per_token);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (smem > 48 * 1024 && smem_set[dev] < smem) {
      err = cudaFuncSetAttribute(kv_append_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
      if (err != cudaSuccess) return err;
      smem_set[dev] = smem;
    }
  }
  dim3 grid(static_cast<unsigned>(n_tokens), 2);
  kv_append_tma_kernel<<<grid, 32, smem, s>>>(static_cast<const uint8_t*>(k_new),
                                              static_cast<const uint8_t*>(v_new), maps.k, maps.v,
                                              cache_len, state, n_tokens, capacity, per_token);
  return cudaGetLastError();
}

cudaError_t launch_kv_append_dev(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const long long* state, int64_t n_max,
                                 int64_t capacity, int heads, int row_bytes,
                                 const AppendMaps* maps, cudaStream_t s) {
  const int CH = row_bytes / 16;
  if (n_max <= 0) return cudaSuccess;
  if (n_max > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (maps != nullptr)
    return launch_tma_append(k_new, v_new, *maps, 0, state, n_max, capacity, heads * row_bytes, s);
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
                             int row_bytes, const AppendMaps* maps, cudaStream_t s) {
  const int CH = row_bytes / 16;
  if (n_new == 0) return cudaSuccess;
  if (n_new > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (maps != nullptr)
    return launch_tma_append(k_new, v_new, *maps, cache_len, nullptr, n_new, capacity,
                             heads * row_bytes, s);
  dim3 grid(static_cast<unsigned>(n_new), 2);
  kv_append_kernel<<<grid, kThreads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), cache_len, capacity, heads, CH);
  return cudaGetLastError();
}

}  // namespace ws
