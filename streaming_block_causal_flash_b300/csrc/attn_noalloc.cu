// attn_noalloc.cu -- ws_block_causal_attn_noalloc: the newest unit's attention
// against the cache, for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer for the split-KV
// workspace: code that runs under a memory pool it does not own, plug-ins
// loaded into a host process that forbids cudaMalloc after start-up, or
// real-time loops that must not call an allocator (cudaMalloc can block and
// synchronise the device).  For them this file holds one file-scope device
// array that serves as the workspace of every call.  The array is part of the
// library's device image: the driver reserves it on each GPU when it loads
// this module there, and it stays reserved until the process exits.
//
// Host code cannot use the array's name as a device address (on the host the
// name refers to a host-side stand-in), so the device address is looked up
// with cudaGetSymbolAddress once per device, with that device current, the
// first time the entry point runs on it.  The address belongs to the device's
// current context: if that context is destroyed and replaced (for example by
// cudaDeviceReset), the module is loaded again at a new address.  So the
// cached address is kept together with the unique id of the context it was
// looked up in, and looked up again when the current context's id differs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/ws.h"
#include "ws_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// 40 MiB: the split-KV partials of one unit call need
// CTAs x 2 x 256 rows x 129 floats (1,032 B a row) -- 39.1 MB with one CTA on
// each of a B300's 148 SMs, whatever the cache length or unit size.  This
// covers any GPU of up to 158 SMs.
constexpr size_t kScratchBytes = WS_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if it cannot be read;
// the cache is then keyed on the device alone).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device and context and cached.
ws_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "ws_block_causal_attn_noalloc: cudaGetDevice: %s",
             cudaGetErrorString(e));
    return ws::record_failure(WS_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices)
    return ws::record_failure(WS_ERR_CUDA, "ws_block_causal_attn_noalloc: device index too large");
  // 0 when the thread has no current context yet: the look-up below creates
  // it, and its id is read again afterwards.
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr || (ctx != 0 && g_scratch_ctx[dev] != ctx)) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg),
               "ws_block_causal_attn_noalloc: cudaGetSymbolAddress of the static scratch: %s",
               cudaGetErrorString(e));
      return ws::record_failure(WS_ERR_CUDA, msg);
    }
    if (ctx == 0) ctx = current_context_id();
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return WS_OK;
}

}  // namespace

extern "C" {

ws_status ws_block_causal_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       void* out, float* lse_or_null, const int32_t* h_offsets,
                                       const int32_t* d_offsets, int n_blocks, int64_t capacity,
                                       int num_heads, int head_dim, float softmax_scale,
                                       ws_dtype dt, ws_stream_t stream) {
  void* scratch = nullptr;
  ws_status st = scratch_address(&scratch);
  if (st != WS_OK) return st;
  // Size check against the static maximum, when the offsets can be read;
  // every other argument problem is reported by the full validation below.
  if (dt == WS_BF16 && h_offsets != nullptr && n_blocks >= 1 && num_heads >= 1 &&
      h_offsets[0] == 0) {
    const int64_t kv_len = h_offsets[n_blocks];
    const int64_t q_len = kv_len - h_offsets[n_blocks - 1];
    const size_t need = ws_block_causal_attn_workspace_size(q_len, kv_len, num_heads, head_dim);
    if (need != SIZE_MAX && need > kScratchBytes) {
      char msg[320];
      snprintf(msg, sizeof(msg),
               "ws_block_causal_attn_noalloc: these sizes need %zu bytes of scratch, more than "
               "the %zu-byte static scratch holds; use ws_block_causal_attn with a caller "
               "workspace",
               need, kScratchBytes);
      return ws::record_failure(WS_ERR_CAPACITY, msg);
    }
  }
  return ws_block_causal_attn(q, k_cache, v_cache, out, lse_or_null, h_offsets, d_offsets,
                              n_blocks, capacity, num_heads, head_dim, softmax_scale, dt, scratch,
                              kScratchBytes, stream);
}

}  // extern "C"
