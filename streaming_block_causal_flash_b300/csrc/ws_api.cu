// ws_api.cu -- the C ABI declared in include/ws.h: argument validation,
// status codes, launch sizing and TMA tensor-map encoding.  Every check runs
// on the host before anything is launched; a call that fails a check
// launches nothing and touches no memory.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/ws.h"
#include "ws_internal.h"

namespace {

thread_local char g_last_error[512] = "";
// Process-wide settings read by every attention call on any thread.  Atomic
// (relaxed: each value stands alone), so a setter racing a call is not a data
// race; a call uses whichever value it reads at its start.
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_force_stall{0};

ws_status fail(ws_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

ws_status cuda_fail(cudaError_t e, const char* what) {
  return fail(WS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

ws_status ok() {
  g_last_error[0] = '\0';
  return WS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t dtype_size(ws_dtype dt) { return dt == WS_BF16 ? 2 : 4; }

bool valid_dtype(ws_dtype dt) { return dt == WS_BF16 || dt == WS_F32; }

// Per-device SM count, queried once.
int device_sms(int* dev_out) {
  static std::mutex mu;
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (dev_out) *dev_out = dev;
  std::lock_guard<std::mutex> lock(mu);
  if (sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    sms[dev] = v;
  }
  return sms[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle, zero fill outside the tensor.
bool encode_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                 const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                  const_cast<void*>(base), dims, strides_bytes, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor maps for the TMA append (see ws::AppendMaps).  Returns false when the
// sizes do not fit that path; the plain-copy kernel then runs instead.
bool encode_append_maps(ws::AppendMaps& m, void* k_cache, void* v_cache, int heads,
                        int64_t row_bytes, int64_t capacity) {
  if (heads > ws::kTmaAppendMaxHeads || row_bytes > ws::kTmaAppendMaxRowBytes ||
      heads * row_bytes > ws::kTmaAppendMaxTokenBytes || capacity > (int64_t)INT32_MAX)
    return false;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)(row_bytes / 2), (cuuint64_t)heads, (cuuint64_t)capacity};
  cuuint64_t strides[2] = {(cuuint64_t)capacity * (cuuint64_t)row_bytes, (cuuint64_t)row_bytes};
  cuuint32_t box[3] = {(cuuint32_t)(row_bytes / 2), (cuuint32_t)heads, 1};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = fn(i == 0 ? &m.k : &m.v, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, i == 0 ? k_cache : v_cache,
                    dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

// Shared validation for the two attention entry points.
ws_status check_attn_args(const char* who, const void* q, const void* k_cache,
                          const void* v_cache, void* out, const float* lse,
                          const int32_t* h_offsets, const int32_t* d_offsets, int n_blocks,
                          int64_t capacity, int num_heads, int head_dim, float softmax_scale,
                          ws_dtype dt, bool side, bool commit) {
  if (!valid_dtype(dt)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: unknown dtype %d", who, (int)dt);
  if (!q || !k_cache || !v_cache || !out || !h_offsets || !d_offsets)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer argument", who);
  if (n_blocks < 1) return fail(WS_ERR_INVALID_ARGUMENT, "%s: n_blocks must be >= 1", who);
  if (num_heads < 1) return fail(WS_ERR_INVALID_ARGUMENT, "%s: num_heads must be >= 1", who);
  if (capacity < 1 || capacity > (int64_t)INT32_MAX)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: capacity out of range", who);
  if (!(softmax_scale >= 0.f) || !std::isfinite(softmax_scale))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: softmax_scale must be finite and >= 0", who);
  if (h_offsets[0] != 0) return fail(WS_ERR_INVALID_ARGUMENT, "%s: offsets[0] must be 0", who);
  for (int b = 0; b < n_blocks; ++b)
    if (h_offsets[b + 1] < h_offsets[b])
      return fail(WS_ERR_INVALID_ARGUMENT, "%s: offsets decrease at block %d", who, b);
  // The cache holds every block read from it: all of them, or, when the
  // newest block comes from side buffers, the ones before it.
  const int cached = (side && !commit) ? n_blocks - 1 : n_blocks;
  if ((int64_t)h_offsets[cached] > capacity)
    return fail(WS_ERR_CAPACITY, "%s: offsets[%d]=%d exceeds capacity %lld", who, cached,
                h_offsets[cached], (long long)capacity);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: q/k/v/out must be 16-byte aligned", who);
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: lse must be 4-byte aligned", who);
  const bool bf16_ok = dt == WS_BF16 && head_dim == 128;
  const bool f32_ok = dt == WS_F32 && (head_dim == 64 || head_dim == 128);
  if (!bf16_ok && !f32_ok)
    return fail(WS_ERR_UNSUPPORTED, "%s: dtype %s with head_dim %d is not implemented", who,
                dt == WS_BF16 ? "bf16" : "f32", head_dim);
  if ((int64_t)num_heads * head_dim > 65535)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: num_heads*head_dim too large", who);
  return WS_OK;
}

ws_status run_attention(const char* who, bool prefill, const void* q, const void* k_cache,
                        const void* v_cache, const void* k_side, const void* v_side, bool commit,
                        void* out, float* lse, const int32_t* h_offsets,
                        const int32_t* d_offsets, int n_blocks, int64_t capacity, int num_heads,
                        int head_dim, float softmax_scale, ws_dtype dt, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  const bool side = k_side != nullptr || v_side != nullptr;
  ws_status st = check_attn_args(who, q, k_cache, v_cache, out, lse, h_offsets, d_offsets,
                                 n_blocks, capacity, num_heads, head_dim, softmax_scale, dt, side,
                                 side && commit);
  if (st != WS_OK) return st;
  if (side) {
    if (!k_side || !v_side)
      return fail(WS_ERR_INVALID_ARGUMENT, "%s: k_side and v_side are both required", who);
    if (!aligned16(k_side) || !aligned16(v_side))
      return fail(WS_ERR_INVALID_ARGUMENT, "%s: side buffers must be 16-byte aligned", who);
    if (dt != WS_BF16)
      return fail(WS_ERR_UNSUPPORTED, "%s: side buffers are implemented for bf16 only", who);
  }
  const int kv_len = h_offsets[n_blocks];
  const int q_row0 = prefill ? 0 : h_offsets[n_blocks - 1];
  const int q_len = kv_len - q_row0;
  if (q_len == 0) return ok();
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)head_dim);

  if (dt == WS_F32) {
    ws::SimtAttnArgs a{};
    a.q = static_cast<const float*>(q);
    a.k = static_cast<const float*>(k_cache);
    a.v = static_cast<const float*>(v_cache);
    a.out = static_cast<float*>(out);
    a.lse = lse;
    a.offs = d_offsets;
    a.n_blocks = n_blocks;
    a.q_len = q_len;
    a.q_row0 = q_row0;
    a.kv_len = kv_len;
    a.heads = num_heads;
    a.head_dim = head_dim;
    a.capacity = capacity;
    a.scale = scale;
    a.prefill = prefill;
    cudaError_t e = ws::launch_attn_simt_f32(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return ok();
  }

  int dev = 0;
  const int sms = device_sms(&dev);
  if (sms <= 0) return fail(WS_ERR_CUDA, "%s: cannot query the current device", who);
  ws::TcAttnPlan plan;
  if (!ws::plan_tc_attn(plan, prefill, num_heads, q_len, q_row0, kv_len, n_blocks, sms,
                        side ? q_len : 0))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: sizes out of range", who);
  if (plan.workspace_bytes > 0) {
    if (!workspace || workspace_bytes < plan.workspace_bytes)
      return fail(WS_ERR_INVALID_ARGUMENT, "%s: workspace of %zu bytes needed, %zu given", who,
                  plan.workspace_bytes, workspace ? workspace_bytes : (size_t)0);
    if (!aligned16(workspace))
      return fail(WS_ERR_INVALID_ARGUMENT, "%s: workspace must be 16-byte aligned", who);
  }
  // TMA maps: Q as a 2-D [q_len][H*D] matrix; K and V as 3-D [H][rows][D]
  // views of the [H][capacity][D] caches, rows = the keys read from the cache
  // (kv_len, or q_row0 with side buffers), so rows beyond read as zeros; the
  // side buffers, like Q, as 2-D [q_len][H*D] matrices.
  CUtensorMap tm_q, tm_k, tm_v, tm_ks, tm_vs;
  const cuuint64_t D = (cuuint64_t)head_dim;
  {
    cuuint64_t dims[2] = {D * (cuuint64_t)num_heads, (cuuint64_t)q_len};
    cuuint64_t strides[1] = {D * (cuuint64_t)num_heads * 2};
    cuuint32_t box[2] = {64, 128};
    if (!encode_bf16(&tm_q, q, 2, dims, strides, box))
      return fail(WS_ERR_CUDA, "%s: cannot encode the Q tensor map", who);
  }
  {
    // a cache part of 0 rows (first unit, side mode) still needs a valid map
    const int rows = side ? (q_row0 > 0 ? q_row0 : 1) : kv_len;
    cuuint64_t dims[3] = {D, (cuuint64_t)rows, (cuuint64_t)num_heads};
    cuuint64_t strides[2] = {D * 2, (cuuint64_t)capacity * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    if (!encode_bf16(&tm_k, k_cache, 3, dims, strides, box) ||
        !encode_bf16(&tm_v, v_cache, 3, dims, strides, box))
      return fail(WS_ERR_CUDA, "%s: cannot encode the K/V tensor maps", who);
  }
  if (side) {
    cuuint64_t dims[2] = {D * (cuuint64_t)num_heads, (cuuint64_t)q_len};
    cuuint64_t strides[1] = {D * (cuuint64_t)num_heads * 2};
    cuuint32_t box[2] = {64, 128};
    if (!encode_bf16(&tm_ks, k_side, 2, dims, strides, box) ||
        !encode_bf16(&tm_vs, v_side, 2, dims, strides, box))
      return fail(WS_ERR_CUDA, "%s: cannot encode the side-buffer tensor maps", who);
  } else {
    tm_ks = tm_k;    // unused without side buffers
    tm_vs = tm_v;
  }
  // the commit's store maps: the caches with rows ending at the unit's last
  // row (cache_len + q_len), so a ragged last side tile is clipped there
  CUtensorMap tm_kc = tm_k, tm_vc = tm_v;
  if (side && commit) {
    cuuint64_t dims[3] = {D, (cuuint64_t)(q_row0 + q_len), (cuuint64_t)num_heads};
    cuuint64_t strides[2] = {D * 2, (cuuint64_t)capacity * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    if (!encode_bf16(&tm_kc, k_cache, 3, dims, strides, box) ||
        !encode_bf16(&tm_vc, v_cache, 3, dims, strides, box))
      return fail(WS_ERR_CUDA, "%s: cannot encode the commit tensor maps", who);
  }
  ws::TcAttnArgs a{};
  a.out = out;
  a.lse = lse;
  a.offs = d_offsets;
  a.capacity = capacity;
  a.scale = scale;
  a.workspace = workspace;
  a.force_stall = g_force_stall.load(std::memory_order_relaxed);
  a.commit = (side && commit) ? 1 : 0;
  cudaError_t e = ws::launch_attn_tc_bf16(plan, a, tm_q, tm_k, tm_v, tm_ks, tm_vs, tm_kc, tm_vc,
                                          g_timeout_ns.load(std::memory_order_relaxed), stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

// Bytes of split-KV workspace for a launch sized by the device-resident
// variant (largest unit q_max, whole cache), or 0 when the plan fails.
size_t dev_workspace_bytes(int64_t q_max, int64_t capacity, int num_heads, int sms) {
  ws::TcAttnPlan plan;
  if (!ws::plan_tc_attn(plan, false, num_heads, (int)q_max, (int)(capacity - q_max), (int)capacity,
                        1, sms, 0, false))
    return 0;
  ws::plan_force_split(plan);
  return plan.workspace_bytes;
}

}  // namespace

namespace ws {

// Lets entry points defined in other files report a failure through
// ws_last_error() on the calling thread.
ws_status record_failure(ws_status s, const char* msg) { return fail(s, "%s", msg); }

}  // namespace ws

extern "C" {

int ws_abi_version(void) { return 101; }

const char* ws_status_string(ws_status s) {
  switch (s) {
    case WS_OK: return "WS_OK";
    case WS_ERR_INVALID_ARGUMENT: return "WS_ERR_INVALID_ARGUMENT";
    case WS_ERR_UNSUPPORTED: return "WS_ERR_UNSUPPORTED";
    case WS_ERR_CAPACITY: return "WS_ERR_CAPACITY";
    case WS_ERR_CUDA: return "WS_ERR_CUDA";
    case WS_ERR_TIMEOUT: return "WS_ERR_TIMEOUT";
  }
  return "WS_ERR_UNKNOWN";
}

const char* ws_last_error(void) { return g_last_error; }

ws_status ws_set_wait_timeout_ns(uint64_t timeout_ns) {
  if (timeout_ns == 0) return fail(WS_ERR_INVALID_ARGUMENT, "ws_set_wait_timeout_ns: must be > 0");
  g_timeout_ns.store(timeout_ns, std::memory_order_relaxed);
  return ok();
}

ws_status ws_debug_force_wait_timeout(int on) {
  g_force_stall.store(on ? 1 : 0, std::memory_order_relaxed);
  return ok();
}

ws_status ws_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       int64_t cache_len, int64_t n_new, int64_t capacity, int num_heads,
                       int head_dim, ws_dtype dt, ws_stream_t stream) {
  const char* who = "ws_kv_append";
  if (!valid_dtype(dt)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: unknown dtype", who);
  if (n_new < 0 || cache_len < 0 || capacity < 0 || num_heads < 1 || head_dim < 1)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: negative or zero size", who);
  if (n_new > capacity || cache_len > capacity - n_new)   // cache_len + n_new > capacity, without overflow
    return fail(WS_ERR_CAPACITY,"%s: cache_len %lld + n_new %lld exceeds capacity %lld", who,
                (long long)cache_len, (long long)n_new, (long long)capacity);
  const int64_t row_bytes = (int64_t)head_dim * (int64_t)dtype_size(dt);
  if (row_bytes % 16 != 0)
    return fail(WS_ERR_UNSUPPORTED, "%s: head_dim*sizeof(dtype) must be a multiple of 16", who);
  if ((int64_t)num_heads * row_bytes > (int64_t)INT32_MAX || n_new > (int64_t)INT32_MAX)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: slice too large", who);
  if (n_new == 0) return ok();
  if (!k_new || !v_new || !k_cache || !v_cache)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer argument", who);
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: pointers must be 16-byte aligned", who);
  ws::AppendMaps maps;
  const bool tma = encode_append_maps(maps, k_cache, v_cache, num_heads, row_bytes, capacity);
  cudaError_t e = ws::launch_kv_append(k_new, v_new, k_cache, v_cache, cache_len, n_new, capacity,
                                       num_heads, (int)row_bytes, tma ? &maps : nullptr, stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

ws_status ws_block_causal_attn(const void* q, const void* k_cache, const void* v_cache, void* out,
                               float* lse_or_null, const int32_t* h_offsets,
                               const int32_t* d_offsets, int n_blocks, int64_t capacity,
                               int num_heads, int head_dim, float softmax_scale, ws_dtype dt,
                               void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  return run_attention("ws_block_causal_attn", false, q, k_cache, v_cache, nullptr, nullptr, false, out,
                       lse_or_null,
                       h_offsets, d_offsets, n_blocks, capacity, num_heads, head_dim,
                       softmax_scale, dt, workspace, workspace_bytes, stream);
}

ws_status ws_block_causal_prefill(const void* q, const void* k_cache, const void* v_cache,
                                  void* out, float* lse_or_null, const int32_t* h_offsets,
                                  const int32_t* d_offsets, int n_blocks, int64_t capacity,
                                  int num_heads, int head_dim, float softmax_scale, ws_dtype dt,
                                  void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  return run_attention("ws_block_causal_prefill", true, q, k_cache, v_cache, nullptr, nullptr, false, out,
                       lse_or_null,
                       h_offsets, d_offsets, n_blocks, capacity, num_heads, head_dim,
                       softmax_scale, dt, workspace, workspace_bytes, stream);
}

ws_status ws_block_causal_attn_side(const void* q, const void* k_cache, const void* v_cache,
                                    const void* k_side, const void* v_side, int commit, void* out,
                                    float* lse_or_null, const int32_t* h_offsets,
                                    const int32_t* d_offsets, int n_blocks, int64_t capacity,
                                    int num_heads, int head_dim, float softmax_scale, ws_dtype dt,
                                    void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  const char* who = "ws_block_causal_attn_side";
  if (!k_side || !v_side)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: k_side and v_side are required", who);
  return run_attention(who, false, q, k_cache, v_cache, k_side, v_side, commit != 0, out, lse_or_null,
                       h_offsets, d_offsets, n_blocks, capacity, num_heads, head_dim,
                       softmax_scale, dt, workspace, workspace_bytes, stream);
}

ws_status ws_fm_euler_step(void* z, ws_dtype z_dt, const void* v, ws_dtype v_dt,
                           void* z_bf16_out_or_null, int64_t n_elems, float dtau,
                           ws_stream_t stream) {
  const char* who = "ws_fm_euler_step";
  if (z_dt != WS_F32) return fail(WS_ERR_UNSUPPORTED, "%s: z must be float32", who);
  if (!valid_dtype(v_dt)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: unknown v dtype", who);
  if (n_elems < 0) return fail(WS_ERR_INVALID_ARGUMENT, "%s: negative n_elems", who);
  if (!std::isfinite(dtau)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: dtau must be finite", who);
  if (n_elems == 0) return ok();
  if (!z || !v) return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer argument", who);
  if (!aligned16(z) || !aligned16(v) || (z_bf16_out_or_null && !aligned16(z_bf16_out_or_null)))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: pointers must be 16-byte aligned", who);
  const int sms = device_sms(nullptr);
  if (sms <= 0) return fail(WS_ERR_CUDA, "%s: cannot query the current device", who);
  cudaError_t e = ws::launch_fm_euler(static_cast<float*>(z), v, v_dt == WS_BF16,
                                      z_bf16_out_or_null, n_elems, dtau, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

ws_status ws_fm_euler_cfg_step(void* z, ws_dtype z_dt, const void* v_uncond, const void* v_cond,
                               ws_dtype v_dt, void* z_bf16_out_or_null, int64_t n_elems,
                               float guidance, float dtau, ws_stream_t stream) {
  const char* who = "ws_fm_euler_cfg_step";
  if (z_dt != WS_F32) return fail(WS_ERR_UNSUPPORTED, "%s: z must be float32", who);
  if (!valid_dtype(v_dt)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: unknown velocity dtype", who);
  if (n_elems < 0) return fail(WS_ERR_INVALID_ARGUMENT, "%s: negative n_elems", who);
  if (!std::isfinite(dtau) || !std::isfinite(guidance))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: dtau and guidance must be finite", who);
  if (n_elems == 0) return ok();
  if (!z || !v_uncond || !v_cond) return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer argument", who);
  if (!aligned16(z) || !aligned16(v_uncond) || !aligned16(v_cond) ||
      (z_bf16_out_or_null && !aligned16(z_bf16_out_or_null)))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: pointers must be 16-byte aligned", who);
  const int sms = device_sms(nullptr);
  if (sms <= 0) return fail(WS_ERR_CUDA, "%s: cannot query the current device", who);
  cudaError_t e = ws::launch_fm_euler_cfg(static_cast<float*>(z), v_uncond, v_cond, v_dt == WS_BF16,
                                          z_bf16_out_or_null, n_elems, guidance, dtau, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

size_t ws_block_causal_attn_workspace_size(int64_t q_len, int64_t kv_len, int num_heads,
                                           int head_dim) {
  if (q_len < 0 || kv_len < q_len || num_heads < 1 || head_dim < 1 || kv_len > INT32_MAX)
    return SIZE_MAX;
  if (head_dim != 128 || q_len == 0) return 0;
  const int sms = device_sms(nullptr);
  if (sms <= 0) return SIZE_MAX;
  // large enough for ws_block_causal_attn and for ws_block_causal_attn_side
  size_t need = 0;
  for (int side = 0; side < 2; ++side) {
    ws::TcAttnPlan plan;
    if (!ws::plan_tc_attn(plan, false, num_heads, (int)q_len, (int)(kv_len - q_len), (int)kv_len, 1,
                          sms, side ? (int)q_len : 0))
      return SIZE_MAX;
    if (plan.workspace_bytes > need) need = plan.workspace_bytes;
  }
  return need;
}

ws_status ws_kv_append_dev(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const ws_unit_state* d_state, int64_t n_max, int64_t capacity,
                           int num_heads, int head_dim, ws_dtype dt, ws_stream_t stream) {
  const char* who = "ws_kv_append_dev";
  if (!valid_dtype(dt)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: unknown dtype", who);
  if (n_max < 1 || capacity < n_max || num_heads < 1 || head_dim < 1)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: need 1 <= n_max <= capacity, heads and head_dim >= 1",
                who);
  const int64_t row_bytes = (int64_t)head_dim * (int64_t)dtype_size(dt);
  if (row_bytes % 16 != 0)
    return fail(WS_ERR_UNSUPPORTED, "%s: head_dim*sizeof(dtype) must be a multiple of 16", who);
  if ((int64_t)num_heads * row_bytes > (int64_t)INT32_MAX || n_max > (int64_t)INT32_MAX)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: slice too large", who);
  if (!k_new || !v_new || !k_cache || !v_cache || !d_state)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer argument", who);
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(d_state) & 7u))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: misaligned pointer", who);
  ws::AppendMaps maps;
  const bool tma = encode_append_maps(maps, k_cache, v_cache, num_heads, row_bytes, capacity);
  cudaError_t e = ws::launch_kv_append_dev(k_new, v_new, k_cache, v_cache,
                                           reinterpret_cast<const long long*>(d_state), n_max,
                                           capacity, num_heads, (int)row_bytes,
                                           tma ? &maps : nullptr, stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

size_t ws_block_causal_attn_dev_workspace_size(int64_t q_max, int64_t capacity, int num_heads,
                                               int head_dim) {
  if (q_max < 1 || capacity < q_max || capacity > INT32_MAX || num_heads < 1 || head_dim != 128)
    return SIZE_MAX;
  const int sms = device_sms(nullptr);
  if (sms <= 0) return SIZE_MAX;
  const size_t need = dev_workspace_bytes(q_max, capacity, num_heads, sms);
  return need == 0 ? SIZE_MAX : need;
}

ws_status ws_block_causal_attn_dev(const void* q, const void* k_cache, const void* v_cache,
                                   void* out, float* lse_or_null, const ws_unit_state* d_state,
                                   int64_t q_max, int64_t capacity, int num_heads, int head_dim,
                                   float softmax_scale, ws_dtype dt, void* workspace,
                                   size_t workspace_bytes, ws_stream_t stream) {
  const char* who = "ws_block_causal_attn_dev";
  if (!valid_dtype(dt)) return fail(WS_ERR_INVALID_ARGUMENT, "%s: unknown dtype %d", who, (int)dt);
  if (dt != WS_BF16 || head_dim != 128)
    return fail(WS_ERR_UNSUPPORTED, "%s: implemented for bf16 with head_dim 128", who);
  if (!q || !k_cache || !v_cache || !out || !d_state || !workspace)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer argument", who);
  if (num_heads < 1 || (int64_t)num_heads * head_dim > 65535)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: num_heads out of range", who);
  if (q_max < 1 || capacity < q_max || capacity > (int64_t)INT32_MAX)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: need 1 <= q_max <= capacity <= INT32_MAX", who);
  if (!(softmax_scale >= 0.f) || !std::isfinite(softmax_scale))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: softmax_scale must be finite and >= 0", who);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(d_state) & 7u) ||
      (lse_or_null && (reinterpret_cast<uintptr_t>(lse_or_null) & 3u)))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: misaligned pointer", who);
  int dev = 0;
  const int sms = device_sms(&dev);
  if (sms <= 0) return fail(WS_ERR_CUDA, "%s: cannot query the current device", who);
  ws::TcAttnPlan plan;
  if (!ws::plan_tc_attn(plan, false, num_heads, (int)q_max, (int)(capacity - q_max), (int)capacity,
                        1, sms, 0, false))
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: sizes out of range", who);
  ws::plan_force_split(plan);
  if (workspace_bytes < plan.workspace_bytes)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: workspace of %zu bytes needed, %zu given", who,
                plan.workspace_bytes, workspace_bytes);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)head_dim);
  // Q as a 2-D [q_max][H*D] matrix (rows past the unit are read, never
  // written back); K and V as 3-D [H][capacity][D] views of the whole cache
  // (the kernels mask keys at the run-time length).
  CUtensorMap tm_q, tm_k, tm_v;
  const cuuint64_t D = (cuuint64_t)head_dim;
  {
    cuuint64_t dims[2] = {D * (cuuint64_t)num_heads, (cuuint64_t)q_max};
    cuuint64_t strides[1] = {D * (cuuint64_t)num_heads * 2};
    cuuint32_t box[2] = {64, 128};
    if (!encode_bf16(&tm_q, q, 2, dims, strides, box))
      return fail(WS_ERR_CUDA, "%s: cannot encode the Q tensor map", who);
  }
  {
    cuuint64_t dims[3] = {D, (cuuint64_t)capacity, (cuuint64_t)num_heads};
    cuuint64_t strides[2] = {D * 2, (cuuint64_t)capacity * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    if (!encode_bf16(&tm_k, k_cache, 3, dims, strides, box) ||
        !encode_bf16(&tm_v, v_cache, 3, dims, strides, box))
      return fail(WS_ERR_CUDA, "%s: cannot encode the K/V tensor maps", who);
  }
  ws::TcAttnArgs a{};
  a.out = out;
  a.lse = lse_or_null;
  a.offs = nullptr;
  a.capacity = capacity;
  a.scale = scale;
  a.workspace = workspace;
  a.force_stall = g_force_stall.load(std::memory_order_relaxed);
  a.dev_state = reinterpret_cast<const long long*>(d_state);
  cudaError_t e = ws::launch_attn_tc_bf16(plan, a, tm_q, tm_k, tm_v, tm_k, tm_v, tm_k, tm_v,
                                          g_timeout_ns.load(std::memory_order_relaxed), stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

ws_status ws_unit_state_advance(ws_unit_state* d_state, const int32_t* d_sizes, int64_t n_sizes,
                                ws_stream_t stream) {
  const char* who = "ws_unit_state_advance";
  if (!d_state || (n_sizes > 0 && !d_sizes) || n_sizes < 0)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: null pointer or negative size", who);
  if (reinterpret_cast<uintptr_t>(d_state) & 7u)
    return fail(WS_ERR_INVALID_ARGUMENT, "%s: misaligned state", who);
  cudaError_t e = ws::launch_unit_state_advance(reinterpret_cast<long long*>(d_state), d_sizes,
                                                n_sizes, stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

ws_status ws_get_device_error(int* code_out, int* info_out) {
  if (!code_out || !info_out) return fail(WS_ERR_INVALID_ARGUMENT, "ws_get_device_error: null");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "ws_get_device_error");
  e = ws::read_attn_device_error(code_out, info_out);
  if (e != cudaSuccess) return cuda_fail(e, "ws_get_device_error");
  if (*code_out == 0) {
    // the append and state kernels keep their own word
    e = ws::read_unit_device_error(code_out, info_out);
    if (e != cudaSuccess) return cuda_fail(e, "ws_get_device_error");
  }
  if (*code_out == 1)
    return fail(WS_ERR_TIMEOUT, "in-kernel wait gave up (site %d, block %d)", *info_out >> 16,
                *info_out & 0xFFFF);
  if (*code_out == 2)
    return fail(WS_ERR_CAPACITY, "device-resident unit sizes out of range (%s); nothing was written",
                *info_out == 1 ? "n_new outside [0, the launch's maximum]"
                               : "cache_len + n_new outside [0, capacity]");
  if (*code_out == 3)
    return fail(WS_ERR_CUDA,
                "debug build: an out-of-bounds access was caught and skipped (check site %d, block %d)",
                *info_out >> 16, *info_out & 0xFFFF);
  if (*code_out != 0) return fail(WS_ERR_CUDA, "unknown device error code %d", *code_out);
  return ok();
}

ws_status ws_clear_device_error(void) {
  cudaError_t e = ws::clear_attn_device_error();
  if (e == cudaSuccess) e = ws::clear_unit_device_error();
  if (e != cudaSuccess) return cuda_fail(e, "ws_clear_device_error");
  return ok();
}

}  // extern "C"
