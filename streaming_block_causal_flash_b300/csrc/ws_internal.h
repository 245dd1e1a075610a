// ws_internal.h -- host-side launchers shared between the C-ABI layer
// (ws_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ws.h"

namespace ws {

// Sets the thread-local ws_last_error() message and returns s (ws_api.cu).
ws_status record_failure(ws_status s, const char* msg);

// ---- KV append (kv_append.cu)
// Tensor maps of the K and V caches for the TMA append: 16-bit elements,
// dims (row_bytes / 2, heads, capacity) with byte strides (capacity *
// row_bytes, row_bytes), box (row_bytes / 2, heads, 1), no swizzle.  Null
// maps select the plain-load/store kernel (sizes the TMA path cannot take).
struct AppendMaps {
  CUtensorMap k;
  CUtensorMap v;
};
// Largest slice row (all heads of one token) the TMA append stages in
// shared memory, and the largest head count of its box.
constexpr int kTmaAppendMaxTokenBytes = 200 * 1024;
constexpr int kTmaAppendMaxHeads = 256;
constexpr int kTmaAppendMaxRowBytes = 512;

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             int64_t cache_len, int64_t n_new, int64_t capacity, int heads,
                             int row_bytes, const AppendMaps* maps, cudaStream_t s);

// Device-resident unit sizes (kv_append.cu): state = {cache_len, n_new, unit}.
cudaError_t launch_kv_append_dev(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const long long* state, int64_t n_max,
                                 int64_t capacity, int heads, int row_bytes,
                                 const AppendMaps* maps, cudaStream_t s);
cudaError_t launch_unit_state_advance(long long* state, const int32_t* sizes, int64_t n_sizes,
                                      cudaStream_t s);
cudaError_t read_unit_device_error(int* code, int* info);
cudaError_t clear_unit_device_error();

// ---- Flow-matching Euler step (fm_euler.cu)
cudaError_t launch_fm_euler(float* z, const void* v, bool v_is_bf16, void* z_bf16_out,
                            int64_t n, float dtau, int num_sms, cudaStream_t s);
cudaError_t launch_fm_euler_cfg(float* z, const void* v_uncond, const void* v_cond, bool v_is_bf16,
                                void* z_bf16_out, int64_t n, float guidance, float dtau,
                                int num_sms, cudaStream_t s);

// ---- fp32 SIMT attention (attn_simt.cu)
struct SimtAttnArgs {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;            // may be null
  const int32_t* offs;   // device offsets
  int n_blocks;
  int q_len;
  int q_row0;            // global token index of q row 0
  int kv_len;            // keys visible to every row (unit mode)
  int heads;
  int head_dim;          // 64 or 128
  int64_t capacity;
  float scale;           // softmax scale (natural units)
  bool prefill;          // per-row limits from offsets
};
cudaError_t launch_attn_simt_f32(const SimtAttnArgs& a, cudaStream_t s);

// ---- bf16 tcgen05 attention (attn_tcgen05.cu)
struct TcAttnPlan {
  int prefill;       // 0: one query block vs. the cache (split-KV groups); 1: prefill
  int heads;
  int q_len;
  int q_row0;
  int kv_len;
  int n_blocks;
  int qtiles;        // ceil(q_len / 128)
  int pairs;         // ceil(qtiles / 2): query-tile pairs per head (one CTA each)
  int kv_tiles;      // ceil(kv_len / 128)
  int groups;        // unit mode: CTA groups over the (head, key tile) space
  int64_t work;      // unit mode: heads * kv_tiles
  int n_items;       // prefill mode: heads * ceil(pairs / 2) (mirrored couples of pairs)
  int grid;          // CTAs launched
  bool split;        // unit mode: some head's key range spans several groups
  size_t workspace_bytes;
  int side_len;      // unit mode: keys of the newest block read from side buffers (0: none)
  int kv_tiles_c;    // side mode: key tiles of the cache part
  int solo;          // unit mode, odd tile count: the last query tile has solo CTAs
                     // (pairs then counts the full pairs, groups the paired groups)
  int solo_groups;   // groups of solo CTAs
};
// Fills the plan for the given sizes; returns false when the sizes do not fit.
// allow_solo: give an unpaired last query tile CTAs of its own (host-sized
// unit launches; launches sized for the largest unit keep plain pairs).
bool plan_tc_attn(TcAttnPlan& p, bool prefill, int heads, int q_len, int q_row0, int kv_len,
                  int n_blocks, int num_sms, int side_len = 0, bool allow_solo = true);

// Q, K and V reach the kernel through the tensor maps alone.
struct TcAttnArgs {
  void* out;
  float* lse;            // may be null
  const int32_t* offs;   // device offsets
  int64_t capacity;
  float scale;           // softmax scale (natural units)
  void* workspace;
  int force_stall;       // test hook (ws_debug_force_wait_timeout)
  int commit;            // side mode: also write the side K/V into the cache
  // Device-resident unit sizes {cache_len, n_new} (ws_unit_state), read by the
  // kernels at run time; null for host-sized launches.  With it the plan
  // must be made for q_len = the largest unit and kv_len = capacity, with
  // split forced on (workspace and merge for any key range).
  const long long* dev_state;
};
// Forces the split-KV merge and its workspace on (device-resident sizes,
// where a launch can split any head's key range).
void plan_force_split(TcAttnPlan& p);
// tm_kc / tm_vc (side mode with commit): the K/V caches as [H][rows][D]
// with rows = cache_len + the side length, 128-byte swizzle, box (64, 128, 1):
// the commit's TMA stores write the side tiles through them, clipped at the
// unit's last row.  Without commit they are not read.
cudaError_t launch_attn_tc_bf16(const TcAttnPlan& plan, const TcAttnArgs& a,
                                const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, const CUtensorMap& tm_ks,
                                const CUtensorMap& tm_vs, const CUtensorMap& tm_kc,
                                const CUtensorMap& tm_vc, uint64_t timeout_ns, cudaStream_t s);
cudaError_t read_attn_device_error(int* code, int* info);
cudaError_t clear_attn_device_error();

}  // namespace ws
