/*
 * ws.h -- C ABI of the streaming block-causal hot path (B300, sm_103a).
 *
 * One streaming unit (about 160 ms of interleaved video-latent, audio and
 * text tokens) is one attention block.  Per unit the path is:
 *   1. ws_kv_append          append the unit's K/V slice to the full-history cache
 *   2. ws_block_causal_attn  the unit's queries against the whole cache
 *   3. ws_fm_euler_step      the flow-matching Euler update, once per solver step
 * and, once per session, ws_block_causal_prefill over a whole token sequence.
 *
 * Sources (web pages about Wan-Streamer, cited by title and section):
 *  [explainer]  Wan Streamer real-time AV explainer (xiaohu-jiedu.pages.dev),
 *               "怎么做到边听边说、随时能打断" -- block-causal visibility;
 *               "点开看部署细节" -- prefill, then the shared full-history cache.
 *  [close-read] "全双工语音模型精读⑫：Wan-Streamer——当全双工长出一张脸"
 *               (alwayszhang.cn), 3.2 -- flow-matching interpolant/velocity;
 *               四、推理 steps 1-3 -- the performer appends the received KV
 *               slice to its full-history cache, then runs the flow solver.
 *  [youleyou]   "阿里通义万相发布亚秒级同步AI视频通话基础模型" (youleyou.com),
 *               3.1 -- block-causal attention over the interleaved sequence;
 *               3.3 -- the performer runs only the flow-matching solver.
 *
 * Conventions shared by every call
 *  - Ownership: the caller owns every buffer; the library allocates no device
 *    memory.  Scratch for split-KV attention is a caller-supplied workspace
 *    sized by ws_block_causal_attn_workspace_size().
 *  - Streams: every call is asynchronous on the caller's stream (NULL = the
 *    legacy default stream) and never synchronises.
 *  - Errors: every call returns a ws_status.  A call that fails validation
 *    launches nothing and touches no memory.  ws_last_error() gives a
 *    thread-local message for the last failure on the calling thread.
 *  - Pointers marked "device" are device addresses.  Pointers marked "host"
 *    are ordinary host memory read during the call only.
 *  - Alignment: every device tensor pointer must be 16-byte aligned.
 *  - Dtypes: WS_BF16 (bfloat16) or WS_F32 (float32).
 */
#ifndef WS_H_
#define WS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WS_API __attribute__((visibility("default")))
#else
#define WS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* ws_stream_t;

typedef enum {
  WS_OK = 0,
  WS_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, bad offsets, misalignment */
  WS_ERR_UNSUPPORTED = 2,      /* dtype / head_dim combination not implemented */
  WS_ERR_CAPACITY = 3,         /* write or read past the cache capacity */
  WS_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
  WS_ERR_TIMEOUT = 5           /* a bounded in-kernel wait gave up (device error word) */
} ws_status;

typedef enum { WS_F32 = 0, WS_BF16 = 1 } ws_dtype;

/*
 * ws_kv_append -- write one unit's K/V slice into the full-history cache.
 * [close-read] 四、推理 step 3; [youleyou] 3.3.
 *
 *   k_cache[h][cache_len + t][:] = k_new[t][h][:]   (same for V)
 *   for 0 <= t < n_new, 0 <= h < num_heads.  A bit copy; no other cache row
 *   changes.
 *
 * k_new, v_new    device, [n_new][num_heads][head_dim], token-major, dtype dt
 * k_cache, v_cache device, [num_heads][capacity][head_dim], dtype dt
 * Requires 0 <= cache_len, n_new >= 0, cache_len + n_new <= capacity
 * (else WS_ERR_CAPACITY), head_dim * sizeof(dt) a multiple of 16.
 * n_new == 0 is a no-op.
 */
WS_API ws_status ws_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       int64_t cache_len, int64_t n_new, int64_t capacity, int num_heads,
                       int head_dim, ws_dtype dt, ws_stream_t stream);

/*
 * ws_block_causal_attn -- attention of the newest unit's tokens against the
 * whole cache.  [explainer] "怎么做到边听边说": tokens see their own block in
 * both directions and every earlier block, never a later one; [youleyou] 3.1.
 *
 * The blocks are given by offsets[0..n_blocks] (offsets[0] = 0,
 * non-decreasing).  The query block is the last one, blk = n_blocks - 1,
 * holding q_len = offsets[n_blocks] - offsets[n_blocks-1] tokens; the cache
 * must already hold blocks 0..blk (append first, then attend).  Every query
 * row therefore sees the keys j < kv_len = offsets[n_blocks]:
 *
 *   O[i][h] = sum_j softmax_j(s * <q[i][h], k[h][j]>) v[h][j],  j < kv_len
 *   lse[h][i] = ln sum_j exp(s * <q[i][h], k[h][j]>)             (natural log)
 *
 * q           device, [q_len][num_heads][head_dim], dtype dt
 * k_cache,
 * v_cache     device, [num_heads][capacity][head_dim], dtype dt
 * out         device, [q_len][num_heads][head_dim], dtype dt
 * lse_or_null device float32 [num_heads][q_len], or NULL
 * h_offsets   host int32 [n_blocks + 1] (validation and launch sizing)
 * d_offsets   device int32 [n_blocks + 1], same values (read by kernels)
 * softmax_scale  s > 0; 0 selects 1/sqrt(head_dim); negative is rejected
 * workspace   device scratch of at least
 *             ws_block_causal_attn_workspace_size(q_len, kv_len, num_heads,
 *             head_dim) bytes (may be NULL when that size is 0); its contents
 *             on entry do not matter; concurrent calls must not share it.
 * Supported: (WS_BF16, head_dim 128) on tcgen05 tensor cores with fp32
 * accumulation and bf16 P; (WS_F32, head_dim 64 or 128) on fp32 CUDA cores.
 * Other combinations return WS_ERR_UNSUPPORTED.
 */
WS_API ws_status ws_block_causal_attn(const void* q, const void* k_cache, const void* v_cache, void* out,
                               float* lse_or_null, const int32_t* h_offsets,
                               const int32_t* d_offsets, int n_blocks, int64_t capacity,
                               int num_heads, int head_dim, float softmax_scale, ws_dtype dt,
                               void* workspace, size_t workspace_bytes, ws_stream_t stream);

/*
 * ws_block_causal_attn_side -- ws_block_causal_attn with the newest block's
 * keys and values read from side buffers instead of the cache.
 * [close-read] 四、推理 step 3 and [explainer] "点开看部署细节": the performer
 * runs the flow solver for the next unit over the full-history cache, and
 * the clean latents are committed to history only once denoised.  While the
 * solver iterates, the unit's own K/V change every step; they live in side
 * buffers, and only the final slice is committed with ws_kv_append.
 *
 * Same result as ws_kv_append(k_side, v_side, ..., cache_len =
 * offsets[n_blocks-1]) followed by ws_block_causal_attn, without touching the
 * cache: every query row of the last block sees the cache keys
 * j < offsets[n_blocks-1] and all q_len side keys.
 *
 * k_side, v_side  device, [q_len][num_heads][head_dim] token-major (the same
 *                 layout as a slice for ws_kv_append), dtype dt
 * commit          0: the cache is not written.  Nonzero: the kernel also
 *                 writes the side K/V into cache rows [offsets[n_blocks-1],
 *                 offsets[n_blocks]) of every head -- the same bytes
 *                 ws_kv_append would write (the append fused into the
 *                 attention: each side tile the kernel loads into shared
 *                 memory for the attention is also stored to the cache by
 *                 TMA, once per tile, before its slot is reused); the
 *                 solver's last step commits the clean slice this way.
 *                 Requires offsets[n_blocks] <= capacity.  Cache rows from
 *                 offsets[n_blocks] on are not written.
 * The cache must hold blocks 0..n_blocks-2 (offsets[n_blocks-1] <= capacity,
 * else WS_ERR_CAPACITY); rows from offsets[n_blocks-1] on are not read.
 * Other arguments, the workspace (same size query) and errors as
 * ws_block_causal_attn.  Implemented for WS_BF16 with head_dim 128 (other
 * combinations return WS_ERR_UNSUPPORTED).
 */
WS_API ws_status ws_block_causal_attn_side(const void* q, const void* k_cache, const void* v_cache,
                                           const void* k_side, const void* v_side, int commit,
                                           void* out,
                                           float* lse_or_null, const int32_t* h_offsets,
                                           const int32_t* d_offsets, int n_blocks,
                                           int64_t capacity, int num_heads, int head_dim,
                                           float softmax_scale, ws_dtype dt, void* workspace,
                                           size_t workspace_bytes, ws_stream_t stream);

/*
 * ws_block_causal_prefill -- full-sequence block-causal attention over all
 * T = offsets[n_blocks] tokens (the session prefill before streaming;
 * [explainer] "点开看部署细节").  Row i sees keys j < e(i), where e(i) is the
 * end offset of the block holding token i.  Key tiles that no row of a query
 * tile can see are skipped.
 *
 * q     device, [T][num_heads][head_dim]; out likewise; lse_or_null [H][T].
 * Caches, offsets, scale, dtype rules and errors as ws_block_causal_attn.
 * The prefill needs no workspace (pass NULL, 0).
 */
WS_API ws_status ws_block_causal_prefill(const void* q, const void* k_cache, const void* v_cache,
                                  void* out, float* lse_or_null, const int32_t* h_offsets,
                                  const int32_t* d_offsets, int n_blocks, int64_t capacity,
                                  int num_heads, int head_dim, float softmax_scale, ws_dtype dt,
                                  void* workspace, size_t workspace_bytes, ws_stream_t stream);

/*
 * ws_fm_euler_step -- one Euler step of the flow-matching solver towards
 * tau = 0.  [close-read] 3.2: z_tau = (1 - tau) z_0 + tau eps, velocity
 * dz/dtau = eps - z_0; the step is  z <- z - dtau * v  (in place).
 *
 * z                  device, n_elems values of dtype z_dt (only WS_F32)
 * v                  device, n_elems values of dtype v_dt (WS_BF16 or WS_F32)
 * z_bf16_out_or_null device bf16 [n_elems], receives the updated z rounded to
 *                    bf16 (the next network input), or NULL
 * One fused multiply-add per element in fp32.  n_elems == 0 is a no-op.
 */
WS_API ws_status ws_fm_euler_step(void* z, ws_dtype z_dt, const void* v, ws_dtype v_dt,
                           void* z_bf16_out_or_null, int64_t n_elems, float dtau,
                           ws_stream_t stream);

/*
 * ws_block_causal_attn_noalloc -- ws_block_causal_attn for callers that
 * cannot allocate device memory.  The paper has no counterpart: this is a
 * deployment convenience of this library.
 *
 * Who needs it: code that may not call cudaMalloc or any allocating library
 * routine -- a plug-in inside a host process whose memory pool it does not
 * own, or a real-time loop where an allocator call (which can block and
 * synchronise the device) is not allowed.  Such a caller cannot provide the
 * split-KV workspace that ws_block_causal_attn takes.
 *
 * What it does: exactly what ws_block_causal_attn does (same arguments
 * without workspace/workspace_bytes, same kernels, same results), with the
 * workspace taken from one static device array of WS_NOALLOC_SCRATCH_BYTES
 * (40 MiB) built into the library.  The driver reserves that array on every
 * GPU that loads the library, and keeps it until the process exits.  The call
 * itself allocates nothing.
 *
 * Limits and rules:
 *  - Sizes whose workspace (ws_block_causal_attn_workspace_size) exceeds
 *    WS_NOALLOC_SCRATCH_BYTES are rejected with WS_ERR_CAPACITY and a message
 *    saying so; nothing is launched.  40 MiB covers every unit call on a GPU
 *    of up to 158 SMs (a B300 has 148).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it together
 *    with the id of the current context; make that first call before any
 *    stream capture on the device.  If the context is replaced (for example
 *    after cudaDeviceReset), the next call looks the address up again in the
 *    new context, so that call too belongs before any stream capture.
 *  - All calls on a device share the one array.  Its contents on entry do not
 *    matter (every value read is written earlier in the same call), but two
 *    calls that may overlap on the GPU -- on different streams, or from
 *    different threads -- race on it and corrupt each other's results.
 *    Serialise them (one stream, or events between them).
 * Errors: as ws_block_causal_attn, plus WS_ERR_CAPACITY for the limit above
 * and WS_ERR_CUDA if the array's address cannot be looked up.
 */
#define WS_NOALLOC_SCRATCH_BYTES ((size_t)40 * 1024 * 1024)
WS_API ws_status ws_block_causal_attn_noalloc(const void* q, const void* k_cache,
                                              const void* v_cache, void* out, float* lse_or_null,
                                              const int32_t* h_offsets, const int32_t* d_offsets,
                                              int n_blocks, int64_t capacity, int num_heads,
                                              int head_dim, float softmax_scale, ws_dtype dt,
                                              ws_stream_t stream);

/*
 * ws_fm_euler_cfg_step -- one Euler step with a classifier-free-guided
 * velocity, in one pass over memory.  [close-read] 五、训练 item 3: the
 * low-latency student is distilled from a teacher that samples with CFG and
 * more solver steps; the pages give no formula, and the standard guidance
 * combination is taken:
 *   v = v_uncond + guidance * (v_cond - v_uncond),   z <- z - dtau * v
 * in fp32 as d = v_cond - v_uncond, v = fma(guidance, d, v_uncond),
 * z = fma(-dtau, v, z).  guidance 0 / 1 give the unconditional / conditional
 * step.
 *
 * z                  device, n_elems float32 (z_dt must be WS_F32), in place
 * v_uncond, v_cond   device, n_elems values of dtype v_dt (WS_BF16 or WS_F32)
 * z_bf16_out_or_null device bf16 [n_elems] receiving the new z rounded to
 *                    bf16, or NULL
 * Errors as ws_fm_euler_step; guidance must be finite.
 */
WS_API ws_status ws_fm_euler_cfg_step(void* z, ws_dtype z_dt, const void* v_uncond,
                                      const void* v_cond, ws_dtype v_dt, void* z_bf16_out_or_null,
                                      int64_t n_elems, float guidance, float dtau,
                                      ws_stream_t stream);

/*
 * Device-resident unit sizes, for a unit step captured once in a CUDA graph
 * and replayed unit after unit.  [youleyou] 3.3 (the performer's path runs
 * under CUDA Graph capture), [explainer] "点开看部署细节" and [close-read]
 * 四、推理, closing paragraph (CUDA graph capture keeps the per-unit path
 * within its 160 ms budget).  A graph replays fixed launches with fixed
 * arguments, so the sizes that change from unit to unit (the cache length,
 * the ragged unit size) live in device memory, where the kernels read them
 * at run time and a small kernel advances them.
 *
 * ws_unit_state lives in device memory (24 bytes, 8-byte aligned), owned by
 * the caller:
 *   cache_len  cache rows (per head) holding the earlier units
 *   n_new      tokens of the current unit (its slice, queries and cache rows
 *              [cache_len, cache_len + n_new))
 *   unit       index of the current unit in the caller's list of unit sizes
 */
typedef struct ws_unit_state {
  int64_t cache_len;
  int64_t n_new;
  int64_t unit;
} ws_unit_state;

/*
 * ws_kv_append_dev -- ws_kv_append with cache_len and n_new read from the
 * device-resident state when the kernel runs.  The launch covers n_max
 * tokens (the largest unit); tokens past n_new do nothing.
 * k_new, v_new  device [n_max][num_heads][head_dim] (rows past n_new unread)
 * d_state       device ws_unit_state
 * A state with n_new outside [0, n_max] or cache_len + n_new outside
 * [0, capacity] writes nothing and sets the device error word, which
 * ws_get_device_error() reports as WS_ERR_CAPACITY.  Other errors as
 * ws_kv_append, checked on the host.
 */
WS_API ws_status ws_kv_append_dev(const void* k_new, const void* v_new, void* k_cache,
                                  void* v_cache, const ws_unit_state* d_state, int64_t n_max,
                                  int64_t capacity, int num_heads, int head_dim, ws_dtype dt,
                                  ws_stream_t stream);

/*
 * ws_block_causal_attn_dev -- ws_block_causal_attn of the current unit, its
 * sizes read from the device-resident state when the kernels run: the query
 * block is the unit's n_new tokens and every query row sees the keys
 * j < kv_len = cache_len + n_new (the unit itself included: append first).
 * The launch is sized for q_max query rows and the whole cache.
 *
 * q             device [q_max][num_heads][head_dim]; rows past n_new are read
 *               and their results dropped, but they must hold finite values
 *               (zero the buffer once; rows left from earlier units are fine):
 *               a row of infinities or NaNs sends its warp to the slow exact
 *               path of the softmax on every key tile
 * out           device [q_max][num_heads][head_dim]; rows < n_new are written
 * lse_or_null   device float32 [num_heads][q_max] (row stride q_max), or NULL
 * d_state       device ws_unit_state
 * k_cache,
 * v_cache       device [num_heads][capacity][head_dim].  Cache rows from
 *               cache_len + n_new up to the next multiple of 128 are read and
 *               masked: V rows there must hold finite values (zero the caches
 *               once when allocating them).
 * workspace     device scratch of at least
 *               ws_block_causal_attn_dev_workspace_size(q_max, capacity,
 *               num_heads, head_dim) bytes (always needed: any unit's key range
 *               may be split); contents on entry do not matter.
 * Implemented for WS_BF16 with head_dim 128 (else WS_ERR_UNSUPPORTED).  A
 * state out of range (n_new outside [0, q_max], cache_len + n_new outside
 * [0, capacity]) writes nothing and sets the device error word
 * (WS_ERR_CAPACITY from ws_get_device_error); n_new == 0 does nothing.
 */
WS_API ws_status ws_block_causal_attn_dev(const void* q, const void* k_cache, const void* v_cache,
                                          void* out, float* lse_or_null,
                                          const ws_unit_state* d_state, int64_t q_max,
                                          int64_t capacity, int num_heads, int head_dim,
                                          float softmax_scale, ws_dtype dt, void* workspace,
                                          size_t workspace_bytes, ws_stream_t stream);

/* Workspace bytes for ws_block_causal_attn_dev on the current device
 * (SIZE_MAX for invalid sizes). */
WS_API size_t ws_block_causal_attn_dev_workspace_size(int64_t q_max, int64_t capacity,
                                                      int num_heads, int head_dim);

/*
 * ws_unit_state_advance -- moves the device-resident state to the next unit
 * (one thread, on the stream): cache_len += n_new; unit += 1; n_new =
 * d_sizes[unit] if unit < n_sizes, else 0.
 * d_sizes  device int32 [n_sizes], the sizes of the caller's units in order
 * (may be NULL when n_sizes is 0).
 */
WS_API ws_status ws_unit_state_advance(ws_unit_state* d_state, const int32_t* d_sizes,
                                       int64_t n_sizes, ws_stream_t stream);

/*
 * Bytes of workspace ws_block_causal_attn (and ws_block_causal_attn_side)
 * needs for these sizes on the current device (0 when no key range is
 * split).  Returns SIZE_MAX when the
 * sizes are invalid or the device cannot be queried.
 */
WS_API size_t ws_block_causal_attn_workspace_size(int64_t q_len, int64_t kv_len, int num_heads,
                                           int head_dim);

/* Static description of a status code. */
WS_API const char* ws_status_string(ws_status s);

/* Message of the last failed call on the calling thread ("" if none). */
WS_API const char* ws_last_error(void);

/*
 * Device error word written by the kernels.  Synchronises the current
 * device.  *code_out = 0 when clean.  Code 2: a kernel with device-resident
 * unit sizes found them out of range and wrote nothing; the call returns
 * WS_ERR_CAPACITY, *info_out = 1 (n_new outside the launch's maximum) or 2
 * (cache_len + n_new outside the capacity).  Code 1: an attention kernel's
 * bounded wait gave up (it then stopped, released its tensor memory and
 * returned); the call returns WS_ERR_TIMEOUT and *info_out says where: (wait site << 16) |
 * (block index & 0xFFFF), the first wait to give up.  Wait sites: 1 producer
 * waiting for the Q slot, 2 producer waiting for a K/V slot, 3 MMA issuer
 * waiting for Q, 4 MMA issuer waiting for a K/V tile, 5 MMA issuer waiting
 * for P, 6 for the O accumulator to be free, 7 softmax waiting for S, 8 for
 * the final O, 9 teardown waiting for MMAs, 10 for copies, 11 the test
 * hook's stalled wait, 12 the MMA issue lock, 13 (no longer used), 14 a
 * solo CTA's softmax merging its two halves (an odd number of query tiles),
 * 15 the KV append waiting for its copy of a token's slice.  The
 * outputs of a launch that gave up are undefined; the context
 * stays usable.  The word stays set until ws_clear_device_error().
 */
WS_API ws_status ws_get_device_error(int* code_out, int* info_out);
WS_API ws_status ws_clear_device_error(void);

/*
 * Limit, in nanoseconds, of every in-kernel wait launched after this call
 * (default 2e9).  Host-side setting, process wide: it applies to calls from
 * every thread.  Setting it is thread-safe, but a call running concurrently
 * on another thread may use either the old or the new value, so change it
 * while no attention call is being made.
 */
WS_API ws_status ws_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * Test hook for failure detection, off by default, process wide.  While on,
 * every tensor-core attention launch makes one of its MMA issuers wait on a
 * barrier that nothing completes.  The wait limit (ws_set_wait_timeout_ns)
 * runs out, the kernel records the wait site in the device error word, every
 * role stops, drains its own copies and MMAs, frees its tensor memory and
 * returns; ws_get_device_error() then reports WS_ERR_TIMEOUT.  Outputs of
 * such a launch are undefined.  Nothing faults, traps or hangs.  Like the
 * wait limit it is process wide (it affects calls from every thread); switch
 * it only while no attention call is being made.
 */
WS_API ws_status ws_debug_force_wait_timeout(int on);

/* ABI version of this header (major * 100 + minor). */
WS_API int ws_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* WS_H_ */
