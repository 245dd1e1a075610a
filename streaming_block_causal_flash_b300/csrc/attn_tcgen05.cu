// attn_tcgen05.cu -- block-causal flash attention, bf16 in / fp32 accumulate,
// head_dim 128, on sm_103a tensor cores (tcgen05 + TMEM + TMA + mbarrier).
//
// What it computes (Wan Streamer real-time AV explainer (xiaohu-jiedu.pages.dev),
// "怎么做到边听边说、随时能打断"; "阿里通义万相发布亚秒级同步AI视频通话基础模型"
// (youleyou.com), 3.1): query row i sees keys j < e(i), where e(i) is the end
// offset of the block (streaming unit) holding token i -- its own block in both
// directions, every earlier block, no later block.
//   O_i = sum_{j<e(i)} softmax_j(s q_i.k_j) v_j,   LSE_i = ln sum_j exp(s q_i.k_j)
//
// CTA layout (one CTA per SM, 384 threads):
//   warps 0-3  softmax for query tile 0 (thread = one query row)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q tiles once per work item, then K_j, V_j into a
//              5-slot ring of 32 KB slots (128 rows x 128 cols, two 128-byte
//              swizzled column halves); 6 slots in solo CTAs (below), which
//              need one Q slot only
//   warp  9    TMEM owner; its lane 0 issues every MMA of query tile 0
//   warp  10   lane 0 issues every MMA of query tile 1 (two issuers keep the
//              tensor pipe fed while the other one waits on barriers)
//   warp  11   idle (it completes the third warpgroup, which gives up
//              registers to the softmax warpgroups)
// TMEM (512 columns): tile t uses S_t = cols [256t, 256t+128) (fp32 logits,
// overwritten in place by bf16 P in its first 64 columns) and
// O_t = cols [256t+128, 256t+256) (fp32 output accumulator).
//
// Per key tile j, the issuer of query tile t waits for K_j, then for P_t(j-1),
// and issues PV_t(j-1) then QK_t(j) as one group under a shared-memory issue
// lock, so the two tiles' groups reach the tensor pipe whole; while one
// softmax group works on S_t(j) the pipe executes the other tile's group.
// tcgen05.mma instructions from one thread execute in issue order, which
// orders QK_t(j) (writes S_t) after PV_t(j-1) (reads P_t from the same
// columns).  One thread issuing both tiles' MMAs left the pipe idle during
// its barrier waits and fences (about 115 cycles per 64-cycle MMA); two
// issuers hide that bookkeeping behind each other's MMAs.
//
// Softmax keeps a per-row running max m (log2 units of the scaled logits) and
// sum l.  O is rescaled only when a row's max grows by more than 2^8 (lazy
// rescale; exact after the final division by l).  After a row's first tile
// the exponentials are computed against the current m with no tile max at
// all; only a tile whose row sum exceeds 2^64 is redone exactly (tile max,
// rescale) from S, which stays in TMEM until P is stored.  P is rounded to
// bf16 before PV.
//
// Work decomposition:
//  * unit mode (the query block is the newest unit; every row sees all keys
//    < kv_len): CTAs form `groups` of `pairs` CTAs; group g walks a contiguous
//    range of the flattened (head, key tile) space and CTA p of the group
//    holds query-tile pair p, so the CTAs of a group read the same K/V tiles at
//    nearly the same time (one HBM read, L2 reuse).  A range that covers only
//    part of a head writes a partial (O/l, log2-sum-exp) into the workspace;
//    attn_combine_kernel merges the partials.
//    With an odd number of query tiles (host-sized launches), the last tile
//    gets solo CTAs of its own: both TMEM halves work on that one tile, on
//    alternate key tiles of the range, and the epilogue merges the two
//    halves' (m, l, O).  A solo CTA runs a range at about twice a paired
//    CTA's rate, so it gets twice the range (half as many groups).
//    Side mode (unit mode only): keys [0, cache_len) come from the cache and
//    the newest unit's keys from token-major side buffers through 2-D TMA
//    maps; the two parts are tiled separately, each with its own ragged tail.
//    With commit, the side tiles are also written to the cache by TMA
//    stores from their ring slots (one CTA per group stores), before each
//    slot is released.
//  * prefill mode: one work item per (head, query-tile pair); key tiles no
//    row of a query tile can see are skipped.  CTAs take, round-robin, a
//    head and a mirrored couple of pairs (z, pairs - 1 - z), which together
//    cost the same for every couple, so the CTAs move through the heads'
//    keys together and L2 serves most K/V tiles.
//
// Every wait is bounded (wall-clock limit): on time-out the kernel records an
// error word, stops all roles, waits (bounded) for its own copies and MMAs in
// flight, frees its tensor memory and returns.
#include <cuda_bf16.h>

#include <mutex>

#include "ws_debug.cuh"
#include "ws_internal.h"
#include "ws_ptx.cuh"

namespace ws {

// Device error word: [0] code (0 = clean, 1 = wait time-out, 2 = device-
// resident sizes out of range, 3 = a debug-build bounds check failed), [1] info.
__device__ unsigned int g_attn_error[2];

namespace {

constexpr int BM = 128;                       // query rows per tile
constexpr int BN = 128;                       // keys per tile
constexpr int HD = 128;                       // head dim
constexpr int NSTAGE = 5;                     // K/V ring slots (paired CTAs)
// Solo CTAs hold one query tile; the second Q slot, which follows the ring in
// shared memory, becomes a sixth ring slot for them.
constexpr int NSTAGE_SOLO = NSTAGE + 1;
constexpr int TILE_BYTES = BM * HD * 2;       // 32 KB
constexpr int HALF_BYTES = TILE_BYTES / 2;    // 128 rows x 64 cols (128-byte rows)
constexpr int NUM_THREADS = 384;
// Register split: the two softmax warpgroups grow to REGS_SOFTMAX per thread,
// the producer/MMA warpgroup shrinks to REGS_OTHER.  The sum must fit in what
// the block is launched with (NUM_THREADS x the kernel's register count); the
// host checks that before every launch.
constexpr int REGS_SOFTMAX = 208;
constexpr int REGS_OTHER = 88;
constexpr int REGS_NEEDED = 256 * REGS_SOFTMAX + 128 * REGS_OTHER;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;
// A tile computed against a row max it has outgrown is accepted while the
// row's sum of p stays within this bound (so every p does).
constexpr float SPEC_SUM_LIMIT = 18446744073709551616.0f;   // 2^64
constexpr float LN2 = 0.69314718055994531f;
// Teardown waits (copies / MMAs still in flight) never use a shorter limit.
constexpr unsigned long long DRAIN_TIMEOUT_NS = 2000000000ull;

// barrier indices
constexpr int BAR_KV_FULL = 0;
constexpr int BAR_KV_EMPTY = NSTAGE_SOLO;
constexpr int BAR_Q_FULL = 2 * NSTAGE_SOLO;
constexpr int BAR_Q_EMPTY = BAR_Q_FULL + 1;
constexpr int BAR_S_FULL = BAR_Q_EMPTY + 1;   // [2]
constexpr int BAR_P_FULL = BAR_S_FULL + 2;    // [2]
constexpr int BAR_O_FULL = BAR_P_FULL + 2;    // [2]
constexpr int BAR_O_FREE = BAR_O_FULL + 2;    // [2]
constexpr int BAR_DRAIN = BAR_O_FREE + 2;    // [2], one per MMA issuer
constexpr int BAR_STALL = BAR_DRAIN + 2;      // never completed (test hook)
constexpr int BAR_MERGE = BAR_STALL + 1;      // solo items: half 1's (m, l) are in shared memory
constexpr int BAR_MERGE_FREE = BAR_MERGE + 1; // solo items: half 0 has read them
constexpr int NUM_BARS = BAR_MERGE_FREE + 1;

// Q slot 0, the K/V ring, Q slot 1 (ring slot NSTAGE of solo CTAs)
constexpr int SMEM_Q = 0;
constexpr int SMEM_KV = TILE_BYTES;
constexpr int SMEM_Q1 = SMEM_KV + NSTAGE * TILE_BYTES;
constexpr int SMEM_BARS = SMEM_Q1 + TILE_BYTES;
constexpr int SMEM_MISC = SMEM_BARS + NUM_BARS * 8;
// tmem slot, abort flag, issue lock, (unused); then the launch's sizes;
// then a solo item's per-row (m, l) of TMEM half 1
constexpr int SMEM_MERGE = SMEM_MISC + 16 + 32;
// side mode with commit: per ring slot, the cache row and (head, K or V) of a
// side tile the producer still has to store from it
constexpr int SMEM_STORE = SMEM_MERGE + 2 * BM * 4;
constexpr int SMEM_USED = SMEM_STORE + NSTAGE_SOLO * 8;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024 B

// wait sites (error info)
enum : int { W_PROD_QE = 1, W_PROD_KVE, W_MMA_Q, W_MMA_KV, W_MMA_P, W_MMA_OF, W_SM_S, W_SM_O,
             W_DRAIN_MMA, W_DRAIN_TMA, W_FORCED, W_LOCK, W_UNUSED_13, W_SM_MERGE };

struct Params {
  int prefill;
  int heads, q_len, q_row0, kv_len, n_blocks;
  int pairs, kv_tiles, groups;
  // Side mode (unit mode only): keys [0, cache_len) come from the cache, in
  // kv_tiles_c tiles; the newest block's n_side keys come from the
  // token-major side buffers, in the remaining kv_tiles - kv_tiles_c tiles.
  int side, kv_tiles_c, cache_len, n_side;
  // Side mode with commit: the side tiles, once in the ring, are also
  // written to cache rows cache_len + (row in the side buffer) by TMA stores
  // (maps tm_kc / tm_vc, whose rows end at cache_len + n_side).
  int commit;
  long long capacity;
  long long work;
  int n_items;
  float scale_log2;
  const int32_t* offs;
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;     // [grid*2][256][HD]
  float* ws_lse;   // [grid*2][256]
  unsigned long long timeout_ns;
  int force_stall;   // test hook: one MMA issuer waits on a barrier nothing completes
  // Device-resident unit sizes (unit mode only): when set, the unit's sizes
  // are read at run time from dev_state = {cache_len, n_new} (the cache holds
  // cache_len rows of earlier units and the n_new rows of the current one),
  // and the launch was sized for at most q_max query rows and capacity keys.
  const long long* dev_state;
  int q_max;
  // Split-stream ("solo") CTAs, unit mode with host sizes: when the query
  // block has an odd number of 128-row tiles, its last tile is not paired.
  // It gets CTAs of its own: the first groups * pairs CTAs hold the full
  // pairs as usual; the solo_groups CTAs after them each hold the last tile
  // on both TMEM halves, which take alternate key tiles of the CTA's range
  // and are merged in the epilogue.  Such a CTA runs its range at the rate of
  // a paired CTA, so solo groups get twice the key range.
  int solo, solo_groups;
};

// The sizes one launch works on: from the host plan, or from the
// device-resident unit state.
struct Dims {
  int q_len;       // query rows
  int kv_len;      // keys every row sees (unit mode)
  int kv_tiles;    // ceil(kv_len / BN)
  int groups;      // unit mode: CTA groups that have work (the others idle)
  int lse_stride;  // row stride of the [H][rows] LSE output
  long long work;  // unit mode: heads * kv_tiles
};

// Reads the sizes of this launch.  Returns false (every thread of every CTA
// alike) when the launch has nothing to do; a device-resident state that is
// out of range sets the device error word (code 2) and does nothing.
__device__ __forceinline__ bool load_dims(const Params& P, Dims& D) {
  if (P.dev_state == nullptr) {
    D.q_len = P.q_len;
    D.kv_len = P.kv_len;
    D.kv_tiles = P.kv_tiles;
    D.groups = P.groups;
    D.lse_stride = P.q_len;
    D.work = P.work;
    return true;
  }
  const long long cache_len = P.dev_state[0];
  const long long n_new = P.dev_state[1];
  if (cache_len < 0 || n_new < 0 || n_new > P.q_max || cache_len > P.capacity - n_new) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && atomicCAS(&g_attn_error[0], 0u, 2u) == 0u)
      g_attn_error[1] = static_cast<unsigned>(n_new > P.q_max || n_new < 0 ? 1 : 2);
    return false;
  }
  if (n_new == 0) return false;
  D.q_len = static_cast<int>(n_new);
  D.kv_len = static_cast<int>(cache_len + n_new);
  D.kv_tiles = (D.kv_len + BN - 1) / BN;
  D.work = static_cast<long long>(P.heads) * D.kv_tiles;
  D.groups = static_cast<int>(D.work < P.groups ? D.work : P.groups);
  D.lse_stride = P.q_max;
  return true;
}

struct Item {
  int h, pair, t0;
  int n[2];        // key tiles for query tile 0 / 1 (0: tile has no rows); for a solo
                   // item, the key tiles of TMEM half 0 (even) and half 1 (odd)
  int slot;        // -1 final output, else partial slot 0/1
  int solo;        // one query tile (2 * pair) on both halves
};

struct ItemIter {
  long long f, fb, fe;
  int p, i, solo;
};

// The q-th K/V load of an item: key tile j (relative to the item's first)
// and which = 0 (K) or 1 (V).  Paired items load K_j, V_j for j in order.
// Solo items (len key tiles, alternating between the two halves) load K_0,
// then K_{j+1} before V_j: K_0, K_1, V_0, K_2, V_1, ..., K_{len-1}, V_{len-2},
// V_{len-1}.  A half holds its V until its next group, so the K it needs
// next must not queue behind it in the ring.
__device__ __forceinline__ void load_order(bool solo, int len, int q, int& j, int& which) {
  if (!solo) {
    j = q >> 1;
    which = q & 1;
    return;
  }
  if (q == 0) {
    j = 0;
    which = 0;
    return;
  }
  const int r = q - 1, m = r >> 1;
  if (r & 1) {
    j = m;
    which = 1;
  } else if (m + 1 < len) {
    j = m + 1;
    which = 0;
  } else {
    j = len - 1;
    which = 1;
  }
}

__device__ __forceinline__ int row_limit_dev(const int32_t* offs, int n_blocks, int token) {
  int lo = 0, hi = n_blocks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= token) lo = mid;
    else hi = mid - 1;
  }
  return __ldg(offs + lo + 1);
}

__device__ __forceinline__ void iter_init(const Params& P, const Dims& D, ItemIter& it) {
  it.solo = 0;
  if (!P.prefill) {
    const int paired = P.solo ? D.groups * P.pairs : static_cast<int>(gridDim.x);
    if (static_cast<int>(blockIdx.x) >= paired) {
      // a solo CTA: the unpaired last query tile, over its own group ranges
      const int g = static_cast<int>(blockIdx.x) - paired;
      it.solo = 1;
      it.p = P.pairs;
      it.fb = static_cast<long long>(g) * D.work / P.solo_groups;
      it.fe = static_cast<long long>(g + 1) * D.work / P.solo_groups;
      it.f = it.fb;
      return;
    }
    const int g = blockIdx.x / P.pairs;
    it.p = blockIdx.x % P.pairs;
    if (g < D.groups && 2 * it.p * BM < D.q_len) {
      it.fb = static_cast<long long>(g) * D.work / D.groups;
      it.fe = static_cast<long long>(g + 1) * D.work / D.groups;
    } else {
      // a group beyond the work, or a query-tile pair past the unit's rows
      // (device-resident sizes, launch sized for a larger unit): idle
      it.fb = it.fe = D.work;
    }
    it.f = it.fb;
  } else {
    it.i = blockIdx.x;   // prefill: the couple (see iter_next)
    it.p = 0;            // 0: the couple's short pair next, 1: its long pair
  }
}

__device__ __forceinline__ bool iter_next(const Params& P, const Dims& D, ItemIter& it, Item& item) {
  if (!P.prefill) {
    if (it.f >= it.fe) return false;
    const int h = static_cast<int>(it.f / D.kv_tiles);
    const int t0 = static_cast<int>(it.f % D.kv_tiles);
    const long long rem = it.fe - it.f;
    const int t1 = static_cast<int>(rem < D.kv_tiles - t0 ? t0 + rem : D.kv_tiles);
    item.h = h;
    item.pair = it.p;
    item.t0 = t0;
    item.slot = (t0 == 0 && t1 == D.kv_tiles) ? -1
                                              : (h == static_cast<int>(it.fb / D.kv_tiles) ? 0 : 1);
    item.solo = it.solo;
    if (it.solo) {
      item.n[0] = (t1 - t0 + 1) / 2;
      item.n[1] = (t1 - t0) / 2;
    } else {
      for (int t = 0; t < 2; ++t)
        item.n[t] = ((2 * it.p + t) * BM < D.q_len) ? (t1 - t0) : 0;
    }
    it.f += t1 - t0;
    return true;
  }
  // Prefill: a work unit is a head and a mirrored couple of query-tile
  // pairs, z and pairs - 1 - z (z < ceil(pairs / 2)), done one after the
  // other, the short one first.  Pair p sees about 2(p + 1) key tiles, so
  // every couple costs the same: the CTAs keep step with each other, each
  // CTA's position in the head's keys stays within a few hundred tiles of
  // the others', and L2 serves those K/V tiles to all of them.  (Single
  // pairs dealt longest first let the CTAs spread over whole heads, more
  // K/V than L2 holds: each tile then left DRAM about 40 times.)
  const int couples = (P.pairs + 1) / 2;
  int z, pair;
  for (;;) {
    if (it.i >= P.n_items) return false;
    z = it.i % couples;
    pair = it.p == 0 ? z : P.pairs - 1 - z;
    if (it.p == 0 || pair != z) break;
    it.p = 0;                 // odd pair count: the middle pair has no mirror
    it.i += gridDim.x;
  }
  item.h = it.i / couples;
  item.pair = pair;
  item.t0 = 0;
  item.slot = -1;
  item.solo = 0;
  for (int t = 0; t < 2; ++t) {
    const int r0 = (2 * item.pair + t) * BM;
    if (r0 < D.q_len) {
      const int last = min(r0 + BM, D.q_len) - 1;
      const int e = row_limit_dev(P.offs, P.n_blocks, P.q_row0 + last);
      item.n[t] = (e + BN - 1) / BN;
    } else {
      item.n[t] = 0;
    }
  }
  // next: the couple's mirror, or the next couple
  if (it.p == 0) {
    it.p = 1;
  } else {
    it.p = 0;
    it.i += gridDim.x;
  }
  return true;
}

__device__ __forceinline__ void record_error(int where) {
  if (atomicCAS(&g_attn_error[0], 0u, 1u) == 0u)
    g_attn_error[1] = (static_cast<unsigned>(where) << 16) | (blockIdx.x & 0xFFFFu);
}

// Bounded wait on an mbarrier phase (slow path, inlined: a call inside a
// setmaxnreg region would pin its register budget).  Returns false on
// time-out or when another role has already aborted the CTA.
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned long long timeout_ns, int where) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        record_error(where);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long timeout_ns, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, abort_flag, timeout_ns, where);
}

// Issue lock shared by the two MMA issuers: a tile's PV and QK go to the
// tensor pipe as one uninterrupted group (interleaving the two tiles' groups
// delays both tiles' logits).  The holder only issues and commits, which
// never blocks indefinitely; waiting for the lock is bounded like every wait.
__device__ __forceinline__ bool issue_lock(int* lk, volatile int* abort_flag,
                                           unsigned long long timeout_ns) {
  if (atomicCAS(lk, 0, 1) == 0) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (atomicCAS(lk, 0, 1) == 0) return true;
    if ((it & 31u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        record_error(W_LOCK);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void issue_unlock(int* lk) { atomicExch(lk, 0); }

// Keys at or beyond the row's limit get -inf logits (ragged key tail and,
// in prefill mode, keys of later blocks).
__device__ __forceinline__ void mask_tail(uint32_t (&s)[4][32], int kv0, int e_row) {
  if (kv0 + BN > e_row) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (kv0 + 32 * c + i >= e_row) s[c][i] = __float_as_uint(-INFINITY);
  }
}

// Row max of the 128 raw logits held by this thread.
__device__ __forceinline__ float tile_max(const uint32_t (&s)[4][32]) {
  float mxc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float a = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      a = max3f(a, __uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1]));
    mxc[c] = a;
  }
  return max3f(mxc[0], mxc[1], fmaxf(mxc[2], mxc[3]));
}

// p = 2^(x*scale - mb) for the 128 logits, in packed fp32x2 arithmetic; the
// bf16 pair k of chunk c overwrites s[c][k] (both of its sources are already
// consumed).  lsum gets the row sum of p in two packed partial sums.
__device__ __forceinline__ void exp_pass(uint32_t (&s)[4][32], uint64_t sc2, float mb,
                                         uint64_t (&lsum)[2]) {
  const uint64_t nm2 = f2_pack(-mb, -mb);
  lsum[0] = 0ull;
  lsum[1] = 0ull;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[c][2 * k]),
                                         __uint_as_float(s[c][2 * k + 1])), sc2, nm2);
      float x0, x1;
      f2_unpack(x2, x0, x1);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      lsum[k & 1] = f2_add(lsum[k & 1], f2_pack(p0, p1));
      s[c][k] = pack_bf16x2(p0, p1);
    }
  }
}

// A slot index that names no ring slot.
constexpr uint32_t NO_SLOT = 0xFFu;

struct Ring {
  uint32_t stage, phase, n;   // n: slots in the ring (NSTAGE or NSTAGE_SOLO)
  __device__ __forceinline__ explicit Ring(uint32_t slots) : stage(0), phase(0), n(slots) {}
  __device__ __forceinline__ void advance() {
    if (++stage == n) { stage = 0; phase ^= 1u; }
  }
};

}  // namespace

__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_tc_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_ks,
                    const __grid_constant__ CUtensorMap tm_vs,
                    const __grid_constant__ CUtensorMap tm_kc,
                    const __grid_constant__ CUtensorMap tm_vc, const Params P) {
  // Sizes of this launch; with device-resident sizes every thread reads the
  // same state, so a launch with nothing to do returns in every thread.
  Dims dims;
  if (!load_dims(P, dims)) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + SMEM_Q;
  const uint32_t sQ1 = sbase + SMEM_Q1;
  const uint32_t sKV = sbase + SMEM_KV;
  const uint32_t sBar = sbase + SMEM_BARS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + SMEM_MISC + 4);
  int* issue_lk = reinterpret_cast<int*>(sgen + SMEM_MISC + 8);
  // the launch's sizes, kept in shared memory (read at item boundaries only,
  // so that they hold no registers through the hot loops)
  Dims* sdims = reinterpret_cast<Dims*>(sgen + SMEM_MISC + 16);
  auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE_SOLO; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), 1);
      // released by both MMA issuers
      mbar_init(bar(BAR_KV_EMPTY + s), 2);
    }
    mbar_init(bar(BAR_Q_FULL), 1);
    mbar_init(bar(BAR_Q_EMPTY), 2);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(BAR_S_FULL + t), 1);
      mbar_init(bar(BAR_P_FULL + t), 128);
      mbar_init(bar(BAR_O_FULL + t), 1);
      mbar_init(bar(BAR_O_FREE + t), 128);
    }
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_DRAIN + 1), 1);
    mbar_init(bar(BAR_STALL), 1);
    mbar_init(bar(BAR_MERGE), 128);
    mbar_init(bar(BAR_MERGE_FREE), 128);
    *abort_flag = 0;
    *issue_lk = 0;
    *sdims = dims;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Dims& D = *sdims;
  // Each role's code sits inside the branch that sets its register budget,
  // so the compiler allocates every region against the right limit.
  if (warp >= 8) {
  setmaxnreg_dec<REGS_OTHER>();
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      if (P.side) {
        tma_prefetch_map(&tm_ks);
        tma_prefetch_map(&tm_vs);
      }
      ItemIter it;
      iter_init(P, D, it);
      Item item;
      Ring ring(it.solo ? NSTAGE_SOLO : NSTAGE);
      uint32_t q_phase = 0;
      int issued = 0, q_issued = 0;
      bool ok = true;
      // Side mode with commit: each side tile is also written to its cache
      // rows, by two TMA stores (one per 64-column half) from the ring slot
      // that holds it for the attention.  The producer issues them just
      // before it refills the slot (the issuers have released it by then,
      // and it still holds the tile), or at teardown for the last slots, so
      // no MMA ever waits for a store.  A group's side tiles are spread over
      // its pair CTAs (tile k's K and V go to pairs (2k) mod P and
      // (2k + 1) mod P); in a launch of solo CTAs only, each stores its own.
      uint32_t store_mask = 0;   // ring slots holding a side tile still to store
      int2* store_info = reinterpret_cast<int2*>(sgen + SMEM_STORE);
      auto flush_store = [&](uint32_t slot) {
        const int2 si = store_info[slot];
        fence_proxy_async_smem();
        const CUtensorMap* map = (si.y >> 16) ? &tm_vc : &tm_kc;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_store_3d(map, sKV + slot * TILE_BYTES + hf * HALF_BYTES, hf * 64, si.x,
                       si.y & 0xFFFF);
        bulk_commit_group();
      };
      while (ok && iter_next(P, D, it, item)) {
        if (!wait_bar(bar(BAR_Q_EMPTY), q_phase ^ 1u, abort_flag, P.timeout_ns, W_PROD_QE)) break;
        q_phase ^= 1u;
        ++q_issued;
        // a solo item has one query tile, whose key tiles alternate between
        // the two halves: the ring carries all of them once, in order
        const int ntiles = (!item.solo && item.n[1] > 0) ? 2 : 1;
        mbar_arrive_expect_tx(bar(BAR_Q_FULL), ntiles * TILE_BYTES);
        for (int t = 0; t < ntiles; ++t) {
          const int row0 = (2 * item.pair + t) * BM;
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d((t ? sQ1 : sQ) + hf * HALF_BYTES, &tm_q, bar(BAR_Q_FULL),
                        item.h * HD + hf * 64, row0);
        }
        const int n_loads = 2 * (item.solo ? item.n[0] + item.n[1] : max(item.n[0], item.n[1]));
        for (int q = 0; q < n_loads && ok; ++q) {
          int j, which;
          load_order(item.solo, item.n[0] + item.n[1], q, j, which);
          const int tile = item.t0 + j;
          const bool from_side = P.side && tile >= P.kv_tiles_c;
          const int kv0 = (from_side ? tile - P.kv_tiles_c : tile) * BN;
          {
            if (!wait_bar(bar(BAR_KV_EMPTY + ring.stage), ring.phase ^ 1u, abort_flag,
                          P.timeout_ns, W_PROD_KVE)) {
              ok = false;
              break;
            }
            if ((store_mask >> ring.stage) & 1u) {
              flush_store(ring.stage);
              bulk_wait_group_read0();   // the stores have read the slot
              store_mask &= ~(1u << ring.stage);
            }
            const uint32_t full = bar(BAR_KV_FULL + ring.stage);
            mbar_arrive_expect_tx(full, TILE_BYTES);
            if (from_side) {
              // side buffer [n_side][H*D]: 128 keys x 64 columns of head h
              const CUtensorMap* map = which == 0 ? &tm_ks : &tm_vs;
              for (int hf = 0; hf < 2; ++hf)
                tma_load_2d(sKV + ring.stage * TILE_BYTES + hf * HALF_BYTES, map, full,
                            item.h * HD + hf * 64, kv0);
              if (P.commit &&
                  (it.solo ? P.pairs == 0 : (2 * (kv0 / BN) + which) % P.pairs == it.p)) {
                store_info[ring.stage] = make_int2(P.cache_len + kv0, item.h | (which << 16));
                store_mask |= 1u << ring.stage;
              }
            } else {
              const CUtensorMap* map = which == 0 ? &tm_k : &tm_v;
              for (int hf = 0; hf < 2; ++hf)
                tma_load_3d(sKV + ring.stage * TILE_BYTES + hf * HALF_BYTES, map, full, hf * 64,
                            kv0, item.h);
            }
            ++issued;
            ring.advance();
          }
        }
      }
      // Teardown: every copy this warp started must have landed before the
      // CTA may exit.  The ring slots filled last (up to a ring's worth) and
      // the last Q load are waited for with bounded waits; loads already
      // consumed return at once.
      volatile int no_abort = 0;
      const int pend = issued < static_cast<int>(ring.n) ? issued : static_cast<int>(ring.n);
      Ring back = ring;
      for (int k = 0; k < pend; ++k) {
        if (back.stage == 0) { back.stage = back.n - 1; back.phase ^= 1u; }
        else --back.stage;
        wait_bar(bar(BAR_KV_FULL + back.stage), back.phase, &no_abort, DRAIN_TIMEOUT_NS, W_DRAIN_TMA);
      }
      if (q_issued > 0)
        wait_bar(bar(BAR_Q_FULL), static_cast<uint32_t>(q_issued - 1) & 1u, &no_abort,
                 DRAIN_TIMEOUT_NS, W_DRAIN_TMA);
      // the side tiles still held in the ring (now all landed), and every
      // cache store to completion
      for (uint32_t slot = 0; slot < ring.n; ++slot)
        if ((store_mask >> slot) & 1u) flush_store(slot);
      if (P.commit) bulk_wait_group0();
    }
    __syncwarp();
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------- MMA issuers, one per query tile
    // Two issuing threads keep the tensor pipe fed: while one waits on its
    // barriers and fences, the other's MMAs execute.  Each issuer walks the
    // same K/V ring and, for every slot use, waits for the slot to be full
    // before it commits its release, so a slot's two releases (count-2
    // barrier) always belong to the same fill.
    if (lane == 0) {
      const int t = warp - 9;
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, HD, 0, 1);
      const uint32_t aQ = t ? sQ1 : sQ;
      const uint32_t tS = tmem + 256u * t;
      const uint32_t tO = tS + 128u;
      ItemIter it;
      iter_init(P, D, it);
      Item item;
      Ring ring(it.solo ? NSTAGE_SOLO : NSTAGE);
      uint32_t q_phase = 0, p_phase = 0, of_phase = 0;
      bool ok = true;

      auto issue_qk_from = [&](uint32_t qaddr, uint32_t kslot) {
        const uint32_t b0 = sKV + kslot * TILE_BYTES;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * HALF_BYTES + (k & 3) * 32;
          mma_ss(tS, smem_desc_sw128(qaddr + off, 16, 1024), smem_desc_sw128(b0 + off, 16, 1024),
                 IDESC_QK, k > 0 ? 1u : 0u);
        }
      };
      auto issue_qk = [&](uint32_t kslot) { issue_qk_from(aQ, kslot); };
      auto issue_pv = [&](uint32_t vslot, bool acc) {
        const uint32_t b0 = sKV + vslot * TILE_BYTES;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          mma_ts(tO, tS + 8u * k, smem_desc_sw128(b0 + k * 16 * 128, HALF_BYTES, 1024), IDESC_PV,
                 (acc || k > 0) ? 1u : 0u);
        }
      };

      if (P.force_stall && t == 0) {
        // Test hook: wait on a barrier that nothing completes, so the wait
        // limit runs out and every role takes the give-up path.
        wait_bar(bar(BAR_STALL), 0u, abort_flag, P.timeout_ns, W_FORCED);
        ok = false;
      }
      while (ok && iter_next(P, D, it, item)) {
        if (item.solo) {
          // One query tile (in Q slot 0) on both halves; this issuer owns the
          // key tiles j = t, t + 2, ...  It walks the whole ring in the
          // producer's order (load_order), waiting for each slot to fill
          // before releasing it: the other half's slots at once, its own K
          // after its QK, its own V after its PV.  At each own K: PV of the
          // previous own tile (once its P is in) and QK of this one, as one
          // group under the issue lock; the last PV follows the walk.
          const int len = item.n[0] + item.n[1];
          if (!wait_bar(bar(BAR_Q_FULL), q_phase, abort_flag, P.timeout_ns, W_MMA_Q)) break;
          q_phase ^= 1u;
          uint32_t pend_v = NO_SLOT;  // V slot of the last own tile (its PV pending); none yet
          int pvs = 0;                // PVs issued in this item
          bool bad = false;
#pragma unroll 1
          for (int q = 0; q <= 2 * len; ++q) {
            // q == 2 * len: past the walk, the last own tile's PV alone
            const bool last = q == 2 * len;
            int j = 0, which = 0;
            uint32_t slot = 0;
            if (!last) {
              load_order(true, len, q, j, which);
              slot = ring.stage;
              if (!wait_bar(bar(BAR_KV_FULL + slot), ring.phase, abort_flag, P.timeout_ns, W_MMA_KV)) {
                bad = true;
                break;
              }
              ring.advance();
              if ((j & 1) != t) {               // the other half's tile
                mbar_arrive(bar(BAR_KV_EMPTY + slot));
                continue;
              }
              if (which == 1) {                 // own V: held until its PV
                pend_v = slot;
                continue;
              }
            } else if (pend_v == NO_SLOT) {
              break;                            // no own tile at all
            }
            if (pend_v != NO_SLOT) {
              if (!wait_bar(bar(BAR_P_FULL + t), p_phase, abort_flag, P.timeout_ns, W_MMA_P)) {
                bad = true;
                break;
              }
              p_phase ^= 1u;
              if (pvs == 0) {   // the item's first PV: the last epilogue must have read O
                if (!wait_bar(bar(BAR_O_FREE + t), of_phase ^ 1u, abort_flag, P.timeout_ns, W_MMA_OF)) {
                  bad = true;
                  break;
                }
                of_phase ^= 1u;
              }
            }
            tc_fence_after();
            if (!issue_lock(issue_lk, abort_flag, P.timeout_ns)) { bad = true; break; }
            if (pend_v != NO_SLOT) issue_pv(pend_v, pvs > 0);
            if (!last) issue_qk_from(sQ, slot);
            mma_commit(bar(last ? BAR_O_FULL + t : BAR_S_FULL + t));
            issue_unlock(issue_lk);
            if (pend_v != NO_SLOT) {
              mma_commit(bar(BAR_KV_EMPTY + pend_v));
              pend_v = NO_SLOT;
              ++pvs;
            }
            if (!last) {
              mma_commit(bar(BAR_KV_EMPTY + slot));
              if (j + 2 >= len) mma_commit(bar(BAR_Q_EMPTY));   // this issuer's last QK
            }
          }
          if (bad) { ok = false; break; }
          if ((t ? item.n[1] : item.n[0]) == 0) mbar_arrive(bar(BAR_Q_EMPTY));   // no QK of ours on this Q
          continue;
        }
        const int n_iter = max(item.n[0], item.n[1]);
        const int n = t ? item.n[1] : item.n[0];
        if (!wait_bar(bar(BAR_Q_FULL), q_phase, abort_flag, P.timeout_ns, W_MMA_Q)) break;
        q_phase ^= 1u;
        // prologue: QK_t(0)
        const uint32_t k0 = ring.stage;
        if (!wait_bar(bar(BAR_KV_FULL + ring.stage), ring.phase, abort_flag, P.timeout_ns,
                      W_MMA_KV)) break;
        ring.advance();
        tc_fence_after();
        if (n > 0) {
          if (!issue_lock(issue_lk, abort_flag, P.timeout_ns)) break;
          issue_qk(k0);
          mma_commit(bar(BAR_S_FULL + t));
          issue_unlock(issue_lk);
        }
        mma_commit(bar(BAR_KV_EMPTY + k0));
        if (n <= 1) mma_commit(bar(BAR_Q_EMPTY));

        for (int jj = 0; jj < n_iter; ++jj) {
          const uint32_t vslot = ring.stage;
          if (!wait_bar(bar(BAR_KV_FULL + ring.stage), ring.phase, abort_flag, P.timeout_ns,
                        W_MMA_KV)) { ok = false; break; }
          ring.advance();
          const bool more = jj + 1 < n_iter;
          uint32_t kslot = 0, kphase = 0;
          if (more) { kslot = ring.stage; kphase = ring.phase; ring.advance(); }
          // every wait and fence of this step before taking the issue lock;
          // K_{j+1} (normally loaded long before) first, so that only the
          // wait for this tile's P sits between its softmax and its MMAs
          if (more && !wait_bar(bar(BAR_KV_FULL + kslot), kphase, abort_flag, P.timeout_ns,
                                W_MMA_KV)) { ok = false; break; }
          if (jj < n) {
            if (!wait_bar(bar(BAR_P_FULL + t), p_phase, abort_flag, P.timeout_ns, W_MMA_P)) {
              ok = false; break;
            }
            p_phase ^= 1u;
            if (jj == 0) {
              if (!wait_bar(bar(BAR_O_FREE + t), of_phase ^ 1u, abort_flag, P.timeout_ns,
                            W_MMA_OF)) { ok = false; break; }
              of_phase ^= 1u;
            }
          }
          if (jj < n) {
            tc_fence_after();
            if (!issue_lock(issue_lk, abort_flag, P.timeout_ns)) { ok = false; break; }
            issue_pv(vslot, jj > 0);
            if (jj + 1 < n) {
              issue_qk(kslot);
              mma_commit(bar(BAR_S_FULL + t));
            } else {
              mma_commit(bar(BAR_O_FULL + t));
            }
            issue_unlock(issue_lk);
          }
          mma_commit(bar(BAR_KV_EMPTY + vslot));
          if (more) mma_commit(bar(BAR_KV_EMPTY + kslot));
          if (jj + 2 == n) mma_commit(bar(BAR_Q_EMPTY));
        }
      }
      // Teardown: all MMAs this thread issued must be complete before the
      // tensor memory is released.
      mma_commit(bar(BAR_DRAIN + t));
      volatile int no_abort = 0;
      wait_bar(bar(BAR_DRAIN + t), 0u, &no_abort, DRAIN_TIMEOUT_NS, W_DRAIN_MMA);
    }
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<REGS_SOFTMAX>();
    // -------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r_in_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + 256u * t;
    const uint32_t tO = tS + 128u;
    uint32_t s_phase = 0, o_phase = 0, merge_phase = 0;
    ItemIter it;
    iter_init(P, D, it);
    Item item;
    bool ok = true;
    while (ok && iter_next(P, D, it, item)) {
      const int n = t ? item.n[1] : item.n[0];
      if (n == 0 && !item.solo) continue;
      // local query row (a solo item's two halves share the one tile's rows)
      const int row = (2 * item.pair + (item.solo ? 0 : t)) * BM + r_in_tile;
      const bool valid = row < D.q_len;
      const int e_row = (P.prefill && valid) ? row_limit_dev(P.offs, P.n_blocks, P.q_row0 + row)
                                             : D.kv_len;
      float m = -INFINITY, l = 0.f;
      for (int jj = 0; jj < n; ++jj) {
        const bool got = wait_bar(bar(BAR_S_FULL + t), s_phase, abort_flag, P.timeout_ns, W_SM_S);
        if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
        s_phase ^= 1u;
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32u * c, s[c]);
        tmem_ld_wait_only();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_reg_fence(s[c]);

        // key range of this tile and the limit its columns are masked at
        // (a solo item's half t takes every other key tile, from t on)
        const int tile = item.t0 + (item.solo ? 2 * jj + t : jj);
        int kv0 = tile * BN, e_lim = e_row;
        if (P.side) {
          if (tile < P.kv_tiles_c) {
            e_lim = P.cache_len;
          } else {
            kv0 = (tile - P.kv_tiles_c) * BN;
            e_lim = P.n_side;
          }
        }
        mask_tail(s, kv0, e_lim);
        // Once a row has a max m, the tile's exponentials are taken against
        // it without looking for the tile max: m only has to keep p finite,
        // and every p <= the row sum, so a row sum <= 2^64 proves the pass
        // good (bf16 P has the same relative precision at any magnitude, and
        // fp32 O and l have range to spare).  A warp whose rows have no max
        // yet, or whose pass overflowed that bound, takes the exact path:
        // tile max first, O and l rescaled, exponentials redone.  S is still
        // intact in TMEM then, because P is stored only after the check.
        const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2);
        uint64_t lsum[2];
        // One instance of the exponential pass serves both attempts: the
        // fast one against the current max, and (at most once, if the fast
        // one overflowed or the rows have no max yet) the exact one after
        // the tile max and the rescale.  A second copy of the pass in the
        // code measured about 1.5% slower.
        bool exact = __any_sync(0xffffffffu, m == -INFINITY);
#pragma unroll 1
        for (;;) {
          if (exact) {
            const float m_tile = tile_max(s) * P.scale_log2;
            const bool need = m_tile > m + RESCALE_LOG2;
            if (__any_sync(0xffffffffu, need)) {
              const float m_new = need ? m_tile : m;
              const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
              if (jj > 0) {
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                  uint32_t o[16];
                  tmem_ld16(tO + 16u * c, o);
                  tmem_ld_wait16(o);
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st16(tO + 16u * c, o);
                }
              }
              l *= alpha;
              m = m_new;
            }
          }
          exp_pass(s, sc2, (m == -INFINITY) ? 0.f : m, lsum);
          if (exact) break;
          float a0, a1, b0, b1;
          f2_unpack(lsum[0], a0, a1);
          f2_unpack(lsum[1], b0, b1);
          const float tile_sum = (a0 + a1) + (b0 + b1);
          if (!__any_sync(0xffffffffu, !(tile_sum <= SPEC_SUM_LIMIT))) break;
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32u * c, s[c]);
          tmem_ld_wait_only();
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_reg_fence(s[c]);
          mask_tail(s, kv0, e_lim);
          exact = true;
        }
        // columns 32h..32h+31 of S_t receive P[64h .. 64h+63] (two 32-column
        // stores measured 0.4% faster than four of 16)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[32];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            pk[k] = s[2 * h2][k];
            pk[16 + k] = s[2 * h2 + 1][k];
          }
          tmem_st32(tS + 32u * h2, pk);
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(lsum[0], a0, a1);
          f2_unpack(lsum[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(BAR_P_FULL + t));
      }
      if (!ok) break;
      // ---- epilogue: O_t / l
      if (n > 0) {
        const bool got = wait_bar(bar(BAR_O_FULL + t), o_phase, abort_flag, P.timeout_ns, W_SM_O);
        if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
        o_phase ^= 1u;
      }
      // A solo item's half 1 hands its row (m, l) to half 0 through shared
      // memory and is done; half 0 merges both halves' O (same rows, same
      // TMEM lanes) and frees both accumulators:
      //   M = max(m0, m1), a_i = 2^(m_i - M), O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1).
      float* merge_ml = reinterpret_cast<float*>(sgen + SMEM_MERGE);
      if (item.solo && t == 1) {
        // the previous solo item's values must have been read by half 0
        const bool freed = wait_bar(bar(BAR_MERGE_FREE), merge_phase ^ 1u, abort_flag, P.timeout_ns,
                                    W_SM_MERGE);
        if (__any_sync(0xffffffffu, !freed)) { ok = false; break; }
        merge_ml[r_in_tile] = n > 0 ? m : -INFINITY;
        merge_ml[BM + r_in_tile] = n > 0 ? l : 0.f;
        tc_fence_before();
        mbar_arrive(bar(BAR_MERGE));
        merge_phase ^= 1u;
        continue;
      }
      float f0 = 1.f / l, f1 = 0.f, lse2 = m + __log2f(l);
      bool two = false;
      if (item.solo) {
        const bool got = wait_bar(bar(BAR_MERGE), merge_phase, abort_flag, P.timeout_ns, W_SM_MERGE);
        if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
        merge_phase ^= 1u;
        tc_fence_after();
        const float m1 = merge_ml[r_in_tile], l1 = merge_ml[BM + r_in_tile];
        mbar_arrive(bar(BAR_MERGE_FREE));
        two = item.n[1] > 0;
        const float mx = fmaxf(m, m1);
        const float a0 = ex2_approx(m - mx);
        const float a1 = l1 > 0.f ? ex2_approx(m1 - mx) : 0.f;
        const float lt = l * a0 + l1 * a1;
        f0 = a0 / lt;
        f1 = a1 / lt;
        lse2 = mx + __log2f(lt);
      }
      const uint32_t tO1 = tO + 256u;   // half 1's accumulator (solo items)
      if (item.slot < 0) {
        __nv_bfloat16* dst = P.out + (static_cast<size_t>(row) * P.heads + item.h) * HD;
        const bool put = valid && WS_BOUND(g_attn_error, (static_cast<long long>(row) * P.heads + item.h) * HD,
                                           static_cast<long long>(D.lse_stride) * P.heads * HD, 21);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32u * c, o);
          tmem_ld_wait(o);
          if (two) {
            uint32_t o1[32];
            tmem_ld32(tO1 + 32u * c, o1);
            tmem_ld_wait(o1);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(fmaf(__uint_as_float(o1[i]), f1, __uint_as_float(o[i]) * f0));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f0);
          }
          if (put) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]), __uint_as_float(o[8 * q + 1]));
              w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]), __uint_as_float(o[8 * q + 3]));
              w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]), __uint_as_float(o[8 * q + 5]));
              w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]), __uint_as_float(o[8 * q + 7]));
              d4[q] = w;
            }
          }
        }
        if (put && P.lse != nullptr &&
            WS_BOUND(g_attn_error, static_cast<long long>(item.h) * D.lse_stride + row,
                     static_cast<long long>(P.heads) * D.lse_stride, 22))
          P.lse[static_cast<size_t>(item.h) * D.lse_stride + row] = lse2 * LN2;
      } else {
        const size_t slot = static_cast<size_t>(blockIdx.x) * 2 + item.slot;
        const size_t prow = slot * 256 + (item.solo ? 0 : t) * BM + r_in_tile;
        float* dst = P.ws_o + prow * HD;
        const bool put = valid && WS_BOUND(g_attn_error, prow, static_cast<long long>(gridDim.x) * 512, 23);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32u * c, o);
          tmem_ld_wait(o);
          if (two) {
            uint32_t o1[32];
            tmem_ld32(tO1 + 32u * c, o1);
            tmem_ld_wait(o1);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(fmaf(__uint_as_float(o1[i]), f1, __uint_as_float(o[i]) * f0));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f0);
          }
          if (put) {
            float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              d4[q] = make_float4(__uint_as_float(o[4 * q + 0]), __uint_as_float(o[4 * q + 1]),
                                  __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
          }
        }
        if (put) P.ws_lse[prow] = lse2;
      }
      tc_fence_before();
      mbar_arrive(bar(BAR_O_FREE + t));
      if (two) mbar_arrive(bar(BAR_O_FREE + 1));   // half 1's accumulator, read above
    }
  }

  // Teardown.  The TMEM address and the warp index are read afresh, so no
  // value stays live through the role branches (one that did would need the
  // same register under both register budgets, and spill in one of them).
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 9) {
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), TMEM_COLS);
  }
}

namespace {

__device__ __forceinline__ long long group_begin(long long g, long long work, int groups) {
  return g * work / groups;
}

// The group whose range holds flattened index f: the largest g with
// group_begin(g) <= f.
__device__ __forceinline__ int group_of(long long f, long long work, int groups) {
  return static_cast<int>(((f + 1) * groups + work - 1) / work) - 1;
}

// Merge the partial results of the groups that share one head:
//   LSE = log2 sum_s 2^{lse_s},  O = sum_s 2^{lse_s - LSE} O_s,
// as one online pass over the partials (running max, rescaled sum and
// accumulator).  One block per (head, 32 query rows); the block first lists
// the partial slots of its head in shared memory (one 64-bit division pair
// per group, spread over the threads), then each warp merges 4 rows with
// lane c holding columns 4c..4c+3, issuing the loads of its 4 rows x 2
// groups together before merging them.
constexpr int COMBINE_ROWS = 32;
constexpr int COMBINE_MAX_GROUPS = 1024;

__global__ void __launch_bounds__(256)
attn_combine_kernel(Params P) {
  __shared__ int s_gs[COMBINE_MAX_GROUPS];
  Dims D;
  if (!load_dims(P, D)) return;
  const int h = blockIdx.y;
  const long long L = D.kv_tiles;
  // Rows of the unpaired last query tile (solo CTAs) have their own groups,
  // after the paired CTAs; a block of 32 rows lies wholly on one side.
  const int solo_row0 = 2 * BM * P.pairs;
  const bool solo_rows = P.solo && static_cast<int>(blockIdx.x) * COMBINE_ROWS >= solo_row0;
  const int groups = solo_rows ? P.solo_groups : D.groups;
  const int g_lo = group_of(h * L, D.work, groups);
  const int g_hi = group_of((h + 1) * L - 1, D.work, groups);
  if (g_lo == g_hi) return;   // one group covered the head: final output already written
  const int cnt = g_hi - g_lo + 1;
  // slot index (partial row block) of group g: paired rows (g * pairs + pair)
  // * 2 + slot, stored without the pair term, which depends on the row; solo
  // rows (groups * pairs + g) * 2 + slot
  for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
    const int g = g_lo + i;
    const int slot = (h == static_cast<int>(group_begin(g, D.work, groups) / L)) ? 0 : 1;
    s_gs[i] = solo_rows ? (D.groups * P.pairs + g) * 2 + slot : g * 2 * P.pairs + slot;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float* __restrict__ ws_o = P.ws_o;
  const float* __restrict__ ws_lse = P.ws_lse;
  constexpr int RW = COMBINE_ROWS / 8;    // rows per warp
  constexpr int CB = 2;                    // groups per load batch
  const int row0 = blockIdx.x * COMBINE_ROWS + warp * RW;
  float m[RW], sum[RW];
  float4 acc[RW];
#pragma unroll
  for (int k = 0; k < RW; ++k) {
    m[k] = -INFINITY;
    sum[k] = 0.f;
    acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i0 = 0; i0 < cnt; i0 += CB) {
    // all loads of this batch (RW rows x 4 groups) before any arithmetic
    float l[RW][CB];
    float4 o[RW][CB];
#pragma unroll
    for (int k = 0; k < RW; ++k) {
      const int row = row0 + k;
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        l[k][u] = -INFINITY;
        o[k][u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < D.q_len && i0 + u < cnt) {
          const size_t prow = solo_rows
              ? static_cast<size_t>(s_gs[i0 + u]) * 256 + (row - solo_row0)
              : static_cast<size_t>(s_gs[i0 + u] + 2 * (row >> 8)) * 256 + (row & 255);
          if (!WS_BOUND(g_attn_error, prow,
                        (static_cast<long long>(P.groups) * P.pairs + (P.solo ? P.solo_groups : 0)) * 512,
                        24))
            continue;
          l[k][u] = ws_lse[prow];
          o[k][u] = reinterpret_cast<const float4*>(ws_o + prow * HD)[lane];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < RW; ++k) {
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        if (!(l[k][u] > -INFINITY)) continue;   // past cnt, or past q_len
        if (l[k][u] > m[k]) {
          const float c = exp2f(m[k] - l[k][u]);   // 0 while m is -inf
          sum[k] *= c;
          acc[k].x *= c; acc[k].y *= c; acc[k].z *= c; acc[k].w *= c;
          m[k] = l[k][u];
        }
        const float w = exp2f(l[k][u] - m[k]);
        sum[k] += w;
        acc[k].x = fmaf(w, o[k][u].x, acc[k].x);
        acc[k].y = fmaf(w, o[k][u].y, acc[k].y);
        acc[k].z = fmaf(w, o[k][u].z, acc[k].z);
        acc[k].w = fmaf(w, o[k][u].w, acc[k].w);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < RW; ++k) {
    const int row = row0 + k;
    if (row >= D.q_len) break;
    const float inv = 1.f / sum[k];
    uint2 packed;
    packed.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
    packed.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
    if (WS_BOUND(g_attn_error, (static_cast<long long>(row) * P.heads + h) * HD,
                 static_cast<long long>(D.lse_stride) * P.heads * HD, 25))
      reinterpret_cast<uint2*>(P.out + (static_cast<size_t>(row) * P.heads + h) * HD)[lane] = packed;
    if (lane == 0 && P.lse != nullptr &&
        WS_BOUND(g_attn_error, static_cast<long long>(h) * D.lse_stride + row,
                 static_cast<long long>(P.heads) * D.lse_stride, 26))
      P.lse[static_cast<size_t>(h) * D.lse_stride + row] = (m[k] + log2f(sum[k])) * LN2;
  }
}

long long host_group_of(long long f, long long work, int groups) {
  return ((f + 1) * groups + work - 1) / work - 1;
}

}  // namespace

namespace {

// Groups of CTAs over `work` (head, key tile) units: at most `cap`; with at
// least one group per head, a multiple of the head count, so that every
// head's key range splits evenly on head boundaries, one work item per CTA
// (the 192x336 unit: 72 groups of a third of a head, 9.5% faster than 74
// groups whose ranges straddle heads).
long long plan_groups(long long cap, int heads, long long work) {
  long long g = cap;
  if (g >= heads) g = (g / heads) * heads;
  if (g < 1) g = 1;
  if (g > work) g = work;
  if (g > COMBINE_MAX_GROUPS) g = COMBINE_MAX_GROUPS;   // the merge lists a head's groups in smem
  return g;
}

bool any_head_split(long long kv_tiles, int heads, long long work, long long groups) {
  for (int h = 0; h < heads; ++h) {
    const long long lo = host_group_of(static_cast<long long>(h) * kv_tiles, work, groups);
    const long long hi = host_group_of(static_cast<long long>(h + 1) * kv_tiles - 1, work, groups);
    if (lo != hi) return true;
  }
  return false;
}

}  // namespace

bool plan_tc_attn(TcAttnPlan& p, bool prefill, int heads, int q_len, int q_row0, int kv_len,
                  int n_blocks, int num_sms, int side_len, bool allow_solo) {
  p = TcAttnPlan{};
  p.prefill = prefill ? 1 : 0;
  p.heads = heads;
  p.q_len = q_len;
  p.q_row0 = q_row0;
  p.kv_len = kv_len;
  p.n_blocks = n_blocks;
  p.qtiles = (q_len + BM - 1) / BM;
  p.pairs = (p.qtiles + 1) / 2;
  p.kv_tiles = (kv_len + BN - 1) / BN;
  if (q_len <= 0 || kv_len <= 0 || heads <= 0 || num_sms <= 0) return false;
  if (side_len < 0 || side_len > kv_len || (prefill && side_len > 0)) return false;
  p.side_len = side_len;
  if (side_len > 0) {
    // the cache part and the side part are tiled separately
    p.kv_tiles_c = (kv_len - side_len + BN - 1) / BN;
    p.kv_tiles = p.kv_tiles_c + (side_len + BN - 1) / BN;
  }
  if (prefill) {
    // work units: a head and a mirrored couple of query-tile pairs
    const long long items = static_cast<long long>(heads) * ((p.pairs + 1) / 2);
    if (items > (1LL << 30)) return false;
    p.n_items = static_cast<int>(items);
    p.grid = p.n_items < num_sms ? p.n_items : num_sms;
    p.split = false;
    p.workspace_bytes = 0;
    return true;
  }
  p.work = static_cast<long long>(heads) * p.kv_tiles;
  if (allow_solo && (p.qtiles & 1)) {
    // The last query tile is unpaired: it gets solo CTAs, which run a key
    // range at twice the rate of a paired CTA, so they get half as many
    // groups of twice the range: full pairs * 2G + G CTAs in all.
    p.solo = 1;
    p.pairs = p.qtiles / 2;
    const long long g1 = plan_groups(num_sms / (2 * p.pairs + 1), heads, p.work);
    const long long g0 = p.pairs > 0 ? plan_groups(2 * g1, heads, p.work) : 0;
    p.groups = static_cast<int>(g0);
    p.solo_groups = static_cast<int>(g1);
    const long long grid = g0 * p.pairs + g1;
    if (grid > (1LL << 30) || grid > num_sms) return false;
    p.grid = static_cast<int>(grid);
    p.split = any_head_split(p.kv_tiles, heads, p.work, g1) ||
              (g0 > 0 && any_head_split(p.kv_tiles, heads, p.work, g0));
  } else {
    const long long g = plan_groups(num_sms / p.pairs, heads, p.work);
    p.groups = static_cast<int>(g);
    const long long grid = g * p.pairs;
    if (grid > (1LL << 30)) return false;
    p.grid = static_cast<int>(grid);
    p.split = any_head_split(p.kv_tiles, heads, p.work, g);
  }
  p.workspace_bytes = p.split ? static_cast<size_t>(p.grid) * 2 * 256 * (HD + 1) * sizeof(float) : 0;
  return true;
}

void plan_force_split(TcAttnPlan& p) {
  p.split = true;
  p.workspace_bytes = static_cast<size_t>(p.grid) * 2 * 256 * (HD + 1) * sizeof(float);
}

cudaError_t launch_attn_tc_bf16(const TcAttnPlan& plan, const TcAttnArgs& a,
                                const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, const CUtensorMap& tm_ks,
                                const CUtensorMap& tm_vs, const CUtensorMap& tm_kc,
                                const CUtensorMap& tm_vc, uint64_t timeout_ns, cudaStream_t s) {
  // One-time set-up per device (shared-memory opt-in, register-split check),
  // under a lock so that threads making their first call at once do it once.
  static std::mutex setup_mu;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(setup_mu);
    if (!attr_done[dev]) {
      err = cudaFuncSetAttribute(attn_tc_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_ALLOC);
      if (err != cudaSuccess) return err;
      // The warpgroup register split must fit in the registers the block is
      // launched with, or setmaxnreg.inc would wait forever: refuse instead.
      cudaFuncAttributes fa{};
      err = cudaFuncGetAttributes(&fa, attn_tc_bf16_kernel);
      if (err != cudaSuccess) return err;
      if (fa.numRegs * NUM_THREADS < REGS_NEEDED) return cudaErrorInvalidConfiguration;
      attr_done[dev] = true;
    }
  }
  Params P{};
  P.prefill = plan.prefill;
  P.heads = plan.heads;
  P.q_len = plan.q_len;
  P.q_row0 = plan.q_row0;
  P.kv_len = plan.kv_len;
  P.n_blocks = plan.n_blocks;
  P.pairs = plan.pairs;
  P.kv_tiles = plan.kv_tiles;
  P.side = plan.side_len > 0 ? 1 : 0;
  P.kv_tiles_c = plan.kv_tiles_c;
  P.cache_len = plan.kv_len - plan.side_len;
  P.n_side = plan.side_len;
  P.commit = (plan.side_len > 0 && a.commit) ? 1 : 0;
  P.capacity = a.capacity;
  P.groups = plan.groups;
  P.work = plan.work;
  P.n_items = plan.n_items;
  P.scale_log2 = a.scale * 1.4426950408889634f;
  P.offs = a.offs;
  P.out = static_cast<__nv_bfloat16*>(a.out);
  P.lse = a.lse;
  if (plan.split) {
    P.ws_o = static_cast<float*>(a.workspace);
    P.ws_lse = P.ws_o + static_cast<size_t>(plan.grid) * 2 * 256 * HD;
  }
  P.timeout_ns = timeout_ns;
  P.force_stall = a.force_stall;
  // device-resident sizes: the plan was made for the largest unit (q_len =
  // q_max) and the whole cache (kv_len = capacity)
  P.dev_state = a.dev_state;
  P.q_max = plan.q_len;
  P.solo = plan.solo;
  P.solo_groups = plan.solo_groups;
  attn_tc_bf16_kernel<<<plan.grid, NUM_THREADS, SMEM_ALLOC, s>>>(tm_q, tm_k, tm_v, tm_ks, tm_vs,
                                                                 tm_kc, tm_vc, P);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (plan.split) {
    dim3 grid((plan.q_len + COMBINE_ROWS - 1) / COMBINE_ROWS, plan.heads);
    attn_combine_kernel<<<grid, 256, 0, s>>>(P);
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t read_attn_device_error(int* code, int* info) {
  unsigned int h[2] = {0u, 0u};
  cudaError_t err = cudaMemcpyFromSymbol(h, g_attn_error, sizeof(h));
  if (err != cudaSuccess) return err;
  *code = static_cast<int>(h[0]);
  *info = static_cast<int>(h[1]);
  return cudaSuccess;
}

cudaError_t clear_attn_device_error() {
  const unsigned int z[2] = {0u, 0u};
  return cudaMemcpyToSymbol(g_attn_error, z, sizeof(z));
}

}  // namespace ws
