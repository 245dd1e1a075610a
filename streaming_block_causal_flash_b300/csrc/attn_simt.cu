// attn_simt.cu -- block-causal attention in fp32 on CUDA cores.
//
// Same visibility rule as the tensor-core path: a token sees its own block in
// both directions and every earlier block, never a later one (Wan Streamer
// real-time AV explainer (xiaohu-jiedu.pages.dev), "怎么做到边听边说、随时能打断").
// Used for fp32 inputs (head_dim 64 or 128), where an fp32 result within
// 1e-5 of the exact value is required and bf16/tf32 tensor cores do not
// reach it.
//
// One warp per (query row, head).  Keys are visited 32 at a time, one key per
// lane: the lane forms the full dot product of its key with the query (held
// in shared memory), the warp keeps an online softmax (running max and sum),
// and each lane accumulates D/32 output columns with the 32 weights
// broadcast by shuffles.
#include "ws_internal.h"

namespace ws {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ int row_limit(const int32_t* offs, int n_blocks, int token) {
  int lo = 0, hi = n_blocks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= token) lo = mid;
    else hi = mid - 1;
  }
  return __ldg(offs + lo + 1);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_f32_kernel(SimtAttnArgs a) {
  constexpr int PER_LANE = D / 32;
  __shared__ float q_s[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_work = static_cast<int64_t>(a.q_len) * a.heads;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + warp; w < n_work;
       w += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int row = static_cast<int>(w / a.heads);
    const int h = static_cast<int>(w % a.heads);
    const int e = a.prefill ? row_limit(a.offs, a.n_blocks, a.q_row0 + row) : a.kv_len;
    const float* qrow = a.q + (static_cast<int64_t>(row) * a.heads + h) * D;
    for (int d = lane; d < D; d += 32) q_s[warp][d] = qrow[d];
    __syncwarp();
    const float* kh = a.k + static_cast<int64_t>(h) * a.capacity * D;
    const float* vh = a.v + static_cast<int64_t>(h) * a.capacity * D;
    float m = -INFINITY, l = 0.f;
    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < e; j0 += 32) {
      const int j = j0 + lane;
      float x = -INFINITY;
      if (j < e) {
        const float4* kr = reinterpret_cast<const float4*>(kh + static_cast<int64_t>(j) * D);
        float dot = 0.f;
#pragma unroll 8
        for (int d4 = 0; d4 < D / 4; ++d4) {
          const float4 kv = kr[d4];
          dot = fmaf(q_s[warp][4 * d4 + 0], kv.x, dot);
          dot = fmaf(q_s[warp][4 * d4 + 1], kv.y, dot);
          dot = fmaf(q_s[warp][4 * d4 + 2], kv.z, dot);
          dot = fmaf(q_s[warp][4 * d4 + 3], kv.w, dot);
        }
        x = dot * a.scale;
      }
      float cmax = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const float m_new = fmaxf(m, cmax);            // finite: key j0 is visible
      const float alpha = expf(m - m_new);           // 0 on the first chunk
      const float p = (j < e) ? expf(x - m_new) : 0.f;
      float psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l = l * alpha + psum;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i) acc[i] *= alpha;
      const int nk = min(32, e - j0);
      for (int jj = 0; jj < nk; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const float* vr = vh + static_cast<int64_t>(j0 + jj) * D;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) acc[i] = fmaf(pj, vr[lane + 32 * i], acc[i]);
      }
      m = m_new;
    }
    const float inv = 1.f / l;
    float* orow = a.out + (static_cast<int64_t>(row) * a.heads + h) * D;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) orow[lane + 32 * i] = acc[i] * inv;
    if (a.lse != nullptr && lane == 0) a.lse[static_cast<int64_t>(h) * a.q_len + row] = m + logf(l);
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_attn_simt_f32(const SimtAttnArgs& a, cudaStream_t s) {
  const int64_t n_work = static_cast<int64_t>(a.q_len) * a.heads;
  if (n_work == 0) return cudaSuccess;
  int64_t blocks = (n_work + kWarps - 1) / kWarps;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  if (a.head_dim == 64)
    attn_simt_f32_kernel<64><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(a);
  else
    attn_simt_f32_kernel<128><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ws
