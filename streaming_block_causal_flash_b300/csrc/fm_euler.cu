// fm_euler.cu -- one Euler step of the flow-matching solver, z <- z - dtau * v.
//
// Interpolant z_tau = (1 - tau) z_0 + tau eps with velocity eps - z_0
// ("全双工语音模型精读⑫：Wan-Streamer" (alwayszhang.cn), 3.2); the solver walks
// tau from 1 (noise) towards 0 (clean latent).  One fp32 FMA per element,
// z in place, v in bf16 or fp32, optionally a bf16 copy of the new z for the
// next network input.  Eight elements per thread step: 32 B of z, 16 B (bf16)
// or 32 B (fp32) of v, 16 B of bf16 output.
#include <cuda_bf16.h>

#include "ws_internal.h"

namespace ws {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float4 ld_f4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

template <bool kVBf16>
__device__ __forceinline__ void load_v8(const void* v_raw, int64_t i, float (&vf)[8]) {
  if constexpr (kVBf16) {
    const uint4 vv = reinterpret_cast<const uint4*>(v_raw)[i];
    bf16x8_to_f32(vv, vf);
  } else {
    const float4 a = ld_f4(static_cast<const float*>(v_raw) + 8 * i);
    const float4 b = ld_f4(static_cast<const float*>(v_raw) + 8 * i + 4);
    vf[0] = a.x; vf[1] = a.y; vf[2] = a.z; vf[3] = a.w;
    vf[4] = b.x; vf[5] = b.y; vf[6] = b.z; vf[7] = b.w;
  }
}

template <bool kOutBf16>
__device__ __forceinline__ void update8(float* __restrict__ z, __nv_bfloat16* __restrict__ zb,
                                        int64_t i, float4 z0, float4 z1, const float (&vf)[8],
                                        float neg) {
  z0.x = fmaf(neg, vf[0], z0.x);
  z0.y = fmaf(neg, vf[1], z0.y);
  z0.z = fmaf(neg, vf[2], z0.z);
  z0.w = fmaf(neg, vf[3], z0.w);
  z1.x = fmaf(neg, vf[4], z1.x);
  z1.y = fmaf(neg, vf[5], z1.y);
  z1.z = fmaf(neg, vf[6], z1.z);
  z1.w = fmaf(neg, vf[7], z1.w);
  reinterpret_cast<float4*>(z)[2 * i] = z0;
  reinterpret_cast<float4*>(z)[2 * i + 1] = z1;
  if constexpr (kOutBf16) {
    uint4 o;
    o.x = f32x2_to_bf16x2(z0.x, z0.y);
    o.y = f32x2_to_bf16x2(z0.z, z0.w);
    o.z = f32x2_to_bf16x2(z1.x, z1.y);
    o.w = f32x2_to_bf16x2(z1.z, z1.w);
    reinterpret_cast<uint4*>(zb)[i] = o;
  }
}

// Each thread step handles two groups of eight elements, one grid stride
// apart, with all loads issued before the stores.
template <bool kVBf16, bool kOutBf16>
__global__ void __launch_bounds__(kThreads)
fm_euler_kernel(float* __restrict__ z, const void* __restrict__ v_raw,
                __nv_bfloat16* __restrict__ zb, int64_t n, float dtau) {
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const float neg = -dtau;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n8;
       i += 2 * stride) {
    const int64_t j = i + stride;
    const bool has_j = j < n8;
    const float4 a0 = ld_f4(z + 8 * i);
    const float4 a1 = ld_f4(z + 8 * i + 4);
    float va[8], vb[8];
    load_v8<kVBf16>(v_raw, i, va);
    float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
    if (has_j) {
      b0 = ld_f4(z + 8 * j);
      b1 = ld_f4(z + 8 * j + 4);
      load_v8<kVBf16>(v_raw, j, vb);
    }
    update8<kOutBf16>(z, zb, i, a0, a1, va, neg);
    if (has_j) update8<kOutBf16>(z, zb, j, b0, b1, vb, neg);
  }
  // ragged tail (n not a multiple of 8): the first block finishes it
  if (blockIdx.x == 0) {
    for (int64_t j = n8 * 8 + threadIdx.x; j < n; j += kThreads) {
      float vj;
      if constexpr (kVBf16)
        vj = __bfloat162float(static_cast<const __nv_bfloat16*>(v_raw)[j]);
      else
        vj = static_cast<const float*>(v_raw)[j];
      const float zn = fmaf(neg, vj, z[j]);
      z[j] = zn;
      if constexpr (kOutBf16) zb[j] = __float2bfloat16_rn(zn);
    }
  }
}

// Guided step (classifier-free guidance on the velocity):
//   v = v_u + w (v_c - v_u),  z <- z - dtau v,
// in fp32 as d = v_c - v_u, v = fma(w, d, v_u), z = fma(-dtau, v, z).  One
// pass reads z and both velocities and writes z (and the bf16 copy): 12 B per
// element with bf16 velocities.  Two groups of eight per thread step, loads
// first.
template <bool kOutBf16>
__device__ __forceinline__ void guided8(float* __restrict__ z, __nv_bfloat16* __restrict__ zb,
                                        int64_t i, float4 z0, float4 z1, const float (&vu)[8],
                                        const float (&vc)[8], float w, float neg) {
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = fmaf(w, vc[e] - vu[e], vu[e]);
  update8<kOutBf16>(z, zb, i, z0, z1, v, neg);
}

template <bool kVBf16, bool kOutBf16>
__global__ void __launch_bounds__(kThreads)
fm_euler_cfg_kernel(float* __restrict__ z, const void* __restrict__ vu_raw,
                    const void* __restrict__ vc_raw, __nv_bfloat16* __restrict__ zb, int64_t n,
                    float w, float dtau) {
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const float neg = -dtau;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n8;
       i += 2 * stride) {
    const int64_t j = i + stride;
    const bool has_j = j < n8;
    const float4 a0 = ld_f4(z + 8 * i);
    const float4 a1 = ld_f4(z + 8 * i + 4);
    float ua[8], ca[8], ub[8], cb[8];
    load_v8<kVBf16>(vu_raw, i, ua);
    load_v8<kVBf16>(vc_raw, i, ca);
    float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
    if (has_j) {
      b0 = ld_f4(z + 8 * j);
      b1 = ld_f4(z + 8 * j + 4);
      load_v8<kVBf16>(vu_raw, j, ub);
      load_v8<kVBf16>(vc_raw, j, cb);
    }
    guided8<kOutBf16>(z, zb, i, a0, a1, ua, ca, w, neg);
    if (has_j) guided8<kOutBf16>(z, zb, j, b0, b1, ub, cb, w, neg);
  }
  if (blockIdx.x == 0) {
    for (int64_t e = n8 * 8 + threadIdx.x; e < n; e += kThreads) {
      float u, c;
      if constexpr (kVBf16) {
        u = __bfloat162float(static_cast<const __nv_bfloat16*>(vu_raw)[e]);
        c = __bfloat162float(static_cast<const __nv_bfloat16*>(vc_raw)[e]);
      } else {
        u = static_cast<const float*>(vu_raw)[e];
        c = static_cast<const float*>(vc_raw)[e];
      }
      const float zn = fmaf(neg, fmaf(w, c - u, u), z[e]);
      z[e] = zn;
      if constexpr (kOutBf16) zb[e] = __float2bfloat16_rn(zn);
    }
  }
}

}  // namespace

cudaError_t launch_fm_euler(float* z, const void* v, bool v_is_bf16, void* z_bf16_out,
                            int64_t n, float dtau, int num_sms, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t n8 = n / 8;
  int64_t blocks = (n8 + 2 * kThreads - 1) / (2 * kThreads);
  const int64_t cap_blocks = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  auto* zb = static_cast<__nv_bfloat16*>(z_bf16_out);
  const unsigned g = static_cast<unsigned>(blocks);
  if (v_is_bf16) {
    if (zb) fm_euler_kernel<true, true><<<g, kThreads, 0, s>>>(z, v, zb, n, dtau);
    else    fm_euler_kernel<true, false><<<g, kThreads, 0, s>>>(z, v, zb, n, dtau);
  } else {
    if (zb) fm_euler_kernel<false, true><<<g, kThreads, 0, s>>>(z, v, zb, n, dtau);
    else    fm_euler_kernel<false, false><<<g, kThreads, 0, s>>>(z, v, zb, n, dtau);
  }
  return cudaGetLastError();
}

}  // namespace ws

namespace ws {

cudaError_t launch_fm_euler_cfg(float* z, const void* v_uncond, const void* v_cond, bool v_is_bf16,
                                void* z_bf16_out, int64_t n, float guidance, float dtau,
                                int num_sms, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t n8 = n / 8;
  int64_t blocks = (n8 + 2 * kThreads - 1) / (2 * kThreads);
  const int64_t cap_blocks = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  auto* zb = static_cast<__nv_bfloat16*>(z_bf16_out);
  const unsigned g = static_cast<unsigned>(blocks);
  if (v_is_bf16) {
    if (zb) fm_euler_cfg_kernel<true, true><<<g, kThreads, 0, s>>>(z, v_uncond, v_cond, zb, n, guidance, dtau);
    else    fm_euler_cfg_kernel<true, false><<<g, kThreads, 0, s>>>(z, v_uncond, v_cond, zb, n, guidance, dtau);
  } else {
    if (zb) fm_euler_cfg_kernel<false, true><<<g, kThreads, 0, s>>>(z, v_uncond, v_cond, zb, n, guidance, dtau);
    else    fm_euler_cfg_kernel<false, false><<<g, kThreads, 0, s>>>(z, v_uncond, v_cond, zb, n, guidance, dtau);
  }
  return cudaGetLastError();
}

}  // namespace ws
