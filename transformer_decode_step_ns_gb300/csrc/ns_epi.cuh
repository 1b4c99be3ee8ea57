// Element formulas of the fused epilogues, written once with explicit roundings so that every
// kernel that applies them (the cluster and persistent projections, the embedding kernel and
// the persistent step kernel) computes them the same way.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace ns {

// RoPE on one (i, i + d/2) pair: (x_lo, x_hi) -> (x_lo c - x_hi s, x_hi c + x_lo s).
__device__ __forceinline__ float rope_lo(float x_lo, float x_hi, float c, float sn) {
  return __fmaf_rn(x_lo, c, -__fmul_rn(x_hi, sn));
}
__device__ __forceinline__ float rope_hi(float x_lo, float x_hi, float c, float sn) {
  return __fmaf_rn(x_hi, c, __fmul_rn(x_lo, sn));
}

// silu(g) * u
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdividef(g, __fadd_rn(1.f, __expf(-g))), u);
}

// 1 / sqrt(mean of squares + eps) from a row's summed squares
__device__ __forceinline__ float rms_scale(float sumsq, int n, float eps) {
  return rsqrtf(__fadd_rn(__fdiv_rn(sumsq, static_cast<float>(n)), eps));
}

// cos and sin of the RoPE angle pos * inv_freq (inv_freq = theta^(-2i/d), an fp64 host table):
// the angle is formed in fp64 and reduced to [-pi, pi] with the two-constant Cody-Waite scheme
// (Cody & Waite, "Software Manual for the Elementary Functions", 1980), then fp32 sincosf.
__device__ __forceinline__ void rope_cos_sin(int pos, double inv_freq, float* cs, float* sn) {
  const double ang = static_cast<double>(pos) * inv_freq;
  const double k = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
  double r = fma(-k, 6.283185307179586, ang);           // 2 pi, high part
  r = fma(-k, 2.4492935982947064e-16, r);               // 2 pi - high part
  sincosf(static_cast<float>(r), sn, cs);
}

}  // namespace ns
