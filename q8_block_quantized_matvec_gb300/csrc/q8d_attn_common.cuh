// Device helpers shared by the two decode-attention kernels.
#pragma once
#include "q8d_attn.cuh"
#include "q8d_internal.cuh"

namespace q8d {

// Decode-step prologue of one head row held by a warp (lane holds elements
// lane + 32t): bias add, per-head RMSNorm, rotary embedding of the pairs
// (i, i + D/2), in that order ("IV.4: One command buffer per token", the
// q/k projections are followed by QK-norm and RoPE).  Pairs sit in one lane.
template <int D>
__device__ __forceinline__ void head_prologue(float (&v)[D / 32], int lane, const float* bias,
                                              const float* norm_w, float eps, const float* cosr,
                                              const float* sinr) {
  constexpr int T = D / 32;
  if (bias) {
#pragma unroll
    for (int t = 0; t < T; ++t) v[t] += bias[lane + 32 * t];
  }
  if (norm_w) {
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < T; ++t) ss = fmaf(v[t], v[t], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / (float)D + eps);
#pragma unroll
    for (int t = 0; t < T; ++t) v[t] = v[t] * inv * norm_w[lane + 32 * t];
  }
  if (cosr) {
#pragma unroll
    for (int t = 0; t < T / 2; ++t) {
      const int i = lane + 32 * t;
      const float c = cosr[i], sn = sinr[i];
      const float a = v[t], bb = v[t + T / 2];
      v[t] = a * c - bb * sn;
      v[t + T / 2] = a * sn + bb * c;
    }
  }
}

}  // namespace q8d
