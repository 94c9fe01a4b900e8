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

// When tickets are in use, the last chunk CTA of (sequence b, KV head g) to
// finish merges the partials of all chunks of that KV head's G query heads
// ({m, l, O}: M = max m, w = 2^(m - M), out = sum w O / sum w l) in chunk
// order, and resets the ticket for the next launch.  `scratch` is shared
// memory free for 2 * G * nact + G floats.  Every thread of the CTA calls it.
template <int D>
__device__ void ticket_combine(const AttnParams& P, int L, int tpc, int b, int g, int G,
                               uint8_t* scratch) {
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* smem = scratch;
  __threadfence();
  __syncthreads();
  const int nact = (L + tpc - 1) / tpc;
  if (tid == 0) s_last = (atomicAdd(&P.tickets[b * P.n_kv_heads + g], 1) == nact - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* wts = reinterpret_cast<float*>(smem);  // [G][nact] chunk weights (first m, then w)
  float* lsm = wts + G * nact;                   // [G][nact] chunk denominators
  float* lh = lsm + G * nact;                    // [G] merged denominators
  // all chunk maxima and denominators of the G heads, loaded together
  for (int e = tid; e < G * nact; e += blockDim.x) {
    const int h = e / nact, cc = e % nact;
    const long long hq = (long long)b * P.n_heads + (long long)g * G + h;
    wts[e] = __ldcg(P.ws_m + hq * P.nc + cc);
    lsm[e] = __ldcg(P.ws_l + hq * P.nc + cc);
  }
  __syncthreads();
  for (int h = warp; h < G; h += (int)(blockDim.x >> 5)) {
    float M = -INFINITY;
    for (int cc = lane; cc < nact; cc += 32) M = fmaxf(M, wts[h * nact + cc]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    __syncwarp();
    float ls = 0.f;
    for (int cc = lane; cc < nact; cc += 32) {
      const float mc = wts[h * nact + cc];
      const float w = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
      wts[h * nact + cc] = w;
      ls = fmaf(lsm[h * nact + cc], w, ls);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) lh[h] = ls;
  }
  __syncthreads();
  // weighted sum of the chunk outputs: eight independent loads in flight
  for (int e = tid; e < G * D; e += blockDim.x) {
    const int h = e / D, j = e % D;
    const long long hq = (long long)b * P.n_heads + (long long)g * G + h;
    const float* O = P.ws_o + hq * P.nc * D + j;
    const float* w = wts + h * nact;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int cc = 0;
    for (; cc + 8 <= nact; cc += 8) {
      float o8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) o8[u] = __ldcg(O + (long long)(cc + u) * D);
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = fmaf(o8[u], w[cc + u], a[u]);
    }
    for (; cc < nact; ++cc) a[0] = fmaf(__ldcg(O + (long long)cc * D), w[cc], a[0]);
    const float acc = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
    P.out[hq * D + j] = acc / lh[h];
  }
  if (tid == 0) P.tickets[b * P.n_kv_heads + g] = 0;  // ready for the next launch
}

}  // namespace q8d
