// Device helpers shared by the two decode-attention kernels.
#pragma once
#include "q8d_attn.cuh"
#include "q8d_internal.cuh"

namespace q8d {

// v = hi + lo with hi = f16(v), lo = f16(v - hi), for a pair of floats.
__device__ __forceinline__ void attn_split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// d += a * b on the tensor cores: m16n8k16, f16 operands, f32 accumulators.
__device__ __forceinline__ void attn_mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four transposed 8x8 b16 tiles from shared memory (the B operand of P.V).
__device__ __forceinline__ void attn_ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                   uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

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

// Q8_0 store of one 32-element block held by a warp (lane j holds element
// j): the packed KV cache's quantizer ("minfer Metal Backend Design",
// "Execution dispatch": the store is byte-identical to the CPU quantizer,
// read as the Q8_0 format's reference quantizer in f32):
//   amax = max |x|, d = amax / 127, id = d != 0 ? 1 / d : 0,
//   q_j = x_j * id rounded to nearest with halves away from zero (roundf),
//   scale = d rounded to binary16 (nearest even).
// Every operation is a correctly rounded f32 operation (IEEE division, a
// single product, no contraction), so the bytes match a scalar CPU
// quantizer bit for bit.  blk: the block's 34 bytes in global memory, at
// an even address (the scale is written with one 16-bit store).
__device__ __forceinline__ void quantize_q8_0_warp(float x, uint8_t* blk, int lane) {
  float amax = fabsf(x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __fdiv_rn(amax, 127.0f);
  const float id = d != 0.f ? __fdiv_rn(1.0f, d) : 0.f;
  const int q = (int)roundf(__fmul_rn(x, id));
  blk[2 + lane] = (uint8_t)(int8_t)q;
  if (lane == 0) *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(__float2half_rn(d));
}

}  // namespace q8d
