// Device helpers of the Q8_0 matvec consumers, shared by the standalone
// matvec kernel (q8d_gemv.cu) and the persistent decode-step kernel
// (q8d_megastep.cu).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "q8d_internal.cuh"

namespace q8d {
namespace mv {

// Shared-memory load of a weight word.  Not volatile: the compiler may
// schedule these loads freely (e.g. the next row's ahead of this row's
// arithmetic).  Callers make the stage address depend on the mbarrier wait
// (after_wait) so that no load moves above it, and every loaded value feeds
// a store that precedes the stage's release.
template <int OFF>
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}

// Returns v through an opaque instruction ordered after the preceding
// volatile asm (the mbarrier wait): addresses derived from it cannot be
// hoisted above the wait.
__device__ __forceinline__ uint32_t after_wait(uint32_t v) {
  asm volatile("" : "+r"(v)::"memory");
  return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// The nine shared-memory words holding the block at byte address `o`
// (2-byte aligned): the 34 bytes of the block start in the first word.
__device__ __forceinline__ void block_words(uint32_t o, uint32_t (&a)[9]) {
  const uint32_t w0 = o & ~3u;
  a[0] = lds32<0>(w0);
  a[1] = lds32<4>(w0);
  a[2] = lds32<8>(w0);
  a[3] = lds32<12>(w0);
  a[4] = lds32<16>(w0);
  a[5] = lds32<20>(w0);
  a[6] = lds32<24>(w0);
  a[7] = lds32<28>(w0);
  a[8] = lds32<32>(w0);
}

// scale * sum_j q_j x_j for the block at byte address `o` whose words are
// `a` (block_words).  Alignment modes: AM = 1, the block starts at byte 2
// of a word (scale = upper half, quants = the next 8 words); AM = 0, it
// starts at a word (scale = lower half, quants from byte 2 on); AM = 2,
// decided per lane from o.
template <int AM>
__device__ __forceinline__ float block_dot_words(uint32_t (&a)[9], uint32_t o,
                                                 const uint64_t (&x2)[16]) {
  float sc;
  uint32_t shift = 16;
  if constexpr (AM == 2) {
    const bool odd = (o & 2u) != 0;
    sc = f16_bits_to_f32(odd ? (a[0] >> 16) : (a[0] & 0xFFFFu));
    shift = odd ? 32u : 16u;
  } else {
    const __half2 sh = *reinterpret_cast<const __half2*>(&a[0]);
    sc = AM ? __high2float(sh) : __low2float(sh);
  }
  const uint64_t bias2 = pack2(-kMagicBias, -kMagicBias);
  uint64_t c[4] = {pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f)};
  if constexpr (AM == 0) {
    // quants start at byte 2 of word 0: quant 4k+i is byte (2+i) mod 4 of
    // word k + (2+i)/4, so each is picked straight from its word (no
    // funnel shift); the sign flip is applied to all nine words once
#pragma unroll
    for (int k = 0; k < 9; ++k) a[k] ^= 0x80808080u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t q01 =
          add2(pack2(magic_byte(a[k], magic_sel(2)), magic_byte(a[k], magic_sel(3))), bias2);
      const uint64_t q23 =
          add2(pack2(magic_byte(a[k + 1], magic_sel(0)), magic_byte(a[k + 1], magic_sel(1))), bias2);
      c[(2 * k) & 3] = fma2(q01, x2[2 * k], c[(2 * k) & 3]);
      c[(2 * k + 1) & 3] = fma2(q23, x2[2 * k + 1], c[(2 * k + 1) & 3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t w;
      if constexpr (AM == 1) w = a[k + 1];
      else w = __funnelshift_rc(a[k], a[k + 1], shift);
      w ^= 0x80808080u;
      const uint64_t q01 = add2(pack2(magic_byte(w, magic_sel(0)), magic_byte(w, magic_sel(1))), bias2);
      const uint64_t q23 = add2(pack2(magic_byte(w, magic_sel(2)), magic_byte(w, magic_sel(3))), bias2);
      c[(2 * k) & 3] = fma2(q01, x2[2 * k], c[(2 * k) & 3]);
      c[(2 * k + 1) & 3] = fma2(q23, x2[2 * k + 1], c[(2 * k + 1) & 3]);
    }
  }
  const uint64_t t = add2(add2(c[0], c[1]), add2(c[2], c[3]));
  float lo, hi;
  unpack2(t, lo, hi);
  return sc * (lo + hi);
}

// scale * sum_j q_j x_j for the block at shared-memory byte address `o`.
template <int AM>
__device__ __forceinline__ float block_dot(uint32_t o, const uint64_t (&x2)[16]) {
  uint32_t a[9];
  block_words(o, a);
  return block_dot_words<AM>(a, o, x2);
}

__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// try_wait that lets the thread sleep (up to a few microseconds) until the
// phase completes instead of returning at once: waiting warps stop taking
// issue slots from the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(4000u)
      : "memory");
  return ok != 0;
}

// Bounded wait (2^21 polls, each sleeping at most the hint: a few seconds)
// that gives up at once when another thread of the CTA already gave up, so
// that every warp still reaches the CTA barriers quickly.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
  for (uint32_t i = 0; i < (1u << 21); ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// Barrier among the consumer warps only (the producer warp runs free).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

}  // namespace mv
}  // namespace q8d
