// Q8_0 block dot products on the tensor cores (mma.sync m16n8k16, f16
// operands, f32 accumulation): the fragment layout shared by the standalone
// matvec (q8d_gemv_mma.cu) and the step kernel's matvec phases.
//
//   y[r] = sum_b scale(r,b) * sum_j q(r,b,j) * x[32b+j]
// ("IV.4: One command buffer per token", "Eight kernels": q8_matvec; the
// product is summed inside the block and scaled once per block).
//
//  * A (16 x 16 per MMA): quants as exact f16 (a sign-flipped byte under the
//    exponent byte 0x64 is 1152 + q; one sub.f16x2 removes the 1152).  The
//    16 A rows are 8 weight rows x 2 column halves, so a unit of work is 8
//    rows x 4 blocks of the same byte alignment (blocks base, base+2,
//    base+4, base+6; half 0 = {base, base+4}, half 1 = {base+2, base+6}),
//    and two units (even and odd blocks) make a pair of 8 consecutive
//    blocks.  Each thread feeds one 32-bit word of quants per MMA (its
//    contraction indices are permuted to match: 4 consecutive bytes).
//  * B (16 x 8): the 8 columns are 4 blocks x (x_hi, x_lo), x = hi + lo in
//    f16 after a power-of-two scale (max |x| of the scaled range in
//    [2^14, 2^15)), so every product is exact in f32; columns that pair a
//    row half with the other half's blocks are zero.  A block's fragment is
//    144 bytes: 8 words x 16 bytes {hi(k0,k1), hi(k2,k3), lo(k0,k1),
//    lo(k2,k3)} in the permuted byte order (word_quant), + 16 pad bytes.
//  * D: every thread ends a unit with the (hi, lo) partials of one (row,
//    block) pair, which it scales by that block's f16 scale.
// Blocks of odd index start two bytes after a word boundary, so their quants
// are word aligned; for even blocks the words at +4 .. +28 hold quants 2..29
// and the last word is assembled from the block's first and last words.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "q8d_internal.cuh"

namespace q8d {
namespace tc {

constexpr int kXfBlock = 144;  // x fragment bytes per block (128 + pad)
constexpr int kSetRows = 8;    // weight rows per unit

__device__ __forceinline__ uint32_t lds32a(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64a(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16a(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds32f(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Four signed quants (one word) -> two exact f16 pairs: bytes (0, 1), (2, 3).
__device__ __forceinline__ void quant_pairs(uint32_t w, uint32_t& h01, uint32_t& h23) {
  const uint32_t f = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(f, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(f, 0x64646464u, 0x7362);
  const uint32_t bias = 0x64806480u;  // (1152, 1152)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(h01) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(h23) : "r"(b), "r"(bias));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Quant index of byte k of word w of a block (the order the A side reads).
__device__ __forceinline__ int word_quant(bool even_block, int w, int k) {
  if (!even_block) return 4 * w + k;
  if (w < 7) return 4 * w + 2 + k;
  return k < 2 ? k : 28 + k;
}

// The x fragment of one word: hi = f16(v), lo = f16(v - hi) for the word's
// four (already scaled) values, 16 bytes at dst.
__device__ __forceinline__ void store_x_word(uint8_t* dst, const float (&v)[4]) {
  const __half2 h01 = __floats2half2_rn(v[0], v[1]), h23 = __floats2half2_rn(v[2], v[3]);
  const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
  const __half2 l01 = __floats2half2_rn(v[0] - f01.x, v[1] - f01.y);
  const __half2 l23 = __floats2half2_rn(v[2] - f23.x, v[3] - f23.y);
  uint4 q;
  q.x = *reinterpret_cast<const uint32_t*>(&h01);
  q.y = *reinterpret_cast<const uint32_t*>(&h23);
  q.z = *reinterpret_cast<const uint32_t*>(&l01);
  q.w = *reinterpret_cast<const uint32_t*>(&l23);
  *reinterpret_cast<uint4*>(dst) = q;
}

// Per-lane constants of the unit loop (byte offsets within a pair of units:
// 8 consecutive blocks 8k .. 8k+7 of a tile row; the even unit is blocks
// 8k + {0, 2, 4, 6}, the odd unit 8k + {1, 3, 5, 7}; half 0 of a unit is
// its blocks +0 and +4, half 1 its blocks +2 and +6).
struct LaneOffs {
  uint32_t e0, e1;    // even unit, halves 0 / 1: this lane's word 2i + wsel, i < 3 (+ 8 i)
  uint32_t e3a, e3b;  // even unit, i = 3: the two words the last word comes from (half 0)
  uint32_t sel3;      // their byte selector (word 6 as is, or bytes {2,3} + {32,33})
  uint32_t o0, o1;    // odd unit, halves 0 / 1: word 2i + wsel (+ 8 i)
  uint32_t s_even;    // this lane's (row, block) scale of the even unit (odd: + 34)
};

// Block of the pair (0, 2, 4 or 6; the odd unit's is + 1) whose (row,
// block) partial lane quad position cq ends a unit with.
__device__ __forceinline__ int lane_block(int cq) { return cq < 2 ? 4 * cq : 2 + 4 * (cq - 2); }

__device__ __forceinline__ LaneOffs lane_offsets(int cq) {
  const int j = cq & 1, wsel = cq >> 1;
  LaneOffs L;
  // even blocks start on a word: words +4 .. +28 hold quants 2 .. 29, the
  // last word is quants {0, 1} (bytes 2, 3) and {30, 31} (bytes 32, 33)
  L.e0 = 136u * j + 4u + 4u * wsel;
  L.e1 = L.e0 + 68u;
  L.e3a = wsel ? 136u * j : 136u * j + 28u;
  L.e3b = 136u * j + 32u;
  L.sel3 = wsel ? 0x5432u : 0x3210u;
  // odd blocks start two bytes past a word: quants are word aligned
  L.o0 = 34u + 136u * j + 2u + 4u * wsel;
  L.o1 = L.o0 + 68u;
  L.s_even = (uint32_t)lane_block(cq) * kQBlockBytes;
  return L;
}

// The unit partials of a pair (8 rows x blocks 8k .. 8k+7) at row32 + base;
// xb: this lane's x fragments of the pair (its B block of the even unit,
// word wsel; the odd unit's are xstep bytes on; the zero pad for lanes whose
// B column is zero).  pe / po: the (row gq, block) sums of the even / odd
// unit for this lane's block (not yet scaled).
__device__ __forceinline__ void pair_units(uint32_t rb, uint32_t xb, uint32_t xstep,
                                           const LaneOffs& L, bool lo_half, float& pe, float& po) {
  float ae[4] = {0.f, 0.f, 0.f, 0.f}, ao[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t we0, we1;
    if (i < 3) {
      we0 = lds32a(rb + L.e0 + 8 * i);
      we1 = lds32a(rb + L.e1 + 8 * i);
    } else {
      we0 = __byte_perm(lds32a(rb + L.e3a), lds32a(rb + L.e3b), L.sel3);
      we1 = __byte_perm(lds32a(rb + L.e3a + 68), lds32a(rb + L.e3b + 68), L.sel3);
    }
    const uint32_t wo0 = lds32a(rb + L.o0 + 8 * i), wo1 = lds32a(rb + L.o1 + 8 * i);
    const uint2 be = lds64a(xb + 32 * i);
    const uint2 bo = lds64a(xb + xstep + 32 * i);
    uint32_t a0, a1, a2, a3;
    quant_pairs(we0, a0, a2);
    quant_pairs(we1, a1, a3);
    mma_f16(ae, a0, a1, a2, a3, be.x, be.y);
    quant_pairs(wo0, a0, a2);
    quant_pairs(wo1, a1, a3);
    mma_f16(ao, a0, a1, a2, a3, bo.x, bo.y);
  }
  // (row gq, block b_cq) of each unit: half 0 for cq < 2, half 1 otherwise
  pe = lo_half ? ae[0] + ae[1] : ae[2] + ae[3];
  po = lo_half ? ao[0] + ao[1] : ao[2] + ao[3];
}

// The f16 weight scale of this lane's (row, block) of the even unit (odd:
// the next block).
__device__ __forceinline__ float unit_scale(uint32_t rb, const LaneOffs& L, bool odd) {
  return __half2float(__ushort_as_half((unsigned short)lds16a(rb + L.s_even + (odd ? 34u : 0u))));
}

// pair_units scaled by the blocks' f16 scales and summed (one power-of-two
// scale for the whole vector, undone by the caller).
__device__ __forceinline__ float pair_dot(uint32_t rb, uint32_t xb, uint32_t xstep, const LaneOffs& L,
                                          bool lo_half) {
  float pe, po;
  pair_units(rb, xb, xstep, L, lo_half, pe, po);
  return fmaf(unit_scale(rb, L, false), pe, unit_scale(rb, L, true) * po);
}

}  // namespace tc
}  // namespace q8d
