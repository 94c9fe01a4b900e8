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
//    f16 after the block's own power-of-two scale (its max |x| into
//    [2^14, 2^15); the inverse scale is applied with the weight scale), so
//    every product is exact in f32; columns that pair a row half with the
//    other half's blocks are zero.  A word's fragment is 16 bytes {hi(k0,k1),
//    hi(k2,k3), lo(k0,k1), lo(k2,k3)} in the permuted byte order
//    (word_quant); the fragments of a pair of 8 blocks (1 KB) are stored in
//    the order the lanes read them (x_word_offset), so the 16 lanes with a
//    nonzero B column read 128 contiguous bytes per load: no bank conflicts
//    and no padding.  The zero columns read a 512-byte zero pad.
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

constexpr int kXfBlock = 128;  // x fragment bytes per block
constexpr int kXfPair = 1024;  // ... per pair of 8 blocks
constexpr int kZeroPad = 512;  // zero bytes the zero B columns read
constexpr int kSetRows = 8;    // weight rows per unit

// Byte offset of word w of block bb in the fragments: pair k = bb / 8; in
// the pair, unit u = bb % 2 (even / odd blocks), step i = w / 2 of the unit
// loop, block q = (bb % 8) / 2 of the unit, word w % 2 of the step.
__host__ __device__ __forceinline__ uint32_t x_word_offset(int bb, int w) {
  const int j = bb & 7;
  return (uint32_t)((bb >> 3) * kXfPair + (j & 1) * 512 + (w >> 1) * 128 + (j >> 1) * 32 +
                    (w & 1) * 16);
}

// This lane's B operand in a pair: its column n = gq = 4 h + 2 jb + hl is
// block 2 h + 4 jb of a unit (q = h + 2 jb), hi or lo (hl); it is nonzero
// when that block is the one the lane's contraction words belong to
// (jb == cq & 1).  off: the lane's offset in a pair's fragments (even unit;
// the odd unit's is step bytes on); zero columns read the pad.
struct XLane {
  uint32_t off, step;
  bool match;
};
__device__ __forceinline__ XLane x_lane(int lane) {
  const int gq = lane >> 2, cq = lane & 3;
  const int bh = gq >> 2, bjb = (gq >> 1) & 1, bhl = gq & 1;
  XLane X;
  X.match = bjb == (cq & 1);
  X.off = X.match ? (uint32_t)((bh + 2 * bjb) * 32 + (cq >> 1) * 16 + bhl * 8) : 0u;
  X.step = X.match ? 512u : 0u;
  return X;
}

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

// The 4 values of word w of block bb (in word_quant order) from v + 32 bb.
// kMode 0: L2 loads (values other CTAs wrote in this kernel), 1: read-only
// global loads, 2: shared memory.
template <int kMode>
__device__ __forceinline__ void load_word(const float* v, int bb, int w, float (&o)[4]) {
  const float* b = v + (size_t)bb * kQBlock;
  auto ld2 = [](const float* p) {
    const float2* q = reinterpret_cast<const float2*>(p);
    return kMode == 0 ? __ldcg(q) : kMode == 1 ? __ldg(q) : *q;
  };
  if (bb & 1) {
    const float4* q = reinterpret_cast<const float4*>(b + 4 * w);
    const float4 a = kMode == 0 ? __ldcg(q) : kMode == 1 ? __ldg(q) : *q;
    o[0] = a.x;
    o[1] = a.y;
    o[2] = a.z;
    o[3] = a.w;
  } else {
    const float2 a = ld2(b + (w < 7 ? 4 * w + 2 : 0));
    const float2 c = ld2(b + (w < 7 ? 4 * w + 4 : 30));
    o[0] = a.x;
    o[1] = a.y;
    o[2] = c.x;
    o[3] = c.y;
  }
}

// Fragment of (block, word) item `it` (block it >> 3, word it & 7) of the
// values v, with the block's own power-of-two scale: the 8 lanes it & ~7 ..
// it | 7 (consecutive lanes of one warp, all calling) share the block's
// max |x| m, and m * 2^e lies in [2^14, 2^15) (e >= -113 for any finite
// m; e <= 125 keeps 2^e and 2^-e normal floats, so blocks below 2^-110
// scale to less).  The word goes to xf + x_word_offset(block, word); the
// block's inverse scale 2^-e to xinv[block].  live: the item exists.
__device__ __forceinline__ void build_x_word(int it, bool live, const float (&v)[4], uint8_t* xf,
                                             float* xinv) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  int ex = 0;
  if (m > 0.f) frexpf(m, &ex);
  const int e = m > 0.f ? min(125, 15 - ex) : 0;
  if (live) {
    const float sc = __int_as_float((127 + e) << 23);
    float t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = v[j] * sc;
    store_x_word(xf + x_word_offset(it >> 3, it & 7), t);
    if ((it & 7) == 0) xinv[it >> 3] = __int_as_float((127 - e) << 23);
  }
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
// xb: this lane's x fragments of the pair (pair base + XLane::off, or the
// zero pad), xstep: XLane::step.  pe / po: the (row gq, block) sums of the
// even / odd unit for this lane's block (not yet scaled).
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
    const uint2 be = lds64a(xb + 128 * i);
    const uint2 bo = lds64a(xb + xstep + 128 * i);
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

// pair_units scaled by the blocks' f16 weight scales and the x blocks'
// inverse scales (xi: this lane's even-unit block's entry of xinv; the odd
// unit's is the next) and summed.
__device__ __forceinline__ float pair_dot(uint32_t rb, uint32_t xb, uint32_t xstep, const LaneOffs& L,
                                          bool lo_half, uint32_t xi) {
  float pe, po;
  pair_units(rb, xb, xstep, L, lo_half, pe, po);
  const float se = unit_scale(rb, L, false) * lds32f(xi);
  const float so = unit_scale(rb, L, true) * lds32f(xi + 4u);
  return fmaf(se, pe, so * po);
}

// pair_dot for MR activation rows sharing every decoded A fragment: xb[r]
// and xi[r] are row r's fragment address and inverse-scale entry (as for
// pair_dot); the weight decode is done once, each row adds two fragment
// loads and two MMAs per step.  y[r] += row r's scaled sum.
template <int MR>
__device__ __forceinline__ void pair_dot_m(uint32_t rb, const uint32_t (&xb)[MR], uint32_t xstep,
                                           const LaneOffs& L, bool lo_half,
                                           const uint32_t (&xi)[MR], float (&y)[MR]) {
  float ae[MR][4], ao[MR][4];
#pragma unroll
  for (int r = 0; r < MR; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k) ae[r][k] = ao[r][k] = 0.f;
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
    uint32_t a0, a1, a2, a3;
    quant_pairs(we0, a0, a2);
    quant_pairs(we1, a1, a3);
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      const uint2 be = lds64a(xb[r] + 128 * i);
      mma_f16(ae[r], a0, a1, a2, a3, be.x, be.y);
    }
    quant_pairs(wo0, a0, a2);
    quant_pairs(wo1, a1, a3);
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      const uint2 bo = lds64a(xb[r] + xstep + 128 * i);
      mma_f16(ao[r], a0, a1, a2, a3, bo.x, bo.y);
    }
  }
  const float we = unit_scale(rb, L, false), wo = unit_scale(rb, L, true);
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    const float pe = lo_half ? ae[r][0] + ae[r][1] : ae[r][2] + ae[r][3];
    const float po = lo_half ? ao[r][0] + ao[r][1] : ao[r][2] + ao[r][3];
    y[r] += fmaf(we * lds32f(xi[r]), pe, wo * lds32f(xi[r] + 4u) * po);
  }
}

// Bank-spread row groups of an 8-row set (rows of a whole number of 8-block
// pairs, m = pairs a row): a 272-byte pair column is 68 words, so row gq's
// words sit 4 * (m * gq mod 8) banks after row 0's, and rows whose m * gq
// agree mod 8 would share banks.  A set is therefore gcd(m, 8) groups of
// 8 / gcd(m, 8) consecutive rows (one copy each), every group 16 bytes
// (4 banks) after the previous group's end; returns log2 of the group size.
__host__ __device__ __forceinline__ int row_group_shift(int m) {
  return (m & 1) ? 3 : (m & 3) ? 2 : (m & 7) ? 1 : 0;
}

}  // namespace tc
}  // namespace q8d
