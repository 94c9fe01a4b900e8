// Split-K decode attention over a packed Q8_0 KV cache on the tensor cores.
//
// The pages' "mechanism A" ("minfer Metal Backend Design", "Execution
// dispatch": the decode kernels read the packed 34-byte blocks natively,
// partials merged by the shared combine): the same contract and split as
// the f16 kernel (q8d_attn_mma.cu) with the cache stored as Q8_0 rows, so a
// KV head's row is D/32 blocks (68 or 136 bytes instead of 128 or 256).
// GB300 organisation:
//  * CTA = (chunk slot, KV head), four warps; each warp walks its own
//    16-token groups with an online softmax, and the warps merge once.
//    The G <= 16 query heads of the KV head are the 16 rows of an
//    mma.sync m16n8k16; every K/V byte is read once for all of them.
//  * Raw blocks stream into a per-warp two-stage ring with 8-byte (head_dim
//    128) or 4-byte (head_dim 64) cp.async copies: a head's slice of a row
//    is 8- (4-) byte aligned but not 16.  Shared rows are padded to 144 (80)
//    bytes so the fragment word reads of eight rows hit distinct banks.
//  * Q.K^T: a quant is an exact f16 after one PRMT into the 0x64xx pattern
//    and one sub.f16x2 per pair.  The 16 contraction indices of a k-step
//    are permuted so that a thread's four quants of a token are one 32-bit
//    word (q, split hi + lo as in the f16 kernel, takes the same
//    permutation).  A block's two k-steps accumulate into a fresh tile
//    that is scaled by the token's f16 block scale in f32 and added to the
//    scores: the products are exact, so the result matches f32 arithmetic.
//  * P.V: the warp converts its V quants to an f16 tile (exact) and reads it
//    transposed with ldmatrix; the V block scale depends on the token (the
//    contraction index), so it is folded into P, per 32-dim block, before
//    the hi + lo split.  To keep P * scale inside f16 range for any scale,
//    every warp carries a power-of-two factor 2^fe set from the largest V
//    scale seen (P * scale * 2^fe < 2^15); when it shrinks, O is rescaled
//    exactly (with the softmax correction), and O / 2^fe is merged.
//  * The in-kernel append of row L-1 quantizes the new k and v rows with
//    the store quantizer (quantize_q8_0_warp), writes them to the cache,
//    and the chunk then reads them back like any other row.
#include <cuda_fp16.h>

#include "q8d_attn.cuh"
#include "q8d_attn_common.cuh"
#include "q8d_internal.cuh"

namespace q8d {
namespace {

constexpr int kWarpsQ = 4;
constexpr int kThreadsQ = kWarpsQ * 32;
constexpr float kLog2eQ = 1.4426950408889634f;
constexpr int kGroupQ = 16;   // tokens per warp step
constexpr int kStagesQ = 2;   // per-warp cp.async ring depth
constexpr int kFeInit = 64;   // range exponent before the first group

template <int D>
struct QCfg {
  static constexpr int kNB = D / 32;                     // blocks per head row
  static constexpr int kRowB = kNB * kQBlockBytes;       // 68 / 136 bytes
  static constexpr int kRS = D == 128 ? 144 : 80;        // padded shared row
  static constexpr int kCopy = D == 128 ? 8 : 4;         // cp.async size
  static constexpr int kPer = kRowB / kCopy;             // copies per row slice
  static constexpr int kRawStage = 2 * kGroupQ * kRS;    // 16 K rows, then 16 V rows
  static constexpr int kVStride = D * 2 + 16;            // f16 V tile row (padded)
  static constexpr int kVTile = kGroupQ * kVStride;
  static constexpr int kWarpBytes = kStagesQ * kRawStage + kVTile;
  static constexpr int kOffQ = kWarpsQ * kWarpBytes;     // f32 q [16][D]
  static constexpr int kOffF = kOffQ + 16 * D * 4;       // per-head score factor [16]
  static constexpr int kSmem = kOffF + 16 * 4;
  static_assert(kRowB % kCopy == 0, "row slice is whole copies");
  static_assert(kWarpsQ * 16 * (D + 2) * 4 <= kOffQ, "merge buffer fits the rings");
  static_assert((kRS / 4) % 32 == 4 || (kRS / 4) % 32 == 20, "conflict-free word reads");
};

template <int N>
__device__ __forceinline__ void cp_async_n(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)), "l"(src), "n"(N)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}




// Four signed quants (one word) -> two exact f16 pairs: bytes (0, 1) and
// (2, 3).  A sign-flipped byte b placed under the exponent byte 0x64 is the
// half 1024 + b = 1152 + q; one sub.f16x2 removes the 1152.
__device__ __forceinline__ void quants_to_h2(uint32_t w, uint32_t& h01, uint32_t& h23) {
  const uint32_t f = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(f, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(f, 0x64646464u, 0x7362);
  const uint32_t bias = 0x64806480u;  // (1152, 1152)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(h01) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(h23) : "r"(b), "r"(bias));
}

// The 32-bit word of quants j0..j0+3 (j0 % 4 == 0) of block `blk` of a
// shared row (the row and the head's slice are 4-byte aligned): block b of
// the slice starts at 34 b, so its quants start at a word boundary for odd
// b and two bytes past one for even b.
template <bool kEvenBlock>
__device__ __forceinline__ uint32_t quant_word(const uint8_t* blk, int j0) {
  if constexpr (kEvenBlock) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(blk + j0);
    return __byte_perm(w[0], w[1], 0x5432);
  } else {
    return *reinterpret_cast<const uint32_t*>(blk + 2 + j0);
  }
}

__device__ __forceinline__ float block_scale(const uint8_t* blk) {
  return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk)));
}

template <int D>
__global__ void __launch_bounds__(kThreadsQ) gqa_q8kv_kernel(const AttnParams P) {
  using C = QCfg<D>;
  constexpr int KS = D / 16;   // k-steps over head_dim (Q.K^T)
  constexpr int NT = D / 8;    // n-tiles over head_dim (P.V)
  constexpr int NB = C::kNB;
  extern __shared__ __align__(128) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + C::kOffQ);
  float* fh = reinterpret_cast<float*>(smem + C::kOffF);
  __shared__ AttnWindow s_win;  // this sequence's window (row t -> cache row)

  const int g = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, cq = lane & 3;
  const int G = P.n_heads / P.n_kv_heads;
  griddep_launch_dependents();  // the combine may be scheduled now
  griddep_wait();  // (a programmatic dependent: the previous work is complete)
  int b, c, n;
  if (!attn_chunk_of(P, blockIdx.x, b, c, n)) return;
  const int L = attn_window_len(P, b);
  if (L < 1) {
    if (g == 0 && tid == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_LEN_RANGE);
    return;
  }
  const int tpc = (L + n - 1) / n;
  const int t_begin = c * tpc;
  if (t_begin >= L) return;
  const int t_end = min(L, t_begin + tpc);
  if (tid == 0) attn_window_store(P, b, &s_win);  // (read after the barrier before the loads)
  const long long rowb = (long long)P.n_kv_heads * C::kRowB;  // packed cache row
  // sequence b's cache starts at its element offset b * stride, i.e. at
  // block b * stride / 32
  const long long seq_off = (long long)b * (P.batch_stride / kQBlock) * kQBlockBytes;
  uint8_t* kbase = reinterpret_cast<uint8_t*>(P.kcache) + seq_off + (long long)g * C::kRowB;
  uint8_t* vbase = reinterpret_cast<uint8_t*>(P.vcache) + seq_off + (long long)g * C::kRowB;

  // In-kernel append of row L-1 by the CTA that owns it (warp 0: k, warp 1:
  // v), quantized by the store quantizer; read back after the barrier.
  const int half = D / 2;
  const float* cosr = P.rope_cos ? P.rope_cos + (long long)(L - 1) * half : nullptr;
  const float* sinr = P.rope_sin ? P.rope_sin + (long long)(L - 1) * half : nullptr;
  if (P.k_new != nullptr && t_end == L && warp < 2) {
    // (the fused decode-step prologue, when given: k bias / norm / RoPE, v bias)
    const long long kvw = (long long)P.n_kv_heads * D;
    const float* src = (warp == 0 ? P.k_new : P.v_new) + (long long)b * kvw + (long long)g * D;
    float v[D / 32];
#pragma unroll
    for (int t = 0; t < D / 32; ++t) v[t] = src[lane + 32 * t];
    if (warp == 0)
      head_prologue<D>(v, lane, P.bk ? P.bk + (long long)g * D : nullptr, P.k_norm, P.eps, cosr, sinr);
    else
      head_prologue<D>(v, lane, P.bv ? P.bv + (long long)g * D : nullptr, nullptr, 0.f, nullptr,
                       nullptr);
    uint8_t* dst = (warp == 0 ? kbase : vbase) + (long long)attn_cell(P, b, L - 1) * rowb;
#pragma unroll
    for (int t = 0; t < NB; ++t) quantize_q8_0_warp(v[t], dst + t * kQBlockBytes, lane);
  }

  // Query rows scaled per head by 2^sh so that max|q| < 2^11; the score
  // factor 2^-sh * scale * log2(e) undoes it in the log2 domain.
  {
    float v[4][D / 32];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int hh = warp + kWarpsQ * u;
#pragma unroll
      for (int t = 0; t < D / 32; ++t)
        v[u][t] = (hh < G) ? P.q[((long long)b * P.n_heads + g * G + hh) * D + lane + 32 * t] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int hh = warp + kWarpsQ * u;
      if (hh < G)
        head_prologue<D>(v[u], lane, P.bq ? P.bq + ((long long)g * G + hh) * D : nullptr, P.q_norm,
                         P.eps, cosr, sinr);
      float mx = 0.f;
#pragma unroll
      for (int t = 0; t < D / 32; ++t) mx = fmaxf(mx, fabsf(v[u][t]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      int e = 0;
      if (mx > 0.f) frexpf(mx, &e);
      const int sh = (mx > 0.f) ? 11 - e : 0;
#pragma unroll
      for (int t = 0; t < D / 32; ++t) qs[hh * D + lane + 32 * t] = ldexpf(v[u][t], sh);
      if (lane == 0) fh[hh] = (hh < G) ? ldexpf(P.scale * kLog2eQ, -sh) : 0.f;
    }
  }
  __syncthreads();  // q rows scaled; the appended row is in the cache
  // the window's first run in registers (a causal window is only that run)
  const int run0_len = s_win.len[0], run0_cell = s_win.cell[0];

  // ---- this warp's cp.async ring over its token groups ----
  const int ngroups = (t_end - t_begin + kGroupQ - 1) / kGroupQ;
  const int my_groups = ngroups > warp ? (ngroups - warp + kWarpsQ - 1) / kWarpsQ : 0;
  uint8_t* ring = smem + warp * C::kWarpBytes;
  uint8_t* vt = ring + kStagesQ * C::kRawStage;  // this warp's f16 V tile
  auto load_group = [&](int i) {
    if (i < my_groups) {
      const int t0 = t_begin + (warp + kWarpsQ * i) * kGroupQ;
      const int nr = min(kGroupQ, t_end - t0);
      uint8_t* st = ring + (i % kStagesQ) * C::kRawStage;
      if (nr == kGroupQ && t0 + kGroupQ <= run0_len) {
        // 16 consecutive cache rows: one base address, no window lookup
        const uint8_t* ks = kbase + (long long)(run0_cell + t0) * rowb;
        const uint8_t* vs = vbase + (long long)(run0_cell + t0) * rowb;
#pragma unroll
        for (int k = 0; k < (kGroupQ * C::kPer + 31) / 32; ++k) {
          const int e = lane + 32 * k;
          if (e < kGroupQ * C::kPer) {
            const int r = e / C::kPer, pc = e % C::kPer;
            const long long off = (long long)r * rowb + pc * C::kCopy;
            cp_async_n<C::kCopy>(st + r * C::kRS + pc * C::kCopy, ks + off);
            cp_async_n<C::kCopy>(st + (kGroupQ + r) * C::kRS + pc * C::kCopy, vs + off);
          }
        }
        cp_commit();
        return;
      }
      for (int e = lane; e < kGroupQ * C::kPer; e += 32) {
        const int r = e / C::kPer, pc = e % C::kPer;
        if (r < nr) {
          const long long off = (long long)(t0 + r < run0_len ? run0_cell + t0 + r : s_win.cell_of(t0 + r)) * rowb + pc * C::kCopy;
          cp_async_n<C::kCopy>(st + r * C::kRS + pc * C::kCopy, kbase + off);
          cp_async_n<C::kCopy>(st + (kGroupQ + r) * C::kRS + pc * C::kCopy, vbase + off);
        }
      }
    }
    cp_commit();  // possibly empty: keeps the group count uniform
  };
#pragma unroll
  for (int i = 0; i < kStagesQ - 1; ++i) load_group(i);

  // A fragments of q, hi and lo parts, with the k-permutation of the quant
  // words: k slots (2cq, 2cq+1) are dims 16kk + 4cq + (0, 1), slots
  // (2cq+8, 2cq+9) dims 16kk + 4cq + (2, 3).
  uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    const int d0 = 16 * kk + 4 * cq;
    attn_split2(qs[gq * D + d0], qs[gq * D + d0 + 1], qh[kk][0], ql[kk][0]);
    attn_split2(qs[(gq + 8) * D + d0], qs[(gq + 8) * D + d0 + 1], qh[kk][1], ql[kk][1]);
    attn_split2(qs[gq * D + d0 + 2], qs[gq * D + d0 + 3], qh[kk][2], ql[kk][2]);
    attn_split2(qs[(gq + 8) * D + d0 + 2], qs[(gq + 8) * D + d0 + 3], qh[kk][3], ql[kk][3]);
  }
  const float f0 = fh[gq], f1 = fh[gq + 8];

  // the V-tile conversion: this lane's word column of every row (fixed per
  // lane, so its block parity is too)
  constexpr int kWordsRow = D / 4;
  const int vc_col = lane % kWordsRow;            // word of the row: dims 4 vc_col ..
  const int vc_blk = vc_col / 8, vc_j0 = (vc_col % 8) * 4;
  const int vc_row0 = lane / kWordsRow;           // first row; rows step by 32 / kWordsRow
  constexpr int kRowStep = 32 / kWordsRow;

  float o[NT][4];
#pragma unroll
  for (int nn = 0; nn < NT; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int fe = kFeInit;

  for (int i = 0; i < my_groups; ++i) {
    load_group(i + kStagesQ - 1);
    cp_wait<kStagesQ - 1>();
    __syncwarp();
    const int nr = min(kGroupQ, t_end - (t_begin + (warp + kWarpsQ * i) * kGroupQ));
    const uint8_t* st = ring + (i % kStagesQ) * C::kRawStage;
    const uint8_t* vraw = st + kGroupQ * C::kRS;

    // ---- V quants -> f16 tile [16 tokens][D] (exact), read by ldmatrix ----
#pragma unroll
    for (int r = vc_row0; r < kGroupQ; r += kRowStep) {
      const uint8_t* blk = vraw + r * C::kRS + vc_blk * kQBlockBytes;
      const uint32_t w = (vc_blk & 1) ? quant_word<false>(blk, vc_j0) : quant_word<true>(blk, vc_j0);
      uint32_t h01, h23;
      quants_to_h2(w, h01, h23);
      *reinterpret_cast<uint2*>(vt + r * C::kVStride + vc_col * 8) = make_uint2(h01, h23);
    }

    // ---- S = Q.K^T: per block, a fresh tile scaled by the token's scale ----
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
      float acc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = 2 * bb + h;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint8_t* blk = st + (8 * j + gq) * C::kRS + bb * kQBlockBytes;
          const uint32_t w = (bb & 1) ? quant_word<false>(blk, 16 * h + 4 * cq)
                                      : quant_word<true>(blk, 16 * h + 4 * cq);
          uint32_t b0, b1;
          quants_to_h2(w, b0, b1);
          attn_mma16816(acc[j], qh[kk], b0, b1);
          attn_mma16816(acc[j], ql[kk], b0, b1);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t0 = 8 * j + 2 * cq;
        const float sa = block_scale(st + t0 * C::kRS + bb * kQBlockBytes);
        const float sb = block_scale(st + (t0 + 1) * C::kRS + bb * kQBlockBytes);
        s[j][0] = fmaf(sa, acc[j][0], s[j][0]);
        s[j][1] = fmaf(sb, acc[j][1], s[j][1]);
        s[j][2] = fmaf(sa, acc[j][2], s[j][2]);
        s[j][3] = fmaf(sb, acc[j][3], s[j][3]);
      }
    }
    // ---- log2-domain scores, mask, online softmax per row ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 8 * j + 2 * cq + (e & 1);
        const float v = s[j][e] * (e < 2 ? f0 : f1);
        s[j][e] = tok < nr ? v : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
      mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
    }
#pragma unroll
    for (int o_ = 1; o_ < 4; o_ <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    float c0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
    float c1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mrow = e < 2 ? mn0 : mn1;
        const float pv = (s[j][e] == -INFINITY) ? 0.f : exp2f(s[j][e] - mrow);
        s[j][e] = pv;
        if (e < 2) rs0 += pv; else rs1 += pv;
      }
    }
#pragma unroll
    for (int o_ = 1; o_ < 4; o_ <<= 1) {
      rs0 += __shfl_xor_sync(0xffffffffu, rs0, o_);
      rs1 += __shfl_xor_sync(0xffffffffu, rs1, o_);
    }
    l0 = l0 * c0 + rs0;
    l1 = l1 * c1 + rs1;
    m0 = mn0;
    m1 = mn1;

    // ---- V scales of this thread's four tokens (0 past the group's rows),
    // the range factor 2^fe: P * scale * 2^fe < 2^15 for every scale seen ----
    const int tk[4] = {2 * cq, 2 * cq + 1, 2 * cq + 8, 2 * cq + 9};
    float sv[NB][4];
    float vmax = 0.f;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float x = tk[u] < nr ? block_scale(vraw + tk[u] * C::kRS + bb * kQBlockBytes) : 0.f;
        sv[bb][u] = x;
        vmax = fmaxf(vmax, fabsf(x));
      }
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o_));
    if (vmax > 0.f) {
      int ev = 0;
      frexpf(vmax, &ev);  // vmax < 2^ev
      const int fe_new = min(fe, 15 - ev);
      if (fe_new < fe) {
        const float r = ldexpf(1.f, fe_new - fe);  // exact power of two (0 from the initial 2^64)
        c0 *= r;
        c1 *= r;
        fe = fe_new;
      }
    }
    if (!__all_sync(0xffffffffu, c0 == 1.f && c1 == 1.f)) {
#pragma unroll
      for (int nn = 0; nn < NT; ++nn) {
        o[nn][0] *= c0;
        o[nn][1] *= c0;
        o[nn][2] *= c1;
        o[nn][3] *= c1;
      }
    }
    __syncwarp();  // the V tile is complete
    // ---- O += (P * Vscale) . Vq, per 32-dim block ----
    const float F = ldexpf(1.f, fe);
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t vrow = smem_u32(vt + ((mi & 1) * 8 + rr) * C::kVStride + (mi >> 1) * 16);
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
      const float a0 = sv[bb][0] * F, a1 = sv[bb][1] * F, a2 = sv[bb][2] * F, a3 = sv[bb][3] * F;
      uint32_t ph[4], pl[4];
      attn_split2(s[0][0] * a0, s[0][1] * a1, ph[0], pl[0]);
      attn_split2(s[0][2] * a0, s[0][3] * a1, ph[1], pl[1]);
      attn_split2(s[1][0] * a2, s[1][1] * a3, ph[2], pl[2]);
      attn_split2(s[1][2] * a2, s[1][3] * a3, ph[3], pl[3]);
#pragma unroll
      for (int dd = 0; dd < 2; ++dd) {
        const int dn = 2 * bb + dd;  // 16 dims
        uint32_t v0, v1, v2, v3;
        attn_ldsm_x4_trans(vrow + dn * 32, v0, v1, v2, v3);
        attn_mma16816(o[2 * dn], ph, v0, v1);
        attn_mma16816(o[2 * dn], pl, v0, v1);
        attn_mma16816(o[2 * dn + 1], ph, v2, v3);
        attn_mma16816(o[2 * dn + 1], pl, v2, v3);
      }
    }
    __syncwarp();  // the stage and the V tile are rewritten next
  }
  cp_wait<0>();

  // ---- merge the four warps' {m, l, O / 2^fe}; write the chunk's partial ----
  __syncthreads();
  const float inv_f = fe == kFeInit ? 0.f : ldexpf(1.f, -fe);  // (no group: O is zero)
  float* mm = reinterpret_cast<float*>(smem);
  float* ll = mm + kWarpsQ * 16;
  float* oo = ll + kWarpsQ * 16;
  if (cq == 0) {
    mm[warp * 16 + gq] = m0;
    mm[warp * 16 + gq + 8] = m1;
    ll[warp * 16 + gq] = l0;
    ll[warp * 16 + gq + 8] = l1;
  }
#pragma unroll
  for (int nn = 0; nn < NT; ++nn) {
    const int col = 8 * nn + 2 * cq;
    oo[(warp * 16 + gq) * D + col] = o[nn][0] * inv_f;
    oo[(warp * 16 + gq) * D + col + 1] = o[nn][1] * inv_f;
    oo[(warp * 16 + gq + 8) * D + col] = o[nn][2] * inv_f;
    oo[(warp * 16 + gq + 8) * D + col + 1] = o[nn][3] * inv_f;
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kThreadsQ) {
    const int h = e / D, j = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarpsQ; ++w) M = fmaxf(M, mm[w * 16 + h]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarpsQ; ++w) {
      const float mw = mm[w * 16 + h];
      if (mw == -INFINITY) continue;
      const float wgt = exp2f(mw - M);
      acc = fmaf(oo[(w * 16 + h) * D + j], wgt, acc);
      lsum = fmaf(ll[w * 16 + h], wgt, lsum);
    }
    const long long hq = (long long)b * P.n_heads + (long long)g * G + h;
    P.ws_o[(hq * P.nc + c) * D + j] = acc;
    if (j == 0) {
      P.ws_m[hq * P.nc + c] = M;
      P.ws_l[hq * P.nc + c] = lsum;
    }
  }
}

template <int D>
int launch_q8kv(const AttnParams& P, cudaStream_t stream) {
  using C = QCfg<D>;
  int rc = configure_kernel(reinterpret_cast<const void*>(gqa_q8kv_kernel<D>), C::kSmem, false);
  if (rc) return rc;
  dim3 grid(P.nct, P.n_kv_heads);
  rc = launch_ex(gqa_q8kv_kernel<D>, grid, dim3(kThreadsQ), (size_t)C::kSmem, stream, true, P);
  if (rc) return rc;
  return attn_combine_launch(P, stream);
}

}  // namespace

int attn_q8kv_launch(const AttnParams& P, cudaStream_t stream) {
  return P.head_dim == 128 ? launch_q8kv<128>(P, stream) : launch_q8kv<64>(P, stream);
}

}  // namespace q8d
