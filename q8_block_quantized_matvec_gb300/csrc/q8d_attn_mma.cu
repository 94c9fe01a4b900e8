// Split-K decode attention over an f16 KV cache on the tensor cores.
//
// Same contract as the CUDA-core kernel in q8d_attn.cu ("IV.4: One command
// buffer per token", attention_decode; "Metal Backend Optimizations" 3.3,
// split partial + combine), organised for GB300:
//  * The G <= 16 query heads of one KV head are the 16 rows of an
//    m16n8k16 MMA; tokens are the N dimension of Q.K^T and the K dimension of
//    P.V.  With G of 2..8 a tcgen05 tile (M >= 64) would be mostly padding
//    and would move the scores out to TMEM between the two products, so the
//    warp-level MMA keeps scores, softmax and P in registers (the
//    accumulator layout of Q.K^T is the A-operand layout of P.V).
//  * f32 accuracy from f16 tensor cores: K and V are f16 already (exact);
//    q is scaled per head by a power of two into f16 range and split into
//    f16 hi + lo parts (q = hi + lo to ~2^-22), and so are the
//    probabilities (scaled by 2^12 first); every product is exact in the f32
//    accumulator, so the result matches f32 CUDA-core arithmetic.
//  * Each warp runs its own online softmax over its token groups (groups
//    w, w+4, w+8, ... of the chunk); the four warps' {m, l, O} are merged once
//    at the end of the chunk and written as the chunk's partial.
//  * Every warp streams its own 16-token groups of K/V rows through a
//    two-stage cp.async ring (16-byte copies; a KV head's row is only 128
//    or 256 bytes, too small for efficient bulk copies) and never waits for
//    the other warps until the final merge.  Two stages keep a CTA at ~70 KB
//    of shared memory, so three CTAs (12 warps) share an SM: more loads in
//    flight per SM than three stages with two CTAs.  Rows are padded by 16
//    bytes so fragment loads and ldmatrix.trans hit distinct banks.
//  * The CTAs of a KV head are split over the batch's sequences in
//    proportion to their lengths (read from device memory by every CTA,
//    q8d_attn.cuh), so a ragged batch's long sequences do not set the time.
#include <cuda_fp16.h>

#include "q8d_attn.cuh"
#include "q8d_attn_common.cuh"
#include "q8d_internal.cuh"

namespace q8d {
namespace {

constexpr int kWarpsA = 4;
constexpr int kThreadsA = kWarpsA * 32;
constexpr float kLog2eA = 1.4426950408889634f;
constexpr float kPScale = 4096.f;      // probabilities scaled by 2^12 before the f16 split

constexpr int kGroup = 16;             // tokens per warp step
constexpr int kWStages = 2;            // per-warp cp.async ring depth

template <int D>
struct MCfg {
  static constexpr int kRow = D * 2;                     // f16 row bytes
  static constexpr int kStride = kRow + 16;              // padded shared-memory row
  static constexpr int kStage = 2 * kGroup * kStride;    // 16 K rows, then 16 V rows
  static constexpr int kWarpRing = kWStages * kStage;    // one warp's ring
  static constexpr int kOffQ = kWarpsA * kWarpRing;      // f32 q [16][D], power-of-two scaled
  static constexpr int kOffF = kOffQ + 16 * D * 4;       // per-head score factor [16]
  static constexpr int kSmem = kOffF + 16 * 4;
  static_assert(kWarpsA * 16 * (D + 2) * 4 <= kOffQ, "merge buffer fits the rings");
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}




template <int D>
__global__ void __launch_bounds__(kThreadsA) gqa_mma_kernel(const AttnParams P) {
  using C = MCfg<D>;
  constexpr int KS = D / 16;  // k-steps over head_dim (Q.K^T)
  constexpr int NT = D / 8;   // n-tiles over head_dim (P.V)
  extern __shared__ __align__(128) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + C::kOffQ);
  float* fh = reinterpret_cast<float*>(smem + C::kOffF);
  __shared__ AttnWindow s_win;  // this sequence's window (row t -> cache row)

  const int g = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, cq = lane & 3;
  const int G = P.n_heads / P.n_kv_heads;
  // the combine kernel, launched as a programmatic dependent, may be
  // scheduled now (it waits for this grid's results before reading them);
  // this grid is itself a programmatic dependent of the previous work in the
  // stream: nothing is read before that work is complete
  griddep_launch_dependents();
  griddep_wait();
  int b, c, n;  // this CTA's sequence and chunk (of n): the balanced split
  if (!attn_chunk_of(P, blockIdx.x, b, c, n)) return;
  const int L = attn_window_len(P, b);
  if (L < 1) {  // (the combine writes NaN outputs)
    if (g == 0 && tid == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_LEN_RANGE);
    return;
  }
  const int tpc = (L + n - 1) / n;
  const int t_begin = c * tpc;
  if (t_begin >= L) return;
  const int t_end = min(L, t_begin + tpc);
  if (tid == 0) attn_window_store(P, b, &s_win);  // (read after the barrier before the loads)
  const long long kvw = (long long)P.n_kv_heads * D;
  __half* kbase = reinterpret_cast<__half*>(P.kcache) + (long long)b * P.batch_stride + (long long)g * D;
  __half* vbase = reinterpret_cast<__half*>(P.vcache) + (long long)b * P.batch_stride + (long long)g * D;

  // In-kernel append of row L-1 by the CTA that owns it; the copies below
  // read it back after the barrier, so attended values are the cached ones.
  const int half = D / 2;
  const float* cosr = P.rope_cos ? P.rope_cos + (long long)(L - 1) * half : nullptr;
  const float* sinr = P.rope_sin ? P.rope_sin + (long long)(L - 1) * half : nullptr;
  if (P.k_new != nullptr && t_end == L && warp < 2) {
    // warp 0: k row (bias, norm, RoPE), warp 1: v row (bias)
    const float* src = (warp == 0 ? P.k_new : P.v_new) + (long long)b * kvw + (long long)g * D;
    float v[D / 32];
#pragma unroll
    for (int t = 0; t < D / 32; ++t) v[t] = src[lane + 32 * t];
    if (warp == 0)
      head_prologue<D>(v, lane, P.bk ? P.bk + (long long)g * D : nullptr, P.k_norm, P.eps, cosr, sinr);
    else
      head_prologue<D>(v, lane, P.bv ? P.bv + (long long)g * D : nullptr, nullptr, 0.f, nullptr,
                       nullptr);
    __half* dst = (warp == 0 ? kbase : vbase) + (long long)attn_cell(P, b, L - 1) * kvw;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) dst[lane + 32 * t] = __float2half_rn(v[t]);
  }

  // Query rows scaled per head by 2^sh so that max|q| < 2^11; the score
  // factor 2^-sh * scale * log2(e) undoes it in the log2 domain.
  {
    // this warp's four query heads: loads first (all in flight), then the
    // prologue and the power-of-two scaling per head
    float v[4][D / 32];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int hh = warp + kWarpsA * u;
#pragma unroll
      for (int t = 0; t < D / 32; ++t)
        v[u][t] = (hh < G) ? P.q[((long long)b * P.n_heads + g * G + hh) * D + lane + 32 * t] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int hh = warp + kWarpsA * u;
      const int hq_ = g * G + hh;
      if (hh < G)
        head_prologue<D>(v[u], lane, P.bq ? P.bq + (long long)hq_ * D : nullptr, P.q_norm, P.eps,
                         cosr, sinr);
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
      if (lane == 0) fh[hh] = (hh < G) ? ldexpf(P.scale * kLog2eA, -sh) : 0.f;
    }
  }
  __syncthreads();  // q rows scaled; the appended row is visible to every thread
  // the window's first run in registers (a causal window is only that run)
  const int run0_len = s_win.len[0], run0_cell = s_win.cell[0];

  // ---- this warp's cp.async ring over its token groups ----
  const int ngroups = (t_end - t_begin + kGroup - 1) / kGroup;
  const int my_groups = ngroups > warp ? (ngroups - warp + kWarpsA - 1) / kWarpsA : 0;
  uint8_t* ring = smem + warp * C::kWarpRing;
  constexpr int kChunks = C::kRow / 16;       // 16-byte pieces per row
  constexpr int kRowsPass = 32 / kChunks;      // rows one pass of the 32 lanes copies
  const long long row_bytes = kvw * 2;
  auto load_group = [&](int i) {  // i-th group of this warp into stage i % kWStages
    if (i < my_groups) {
      const int t0 = t_begin + (warp + kWarpsA * i) * kGroup;
      const int nr = min(kGroup, t_end - t0);
      uint8_t* st = ring + (i % kWStages) * C::kStage;
      if (nr == kGroup && t0 + kGroup <= run0_len) {
        // 16 consecutive cache rows: one base address, fixed strides
        const int r = lane / kChunks, pc = lane % kChunks;
        const long long off = (long long)(run0_cell + t0 + r) * row_bytes + pc * 16;
        const uint8_t* ks = reinterpret_cast<const uint8_t*>(kbase) + off;
        const uint8_t* vs = reinterpret_cast<const uint8_t*>(vbase) + off;
        uint8_t* kd = st + r * C::kStride + pc * 16;
#pragma unroll
        for (int k = 0; k < kGroup / kRowsPass; ++k) {
          cp_async16(kd + k * kRowsPass * C::kStride, ks + k * kRowsPass * row_bytes);
          cp_async16(kd + (kGroup + k * kRowsPass) * C::kStride, vs + k * kRowsPass * row_bytes);
        }
        cp_async_commit();
        return;
      }
#pragma unroll
      for (int e = lane; e < kGroup * kChunks; e += 32) {
        const int r = e / kChunks, pc = e % kChunks;
        if (r < nr) {
          const long long off = (long long)(t0 + r < run0_len ? run0_cell + t0 + r : s_win.cell_of(t0 + r)) * kvw * 2 + pc * 16;
          cp_async16(st + r * C::kStride + pc * 16, reinterpret_cast<const uint8_t*>(kbase) + off);
          cp_async16(st + (kGroup + r) * C::kStride + pc * 16,
                     reinterpret_cast<const uint8_t*>(vbase) + off);
        }
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
  };
#pragma unroll
  for (int i = 0; i < kWStages - 1; ++i) load_group(i);

  // A fragments of q (rows gq and gq + 8, K = head_dim), hi and lo parts.
  uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    const int d0 = 16 * kk + 2 * cq;
    attn_split2(qs[gq * D + d0], qs[gq * D + d0 + 1], qh[kk][0], ql[kk][0]);
    attn_split2(qs[(gq + 8) * D + d0], qs[(gq + 8) * D + d0 + 1], qh[kk][1], ql[kk][1]);
    attn_split2(qs[gq * D + d0 + 8], qs[gq * D + d0 + 9], qh[kk][2], ql[kk][2]);
    attn_split2(qs[(gq + 8) * D + d0 + 8], qs[(gq + 8) * D + d0 + 9], qh[kk][3], ql[kk][3]);
  }
  const float f0 = fh[gq], f1 = fh[gq + 8];

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int i = 0; i < my_groups; ++i) {
    load_group(i + kWStages - 1);
    cp_async_wait<kWStages - 1>();
    __syncwarp();
    const int nr = min(kGroup, t_end - (t_begin + (warp + kWarpsA * i) * kGroup));
    const uint8_t* st = ring + (i % kWStages) * C::kStage;
    const int base_t = 0;

    // ---- S = Q.K^T for this warp's 16 tokens (two n-tiles of 8) ----
    // hi and lo products accumulate in separate chains (4 independent MMA
    // chains per warp) and are added at the end
    float s[2][4], sl[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
      sl[j][0] = sl[j][1] = sl[j][2] = sl[j][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = min(base_t + 8 * j + gq, nr - 1);
        const uint8_t* krow = st + tok * C::kStride + 4 * cq + 32 * kk;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + 16);
        attn_mma16816(s[j], qh[kk], b0, b1);
        attn_mma16816(sl[j], ql[kk], b0, b1);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] += sl[j][e];
    // ---- log2-domain scores, mask, online softmax per row ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = base_t + 8 * j + 2 * cq + (e & 1);
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
    const float c0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
    const float c1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
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
    if (!__all_sync(0xffffffffu, c0 == 1.f && c1 == 1.f)) {  // skipped when no row max moved
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= c0;
        o[n][1] *= c0;
        o[n][2] *= c1;
        o[n][3] *= c1;
      }
    }
    // ---- P (16 heads x 16 tokens) as the A operand, hi/lo ----
    uint32_t ph[4], pl[4];
    attn_split2(s[0][0] * kPScale, s[0][1] * kPScale, ph[0], pl[0]);
    attn_split2(s[0][2] * kPScale, s[0][3] * kPScale, ph[1], pl[1]);
    attn_split2(s[1][0] * kPScale, s[1][1] * kPScale, ph[2], pl[2]);
    attn_split2(s[1][2] * kPScale, s[1][3] * kPScale, ph[3], pl[3]);
    // ---- O += P.V ----
    {
      const int mi = lane >> 3, r = lane & 7;
      const int tok = min(base_t + (mi & 1) * 8 + r, nr - 1);
      const uint32_t vrow = smem_u32(st + (kGroup + tok) * C::kStride + (mi >> 1) * 16);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t v0, v1, v2, v3;
        attn_ldsm_x4_trans(vrow + dn * 32, v0, v1, v2, v3);
        attn_mma16816(o[2 * dn], ph, v0, v1);
        attn_mma16816(o[2 * dn], pl, v0, v1);
        attn_mma16816(o[2 * dn + 1], ph, v2, v3);
        attn_mma16816(o[2 * dn + 1], pl, v2, v3);
      }
    }
    __syncwarp();  // the stage is refilled by the next iteration's load
  }
  cp_async_wait<0>();

  // ---- merge the four warps' {m, l, O}; write the chunk's partial ----
  __syncthreads();
  float* mm = reinterpret_cast<float*>(smem);  // stages are idle now
  float* ll = mm + kWarpsA * 16;
  float* oo = ll + kWarpsA * 16;
  if (cq == 0) {
    mm[warp * 16 + gq] = m0;
    mm[warp * 16 + gq + 8] = m1;
    ll[warp * 16 + gq] = l0;
    ll[warp * 16 + gq + 8] = l1;
  }
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int col = 8 * n + 2 * cq;
    oo[(warp * 16 + gq) * D + col] = o[n][0];
    oo[(warp * 16 + gq) * D + col + 1] = o[n][1];
    oo[(warp * 16 + gq + 8) * D + col] = o[n][2];
    oo[(warp * 16 + gq + 8) * D + col + 1] = o[n][3];
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kThreadsA) {
    const int h = e / D, j = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarpsA; ++w) M = fmaxf(M, mm[w * 16 + h]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarpsA; ++w) {
      const float mw = mm[w * 16 + h];
      if (mw == -INFINITY) continue;
      const float wgt = exp2f(mw - M);
      acc = fmaf(oo[(w * 16 + h) * D + j], wgt, acc);
      lsum = fmaf(ll[w * 16 + h], wgt, lsum);
    }
    const long long hq = (long long)b * P.n_heads + (long long)g * G + h;
    P.ws_o[(hq * P.nc + c) * D + j] = acc * (1.f / kPScale);
    if (j == 0) {
      P.ws_m[hq * P.nc + c] = M;
      P.ws_l[hq * P.nc + c] = lsum;
    }
  }
}

template <int D>
int launch_mma(const AttnParams& P, cudaStream_t stream) {
  using C = MCfg<D>;
  int rc = configure_kernel(reinterpret_cast<const void*>(gqa_mma_kernel<D>), C::kSmem, false);
  if (rc) return rc;
  dim3 grid(P.nct, P.n_kv_heads);
  rc = launch_ex(gqa_mma_kernel<D>, grid, dim3(kThreadsA), (size_t)C::kSmem, stream, true, P);
  if (rc) return rc;
  return attn_combine_launch(P, stream);
}

}  // namespace

int attn_mma_launch(const AttnParams& P, cudaStream_t stream) {
  return P.head_dim == 128 ? launch_mma<128>(P, stream) : launch_mma<64>(P, stream);
}

}  // namespace q8d
