// KV append and grouped-query decode attention with split-K (sm_103a).
//
// Semantics ("IV.4: One command buffer per token", "Eight kernels":
// append_kv and attention_decode): query head h attends with KV head
// h / (H/Hk) over the first L cached rows; softmax(scale * q.K) weights V.
//
// Design for GB300 (the pages' kernel keeps one threadgroup per query head
// and the whole score row in 16 KB of threadgroup memory, capped at 4096
// positions; "Metal Backend Optimizations" 3.3 replaces it with a split
// pass plus a combine):
//  * One CTA per (sequence, KV head, context chunk).  It serves all G query
//    heads of its KV head, so each K/V byte is read from HBM exactly once.
//  * The chunk layout is derived on the device from the length in device
//    memory (chunk = max(128, ceil(L / NC)) rows, NC fixed at launch), so a
//    captured graph replays at any length; CTAs past the last chunk exit.
//  * K/V rows (one KV head's head_dim slice: 128-256 bytes) stream into a
//    two-stage shared-memory ring with 1-D cp.async.bulk copies completing
//    on an mbarrier; K rows are padded by 16 bytes so the per-token score
//    loop reads shared memory without bank conflicts.
//  * Online softmax in the log2 domain (scores pre-scaled by log2 e), packed
//    f32x2 FMAs for P.V, partials {m, l, O} per (query head, chunk) in the
//    workspace; a second kernel merges them in chunk order (deterministic).
//  * The append of row L-1 happens inside the CTA owning that row: it writes
//    the rounded row to the cache, fences the async proxy and then streams
//    it like any other row, so the attended values are exactly the cached.
#include <algorithm>
#include <cmath>

#include "q8d_attn.cuh"
#include "q8d_attn_common.cuh"
#include "q8d_internal.cuh"

namespace q8d {

namespace {

constexpr int kAttnThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

template <typename KT>
__device__ __forceinline__ KT to_cache(float v);
template <>
__device__ __forceinline__ __half to_cache<__half>(float v) {
  return __float2half_rn(v);
}
template <>
__device__ __forceinline__ float to_cache<float>(float v) {
  return v;
}

// Converts 16 bytes of cache elements into floats.
template <typename KT>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const void* p, float (&f)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  }
};

template <int D, typename KT, int GMAX>
struct AttnCfg {
  static constexpr int kRowBytes = D * (int)sizeof(KT);
  static constexpr int kTS = 16384 / kRowBytes;            // tokens per sub-tile
  static constexpr int kKStride = kRowBytes + 16;          // padded K row
  static constexpr int kTPT = kAttnThreads / kTS;          // threads per token (scores)
  static constexpr int kEPT = D / kTPT;                    // elements per thread (scores)
  static constexpr int kPairs = D / 2;                     // output column pairs
  static constexpr int kTG = kAttnThreads / kPairs;        // token groups (P.V)
  static constexpr int kStageBytes = kTS * kKStride + kTS * kRowBytes;
  // shared memory carve-up (bytes)
  static constexpr int kOffStage = 0;
  static constexpr int kOffQ = kOffStage + 2 * kStageBytes;
  static constexpr int kOffS = kOffQ + GMAX * D * 4;              // scores [TPT][TS][GMAX]
  static constexpr int kOffMisc = kOffS + kTPT * kTS * GMAX * 4;  // m, l, corr [3][GMAX]
  static constexpr int kOffBar = kOffMisc + 3 * GMAX * 4;
  static constexpr int kSmem = kOffBar + 2 * 8;
  static_assert(kTS * kTPT == kAttnThreads, "token mapping");
  static_assert(kPairs * kTG == kAttnThreads, "column mapping");
  static_assert((kTG * GMAX * D * 4) <= 2 * kStageBytes, "reduction buffer fits the stages");
};

template <int D, typename KT, int GMAX>
__global__ void __launch_bounds__(kAttnThreads) gqa_split_kernel(const AttnParams P) {
  using C = AttnCfg<D, KT, GMAX>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + C::kOffQ);
  float* sp = reinterpret_cast<float*>(smem + C::kOffS);
  float* m_run = reinterpret_cast<float*>(smem + C::kOffMisc);
  float* l_run = m_run + GMAX;
  float* corr = l_run + GMAX;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  __shared__ AttnWindow s_win;  // this sequence's window (row t -> cache row)

  const int g = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  KT* kbase = reinterpret_cast<KT*>(P.kcache) + (long long)b * P.batch_stride + (long long)g * D;
  KT* vbase = reinterpret_cast<KT*>(P.vcache) + (long long)b * P.batch_stride + (long long)g * D;

  // In-kernel append of row L-1 by the CTA that owns it (warp 0 the k row
  // with its bias / norm / RoPE prologue, warp 1 the v row with its bias).
  const int half = D / 2;
  const float* cosr = P.rope_cos ? P.rope_cos + (long long)(L - 1) * half : nullptr;
  const float* sinr = P.rope_sin ? P.rope_sin + (long long)(L - 1) * half : nullptr;
  if (P.k_new != nullptr && t_end == L && warp < 2) {
    const float* src = (warp == 0 ? P.k_new : P.v_new) + (long long)b * kvw + (long long)g * D;
    float v[D / 32];
#pragma unroll
    for (int t = 0; t < D / 32; ++t) v[t] = src[lane + 32 * t];
    if (warp == 0)
      head_prologue<D>(v, lane, P.bk ? P.bk + (long long)g * D : nullptr, P.k_norm, P.eps, cosr, sinr);
    else
      head_prologue<D>(v, lane, P.bv ? P.bv + (long long)g * D : nullptr, nullptr, 0.f, nullptr,
                       nullptr);
    KT* dst = (warp == 0 ? kbase : vbase) + (long long)attn_cell(P, b, L - 1) * kvw;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) dst[lane + 32 * t] = to_cache<KT>(v[t]);
    fence_proxy_async_global();
  }

  // Query rows of the group (with the step prologue), scaled into the log2 domain.
  const float qscale = P.scale * kLog2e;
  for (int hh = warp; hh < G; hh += kAttnThreads / 32) {
    const int hq_ = g * G + hh;
    float v[D / 32];
#pragma unroll
    for (int t = 0; t < D / 32; ++t) v[t] = P.q[((long long)b * P.n_heads + hq_) * D + lane + 32 * t];
    head_prologue<D>(v, lane, P.bq ? P.bq + (long long)hq_ * D : nullptr, P.q_norm, P.eps, cosr,
                     sinr);
#pragma unroll
    for (int t = 0; t < D / 32; ++t) qs[hh * D + lane + 32 * t] = v[t] * qscale;
  }
  if (tid < GMAX) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
  }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t pol = policy_evict_first();
  const int n_sub = (t_end - t_begin + C::kTS - 1) / C::kTS;
  // the window's first run in registers (a causal window is only that run)
  const int run0_len = s_win.len[0], run0_cell = s_win.cell[0];
  auto issue = [&](int k) {  // warp 0 only
    if (k >= n_sub) return;
    const int r0 = t_begin + k * C::kTS;
    const int nr = min(C::kTS, t_end - r0);
    uint8_t* st = smem + C::kOffStage + (k & 1) * C::kStageBytes;
    if (lane == 0) mbar_arrive_expect_tx(&bar[k & 1], (uint32_t)(2 * nr * C::kRowBytes));
    __syncwarp();
    for (int r = lane; r < nr; r += 32) {
      const long long row = (long long)(r0 + r < run0_len ? run0_cell + r0 + r : s_win.cell_of(r0 + r)) * kvw;
      bulk_g2s(st + r * C::kKStride, kbase + row, C::kRowBytes, &bar[k & 1], pol);
      bulk_g2s(st + C::kTS * C::kKStride + r * C::kRowBytes, vbase + row, C::kRowBytes,
               &bar[k & 1], pol);
    }
  };
  if (warp == 0) {
    issue(0);
    issue(1);
  }

  // P.V accumulators: column pair `pair`, tokens t % kTG == tg.
  const int pair = tid % C::kPairs, tg = tid / C::kPairs;
  uint64_t acc2[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) acc2[h] = pack2(0.f, 0.f);

  // Score mapping: token st_tok of the sub-tile, element slice st_part.
  // Slices are spread over warps (st_part uniform within a warp) so that the
  // K reads of a quarter-warp hit distinct banks and the q reads broadcast.
  const int st_tok = tid % C::kTS, st_part = tid / C::kTS;

  for (int k = 0; k < n_sub; ++k) {
    const int r0 = t_begin + k * C::kTS;
    const int nr = min(C::kTS, t_end - r0);
    const bool ok = mbar_wait(&bar[k & 1], (uint32_t)(k >> 1) & 1u);
    if (!__syncthreads_and(ok)) {
      if (tid == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
      return;
    }
    const uint8_t* st = smem + C::kOffStage + (k & 1) * C::kStageBytes;

    // ---- partial scores s[part][t][h] = q_h . K_t over one slice (log2 domain) ----
    {
      float acc[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) acc[h] = 0.f;
      const uint8_t* krow = st + st_tok * C::kKStride + st_part * C::kEPT * (int)sizeof(KT);
      const float* qp = qs + st_part * C::kEPT;
#pragma unroll 2
      for (int e = 0; e < C::kEPT; e += Vec16<KT>::N) {
        float kf[Vec16<KT>::N];
        Vec16<KT>::load(krow + e * sizeof(KT), kf);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          if (h < G) {
#pragma unroll
            for (int u = 0; u < Vec16<KT>::N; u += 4) {
              const float4 qv = *reinterpret_cast<const float4*>(qp + h * D + e + u);
              acc[h] = fmaf(qv.x, kf[u], acc[h]);
              acc[h] = fmaf(qv.y, kf[u + 1], acc[h]);
              acc[h] = fmaf(qv.z, kf[u + 2], acc[h]);
              acc[h] = fmaf(qv.w, kf[u + 3], acc[h]);
            }
          }
        }
      }
      float* spp = sp + (st_part * C::kTS + st_tok) * GMAX;
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) spp[h] = acc[h];
    }
    __syncthreads();

    // ---- online softmax update, one warp per head ----
    for (int h = warp; h < G; h += kAttnThreads / 32) {
      // total score of token t: the kTPT slice partials, added in slice order
      float mx = -INFINITY;
      for (int t = lane; t < nr; t += 32) {
        float sc = sp[t * GMAX + h];
#pragma unroll
        for (int q = 1; q < C::kTPT; ++q) sc += sp[(q * C::kTS + t) * GMAX + h];
        sp[t * GMAX + h] = sc;
        mx = fmaxf(mx, sc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = m_run[h];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (int t = lane; t < C::kTS; t += 32) {
        const float pt = (t < nr) ? exp2f(sp[t * GMAX + h] - m_new) : 0.f;
        sp[t * GMAX + h] = pt;
        sum += pt;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float cf = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
        corr[h] = cf;
        l_run[h] = l_run[h] * cf + sum;
        m_run[h] = m_new;
      }
    }
    __syncthreads();

    // ---- O_h = corr_h * O_h + sum_t p[t][h] * V_t ----
    {
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) acc2[h] = fma2(acc2[h], pack2(corr[h], corr[h]), pack2(0.f, 0.f));
      const uint8_t* vt = st + C::kTS * C::kKStride;
      for (int t = tg; t < nr; t += C::kTG) {
        float v0, v1;
        if constexpr (sizeof(KT) == 2) {
          const float2 f = __half22float2(
              *reinterpret_cast<const __half2*>(vt + t * C::kRowBytes + pair * 4));
          v0 = f.x;
          v1 = f.y;
        } else {
          const float2 f = *reinterpret_cast<const float2*>(vt + t * C::kRowBytes + pair * 8);
          v0 = f.x;
          v1 = f.y;
        }
        const uint64_t v2 = pack2(v0, v1);
        const float* pr = sp + t * GMAX;
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
          if (h < G) acc2[h] = fma2(v2, pack2(pr[h], pr[h]), acc2[h]);
      }
    }
    __syncthreads();
    if (warp == 0) issue(k + 2);
  }

  // ---- reduce token groups, write the partial {m, l, O} ----
  float* red = reinterpret_cast<float*>(smem + C::kOffStage);  // stages are idle now
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    if (h < G) {
      float lo, hi;
      unpack2(acc2[h], lo, hi);
      red[(tg * GMAX + h) * D + 2 * pair] = lo;
      red[(tg * GMAX + h) * D + 2 * pair + 1] = hi;
    }
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kAttnThreads) {
    const int h = e / D, j = e % D;
    float s = 0.f;
    for (int q = 0; q < C::kTG; ++q) s += red[(q * GMAX + h) * D + j];
    const long long hq = (long long)b * P.n_heads + (long long)g * G + h;
    P.ws_o[(hq * P.nc + c) * D + j] = s;
    if (j == 0) {
      P.ws_m[hq * P.nc + c] = m_run[h];
      P.ws_l[hq * P.nc + c] = l_run[h];
    }
  }
}

// Merges the chunk partials of one (sequence, query head):
//   M = max_c m_c,  w_c = 2^(m_c - M),  out = sum_c w_c O_c / sum_c w_c l_c
// kCombGroups groups of D threads (thread j of a group: output element j)
// take every kCombGroups-th chunk; each thread issues all loads of its
// chunks before using any (one L2 round trip, up to kCombLoads chunks per
// pass), merges them, and the groups' {m, l, o} are merged in group order
// through shared memory.  Fixed order throughout: deterministic.
constexpr int kCombGroups = 4;
constexpr int kCombLoads = 8;

template <int D>
__global__ void __launch_bounds__(kCombGroups * D) gqa_combine_kernel(const AttnParams P) {
  __shared__ float gm[kCombGroups], gl[kCombGroups];
  __shared__ float go[kCombGroups][D];
  const int hq = blockIdx.x;  // b * H + h
  const int b = hq / P.n_heads;
  const int j = threadIdx.x % D, grp = threadIdx.x / D;
  griddep_wait();  // the partials of the attention grid are complete and visible
  // the next kernel may be scheduled now (it waits for this grid before it
  // reads anything); not earlier, so that launches do not run ahead of the
  // work in flight and take its SMs
  griddep_launch_dependents();
  const int L = attn_window_len(P, b);
  float* o = P.out + (long long)hq * D;
  if (L < 1) {
    if (grp == 0) o[j] = __int_as_float(0x7fc00000);
    return;
  }
  // the kernels' split of this sequence (chunks past the rows are unused)
  const int n = attn_nchunks(P, L, attn_total_rows(P));
  const int tpc = (L + n - 1) / n;
  const int nact = (L + tpc - 1) / tpc;
  const float* M = P.ws_m + (long long)hq * P.nc;
  const float* S = P.ws_l + (long long)hq * P.nc;
  const float* O = P.ws_o + (long long)hq * P.nc * D + j;
  float m = -INFINITY, l = 0.f, acc = 0.f;
  for (int c0 = grp; c0 < nact; c0 += kCombGroups * kCombLoads) {
    float mc[kCombLoads], sc[kCombLoads], oc[kCombLoads];
#pragma unroll
    for (int u = 0; u < kCombLoads; ++u) {
      const int c = c0 + u * kCombGroups;
      const bool ok = c < nact;
      mc[u] = ok ? __ldcg(M + c) : -INFINITY;
      sc[u] = ok ? __ldcg(S + c) : 0.f;
      oc[u] = ok ? __ldcg(O + (long long)c * D) : 0.f;
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < kCombLoads; ++u) mn = fmaxf(mn, mc[u]);
    if (mn == -INFINITY) continue;
    const float r = exp2f(m - mn);  // 0 when m was -inf
    l *= r;
    acc *= r;
#pragma unroll
    for (int u = 0; u < kCombLoads; ++u) {
      const float w = mc[u] == -INFINITY ? 0.f : exp2f(mc[u] - mn);
      l = fmaf(sc[u], w, l);
      acc = fmaf(oc[u], w, acc);
    }
    m = mn;
  }
  if (j == 0) {
    gm[grp] = m;
    gl[grp] = l;
  }
  go[grp][j] = acc;
  __syncthreads();
  if (grp != 0) return;
  float mx = -INFINITY;
#pragma unroll
  for (int g = 0; g < kCombGroups; ++g) mx = fmaxf(mx, gm[g]);
  float lt = 0.f, at = 0.f;
#pragma unroll
  for (int g = 0; g < kCombGroups; ++g) {
    if (gm[g] == -INFINITY) continue;
    const float w = exp2f(gm[g] - mx);
    lt = fmaf(gl[g], w, lt);
    at = fmaf(go[g][j], w, at);
  }
  o[j] = at / lt;
}

template <typename KT>
__global__ void kv_append_kernel(const float* k, const float* v, KT* kc, KT* vc, int kvw, int cap,
                                 const int* d_pos, int* d_err) {
  const int pos = *d_pos;
  if (pos < 0 || pos >= cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && d_err) atomicOr(d_err, Q8D_DERR_POS_RANGE);
    return;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < kvw; i += gridDim.x * blockDim.x) {
    kc[(long long)pos * kvw + i] = to_cache<KT>(k[i]);
    vc[(long long)pos * kvw + i] = to_cache<KT>(v[i]);
  }
}

// Packed Q8_0 store: one warp per 32-element block, the k blocks then the
// v blocks of the row.
__global__ void kv_append_q8_kernel(const float* k, const float* v, uint8_t* kc, uint8_t* vc,
                                    int kvw, int cap, const int* d_pos, int* d_err) {
  const int pos = *d_pos;
  if (pos < 0 || pos >= cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && d_err) atomicOr(d_err, Q8D_DERR_POS_RANGE);
    return;
  }
  const int nb = kvw / kQBlock, lane = threadIdx.x & 31;
  const long long rowb = (long long)nb * kQBlockBytes;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < 2 * nb; w += nwarps) {
    const bool isv = w >= nb;
    const int b = isv ? w - nb : w;
    const float x = (isv ? v : k)[b * kQBlock + lane];
    quantize_q8_0_warp(x, (isv ? vc : kc) + (long long)pos * rowb + (long long)b * kQBlockBytes,
                       lane);
  }
}

template <int D, typename KT, int GMAX>
int launch_attn_t(const AttnParams& P, cudaStream_t stream) {
  using C = AttnCfg<D, KT, GMAX>;
  auto fn = gqa_split_kernel<D, KT, GMAX>;
  int rc = configure_kernel(reinterpret_cast<const void*>(fn), C::kSmem, false);
  if (rc) return rc;
  dim3 grid(P.nct, P.n_kv_heads);
  rc = launch_ex(fn, grid, dim3(kAttnThreads), (size_t)C::kSmem, stream, true, P);
  if (rc) return rc;
  return attn_combine_launch(P, stream);
}

template <int D, typename KT>
int launch_attn_g(const AttnParams& P, cudaStream_t stream) {
  const int G = P.n_heads / P.n_kv_heads;
  if (G <= 2) return launch_attn_t<D, KT, 2>(P, stream);
  if (G <= 4) return launch_attn_t<D, KT, 4>(P, stream);
  if (G <= 8) return launch_attn_t<D, KT, 8>(P, stream);
  return launch_attn_t<D, KT, 16>(P, stream);
}

}  // namespace

int attn_combine_launch(const AttnParams& P, cudaStream_t stream) {
  // a programmatic dependent of the attention grid: its launch overlaps
  // that grid's tail
  const dim3 grid((unsigned)(P.batch * P.n_heads));
  if (P.head_dim == 128)
    return launch_ex(gqa_combine_kernel<128>, grid, dim3(kCombGroups * 128), 0, stream, true, P);
  return launch_ex(gqa_combine_kernel<64>, grid, dim3(kCombGroups * 64), 0, stream, true, P);
}

int attn_ctas_per_head(int batch, int n_kv_heads, int max_len) {
  // two per SM in all: one wave at the f16 kernel's two resident CTAs per SM
  const int per_head = (2 * sm_count() + n_kv_heads - 1) / n_kv_heads;
  // no more than the sequences could use at one chunk per kMinChunk rows
  const long long by_len = (long long)batch * ((std::max(max_len, 1) + kMinChunk - 1) / kMinChunk);
  return (int)std::max<long long>(batch, std::min<long long>(per_head, by_len));
}

int attn_chunks(int batch, int n_kv_heads, int max_len) {
  const int nct = attn_ctas_per_head(batch, n_kv_heads, max_len);
  const int share = std::max(8, 4 * ((nct + batch - 1) / batch));
  const int by_len = (std::max(max_len, 1) + kMinChunk - 1) / kMinChunk;
  return std::max(1, std::min(std::min(nct, share), by_len));
}

size_t attn_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim, int max_len) {
  const size_t nc = (size_t)attn_chunks(batch, n_kv_heads, max_len);
  return (size_t)batch * n_heads * nc * ((size_t)head_dim + 2) * sizeof(float);
}

int attn_launch(AttnParams P, cudaStream_t stream) {
  const size_t nc = (size_t)P.nc;
  float* ws = reinterpret_cast<float*>(P.workspace);
  P.ws_o = ws;
  P.ws_m = ws + (size_t)P.batch * P.n_heads * nc * P.head_dim;
  P.ws_l = P.ws_m + (size_t)P.batch * P.n_heads * nc;
  if (P.kv_dtype == Q8D_KV_F16) return attn_mma_launch(P, stream);
  if (P.kv_dtype == Q8D_KV_Q8_0) return attn_q8kv_launch(P, stream);
  if (P.head_dim == 128) return launch_attn_g<128, float>(P, stream);
  return launch_attn_g<64, float>(P, stream);
}

int kv_append_launch(const float* k, const float* v, void* kc, void* vc, int kv_dtype, int kvw,
                     int cap, const int* d_pos, int* d_err, cudaStream_t stream) {
  const int threads = 256, blocks = std::max(1, std::min(64, (kvw + threads - 1) / threads));
  if (kv_dtype == Q8D_KV_Q8_0) {
    const int qblocks = std::max(1, std::min(64, (2 * (kvw / kQBlock) * 32 + threads - 1) / threads));
    kv_append_q8_kernel<<<qblocks, threads, 0, stream>>>(k, v, static_cast<uint8_t*>(kc),
                                                         static_cast<uint8_t*>(vc), kvw, cap,
                                                         d_pos, d_err);
    return check_launch();
  }
  if (kv_dtype == Q8D_KV_F16)
    kv_append_kernel<__half><<<blocks, threads, 0, stream>>>(
        k, v, reinterpret_cast<__half*>(kc), reinterpret_cast<__half*>(vc), kvw, cap, d_pos, d_err);
  else
    kv_append_kernel<float><<<blocks, threads, 0, stream>>>(
        k, v, reinterpret_cast<float*>(kc), reinterpret_cast<float*>(vc), kvw, cap, d_pos, d_err);
  return check_launch();
}

}  // namespace q8d
