// The whole decode step in one persistent cooperative kernel (sm_103a).
//
// What the step computes is the pages' decoder ("IV.4: One command buffer
// per token": embed_row; per layer RMSNorm, q|k|v matvecs, bias / QK-norm,
// RoPE, append_kv, attention_decode, o matvec + residual, RMSNorm, gate|up
// matvecs, SiLU*up, down matvec + residual; final RMSNorm, lm_head matvec,
// argmax_row).  How it runs is GB300-specific:
//  * One CTA per SM, 20 consumer warps and one producer warp.  The producer
//    streams the weight tiles of this CTA's rows of every matvec phase, in
//    phase order, through a ring of shared-memory stages with 1-D bulk
//    copies (TMA) completing on mbarriers.  Weights do not depend on
//    activations, so the stream runs ahead across phase boundaries, grid
//    barriers and attention: HBM stays busy while the consumers wait.
//  * Consumers walk the phase table; a grid-wide barrier (a counter in
//    global memory, bounded spin) separates phases.  Activations written by
//    other CTAs are read through L2 (ld.global.cg), never through the
//    non-coherent L1 / read-only path.
//  * Matvec phases use the layout of the standalone matvec kernel: warp
//    pairs own the even / odd block columns of 64-column segments, the
//    lane's 32 activations in registers (RMSNorm applied while loading),
//    lane partials folded within the warp and reduced in double-buffered
//    row windows; the gate|up phase forms SiLU(gate) * up as it writes the
//    up rows.
//  * Attention: one CTA per (KV head, context chunk) computes the G query
//    heads' online-softmax partial over its chunk on CUDA cores (f32); the
//    CTA owning row L-1 applies bias / QK-norm / RoPE to the new k, v,
//    appends them to the cache and patches them into its chunk; a combine
//    phase (one CTA per query head) merges the chunks.  The producer warp
//    prefetches each CTA's K/V chunk into L2 a phase ahead.
#include <algorithm>
#include <cmath>
#include <type_traits>

#include "q8d_attn_common.cuh"
#include "q8d_gemv.cuh"
#include "q8d_internal.cuh"
#include "q8d_megastep.cuh"
#include "q8d_mma_frag.cuh"

namespace q8d {

namespace {

using namespace mv;

constexpr int kW = kMsWarps;
constexpr int kCT = kW * 32;  // consumer threads
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxStages = 8;
// Partials a warp keeps per row: its 32 lane partials folded to 4 with
// three shuffles, so a reduction window (a shared buffer) holds 8x the rows
// (and a row's partials stay whole 16-byte vectors for any NS).
constexpr int kPW = 4;

// Per-CTA state at fixed shared addresses (no registers to hold pointers).
__shared__ uint64_t ms_full[kMaxStages];   // stage s filled (TMA complete_tx)
__shared__ uint64_t ms_empty[kMaxStages];  // stage s released by all consumer warps
__shared__ int ms_abort;                   // a wait of this CTA was abandoned
__shared__ int ms_flag;
__shared__ unsigned ms_target;             // grid barrier arrivals to wait for
__shared__ unsigned ms_spin;               // grid barrier polls before giving up
__shared__ int ms_L;                       // attended length of this step
// Per-row values of the CTA's rows of a matvec phase: the residual rows it
// accumulates into (prefetched at the phase start), or its gate rows of a
// gate|up phase (kept for the up rows): no global round trip in the window
// reductions.
constexpr int kRowsMax = 512;
__shared__ __align__(16) float ms_rows[kRowsMax];

__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }

// A pointer field of a read-only table.
template <typename T>
__device__ __forceinline__ T* ldg_ptr(T* const* p) {
  return reinterpret_cast<T*>(__ldg(reinterpret_cast<const unsigned long long*>(p)));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of the consumer threads of all CTAs, in two halves:
// grid_arrive (this CTA is done with the phase) and grid_wait (every CTA
// is); work that depends on no other CTA may run in between.  grid_wait
// returns false if the step was aborted (a CTA gave up a wait); then every
// CTA stops.
__device__ void grid_arrive(const MParams& P) {
  volatile int* s_abort = &ms_abort;
  volatile int* s_flag = &ms_flag;
  consumer_sync(kCT);
  if (threadIdx.x == 0) {
    ms_target += gridDim.x;
    if (*s_abort) {
      atomicExch(P.abort, 1);
      *s_flag = 0;
    } else {
      // release: this CTA's writes of the phase (ordered before by the CTA
      // barrier above) are visible to every CTA that acquires the count
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.bar) : "memory");
      *s_flag = 1;
    }
  }
}

__device__ bool grid_wait(const MParams& P) {
  volatile int* s_abort = &ms_abort;
  volatile int* s_flag = &ms_flag;
  if (threadIdx.x == 0) {
    const unsigned target = ms_target;
    int ok = *s_flag;
    if (ok) {
      for (uint32_t i = 0;; ++i) {
        if ((int)(ld_acquire(P.bar) - target) >= 0) break;
        if (*(volatile int*)P.abort) {
          ok = 0;
          break;
        }
        if (i >= ms_spin) {
          ok = 0;
          atomicExch(P.abort, 1);
          if (P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
          break;
        }
      }
      // (no fence here: the acquire load that saw the count synchronizes
      // with every CTA's release add, the CTA barrier below orders this
      // CTA's other threads after it, and their reads of other CTAs' data
      // go through L2 (ld.global.cg, cp.async.cg); a gpu-scope fence here
      // measured ~0.5 us per phase boundary)
    }
    if (!ok) *s_abort = 1;
    *s_flag = ok;
  }
  cp_async_wait_all();  // this thread's staging copies of the next phase
  consumer_sync(kCT);
  return *s_flag != 0;
}

// Whether a tensor-core phase's RMSNorm weights fit behind its fragments.
__device__ __forceinline__ bool tc_weights_staged(const MPhase& F) {
  return F.bpr * 260 + tc::kZeroPad <= kMsRegion;  // bpr * (128 + 4) + pad + n * 4
}

// Work of matvec phase F that depends on no other CTA, done between the
// halves of the grid barrier before it: the residual rows this CTA adds to
// (written by this CTA, or before an earlier barrier) and the RMSNorm
// weights staged where the activation pass reads them.
// The copies are asynchronous (cp.async through L2, completed by grid_wait),
// so their latency overlaps the barrier.  Thread 0 polls the barrier and
// issues none.  The residual rows are copied in 16-byte units from the
// 16-byte boundary at or below the CTA's first row (ms_rows_off floats
// before it; the extra values are never used).
__device__ void matvec_pre(const MPhase& F, uint8_t* region) {
  const int t = threadIdx.x - 32;  // (warps 1 .. kW-1)
  if (F.accumulate && F.rows_per_cta + 3 <= kRowsMax) {
    const int r0 = blockIdx.x * F.rows_per_cta;
    const int r1 = min(F.total_rows, r0 + F.rows_per_cta);
    const int a0 = r0 & ~3, n4 = (r1 - a0 + 3) / 4;  // (the rows end 16-byte aligned)
    for (int i = t; i >= 0 && i < n4; i += kCT - 32) cp_async16(ms_rows + 4 * i, F.y[0] + a0 + 4 * i);
  }
  if (F.tc) {
    // tensor-core phase: the RMSNorm weights at the end of the region
    // (clear of the fragments the activation pass writes)
    if (F.xmode == kXRmsNorm && tc_weights_staged(F)) {
      float4* ws = reinterpret_cast<float4*>(region + kMsRegion) - F.n / 4;
      for (int i = t; i >= 0 && i < F.n / 4; i += kCT - 32)
        cp_async16(ws + i, reinterpret_cast<const float4*>(F.xw) + i);
    }
    return;
  }
  const int pass4 = kMsRegion / 32;
  if (F.xmode == kXRmsNorm && F.n / 4 <= pass4) {
    float4* ws = reinterpret_cast<float4*>(region) + pass4;
    const int n4 = F.n / 4;
    const int rot = (int)((blockIdx.x * 97u) % (unsigned)n4);
    for (int i = t; i >= 0 && i < n4; i += kCT - 32) {
      int j = i + rot;
      if (j >= n4) j -= n4;
      const int ph = (j & ~7) | (((j & 7) + (j >> 4)) & 7);
      cp_async16(ws + ph, reinterpret_cast<const float4*>(F.xw) + j);
    }
  }
}

// The matrix row held in ms_rows[0] for phase F (the 16-byte boundary at or
// below the CTA's first row), or -1 when ms_rows is not used (no residual
// or gate rows, or too many rows: values then go through L2).
__device__ __forceinline__ int ms_rbase(const MPhase& F) {
  return (F.accumulate || F.glu) && F.rows_per_cta + 3 <= kRowsMax
             ? (int)(blockIdx.x * F.rows_per_cta) & ~3
             : -1;
}

// ---------------------------------------------------------------- matvec
// Tiles of the CTA's virtual rows of phase F (at most F.R rows, never across
// a matrix end).  Fields come from the phase copy in shared memory.
struct MCursor {
  int cur, r0, seg, seg_end;
  __device__ void start(const MPhase& F, int v0) {
    cur = v0;
    seg = 0;
    while (seg + 1 < F.nseg && v0 >= F.vbegin[seg + 1]) ++seg;
    r0 = v0 - F.vbegin[seg];
    seg_end = F.vbegin[seg + 1];
  }
  __device__ int rows(int R, int v1) const { return min(R, min(seg_end, v1) - cur); }
  __device__ void advance(const MPhase& F, int n) {
    cur += n;
    r0 += n;
    if (cur == seg_end && seg + 1 < F.nseg) {
      ++seg;
      r0 = 0;
      seg_end = F.vbegin[seg + 1];
    }
  }
};

// Ring position shared by consecutive phases (tile index modulo the stages).
struct RingPos {
  int s;
  uint32_t ph;
  uint32_t stage32;
};

// The CTA's virtual row ranges of phase F: one contiguous range, or for a
// gate|up phase the same rows of both matrices (two ranges).
__device__ __forceinline__ void piece_range(int glu, int nrows0, int rpc, int total, int piece,
                                            int& v0, int& v1) {
  if (glu) {
    v0 = blockIdx.x * rpc;
    v1 = min(nrows0, v0 + rpc);
    if (v0 > v1) v0 = v1;
    v0 += piece * nrows0;
    v1 += piece * nrows0;
  } else {
    v0 = blockIdx.x * rpc;
    v1 = min(total, v0 + rpc);
  }
}

// Writes the dot product `sum` of virtual row vr of phase F: adds the
// residual, forms SiLU(gate) * up, tracks the argmax.
// rbase: ms_rbase(F).
__device__ __forceinline__ void ms_store_row(const MPhase& F, int vr, float sum, int rbase,
                                             float& bv, int& bi) {
  int sg = 0;
  while (sg + 1 < F.nseg && vr >= F.vbegin[sg + 1]) ++sg;
  const int ri = vr - F.vbegin[sg];
  float* y = F.y[sg] + ri;
  float out = sum;
  if (F.accumulate) out += rbase >= 0 ? ms_rows[ri - rbase] : __ldcg(y);
  if (F.glu) {
    // gate rows are kept; an up row combines with its gate row (computed
    // by this CTA in an earlier window) into h = silu(gate) * up, stored
    // over the gate half (the only half read afterwards)
    if (sg == 0) {
      if (rbase >= 0) ms_rows[ri - rbase] = out;
      else *y = out;
    } else {
      const float gt = rbase >= 0 ? ms_rows[ri - rbase] : __ldcg(F.y[0] + ri);
      F.y[0][ri] = gt / (1.0f + expf(-gt)) * out;
    }
  } else {
    *y = out;
  }
  if (F.argmax && !isnan(out) && am_better(out, ri, bv, bi)) {
    bv = out;
    bi = ri;
  }
}

// Window reduction: sums each row's warp partials over segments and lanes
// in a fixed order and writes the row.
__device__ void ms_window_reduce(const MPhase& F, const float* part, int nrow, int wbeg, int rbase,
                                 float& bv, int& bi) {
  // 8 threads per row, four rows per warp at a time: windows of up to 80
  // rows take one pass, so no warp carries a second pass into the next
  // window (stage releases and the next window barrier wait for the last)
  // (rows go to the highest warps first: row group 0, the low warps, has
  // the most rows of a ragged tile)
  const int lane = threadIdx.x & 31, warp = kW - 1 - (threadIdx.x >> 5);
  const int sub = lane & 7;
  const int n4 = F.NS * kPW / 4;  // float4s per row
  for (int r0 = warp * 4; r0 < nrow; r0 += kW * 4) {
    const int r = r0 + (lane >> 3);
    const bool valid = r < nrow;
    const float4* pr = reinterpret_cast<const float4*>(part + (size_t)(valid ? r : r0) * n4 * 4);
    uint64_t acc0 = pack2(0.f, 0.f), acc1 = acc0;
    for (int k = sub; k < n4; k += 8) {
      const float4 v = pr[k];
      acc0 = add2(acc0, pack2(v.x, v.y));
      acc1 = add2(acc1, pack2(v.z, v.w));
    }
    float lo, hi;
    unpack2(add2(acc0, acc1), lo, hi);
    float sum = lo + hi;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (valid && sub == 0) ms_store_row(F, wbeg + r, sum, rbase, bv, bi);
  }
}

// The CTA's argmax candidate (over the threads' (bv, bi)) to P.am_val /
// P.am_idx[blockIdx.x].
__device__ void ms_argmax_cta(const MParams& P, float bv, int bi, float* s_f, int* s_i) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (am_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    s_f[warp] = bv;
    s_i[warp] = bi;
  }
  consumer_sync(kCT);
  if (threadIdx.x == 0) {
    for (int w = 1; w < kW; ++w)
      if (am_better(s_f[w], s_i[w], bv, bi)) {
        bv = s_f[w];
        bi = s_i[w];
      }
    P.am_val[blockIdx.x] = bv;
    P.am_idx[blockIdx.x] = bi;
  }
}

// Consumes up to F.win tiles of the CTA's rows [c.cur, v1) of phase F (one
// reduction window), storing the lanes' partials at window buffer `buf`
// (bytes); returns the rows consumed.  AM: alignment mode of this warp.
template <int AM>
__device__ int ms_consume_window(const MPhase& F, const MParams& P, RingPos& rp,
                                 uint32_t smem32, MCursor& c,
                                 uint32_t& delta, int v1, uint32_t lane_buf, int rg, bool active,
                                 uint32_t boff, const uint64_t (&x2)[16], bool& ok) {
  const int lane = threadIdx.x & 31;
  const int RG = F.RG, R = F.R;
  const int nP = F.NS * kPW;  // partials per row
  const uint32_t rowb = (uint32_t)F.row_bytes;
  const uint32_t step = (uint32_t)RG * rowb;
  const uint32_t pstep = (uint32_t)(RG * nP * 4);
  const uint32_t rb15 = rowb & 15u;
  int wrow = 0;
#pragma unroll 1
  for (int wt = 0; wt < F.win && c.cur < v1; ++wt) {
    const int rows = c.rows(R, v1);
    const int rows_st = active ? rows : 0;  // rows whose partials this warp stores
    ok = wait_or_abort(&ms_full[rp.s], rp.ph, &ms_abort) && ok;
    // (warps beyond NS * RG, when NS does not divide the warp count, run the
    // same code on row group 0's rows and store nothing)
    uint32_t o = after_wait(rp.stage32 + delta + boff + (uint32_t)rg * rowb);
    uint32_t d = lane_buf + (uint32_t)(wrow * nP) * 4u;
    // this warp's rows of the tile, one block at a time (a ragged tile stops
    // at the warp's last row)
#pragma unroll 1
    for (int rl = rg; rl < rows; rl += RG) {
      float va = block_dot<AM>(o, x2);
      va += __shfl_xor_sync(0xffffffffu, va, 16);
      va += __shfl_xor_sync(0xffffffffu, va, 8);
      va += __shfl_xor_sync(0xffffffffu, va, 4);
      if (rl < rows_st && lane < kPW) sts32(d, va);
      o += step;
      d += pstep;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms_empty[rp.s]);
    rp.stage32 += (uint32_t)P.stage_bytes;
    if (++rp.s == P.nstages) {
      rp.s = 0;
      rp.ph ^= 1u;
      rp.stage32 = smem32;
    }
    const int seg_before = c.seg;
    c.advance(F, rows);
    delta = c.seg == seg_before ? (delta + (uint32_t)rows * rb15) & 15u : 0u;
    wrow += rows;
  }
  return wrow;
}

__device__ bool matvec_phase(const MPhase& F, const MParams& P, RingPos& rp, uint32_t smem32,
                             uint8_t* region,
                             float* s_f, int* s_i) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = F.NS, RG = F.RG;
  const bool active = warp < NS * RG;
  const int ci = warp % NS, rg = active ? warp / NS : 0;
  int col, col_read;
  if (F.paired) {
    const int par = ci & 1;
    col = 64 * (ci >> 1) + 2 * lane + par;
    col_read = min(col, F.bpr - 1 - ((F.bpr - 1 - par) & 1));
  } else {
    col = lane;
    col_read = min(col, F.bpr - 1);
  }
  // Activations: every CTA needs all of x, and the warps of a column class
  // share it, so x (and the RMSNorm weights) pass through shared memory in
  // chunks of the region, loaded with coalesced 16-byte loads (each CTA
  // starting at its own offset, so the CTAs released together by the grid
  // barrier spread over L2 lines).  A lane's column is 8 chunks of 16 bytes
  // and lanes read columns 256 bytes apart, so chunk t of column c is stored
  // at position (t + c/2) mod 8 of the column: a warp's reads then cover all
  // bank groups.
  uint64_t x2[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) x2[t] = 0;
  const bool rms = F.xmode == kXRmsNorm;
  const int pass4 = (rms ? kMsRegion / 32 : kMsRegion / 16);  // float4s of x per pass
  float inv = 1.f;
  if (rms && F.n / 4 > pass4) {
    // x does not fit in one pass: the sum of squares straight from L2
    float ss = 0.f;
    const float4* x4 = reinterpret_cast<const float4*>(F.X);
    for (int i = threadIdx.x; i < F.n / 4; i += kCT) {
      const float4 v = __ldcg(x4 + i);
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_f[warp] = ss;
    consumer_sync(kCT);
    float tot = 0.f;
    for (int w = 0; w < kW; ++w) tot += s_f[w];
    inv = 1.0f / sqrtf(tot / (float)F.n + P.eps);
    consumer_sync(kCT);  // s_f is reused below
  }
  // (the residual rows and, for one pass, the RMSNorm weights were staged
  // by matvec_pre)
  const bool ws_staged = rms && F.n / 4 <= pass4;
  float4* xs = reinterpret_cast<float4*>(region);
  float4* ws = xs + pass4;
  for (int e0 = 0; e0 < F.n / 4; e0 += pass4) {
    const int n4 = min(pass4, F.n / 4 - e0);
    const int rot = (int)((blockIdx.x * 97u) % (unsigned)n4);
    for (int i = threadIdx.x; i < n4; i += kCT) {
      int j = i + rot;
      if (j >= n4) j -= n4;
      const int ph = (j & ~7) | (((j & 7) + (j >> 4)) & 7);
      xs[ph] = __ldcg(reinterpret_cast<const float4*>(F.X) + e0 + j);
      if (rms && !ws_staged) ws[ph] = __ldg(reinterpret_cast<const float4*>(F.xw) + e0 + j);
    }
    consumer_sync(kCT);
    if (rms && F.n / 4 <= pass4) {
      // sum of squares (all of x is in this pass), the same order in every CTA
      float ss = 0.f;
      for (int i = threadIdx.x; i < n4; i += kCT) {
        const float4 v = xs[i];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_f[warp] = ss;
      consumer_sync(kCT);
      float tot = 0.f;
      for (int w = 0; w < kW; ++w) tot += s_f[w];
      inv = 1.0f / sqrtf(tot / (float)F.n + P.eps);
    }
    const int cl = col - e0 / 8;  // column within this pass
    if (active && col < F.bpr && cl >= 0 && cl * 8 < n4) {
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int ph = cl * 8 + ((t + (cl >> 1)) & 7);
        float4 v = xs[ph];
        if (rms) {
          const float4 wv = ws[ph];
          v.x = v.x * inv * wv.x;
          v.y = v.y * inv * wv.y;
          v.z = v.z * inv * wv.z;
          v.w = v.w * inv * wv.w;
        }
        x2[2 * t] = pack2(v.x, v.y);
        x2[2 * t + 1] = pack2(v.z, v.w);
      }
    }
    consumer_sync(kCT);  // the region is refilled next (or holds window partials)
  }
  const uint32_t boff = (uint32_t)col_read * kQBlockBytes;
  float* part = reinterpret_cast<float*>(region);
  const uint32_t part32 = smem_u32(region);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool ok = true;
  // With an even number of blocks per row every row starts at a multiple of
  // 4 bytes, so all blocks of a paired warp start at 2*(col & 1) mod 4.
  const int am = (F.paired && (F.bpr & 1) == 0) ? (ci & 1) : 2;
  const uint32_t nP = (uint32_t)F.NS * kPW;
  const uint32_t lane_part =
      part32 + ((uint32_t)(ci * kPW + (lane & (kPW - 1))) + (uint32_t)rg * nP) * 4u;
  const uint32_t buf_bytes = (uint32_t)F.win * (uint32_t)F.R * nP * 4u;
  uint32_t buf = 0;
  const int rbase = ms_rbase(F);
  const int npieces = F.glu ? 2 : 1;
  for (int piece = 0; piece < npieces; ++piece) {
    int v0, v1;
    piece_range(F.glu, F.vbegin[1], F.rows_per_cta, F.total_rows, piece, v0, v1);
    MCursor c;
    c.start(F, v0);
    uint32_t delta = ((uint32_t)c.r0 * ((uint32_t)F.row_bytes & 15u)) & 15u;
    while (c.cur < v1) {
      const int wbeg = c.cur;
      int nrow;
      if (am == 0)
        nrow = ms_consume_window<0>(F, P, rp, smem32, c, delta, v1,
                                    lane_part + buf, rg, active, boff, x2, ok);
      else if (am == 1)
        nrow = ms_consume_window<1>(F, P, rp, smem32, c, delta, v1,
                                    lane_part + buf, rg, active, boff, x2, ok);
      else
        nrow = ms_consume_window<2>(F, P, rp, smem32, c, delta, v1,
                                    lane_part + buf, rg, active, boff, x2, ok);
      // window complete: every consumer warp has stored its partials.  The
      // other buffer was reduced before this barrier, so the next window may
      // overwrite it.
      consumer_sync(kCT);
      ms_window_reduce(F, part + buf / 4, nrow, wbeg, rbase, bv, bi);
      buf = buf ? 0u : buf_bytes;
    }
  }
  if (F.argmax) ms_argmax_cta(P, bv, bi, s_f, s_i);
  return ok;
}

// ---------------------------------------------------------------- tensor-core matvec
// Matvec phases whose rows are whole pairs of 8 blocks (n % 256 == 0) and
// whose x fragments fit the shared region: the block dot products run on
// mma.sync (layout in q8d_mma_frag.cuh).  A tile is 8 consecutive rows of
// the CTA's range (the last one may hold fewer), each in a row slot of F.SR
// bytes; the unit pairs of all the CTA's tiles are dealt to the warps in
// turn (pair k of the CTA's t-th tile goes to warp (t * pairs + k) mod 20),
// so no warp waits for another within a window.  Each 32-element block of
// the activation vector gets its own power-of-two scale before the f16
// hi/lo split (the 8 threads that build a block's fragment share its max),
// and the block's inverse scale multiplies its partial with the weight
// scale: no CTA-wide reduction is needed for it.
//
// Region layout: x fragments (128 bytes a block, tc::x_word_offset), a
// 512-byte zero pad, the blocks' inverse scales [bpr] (f32), then the
// double-buffered window partials [2][win * 8][kW].

constexpr int kTcItems = 4;  // (block, word) items per consumer thread: bpr <= 320

__device__ bool tc_matvec_phase(const MPhase& F, const MParams& P, RingPos& rp, uint32_t smem32,
                                uint8_t* region, float* s_f, int* s_i) {
  using namespace tc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bpr = F.bpr;
  uint8_t* xf = region;
  uint8_t* zpad = xf + (size_t)bpr * kXfBlock;
  float* xinv = reinterpret_cast<float*>(zpad + kZeroPad);
  float* part = xinv + bpr;
  // ---- x fragments (RMSNorm applied first where the phase has it) ----
  const bool rms = F.xmode == kXRmsNorm;
  const int nit = bpr * 8;
  float v[kTcItems][4];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kTcItems; ++k) {
    const int it = threadIdx.x + k * kCT;
    if (it < nit) {
      load_word<0>(F.X, it >> 3, it & 7, v[k]);
    } else {
      v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0.f;
    }
    ss = fmaf(v[k][0], v[k][0], ss);
    ss = fmaf(v[k][1], v[k][1], ss);
    ss = fmaf(v[k][2], v[k][2], ss);
    ss = fmaf(v[k][3], v[k][3], ss);
  }
  if (rms) {
    // (every element is in exactly one (block, word) item; the sum's order
    // is the same in every CTA)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_f[warp] = ss;
    consumer_sync(kCT);
    float tot = 0.f;
    for (int w = 0; w < kW; ++w) tot += s_f[w];
    const float inv = 1.0f / sqrtf(tot / (float)F.n + P.eps);
    const bool staged = tc_weights_staged(F);  // (by matvec_pre)
    const float* wsm = reinterpret_cast<const float*>(region + kMsRegion) - F.n;
#pragma unroll
    for (int k = 0; k < kTcItems; ++k) {
      const int it = threadIdx.x + k * kCT;
      float wv[4] = {0.f, 0.f, 0.f, 0.f};
      if (it < nit) {
        if (staged) load_word<2>(wsm, it >> 3, it & 7, wv);
        else load_word<1>(F.xw, it >> 3, it & 7, wv);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) v[k][j] = v[k][j] * inv * wv[j];
    }
  }
#pragma unroll
  for (int k = 0; k < kTcItems; ++k) {
    const int it = threadIdx.x + k * kCT;
    if (k * kCT >= nit) break;  // (uniform over the CTA)
    build_x_word(it, it < nit, v[k], xf, xinv);
  }
  if (threadIdx.x < kZeroPad / 4) reinterpret_cast<uint32_t*>(zpad)[threadIdx.x] = 0u;
  consumer_sync(kCT);

  // ---- units ----
  const int gq = lane >> 2, cq = lane & 3;
  const LaneOffs LO = lane_offsets(cq);
  const XLane XL = x_lane(lane);
  const uint32_t xf32 = smem_u32(xf), z32 = smem_u32(zpad);
  const uint32_t xi32 = smem_u32(xinv) + 4u * (uint32_t)lane_block(cq);
  const bool lo_half = cq < 2;
  const int P8 = bpr / 8;  // unit pairs per row
  const int T = F.T;
  // this lane's row gq of a set: groups of 1 << gsh rows, 16 bytes apart
  const uint32_t rowoff = (uint32_t)(gq * F.row_bytes) + (uint32_t)((gq >> F.gsh) << 4);
  const uint32_t part32 = smem_u32(part);
  const int tile_rows = kSetRows * T;
  const uint32_t buf_bytes = (uint32_t)(F.win * tile_rows * kW) * 4u;
  const int rbase = ms_rbase(F);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool ok = true;
  uint32_t buf = 0;
  int first = warp;  // this warp's first pair of the next tile
  const int npieces = F.glu ? 2 : 1;
  for (int piece = 0; piece < npieces; ++piece) {
    int v0, v1;
    piece_range(F.glu, F.vbegin[1], F.rows_per_cta, F.total_rows, piece, v0, v1);
    int wt = 0, wbeg = v0;
    for (int r0 = v0; r0 < v1; r0 += tile_rows) {
      const int nsets = min(T, (v1 - r0 + kSetRows - 1) / kSetRows);
      const int items = nsets * P8;
      ok = wait_or_abort(&ms_full[rp.s], rp.ph, &ms_abort) && ok;
      const uint32_t row32 = after_wait(rp.stage32 + rowoff);
      float y0 = 0.f, y1 = 0.f;  // row gq of the tile's sets 0 / 1
      for (int j = first; j < items; j += kW) {
        const int sl = j >= P8 ? 1 : 0;  // (T <= 2)
        const int k = j - sl * P8;
        const uint32_t rb = row32 + (uint32_t)(sl * F.SR) + 272u * (uint32_t)k;
        const uint32_t xb = XL.match ? xf32 + (uint32_t)(k * kXfPair) + XL.off : z32;
        float pe, po;
        pair_units(rb, xb, XL.step, LO, lo_half, pe, po);
        const float se = unit_scale(rb, LO, false) * lds32f(xi32 + 32u * (uint32_t)k);
        const float so = unit_scale(rb, LO, true) * lds32f(xi32 + 32u * (uint32_t)k + 4u);
        const float d = fmaf(se, pe, so * po);
        if (sl) y1 += d;
        else y0 += d;
      }
      first = ((first - items) % kW + kW) % kW;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms_empty[rp.s]);
      rp.stage32 += (uint32_t)P.stage_bytes;
      if (++rp.s == P.nstages) {
        rp.s = 0;
        rp.ph ^= 1u;
        rp.stage32 = smem32;
      }
      // the warp's partials of rows r0 + gq and r0 + 8 + gq (4 lanes per row)
      y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
      y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
      y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
      y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
      if (cq == 0) {
        const uint32_t a = part32 + buf + (uint32_t)(((wt * tile_rows + gq) * kW + warp) * 4);
        sts32(a, y0);
        if (T > 1) sts32(a + (uint32_t)(kSetRows * kW * 4), y1);
      }
      ++wt;
      if (wt == F.win || r0 + tile_rows >= v1) {
        // window complete: sum each row's warp partials (4 threads a row,
        // 5 warps each, in a fixed order) and write the rows
        consumer_sync(kCT);
        const int nrow = min(wt * tile_rows, v1 - wbeg);
        const float* pw = part + buf / 4;
        for (int i0 = 0; i0 < nrow; i0 += kCT / 4) {
          const int i = i0 + (threadIdx.x >> 2), sub = threadIdx.x & 3;
          float sum = 0.f;
          if (i < nrow) {
            const float* pr = pw + (size_t)i * kW;
#pragma unroll
            for (int w = 0; w < kW / 4; ++w) sum += pr[sub + 4 * w];
          }
          sum += __shfl_xor_sync(0xffffffffu, sum, 1);
          sum += __shfl_xor_sync(0xffffffffu, sum, 2);
          if (i < nrow && sub == 0) ms_store_row(F, wbeg + i, sum, rbase, bv, bi);
        }
        buf = buf ? 0u : buf_bytes;
        wt = 0;
        wbeg = r0 + tile_rows;
      }
    }
  }
  if (F.argmax) ms_argmax_cta(P, bv, bi, s_f, s_i);
  return ok;
}

// ---------------------------------------------------------------- embedding
__device__ void embed_phase(const MParams& P, int tok, bool len_ok) {
  const bool bad = tok < 0 || tok >= P.vocab;
  if (blockIdx.x == 0 && threadIdx.x == 0 && P.d_err) {
    if (bad) atomicOr(P.d_err, Q8D_DERR_TOKEN_RANGE);
    if (!len_ok) atomicOr(P.d_err, Q8D_DERR_LEN_RANGE);
  }
  const long long rb = (long long)(P.hidden / kQBlock) * kQBlockBytes;
  for (int i = blockIdx.x * kCT + threadIdx.x; i < P.hidden; i += gridDim.x * kCT) {
    if (bad) {
      P.x[i] = __int_as_float(0x7fc00000);
      continue;
    }
    const uint8_t* blk = P.embed + (long long)tok * rb + (long long)(i / kQBlock) * kQBlockBytes;
    const float sc = f16_bits_to_f32((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
    P.x[i] = sc * (float)(int8_t)blk[2 + (i % kQBlock)];
  }
}

// ---------------------------------------------------------------- attention
template <typename KT>
__device__ __forceinline__ KT ms_to_cache(float v);
template <>
__device__ __forceinline__ __half ms_to_cache<__half>(float v) {
  return __float2half_rn(v);
}
template <>
__device__ __forceinline__ float ms_to_cache<float>(float v) {
  return v;
}

// DPL consecutive cache elements at p as floats.
template <typename KT, int DPL>
__device__ __forceinline__ void ld_row_part(const KT* p, float (&f)[DPL]) {
  if constexpr (sizeof(KT) == 2) {
    const __half2* h = reinterpret_cast<const __half2*>(p);
#pragma unroll
    for (int j = 0; j < DPL / 2; ++j) {
      const float2 t = __half22float2(h[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < DPL; ++j) f[j] = reinterpret_cast<const float*>(p)[j];
  }
}


// Context chunks per KV head for attended length L: P.nc (every CTA takes a
// chunk) unless that leaves chunks of fewer than 16 rows; producer, attention
// and combine agree on it.
__device__ __forceinline__ int attn_chunks_for(const MParams& P, int L) {
  return max(1, min(P.nc, (L + 15) / 16));
}

template <int D, typename KT>
struct MsAttnCfg {
  static constexpr int kST = 16384 / (D * (int)sizeof(KT)) < 64 ? 16384 / (D * (int)sizeof(KT)) : 64;  // tokens per sub-tile
  static constexpr int kDPL = D / 32;                        // dims per lane
  static constexpr int kRowB = D * (int)sizeof(KT);
  static constexpr int kGMax = 16;
  static constexpr int kOffQ = 0;                            // f32 [G][D]
  static constexpr int kOffS = kOffQ + kGMax * D * 4;        // f32 [G][ST]
  static constexpr int kOffK = kOffS + kGMax * kST * 4;      // KT [ST][D]
  static constexpr int kOffV = kOffK + kST * kRowB;
  static constexpr int kBytes = kOffV + kST * kRowB;
  static_assert(kBytes <= kMsRegion, "attention scratch fits the shared region");
  static_assert(kST <= 64, "two tokens per lane at most in the softmax");
};

template <int D, typename KT>
__device__ void attn_phase(const MParams& P, const MPhase& F, int L, bool len_ok,
                           uint8_t* region) {
  using C = MsAttnCfg<D, KT>;
  constexpr int DPL = C::kDPL, ST = C::kST;
  const int Hk = P.n_kv_heads, G = P.n_heads / Hk;
  const int item = blockIdx.x;
  if (!len_ok) return;  // the combine writes NaN outputs
  const int nc = attn_chunks_for(P, L);
  if (item >= Hk * nc) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = item / nc, c = item % nc;
  const MLayer* Ly = P.layers + F.layer;
  float* pm = P.ws_m + (size_t)item * G;
  float* pl = P.ws_l + (size_t)item * G;
  float* po = P.ws_o + (size_t)item * G * D;
  const int T = (L + nc - 1) / nc;
  const int t0 = c * T, t1 = min(L, t0 + T);
  // (chunks of T = ceil(L / nc) rows: for some L the last chunk is empty,
  // t0 >= L; it then writes m = -inf, l = 0, which the combine skips, and
  // it also takes the owner branch below, appending the same rounded row
  // as the chunk that holds row L-1)
  float* qs = reinterpret_cast<float*>(region + C::kOffQ);
  float* sc = reinterpret_cast<float*>(region + C::kOffS);
  uint8_t* Ks = region + C::kOffK;
  uint8_t* Vs = region + C::kOffV;
  const int pos = L - 1;
  const float* cosr = P.rope_cos + (size_t)pos * (D / 2);
  const float* sinr = P.rope_sin + (size_t)pos * (D / 2);
  const long long kvw = (long long)Hk * D;
  KT* kc = reinterpret_cast<KT*>(ldg_ptr(&Ly->kcache));
  KT* vc = reinterpret_cast<KT*>(ldg_ptr(&Ly->vcache));
  const float* bq = ldg_ptr(&Ly->bq);
  const float* bk = ldg_ptr(&Ly->bk);
  const float* bvp = ldg_ptr(&Ly->bv);
  const float* qn = ldg_ptr(&Ly->q_norm);
  const float* kn = ldg_ptr(&Ly->k_norm);

  constexpr int kChunks = C::kRowB / 16;
  const bool owner = t1 == L;  // this CTA's chunk ends with the new row L-1
  // K/V rows [tb, tb + nt) of head g into the sub-tile buffers, except the
  // new row, which the owner writes in from registers.
  auto issue = [&](int tb) {
    const int nt = min(ST, t1 - tb);
    const int nl = (owner && tb + nt == L) ? nt - 1 : nt;
    for (int e = threadIdx.x; e < 2 * nl * kChunks; e += kCT) {
      const int which = e / (nl * kChunks);
      const int r = (e / kChunks) % nl, pc = e % kChunks;
      const KT* src = (which ? vc : kc) + (long long)(tb + r) * kvw + (long long)g * D;
      cp_async16((which ? Vs : Ks) + r * C::kRowB + pc * 16,
                 reinterpret_cast<const uint8_t*>(src) + pc * 16);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  issue(t0);  // the loads overlap the prologues below

  // query heads of KV head g: bias, QK-norm, RoPE, then scale * log2(e)
  if (warp < G) {
    const int hq = g * G + warp;
    float v[D / 32];
#pragma unroll
    for (int t = 0; t < D / 32; ++t) v[t] = ldcg(P.q + (size_t)hq * D + lane + 32 * t);
    head_prologue<D>(v, lane, bq ? bq + (size_t)hq * D : nullptr, qn, P.eps, cosr, sinr);
#pragma unroll
    for (int t = 0; t < D / 32; ++t) qs[warp * D + lane + 32 * t] = v[t] * (P.scale * kLog2e);
  }
  // the owner appends the new k (bias, norm, RoPE) and v (bias) to the cache
  // and keeps them, rounded to the cache type, for its last sub-tile
  float nv[D / 32];
  const bool appender = owner && (warp == G || warp == G + 1);
  if (appender) {
    const bool isk = warp == G;
    const float* src = (isk ? P.k : P.v) + (size_t)g * D;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) nv[t] = ldcg(src + lane + 32 * t);
    if (isk)
      head_prologue<D>(nv, lane, bk ? bk + (size_t)g * D : nullptr, kn, P.eps, cosr, sinr);
    else
      head_prologue<D>(nv, lane, bvp ? bvp + (size_t)g * D : nullptr, nullptr, 0.f, nullptr,
                       nullptr);
    KT* dst = (isk ? kc : vc) + (long long)pos * kvw + (long long)g * D;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) dst[lane + 32 * t] = ms_to_cache<KT>(nv[t]);
  }

  float m_run = -INFINITY, l_run = 0.f;
  float o[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) o[j] = 0.f;
  for (int tb = t0; tb < t1; tb += ST) {
    const int nt = min(ST, t1 - tb);
    if (tb != t0) issue(tb);
    if (appender && tb + nt == L) {
      KT* row = reinterpret_cast<KT*>((warp == G ? Ks : Vs) + (nt - 1) * C::kRowB);
#pragma unroll
      for (int t = 0; t < D / 32; ++t) row[lane + 32 * t] = ms_to_cache<KT>(nv[t]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    consumer_sync(kCT);  // q rows, this sub-tile's K/V rows and the new row are in place
    // scores (log2 domain): warp per token, lanes over dims; the lanes'
    // partial dot products of 4 heads are reduce-scattered across the warp
    // (lane octet k ends with head k's sum: 6 shuffles instead of 20)
    for (int r = warp; r < nt; r += kW) {
      float kv[DPL];
      ld_row_part<KT, DPL>(reinterpret_cast<const KT*>(Ks + r * C::kRowB) + lane * DPL, kv);
      for (int h0 = 0; h0 < G; h0 += 4) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4* qh = reinterpret_cast<const float4*>(qs + min(h0 + i, G - 1) * D + lane * DPL);
          float part = 0.f;
#pragma unroll
          for (int j = 0; j < DPL / 4; ++j) {
            const float4 qq = qh[j];
            part = fmaf(qq.x, kv[4 * j], part);
            part = fmaf(qq.y, kv[4 * j + 1], part);
            part = fmaf(qq.z, kv[4 * j + 2], part);
            part = fmaf(qq.w, kv[4 * j + 3], part);
          }
          if constexpr (DPL % 4 != 0) {
#pragma unroll
            for (int j = DPL - DPL % 4; j < DPL; ++j)
              part = fmaf(qs[min(h0 + i, G - 1) * D + lane * DPL + j], kv[j], part);
          }
          v[i] = part;
        }
        const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
        float w2[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
          w2[i] = (b4 ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 2], 16);
        float z = (b3 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? w2[0] : w2[1], 8);
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        const int hh = h0 + ((lane >> 3) & 3);
        if ((lane & 7) == 0 && hh < G) sc[hh * ST + r] = z;
      }
    }
    consumer_sync(kCT);
    if (warp < G) {
      // online softmax of head `warp` over the sub-tile, then O += P.V
      float* sh = sc + warp * ST;
      const float s0 = lane < nt ? sh[lane] : -INFINITY;
      const float s1 = lane + 32 < nt ? sh[lane + 32] : -INFINITY;
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m_run, mx);
      const float corr = exp2f(m_run - mn);
      const float p0 = exp2f(s0 - mn), p1 = exp2f(s1 - mn);
      __syncwarp();
      if (lane < nt) sh[lane] = p0;
      if (lane + 32 < nt) sh[lane + 32] = p1;
      float ps = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l_run = l_run * corr + ps;
      m_run = mn;
      __syncwarp();
      // P.V with two independent accumulator sets
      float pa[DPL], pb[DPL];
#pragma unroll
      for (int j = 0; j < DPL; ++j) pa[j] = pb[j] = 0.f;
      int r = 0;
      for (; r + 1 < nt; r += 2) {
        const float p0r = sh[r], p1r = sh[r + 1];
        float va[DPL], vb[DPL];
        ld_row_part<KT, DPL>(reinterpret_cast<const KT*>(Vs + r * C::kRowB) + lane * DPL, va);
        ld_row_part<KT, DPL>(reinterpret_cast<const KT*>(Vs + (r + 1) * C::kRowB) + lane * DPL, vb);
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          pa[j] = fmaf(p0r, va[j], pa[j]);
          pb[j] = fmaf(p1r, vb[j], pb[j]);
        }
      }
      if (r < nt) {
        const float p0r = sh[r];
        float va[DPL];
        ld_row_part<KT, DPL>(reinterpret_cast<const KT*>(Vs + r * C::kRowB) + lane * DPL, va);
#pragma unroll
        for (int j = 0; j < DPL; ++j) pa[j] = fmaf(p0r, va[j], pa[j]);
      }
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[j] = fmaf(o[j], corr, pa[j] + pb[j]);
    }
    consumer_sync(kCT);  // the sub-tile buffers are refilled next
  }
  if (warp < G) {
    if (lane == 0) {
      pm[warp] = m_run;
      pl[warp] = l_run;
    }
#pragma unroll
    for (int j = 0; j < DPL; ++j) po[(size_t)warp * D + lane * DPL + j] = o[j];
  }
}

// out[hq] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the chunks of
// query head hq (one CTA per query head).  Warp w takes chunks w, w + 20,
// ... with all loads issued before use; the warps' partials are merged in
// warp order (deterministic).
// Attention phase over an f16 cache on the tensor cores (the layout of the
// standalone attention kernel): the G <= 16 query heads of KV head g are
// the 16 rows of m16n8k16 products.  The chunk's 16-token groups go to 4
// warp pairs (warps 0..7) in turn (groups p, p + 4, ...); both warps of a
// pair compute the group's scores and online softmax (kept in registers)
// and each owns half of head_dim in P.V, so a warp holds 32 (D = 128)
// accumulators.  q is split into f16 hi + lo after a power-of-two scale
// per head, and so are the probabilities (after a 2^12 scale), so every
// product is exact in the f32 accumulators.  Warps 8.. prepare q: each
// head row is written to shared memory already as the hi / lo A fragments
// of the MMA (conflict-free 32-bit reads, no splitting in the token loop).
// Each pair's first group is copied (cp.async) before the q prologue and the
// append; the owner CTA writes the new row into that group's tile itself
// when it is there, and later groups read it back from the cache.  Pair 0
// merges the pairs' {m, l, O} from shared memory and writes the partial.
template <int D>
struct MsMmaCfg {
  static constexpr int kPairs = 4;                   // warp pairs (token-group slots)
  static constexpr int kRow = D * 2;                 // f16 row bytes
  static constexpr int kStride = kRow + 16;          // padded tile row
  static constexpr int kStage = 2 * 16 * kStride;    // 16 K rows, then 16 V rows
  static constexpr int kOffQ = kPairs * kStage;      // q fragments [2 hi/lo][D/16][4][32] (u32)
  static constexpr int kOffF = kOffQ + 64 * D;       // per-head score factors [16]
  static constexpr int kBytes = kOffF + 16 * 4;
  static_assert(kBytes <= kMsRegion, "attention tiles fit the shared region");
  // merge buffer of the pairs in the tiles: m, l [4][16], O [4][16][D]
  static_assert(kPairs * 16 * (D + 2) * 4 <= kOffQ, "the merge buffer fits the tiles");
};

// Barrier of warp pair p (64 threads; ids 2.. are free: 0 is the CTA's, 1
// the consumer warps'), and of the 8 warps of the pairs (id 6).
__device__ __forceinline__ void pair_sync(int p) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + p) : "memory");
}
__device__ __forceinline__ void pairs_sync() { asm volatile("bar.sync 6, 256;" ::: "memory"); }

template <int D>
__device__ void attn_phase_mma(const MParams& P, const MPhase& F, int L, bool len_ok,
                               uint8_t* region) {
  using C = MsMmaCfg<D>;
  constexpr int KS = D / 16, NH = D / 16;  // k-steps of Q.K^T; n-tiles of a dim half in P.V
  constexpr int kPairs = C::kPairs;
  constexpr float kPS = 4096.f;  // probabilities scaled by 2^12 before the f16 split
  const int Hk = P.n_kv_heads, G = P.n_heads / Hk;
  const int item = blockIdx.x;
  if (!len_ok) return;  // the combine writes NaN outputs
  const int nc = attn_chunks_for(P, L);
  if (item >= Hk * nc) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int g = item / nc, c = item % nc;
  const MLayer* Ly = P.layers + F.layer;
  const int T = (L + nc - 1) / nc;
  const int t0 = c * T, t1 = min(L, t0 + T);
  const int nrows = max(0, t1 - t0);
  const int ngroups = (nrows + 15) / 16;
  // (chunks of T = ceil(L / nc) rows: for some L the last chunk is empty;
  // it writes m = -inf, l = 0, which the combine skips, and it also takes
  // the owner branch, appending the same rounded row as the chunk holding
  // row L-1)
  const bool owner = t1 == L;
  const int pos = L - 1;
  const int new_gi = owner && nrows > 0 ? (pos - t0) / 16 : -1;  // the new row's group
  const float* cosr = P.rope_cos + (size_t)pos * (D / 2);
  const float* sinr = P.rope_sin + (size_t)pos * (D / 2);
  const long long kvw = (long long)Hk * D;
  __half* kc = reinterpret_cast<__half*>(ldg_ptr(&Ly->kcache));
  __half* vc = reinterpret_cast<__half*>(ldg_ptr(&Ly->vcache));
  const uint8_t* kb = reinterpret_cast<const uint8_t*>(kc + (long long)g * D);
  const uint8_t* vb = reinterpret_cast<const uint8_t*>(vc + (long long)g * D);
  uint32_t* qf = reinterpret_cast<uint32_t*>(region + C::kOffQ);  // [hi/lo][kk][reg][lane]
  float* fh = reinterpret_cast<float*>(region + C::kOffF);
  const int pr = warp & (kPairs - 1), dh = warp / kPairs;  // (pair warps: warp < 2 * kPairs)
  uint8_t* st = region + pr * C::kStage;

  // this warp's half (rows 8 dh .. 8 dh + 7) of group gi into its pair's
  // tile; skip_new leaves the new row to the appender
  constexpr int kChunks = C::kRow / 16;
  auto load_half = [&](int gi, bool skip_new) {
    const int r0 = t0 + 16 * gi, nr = min(16, t1 - r0);
    const uint8_t* ks = kb + (long long)r0 * kvw * 2;
    const uint8_t* vs = vb + (long long)r0 * kvw * 2;
#pragma unroll
    for (int k = 0; k < 8 * kChunks / 32; ++k) {
      const int e = lane + 32 * k;
      const int r = 8 * dh + e / kChunks, pc = e % kChunks;
      if (r < nr && !(skip_new && r0 + r == pos)) {
        const long long off = (long long)r * kvw * 2 + pc * 16;
        cp_async16(st + r * C::kStride + pc * 16, ks + off);
        cp_async16(st + (16 + r) * C::kStride + pc * 16, vs + off);
      }
    }
  };
  if (warp < 2 * kPairs) {
    if (pr < ngroups) load_half(pr, true);
  } else if (warp < 2 * kPairs + 16) {
    // q row hh = warp - 8 (rows past G are zero; the 12 warps cover G <= 12,
    // which the step's set-up checks for f16 caches): bias / QK-norm / RoPE,
    // scaled by 2^sh so that max|q| < 2^11 (the score factor 2^-sh * scale
    // * log2(e) undoes it), split into hi / lo A fragments: the pair of
    // columns (d, d + 1) of row hh is register (hh >= 8) + 2 (d % 16 >= 8)
    // of lane (hh % 8) * 4 + (d % 8) / 2 at k-step d / 16
    const int hh = warp - 2 * kPairs;
    float v[D / 32];
    if (hh < G) {
      const int hq = g * G + hh;
      const float* bq = ldg_ptr(&Ly->bq);
#pragma unroll
      for (int t = 0; t < D / 32; ++t) v[t] = ldcg(P.q + (size_t)hq * D + lane + 32 * t);
      head_prologue<D>(v, lane, bq ? bq + (size_t)hq * D : nullptr, ldg_ptr(&Ly->q_norm), P.eps,
                       cosr, sinr);
    } else {
#pragma unroll
      for (int t = 0; t < D / 32; ++t) v[t] = 0.f;
    }
    float mx = 0.f;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) mx = fmaxf(mx, fabsf(v[t]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int e = 0;
    if (mx > 0.f) frexpf(mx, &e);
    // (sh >= -117 for any finite q; at most 125 keeps 2^sh a normal float:
    // rows below 2^-114 then scale to less)
    const int sh = mx > 0.f ? min(125, 11 - e) : 0;
    const float sc = __int_as_float((127 + sh) << 23);
#pragma unroll
    for (int t = 0; t < D / 32; ++t) {
      const float a = v[t] * sc;
      const float b = __shfl_down_sync(0xffffffffu, a, 1);  // column d + 1
      if ((lane & 1) == 0) {
        const int d = lane + 32 * t;
        uint32_t hi, lo;
        attn_split2(a, b, hi, lo);
        const int reg = (hh >= 8 ? 1 : 0) + ((d & 15) >= 8 ? 2 : 0);
        const int ln = (hh & 7) * 4 + ((d & 7) >> 1);
        qf[((d >> 4) * 4 + reg) * 32 + ln] = hi;
        qf[((KS + (d >> 4)) * 4 + reg) * 32 + ln] = lo;
      }
    }
    if (lane == 0) fh[hh] = hh < G ? ldexpf(P.scale * kLog2e, -sh) : 0.f;
  }
  // the owner appends the new k (bias, norm, RoPE) and v (bias) to the cache
  // (warps 6 and 7, after their copies are issued) and, when its group is a
  // pair's first, into that tile
  if (owner && (warp == 6 || warp == 7)) {
    const bool isk = warp == 6;
    float nv[D / 32];
    const float* src = (isk ? P.k : P.v) + (size_t)g * D;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) nv[t] = ldcg(src + lane + 32 * t);
    if (isk) {
      const float* bk = ldg_ptr(&Ly->bk);
      head_prologue<D>(nv, lane, bk ? bk + (size_t)g * D : nullptr, ldg_ptr(&Ly->k_norm), P.eps,
                       cosr, sinr);
    } else {
      const float* bv = ldg_ptr(&Ly->bv);
      head_prologue<D>(nv, lane, bv ? bv + (size_t)g * D : nullptr, nullptr, 0.f, nullptr,
                       nullptr);
    }
    __half* dst = (isk ? kc : vc) + (long long)pos * kvw + (long long)g * D;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) dst[lane + 32 * t] = __float2half_rn(nv[t]);
    if (new_gi >= 0 && new_gi < kPairs) {
      __half* row = reinterpret_cast<__half*>(region + new_gi * C::kStage +
                                              ((isk ? 0 : 16) + (pos - t0) % 16) * C::kStride);
#pragma unroll
      for (int t = 0; t < D / 32; ++t) row[lane + 32 * t] = __float2half_rn(nv[t]);
    }
  }
  cp_async_wait_all();
  consumer_sync(kCT);  // q fragments, first tiles and the new row in place; the cache row written
  if (warp >= 2 * kPairs) return;  // (the pair warps finish the phase)

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[NH][4];  // this warp's dim half: columns 8 n + 2 cq (+1) of the half
#pragma unroll
  for (int n = 0; n < NH; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const float f0 = fh[gq], f1 = fh[gq + 8];
  for (int gi = pr; gi < ngroups; gi += kPairs) {
    if (gi != pr) {  // later groups: one tile, refilled once the pair is done with it
      pair_sync(pr);
      load_half(gi, false);
      cp_async_wait_all();
      pair_sync(pr);
    }
    const int nr = min(16, t1 - (t0 + 16 * gi));
    // ---- S = Q.K^T for the group's 16 tokens (two n-tiles of 8): hi and
    // lo products in separate accumulators (four independent chains) ----
    float sh_[2][4], sl_[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      sh_[j][0] = sh_[j][1] = sh_[j][2] = sh_[j][3] = 0.f;
      sl_[j][0] = sl_[j][1] = sl_[j][2] = sl_[j][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t qh[4], ql[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        qh[r] = qf[(kk * 4 + r) * 32 + lane];
        ql[r] = qf[((KS + kk) * 4 + r) * 32 + lane];
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = min(8 * j + gq, nr - 1);
        const uint8_t* krow = st + tok * C::kStride + 4 * cq + 32 * kk;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + 16);
        attn_mma16816(sh_[j], qh, b0, b1);
        attn_mma16816(sl_[j], ql, b0, b1);
      }
    }
    // ---- log2-domain scores, mask, online softmax per row ----
    float sc[2][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 8 * j + 2 * cq + (e & 1);
        const float v = (sh_[j][e] + sl_[j][e]) * (e < 2 ? f0 : f1);
        sc[j][e] = tok < nr ? v : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(sc[j][0], sc[j][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[j][2], sc[j][3]));
    }
#pragma unroll
    for (int o_ = 1; o_ < 4; o_ <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float c0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
    const float c1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mrow = e < 2 ? mn0 : mn1;
        const float pv = sc[j][e] == -INFINITY ? 0.f : exp2f(sc[j][e] - mrow);
        sc[j][e] = pv;
        if (e < 2) rs0 += pv;
        else rs1 += pv;
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
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      o[n][0] *= c0;
      o[n][1] *= c0;
      o[n][2] *= c1;
      o[n][3] *= c1;
    }
    // ---- P (16 heads x 16 tokens) as the A operand, hi / lo ----
    uint32_t ph[4], pl[4];
    attn_split2(sc[0][0] * kPS, sc[0][1] * kPS, ph[0], pl[0]);
    attn_split2(sc[0][2] * kPS, sc[0][3] * kPS, ph[1], pl[1]);
    attn_split2(sc[1][0] * kPS, sc[1][1] * kPS, ph[2], pl[2]);
    attn_split2(sc[1][2] * kPS, sc[1][3] * kPS, ph[3], pl[3]);
    // ---- O += P.V over this warp's dims [D/2 dh, D/2 (dh + 1)) ----
    const int mi = lane >> 3, r = lane & 7;
    const int tok = min((mi & 1) * 8 + r, nr - 1);
    const uint32_t vrow =
        smem_u32(st + (16 + tok) * C::kStride + (mi >> 1) * 16) + (uint32_t)(dh * D);  // D/2 f16
#pragma unroll
    for (int dn = 0; dn < NH / 2; ++dn) {
      uint32_t v0, v1, v2, v3;
      attn_ldsm_x4_trans(vrow + dn * 32, v0, v1, v2, v3);
      attn_mma16816(o[2 * dn], ph, v0, v1);
      attn_mma16816(o[2 * dn], pl, v0, v1);
      attn_mma16816(o[2 * dn + 1], ph, v2, v3);
      attn_mma16816(o[2 * dn + 1], pl, v2, v3);
    }
  }
  // ---- the pairs' {m, l, O} merged by all 8 pair warps, output elements
  // dealt over their threads (in the order of the single-pair merge: the
  // same results); the chunk's partial written ----
  pairs_sync();  // every pair is done with its tile: each parks its state there
  float* mm = reinterpret_cast<float*>(region);  // [4][16]
  float* ll = mm + kPairs * 16;                  // [4][16]
  float* oo = ll + kPairs * 16;                  // [4][16][D]
  if (cq == 0 && dh == 0) {
    mm[pr * 16 + gq] = m0;
    mm[pr * 16 + gq + 8] = m1;
    ll[pr * 16 + gq] = l0;
    ll[pr * 16 + gq + 8] = l1;
  }
#pragma unroll
  for (int n = 0; n < NH; ++n) {
    const int col = dh * (D / 2) + 8 * n + 2 * cq;
    *reinterpret_cast<float2*>(oo + (pr * 16 + gq) * D + col) = make_float2(o[n][0], o[n][1]);
    *reinterpret_cast<float2*>(oo + (pr * 16 + gq + 8) * D + col) = make_float2(o[n][2], o[n][3]);
  }
  pairs_sync();
  float* po = P.ws_o + (size_t)item * G * D;
  for (int e = threadIdx.x; e < G * D; e += 2 * kPairs * 32) {  // (threads 0..255: the pair warps)
    const int h = e / D, d = e % D;
    float M = mm[h];
#pragma unroll
    for (int q = 1; q < kPairs; ++q) M = fmaxf(M, mm[q * 16 + h]);
    float Ls = 0.f, acc = 0.f;
#pragma unroll
    for (int q = 0; q < kPairs; ++q) {
      const float mq = mm[q * 16 + h];
      const float w = mq == -INFINITY ? 0.f : exp2f(mq - M);
      Ls = fmaf(ll[q * 16 + h], w, Ls);
      acc = fmaf(oo[(q * 16 + h) * D + d], w, acc);
    }
    po[e] = acc / kPS;
    if (d == 0) {
      P.ws_m[(size_t)item * G + h] = M;
      P.ws_l[(size_t)item * G + h] = Ls;
    }
  }
}

template <int D>
__device__ void combine_phase(const MParams& P, int L, bool len_ok, uint8_t* region) {
  // Every CTA merges a contiguous slice of the H * D outputs: a group of LW
  // lanes per output element (two elements a warp for up to 80 chunks),
  // lanes over the context chunks (loaded together, then max / sums by
  // shuffles in a fixed order), so the merge is one round of L2 loads
  // wherever it runs.
  (void)region;
  const int H = P.n_heads, Hk = P.n_kv_heads, G = H / Hk;
  const int nc = attn_chunks_for(P, L);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int LW = nc > 80 ? 32 : 16, per_warp = 32 / LW;
  const int grp = lane / LW, gl = lane % LW;
  const int total = H * D, per = (total + gridDim.x - 1) / gridDim.x;
  const int e0 = blockIdx.x * per, e1 = min(total, e0 + per);
  for (int eb = e0 + warp * per_warp; eb < e1; eb += kW * per_warp) {
    const int e = eb + grp;  // (warp-uniform loop: every lane reaches the shuffles)
    const bool live = e < e1;
    if (!len_ok) {
      if (live && gl == 0) P.attn[e] = __int_as_float(0x7fc00000);
      continue;
    }
    const int hq = live ? e / D : 0, d = live ? e % D : 0;
    const int g = hq / G, h = hq % G;
    // chunks c = gl + LW j of KV head g: (m, l, O[d]) of query head h
    constexpr int kJ = 5;  // nc <= 5 * LW (at most 160: one chunk per CTA)
    float m[kJ], l[kJ], o[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int c = gl + LW * j;
      m[j] = -INFINITY;
      l[j] = o[j] = 0.f;
      if (live && c < nc) {
        const size_t i = ((size_t)g * nc + c) * G + h;
        m[j] = ldcg(P.ws_m + i);
        l[j] = ldcg(P.ws_l + i);
        o[j] = ldcg(P.ws_o + i * D + d);
      }
    }
    float M = m[0];
#pragma unroll
    for (int j = 1; j < kJ; ++j) M = fmaxf(M, m[j]);
    for (int off = LW / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float ls = 0.f, acc = 0.f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      // (empty chunks: m = -inf, l = 0, O = 0 weigh nothing)
      const float w = m[j] == -INFINITY ? 0.f : exp2f(m[j] - M);
      ls = fmaf(l[j], w, ls);
      acc = fmaf(o[j], w, acc);
    }
    for (int off = LW / 2; off > 0; off >>= 1) {
      ls += __shfl_xor_sync(0xffffffffu, ls, off);
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    }
    if (live && gl == 0) P.attn[e] = acc / ls;
  }
}

// ---------------------------------------------------------------- argmax
// One warp: each lane loads every 32nd CTA's (value, index) pair, all loads
// in flight together, then the lanes' bests are merged by shuffles.  The
// order (larger value, then lower index) is total, so the result does not
// depend on the merge order.  Out of line: inlined, this phase changed the
// register allocation of the matvec loops (measured ~30 µs slower a 7B step).
constexpr int kAmPerLane = 8;  // up to 256 CTAs (the step refuses larger grids)
__device__ __noinline__ void argmax_phase(const MParams& P, int pos) {
  if (blockIdx.x != 0 || threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float v[kAmPerLane];
  int ix[kAmPerLane];
#pragma unroll
  for (int k = 0; k < kAmPerLane; ++k) {
    const int b = lane + 32 * k;
    const bool live = b < (int)gridDim.x;
    v[k] = live ? ldcg(P.am_val + b) : -INFINITY;
    ix[k] = live ? __ldcg(P.am_idx + b) : 0x7fffffff;
  }
  float bv = v[0];
  int bi = ix[0];
#pragma unroll
  for (int k = 1; k < kAmPerLane; ++k)
    if (am_better(v[k], ix[k], bv, bi)) {
      bv = v[k];
      bi = ix[k];
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (am_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    *P.d_token = bi;
    *P.d_pos = pos + 1;
  }
}

// ---------------------------------------------------------------- producer
// Issues every weight tile of this CTA's rows of all matvec phases, in
// order, into the ring.  Returns the number of tiles issued (fewer if a
// wait was abandoned).
// Pulls the 128-byte lines of [p, p + bytes) into L2, line j by CTA j mod
// the grid (small vectors every CTA reads right after a grid barrier).
__device__ __forceinline__ void prefetch_l2_spread(const void* p, size_t bytes) {
  if (!p || !bytes) return;
  const unsigned long long a = reinterpret_cast<unsigned long long>(p), e = a + bytes;
  for (unsigned long long l = (a >> 7) + blockIdx.x; l <= ((e - 1) >> 7); l += gridDim.x) {
    const unsigned long long q = (l << 7) > a ? (l << 7) : a;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(q) : "memory");
  }
}

__device__ __noinline__ int produce_all(const MParams& P, uint8_t* smem) {
  uint64_t* full = ms_full;
  uint64_t* empty = ms_empty;
  int* s_abort = &ms_abort;
  const uint64_t pol = policy_evict_first();
  int s = 0, issued = 0;
  uint32_t ph = 0;
  const int pos = *(volatile const int*)P.d_pos;
  const int L = pos + 1;
  const bool len_ok = pos >= 0 && L <= P.cap;
  for (int pi = 0; pi < P.nphases; ++pi) {
    const MPhase* F = P.phases + pi;
    const int kind = __ldg(&F->kind);
    if (kind == kPhAttn && len_ok) {
      // the layer's biases, QK-norm weights and this position's RoPE row
      const MLayer* Ly = P.layers + __ldg(&F->layer);
      const size_t qb = (size_t)P.n_heads * P.head_dim * 4, kb = (size_t)P.n_kv_heads * P.head_dim * 4;
      prefetch_l2_spread(ldg_ptr(&Ly->bq), qb);
      prefetch_l2_spread(ldg_ptr(&Ly->bk), kb);
      prefetch_l2_spread(ldg_ptr(&Ly->bv), kb);
      prefetch_l2_spread(ldg_ptr(&Ly->q_norm), (size_t)P.head_dim * 4);
      prefetch_l2_spread(ldg_ptr(&Ly->k_norm), (size_t)P.head_dim * 4);
      prefetch_l2_spread(P.rope_cos + (size_t)pos * (P.head_dim / 2), (size_t)P.head_dim * 2);
      prefetch_l2_spread(P.rope_sin + (size_t)pos * (P.head_dim / 2), (size_t)P.head_dim * 2);
    }
    if (kind == kPhMatvec && __ldg(&F->xmode) == kXRmsNorm)
      prefetch_l2_spread(ldg_ptr(&F->xw), (size_t)__ldg(&F->n) * 4);  // the RMSNorm weights
    if (kind == kPhAttn && P.pf_permille > 0) {
      // Through the short phases that follow (attention, combine, o: their
      // weight tiles are in the ring by now) the ring is full and HBM idles:
      // pull the first share of this CTA's rows of the next gate|up phase
      // (both matrices) into L2 meanwhile, so that phase starts partly from
      // L2.
      for (int k = 1; k <= 4 && pi + k < P.nphases; ++k) {
        const MPhase* G = F + k;
        if (__ldg(&G->kind) != kPhMatvec || !__ldg(&G->glu)) continue;
        if (!__ldg(&G->tc)) break;  // (tensor-core phases only: measured there)
        const int rpc_g = __ldg(&G->rows_per_cta), nr0 = __ldg(&G->vbegin[1]);
        const long long rb = __ldg(&G->row_bytes);
        const int v0 = blockIdx.x * rpc_g, v1 = min(nr0, v0 + rpc_g);
        if (v0 < v1) {
          const long long want = (long long)(v1 - v0) * rb * P.pf_permille / 1000;
          for (int sg = 0; sg < 2; ++sg) {
            // bulk prefetches take 16-byte aligned ranges: the start rounded
            // down and the end rounded down stay inside the matrix (its base
            // is 16-byte aligned)
            const uintptr_t b0 = reinterpret_cast<uintptr_t>(ldg_ptr(&G->w[sg])) + (uintptr_t)(v0 * rb);
            const uintptr_t s0 = b0 & ~(uintptr_t)15, e0 = (b0 + (uintptr_t)want) & ~(uintptr_t)15;
            for (uintptr_t a = s0; a < e0; a += 32768) {
              const uint32_t n = (uint32_t)min((uintptr_t)32768, e0 - a);
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(n) : "memory");
            }
          }
        }
        break;
      }
    }
    if (kind == kPhAttn && len_ok && (int)blockIdx.x < attn_chunks_for(P, L)) {
      // pull context chunk c's K/V rows (all KV heads: whole cache rows,
      // contiguous; the rows before the new one) into L2 now, a phase or
      // more before the attention phase reads them: the CTA of chunk c and
      // KV head 0 does it for the chunk's CTAs of every head, in a few large
      // requests
      const int nc = attn_chunks_for(P, L);
      const int c = blockIdx.x;
      const int T = (L + nc - 1) / nc;
      const int t0 = c * T, t1 = min(L - 1, t0 + T);
      if (t1 > t0) {
        const MLayer* Ly = P.layers + __ldg(&F->layer);
        const uint8_t* kc = reinterpret_cast<const uint8_t*>(ldg_ptr(&Ly->kcache));
        const uint8_t* vc = reinterpret_cast<const uint8_t*>(ldg_ptr(&Ly->vcache));
        const long long stride = (long long)P.head_dim * P.kv_esize * P.n_kv_heads;  // a cache row
        const long long a = (long long)t0 * stride, bytes = (long long)(t1 - t0) * stride;
        for (long long o = 0; o < bytes; o += 32768) {
          const uint32_t n = (uint32_t)min(32768LL, bytes - o);  // (rows are 16-byte multiples)
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kc + a + o), "r"(n)
                       : "memory");
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vc + a + o), "r"(n)
                       : "memory");
        }
      }
      continue;
    }
    if (kind != kPhMatvec) continue;
    const int nseg = __ldg(&F->nseg), R = __ldg(&F->R), rpc = __ldg(&F->rows_per_cta);
    const int total = __ldg(&F->total_rows), glu = __ldg(&F->glu);
    const long long rowb = __ldg(&F->row_bytes);
    if (__ldg(&F->tc)) {
      // tiles of T sets of 8 rows (fewer at the end of a range); a set is
      // groups of consecutive rows, one bulk copy per group (per row where
      // a group crosses into the next matrix); rows are 16-byte multiples
      // at 16-byte aligned addresses (n % 256 == 0)
      const uint32_t SR = (uint32_t)__ldg(&F->SR);
      const int gsh = __ldg(&F->gsh), gsz = 1 << gsh, T = __ldg(&F->T);
      const uint32_t gbytes = (uint32_t)(gsz * rowb) + 16u;
      for (int piece = 0; piece < (glu ? 2 : 1); ++piece) {
        int v0, v1;
        piece_range(glu, __ldg(&F->vbegin[1]), rpc, total, piece, v0, v1);
        int seg = 0;
        while (seg + 1 < nseg && v0 >= __ldg(&F->vbegin[seg + 1])) ++seg;
        int seg_beg = __ldg(&F->vbegin[seg]), seg_end = __ldg(&F->vbegin[seg + 1]);
        const uint8_t* wseg = ldg_ptr(&F->w[seg]);
        for (int r0 = v0; r0 < v1; r0 += 8 * T) {
          if (issued >= P.nstages && !wait_or_abort(&empty[s], ph ^ 1u, s_abort)) return issued;
          const int nrows = min(8 * T, v1 - r0);
          uint8_t* dst = smem + (size_t)P.stage_bytes * s;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(nrows * rowb));
          for (int a = 0; a < nrows; a += gsz) {
            const int b = min(a + gsz, nrows);
            uint8_t* gd = dst + (a >> 3) * SR + ((a & 7) >> gsh) * gbytes;
            for (int r = a; r < b;) {
              const int vr = r0 + r;
              while (vr >= seg_end) {  // (the next matrix of the phase)
                ++seg;
                seg_beg = seg_end;
                seg_end = __ldg(&F->vbegin[seg + 1]);
                wseg = ldg_ptr(&F->w[seg]);
              }
              const int nr = min(b, r + (seg_end - vr)) - r;
              bulk_g2s(gd + (r - a) * rowb, wseg + (long long)(vr - seg_beg) * rowb,
                       (uint32_t)(nr * rowb), &full[s], pol);
              r += nr;
            }
          }
          ++issued;
          if (++s == P.nstages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      continue;
    }
    for (int piece = 0; piece < (glu ? 2 : 1); ++piece) {
    int v0, v1;
    piece_range(glu, __ldg(&F->vbegin[1]), rpc, total, piece, v0, v1);
    int cur = v0, seg = 0;
    while (seg + 1 < nseg && v0 >= __ldg(&F->vbegin[seg + 1])) ++seg;
    int r0 = v0 - __ldg(&F->vbegin[seg]);
    int seg_end = __ldg(&F->vbegin[seg + 1]);
    while (cur < v1) {
      if (issued >= P.nstages && !wait_or_abort(&empty[s], ph ^ 1u, s_abort)) return issued;
      const int rows = min(R, min(seg_end, v1) - cur);
      const uint8_t* w = ldg_ptr(&F->w[seg]);
      const long long segp = seg_end - __ldg(&F->vbegin[seg]);
      const long long start = (long long)r0 * rowb;
      const long long end = start + (long long)rows * rowb;
      const long long cap16 = (segp * rowb) & ~15LL;
      const long long a0 = start & ~15LL;
      long long a1 = (end + 15) & ~15LL;
      uint8_t* dst = smem + (size_t)P.stage_bytes * s;
      if (a1 > cap16) {
        a1 = cap16 > a0 ? cap16 : a0;
        for (long long o = a1; o < end; ++o) dst[o - a0] = __ldg(w + o);
      }
      const uint32_t bytes = (uint32_t)(a1 - a0);
      mbar_arrive_expect_tx(&full[s], bytes);
      if (bytes) bulk_g2s(dst, w + a0, bytes, &full[s], pol);
      cur += rows;
      r0 += rows;
      if (cur == seg_end && seg + 1 < nseg) {
        ++seg;
        r0 = 0;
        seg_end = __ldg(&F->vbegin[seg + 1]);
      }
      ++issued;
      if (++s == P.nstages) {
        s = 0;
        ph ^= 1u;
      }
    }
    }
  }
  return issued;
}

// ---------------------------------------------------------------- kernel
template <int D, typename KT>
__global__ void __launch_bounds__(kMsThreads, 1) q8_step_kernel(const MParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) MPhase s_ph2[2];  // this phase's record and the next one's
  __shared__ float s_f[kW];
  __shared__ int s_i[kW];
  uint8_t* region = smem + (size_t)P.stage_bytes * P.nstages;  // 128-byte aligned
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nstages; ++s) {
      mbar_init(&ms_full[s], 1);
      mbar_init(&ms_empty[s], kW);
    }
    ms_abort = 0;
    ms_target = 0;
    ms_spin = *(volatile const unsigned*)P.wait_limit;
    fence_barrier_init();
  }
  __syncthreads();

  int issued = 0;
  if (warp == kW) {
    // ---- producer warp ----
    if (lane == 0) issued = produce_all(P, smem);
  } else {
    // ---- consumers ----
    // the step's position: read once, kept in shared memory (fewer live
    // registers across the phases)
    if (threadIdx.x == 0) ms_L = *(volatile const int*)P.d_pos + 1;
    consumer_sync(kCT);
    RingPos rp{0, 0u, smem_u32(smem)};
    const uint32_t smem32 = smem_u32(smem);
    // phase records come in by cp.async a phase ahead (16 bytes a thread)
    constexpr int kRecChunks = (int)(sizeof(MPhase) / 16);
    static_assert(sizeof(MPhase) % 16 == 0, "phase records are whole 16-byte chunks");
    if (threadIdx.x < kRecChunks)
      cp_async16(reinterpret_cast<uint8_t*>(&s_ph2[0]) + 16 * threadIdx.x,
                 reinterpret_cast<const uint8_t*>(P.phases) + 16 * threadIdx.x);
    for (int pi = 0; pi < P.nphases; ++pi) {
      if (pi > 0) grid_arrive(P);
      if (threadIdx.x < kRecChunks) cp_async_wait_all();
      consumer_sync(kCT);
      MPhase& s_ph = s_ph2[pi & 1];
      if (pi + 1 < P.nphases && threadIdx.x < kRecChunks)
        cp_async16(reinterpret_cast<uint8_t*>(&s_ph2[(pi + 1) & 1]) + 16 * threadIdx.x,
                   reinterpret_cast<const uint8_t*>(P.phases + pi + 1) + 16 * threadIdx.x);
      const int kind = s_ph.kind;
      if (kind == kPhMatvec) matvec_pre(s_ph, region);
      if (pi > 0 && !grid_wait(P)) break;
      if (kind == kPhMatvec) {
        const bool ok = s_ph.tc ? tc_matvec_phase(s_ph, P, rp, smem32, region, s_f, s_i)
                                : matvec_phase(s_ph, P, rp, smem32, region, s_f, s_i);
        if (!ok) ms_abort = 1;  // seen at the next grid barrier
      } else if (kind == kPhAttn) {
        const int L = ms_L;
        if constexpr (std::is_same<KT, __half>::value)
          attn_phase_mma<D>(P, s_ph, L, L >= 1 && L <= P.cap, region);
        else
          attn_phase<D, KT>(P, s_ph, L, L >= 1 && L <= P.cap, region);
      } else if (kind == kPhCombine) {
        const int L = ms_L;
        combine_phase<D>(P, L, L >= 1 && L <= P.cap, region);
      } else if (kind == kPhEmbed) {
        const int L = ms_L;
        embed_phase(P, *(volatile const int*)P.d_token, L >= 1 && L <= P.cap);
      } else {
        argmax_phase(P, ms_L - 1);
      }
    }
    if (ms_abort && threadIdx.x == 0) {
      atomicExch(P.abort, 1);
      if (P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
    }
  }
  __syncthreads();
  if (warp == kW && lane == 0 && ms_abort) {
    // the step was abandoned: tiles issued but never consumed may still be
    // in flight; wait (bounded) for the last copy of every stage before the
    // CTA's shared memory is released
    for (int j = max(0, issued - P.nstages); j < issued; ++j)
      mbar_wait(&ms_full[j % P.nstages], (uint32_t)(j / P.nstages) & 1u);
  }
}

template <int D, typename KT>
int launch_typed(const MParams& P, int grid, cudaStream_t st) {
  auto fn = q8_step_kernel<D, KT>;
  const size_t smem = megastep_smem(P);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return record_cuda(e);
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kMsThreads, smem);
  if (e != cudaSuccess) return record_cuda(e);
  if (occ < 1) return Q8D_EUNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kMsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fn, P);
  return e == cudaSuccess ? Q8D_OK : record_cuda(e);
}

}  // namespace

int megastep_plan_tc(MPhase& F, int grid) {
  F.bpr = F.n / kQBlock;
  F.row_bytes = (long long)F.bpr * kQBlockBytes;
  F.tc = 0;
  if (F.n % 256 || F.bpr < 32 || F.bpr * 8 > kTcItems * kCT) return 0;
  // sets of bank-spread row groups (tc::row_group_shift)
  F.gsh = tc::row_group_shift(F.bpr / 8);
  F.SR = (int)(8 * F.row_bytes + 16 * (8 >> F.gsh));
  // two sets a tile when three such stages fit the ring, else one
  F.T = 3LL * ((2LL * F.SR + 127) / 128 * 128) <= megastep_ring_bytes() ? 2 : 1;
  const long long tile = ((long long)F.T * F.SR + 127) / 128 * 128;
  if (tile > megastep_ring_bytes() / 3) return 0;
  const long long frag = (long long)F.bpr * (tc::kXfBlock + 4) + tc::kZeroPad;
  const long long per_tile = 2LL * F.T * tc::kSetRows * kW * 4;  // double-buffered partials
  if (frag + per_tile > kMsRegion) return 0;
  const int total = F.vbegin[F.nseg];
  const int rpc = F.glu ? (F.vbegin[1] + grid - 1) / grid : (total + grid - 1) / grid;
  // Rows of 32 blocks give a 16-row tile only 8 unit pairs for the 20
  // warps: on the tensor cores they pay off in short phases (a few tiles a
  // CTA, latency-bound) but not in long ones (the Qwen3-0.6B lm_head, 1000
  // rows a CTA, streamed 2.4x slower than on the CUDA cores).
  if (F.bpr < 64 && rpc > 128) return 0;
  F.tc = 1;
  F.win = (int)std::min<long long>(8, (kMsRegion - frag) / per_tile);
  F.total_rows = total;
  F.rows_per_cta = rpc;
  return (int)tile;
}

bool megastep_plan_matvec(MPhase& F, int grid, int stage_target) {
  F.bpr = F.n / kQBlock;
  F.row_bytes = (long long)F.bpr * kQBlockBytes;
  F.paired = F.bpr > 32 ? 1 : 0;
  F.NS = F.paired ? 2 * ((F.bpr + 63) / 64) : 1;
  if (F.NS > kMsWarps) return false;
  F.RG = kMsWarps / F.NS;
  // R = RG * k rows (each warp takes k rows of a tile), k the largest up to
  // 8 within the stage target that still gives every CTA at least two
  // tiles of the phase
  const long long rows_cta = F.glu ? ((long long)F.vbegin[1] + grid - 1) / grid * 2
                                   : ((long long)F.vbegin[F.nseg] + grid - 1) / grid;
  int k = 8;
  while (k > 1 && ((long long)F.RG * k * F.row_bytes + 32 > stage_target ||
                   rows_cta < 2LL * F.RG * k))
    --k;
  F.R = F.RG * k;
  // window tiles: double-buffered partials within the shared region
  const long long per_tile = 2LL * F.R * F.NS * kPW * 4;
  if (per_tile > kMsRegion) return false;
  F.win = (int)std::max<long long>(1, kMsRegion / per_tile);
  F.total_rows = F.vbegin[F.nseg];
  F.rows_per_cta = F.glu ? (F.vbegin[1] + grid - 1) / grid : (F.total_rows + grid - 1) / grid;
  return true;
}

// dynamic shared memory per CTA (one CTA per SM; the rest is static)
constexpr int kMsDynamicBudget = 224 * 1024;

int megastep_ring_bytes() { return kMsDynamicBudget - kMsRegion; }

int megastep_max_stages(int stage_bytes) { return megastep_ring_bytes() / stage_bytes; }

size_t megastep_smem(const MParams& P) {
  return (size_t)P.stage_bytes * P.nstages + kMsRegion;
}

int megastep_launch(const MParams& P, int head_dim, int kv_dtype, int grid, cudaStream_t st) {
  if (head_dim == 128)
    return kv_dtype == Q8D_KV_F16 ? launch_typed<128, __half>(P, grid, st)
                                  : launch_typed<128, float>(P, grid, st);
  if (head_dim == 64)
    return kv_dtype == Q8D_KV_F16 ? launch_typed<64, __half>(P, grid, st)
                                  : launch_typed<64, float>(P, grid, st);
  return Q8D_EUNSUPPORTED;
}

}  // namespace q8d
