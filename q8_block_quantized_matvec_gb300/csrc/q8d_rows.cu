// Q8_0 matrix-vector and small-M products on CUDA cores (sm_103a).
//
// Computes, for up to three Q8_0 matrices that share the same activations,
//   Y[i][r] (+)= sum_b scale(r,b) * sum_j q(r,b,j) * X[i][32b+j]
// ("IV.4: One command buffer per token", "Eight kernels": q8_matvec; the
// batched form is "Metal Backend Optimizations"' nt in [2, 8] matvec).
// A single vector (m == 1) goes to the matvec kernel of q8d_gemv.cu when its
// rows fit it; this kernel serves several vectors and very long rows.
//
// Design for GB300 (the pages' kernel gives one 32-lane SIMD-group per
// output row with scalar byte loads; that shape would leave HBM idle here):
//  * Weight bytes are streamed by the TMA engine: each CTA walks a list of
//    tiles (R whole rows = one contiguous byte range of the 34-byte block
//    stream) through an NSTAGE-deep ring of shared-memory stages filled with
//    1-D cp.async.bulk copies that complete on an mbarrier.  Blocks are only
//    2-byte aligned, so the copy starts at the 16-byte boundary below the
//    tile and the kernel indexes from the remainder.
//  * A warp owns a segment of 32*K block columns of a row; lane l owns
//    columns l, l+32, ... of that segment, so its activations stay in
//    registers for every row it visits and each weight byte is read from
//    shared memory exactly once.
//  * Dequantisation is integer-free of I2F: a quant byte (sign-flipped) is
//    placed in the mantissa of 2^23 with one PRMT, one packed f32x2 add
//    removes the bias exactly, and packed f32x2 FMAs do the dot product.
//    The block sum is scaled by the f16 scale once per block.
//  * Per-row partials of the warps covering a row are reduced in a fixed
//    order (warp shuffle, then shared memory), so results are deterministic.
#include <algorithm>
#include <cstdio>

#include "q8d_internal.cuh"
#include "q8d_rows.cuh"

namespace q8d {

namespace {

constexpr int kWarpsSmall = 8;   // warps per CTA

// Decodes the 32 quants of the block at byte offset `o` of the 4-byte
// aligned shared buffer `s32` into 16 packed f32x2 pairs, and returns the
// block's scale.  o is even; bytes o..o+33 are the block.
__device__ __forceinline__ float decode_block(const uint32_t* __restrict__ s32, uint32_t o,
                                              uint64_t (&q2)[16]) {
  const uint32_t wi = o >> 2;
  const bool odd = (o & 2u) != 0;
  uint32_t a[9];
#pragma unroll
  for (int k = 0; k < 9; ++k) a[k] = s32[wi + k];
  const uint32_t sbits = odd ? (a[0] >> 16) : (a[0] & 0xFFFFu);
  const uint32_t sh = odd ? 32u : 16u;
  const uint64_t bias2 = pack2(-kMagicBias, -kMagicBias);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t w = __funnelshift_rc(a[k], a[k + 1], sh) ^ 0x80808080u;
    const float f0 = magic_byte(w, magic_sel(0));
    const float f1 = magic_byte(w, magic_sel(1));
    const float f2 = magic_byte(w, magic_sel(2));
    const float f3 = magic_byte(w, magic_sel(3));
    q2[2 * k] = add2(pack2(f0, f1), bias2);
    q2[2 * k + 1] = add2(pack2(f2, f3), bias2);
  }
  return f16_bits_to_f32(sbits);
}

// sum_j q_j x_j over one block with four independent f32x2 chains.
__device__ __forceinline__ float block_dot(const uint64_t (&q2)[16], const uint64_t (&x2)[16]) {
  uint64_t c0 = pack2(0.f, 0.f), c1 = c0, c2 = c0, c3 = c0;
#pragma unroll
  for (int j = 0; j < 16; j += 4) {
    c0 = fma2(q2[j], x2[j], c0);
    c1 = fma2(q2[j + 1], x2[j + 1], c1);
    c2 = fma2(q2[j + 2], x2[j + 2], c2);
    c3 = fma2(q2[j + 3], x2[j + 3], c3);
  }
  const uint64_t s = add2(add2(c0, c1), add2(c2, c3));
  float lo, hi;
  unpack2(s, lo, hi);
  return lo + hi;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Loads the activation pairs of vectors v0..v0+MV-1 for block columns
// seg*32K + k*32 + lane into registers (zeros past the row end / m).
template <int K, int MV>
__device__ __forceinline__ void load_x(const RowsParams& P, int v0, int seg, int lane,
                                       uint64_t (&xr)[MV][K][16]) {
#pragma unroll
  for (int i = 0; i < MV; ++i) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int b = seg * 32 * K + k * 32 + lane;
      const bool ok = (v0 + i < P.m) && (b < P.bpr);
      const size_t base = (size_t)(v0 + i) * P.ldx + (size_t)b * kQBlock;
      const float4* xp = reinterpret_cast<const float4*>(P.X + base);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float4 v = ok ? __ldg(xp + t) : make_float4(0.f, 0.f, 0.f, 0.f);
        xr[i][k][2 * t] = pack2(v.x, v.y);
        xr[i][k][2 * t + 1] = pack2(v.z, v.w);
      }
    }
  }
}

// Bounded wait that gives up at once when another warp of the CTA already
// gave up (so every warp still reaches the CTA's barriers quickly).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// One tile of the CTA's contiguous row range: rows [r0, r0 + rows) of
// segment `seg`, which are rows [vrow0, vrow0 + rows) of the CTA.
struct Tile {
  int seg, rows, vrow0;
  long long r0;
};

__device__ __forceinline__ Tile tile_at(const RowsParams& P, long long cur, long long v0,
                                        long long v1) {
  Tile t;
  int sg = 0;
  while (sg + 1 < P.nseg && cur >= P.vbegin[sg + 1]) ++sg;
  t.seg = sg;
  t.r0 = cur - P.vbegin[sg];
  const long long seg_end = P.vbegin[sg] + P.seg[sg].p;
  t.rows = (int)min((long long)P.rows_per_tile, min(seg_end, v1) - cur);
  t.vrow0 = (int)(cur - v0);
  return t;
}

// Streaming kernel: lane 0 of warp 0 fills a ring of stages with bulk
// copies (recycled through per-stage "empty" barriers that every warp
// arrives on); all warps consume.  Each CTA owns a contiguous range of output rows;
// per-(row, segment) partials wait in shared memory and are reduced in a
// fixed order once, at the end, so no CTA-wide barrier runs per tile.
template <int MV, int W>
__global__ void __launch_bounds__(W * 32, MV >= 4 ? 1 : 2)
    q8_rows_kernel(const RowsParams P) {
  constexpr int K = 1;
  constexpr int kWarps = W;
  constexpr int kThreads = W * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = P.segs_per_row;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)P.stage_bytes * P.nstages);
  uint64_t* empty = full + P.nstages;
  float* part = reinterpret_cast<float*>(empty + P.nstages);  // [rows_cta][NS][m]

  const long long v0 = (long long)blockIdx.x * P.rows_per_cta;
  const long long v1 = min(P.total_rows, v0 + P.rows_per_cta);
  const int rows_cta = (int)max(0LL, v1 - v0);

  __shared__ int s_abort;
  // Launched as a programmatic dependent: the next kernel may start its
  // prologue now; this one waits for the previous kernel before it reads
  // anything or writes y.
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  griddep_wait();
  __syncthreads();

  bool ok = true;
  // Producer state (lane 0 of warp 0): next tile index and its first row.
  // A stage is refilled as soon as every warp has released it, so up to
  // nstages tiles are in flight while the warps compute.
  long long pcur = v0;
  int pi = 0;
  const uint64_t pol = policy_evict_first();
  auto produce = [&](int upto) {
    while (pi < upto && pcur < v1) {
      const Tile t = tile_at(P, pcur, v0, v1);
      const int s = pi % P.nstages;
      if (pi >= P.nstages && !wait_or_abort(&empty[s], (uint32_t)((pi / P.nstages) - 1) & 1u, &s_abort)) {
        ok = false;
        pcur = v1;  // stop producing
        return;
      }
      const RowSeg& S = P.seg[t.seg];
      const long long start = t.r0 * P.row_bytes, end = (t.r0 + t.rows) * P.row_bytes;
      const long long total = (long long)S.p * P.row_bytes;
      const long long a0 = start & ~15LL;
      long long a1 = (end + 15) & ~15LL;
      const long long cap16 = total & ~15LL;
      uint8_t* dst = smem + (size_t)P.stage_bytes * s;
      if (a1 > cap16) {
        // Last tile of a matrix whose byte size is not a multiple of 16:
        // the final bytes are copied by hand before the arrive publishes them.
        a1 = cap16 > a0 ? cap16 : a0;
        for (long long o = a1; o < end; ++o) dst[o - a0] = __ldg(S.w + o);
      }
      const uint32_t bytes = (uint32_t)(a1 - a0);
      mbar_arrive_expect_tx(&full[s], bytes);
      if (bytes) bulk_g2s(dst, S.w + a0, bytes, &full[s], pol);
      pcur += t.rows;
      ++pi;
    }
  };
  const bool producer = (warp == 0 && lane == 0);
  if (producer) produce(P.nstages);
  {
    // ---------------- consumers ----------------
    const bool x_static = (NS <= kWarps) && (P.m <= MV);
    const int RG = NS <= kWarps ? kWarps / NS : 1;
    const int my_seg0 = NS <= kWarps ? warp % NS : warp;
    const int seg_step = NS <= kWarps ? NS : kWarps;
    const int my_rg = NS <= kWarps ? warp / NS : 0;
    const bool active = (NS <= kWarps) ? (warp < NS * RG) : true;

    uint64_t xr[MV][K][16];
    if (x_static && active) load_x<K, MV>(P, 0, my_seg0, lane, xr);

    {
    long long cur = v0;
    for (int i = 0; cur < v1; ++i) {
      const Tile t = tile_at(P, cur, v0, v1);
      const int s = i % P.nstages;
      if (!mbar_wait(&full[s], (uint32_t)(i / P.nstages) & 1u)) {
        ok = false;
        break;
      }
      if (active) {
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(smem + (size_t)P.stage_bytes * s);
        const uint32_t delta = (uint32_t)((t.r0 * P.row_bytes) & 15LL);
        const int first = ((my_rg - t.vrow0) % RG + RG) % RG;
        for (int v0m = 0; v0m < P.m; v0m += MV) {
          for (int seg = my_seg0; seg < NS; seg += seg_step) {
            if (!x_static) load_x<K, MV>(P, v0m, seg, lane, xr);
            for (int rl = first; rl < t.rows; rl += RG) {
              float acc[MV];
#pragma unroll
              for (int m = 0; m < MV; ++m) acc[m] = 0.f;
#pragma unroll
              for (int k = 0; k < K; ++k) {
                const int b = seg * 32 * K + k * 32 + lane;
                const uint32_t o =
                    delta + (uint32_t)(rl * P.bpr + (b < P.bpr ? b : P.bpr - 1)) * kQBlockBytes;
                uint64_t q[16];
                const float sc = decode_block(s32, o, q);
#pragma unroll
                for (int m = 0; m < MV; ++m) acc[m] = fmaf(sc, block_dot(q, xr[m][k]), acc[m]);
              }
#pragma unroll
              for (int m = 0; m < MV; ++m) {
                const float v = warp_sum(acc[m]);
                if (lane == 0 && v0m + m < P.m)
                  part[((size_t)(t.vrow0 + rl) * NS + seg) * P.m + v0m + m] = v;
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (producer) produce(i + 1 + P.nstages);
      cur += t.rows;
    }
    }
  }

  // ---- reduce the segment partials of each (row, vector) in order ----
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
    return;
  }
  for (int e = threadIdx.x; e < rows_cta * P.m; e += kThreads) {
    const int rc = e / P.m, m = e % P.m;
    float sum = 0.f;
    for (int seg = 0; seg < NS; ++seg) sum += part[((size_t)rc * NS + seg) * P.m + m];
    const long long vr = v0 + rc;
    int sg = 0;
    while (sg + 1 < P.nseg && vr >= P.vbegin[sg + 1]) ++sg;
    P.seg[sg].y[(size_t)m * P.ldy + (vr - P.vbegin[sg])] = sum;
  }
}

__global__ void fill_zero_kernel(float* y, int ldy, int m, int p) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < (long long)m * p;
       e += (long long)gridDim.x * blockDim.x)
    y[(e / p) * ldy + (e % p)] = 0.f;
}

template <int MV, int W>
int launch_rows(RowsParams P, long long R, cudaStream_t stream, int* grid_out) {
  auto fn = q8_rows_kernel<MV, W>;
  constexpr int kThreads = W * 32;
  const int rc = configure_kernel(reinterpret_cast<const void*>(fn), 200 * 1024, true);
  if (rc) return rc;
  // One wave of resident CTAs, each owning a contiguous row range.
  const int sms = sm_count();
  const long long p_total = P.total_rows;
  auto smem_for = [&](long long rows_cta) {
    const long long part = rows_cta * P.segs_per_row * P.m;
    return (long long)P.stage_bytes * P.nstages + 16LL * P.nstages + 4LL * part;
  };
  long long smem = smem_for((p_total + sms - 1) / sms);
  if (smem > 200 * 1024) return Q8D_EUNSUPPORTED;
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, (size_t)smem);
  if (e != cudaSuccess) return record_cuda(e);
  occ = std::max(occ, 1);
  long long grid = std::min<long long>(p_total, (long long)sms * occ);
  long long rows_cta = (p_total + grid - 1) / grid;
  grid = (p_total + rows_cta - 1) / rows_cta;
  P.rows_per_cta = rows_cta;
  P.rows_per_tile = (int)std::min<long long>(R, rows_cta);
  smem = smem_for(rows_cta);
  if (grid_out) *grid_out = (int)grid;
  return launch_ex(fn, dim3((unsigned)grid), dim3(kThreads), (size_t)smem, stream, true, P);
}

}  // namespace

int rows_plan_and_launch(RowsParams P, cudaStream_t stream, int* grid_out) {
  if (P.m <= 0) return Q8D_OK;
  long long p_total = 0;
  for (int s = 0; s < P.nseg; ++s) {
    P.vbegin[s] = p_total;
    p_total += P.seg[s].p;
  }
  if (p_total == 0) return Q8D_OK;
  if (P.n == 0) {
    for (int s = 0; s < P.nseg; ++s) {
      if (!P.seg[s].p) continue;
      fill_zero_kernel<<<std::min(1024, (P.m * P.seg[s].p + 255) / 256), 256, 0, stream>>>(
          P.seg[s].y, P.ldy, P.m, P.seg[s].p);
      int rc = check_launch();
      if (rc) return rc;
    }
    return Q8D_OK;
  }
  P.bpr = P.n / kQBlock;
  P.row_bytes = (long long)P.bpr * kQBlockBytes;
  P.total_rows = p_total;
  if (P.m == 1) {
    int rc = gemv_mma_plan_and_launch(P, stream, grid_out);
    if (rc != Q8D_EUNSUPPORTED) return rc;
    rc = gemv_plan_and_launch(P, stream, grid_out);
    if (rc != Q8D_EUNSUPPORTED) return rc;
  } else if (P.m <= 8 && P.nseg == 1) {
    // the activation rows in one launch of the tensor-core matvec (each
    // decoded weight block shared by the rows' MMAs) if the shape and the
    // rows' fragments suit it, else in two launches of up to four rows
    int rc = gemv_mma_plan_and_launch(P, stream, grid_out);
    if (rc != Q8D_EUNSUPPORTED) return rc;
    if (P.m > 4) {
      RowsParams Q = P;
      Q.m = 4;
      rc = gemv_mma_plan_and_launch(Q, stream, grid_out);
      if (rc != Q8D_EUNSUPPORTED) {
        if (rc) return rc;
        Q.m = P.m - 4;
        Q.X = P.X + 4LL * P.ldx;
        Q.seg[0].y = P.seg[0].y + 4LL * P.ldy;
        return gemv_mma_plan_and_launch(Q, stream, grid_out);
      }
    }
  }

  // Several activation vectors (or a row too long for the matvec kernel):
  // one 32-block segment of a row per warp (lane l owns block column l of
  // it), 8-warp CTAs.  Rows of up to 8 segments keep the activations in
  // registers; longer rows reload them per segment and tile.
  const int NS = (P.bpr + 31) / 32;
  // activation rows held in registers per pass (four: one CTA per SM, up
  // to 255 registers a thread; each block is decoded once for all of them)
  const int MV = P.m == 1 ? 1 : (P.m == 2 ? 2 : 4);
  P.segs_per_row = NS;
  constexpr int W = kWarpsSmall;

  // Stages of ~36 KB of whole rows (quads per row group where they fit).
  const int RG = NS <= W ? W / NS : 1;
  long long R = std::max<long long>(1, 36864 / P.row_bytes);
  if (R >= 4 * RG) R -= R % (4 * RG);
  else if (R >= 2 * RG) R -= R % (2 * RG);
  P.stage_bytes = (int)(((R * P.row_bytes + 32 + 127) / 128) * 128);
  const int ring = W == kWarpsSmall ? 96 * 1024 : 160 * 1024;  // per-CTA stage budget
  P.nstages = std::max(2, std::min(8, ring / P.stage_bytes));
  if (MV == 1) return launch_rows<1, kWarpsSmall>(P, R, stream, grid_out);
  if (MV == 2) return launch_rows<2, kWarpsSmall>(P, R, stream, grid_out);
  return launch_rows<4, kWarpsSmall>(P, R, stream, grid_out);
}

}  // namespace q8d
