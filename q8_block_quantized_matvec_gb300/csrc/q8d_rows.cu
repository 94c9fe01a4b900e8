// Q8_0 matrix-vector and small-M products on CUDA cores (sm_103a).
//
// Computes, for up to three Q8_0 matrices that share the same activations,
//   Y[i][r] (+)= sum_b scale(r,b) * sum_j q(r,b,j) * X[i][32b+j]
// ("IV.4: One command buffer per token", "Eight kernels": q8_matvec; the
// batched form is "Metal Backend Optimizations"' nt in [2, 8] matvec).
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

constexpr int kWarps = 8;        // warps per CTA
constexpr int kThreads = kWarps * 32;

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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Loads the activation pairs of `m_here` vectors for block columns
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
      const float4* xp =
          reinterpret_cast<const float4*>(P.X + (size_t)(v0 + i) * P.ldx + (size_t)b * kQBlock);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        float4 v = ok ? __ldg(xp + t) : make_float4(0.f, 0.f, 0.f, 0.f);
        xr[i][k][2 * t] = pack2(v.x, v.y);
        xr[i][k][2 * t + 1] = pack2(v.z, v.w);
      }
    }
  }
}

template <int K, int MV>
__global__ void __launch_bounds__(kThreads) q8_rows_kernel(const RowsParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = P.segs_per_row;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)P.stage_bytes * P.nstages);
  float* part = reinterpret_cast<float*>(full + P.nstages);  // [2][R][NS][MV]
  const int part_stride = P.rows_per_tile * NS * MV;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nstages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t pol = policy_evict_first();

  // Producer (thread 0): fill stage i % nstages with this CTA's i-th tile.
  auto issue = [&](int i) {
    const int t = blockIdx.x + i * gridDim.x;
    if (t >= P.total_tiles) return;
    int sg = 0;
    while (sg + 1 < P.nseg && t >= P.seg[sg + 1].tile_begin) ++sg;
    const RowSeg& S = P.seg[sg];
    const long long r0 = (long long)(t - S.tile_begin) * P.rows_per_tile;
    const long long r1 = min((long long)S.p, r0 + P.rows_per_tile);
    const long long start = r0 * P.row_bytes, end = r1 * P.row_bytes;
    const long long total = (long long)S.p * P.row_bytes;
    const long long a0 = start & ~15LL;
    long long a1 = (end + 15) & ~15LL;
    const long long cap16 = total & ~15LL;
    uint8_t* dst = smem + (size_t)P.stage_bytes * (i % P.nstages);
    if (a1 > cap16) {
      // Last tile of a matrix whose byte size is not a multiple of 16: the
      // final few bytes are copied by hand (generic proxy), before the
      // arrive that publishes the stage.
      a1 = cap16 > a0 ? cap16 : a0;
      for (long long o = a1; o < end; ++o) dst[o - a0] = __ldg(S.w + o);
    }
    const uint32_t bytes = (uint32_t)(a1 - a0);
    uint64_t* bar = &full[i % P.nstages];
    mbar_arrive_expect_tx(bar, bytes);
    if (bytes) bulk_g2s(dst, S.w + a0, bytes, bar, pol);
  };

  if (threadIdx.x == 0)
    for (int i = 0; i < P.nstages; ++i) issue(i);

  // Ownership of (segment, rows) inside a tile.
  const bool x_static = (NS <= kWarps) && (P.m <= MV);
  const int RG = NS <= kWarps ? kWarps / NS : 1;
  const int my_seg0 = NS <= kWarps ? warp % NS : warp;
  const int seg_step = NS <= kWarps ? NS : kWarps;   // only used when NS > kWarps
  const int my_rg = NS <= kWarps ? warp / NS : 0;
  const bool active_warp = (NS <= kWarps) ? (warp < NS * RG) : true;

  uint64_t xr[MV][K][16];
  if (x_static && active_warp) load_x<K, MV>(P, 0, my_seg0, lane, xr);

  for (int i = 0;; ++i) {
    const int t = blockIdx.x + i * gridDim.x;
    if (t >= P.total_tiles) break;
    int sg = 0;
    while (sg + 1 < P.nseg && t >= P.seg[sg + 1].tile_begin) ++sg;
    const RowSeg& S = P.seg[sg];
    const long long r0 = (long long)(t - S.tile_begin) * P.rows_per_tile;
    const int rows = (int)min((long long)P.rows_per_tile, (long long)S.p - r0);
    const int stage = i % P.nstages;
    const uint32_t parity = (uint32_t)(i / P.nstages) & 1u;
    const bool ok = mbar_wait(&full[stage], parity);
    if (!__syncthreads_and(ok)) {
      if (threadIdx.x == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
      return;
    }
    const uint32_t* s32 = reinterpret_cast<const uint32_t*>(smem + (size_t)P.stage_bytes * stage);
    const uint32_t delta = (uint32_t)((r0 * P.row_bytes) & 15LL);

    for (int v0 = 0; v0 < P.m; v0 += MV) {
      float* pb = part + (size_t)(i & 1) * part_stride;
      if (active_warp) {
        for (int seg = my_seg0; seg < NS; seg += (NS <= kWarps ? NS : seg_step)) {
          if (!x_static) load_x<K, MV>(P, v0, seg, lane, xr);
          for (int rl = my_rg; rl < rows; rl += RG) {
            float acc[MV];
#pragma unroll
            for (int m = 0; m < MV; ++m) acc[m] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
              const int b = seg * 32 * K + k * 32 + lane;
              if (b < P.bpr) {
                uint64_t q2[16];
                const uint32_t o = delta + (uint32_t)(rl * P.bpr + b) * kQBlockBytes;
                const float sc = decode_block(s32, o, q2);
#pragma unroll
                for (int m = 0; m < MV; ++m) {
                  uint64_t s2 = pack2(0.f, 0.f);
#pragma unroll
                  for (int j = 0; j < 16; ++j) s2 = fma2(q2[j], xr[m][k][j], s2);
                  float lo, hi;
                  unpack2(s2, lo, hi);
                  acc[m] = fmaf(sc, lo + hi, acc[m]);
                }
              }
            }
#pragma unroll
            for (int m = 0; m < MV; ++m) {
              const float v = warp_sum(acc[m]);
              if (lane == 0) pb[((size_t)rl * NS + seg) * MV + m] = v;
            }
          }
          if (NS <= kWarps) break;
        }
      }
      __syncthreads();
      // Reduce the NS segment partials of each (row, vector) in order.
      const int mv_here = min(MV, P.m - v0);
      for (int e = threadIdx.x; e < rows * mv_here; e += kThreads) {
        const int rl = e / mv_here, m = e % mv_here;
        float s = 0.f;
        for (int seg = 0; seg < NS; ++seg) s += pb[((size_t)rl * NS + seg) * MV + m];
        float* y = S.y + (size_t)(v0 + m) * P.ldy + (r0 + rl);
        *y = P.accumulate ? (*y + s) : s;
      }
      if (v0 + MV < P.m) __syncthreads();
    }
    // Stage `stage` is free once every warp passed the barrier above.
    if (threadIdx.x == 0) issue(i + P.nstages);
  }
}

__global__ void fill_zero_kernel(float* y, int ldy, int m, int p) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < (long long)m * p;
       e += (long long)gridDim.x * blockDim.x)
    y[(e / p) * ldy + (e % p)] = 0.f;
}

template <int K, int MV>
int launch_rows(const RowsParams& P, int smem_bytes, cudaStream_t stream) {
  auto fn = q8_rows_kernel<K, MV>;
  static int configured_bytes[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_bytes[dev] < smem_bytes) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return record_cuda(e);
    configured_bytes[dev] = 200 * 1024;
  }
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, smem_bytes);
  if (e != cudaSuccess) return record_cuda(e);
  occ = std::max(occ, 1);
  const int grid = std::min(P.total_tiles, sm_count() * occ);
  fn<<<grid, kThreads, smem_bytes, stream>>>(P);
  return check_launch();
}

}  // namespace

int rows_plan_and_launch(RowsParams P, cudaStream_t stream) {
  if (P.m <= 0) return Q8D_OK;
  long long p_total = 0;
  for (int s = 0; s < P.nseg; ++s) p_total += P.seg[s].p;
  if (p_total == 0) return Q8D_OK;
  if (P.n == 0) {
    if (P.accumulate) return Q8D_OK;
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

  // Blocks per lane K (1..4): fewest segments per row up to 8 warps with
  // little idle; x for MV vectors stays in registers (32*K*MV floats <= 128).
  int K = 1;
  for (K = 1; K < 4; ++K) {
    const int ns = (P.bpr + 32 * K - 1) / (32 * K);
    if (ns <= kWarps) break;
  }
  if (P.m > 1) K = 1;  // activations of several vectors compete for registers
  const int NS = (P.bpr + 32 * K - 1) / (32 * K);
  const int MV = (K > 1 || P.m == 1) ? 1 : (P.m == 2 ? 2 : 4);
  P.segs_per_row = NS;

  // Tile rows: ~16 KB stages, but enough tiles to give every SM work.
  const int sms = sm_count();
  long long R = std::max<long long>(1, 16384 / P.row_bytes);
  R = std::min<long long>(R, std::max<long long>(1, p_total / (2LL * sms)));
  R = std::min<long long>(R, 64);
  P.rows_per_tile = (int)R;
  int tiles = 0;
  for (int s = 0; s < P.nseg; ++s) {
    P.seg[s].tile_begin = tiles;
    tiles += (int)((P.seg[s].p + R - 1) / R);
  }
  P.total_tiles = tiles;
  P.stage_bytes = (int)(((R * P.row_bytes + 32 + 127) / 128) * 128);
  P.nstages = P.stage_bytes <= 12 * 1024 ? 6 : (P.stage_bytes <= 24 * 1024 ? 4 : 3);
  const int part_floats = (int)R * NS * MV;
  const int smem = P.stage_bytes * P.nstages + 8 * P.nstages + 4 * 2 * part_floats;
  if (smem > 200 * 1024) return Q8D_EUNSUPPORTED;

  switch (K * 10 + MV) {
    case 11: return launch_rows<1, 1>(P, smem, stream);
    case 12: return launch_rows<1, 2>(P, smem, stream);
    case 14: return launch_rows<1, 4>(P, smem, stream);
    case 21: return launch_rows<2, 1>(P, smem, stream);
    case 31: return launch_rows<3, 1>(P, smem, stream);
    case 41: return launch_rows<4, 1>(P, smem, stream);
    default: return Q8D_EUNSUPPORTED;
  }
}

}  // namespace q8d
