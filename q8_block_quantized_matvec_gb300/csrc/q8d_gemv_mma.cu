// Q8_0 matrix-vector product with the block dot products on the tensor
// cores (mma.sync m16n8k16, f16 operands, f32 accumulation), sm_103a.
//
//   y[r] = sum_b scale(r,b) * sum_j q(r,b,j) * x[32b+j]
// ("IV.4: One command buffer per token", "Eight kernels": q8_matvec; the
// per-block product is summed inside the block and scaled once, as the
// pages' kernel does).
//
// Why: on CUDA cores every quant costs a byte permute, a bias add and an FMA
// (half of them on the half-rate ALU pipe), which holds the matvec near 50 %
// issue and 0.5 of HBM.  Here a quant pair costs one PRMT and one sub.f16x2,
// and the products go to the tensor pipe (the operand layout is in
// q8d_mma_frag.cuh).  The x fragments (each block with its own power-of-two
// scale) are built once per launch in shared memory, in one pass over x.
//  * Weights stream in through a ring of shared-memory stages filled with
//    1-D bulk copies (TMA) by one producer warp: a tile is 8 or 16 rows of
//    up to 136 blocks.  Whole rows come as bank-spread groups of
//    consecutive rows (one copy per group); rows longer than that are cut
//    into slices, one copy per row into a row slot padded so that the
//    lanes' word reads hit distinct banks.
//  * 4 lanes share a row; the warps' row partials are summed in a fixed
//    order (deterministic).
#include <algorithm>

#include "q8d_gemv.cuh"
#include "q8d_internal.cuh"
#include "q8d_mma_frag.cuh"
#include "q8d_rows.cuh"

namespace q8d {
namespace {

using namespace mv;
using namespace tc;

constexpr int kMvMaxWarps = 16;                         // consumer warps (at most)
constexpr int kMvThreads = (kMvMaxWarps + 1) * 32;      // + the producer warp
// more activation rows, fewer consumer warps, so that a thread may hold the
// accumulators of every row: 128 registers for three or four rows, ~168
// for five to eight
__host__ __device__ constexpr int mv_max_warps(int mr) {
  return mr <= 2 ? kMvMaxWarps : mr <= 4 ? 12 : 11;
}
constexpr int kWinSets = 4;                             // row sets per reduction window

struct MvParams {
  const uint8_t* w;
  float* y;          // row i of the output at y + i * ldy
  const float* x;    // activation row i at x + i * ldx
  int ldx, ldy;      // (m > 1)
  int n, bpr, p;
  int row_bytes;     // bpr * 34, a multiple of 272
  int rows_per_cta;  // a multiple of 8
  int S, nslices;    // blocks per slice (a multiple of 8), slices per row
  int SR;            // shared-memory row stride (bytes, multiple of 16)
  int gsh;           // a set is groups of 1 << gsh rows, 16 bytes apart (whole
                     // rows: one copy per group; sliced rows: gsh = 3, a copy a row)
  int set_bytes;     // an 8-row set: 8 * SR + 16 * (8 >> gsh)
  int stage_bytes, nstages;
  int W;             // consumer warps
  int T;             // 8-row sets per tile (1 or 2)
  int* d_err;
};

// Run by the whole producer warp: every lane walks the same tiles; lane 0
// waits for a free stage (bounded) and posts the transaction count, the
// warp follows its result, and the tile's row (or row-group) copies are
// dealt over the lanes.
__device__ int mv_produce(const MvParams& P, uint8_t* smem, uint64_t* full, uint64_t* empty,
                          int* abort_flag, int v0, int v1) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol = policy_evict_first();
  int s = 0, issued = 0;
  uint32_t ph = 0;
  const int tile_rows = kSetRows * P.T;
  const int gsz = P.nslices == 1 ? 1 << P.gsh : 1;  // rows a copy
  for (int r0 = v0; r0 < v1; r0 += tile_rows) {
    const int nrows = min(tile_rows, v1 - r0);
    for (int sl = 0; sl < P.nslices; ++sl) {
      if (issued >= P.nstages) {
        int ok = 1;
        if (lane == 0) ok = wait_or_abort(&empty[s], ph ^ 1u, abort_flag) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) return issued;
      }
      const int c0 = sl * P.S;
      const int nb = min(P.S, P.bpr - c0);
      const uint32_t bytes = (uint32_t)nb * kQBlockBytes;
      uint8_t* dst = smem + (size_t)P.stage_bytes * s;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes * nrows);
      __syncwarp();
      for (int r = lane * gsz; r < nrows; r += 32 * gsz)
        bulk_g2s(dst + (r >> 3) * P.set_bytes + (r & 7) * P.SR + ((r & 7) >> P.gsh) * 16,
                 P.w + (long long)(r0 + r) * P.row_bytes + (long long)c0 * kQBlockBytes,
                 bytes * (uint32_t)min(gsz, nrows - r), &full[s], pol);
      ++issued;
      if (++s == P.nstages) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  return issued;
}

// MR activation rows (1..8) against the same weights: each decoded weight
// fragment feeds MR MMAs (one per row's x fragments), so the weight decode
// and the weight stream are shared by the rows.
template <int MR>
__global__ void __launch_bounds__((mv_max_warps(MR) + 1) * 32, 1) q8_gemv_mma_kernel(const MvParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = P.W;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)P.stage_bytes * P.nstages);
  uint64_t* empty = full + P.nstages;
  uint8_t* xf = reinterpret_cast<uint8_t*>(empty + P.nstages);   // [MR][bpr] x fragments
  uint8_t* zpad = xf + (size_t)MR * P.bpr * kXfBlock;            // kZeroPad zero bytes
  float* xinv = reinterpret_cast<float*>(zpad + kZeroPad);       // [MR][bpr] inverse block scales
  float* part = xinv + MR * P.bpr;                               // [MR][2][kWinSets*8][W]
  const int v0 = blockIdx.x * P.rows_per_cta;
  const int v1 = min(P.p, v0 + P.rows_per_cta);
  // Launched as a programmatic dependent: the next kernel may start its
  // prologue now; this one waits for the previous kernel before it copies
  // weights into shared memory, reads x or writes y.  Until then the
  // producer pulls the first ring-full of this CTA's rows (contiguous in
  // memory) into L2, which reads nothing it depends on.
  griddep_launch_dependents();
  if (warp == W && v0 < v1) {
    const long long bytes =
        min((long long)P.stage_bytes * P.nstages, (long long)(v1 - v0) * P.row_bytes) & ~15LL;
    const uint8_t* base = P.w + (long long)v0 * P.row_bytes;
    for (long long o = (long long)lane * 16384; o < bytes; o += 32LL * 16384)
      bulk_prefetch_l2(base + o, (uint32_t)min(16384LL, bytes - o));
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  griddep_wait();
  __syncthreads();

  int issued = 0;
  bool ok = true;
  if (warp == W) {
    issued = mv_produce(P, smem, full, empty, &s_abort, v0, v1);
  } else {
    const int nct = W * 32;
    // ---- x fragments, one pass: up to kXItems (block, word) items a
    // thread per round, all loads issued before the first use (one round
    // for rows of up to kXItems * 480 / 8 blocks) ----
    // (items of all MR rows in one pass: item it is word it % nit of row
    // it / nit; a row's items are whole blocks, so the 8 lanes of a block
    // stay in one row)
    constexpr int kXItems = 12;
    const int nit = P.bpr * 8, nall = MR * nit;
    for (int it0 = 0; it0 < nall; it0 += kXItems * nct) {
      float v[kXItems][4];
#pragma unroll
      for (int k = 0; k < kXItems; ++k) {
        const int it = it0 + k * nct + threadIdx.x;
        if (it < nall) {
          const int r = it / nit, ii = it - r * nit;
          load_word<1>(P.x + (long long)r * P.ldx, ii >> 3, ii & 7, v[k]);
        } else {
          v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < kXItems; ++k) {
        const int it = it0 + k * nct + threadIdx.x;
        if (it0 + k * nct >= nall) break;  // (uniform over the warps)
        const int r = min(it / nit, MR - 1), ii = it - r * nit;
        build_x_word(ii, it < nall, v[k], xf + (size_t)r * P.bpr * kXfBlock, xinv + r * P.bpr);
      }
    }
    for (int i = threadIdx.x; i < kZeroPad / 4; i += nct) reinterpret_cast<uint32_t*>(zpad)[i] = 0u;
    consumer_sync(nct);

    // ---- main loop ----
    const int gq = lane >> 2, cq = lane & 3;
    const LaneOffs LO = lane_offsets(cq);
    const XLane XL = x_lane(lane);
    const uint32_t xf32 = smem_u32(xf), z32 = smem_u32(zpad);
    const uint32_t xi32 = smem_u32(xinv) + 4u * (uint32_t)lane_block(cq);
    const uint32_t smem32 = smem_u32(smem);
    const bool lo_half = cq < 2;
    const int S = P.S, bpr = P.bpr, nslices = P.nslices, nst = P.nstages;
    const uint32_t stage_b = (uint32_t)P.stage_bytes;
    const uint32_t rowoff = (uint32_t)(gq * P.SR + ((gq >> P.gsh) << 4));
    const int T = P.T;
    const uint32_t set_b = (uint32_t)P.set_bytes;  // bytes between the row sets of a tile
    int s = 0;
    uint32_t ph = 0;
    int set = 0, buf = 0;
    const uint32_t xf_row = (uint32_t)bpr * kXfBlock, xi_row = 4u * (uint32_t)bpr;
    for (int r0 = v0; r0 < v1; r0 += kSetRows * T) {
      float yacc[2][MR];  // this thread's row gq of the tile's sets, per activation row
#pragma unroll
      for (int r = 0; r < MR; ++r) yacc[0][r] = yacc[1][r] = 0.f;
      for (int sl = 0; sl < nslices; ++sl) {
        ok = wait_or_abort(&full[s], ph, &s_abort) && ok;
        const uint32_t row32 = after_wait(smem32 + stage_b * (uint32_t)s + rowoff);
        const int c0 = sl * S;
        const int pairs = min(S, bpr - c0) / 8;
        for (int k = warp; k < pairs; k += W) {
          const uint32_t xb0 = XL.match ? xf32 + (uint32_t)((c0 / 8 + k) * kXfPair) + XL.off : z32;
          const uint32_t xi0 = xi32 + 4u * (uint32_t)(c0 + 8 * k);
          uint32_t xb[MR], xi[MR];
#pragma unroll
          for (int r = 0; r < MR; ++r) {
            xb[r] = XL.match ? xb0 + (uint32_t)r * xf_row : z32;
            xi[r] = xi0 + (uint32_t)r * xi_row;
          }
          const uint32_t rb = row32 + 272u * (uint32_t)k;
          pair_dot_m<MR>(rb, xb, XL.step, LO, lo_half, xi, yacc[0]);
          if (T == 2) pair_dot_m<MR>(rb + set_b, xb, XL.step, LO, lo_half, xi, yacc[1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == nst) {
          s = 0;
          ph ^= 1u;
        }
      }
      // the tile's row sets are complete: the warp's partials of rows r0 + 8t + gq
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t >= T || r0 + kSetRows * t >= v1) break;
        const int rs0 = r0 + kSetRows * t;
        const int slot = set % kWinSets;
#pragma unroll
        for (int r = 0; r < MR; ++r) {
          float y = yacc[t][r];
          y += __shfl_xor_sync(0xffffffffu, y, 1);
          y += __shfl_xor_sync(0xffffffffu, y, 2);
          if (cq == 0) part[(((r * 2 + buf) * kWinSets + slot) * kSetRows + gq) * W + warp] = y;
        }
        if (slot == kWinSets - 1 || rs0 + kSetRows >= v1) {
          consumer_sync(nct);
          // window reduction: rows of the window's sets, warp partials in order
          const int wr0 = rs0 - slot * kSetRows;
          for (int i = threadIdx.x; i < MR * (slot + 1) * kSetRows; i += nct) {
            const int r = i / ((slot + 1) * kSetRows), ii = i % ((slot + 1) * kSetRows);
            const int row = wr0 + ii;
            if (row < v1) {
              const float* pr = part + (((size_t)(r * 2 + buf) * kWinSets) * kSetRows + ii) * W;
              float sum = 0.f;
              for (int w = 0; w < W; ++w) sum += pr[w];
              P.y[(long long)r * P.ldy + row] = sum;
            }
          }
          buf ^= 1;
        }
        ++set;
      }
    }
  }
  if (!__syncthreads_and(ok && !*(volatile int*)&s_abort)) {
    if (threadIdx.x == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
  }
  if (warp == W && lane == 0 && *(volatile int*)&s_abort) {
    for (int j = max(0, issued - P.nstages); j < issued; ++j)
      mbar_wait(&full[j % P.nstages], (uint32_t)(j / P.nstages) & 1u);
  }
}

}  // namespace

// Plans and launches the tensor-core matvec for R.m (1..8) activation rows.
// Q8D_EUNSUPPORTED when the shape does not suit it (one matrix, n % 256 ==
// 0 and n >= 2048, enough rows to give every SM two 8-row sets, the rows'
// x fragments and three stages within shared memory); the caller then runs
// a CUDA-core kernel.
int gemv_mma_plan_and_launch(const RowsParams& R, cudaStream_t stream, int* grid_out) {
  if (R.m < 1 || R.m > 8 || R.nseg != 1 || R.bpr % 8 || R.bpr < 64) return Q8D_EUNSUPPORTED;
  const int sms = sm_count();
  const long long p = R.seg[0].p;
  if (p < 2LL * kSetRows * sms || p > 0x7fffffffLL) return Q8D_EUNSUPPORTED;
  MvParams P{};
  P.w = R.seg[0].w;
  P.y = R.seg[0].y;
  P.x = R.X;
  P.ldx = R.ldx;
  P.ldy = R.ldy;
  P.n = R.n;
  P.bpr = R.bpr;
  P.p = (int)p;
  P.row_bytes = R.bpr * kQBlockBytes;
  P.d_err = R.d_err;
  // slices of at most ~4.6 KB per row (8 rows: ~37 KB a stage)
  const int max_blocks = 136;
  P.nslices = (P.bpr + max_blocks - 1) / max_blocks;
  P.S = ((P.bpr + P.nslices - 1) / P.nslices + 7) / 8 * 8;
  P.nslices = (P.bpr + P.S - 1) / P.S;
  if (P.nslices == 1) {
    // whole rows: bank-spread groups of consecutive rows, one copy each
    P.SR = P.row_bytes;
    P.gsh = row_group_shift(P.bpr / 8);
  } else {
    // row slot: >= the slice, 16-byte multiple, 4 banks apart row to row
    int SR = (P.S * kQBlockBytes + 15) / 16 * 16;
    while ((SR / 4) % 32 != 4) SR += 16;
    P.SR = SR;
    P.gsh = 3;  // (one group: no offsets; the slots spread the banks)
  }
  P.set_bytes = kSetRows * P.SR + 16 * (8 >> P.gsh);
  P.stage_bytes = P.set_bytes;
  // consumer warps: the count in [8, 16] that splits a slice's unit pairs
  // (8 blocks of 8 rows) most evenly
  const int U = P.S / 8;
  const int maxW = mv_max_warps(R.m);
  int bestW = maxW;
  double best = 0.0;
  for (int w = maxW; w >= 8; --w) {
    const double eff = (double)U / (w * ((U + w - 1) / w));
    if (eff > best + 1e-9) {
      best = eff;
      bestW = w;
    }
  }
  P.W = bestW;
  const int MR = R.m;
  const long long fixed = (long long)MR * P.bpr * (kXfBlock + 4) + kZeroPad +
                          2LL * MR * kWinSets * kSetRows * P.W * 4;
  const long long budget = 220 * 1024;
  // two row sets per tile (each warp's per-tile work twice as long) when
  // three such stages fit
  P.T = (budget - fixed) / (2LL * P.stage_bytes + 16) >= 3 ? 2 : 1;
  P.stage_bytes *= P.T;
  P.nstages = (int)std::min<long long>(8, (budget - fixed) / (P.stage_bytes + 16));
  if (P.nstages < 3) return Q8D_EUNSUPPORTED;
  const long long smem = (long long)P.stage_bytes * P.nstages + 16LL * P.nstages + fixed;
  // 8-row sets spread evenly over one wave of CTAs (one per SM)
  const long long sets = (p + kSetRows - 1) / kSetRows;
  const long long sets_cta = (sets + sms - 1) / sms;
  P.rows_per_cta = (int)(sets_cta * kSetRows);  // (a CTA's last tile may hold one set)
  const int grid = (int)((p + P.rows_per_cta - 1) / P.rows_per_cta);
  void (*const kFns[8])(MvParams) = {q8_gemv_mma_kernel<1>, q8_gemv_mma_kernel<2>,
                                     q8_gemv_mma_kernel<3>, q8_gemv_mma_kernel<4>,
                                     q8_gemv_mma_kernel<5>, q8_gemv_mma_kernel<6>,
                                     q8_gemv_mma_kernel<7>, q8_gemv_mma_kernel<8>};
  const auto fn = kFns[MR - 1];
  const int rc = configure_kernel(reinterpret_cast<const void*>(fn), 220 * 1024, true);
  if (rc) return rc;
  if (grid_out) *grid_out = grid;
  return launch_ex(fn, dim3(grid), dim3((P.W + 1) * 32), (size_t)smem, stream, true, P);
}

}  // namespace q8d
