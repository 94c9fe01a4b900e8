// Q8_0 matrix-vector product (one activation vector) on CUDA cores, sm_103a.
//
//   y[r] (+)= sum_b scale(r,b) * sum_j q(r,b,j) * x[32b+j]
// ("IV.4: One command buffer per token", "Eight kernels": q8_matvec), for up
// to three matrices that share x in one launch.
//
// The product reads every weight byte once and does ~2.5 instructions per
// quant, so at HBM speed it is bound by instruction issue as much as by
// DRAM.  The layout is chosen to keep the per-block instruction count at the
// decode's own cost:
//  * Weight tiles (R whole rows, one contiguous byte range) are streamed into
//    a ring of shared-memory stages with 1-D bulk copies (TMA) that complete
//    on mbarriers.  One producer warp issues them, refilling a stage as soon
//    as every consumer warp has released it; the consumer warps do nothing
//    but the products, and per-tile bookkeeping is incremental 32-bit
//    arithmetic.
//  * A row is covered by NS warps.  For rows of more than 32 blocks the
//    warps come in pairs that own the even and the odd block columns of a
//    64-column segment: lane l of the pair's warps owns column 64s + 2l (+1).
//    Blocks are 34 bytes, so all blocks of one warp then have the same
//    alignment modulo 4 (the scale in the upper or lower half of a word),
//    and the 17-word lane stride is free of shared-memory bank conflicts.
//    Rows of up to 32 blocks use one warp with lane l on column l.
//  * A lane keeps the 32 activations of its column in registers for every
//    row it visits; its partial for a row (scale * block dot product) goes
//    to shared memory, and windows of rows are summed over segments and lanes
//    in a fixed order (deterministic results).  Windows are double-buffered,
//    so one barrier of the consumer warps per window suffices.
//  * Dequantisation: a sign-flipped quant byte is placed in the mantissa of
//    2^23 with one PRMT, one packed f32x2 add removes the bias exactly, and
//    packed f32x2 FMAs accumulate in four chains.
#include <algorithm>

#include "q8d_gemv.cuh"
#include "q8d_internal.cuh"
#include "q8d_rows.cuh"

namespace q8d {

namespace {

using namespace mv;

constexpr int kMaxWarps = 20;
constexpr int kSmallThreads = 17 * 32;              // 16 consumer warps + the producer
constexpr int kLargeThreads = (kMaxWarps + 1) * 32;  // 20 + 1

// Activations of block column `col` (32 floats) as 16 packed pairs; zeros
// when col is past the row end.
__device__ __forceinline__ void load_x_col(const RowsParams& P, int col, uint64_t (&x2)[16]) {
  const bool ok = col < P.bpr;
  const size_t base = (size_t)col * kQBlock;
  const float4* xp = reinterpret_cast<const float4*>(P.X + base);
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const float4 v = ok ? __ldg(xp + t) : make_float4(0.f, 0.f, 0.f, 0.f);
    x2[2 * t] = pack2(v.x, v.y);
    x2[2 * t + 1] = pack2(v.z, v.w);
  }
}

// Sums the lane partials of `nrow` rows (the window starting at virtual row
// wbeg) over segments and lanes in a fixed order and writes y.  Eight
// threads per row, four rows per consumer warp at a time; every lane of a
// warp runs the same iterations.  part = [row][NS][32] floats, 16-byte
// aligned rows.
__device__ __forceinline__ void window_reduce(const RowsParams& P, const float* part, int nrow,
                                              int NS, int nwarps, int wbeg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane & 7;
  for (int r0 = warp * 4; r0 < nrow; r0 += nwarps * 4) {
    const int r = r0 + (lane >> 3);
    const bool valid = r < nrow;
    const float4* pr = reinterpret_cast<const float4*>(part + (size_t)(valid ? r : r0) * NS * 32) + sub;
    uint64_t acc0 = pack2(0.f, 0.f), acc1 = acc0;
    for (int k = 0; k < NS; ++k) {
      const float4 v = pr[8 * k];
      acc0 = add2(acc0, pack2(v.x, v.y));
      acc1 = add2(acc1, pack2(v.z, v.w));
    }
    float lo, hi;
    unpack2(add2(acc0, acc1), lo, hi);
    float sum = lo + hi;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (valid && sub == 0) {
      const int vr = wbeg + r;
      int sg = 0;
      while (sg + 1 < P.nseg && vr >= P.vbegin[sg + 1]) ++sg;
      const int ri = vr - (int)P.vbegin[sg];
      P.seg[sg].y[ri] = sum;
    }
  }
}

struct Ring {
  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  float* part;  // [2][win_rows][NS][32] lane partials
  int* abort_flag;
};

// Tiles of the CTA's contiguous range of virtual rows (the matrices' rows
// concatenated): at most R rows each, never across a matrix end.
struct Cursor {
  int cur;   // first virtual row of the tile
  int r0;    // its row within matrix `seg`
  int seg;
  int seg_end;  // virtual row where matrix `seg` ends
  __device__ void start(const RowsParams& P, int v0) {
    cur = v0;
    seg = 0;
    while (seg + 1 < P.nseg && v0 >= P.vbegin[seg + 1]) ++seg;
    r0 = v0 - (int)P.vbegin[seg];
    seg_end = (int)P.vbegin[seg] + P.seg[seg].p;
  }
  __device__ int rows(int R, int v1) const { return min(R, min(seg_end, v1) - cur); }
  __device__ void advance(const RowsParams& P, int n) {
    cur += n;
    r0 += n;
    if (cur == seg_end && seg + 1 < P.nseg) {
      ++seg;
      r0 = 0;
      seg_end = cur + P.seg[seg].p;
    }
  }
};

// Producer: one thread issues every tile of the CTA into the ring, waiting
// for a stage only until all consumer warps have released it.  Returns the
// number of tiles issued (fewer if a wait timed out).
__device__ int produce_all(const RowsParams& P, const Ring& ring, int v0, int v1) {
  const uint64_t pol = policy_evict_first();
  Cursor c;
  c.start(P, v0);
  int s = 0;
  uint32_t ph = 0;
  int i = 0;
  for (; c.cur < v1; ++i) {
    if (i >= P.nstages && !wait_or_abort(&ring.empty[s], ph ^ 1u, ring.abort_flag)) break;
    const int rows = c.rows(P.rows_per_tile, v1);
    const RowSeg& S = P.seg[c.seg];
    const long long start = (long long)c.r0 * P.row_bytes;
    const long long end = start + (long long)rows * P.row_bytes;
    const long long cap16 = ((long long)S.p * P.row_bytes) & ~15LL;
    const long long a0 = start & ~15LL;
    long long a1 = (end + 15) & ~15LL;
    uint8_t* dst = ring.smem + (size_t)P.stage_bytes * s;
    if (a1 > cap16) {
      // last tile of a matrix whose size is not a multiple of 16 bytes: the
      // bytes past the last 16-byte boundary are copied by hand (published
      // by the arrive below)
      a1 = cap16 > a0 ? cap16 : a0;
      for (long long o = a1; o < end; ++o) dst[o - a0] = __ldg(S.w + o);
    }
    const uint32_t bytes = (uint32_t)(a1 - a0);
    mbar_arrive_expect_tx(&ring.full[s], bytes);
    if (bytes) bulk_g2s(dst, S.w + a0, bytes, &ring.full[s], pol);
    c.advance(P, rows);
    if (++s == P.nstages) {
      s = 0;
      ph ^= 1u;
    }
  }
  return i;
}

// Consumer loop of one warp.  AM: alignment mode of the warp's blocks.  A
// warp takes P.np pairs of rows per tile (a tile has R = 2 * RG * np rows).  A tile
// with fewer rows (the end of a matrix or of the CTA's range) is computed
// over all R rows of its stage, which the stage's size covers, and only
// the partials of its real rows are stored.
template <int AM>
__device__ __forceinline__ bool consume(const RowsParams& P, const Ring& ring, uint32_t part32,
                                        int v0, int v1, int ci, int rg, int RG, int nwarps,
                                        uint32_t boff, const uint64_t (&x2)[16]) {
  const int lane = threadIdx.x & 31;
  const int NS = P.segs_per_row;
  const int n32 = NS * 32;
  const uint32_t rowb = (uint32_t)P.row_bytes;
  const uint32_t step = (uint32_t)RG * rowb;        // stage bytes between a warp's rows
  const uint32_t pstep = (uint32_t)(RG * n32 * 4);  // partial bytes between them
  const uint32_t rb15 = rowb & 15u;
  const uint32_t smem32 = smem_u32(ring.smem);
  const uint32_t lane_part = part32 + (uint32_t)(ci * 32 + lane) * 4u + (uint32_t)(rg * n32) * 4u;
  const uint32_t buf_bytes = (uint32_t)(P.win_rows * n32 * 4);
  bool ok = true;
  Cursor c;
  c.start(P, v0);
  uint32_t delta = ((uint32_t)c.r0 * rb15) & 15u;  // tile start mod 16 (matrices are 16-aligned)
  int s = 0;
  uint32_t ph = 0;
  uint32_t stage32 = smem32;
  int wbeg = v0, wt = 0, wrow = 0;
  uint32_t buf = 0;  // byte offset of the current window buffer
  while (c.cur < v1) {
    const int rows = c.rows(P.rows_per_tile, v1);
    // On a timeout the loop still runs (over whatever the stage holds; the
    // launch then reports Q8D_DERR_WAIT) so that every consumer warp reaches
    // the window barriers.
    ok = wait_or_abort(&ring.full[s], ph, ring.abort_flag) && ok;
    uint32_t o = after_wait(stage32 + delta + boff + (uint32_t)rg * rowb);
    uint32_t d = lane_part + buf + (uint32_t)(wrow * n32) * 4u;
    int rl = rg;
#pragma unroll 1
    for (int j = 0; j < P.np; ++j) {
      // both rows' words first: the two decodes are independent work for
      // the scheduler to interleave
      uint32_t wa[9], wb[9];
      block_words(o, wa);
      block_words(o + step, wb);
      const float va = block_dot_words<AM>(wa, o, x2);
      const float vb = block_dot_words<AM>(wb, o + step, x2);
      if (rl < rows) sts32(d, va);
      if (rl + RG < rows) sts32(d + pstep, vb);
      o += 2 * step;
      d += 2 * pstep;
      rl += 2 * RG;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[s]);
    stage32 += (uint32_t)P.stage_bytes;
    if (++s == P.nstages) {
      s = 0;
      ph ^= 1u;
      stage32 = smem32;
    }
    const int seg_before = c.seg;
    c.advance(P, rows);
    delta = c.seg == seg_before ? (delta + (uint32_t)rows * rb15) & 15u : 0u;
    wrow += rows;
    if (++wt == P.win || c.cur >= v1) {
      // window complete: every consumer warp has stored its partials.  The
      // other buffer was reduced before this barrier, so the next window may
      // overwrite it.
      consumer_sync(nwarps * 32);
      window_reduce(P, ring.part + buf / 4, wrow, NS, nwarps, wbeg);
      buf = buf ? 0u : buf_bytes;
      wt = 0;
      wrow = 0;
      wbeg = c.cur;
    }
  }
  return ok;
}

// Block of W consumer warps plus one producer warp (the last), at most
// NT / 32 warps in all: up to 17 warps (at most five per SM sub-partition)
// a thread may hold 96 registers, 80 with 21.
template <int NT>
__global__ void __launch_bounds__(NT) q8_gemv_kernel(const RowsParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = (blockDim.x >> 5) - 1;  // consumer warps
  const int NS = P.segs_per_row;
  __shared__ int s_abort;

  Ring ring;
  ring.smem = smem;
  ring.full = reinterpret_cast<uint64_t*>(smem + (size_t)P.stage_bytes * P.nstages);
  ring.empty = ring.full + P.nstages;
  ring.abort_flag = &s_abort;
  ring.part = reinterpret_cast<float*>(ring.empty + P.nstages);

  const int v0 = blockIdx.x * (int)P.rows_per_cta;
  const int v1 = (int)min(P.total_rows, (long long)v0 + P.rows_per_cta);
  // Launched as a programmatic dependent: the next kernel may start its
  // prologue now; this one waits for the previous kernel before it copies
  // weights into shared memory, reads x or writes y.  Until then the
  // producer warp pulls the first ring-full of this CTA's rows (one byte
  // range of one matrix, widened to 16-byte boundaries inside it) into L2,
  // which reads nothing it depends on.
  griddep_launch_dependents();
  if (warp == W && P.nseg == 1 && v0 < v1) {
    const long long want = min((long long)P.stage_bytes * P.nstages, (long long)(v1 - v0) * P.row_bytes);
    const long long cap16 = ((long long)P.seg[0].p * P.row_bytes) & ~15LL;
    const long long a0 = ((long long)v0 * P.row_bytes) & ~15LL;
    const long long a1 = min(cap16, ((long long)v0 * P.row_bytes + want + 15) & ~15LL);
    for (long long o = a0 + (long long)lane * 16384; o < a1; o += 32LL * 16384)
      bulk_prefetch_l2(P.seg[0].w + o, (uint32_t)min(16384LL, a1 - o));
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nstages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], W);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  griddep_wait();
  __syncthreads();

  bool ok = true;
  if (warp == W) {
    // ---- producer warp ----
    if (lane == 0) {
      const int issued = produce_all(P, ring, v0, v1);
      if (*(volatile int*)&s_abort) {
        // Wait (bounded) for the copies still in flight before the CTA's
        // shared memory can be released.
        for (int j = max(0, issued - P.nstages); j < issued; ++j)
          mbar_wait(&ring.full[j % P.nstages], (uint32_t)(j / P.nstages) & 1u);
      }
    }
  } else {
    // This warp's block column class and row group (W is a multiple of NS).
    const int ci = warp % NS, rg = warp / NS, RG = W / NS;
    int col, col_read;
    if (P.paired) {
      const int par = ci & 1;
      col = 64 * (ci >> 1) + 2 * lane + par;
      // lanes past the row end read the last block of the same parity (so
      // the warp's alignment holds) with zero activations
      col_read = min(col, P.bpr - 1 - ((P.bpr - 1 - par) & 1));
    } else {
      col = lane;
      col_read = min(col, P.bpr - 1);
    }
    uint64_t x2[16];
    load_x_col(P, col, x2);
    const uint32_t boff = (uint32_t)col_read * kQBlockBytes;
    // With an even number of blocks per row every row starts at a multiple
    // of 4 bytes, so all blocks of a paired warp start at 2*(col & 1) mod 4.
    const uint32_t part32 = smem_u32(ring.part);
    if (P.paired && (P.bpr & 1) == 0) {
      if (ci & 1)
        ok = consume<1>(P, ring, part32, v0, v1, ci, rg, RG, W, boff, x2);
      else
        ok = consume<0>(P, ring, part32, v0, v1, ci, rg, RG, W, boff, x2);
    } else {
      ok = consume<2>(P, ring, part32, v0, v1, ci, rg, RG, W, boff, x2);
    }
  }

  if (!__syncthreads_and(ok && !*(volatile int*)&s_abort)) {
    if (threadIdx.x == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
  }
}

}  // namespace

// Plans and launches the matvec kernel (m == 1, rows of at most 20 warps).
// Returns Q8D_EUNSUPPORTED when the shape does not fit it.
int gemv_plan_and_launch(RowsParams P, cudaStream_t stream, int* grid_out) {
  const int bpr = P.bpr;
  const bool paired = bpr > 32;
  const int NS = paired ? 2 * ((bpr + 63) / 64) : 1;  // warps per row
  if (P.m != 1 || NS > kMaxWarps || P.total_rows > 0x7fffffffLL) return Q8D_EUNSUPPORTED;
  // One CTA per SM with 16 consumer warps (20 for the longest rows), a
  // multiple of NS, plus the producer warp; RG rows are in work at once.
  const int W = NS <= 8 ? NS * (16 / NS) : NS * (kMaxWarps / NS);
  const int RG = W / NS;
  const int sms = sm_count();
  constexpr long long kSmemCta = 220 * 1024;

  // Tiles of R = 2 * RG * NP rows (each warp takes NP pairs of rows per
  // tile), NP = 4, 2 or 1: the largest whose tile is at most ~64 KB (and
  // 128 rows) and leaves room for three stages.  Reduction windows are
  // double-buffered within ~40 KB of partials.
  long long R = 0, stage = 0, part_bytes = 0;
  int nst = 0, wt = 0, np = 4;
  for (;; np /= 2) {
    R = 2LL * RG * np;
    const long long win_rows = std::max<long long>(R, 40960 / (2LL * NS * 32 * 4));
    wt = (int)(win_rows / R);
    part_bytes = 2LL * wt * R * NS * 32 * 4;
    stage = ((R * P.row_bytes + 32 + 127) / 128) * 128;
    nst = (int)std::min<long long>(8, (kSmemCta - part_bytes - 1024) / (stage + 16));
    if (np == 1 || (R <= 128 && R * P.row_bytes <= 65536 && nst >= 3)) break;
  }
  P.paired = paired ? 1 : 0;
  P.segs_per_row = NS;
  P.stage_bytes = (int)stage;
  P.nstages = nst;
  P.win = wt;
  P.win_rows = (int)(wt * R);
  P.np = np;
  const long long smem = stage * nst + 16LL * nst + part_bytes;

  const bool small = (W + 1) * 32 <= kSmallThreads;
  void (*fn)(const RowsParams) = small ? q8_gemv_kernel<kSmallThreads> : q8_gemv_kernel<kLargeThreads>;
  const int rc = configure_kernel(reinterpret_cast<const void*>(fn), 220 * 1024, true);
  if (rc) return rc;
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, (W + 1) * 32, (size_t)smem);
  if (e != cudaSuccess) return record_cuda(e);
  occ = std::max(occ, 1);
  // One wave of resident CTAs, each owning a contiguous range of rows.
  long long grid = std::min<long long>(P.total_rows, (long long)sms * occ);
  const long long rows_cta = (P.total_rows + grid - 1) / grid;
  grid = (P.total_rows + rows_cta - 1) / rows_cta;
  P.rows_per_cta = rows_cta;
  P.rows_per_tile = (int)std::min<long long>(R, rows_cta);
  if (grid_out) *grid_out = (int)grid;
  if (rows_cta < R) {
    // Fewer rows a CTA than one tile (small matrices: 7B k and v, 512 rows
    // over the SMs): one tile of exactly its rows in one stage, RG = half of
    // them (at most the full plan's), one window.  A few KB of shared memory
    // and a few warps a CTA, so the next call's CTAs (another small matrix)
    // fit beside this call's and pull their weights into L2 while it runs.
    const int rgc = std::max(1, std::min(RG, (int)(rows_cta / 2)));
    const int npc = (int)((rows_cta + 2LL * rgc - 1) / (2LL * rgc));
    const long long Rc = 2LL * rgc * npc;
    P.np = npc;
    P.rows_per_tile = (int)rows_cta;
    P.stage_bytes = (int)(((Rc * P.row_bytes + 32 + 127) / 128) * 128);
    P.nstages = 1;
    P.win = 1;
    P.win_rows = (int)Rc;
    const int Wc = rgc * NS;
    const long long smc = (long long)P.stage_bytes + 16 + 2LL * Rc * NS * 32 * 4;
    return launch_ex(fn, dim3((unsigned)grid), dim3((Wc + 1) * 32), (size_t)smc, stream, true, P);
  }
  return launch_ex(fn, dim3((unsigned)grid), dim3((W + 1) * 32), (size_t)smem, stream, true, P);
}

}  // namespace q8d
