// Tensor-core path of q8d_matmul_small_m (m >= 9): Y[i][r] = sum_k X[i][k] W[r][k].
//
// At m >= 9 activation rows the product is a real dense contraction (2m
// flops per weight element, 30-120 flop/byte at m = 16..64) that would make
// the CUDA cores the bottleneck, so it runs on the 5th-generation tensor
// cores ("Metal Backend Optimizations": the quantised GEMM tier used once
// more than one token is in flight stages dequantised weights in on-chip
// memory; here the tile feeds tcgen05.mma instead of SIMD-group matrices).
//
//  * The activations are rounded to f16 once per call by a small kernel
//    (q8_ximage_kernel, one CTA per activation row) under a power-of-two
//    scale per row (its max |x| into [2^14, 2^15), undone on the result)
//    into a workspace that holds, for every 128-row block of X and every
//    128-element K half, the B operand exactly as the MMA reads it from
//    shared memory (canonical K-major 128-byte-swizzled layout); the main
//    kernel starts as its programmatic dependent and copies a chunk's B
//    tile with a single 1-D bulk copy.
//  * CTA = 128 weight rows (the MMA's M) x a K range; a thread-block cluster
//    of `ksplit` CTAs along K shares one output tile and reduces the fp32
//    partials through distributed shared memory in rank order
//    (deterministic, no global scratch, no atomics).
//  * Warp roles, so that dequantisation, copies and MMAs overlap: a weight
//    producer warp streams raw Q8_0 bytes (8 blocks = 272 bytes per row per
//    256-element chunk, the 128 rows a weight-row stride apart) by one 2-D
//    tensor copy per chunk (TMA: 68 32-bit elements x 128 rows; every x
//    coordinate a multiple of 16 bytes; rows past the matrix zero-filled)
//    into a ring of stages; an activation producer warp copies the B tiles;
//    16 dequantising warps turn each chunk (256 K elements) into the bf16 A
//    operand in tensor memory (TMEM): warp w owns TMEM lanes 32 (w % 4) +
//    [0, 32) = weight rows and blocks w / 4 and w / 4 + 4 of the chunk; a
//    thread reads a block with three conflict-free 16-byte shared loads,
//    turns the quants into exact f16 pairs (one byte permute and one
//    sub.f16x2 a pair), multiplies them by the block's f16 scale (one
//    mul.f16x2: the exact product rounded once) and writes the block's 16
//    columns with one tcgen05.st.  A ring of two or three slots,
//    each a chunk's A tile (128 TMEM columns) and B tile (shared memory)
//    with one "full" mbarrier (16 warp arrivals + the B copy's bytes) and
//    one "empty" mbarrier; one MMA warp issues
//    tcgen05.mma.cta_group::1.kind::f16 with A from TMEM and B from shared
//    memory (f16 x f16 -> f32, M = 128, N = m rounded up to 16, K = 16 per
//    instruction: ~93 cycles each on this part whatever N <= 128, so the 16
//    of a chunk bound the loop) and commits to the slot's "empty"
//    barrier.  The accumulator (TMEM columns [0, N)) is read with
//    tcgen05.ld and stored to Y directly, or, for a K split, reduced across
//    the cluster through distributed shared memory.
// Accuracy: one f16 rounding of each weight (scale * q) and activation
// (x * 2^e), f32 accumulation: |error| <= ~2^-10 * sum|terms| per output
// (plus 2^-25 * sum|x| where scale * q falls below f16's normal range).  A
// block scale above 511.75 could make scale * q overflow f16: the kernel
// checks every scale and then writes NaN for its row tile.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is looked up at run time
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "q8d_gemv.cuh"
#include "q8d_internal.cuh"

namespace q8d {
namespace {

using mv::wait_or_abort;

// One plain poll first (the phase is usually complete), then the bounded
// sleeping wait.
__device__ __forceinline__ bool wait_ready(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || wait_or_abort(bar, parity, abort_flag);
}

constexpr int kDeqWarps = 16;                   // dequantising warps
constexpr int kDeqThreads = kDeqWarps * 32;
constexpr int kWProducer = kDeqWarps;           // weight producer warp
constexpr int kXProducer = kDeqWarps + 1;       // activation producer warp
constexpr int kMmaWarp = kDeqWarps + 2;         // MMA issuer warp
constexpr int kThreads = kDeqThreads + 96;
constexpr int kM = 128;                         // weight rows per CTA (MMA M)
constexpr int kKC = 256;                        // K elements per raw chunk (one tensor copy)
constexpr int kRawRow = (kKC / kQBlock) * kQBlockBytes;  // 272 bytes
constexpr int kRawStage = kM * kRawRow;         // 34816 bytes
constexpr int kACols = kKC / 2;                 // TMEM columns of a chunk's A tile (two bf16 a column)
constexpr int kAColBase = 128;                  // first TMEM column of the A slots
constexpr int kMaxN = 128;
constexpr int kMaxStages = 3;                   // A|B slots: TMEM columns 128 + 3 * 128 <= 512
constexpr int kSmemLimit = 224 * 1024;
constexpr int kSmemFixed = 1024 + 256;                // alignment slack, barriers
constexpr int kMaxRawStages = 4;

struct MmaParams {
  CUtensorMap wmap;      // the weights as [p][row_bytes / 4] 32-bit elements, box [128][68]
  const uint8_t* ximg;   // B operand image of this launch's activation rows
  const float* xinv;     // their inverse power-of-two scales
  float* Y;
  int ldy;
  int m, p, npad;        // npad = m rounded up to 16: B rows = accumulator columns
  int nchunks, ksplit, raw_stages, stages;
};

// ---- tcgen05 / cluster PTX wrappers ----------------------------------------
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// D (TMEM) += A * B^T, A read from tensor memory (lanes 0..127, columns
// from a_tmem), B from shared memory (descriptor b).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-collective store of 16 consecutive 32-bit columns of the warp's 32
// TMEM lanes (lane i of the warp writes TMEM lane (taddr >> 16) + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ float ld_peer(uint32_t local_saddr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}


// Block BLK (0..7) of a 272-byte raw row chunk as 32 f16 of scale * q (two
// a word, lower K first): the quants as exact f16 pairs (the sign-flipped
// byte under the exponent byte 0x64 is 1152 + q; one sub.f16x2 removes the
// 1152), times the block's f16 scale with one mul.f16x2 (the exact product
// rounded once).  v = the 48 bytes from byte 32 * BLK of the row, the
// block's scale at byte 2 * BLK of v.  range_ok: |scale| <= 511.75, so
// that |q * scale| <= 65504 (else the call's outputs become NaN).
template <int BLK>
__device__ __forceinline__ void decode_block_f16(const uint32_t (&v)[12], uint32_t (&pk)[16],
                                                 bool& range_ok) {
  constexpr int kScaleWord = BLK >> 1, kScaleShift = (BLK & 1) * 16;
  constexpr int kQWord = (BLK + 1) >> 1;  // odd BLK: quants word-aligned; even: from byte 2
  const uint32_t sb = (v[kScaleWord] >> kScaleShift) & 0xFFFFu;
  range_ok = range_ok && (sb & 0x7FFFu) <= 0x5FFFu;
  const uint32_t sc2 = sb | (sb << 16);
  const uint32_t bias = 0x64806480u;  // (1152, 1152)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t w;
    if constexpr ((BLK & 1) != 0)
      w = v[kQWord + k];
    else
      w = __funnelshift_r(v[kQWord + k], v[kQWord + k + 1], 16);
    w ^= 0x80808080u;
    uint32_t a = __byte_perm(w, 0x64646464u, 0x5140), b = __byte_perm(w, 0x64646464u, 0x7362);
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a) : "r"(a), "r"(bias));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(b) : "r"(b), "r"(bias));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(pk[2 * k]) : "r"(a), "r"(sc2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(pk[2 * k + 1]) : "r"(b), "r"(sc2));
  }
}


// 2-D tensor copy of the box at element (x, y) of the map into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Rows of the B operand of a 128-row block of mb activation rows: mb
// rounded up to 16 (zero rows past mb).
__host__ __device__ __forceinline__ int ximage_mp(int mb) { return (mb + 15) / 16 * 16; }

// The B operand image of the activations: for every 128-row block rb of X
// (mb rows, mp = ximage_mp(mb)) and every 128-element K half kh, the bytes
// [2 atoms][mp rows][128 B] at the block's base + kh * mp * 256, row r of an
// atom holding K elements 64 * atom + [0, 64) of activation row r as f16 of
// x * 2^e_r (rounded once; e_r puts the row's max |x| into [2^14, 2^15)),
// its 16-byte chunk c at position c ^ (r & 7) (canonical K-major 128-byte
// swizzle); inv[r] = 2^-e_r.  One CTA per activation row (grid = m), which
// also writes its share of the block's zero rows.
__global__ void __launch_bounds__(256) q8_ximage_kernel(const float* __restrict__ X, int ldx, int m,
                                                         int n, uint8_t* __restrict__ img,
                                                         float* __restrict__ inv) {
  griddep_wait();               // X (and the workspace's last readers) are done
  griddep_launch_dependents();  // the matmul kernel may start its prologue
  __shared__ float s_max[8];
  const int i = blockIdx.x, tid = threadIdx.x;
  const float* xr = X + (long long)i * ldx;
  // max |x| of the row (n % 256 == 0: whole float4s)
  float mx = 0.f;
  for (int k = 4 * tid; k < n; k += 1024) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) s_max[tid >> 5] = mx;
  __syncthreads();
  mx = s_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) mx = fmaxf(mx, s_max[w]);
  int ex = 0;
  if (mx > 0.f) frexpf(mx, &ex);
  const int e = mx > 0.f ? min(125, 15 - ex) : 0;  // (e >= -113 for any finite max)
  const float sc = __int_as_float((127 + e) << 23);
  if (tid == 0) inv[i] = __int_as_float((127 - e) << 23);
  const int rb = i / kMaxN, r = i % kMaxN;
  const int mb = min(kMaxN, m - rb * kMaxN), mp = ximage_mp(mb);
  uint8_t* base = img + (long long)rb * 256 * n;  // (full blocks before it: 128 rows)
  auto at = [&](int row, int kh, int c) {  // 16-byte chunk c (of 16) of image row `row`, half kh
    return base + (long long)kh * mp * 256 + (c >> 3) * mp * 128 + (row >> 3) * 1024 +
           (row & 7) * 128 + (((c & 7) ^ (row & 7)) << 4);
  };
  for (int q = tid; q < n / 8; q += 256) {  // 8 elements a chunk
    const float4 a = __ldg(reinterpret_cast<const float4*>(xr + 8 * q));
    const float4 b = __ldg(reinterpret_cast<const float4*>(xr + 8 * q + 4));
    const __half2 h0 = __floats2half2_rn(a.x * sc, a.y * sc), h1 = __floats2half2_rn(a.z * sc, a.w * sc);
    const __half2 h2 = __floats2half2_rn(b.x * sc, b.y * sc), h3 = __floats2half2_rn(b.z * sc, b.w * sc);
    const uint4 v = make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                               *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
    const int kh = q / 16, c = q % 16;
    *reinterpret_cast<uint4*>(at(r, kh, c)) = v;
    // zero rows mb .. mp - 1: this row takes every mb-th
    for (int zr = mb + r; zr < mp; zr += mb)
      *reinterpret_cast<uint4*>(at(zr, kh, c)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(kThreads, 1) q8_mma_kernel(const __grid_constant__ MmaParams P) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled B atoms
  const uint32_t base_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (base_s & 1023)) & 1023);
  const int b_atom = P.npad * 128;             // one 64-element K atom of B
  const int b_half = 2 * b_atom;               // B of 128 K elements (one image half)
  const int b_tile = 2 * b_half;               // B of a chunk
  const int S = P.stages;
  uint8_t* B = smem;                           // [S][2 halves][2 atoms][npad rows][128 B]
  uint8_t* raw = B + (size_t)S * b_tile;       // [raw_stages][128 rows][272 B]
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(raw + (size_t)P.raw_stages * kRawStage);
  uint64_t* raw_empty = raw_full + P.raw_stages;
  uint64_t* full = raw_empty + P.raw_stages;  // [S]: A tile written, B tile arrived
  uint64_t* empty = full + S;                 // [S]: their MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty + S);
  __shared__ int s_abort;
  __shared__ float s_ok;  // 1 if this CTA's partials are good (read by its cluster peers)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int r0 = blockIdx.x * kM;
  const int c_begin = (int)((long long)rank * P.nchunks / P.ksplit);
  const int c_end = (int)((long long)(rank + 1) * P.nchunks / P.ksplit);
  const int nloc = c_end - c_begin;
  // accumulator in columns [0, npad), A slots from kAColBase
  static_assert(kAColBase + kMaxStages * kACols <= 512, "TMEM columns");
  constexpr uint32_t kCols = 512;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  bool ok = true;
  int issued = 0;  // copies issued by this thread (producers)
  if (warp == kWProducer && lane == 0) {
    // every barrier, then the first weight copies at once (they need
    // neither TMEM nor the other warps)
    for (int s = 0; s < P.raw_stages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDeqWarps);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], kDeqWarps + 1);  // + the B copy's arrive (with its bytes)
      mbar_init(&empty[s], 1);
    }
    s_abort = 0;
    fence_barrier_init();
    const uint64_t pol = policy_evict_first();
    for (; issued < min(nloc, P.raw_stages); ++issued) {
      mbar_arrive_expect_tx(&raw_full[issued], (uint32_t)kRawStage);  // the whole box (zero-filled past p)
      tma_load_2d(raw + (size_t)issued * kRawStage, &P.wmap, (c_begin + issued) * (kRawRow / 4), r0,
                  &raw_full[issued], pol);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int valid_rows = min(kM, P.p - r0);

  if (warp == kWProducer) {
    // ---- one 2-D tensor copy per 8-block chunk of the 128 rows ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int i = issued; i < nloc; ++i) {
        const int st = i % P.raw_stages;
        if (!wait_or_abort(&raw_empty[st], (uint32_t)((i / P.raw_stages) - 1) & 1u, &s_abort))
          break;
        mbar_arrive_expect_tx(&raw_full[st], (uint32_t)kRawStage);
        tma_load_2d(raw + (size_t)st * kRawStage, &P.wmap, (c_begin + i) * (kRawRow / 4), r0,
                    &raw_full[st], pol);
        ++issued;
      }
    }
  } else if (warp == kXProducer) {
    // ---- one bulk copy per chunk of the B operand image (its two halves) ----
    if (lane == 0) {
      griddep_wait();  // the image is written by the kernel before this one
      fence_proxy_async_global();
      const uint64_t pol = policy_evict_last();  // every row tile reads it
      const uint8_t* src = P.ximg + (size_t)c_begin * b_tile;
      for (int i = 0; i < nloc; ++i) {
        const int st = i % S;
        if (i >= S && !wait_or_abort(&empty[st], (uint32_t)((i / S) - 1) & 1u, &s_abort)) break;
        mbar_arrive_expect_tx(&full[st], (uint32_t)b_tile);
        bulk_g2s(B + (size_t)st * b_tile, src + (size_t)i * b_tile, (uint32_t)b_tile, &full[st], pol);
        ++issued;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- 16 UMMAs (K = 16 each) per chunk, then commit ----
    if (lane == 0) {
      // f32 accumulator, f16 A and B, both K-major; N = npad, M = 128
      const uint32_t idesc = (1u << 4) | ((uint32_t)(P.npad >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
      // a K step adds its byte offset / 16 to the B descriptor's start
      // address (every address stays below 256 KB) and 8 columns to A's
      const uint64_t b_desc0 = sw128_desc(smem_u32(B));
      int st = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nloc; ++i) {
        if (!wait_ready(&full[st], ph, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t at = tmem + (uint32_t)(kAColBase + st * kACols);
        const uint64_t bd = b_desc0 + (uint64_t)((st * b_tile) >> 4);
#pragma unroll
        for (int s = 0; s < kKC / 16; ++s)
          umma_bf16_ts(tmem, at + (uint32_t)(8 * s),
                       bd + (((s >> 3) * b_half + ((s >> 2) & 1) * b_atom + (s & 3) * 32) >> 4), idesc,
                       (i > 0 || s > 0) ? 1u : 0u);
        umma_commit(&empty[st]);
        if (++st == S) {
          st = 0;
          ph ^= 1u;
        }
      }
    }
  } else {
    // ---- dequantisation warps: weight row 32 (warp % 4) + lane (the
    // thread's TMEM lane), blocks bsel and bsel + 4 of each chunk ----
    const int q = warp & 3, bsel = warp >> 2;
    const int row = 32 * q + lane;
    bool range_ok = true;  // every block scale keeps scale * q within f16
    // 48 bytes from byte 32 * blk of the row: 16-byte aligned, and the 34
    // bytes of block blk start 2 * blk bytes in (rows of 272 bytes: the
    // loads of 8 consecutive rows cover the 32 banks once)
    const uint32_t src0 = smem_u32(raw) + (uint32_t)(row * kRawRow + 32 * bsel);
    // TMEM address of this warp's lanes, slot 0, block bsel's 16 columns
    // (block bsel + 4: 64 columns further)
    const uint32_t a_lane = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kAColBase + 16 * bsel);
    int rs = 0, st = 0;
    uint32_t rph = 0, ph = 0;  // raw stage, A|B slot, their parities
    for (int i = 0; i < nloc; ++i) {
      ok = wait_ready(&raw_full[rs], rph, &s_abort) && ok;
      const uint32_t src = src0 + (uint32_t)(rs * kRawStage);
      uint32_t v[12], u[12];
      {
        const uint4 v0 = lds128(src), v1 = lds128(src + 16), v2 = lds128(src + 32);
        const uint4 u0 = lds128(src + 128), u1 = lds128(src + 144), u2 = lds128(src + 160);
        v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
        v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        v[8] = v2.x; v[9] = v2.y; v[10] = v2.z; v[11] = v2.w;
        u[0] = u0.x; u[1] = u0.y; u[2] = u0.z; u[3] = u0.w;
        u[4] = u1.x; u[5] = u1.y; u[6] = u1.z; u[7] = u1.w;
        u[8] = u2.x; u[9] = u2.y; u[10] = u2.z; u[11] = u2.w;
      }
      // the raw stage is read once the values are in registers
      __syncwarp();
      if (lane == 0) mbar_arrive(&raw_empty[rs]);
      if (++rs == P.raw_stages) {
        rs = 0;
        rph ^= 1u;
      }
      uint32_t pa[16], pb[16];
      switch (bsel) {  // the same for the warp's 32 lanes
        case 0: decode_block_f16<0>(v, pa, range_ok); decode_block_f16<4>(u, pb, range_ok); break;
        case 1: decode_block_f16<1>(v, pa, range_ok); decode_block_f16<5>(u, pb, range_ok); break;
        case 2: decode_block_f16<2>(v, pa, range_ok); decode_block_f16<6>(u, pb, range_ok); break;
        default: decode_block_f16<3>(v, pa, range_ok); decode_block_f16<7>(u, pb, range_ok); break;
      }
      // slot st is free once the MMAs of chunk i - S completed
      if (i >= S) {
        ok = wait_ready(&empty[st], ph ^ 1u, &s_abort) && ok;
        tc_fence_after();
      }
      const uint32_t ta = a_lane + (uint32_t)(st * kACols);
      tmem_st16(ta, pa);
      tmem_st16(ta + 64u, pb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
      if (++st == S) {
        st = 0;
        ph ^= 1u;
      }
    }
    ok = ok && range_ok;
  }

  // every MMA of the CTA has completed once the last chunk's commit arrives
  if (nloc > 0)
    ok = wait_or_abort(&empty[(nloc - 1) % S], (uint32_t)((nloc - 1) / S) & 1u, &s_abort) && ok;
  ok = __syncthreads_and(ok && !*(volatile int*)&s_abort);
  // the next call's image kernel may start during the epilogue (it waits
  // for this grid before it touches X or the workspace)
  griddep_launch_dependents();
  if (!ok && lane == 0) {
    // copies issued but never consumed may still be in flight
    if (warp == kWProducer)
      for (int k = max(0, issued - P.raw_stages); k < issued; ++k)
        mbar_wait(&raw_full[k % P.raw_stages], (uint32_t)(k / P.raw_stages) & 1u);
    if (warp == kXProducer)
      for (int k = max(0, issued - S); k < issued; ++k) mbar_wait(&full[k % S], (uint32_t)(k / S) & 1u);
  }
  __syncthreads();
  tc_fence_after();
  // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) + [0, 32) (rows),
  // columns 16 g + [0, 16) (activation rows) for g = w / 4, w / 4 + 4, ...,
  // and undoes the rows' power-of-two scales
  const float nan = __int_as_float(0x7fc00000);
  auto read_cols = [&](int g, float (&v)[16]) {
    if (nloc > 0) {
      tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(16 * g), v);
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] *= __ldg(P.xinv + min(16 * g + k, P.m - 1));
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 0.f;
    }
  };
  if (P.ksplit == 1) {
    if (warp < kDeqWarps) {
      const int r = 32 * (warp & 3) + lane;
      for (int g = warp >> 2; 16 * g < P.npad; g += kDeqWarps / 4) {
        float v[16];
        read_cols(g, v);
        if (r < valid_rows) {
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (16 * g + k < P.m) P.Y[(long long)(16 * g + k) * P.ldy + r0 + r] = ok ? v[k] : nan;
        }
      }
    }
  } else {
    // partial tile [npad][128] in the raw ring, then rank r sums and stores
    // every ksplit-th element of the tile, the partials of all ranks added
    // in rank order
    float* part = reinterpret_cast<float*>(raw);
    if (warp < kDeqWarps) {
      const int r = 32 * (warp & 3) + lane;
      for (int g = warp >> 2; 16 * g < P.npad; g += kDeqWarps / 4) {
        float v[16];
        read_cols(g, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) part[(16 * g + k) * kM + r] = v[k];
      }
    }
    if (tid == 0) s_ok = ok ? 1.f : 0.f;
    __syncthreads();
    cluster_sync();  // every CTA's partial tile is complete
    const uint32_t part_s = smem_u32(part);
    bool ok_all = true;  // every rank's partials are good
    for (int k = 0; k < P.ksplit; ++k) ok_all = ok_all && ld_peer(smem_u32(&s_ok), (uint32_t)k) != 0.f;
    for (int e = tid * P.ksplit + (int)rank; e < P.m * kM; e += kThreads * P.ksplit) {
      const int col = e / kM, r = e % kM;
      if (r >= valid_rows) continue;
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < P.ksplit) v[k] = ld_peer(part_s + (uint32_t)(col * kM + r) * 4u, (uint32_t)k);
      float sum = v[0];
#pragma unroll
      for (int k = 1; k < 8; ++k)
        if (k < P.ksplit) sum += v[k];
      P.Y[(long long)col * P.ldy + r0 + r] = ok_all ? sum : nan;
    }
    cluster_sync();  // every CTA keeps its shared memory until its peers have read it
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
  }
}

}  // namespace

// cuTensorMapEncodeTiled from the driver (looked up once, no link-time
// dependency on libcuda); null if unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Clusters of `ksplit` CTAs (one per SM, smem bytes each) that the device
// runs at once; cached per (device, ksplit, smem).
int max_active_clusters(int ksplit, int smem) {
  static std::mutex mu;
  static std::map<std::pair<int, std::pair<int, int>>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_pair(dev, std::make_pair(ksplit, smem));
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, ksplit, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = ksplit;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, q8_mma_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

// Bytes of the B operand image of m activation rows of n elements: two
// bytes per element, rows rounded up to 16 per 128-row block.
size_t mma_small_m_image_bytes(int m, int n) {
  size_t rows = 0;
  for (int i0 = 0; i0 < m; i0 += kMaxN) rows += (size_t)ximage_mp(std::min(kMaxN, m - i0));
  return rows * (size_t)n * 2;
}

// Workspace bytes of the tensor-core path: the image and m inverse scales
// (f32, 16-byte padded); 0 when it does not take the shape (m < 9 or n not a
// multiple of 256).  Host arithmetic only.
size_t mma_small_m_workspace(int m, int n) {
  if (m < 9 || n <= 0 || n % kKC != 0) return 0;
  return mma_small_m_image_bytes(m, n) + (size_t)(m + 3) / 4 * 16;  // + the rows' inverse scales
}

// Runs the tensor-core path with `ws` (mma_small_m_workspace(m, n) bytes,
// 16-byte aligned) holding the activation image; Q8D_EUNSUPPORTED for
// shapes it does not take or without a tensor-map encoder, which the caller
// routes to the CUDA-core path.
int mma_small_m_launch(const float* X, int ldx, const uint8_t* w, float* Y, int ldy, int m, int n,
                       int p, void* ws, cudaStream_t stream) {
  const EncodeTiledFn encode = encode_tiled();
  if (mma_small_m_workspace(m, n) == 0 || !encode) return Q8D_EUNSUPPORTED;
  // the weights as p rows of row_bytes / 4 32-bit elements (row_bytes is a
  // multiple of 272, so of 16), box = one chunk of 128 rows
  const long long row_bytes = (long long)(n / kQBlock) * kQBlockBytes;
  CUtensorMap wmap;
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)p};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(kRawRow / 4), (cuuint32_t)kM};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(w), gdim, gstride, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return Q8D_EUNSUPPORTED;
  }
  const int crc = configure_kernel(reinterpret_cast<const void*>(q8_mma_kernel), kSmemLimit, false);
  if (crc) return crc;
  uint8_t* img = static_cast<uint8_t*>(ws);
  float* inv = reinterpret_cast<float*>(img + mma_small_m_image_bytes(m, n));
  {
    const int rc = launch_ex(q8_ximage_kernel, dim3((unsigned)m), dim3(256), 0, stream, true, X, ldx,
                             m, n, img, inv);
    if (rc) return rc;
  }
  const int row_tiles = (p + kM - 1) / kM;
  const int nchunks = n / kKC;
  const int sms = sm_count();
  for (int i0 = 0; i0 < m; i0 += kMaxN) {
    MmaParams P{};
    P.wmap = wmap;
    P.m = std::min(kMaxN, m - i0);
    P.npad = ximage_mp(P.m);
    P.ximg = img + (size_t)i0 * 2 * n;
    P.xinv = inv + i0;
    P.Y = Y + (long long)i0 * ldy;
    P.ldy = ldy;
    P.p = p;
    P.nchunks = nchunks;
    // three A|B slots (two when three leave fewer than three weight
    // stages) and as many weight stages as fit (2..kMaxRawStages)
    const int b_tile = P.npad * 512, left = kSmemLimit - kSmemFixed;
    P.stages = kMaxStages;
    if (left - P.stages * b_tile < 3 * kRawStage) P.stages = 2;
    P.raw_stages = std::min(kMaxRawStages, (left - P.stages * b_tile) / kRawStage);
    if (P.raw_stages < 2) return Q8D_EUNSUPPORTED;
    const int smem = kSmemFixed + P.stages * b_tile + P.raw_stages * kRawStage;
    // K split: the largest (<= 8, <= the chunks) whose row_tiles clusters
    // all run at once (clusters of 5 or 6 pack worse into the GPCs than 4)
    P.ksplit = std::max(1, std::min({8, sms / row_tiles, nchunks}));
    while (P.ksplit > 1 && max_active_clusters(P.ksplit, smem) < row_tiles) --P.ksplit;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(row_tiles, P.ksplit, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = P.ksplit;
    attr[0].val.clusterDim.z = 1;
    // a programmatic dependent: the prologue and the weight stream start
    // while the image is written; the activation producer waits for it
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, q8_mma_kernel, P);
    if (e != cudaSuccess) return record_cuda(e);
  }
  return Q8D_OK;
}

}  // namespace q8d
