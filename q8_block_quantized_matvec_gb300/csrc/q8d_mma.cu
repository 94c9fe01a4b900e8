// Tensor-core path of q8d_matmul_small_m (m >= 9): Y[i][r] = sum_k X[i][k] W[r][k].
//
// At m >= 9 activation rows the product is a real dense contraction (2m
// flops per weight element, 30-120 flop/byte at m = 16..64) that would make
// the CUDA cores the bottleneck, so it runs on the 5th-generation tensor
// cores ("Metal Backend Optimizations": the quantised GEMM tier used once
// more than one token is in flight stages dequantised weights in on-chip
// memory; here the tile feeds tcgen05.mma instead of SIMD-group matrices).
//
//  * CTA = 128 weight rows (the MMA's M) x a K range; a thread-block cluster
//    of `ksplit` CTAs along K shares one output tile and reduces the fp32
//    partials through distributed shared memory in rank order
//    (deterministic, no global scratch, no atomics).
//  * Warp roles, so that dequantisation, weight streaming and MMAs overlap:
//    one producer warp streams raw Q8_0 bytes (8 blocks = 272 bytes per row
//    per 256-element chunk, the 128 rows a weight-row stride apart) by one
//    2-D tensor copy per chunk (TMA: 68 32-bit elements x 128 rows; every x
//    coordinate a multiple of 16 bytes; rows past the matrix zero-filled)
//    into a ring of stages; 16 dequantising warps turn each half chunk (128
//    K elements) into bf16 A and B tiles in the canonical K-major
//    128-byte-swizzled layout (a thread: one (row, block) of scale * q,
//    computed exactly in f32 and rounded once, and its share of the X rows
//    rounded to bf16), double-buffered; one MMA warp issues
//    tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 -> f32, M = 128,
//    N = m rounded up to 16, K = 16 per instruction) on a buffer as soon as
//    it is written and commits to that buffer's mbarrier, which frees it
//    for the half chunk after next.  The epilogue reads TMEM with
//    tcgen05.ld.
// Accuracy: one bf16 rounding of each weight and activation, f32
// accumulation: |error| <= ~2^-8 * sum|terms| per output.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is looked up at run time
#include <cuda_bf16.h>

#include <algorithm>

#include "q8d_gemv.cuh"
#include "q8d_internal.cuh"

namespace q8d {
namespace {

using mv::wait_or_abort;

constexpr int kDeqWarps = 16;                   // dequantising warps
constexpr int kDeqThreads = kDeqWarps * 32;
constexpr int kThreads = kDeqThreads + 64;      // + the TMA producer warp + the MMA warp
constexpr int kM = 128;                         // weight rows per CTA (MMA M)
constexpr int kKC = 256;                        // K elements per raw chunk (one tensor copy)
constexpr int kHalfK = 128;                     // K elements per A/B tile (half a chunk)
constexpr int kRawRow = (kKC / kQBlock) * kQBlockBytes;  // 272 bytes
constexpr int kRawStage = kM * kRawRow;         // 34816 bytes
constexpr int kAtomBytes = kM * 128;            // one 64-element K atom of A
constexpr int kAHalf = 2 * kAtomBytes;          // an A tile of 128 K elements: 32 KB
constexpr int kMaxN = 128;
constexpr int kMaxPieces = kMaxN * (kHalfK / 8) / kDeqThreads;  // B pieces per thread (<= 4)

struct MmaParams {
  CUtensorMap wmap;  // the weights as [p][row_bytes / 4] 32-bit elements, box [128][68]
  const float* X;
  int ldx;
  const uint8_t* w;
  float* Y;
  int ldy;
  int m, n, p, npad;
  int nchunks, ksplit, raw_stages;
  long long row_bytes;
  int* d_err;
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

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
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

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of the 16-byte chunk holding K elements [8c, 8c+8) of row r
// inside a K-major SW128 tile whose 64-element atoms are atom_bytes apart.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c, int atom_bytes) {
  const int atom = c >> 3, cc = c & 7;
  return (uint32_t)(atom * atom_bytes + (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4));
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

__global__ void __launch_bounds__(kThreads, 1) q8_mma_kernel(const __grid_constant__ MmaParams P) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled atoms
  const uint32_t base_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (base_s & 1023)) & 1023);
  const int b_atom = P.npad * 128;             // one 64-element K atom of B
  uint8_t* A = smem;                           // [2][2 atoms][128 rows][128 B]
  uint8_t* B = A + 2 * kAHalf;                 // [2][2 atoms][npad rows][128 B]
  uint8_t* raw = B + 2 * 2 * b_atom;           // [raw_stages][128 rows][272 B]
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(raw + (size_t)P.raw_stages * kRawStage);
  uint64_t* raw_empty = raw_full + P.raw_stages;
  uint64_t* ab_full = raw_empty + P.raw_stages;  // [2]: half-chunk tiles written
  uint64_t* ab_empty = ab_full + 2;              // [2]: their MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ab_empty + 2);
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int r0 = blockIdx.x * kM;
  const int c_begin = (int)((long long)rank * P.nchunks / P.ksplit);
  const int c_end = (int)((long long)(rank + 1) * P.nchunks / P.ksplit);
  const int nloc = c_end - c_begin;
  const int nhalf = 2 * nloc;
  const uint32_t ncols = P.npad <= 32 ? 32u : (P.npad <= 64 ? 64u : 128u);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < P.raw_stages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDeqWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ab_full[b], kDeqWarps);
      mbar_init(&ab_empty[b], 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int valid_rows = min(kM, P.p - r0);
  bool ok = true;
  int issued = 0;

  if (warp == kDeqWarps) {
    // ---- producer: one 2-D tensor copy per 8-block chunk of the 128 rows ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < nloc; ++i) {
        const int st = i % P.raw_stages;
        if (i >= P.raw_stages &&
            !wait_or_abort(&raw_empty[st], (uint32_t)((i / P.raw_stages) - 1) & 1u, &s_abort))
          break;
        mbar_arrive_expect_tx(&raw_full[st], (uint32_t)kRawStage);  // the whole box (zero-filled past p)
        tma_load_2d(raw + (size_t)st * kRawStage, &P.wmap, (c_begin + i) * (kRawRow / 4), r0,
                    &raw_full[st], pol);
        ++issued;
      }
    }
  } else if (warp == kDeqWarps + 1) {
    // ---- MMA issuer: 8 UMMAs (K = 16 each) per half-chunk, then commit ----
    if (lane == 0) {
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                             ((uint32_t)(P.npad >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
      for (int j = 0; j < nhalf; ++j) {
        const int b = j & 1;
        if (!wait_or_abort(&ab_full[b], (uint32_t)(j >> 1) & 1u, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(A + b * kAHalf), b0 = smem_u32(B + b * 2 * b_atom);
#pragma unroll
        for (int s = 0; s < kHalfK / 16; ++s) {
          const uint32_t koff = (uint32_t)((s & 3) * 32);
          umma_bf16(tmem, sw128_desc(a0 + (s >> 2) * kAtomBytes + koff),
                    sw128_desc(b0 + (s >> 2) * b_atom + koff), idesc, (j > 0 || s > 0) ? 1u : 0u);
        }
        umma_commit(&ab_empty[b]);
      }
    }
  } else {
    // ---- dequantisation warps: one (row, block) item and up to npad/32 B
    // pieces per thread and half-chunk ----
    const int rr = (tid & 7) | ((tid >> 5) << 3);
    const int blk = (tid >> 3) & 3;
    const int nb = P.npad * (kHalfK / 8) / kDeqThreads;  // B pieces per thread (may be 0 or fractional)
    const int npieces = P.npad * (kHalfK / 8);
    for (int j = 0; j < nhalf; ++j) {
      const int i = j >> 1, h = j & 1, b = j & 1, c = c_begin + i;
      const int st = i % P.raw_stages;
      // B pieces of this half: X rows, K elements c*256 + h*128 + [8 cch, 8 cch + 8)
      float4 xa[kMaxPieces], xb[kMaxPieces];
#pragma unroll
      for (int u = 0; u < kMaxPieces; ++u) {
        const int e = tid + u * kDeqThreads;
        const int row = (e & 7) | ((e >> 7) << 3), cch = (e >> 3) & 15;
        xa[u] = xb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (u <= nb && e < npieces && row < P.m) {
          const float4* xp = reinterpret_cast<const float4*>(
              P.X + (long long)row * P.ldx + (long long)c * kKC + h * kHalfK + cch * 8);
          xa[u] = __ldg(xp);
          xb[u] = __ldg(xp + 1);
        }
      }
      if (h == 0) ok = wait_or_abort(&raw_full[st], (uint32_t)(i / P.raw_stages) & 1u, &s_abort) && ok;
      // the item's block (raw row rr, block 4h + blk) as bf16 of scale * q
      const uint8_t* rs = raw + (size_t)st * kRawStage;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) pk[k] = 0u;
      if (rr < valid_rows) {
        const uint32_t off = (uint32_t)(rr * kRawRow + (4 * h + blk) * kQBlockBytes);
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(rs);
        const uint32_t wi = off >> 2;
        const bool odd = (off & 2u) != 0;
        uint32_t a[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) a[k] = s32[wi + k];
        const float sc = f16_bits_to_f32(odd ? (a[0] >> 16) : (a[0] & 0xFFFFu));
        const uint32_t sh = odd ? 32u : 16u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t wq = __funnelshift_rc(a[k], a[k + 1], sh) ^ 0x80808080u;
          const float q0 = magic_byte(wq, magic_sel(0)) - kMagicBias;
          const float q1 = magic_byte(wq, magic_sel(1)) - kMagicBias;
          const float q2 = magic_byte(wq, magic_sel(2)) - kMagicBias;
          const float q3 = magic_byte(wq, magic_sel(3)) - kMagicBias;
          pk[2 * k] = bf16x2(q0 * sc, q1 * sc);
          pk[2 * k + 1] = bf16x2(q2 * sc, q3 * sc);
        }
      }
      // (the raw stage is read: release it after the chunk's second half)
      if (h == 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[st]);
      }
      // tiles of buffer b are free once the MMAs of half j - 2 completed
      if (j >= 2) ok = wait_or_abort(&ab_empty[b], (uint32_t)((j >> 1) - 1) & 1u, &s_abort) && ok;
      uint8_t* Ab = A + b * kAHalf;
      const int c0 = blk * 4;  // 16-byte chunk index of the block's first 8 elements (in the half)
      *reinterpret_cast<uint4*>(Ab + sw128_offset(rr, c0 + 0, kAtomBytes)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(Ab + sw128_offset(rr, c0 + 1, kAtomBytes)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      *reinterpret_cast<uint4*>(Ab + sw128_offset(rr, c0 + 2, kAtomBytes)) = make_uint4(pk[8], pk[9], pk[10], pk[11]);
      *reinterpret_cast<uint4*>(Ab + sw128_offset(rr, c0 + 3, kAtomBytes)) = make_uint4(pk[12], pk[13], pk[14], pk[15]);
      uint8_t* Bb = B + b * 2 * b_atom;
#pragma unroll
      for (int u = 0; u < kMaxPieces; ++u) {
        const int e = tid + u * kDeqThreads;
        if (u <= nb && e < npieces) {
          const int row = (e & 7) | ((e >> 7) << 3), cch = (e >> 3) & 15;
          *reinterpret_cast<uint4*>(Bb + sw128_offset(row, cch, b_atom)) =
              make_uint4(bf16x2(xa[u].x, xa[u].y), bf16x2(xa[u].z, xa[u].w),
                         bf16x2(xb[u].x, xb[u].y), bf16x2(xb[u].z, xb[u].w));
        }
      }
      // generic-proxy shared writes -> visible to the tensor core (async proxy)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&ab_full[b]);
    }
  }

  // every MMA of the CTA has completed once the last half's commit arrives
  if (nhalf > 0)
    ok = wait_or_abort(&ab_empty[(nhalf - 1) & 1], (uint32_t)((nhalf - 1) >> 1) & 1u, &s_abort) && ok;
  ok = __syncthreads_and(ok && !*(volatile int*)&s_abort);
  if (!ok && warp == kDeqWarps && lane == 0) {
    // copies issued but never consumed may still be in flight
    for (int k = max(0, issued - P.raw_stages); k < issued; ++k)
      mbar_wait(&raw_full[k % P.raw_stages], (uint32_t)(k / P.raw_stages) & 1u);
  }
  // ---- epilogue: TMEM -> shared partial tile [npad][128] (reusing A) ----
  tc_fence_after();
  float* part = reinterpret_cast<float*>(A);
  if (warp < 4) {
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < P.npad; c0 += 16) {
      float v[16];
      if (nloc > 0) {
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) part[(c0 + j) * kM + row] = v[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (!ok && tid == 0 && P.d_err) atomicOr(P.d_err, Q8D_DERR_WAIT);
  cluster_sync();  // every CTA's partial tile is complete
  if (rank == 0) {
    const uint32_t part_s = smem_u32(part);
    for (int e = tid; e < P.m * kM; e += kThreads) {
      const int col = e / kM, row = e % kM;
      if (row >= valid_rows) continue;
      float s = part[col * kM + row];
      for (int q = 1; q < P.ksplit; ++q) s += ld_peer(part_s + (uint32_t)(col * kM + row) * 4u, q);
      P.Y[(long long)col * P.ldy + r0 + row] = ok ? s : __int_as_float(0x7fc00000);
    }
  }
  cluster_sync();  // peers keep their shared memory until rank 0 has read it
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols)
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

// Runs the tensor-core path; Q8D_EUNSUPPORTED for shapes it does not take
// (n not a multiple of 256, or no tensor-map encoder), which the caller
// routes to the CUDA-core path.
int mma_small_m_launch(const float* X, int ldx, const uint8_t* w, float* Y, int ldy, int m, int n,
                       int p, cudaStream_t stream) {
  if (n % kKC != 0) return Q8D_EUNSUPPORTED;
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return Q8D_EUNSUPPORTED;
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
  const int crc = configure_kernel(reinterpret_cast<const void*>(q8_mma_kernel), 224 * 1024, false);
  if (crc) return crc;
  const int row_tiles = (p + kM - 1) / kM;
  const int nchunks = n / kKC;
  const int sms = sm_count();
  for (int i0 = 0; i0 < m; i0 += kMaxN) {
    MmaParams P{};
    P.wmap = wmap;
    P.m = std::min(kMaxN, m - i0);
    P.npad = (P.m + 15) / 16 * 16;
    P.X = X + (long long)i0 * ldx;
    P.ldx = ldx;
    P.w = w;
    P.Y = Y + (long long)i0 * ldy;
    P.ldy = ldy;
    P.n = n;
    P.p = p;
    P.nchunks = nchunks;
    P.row_bytes = row_bytes;
    P.ksplit = std::max(1, std::min({8, sms / row_tiles, nchunks}));
    const int fixed = 2 * kAHalf + 2 * 2 * P.npad * 128 + 1024 + 128;
    P.raw_stages = (fixed + 3 * kRawStage <= 224 * 1024) ? 3 : 2;
    const int smem = fixed + P.raw_stages * kRawStage;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(row_tiles, P.ksplit, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = P.ksplit;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, q8_mma_kernel, P);
    if (e != cudaSuccess) return record_cuda(e);
  }
  return Q8D_OK;
}

}  // namespace q8d
