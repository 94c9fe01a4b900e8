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
//  * Raw Q8_0 bytes (8 blocks = 272 bytes per row per 256-element chunk) are
//    streamed into a ring of stages, a chunk's 128 rows by one 2-D tensor
//    copy (TMA: the rows are a weight-row stride apart in global memory;
//    the 272 bytes are 68 32-bit elements, so the box stays within TMA's 256
//    elements per dimension and every x coordinate is a multiple of 16
//    bytes; rows past the matrix are zero-filled).  All threads
//    dequantise scale*q exactly in f32, round once to bf16 and store the A
//    tile in the canonical K-major 128-byte-swizzled layout; X rows are
//    rounded to bf16 into the B tile the same way.
//  * One thread issues tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 ->
//    f32, M = 128, N = m rounded up to 16, K = 16 per instruction) into a
//    TMEM accumulator; tcgen05.commit signals an mbarrier when the tiles may
//    be overwritten.  The epilogue reads TMEM with tcgen05.ld.
// Accuracy: one bf16 rounding of each weight and activation, f32
// accumulation: |error| <= ~2^-8 * sum|terms| per output.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is looked up at run time
#include <cuda_bf16.h>

#include <algorithm>

#include "q8d_internal.cuh"

namespace q8d {
namespace {

constexpr int kThreads = 512;
constexpr int kM = 128;                         // weight rows per CTA (MMA M)
constexpr int kKC = 256;                        // K elements per chunk
constexpr int kRawRow = (kKC / kQBlock) * kQBlockBytes;  // 272 bytes
constexpr int kRawStage = kM * kRawRow;         // 34816 bytes
constexpr int kAtomBytes = kM * 128;            // one 64-element K atom of A
constexpr int kATile = 4 * kAtomBytes;          // 65536 bytes
constexpr int kMaxN = 128;
constexpr int kBGroup = 4;                      // B-tile pieces a thread loads at once

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
  uint8_t* A = smem;
  uint8_t* B = A + kATile;
  const int b_atom = P.npad * 128;
  uint8_t* raw = B + 4 * b_atom;
  uint64_t* raw_bar = reinterpret_cast<uint64_t*>(raw + (size_t)P.raw_stages * kRawStage);
  uint64_t* mma_bar = raw_bar + P.raw_stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int r0 = blockIdx.x * kM;
  const int c_begin = (int)((long long)rank * P.nchunks / P.ksplit);
  const int c_end = (int)((long long)(rank + 1) * P.nchunks / P.ksplit);
  const int nloc = c_end - c_begin;
  const uint32_t ncols = P.npad <= 32 ? 32u : (P.npad <= 64 ? 64u : 128u);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < P.raw_stages; ++s) mbar_init(&raw_bar[s], 1);
    mbar_init(mma_bar, 1);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t pol = policy_evict_first();
  const int valid_rows = min(kM, P.p - r0);

  auto issue = [&](int i) {  // warp 0: one tensor copy of the chunk's 128 rows
    if (i >= nloc || lane != 0) return;
    const int c = c_begin + i;
    uint64_t* bar = &raw_bar[i % P.raw_stages];
    uint8_t* dst = raw + (size_t)(i % P.raw_stages) * kRawStage;
    mbar_arrive_expect_tx(bar, (uint32_t)kRawStage);  // the whole box (zero-filled past p)
    tma_load_2d(dst, &P.wmap, c * (kRawRow / 4), r0, bar, pol);
  };
  if (warp == 0)
    for (int i = 0; i < P.raw_stages; ++i) issue(i);

  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(P.npad >> 3) << 17) |
                         ((uint32_t)(kM >> 4) << 24);
  bool ok = true;

  // B tile pieces: thread tid takes pieces tid + k * kThreads (k < nit), 8
  // K elements of one X row each, loaded kBGroup at a time (one L2 round
  // trip per group) before they are rounded and stored
  const int nit = P.npad * 32 / kThreads;
  auto b_load = [&](int c, int k0, float4 (&va)[kBGroup], float4 (&vb)[kBGroup]) {
#pragma unroll
    for (int u = 0; u < kBGroup; ++u) {
      const int e = tid + (k0 + u) * kThreads;
      const int row = e & 7 | ((e >> 8) << 3), cch = (e >> 3) & 31;  // 8 rows per quarter-warp
      va[u] = vb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k0 + u < nit && row < P.m) {
        const float4* xp = reinterpret_cast<const float4*>(P.X + (long long)row * P.ldx +
                                                           (long long)c * kKC + cch * 8);
        va[u] = __ldg(xp);
        vb[u] = __ldg(xp + 1);
      }
    }
  };
  auto b_store = [&](int k0, const float4 (&va)[kBGroup], const float4 (&vb)[kBGroup]) {
#pragma unroll
    for (int u = 0; u < kBGroup; ++u) {
      if (k0 + u >= nit) break;
      const int e = tid + (k0 + u) * kThreads;
      const int row = e & 7 | ((e >> 8) << 3), cch = (e >> 3) & 31;
      const uint4 v = make_uint4(bf16x2(va[u].x, va[u].y), bf16x2(va[u].z, va[u].w),
                                 bf16x2(vb[u].x, vb[u].y), bf16x2(vb[u].z, vb[u].w));
      *reinterpret_cast<uint4*>(B + sw128_offset(row, cch, b_atom)) = v;
    }
  };

  // the first group of chunk i's B pieces is loaded during chunk i - 1 (all
  // of a thread's pieces for m <= 64): its L2 latency overlaps the previous
  // chunk's dequantisation and MMAs
  float4 va[kBGroup], vb[kBGroup];
  if (nloc > 0) b_load(c_begin, 0, va, vb);
  for (int i = 0; i < nloc; ++i) {
    const int c = c_begin + i;
    // (a) the previous chunk's MMAs must have finished reading A and B
    if (i > 0) ok = ok && mbar_wait(mma_bar, (uint32_t)(i - 1) & 1u);
    // (b) B tile: X[0..m) rows, K elements [c*256, c*256+256), rounded to bf16
    b_store(0, va, vb);
    for (int k0 = kBGroup; k0 < nit; k0 += kBGroup) {
      b_load(c, k0, va, vb);
      b_store(k0, va, vb);
    }
    if (i + 1 < nloc) b_load(c + 1, 0, va, vb);
    // (c) raw weight bytes of this chunk
    ok = ok && mbar_wait(&raw_bar[i % P.raw_stages], (uint32_t)(i / P.raw_stages) & 1u);
    if (!__syncthreads_and(ok)) break;
    // (d) dequantise 128 rows x 8 blocks into the A tile
    const uint8_t* rs = raw + (size_t)(i % P.raw_stages) * kRawStage;
    for (int f = tid; f < kM * 8; f += kThreads) {
      const int rr = (f & 7) | (((f >> 5) & 15) << 3);
      const int blk = ((f >> 3) & 3) | ((f >> 9) << 2);
      uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0, o2 = o0, o3 = o0;
      if (rr < valid_rows) {
        const uint32_t off = (uint32_t)(rr * kRawRow + blk * kQBlockBytes);
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(rs);
        const uint32_t wi = off >> 2;
        const bool odd = (off & 2u) != 0;
        uint32_t a[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) a[k] = s32[wi + k];
        const float sc = f16_bits_to_f32(odd ? (a[0] >> 16) : (a[0] & 0xFFFFu));
        const uint32_t sh = odd ? 32u : 16u;
        uint32_t pk[16];
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
        o0 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        o1 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        o2 = make_uint4(pk[8], pk[9], pk[10], pk[11]);
        o3 = make_uint4(pk[12], pk[13], pk[14], pk[15]);
      }
      const int c0 = blk * 4;  // 16-byte chunk index of the block's first 8 elements
      *reinterpret_cast<uint4*>(A + sw128_offset(rr, c0 + 0, kAtomBytes)) = o0;
      *reinterpret_cast<uint4*>(A + sw128_offset(rr, c0 + 1, kAtomBytes)) = o1;
      *reinterpret_cast<uint4*>(A + sw128_offset(rr, c0 + 2, kAtomBytes)) = o2;
      *reinterpret_cast<uint4*>(A + sw128_offset(rr, c0 + 3, kAtomBytes)) = o3;
    }
    // generic-proxy smem writes -> visible to the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
      if (lane == 0) {
        tc_fence_after();
        const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
#pragma unroll
        for (int s = 0; s < kKC / 16; ++s) {
          const uint32_t koff = (uint32_t)((s & 3) * 32);
          umma_bf16(tmem, sw128_desc(a0 + (s >> 2) * kAtomBytes + koff),
                    sw128_desc(b0 + (s >> 2) * b_atom + koff), idesc, (i > 0 || s > 0) ? 1u : 0u);
        }
        umma_commit(mma_bar);
      }
      __syncwarp();
      issue(i + P.raw_stages);  // the raw stage just consumed is free again
    }
  }

  // ---- epilogue: TMEM -> shared partial tile [npad][128] (reusing A) ----
  if (nloc > 0) ok = ok && mbar_wait(mma_bar, (uint32_t)(nloc - 1) & 1u);
  ok = __syncthreads_and(ok);
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
  const int crc = configure_kernel(reinterpret_cast<const void*>(q8_mma_kernel), 227 * 1024, false);
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
    const int fixed = kATile + 4 * P.npad * 128 + 1024 + 64;
    P.raw_stages = (fixed + 3 * kRawStage <= 227 * 1024) ? 3 : 2;
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
