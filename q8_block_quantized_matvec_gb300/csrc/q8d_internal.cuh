// Internal helpers shared by the q8d CUDA translation units (sm_103a only).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q8d.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "q8d is written for Blackwell (sm_103a); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace q8d {

constexpr int kQBlock = 32;       // quants per Q8_0 block
constexpr int kQBlockBytes = 34;  // 2-byte scale + 32 quants

// Upper bound on polls of an mbarrier before a kernel gives up, records
// Q8D_DERR_WAIT and leaves.  try_wait itself suspends for a hardware-chosen
// interval, so this is far longer than any legitimate wait (seconds).
constexpr uint32_t kWaitLimit = 1u << 24;

// ---- host-side error bookkeeping (q8d_api.cu) -----------------------------
int record_cuda(cudaError_t e);  // stores e for q8d_last_cuda_error, returns Q8D_ECUDA
int sm_count();                  // SMs of the current device (cached per device)
int check_launch();              // cudaGetLastError -> status
// Sets a kernel's dynamic shared-memory limit to smem_bytes (and, with
// max_carveout, prefers the largest shared-memory carveout) the first time
// it is called for that kernel on the current device.  Thread-safe; returns
// a status (Q8D_ECUDA if cudaGetDevice or an attribute call fails).
int configure_kernel(const void* fn, int smem_bytes, bool max_carveout);
// Polls `ev` for at most timeout_ms (<= 0: 10 s); then *dst = *src.
int wait_event_bounded(cudaEvent_t ev, int timeout_ms, const int* src, int* dst);

// ---- shared memory / mbarrier / bulk-copy PTX wrappers --------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity`; returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// L2 policy: data read exactly once (weights, KV) should not evict reused data.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy: data that many CTAs read (a shared operand) stays in L2.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk async copy global -> shared (TMA engine), completion counted on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Pulls [src, src + bytes) into L2 (TMA engine, nothing to wait for).
// src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Orders this thread's earlier generic-proxy global writes before later
// async-proxy (bulk copy) reads of the same addresses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- programmatic dependent launch ---------------------------------------
// Lets the next kernel in the stream start its prologue now.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the kernels this one depends on have completed and their
// writes are visible (returns at once for an ordinary launch).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kernel` on `stream`, as a programmatic dependent of the previous
// work in the stream when `pdl` is set.
template <typename... Args>
int launch_ex(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
              bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e == cudaSuccess ? Q8D_OK : record_cuda(e);
}

// ---- packed f32x2 arithmetic (Blackwell) ---------------------------------
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- Q8_0 decoding helpers ------------------------------------------------
// Signed byte q placed in the mantissa of 2^23: the float 2^23 + (q + 128)
// is exact, so subtracting 2^23 + 128 yields q exactly with one add.  The
// caller flips the sign bit of each byte (xor 0x80) once per 32-bit word.
constexpr uint32_t kMagicHi = 0x4B000000u;  // 2^23
constexpr float kMagicBias = 8388736.0f;   // 2^23 + 128

__device__ __forceinline__ float magic_byte(uint32_t word_flipped, uint32_t sel) {
  return __uint_as_float(__byte_perm(word_flipped, kMagicHi, sel));
}

// Selector nibbles: byte k of `word` into byte 0, bytes 4,5 (zero) and 7
// (0x4B) of kMagicHi into bytes 1..3.
__device__ __forceinline__ constexpr uint32_t magic_sel(int k) { return 0x7540u | (uint32_t)k; }

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

}  // namespace q8d
