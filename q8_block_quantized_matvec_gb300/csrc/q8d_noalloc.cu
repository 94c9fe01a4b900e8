// q8d_gqa_decode_attn_noalloc: the split-K decode attention with its
// scratch in a fixed device array owned by this library, for callers that
// cannot allocate device memory themselves.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// libq8d holds it (kNoAllocScratchBytes) until the process exits.  Host code
// must not pass the symbol itself to a kernel (in host code it names a host
// stand-in); the device address is obtained once per device with
// cudaGetSymbolAddress, with that device current, and cached.
#include <mutex>

#include "q8d_attn.cuh"
#include "q8d_internal.cuh"

namespace q8d {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_attn_scratch on the current device (set up on first use).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return Q8D_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return record_cuda(e);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return Q8D_OK;
}

}  // namespace
}  // namespace q8d

using namespace q8d;

extern "C" {

size_t q8d_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int q8d_gqa_decode_attn_noalloc(const float* q, const float* k_new, const float* v_new,
                                void* kcache, void* vcache, int kv_dtype, float* out, int batch,
                                int n_heads, int n_kv_heads, int head_dim, int cap,
                                long long cache_batch_stride, const int* d_lens, float scale,
                                int* d_err, void* stream) {
  if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || cap <= 0)
    return Q8D_EINVAL;
  const size_t need = attn_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, cap);
  if (need > kNoAllocScratchBytes) return Q8D_ERANGE;
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc) return rc;
  return q8d_gqa_decode_attn(q, k_new, v_new, kcache, vcache, kv_dtype, out, batch, n_heads,
                             n_kv_heads, head_dim, cap, cache_batch_stride, d_lens, scale, ws,
                             kNoAllocScratchBytes, d_err, stream);
}

}  // extern "C"
