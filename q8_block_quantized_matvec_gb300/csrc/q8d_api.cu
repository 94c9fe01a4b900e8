// C-ABI entry points of libq8d: argument validation, then the kernels.
// Every check happens on the host before anything is enqueued; a refused
// call launches nothing and never falls back to another implementation
// ("minfer Metal Backend Design": an unsupported case returns an error and
// never runs the wrong kernel).
#include <chrono>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <thread>
#include <utility>

#include "q8d_attn.cuh"
#include "q8d_internal.cuh"
#include "q8d_rows.cuh"

namespace q8d {

static thread_local int g_last_cuda = 0;

int record_cuda(cudaError_t e) {
  g_last_cuda = (int)e;
  return Q8D_ECUDA;
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? Q8D_OK : record_cuda(e);
}

int configure_kernel(const void* fn, int smem_bytes, bool max_carveout) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return record_cuda(ge);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({fn, dev})) return Q8D_OK;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return record_cuda(e);
  if (max_carveout) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return record_cuda(e);
  }
  done.insert({fn, dev});
  return Q8D_OK;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) return 1;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 1;
  }
  return cached[dev];
}

size_t mma_small_m_workspace(int m, int n);
int mma_small_m_launch(const float* X, int ldx, const uint8_t* w, float* Y, int ldy, int m, int n,
                       int p, void* ws, cudaStream_t stream);

// Polls an event with a wall-clock limit; on completion copies *src to *dst.
int wait_event_bounded(cudaEvent_t ev, int timeout_ms, const int* src, int* dst) {
  const auto limit = std::chrono::milliseconds(timeout_ms > 0 ? timeout_ms : 10000);
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) return record_cuda(e);
    if (std::chrono::steady_clock::now() - t0 > limit) return Q8D_ETIMEOUT;
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  *dst = *src;
  return Q8D_OK;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

static size_t q8_bytes(long long rows, int n) { return (size_t)rows * (size_t)(n / 32) * 34; }

int step_validate(const q8d_step_desc* d) {
  if (!d || !d->layers || !d->embed || !d->out_norm || !d->lm_head || !d->d_token || !d->d_pos ||
      !d->d_err)
    return Q8D_EINVAL;
  if (d->hidden <= 0 || d->n_layers <= 0 || d->n_heads <= 0 || d->n_kv_heads <= 0 ||
      d->head_dim <= 0 || d->ffn <= 0 || d->vocab <= 0 || d->cap <= 0)
    return Q8D_EINVAL;
  if (d->head_dim != 64 && d->head_dim != 128) return Q8D_EUNSUPPORTED;
  if (d->n_heads % d->n_kv_heads) return Q8D_EUNSUPPORTED;
  if (d->n_heads / d->n_kv_heads > 16) return Q8D_EUNSUPPORTED;
  // the step's f16-cache attention prepares the query rows of a KV head's
  // group with the 12 warps beside its 8 pair warps
  if (d->kv_dtype == Q8D_KV_F16 && d->n_heads / d->n_kv_heads > 12) return Q8D_EUNSUPPORTED;
  if (d->hidden % 32 || d->ffn % 32) return Q8D_EUNSUPPORTED;
  if (d->kv_dtype != Q8D_KV_F32 && d->kv_dtype != Q8D_KV_F16) return Q8D_EUNSUPPORTED;
  if (!(d->rms_eps >= 0.f) || !(d->rope_theta > 0.f)) return Q8D_EINVAL;
  // the RMSNorm weights are read as 16-byte vectors, the other f32 vectors
  // element by element
  if (!aligned(d->embed, 16) || !aligned(d->lm_head, 16) || !aligned(d->out_norm, 16))
    return Q8D_EALIGN;
  for (int i = 0; i < d->n_layers; ++i) {
    const q8d_layer_desc& L = d->layers[i];
    if (!L.wq || !L.wk || !L.wv || !L.wo || !L.wg || !L.wu || !L.wd || !L.attn_norm ||
        !L.ffn_norm || !L.kcache || !L.vcache)
      return Q8D_EINVAL;
    if (d->qk_norm && (!L.q_norm || !L.k_norm)) return Q8D_EINVAL;
    if (d->qkv_bias && (!L.bq || !L.bk || !L.bv)) return Q8D_EINVAL;
    const void* w[] = {L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd, L.kcache, L.vcache,
                       L.attn_norm, L.ffn_norm};
    for (const void* p : w)
      if (!aligned(p, 16)) return Q8D_EALIGN;
    const void* v[] = {L.q_norm, L.k_norm, L.bq, L.bk, L.bv};
    for (const void* p : v)
      if (p && !aligned(p, 4)) return Q8D_EALIGN;
  }
  return Q8D_OK;
}

}  // namespace q8d

using namespace q8d;

extern "C" {

int q8d_version(void) { return 100; }

const char* q8d_strerror(int s) {
  switch (s) {
    case Q8D_OK: return "ok";
    case Q8D_EINVAL: return "invalid argument (null pointer, bad size or overlap)";
    case Q8D_EALIGN: return "misaligned pointer or stride";
    case Q8D_EUNSUPPORTED: return "unsupported shape or dtype";
    case Q8D_ERANGE: return "index or length outside its buffer";
    case Q8D_ECUDA: return "CUDA error (see q8d_last_cuda_error)";
    case Q8D_ETIMEOUT: return "bounded wait timed out";
    case Q8D_ENOMEM: return "device allocation failed";
    default: return "unknown status";
  }
}

int q8d_last_cuda_error(void) { return g_last_cuda; }

int q8d_matvec(const float* x, const void* w_q8, float* out, int n, int p, void* stream) {
  if (n < 0 || p < 0) return Q8D_EINVAL;
  if (p == 0) return Q8D_OK;
  if (!out) return Q8D_EINVAL;
  if (n % 32) return Q8D_EUNSUPPORTED;
  if (n > 0 && (!x || !w_q8)) return Q8D_EINVAL;
  if (!aligned(out, 4)) return Q8D_EALIGN;
  if (n > 0) {
    if (!aligned(w_q8, 16) || !aligned(x, 16)) return Q8D_EALIGN;
    if (overlap(out, 4ull * p, x, 4ull * n) || overlap(out, 4ull * p, w_q8, q8_bytes(p, n)))
      return Q8D_EINVAL;
  }
  RowsParams P{};
  P.seg[0] = {static_cast<const uint8_t*>(w_q8), out, p, 0};
  P.nseg = 1;
  P.n = n;
  P.X = x;
  P.ldx = n;
  P.ldy = p;
  P.m = 1;
  return rows_plan_and_launch(P, static_cast<cudaStream_t>(stream));
}

namespace {
// Argument checks shared by both small-M entry points (Q8D_OK: go on).
int small_m_check(const float* X, int ldx, const void* w_q8, const float* Y, int ldy, int m, int n,
                  int p) {
  if (m < 0 || n < 0 || p < 0) return Q8D_EINVAL;
  if (m > 256) return Q8D_EUNSUPPORTED;
  if (m == 0 || p == 0) return Q8D_OK;
  if (!Y || ldy < p) return Q8D_EINVAL;
  if (n % 32) return Q8D_EUNSUPPORTED;
  if (n > 0 && (!X || !w_q8 || ldx < n)) return Q8D_EINVAL;
  if (!aligned(Y, 4)) return Q8D_EALIGN;
  if (n > 0) {
    if (!aligned(w_q8, 16) || !aligned(X, 16) || (ldx % 4)) return Q8D_EALIGN;
    const size_t ybytes = 4ull * ((size_t)(m - 1) * ldy + p);
    if (overlap(Y, ybytes, X, 4ull * ((size_t)(m - 1) * ldx + n)) ||
        overlap(Y, ybytes, w_q8, q8_bytes(p, n)))
      return Q8D_EINVAL;
  }
  return Q8D_OK;
}

int small_m_cuda_cores(const float* X, int ldx, const void* w_q8, float* Y, int ldy, int m, int n,
                       int p, cudaStream_t st) {
  RowsParams P{};
  P.seg[0] = {static_cast<const uint8_t*>(w_q8), Y, p, 0};
  P.nseg = 1;
  P.n = n;
  P.X = X;
  P.ldx = ldx;
  P.ldy = ldy;
  P.m = m;
  return rows_plan_and_launch(P, st);
}
}  // namespace

size_t q8d_matmul_small_m_workspace_bytes(int m, int n) {
  if (m < 9 || m > 256 || n <= 0 || n % 32) return 0;
  return mma_small_m_workspace(m, n);
}

int q8d_matmul_small_m_ws(const float* X, int ldx, const void* w_q8, float* Y, int ldy, int m,
                          int n, int p, void* workspace, size_t workspace_bytes, void* stream) {
  const int crc = small_m_check(X, ldx, w_q8, Y, ldy, m, n, p);
  if (crc || m == 0 || p == 0) return crc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t need = q8d_matmul_small_m_workspace_bytes(m, n);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return Q8D_EINVAL;
    if (!aligned(workspace, 16)) return Q8D_EALIGN;
    const size_t ybytes = 4ull * ((size_t)(m - 1) * ldy + p);
    if (overlap(workspace, need, Y, ybytes) ||
        overlap(workspace, need, X, 4ull * ((size_t)(m - 1) * ldx + n)) ||
        overlap(workspace, need, w_q8, q8_bytes(p, n)))
      return Q8D_EINVAL;
    const int rc =
        mma_small_m_launch(X, ldx, static_cast<const uint8_t*>(w_q8), Y, ldy, m, n, p, workspace, st);
    if (rc != Q8D_EUNSUPPORTED) return rc;
  }
  return small_m_cuda_cores(X, ldx, w_q8, Y, ldy, m, n, p, st);
}

int q8d_matmul_small_m(const float* X, int ldx, const void* w_q8, float* Y, int ldy, int m, int n,
                       int p, void* stream) {
  const int crc = small_m_check(X, ldx, w_q8, Y, ldy, m, n, p);
  if (crc || m == 0 || p == 0) return crc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t need = q8d_matmul_small_m_workspace_bytes(m, n);
  if (need == 0) return small_m_cuda_cores(X, ldx, w_q8, Y, ldy, m, n, p, st);
  // the activation image in stream-ordered memory, freed behind the kernels
  void* ws = nullptr;
  const cudaError_t e = cudaMallocAsync(&ws, need, st);
  if (e != cudaSuccess) return record_cuda(e);
  const int rc = q8d_matmul_small_m_ws(X, ldx, w_q8, Y, ldy, m, n, p, ws, need, stream);
  const cudaError_t f = cudaFreeAsync(ws, st);
  if (rc) return rc;
  return f == cudaSuccess ? Q8D_OK : record_cuda(f);
}

int q8d_kv_append(const float* k, const float* v, void* kcache, void* vcache, int kv_dtype,
                  int kv_width, int cap, const int* d_pos, int* d_err, void* stream) {
  if (!k || !v || !kcache || !vcache || !d_pos || kv_width <= 0 || cap <= 0) return Q8D_EINVAL;
  if (kv_dtype != Q8D_KV_F32 && kv_dtype != Q8D_KV_F16 && kv_dtype != Q8D_KV_Q8_0)
    return Q8D_EUNSUPPORTED;
  if (kv_dtype == Q8D_KV_Q8_0 && kv_width % 32) return Q8D_EUNSUPPORTED;
  // (a packed cache's blocks are written with 16-bit scale stores)
  const size_t es = kv_dtype == Q8D_KV_F32 ? 4 : (kv_dtype == Q8D_KV_F16 ? 2 : 16);
  if (!aligned(kcache, es) || !aligned(vcache, es) || !aligned(k, 4) || !aligned(v, 4))
    return Q8D_EALIGN;
  const size_t cb = kv_dtype == Q8D_KV_Q8_0 ? q8_bytes(cap, kv_width) : es * (size_t)kv_width * cap;
  if (overlap(kcache, cb, vcache, cb)) return Q8D_EINVAL;
  return kv_append_launch(k, v, kcache, vcache, kv_dtype, kv_width, cap, d_pos, d_err,
                          static_cast<cudaStream_t>(stream));
}

size_t q8d_gqa_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim, int max_len) {
  if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_len <= 0) return 0;
  return attn_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, max_len);
}

}  // extern "C"

namespace q8d {
// Shared checks and launch of the causal (d_lens) and windowed (d_runs)
// decode attention; shared_cache: sequences may share one cache (stride 0).
static int attn_entry(const float* q, const float* k_new, const float* v_new, void* kcache,
                      void* vcache, int kv_dtype, float* out, int batch, int n_heads,
                      int n_kv_heads, int head_dim, int cap, long long cache_batch_stride,
                      const int* d_lens, const int* d_runs, float scale, void* workspace,
                      size_t ws_bytes, int* d_err, cudaStream_t stream) {
  if (!q || !kcache || !vcache || !out || !(d_lens || d_runs) || !workspace) return Q8D_EINVAL;
  if ((k_new == nullptr) != (v_new == nullptr)) return Q8D_EINVAL;
  if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || cap <= 0) return Q8D_EINVAL;
  if (head_dim != 64 && head_dim != 128) return Q8D_EUNSUPPORTED;
  if (n_heads % n_kv_heads || n_heads / n_kv_heads > 16) return Q8D_EUNSUPPORTED;
  if (kv_dtype != Q8D_KV_F32 && kv_dtype != Q8D_KV_F16 && kv_dtype != Q8D_KV_Q8_0)
    return Q8D_EUNSUPPORTED;
  if (!std::isfinite(scale)) return Q8D_EINVAL;
  const long long kvw = (long long)n_kv_heads * head_dim;
  if (cache_batch_stride < 0) return Q8D_EINVAL;
  // sequences own disjoint caches, or (run maps only) share one cache
  if (batch > 1 && cache_batch_stride < kvw * cap && !(d_runs && cache_batch_stride == 0))
    return Q8D_EINVAL;
  // sequence starts 16-byte aligned: for a packed cache the stride (in
  // elements) is a whole number of blocks, 34 bytes per 32 elements
  const long long stride_bytes =
      kv_dtype == Q8D_KV_Q8_0
          ? (cache_batch_stride % 32 ? 1 : cache_batch_stride / 32 * 34)
          : cache_batch_stride * (kv_dtype == Q8D_KV_F16 ? 2 : 4);
  if (!aligned(kcache, 16) || !aligned(vcache, 16) || (stride_bytes % 16)) return Q8D_EALIGN;
  if (!aligned(q, 4) || !aligned(out, 4) || !aligned(workspace, 16)) return Q8D_EALIGN;
  if (d_runs && !aligned(d_runs, 4)) return Q8D_EALIGN;
  if (ws_bytes < attn_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, cap))
    return Q8D_ERANGE;
  AttnParams A{};
  A.q = q;
  A.k_new = k_new;
  A.v_new = v_new;
  A.kcache = kcache;
  A.vcache = vcache;
  A.kv_dtype = kv_dtype;
  A.out = out;
  A.batch = batch;
  A.n_heads = n_heads;
  A.n_kv_heads = n_kv_heads;
  A.head_dim = head_dim;
  A.cap = cap;
  A.batch_stride = cache_batch_stride;
  A.d_lens = d_lens;
  A.d_runs = d_runs;
  A.scale = scale;
  A.workspace = workspace;
  A.nc = attn_chunks(batch, n_kv_heads, cap);
  A.nct = attn_ctas_per_head(batch, n_kv_heads, cap);
  A.d_err = d_err;
  return attn_launch(A, stream);
}
}  // namespace q8d

extern "C" {

int q8d_gqa_decode_attn(const float* q, const float* k_new, const float* v_new, void* kcache,
                        void* vcache, int kv_dtype, float* out, int batch, int n_heads,
                        int n_kv_heads, int head_dim, int cap, long long cache_batch_stride,
                        const int* d_lens, float scale, void* workspace, size_t ws_bytes,
                        int* d_err, void* stream) {
  if (!d_lens) return Q8D_EINVAL;
  return attn_entry(q, k_new, v_new, kcache, vcache, kv_dtype, out, batch, n_heads, n_kv_heads,
                    head_dim, cap, cache_batch_stride, d_lens, nullptr, scale, workspace,
                    ws_bytes, d_err, static_cast<cudaStream_t>(stream));
}

int q8d_gqa_decode_attn_window(const float* q, const float* k_new, const float* v_new,
                               void* kcache, void* vcache, int kv_dtype, float* out, int batch,
                               int n_heads, int n_kv_heads, int head_dim, int cap,
                               long long cache_batch_stride, const int* d_runs, float scale,
                               void* workspace, size_t ws_bytes, int* d_err, void* stream) {
  if (!d_runs) return Q8D_EINVAL;
  return attn_entry(q, k_new, v_new, kcache, vcache, kv_dtype, out, batch, n_heads, n_kv_heads,
                    head_dim, cap, cache_batch_stride, nullptr, d_runs, scale, workspace,
                    ws_bytes, d_err, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
