// Parameters of the KV-append and split-K decode-attention kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace q8d {

struct AttnParams {
  const float* q;       // [batch][H*D]
  const float* k_new;   // [batch][Hk*D] or nullptr
  const float* v_new;
  void* kcache;         // sequence b at element b*batch_stride, rows of Hk*D
  void* vcache;
  int kv_dtype;
  float* out;           // [batch][H*D]
  int batch, n_heads, n_kv_heads, head_dim, cap;
  long long batch_stride;
  const int* d_lens;    // [batch]
  float scale;
  void* workspace;
  int nc;               // context chunks per (sequence, KV head)
  int* d_err;
  // Decode-step prologue fused into the f16 kernel (all null / 0 for the
  // plain C-ABI call): q/k/v biases, per-head q/k RMSNorm gains, RoPE table
  // [cap][head_dim/2] at position L-1, applied to q and to the appended row.
  const float* bq;
  const float* bk;
  const float* bv;
  const float* q_norm;
  const float* k_norm;
  float eps;
  const float* rope_cos;
  const float* rope_sin;
  // Zero-initialised tickets [batch * n_kv_heads]: when set, the last chunk
  // CTA of each (sequence, KV head) merges the partials itself (and resets
  // its ticket); when null a separate combine kernel runs.
  int* tickets;
  int pdl;              // launched as a programmatic dependent
  // carved from the workspace by attn_launch
  float* ws_o;
  float* ws_m;
  float* ws_l;
};

// Context rows per chunk for attended length L with nc chunk slots: at least
// kMinChunk rows so the partials stay small next to the K/V they summarise.
constexpr int kMinChunk = 128;
__host__ __device__ __forceinline__ int chunk_rows(int L, int nc) {
  const int c = (L + nc - 1) / nc;
  return c > kMinChunk ? c : kMinChunk;
}

int attn_chunks(int batch, int n_kv_heads, int max_len);
int attn_combine_launch(const AttnParams& P, cudaStream_t stream);
int attn_mma_launch(const AttnParams& P, cudaStream_t stream);  // f16 cache, tensor cores
size_t attn_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim, int max_len);
int attn_launch(AttnParams P, cudaStream_t stream);
int kv_append_launch(const float* k, const float* v, void* kc, void* vc, int kv_dtype, int kvw,
                     int cap, const int* d_pos, int* d_err, cudaStream_t stream);

}  // namespace q8d
