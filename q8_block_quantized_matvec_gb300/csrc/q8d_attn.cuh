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
  const int* d_lens;    // [batch] attended lengths (causal windows [0, L))
  const int* d_runs;    // [batch][kMaxRuns][2] (cell, len) run maps, or nullptr
  float scale;
  void* workspace;
  int nc;               // chunk slots per (sequence, KV head) in the workspace
  int nct;              // chunk CTAs per KV head (the grid's x)
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
  // carved from the workspace by attn_launch
  float* ws_o;
  float* ws_m;
  float* ws_l;
};

// Split-K over a ragged batch.  The host fixes the grid (nct chunk CTAs per
// KV head) without knowing the lengths, which live in device memory; every
// CTA (and the combine) derives the same split from them: sequence s gets
// n_s = 1 + floor((nct - batch) * L_s / sum L) chunks (its share of the
// batch's rows), at most one per kMinChunk rows and at most nc (the
// workspace slots), and its rows [0, L_s) go to them in equal parts.  CTA k
// of a KV head takes chunk k - (n_0 + ... + n_{s-1}) of the sequence s whose
// range holds k; CTAs past the last chunk have no work.
constexpr int kMinChunk = 128;
constexpr int kMaxRuns = 4;  // runs per window map ("minfer Metal Backend Design": <= 4 spans)

// A sequence's attended cache rows: the causal window [0, L), or the cells
// of up to kMaxRuns (cell, len) runs in order ("minfer Metal Backend
// Design", "Execution dispatch", window modes).  Window row t is cache row
// cell(t).
struct AttnWindow {
  int cell[kMaxRuns], len[kMaxRuns];
  __device__ __forceinline__ int cell_of(int t) const {
#pragma unroll
    for (int i = 0; i < kMaxRuns; ++i) {
      if (t < len[i]) return cell[i] + t;
      t -= len[i];
    }
    return cell[kMaxRuns - 1];  // (t >= total: not used)
  }
};

// Stores the window of sequence b in shared memory (one thread; readers
// wait for a barrier).  Invalid windows are not stored: their sequences do
// no work.
__device__ __forceinline__ void attn_window_store(const AttnParams& P, int b, AttnWindow* w) {
  if (!P.d_runs) {
    w->cell[0] = 0;
    w->len[0] = P.d_lens[b];
#pragma unroll
    for (int i = 1; i < kMaxRuns; ++i) w->cell[i] = w->len[i] = 0;
  } else {
    const int* r = P.d_runs + (long long)b * 2 * kMaxRuns;
#pragma unroll
    for (int i = 0; i < kMaxRuns; ++i) {
      w->cell[i] = r[2 * i];
      w->len[i] = r[2 * i + 1];
    }
  }
}

// Cache row of window row t of sequence b (a valid window, t inside it),
// read from the run map in global memory.
__device__ __forceinline__ int attn_cell(const AttnParams& P, int b, int t) {
  if (!P.d_runs) return t;
  const int* r = P.d_runs + (long long)b * 2 * kMaxRuns;
#pragma unroll
  for (int i = 0; i < kMaxRuns; ++i) {
    const int len = r[2 * i + 1];
    if (t < len) return r[2 * i] + t;
    t -= len;
  }
  return r[2 * (kMaxRuns - 1)];
}

// Rows attended by sequence b (-1 if its window is invalid): the total of
// attn_window without building the run table.
__device__ __forceinline__ int attn_window_len(const AttnParams& P, int b) {
  if (!P.d_runs) {
    const int L = P.d_lens[b];
    return (L >= 1 && L <= P.cap) ? L : -1;
  }
  const int* r = P.d_runs + (long long)b * 2 * kMaxRuns;
  long long tot = 0;
  bool ok = true;
#pragma unroll
  for (int i = 0; i < kMaxRuns; ++i) {
    const int cell = r[2 * i], len = r[2 * i + 1];
    ok = ok && cell >= 0 && len >= 0 && (long long)cell + len <= P.cap;
    tot += len > 0 ? len : 0;
  }
  return (ok && tot >= 1) ? (int)tot : -1;
}

// Sum of the valid window lengths of the batch.
__device__ __forceinline__ long long attn_total_rows(const AttnParams& P) {
  long long t = 0;
  for (int s = 0; s < P.batch; ++s) {
    const int L = attn_window_len(P, s);
    if (L >= 1) t += L;
  }
  return t;
}

// Chunks of a sequence attending L rows (1 for an invalid window, L < 1).
__device__ __forceinline__ int attn_nchunks(const AttnParams& P, int L, long long total) {
  if (L < 1 || total <= 0) return 1;
  long long n = 1 + (long long)(P.nct - P.batch) * L / total;
  n = n < (L + kMinChunk - 1) / kMinChunk ? n : (L + kMinChunk - 1) / kMinChunk;
  n = n < P.nc ? n : P.nc;
  return n > 1 ? (int)n : 1;
}

// Sequence b, chunk c of n for CTA k of a KV head; false if it has no work.
__device__ __forceinline__ bool attn_chunk_of(const AttnParams& P, int k, int& b, int& c, int& n) {
  const long long total = attn_total_rows(P);
  int first = 0;
  for (int s = 0; s < P.batch; ++s) {
    const int ns = attn_nchunks(P, attn_window_len(P, s), total);
    if (k < first + ns) {
      b = s;
      c = k - first;
      n = ns;
      return true;
    }
    first += ns;
  }
  return false;
}

// Chunk CTAs per KV head (grid.x): about two per SM in all, at least one
// per sequence, at most one per kMinChunk rows of every cache.
int attn_ctas_per_head(int batch, int n_kv_heads, int max_len);
// Workspace chunk slots per (sequence, KV head): up to 4x a sequence's even
// share of the CTAs (at least 8), one per kMinChunk rows of the cache.
int attn_chunks(int batch, int n_kv_heads, int max_len);
int attn_combine_launch(const AttnParams& P, cudaStream_t stream);
int attn_mma_launch(const AttnParams& P, cudaStream_t stream);  // f16 cache, tensor cores
int attn_q8kv_launch(const AttnParams& P, cudaStream_t stream);  // packed Q8_0 cache
size_t attn_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim, int max_len);
int attn_launch(AttnParams P, cudaStream_t stream);
int kv_append_launch(const float* k, const float* v, void* kc, void* vc, int kv_dtype, int kvw,
                     int cap, const int* d_pos, int* d_err, cudaStream_t stream);

}  // namespace q8d
