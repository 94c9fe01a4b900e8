// Whole decode step captured as one CUDA graph ("IV.4: One command buffer
// per token", "One command buffer": every operation of the step encoded
// once, submitted as one unit, one integer read back).  On GB300 the
// analogue of the pages' single command buffer is a CUDA graph: the host
// launches it with one call, the token id and position live in device
// memory, and the argmax kernel writes the next token and advances the
// position so the same graph decodes the next token when launched again.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "q8d_attn.cuh"
#include "q8d_internal.cuh"
#include "q8d_rows.cuh"

namespace q8d {
namespace {

constexpr int kArgmaxBlocks = 148;
constexpr int kArgmaxThreads = 512;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < nw; ++w) s += red[w];  // same order in every thread
  return s;
}

// x = dequantised embedding row of *d_token ("The decoder: kernels and
// helpers": embed_row); also publishes the attended length L = pos + 1.
__global__ void embed_kernel(const uint8_t* __restrict__ embed, int hidden, int vocab,
                             const int* d_token, const int* d_pos, int cap, float* x, int* d_len,
                             int* d_err) {
  const int tok = *d_token;
  const bool bad = tok < 0 || tok >= vocab;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (bad && d_err) atomicOr(d_err, Q8D_DERR_TOKEN_RANGE);
    const int pos = *d_pos;
    *d_len = pos + 1;  // checked against cap by the append/attention kernels
    (void)cap;
  }
  const long long rb = (long long)(hidden / kQBlock) * kQBlockBytes;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < hidden; i += gridDim.x * blockDim.x) {
    if (bad) {
      x[i] = __int_as_float(0x7fc00000);
      continue;
    }
    const uint8_t* blk = embed + (long long)tok * rb + (long long)(i / kQBlock) * kQBlockBytes;
    const float sc = f16_bits_to_f32((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
    x[i] = sc * (float)(int8_t)blk[2 + (i % kQBlock)];
  }
}

// out = x / sqrt(mean(x^2) + eps) * w   (one CTA; "Eight kernels": rms_norm_row)
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ w,
                               float* __restrict__ out, int dim, float eps) {
  __shared__ float red[32];
  float ss = 0.f;
  for (int i = threadIdx.x; i < dim; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)dim + eps);
  for (int i = threadIdx.x; i < dim; i += blockDim.x) out[i] = x[i] * inv * w[i];
}

// Per head: bias add, optional per-head RMSNorm (q and k), RoPE (q and k).
// Blocks [0, H) are query heads, [H, H+Hk) key heads, [H+Hk, H+2Hk) value
// heads (bias only).  RoPE pairs (i, i + D/2) rotate by pos * theta^(-i/(D/2))
// using a cos/sin table built once in double precision.
__global__ void qkv_post_kernel(float* q, float* k, float* v, const float* bq, const float* bk,
                                const float* bv, const float* q_norm, const float* k_norm,
                                const float* rope_cos, const float* rope_sin, const int* d_pos,
                                int cap, int H, int Hk, int D, int qkv_bias, int qk_norm,
                                float eps) {
  __shared__ float red[32];
  __shared__ float row[256];
  const int blk = blockIdx.x, j = threadIdx.x;
  float* base;
  const float* bias;
  const float* nw = nullptr;
  bool rope = true;
  if (blk < H) {
    base = q + (long long)blk * D;
    bias = bq ? bq + (long long)blk * D : nullptr;
    nw = qk_norm ? q_norm : nullptr;
  } else if (blk < H + Hk) {
    base = k + (long long)(blk - H) * D;
    bias = bk ? bk + (long long)(blk - H) * D : nullptr;
    nw = qk_norm ? k_norm : nullptr;
  } else {
    base = v + (long long)(blk - H - Hk) * D;
    bias = bv ? bv + (long long)(blk - H - Hk) * D : nullptr;
    rope = false;
  }
  float val = base[j];
  if (qkv_bias && bias) val += bias[j];
  if (nw) {
    const float ss = block_sum(val * val, red);
    const float inv = 1.0f / sqrtf(ss / (float)D + eps);
    val = val * inv * nw[j];
  }
  if (!rope) {
    base[j] = val;
    return;
  }
  row[j] = val;
  __syncthreads();
  int pos = *d_pos;
  pos = pos < 0 ? 0 : (pos >= cap ? cap - 1 : pos);  // out-of-range is flagged by the append
  const int half = D / 2;
  const int i = j < half ? j : j - half;
  const float c = rope_cos[(long long)pos * half + i];
  const float s = rope_sin[(long long)pos * half + i];
  const float a = row[i], b = row[i + half];
  base[j] = (j < half) ? (a * c - b * s) : (a * s + b * c);
}

__global__ void rope_table_kernel(float* cosv, float* sinv, int cap, int half, double theta) {
  const long long n = (long long)cap * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e % half);
    const double freq = 1.0 / pow(theta, (double)i / (double)half);
    double s, c;
    sincos((double)p * freq, &s, &c);
    cosv[e] = (float)c;
    sinv[e] = (float)s;
  }
}

// h = silu(g) * u with gu = [g | u]  ("Eight kernels": silu_hadamard)
__global__ void silu_mul_kernel(const float* __restrict__ gu, float* __restrict__ h, int F) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < F; i += gridDim.x * blockDim.x) {
    const float g = gu[i];
    h[i] = g / (1.0f + expf(-g)) * gu[F + i];
  }
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Argmax, ties to the lowest index, NaN never wins ("Eight kernels":
// argmax_row), in two deterministic passes.
__global__ void argmax_partial_kernel(const float* __restrict__ x, int n, float* pv, int* pi) {
  __shared__ float sv[32];
  __shared__ int si[32];
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float v = x[i];
    if (!isnan(v) && better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (better(sv[w], si[w], bv, bi)) {
        bv = sv[w];
        bi = si[w];
      }
    pv[blockIdx.x] = bv;
    pi[blockIdx.x] = bi;
  }
}

__global__ void argmax_final_kernel(const float* pv, const int* pi, int np, int* d_token,
                                    int* d_pos) {
  if (threadIdx.x != 0) return;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int b = 0; b < np; ++b)
    if (better(pv[b], pi[b], bv, bi)) {
      bv = pv[b];
      bi = pi[b];
    }
  *d_token = bi;
  *d_pos = *d_pos + 1;
}

}  // namespace
}  // namespace q8d

using namespace q8d;

struct q8d_step {
  q8d_step_desc desc;
  std::vector<q8d_layer_desc> layers;
  // workspace (one allocation)
  void* ws = nullptr;
  float *x, *xn, *q, *k, *v, *attn, *gu, *h, *logits, *rope_cos, *rope_sin, *am_val;
  int *am_idx, *d_len;
  void* attn_ws;
  size_t attn_ws_bytes;
  int attn_nc;
  int* h_err = nullptr;  // pinned
  cudaEvent_t ev = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int kernel_nodes = 0;
};

namespace q8d {
int step_validate(const q8d_step_desc* d);

static int enqueue_step(q8d_step* S, cudaStream_t st) {
  const q8d_step_desc& d = S->desc;
  const int H = d.n_heads, Hk = d.n_kv_heads, D = d.head_dim;
  const int qw = H * D, kvw = Hk * D;
  int rc;
  embed_kernel<<<(d.hidden + 255) / 256, 256, 0, st>>>(
      static_cast<const uint8_t*>(d.embed), d.hidden, d.vocab, d.d_token, d.d_pos, d.cap, S->x,
      S->d_len, d.d_err);
  if ((rc = check_launch())) return rc;
  for (int li = 0; li < d.n_layers; ++li) {
    const q8d_layer_desc& L = S->layers[li];
    rmsnorm_kernel<<<1, 1024, 0, st>>>(S->x, L.attn_norm, S->xn, d.hidden, d.rms_eps);
    if ((rc = check_launch())) return rc;
    {  // q | k | v projections, one launch
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wq), S->q, qw, 0};
      P.seg[1] = {static_cast<const uint8_t*>(L.wk), S->k, kvw, 0};
      P.seg[2] = {static_cast<const uint8_t*>(L.wv), S->v, kvw, 0};
      P.nseg = 3;
      P.n = d.hidden;
      P.X = S->xn;
      P.ldx = d.hidden;
      P.ldy = 0;
      P.m = 1;
      P.accumulate = 0;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
    qkv_post_kernel<<<H + 2 * Hk, D, 0, st>>>(S->q, S->k, S->v, L.bq, L.bk, L.bv, L.q_norm,
                                              L.k_norm, S->rope_cos, S->rope_sin, d.d_pos, d.cap,
                                              H, Hk, D, d.qkv_bias, d.qk_norm, d.rms_eps);
    if ((rc = check_launch())) return rc;
    {
      AttnParams A{};
      A.q = S->q;
      A.k_new = S->k;
      A.v_new = S->v;
      A.kcache = L.kcache;
      A.vcache = L.vcache;
      A.kv_dtype = d.kv_dtype;
      A.out = S->attn;
      A.batch = 1;
      A.n_heads = H;
      A.n_kv_heads = Hk;
      A.head_dim = D;
      A.cap = d.cap;
      A.batch_stride = 0;
      A.d_lens = S->d_len;
      A.scale = (float)(1.0 / std::sqrt((double)D));
      A.workspace = S->attn_ws;
      A.nc = S->attn_nc;
      A.d_err = d.d_err;
      if ((rc = attn_launch(A, st))) return rc;
    }
    {  // x += Wo . attn
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wo), S->x, d.hidden, 0};
      P.nseg = 1;
      P.n = qw;
      P.X = S->attn;
      P.ldx = qw;
      P.m = 1;
      P.accumulate = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
    rmsnorm_kernel<<<1, 1024, 0, st>>>(S->x, L.ffn_norm, S->xn, d.hidden, d.rms_eps);
    if ((rc = check_launch())) return rc;
    {  // gate | up
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wg), S->gu, d.ffn, 0};
      P.seg[1] = {static_cast<const uint8_t*>(L.wu), S->gu + d.ffn, d.ffn, 0};
      P.nseg = 2;
      P.n = d.hidden;
      P.X = S->xn;
      P.ldx = d.hidden;
      P.m = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
    silu_mul_kernel<<<(d.ffn + 255) / 256, 256, 0, st>>>(S->gu, S->h, d.ffn);
    if ((rc = check_launch())) return rc;
    {  // x += Wd . h
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wd), S->x, d.hidden, 0};
      P.nseg = 1;
      P.n = d.ffn;
      P.X = S->h;
      P.ldx = d.ffn;
      P.m = 1;
      P.accumulate = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
  }
  rmsnorm_kernel<<<1, 1024, 0, st>>>(S->x, d.out_norm, S->xn, d.hidden, d.rms_eps);
  if ((rc = check_launch())) return rc;
  {
    RowsParams P{};
    P.seg[0] = {static_cast<const uint8_t*>(d.lm_head), S->logits, d.vocab, 0};
    P.nseg = 1;
    P.n = d.hidden;
    P.X = S->xn;
    P.ldx = d.hidden;
    P.m = 1;
    P.d_err = d.d_err;
    if ((rc = rows_plan_and_launch(P, st))) return rc;
  }
  argmax_partial_kernel<<<kArgmaxBlocks, kArgmaxThreads, 0, st>>>(S->logits, d.vocab, S->am_val,
                                                                  S->am_idx);
  if ((rc = check_launch())) return rc;
  argmax_final_kernel<<<1, 32, 0, st>>>(S->am_val, S->am_idx, kArgmaxBlocks, d.d_token, d.d_pos);
  return check_launch();
}

}  // namespace q8d

extern "C" {

int q8d_step_create(const q8d_step_desc* desc, void* stream, q8d_step** out) {
  if (!out) return Q8D_EINVAL;
  *out = nullptr;
  int rc = step_validate(desc);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  q8d_step* S = new (std::nothrow) q8d_step();
  if (!S) return Q8D_ENOMEM;
  S->desc = *desc;
  S->layers.assign(desc->layers, desc->layers + desc->n_layers);
  const q8d_step_desc& d = S->desc;
  const int qw = d.n_heads * d.head_dim, kvw = d.n_kv_heads * d.head_dim, half = d.head_dim / 2;
  S->attn_nc = attn_chunks(1, d.n_kv_heads, d.cap);
  S->attn_ws_bytes = attn_workspace_bytes(1, d.n_heads, d.n_kv_heads, d.head_dim, d.cap);

  // carve one allocation (256-byte aligned pieces)
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t o_x = take(4ull * d.hidden), o_xn = take(4ull * d.hidden), o_q = take(4ull * qw),
               o_k = take(4ull * kvw), o_v = take(4ull * kvw), o_attn = take(4ull * qw),
               o_gu = take(8ull * d.ffn), o_h = take(4ull * d.ffn),
               o_logits = d.d_logits ? 0 : take(4ull * d.vocab),
               o_cos = take(4ull * d.cap * half), o_sin = take(4ull * d.cap * half),
               o_amv = take(4ull * kArgmaxBlocks), o_ami = take(4ull * kArgmaxBlocks),
               o_len = take(16), o_aws = take(S->attn_ws_bytes);
  cudaError_t e = cudaMalloc(&S->ws, off);
  if (e != cudaSuccess) {
    delete S;
    record_cuda(e);
    return Q8D_ENOMEM;
  }
  uint8_t* base = static_cast<uint8_t*>(S->ws);
  S->x = reinterpret_cast<float*>(base + o_x);
  S->xn = reinterpret_cast<float*>(base + o_xn);
  S->q = reinterpret_cast<float*>(base + o_q);
  S->k = reinterpret_cast<float*>(base + o_k);
  S->v = reinterpret_cast<float*>(base + o_v);
  S->attn = reinterpret_cast<float*>(base + o_attn);
  S->gu = reinterpret_cast<float*>(base + o_gu);
  S->h = reinterpret_cast<float*>(base + o_h);
  S->logits = d.d_logits ? d.d_logits : reinterpret_cast<float*>(base + o_logits);
  S->rope_cos = reinterpret_cast<float*>(base + o_cos);
  S->rope_sin = reinterpret_cast<float*>(base + o_sin);
  S->am_val = reinterpret_cast<float*>(base + o_amv);
  S->am_idx = reinterpret_cast<int*>(base + o_ami);
  S->d_len = reinterpret_cast<int*>(base + o_len);
  S->attn_ws = base + o_aws;

  auto fail = [&](int code) {
    q8d_step_destroy(S);
    return code;
  };
  if ((e = cudaMallocHost(&S->h_err, sizeof(int))) != cudaSuccess) return fail(record_cuda(e));
  if ((e = cudaEventCreateWithFlags(&S->ev, cudaEventDisableTiming)) != cudaSuccess)
    return fail(record_cuda(e));

  rope_table_kernel<<<256, 256, 0, st>>>(S->rope_cos, S->rope_sin, d.cap, half,
                                         (double)d.rope_theta);
  if ((rc = check_launch())) return fail(rc);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(record_cuda(e));

  cudaStream_t cs;
  if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess)
    return fail(record_cuda(e));
  if ((e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return fail(record_cuda(e));
  }
  rc = enqueue_step(S, cs);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (rc) {
    if (g) cudaGraphDestroy(g);
    return fail(rc);
  }
  if (e != cudaSuccess) return fail(record_cuda(e));
  S->graph = g;
  if ((e = cudaGraphInstantiate(&S->exec, g, 0)) != cudaSuccess) return fail(record_cuda(e));
  size_t nn = 0;
  cudaGraphGetNodes(g, nullptr, &nn);
  std::vector<cudaGraphNode_t> nodes(nn);
  cudaGraphGetNodes(g, nodes.data(), &nn);
  int kn = 0;
  for (auto n : nodes) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(n, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kn;
  }
  S->kernel_nodes = kn;
  *out = S;
  return Q8D_OK;
}

int q8d_step_launch(q8d_step* S, void* stream) {
  if (!S || !S->exec) return Q8D_EINVAL;
  cudaError_t e = cudaGraphLaunch(S->exec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q8D_OK : record_cuda(e);
}

int q8d_step_status(q8d_step* S, void* stream, int timeout_ms, int* err) {
  if (!S || !err) return Q8D_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(S->h_err, S->desc.d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return record_cuda(e);
  if ((e = cudaEventRecord(S->ev, st)) != cudaSuccess) return record_cuda(e);
  return wait_event_bounded(S->ev, timeout_ms, S->h_err, err);
}

int q8d_step_kernel_count(const q8d_step* S) { return S ? S->kernel_nodes : 0; }

float* q8d_step_logits(q8d_step* S) { return S ? S->logits : nullptr; }

void q8d_step_destroy(q8d_step* S) {
  if (!S) return;
  if (S->exec) cudaGraphExecDestroy(S->exec);
  if (S->graph) cudaGraphDestroy(S->graph);
  if (S->ev) cudaEventDestroy(S->ev);
  if (S->h_err) cudaFreeHost(S->h_err);
  if (S->ws) cudaFree(S->ws);
  delete S;
}

}  // extern "C"
