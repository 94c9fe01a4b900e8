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

constexpr int kMaxRowCtas = 1024;  // upper bound on the lm_head launch's CTAs (argmax partials)

// x = dequantised embedding row of *d_token ("The decoder: kernels and
// helpers": embed_row); also publishes the attended length L = pos + 1.
__global__ void embed_kernel(const uint8_t* __restrict__ embed, int hidden, int vocab,
                             const int* d_token, const int* d_pos, int cap, float* x, int* d_len,
                             int* d_err) {
  griddep_launch_dependents();
  griddep_wait();  // the previous step's argmax wrote the token
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

// cos/sin of pos * theta^(-i/half) for every cached position, computed in
// double and rounded once (the RoPE of "Eight kernels": rope_row).
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

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Final argmax over the lm_head CTAs' partial winners (ties to the lowest
// index; "Eight kernels": argmax_row); writes the next token and advances
// the position for the next launch of the graph.

__global__ void argmax_final_kernel(const float* pv, const int* pi, int np, int* d_token,
                                    int* d_pos) {
  griddep_wait();
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

__global__ void zero_ints(int* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
}

}  // namespace
}  // namespace q8d

using namespace q8d;

struct q8d_step {
  q8d_step_desc desc;
  std::vector<q8d_layer_desc> layers;
  // workspace (one allocation)
  void* ws = nullptr;
  float *x, *q, *k, *v, *attn, *gu, *logits, *rope_cos, *rope_sin, *am_val;
  int *am_idx, *d_len, *tickets;
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

// The step, five kernels per layer, each a programmatic dependent of the
// previous one (its weight stream starts while the previous kernel drains):
//   q|k|v matvec with RMSNorm folded into the activation load
//   attention with bias / QK-norm / RoPE / KV append / combine folded in
//   o matvec accumulating into the residual stream
//   gate|up matvec with RMSNorm folded in
//   down matvec with SiLU(gate)*up folded in, accumulating into the residual
// then the lm_head matvec (final RMSNorm folded in, per-CTA argmax) and the
// final argmax that writes the next token and advances the position.
static int enqueue_step(q8d_step* S, cudaStream_t st) {
  const q8d_step_desc& d = S->desc;
  const int H = d.n_heads, Hk = d.n_kv_heads, D = d.head_dim;
  const int qw = H * D, kvw = Hk * D;
  int rc;
  if ((rc = launch_ex(embed_kernel, dim3((d.hidden + 255) / 256), dim3(256), 0, st, true,
                      static_cast<const uint8_t*>(d.embed), d.hidden, d.vocab,
                      (const int*)d.d_token, (const int*)d.d_pos, d.cap, S->x, S->d_len, d.d_err)))
    return rc;
  for (int li = 0; li < d.n_layers; ++li) {
    const q8d_layer_desc& L = S->layers[li];
    {  // q | k | v projections of RMSNorm(x)
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wq), S->q, qw, 0};
      P.seg[1] = {static_cast<const uint8_t*>(L.wk), S->k, kvw, 0};
      P.seg[2] = {static_cast<const uint8_t*>(L.wv), S->v, kvw, 0};
      P.nseg = 3;
      P.n = d.hidden;
      P.X = S->x;
      P.ldx = d.hidden;
      P.m = 1;
      P.xmode = kXRmsNorm;
      P.xw = L.attn_norm;
      P.eps = d.rms_eps;
      P.pdl = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
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
      A.bq = d.qkv_bias ? L.bq : nullptr;
      A.bk = d.qkv_bias ? L.bk : nullptr;
      A.bv = d.qkv_bias ? L.bv : nullptr;
      A.q_norm = d.qk_norm ? L.q_norm : nullptr;
      A.k_norm = d.qk_norm ? L.k_norm : nullptr;
      A.eps = d.rms_eps;
      A.rope_cos = S->rope_cos;
      A.rope_sin = S->rope_sin;
      A.tickets = S->tickets;
      A.pdl = 1;
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
      P.pdl = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
    {  // gate | up of RMSNorm(x)
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wg), S->gu, d.ffn, 0};
      P.seg[1] = {static_cast<const uint8_t*>(L.wu), S->gu + d.ffn, d.ffn, 0};
      P.nseg = 2;
      P.n = d.hidden;
      P.X = S->x;
      P.ldx = d.hidden;
      P.m = 1;
      P.xmode = kXRmsNorm;
      P.xw = L.ffn_norm;
      P.eps = d.rms_eps;
      P.pdl = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
    {  // x += Wd . (silu(gate) * up)
      RowsParams P{};
      P.seg[0] = {static_cast<const uint8_t*>(L.wd), S->x, d.hidden, 0};
      P.nseg = 1;
      P.n = d.ffn;
      P.X = S->gu;
      P.ldx = d.ffn;
      P.m = 1;
      P.accumulate = 1;
      P.xmode = kXSiluMul;
      P.pdl = 1;
      P.d_err = d.d_err;
      if ((rc = rows_plan_and_launch(P, st))) return rc;
    }
  }
  int np = 0;
  {  // logits = lm_head . RMSNorm(x), with per-CTA argmax partials
    RowsParams P{};
    P.seg[0] = {static_cast<const uint8_t*>(d.lm_head), S->logits, d.vocab, 0};
    P.nseg = 1;
    P.n = d.hidden;
    P.X = S->x;
    P.ldx = d.hidden;
    P.m = 1;
    P.xmode = kXRmsNorm;
    P.xw = d.out_norm;
    P.eps = d.rms_eps;
    P.am_val = S->am_val;
    P.am_idx = S->am_idx;
    P.pdl = 1;
    P.d_err = d.d_err;
    if ((rc = rows_plan_and_launch(P, st, &np))) return rc;
  }
  if (np > kMaxRowCtas) return Q8D_EUNSUPPORTED;
  return launch_ex(argmax_final_kernel, dim3(1), dim3(32), 0, st, true, (const float*)S->am_val,
                   (const int*)S->am_idx, np, d.d_token, d.d_pos);
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
  const size_t o_x = take(4ull * d.hidden), o_q = take(4ull * qw), o_k = take(4ull * kvw),
               o_v = take(4ull * kvw), o_attn = take(4ull * qw), o_gu = take(8ull * d.ffn),
               o_logits = d.d_logits ? 0 : take(4ull * d.vocab),
               o_cos = take(4ull * d.cap * half), o_sin = take(4ull * d.cap * half),
               o_amv = take(4ull * kMaxRowCtas), o_ami = take(4ull * kMaxRowCtas),
               o_len = take(16), o_tk = take(4ull * d.n_kv_heads), o_aws = take(S->attn_ws_bytes);
  cudaError_t e = cudaMalloc(&S->ws, off);
  if (e != cudaSuccess) {
    delete S;
    record_cuda(e);
    return Q8D_ENOMEM;
  }
  uint8_t* base = static_cast<uint8_t*>(S->ws);
  S->x = reinterpret_cast<float*>(base + o_x);
  S->q = reinterpret_cast<float*>(base + o_q);
  S->k = reinterpret_cast<float*>(base + o_k);
  S->v = reinterpret_cast<float*>(base + o_v);
  S->attn = reinterpret_cast<float*>(base + o_attn);
  S->gu = reinterpret_cast<float*>(base + o_gu);
  S->logits = d.d_logits ? d.d_logits : reinterpret_cast<float*>(base + o_logits);
  S->rope_cos = reinterpret_cast<float*>(base + o_cos);
  S->rope_sin = reinterpret_cast<float*>(base + o_sin);
  S->am_val = reinterpret_cast<float*>(base + o_amv);
  S->am_idx = reinterpret_cast<int*>(base + o_ami);
  S->d_len = reinterpret_cast<int*>(base + o_len);
  S->tickets = reinterpret_cast<int*>(base + o_tk);
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
  zero_ints<<<1, 32, 0, st>>>(S->tickets, d.n_kv_heads);  // attention tickets start at zero
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
