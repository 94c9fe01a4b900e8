// Whole decode step captured as one CUDA graph ("IV.4: One command buffer
// per token", "One command buffer": every operation of the step encoded
// once, submitted as one unit, one integer read back).  On GB300 the graph
// holds one memset (the grid barrier counter) and one persistent
// cooperative kernel that runs every phase of the step (q8d_megastep.cu);
// the token id and position live in device memory, and the kernel's last
// phase writes the next token and advances the position, so the same graph
// decodes the next token when launched again.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "q8d_internal.cuh"
#include "q8d_megastep.cuh"

namespace q8d {
namespace {

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

}  // namespace
}  // namespace q8d

using namespace q8d;

struct q8d_step {
  q8d_step_desc desc;
  std::vector<q8d_layer_desc> layers;
  void* ws = nullptr;  // activations, tables and phase table (one allocation)
  float *x, *q, *k, *v, *attn, *gu, *logits, *rope_cos, *rope_sin, *am_val;
  int* am_idx;
  unsigned* bar;  // grid barrier counter, abort flag (both reset per launch), wait limit
  MParams mp;
  int grid = 0;
  int* h_err = nullptr;  // pinned
  cudaEvent_t ev = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int kernel_nodes = 0;
};

namespace q8d {
int step_validate(const q8d_step_desc* d);

// Share (1/1000) of each CTA's rows of a gate|up phase that the producer
// pulls into L2 while the short phases before it run.
constexpr int kGluPrefetchPermille = 250;

// Default number of polls a grid-barrier wait of the step kernel makes
// before the step gives up (each poll is an L2 round trip: about a second).
constexpr unsigned kStepWaitPolls = 1u << 21;

// The step: reset the grid barrier, then the persistent step kernel.
static int enqueue_step(q8d_step* S, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(S->bar, 0, 2 * sizeof(unsigned), st);
  if (e != cudaSuccess) return record_cuda(e);
  return megastep_launch(S->mp, S->desc.head_dim, S->desc.kv_dtype, S->grid, st);
}

// Phase table of the step: embedding; per layer q|k|v (RMSNorm folded in),
// attention partials (bias / QK-norm / RoPE / append folded in), combine,
// o (+ residual), gate|up (RMSNorm folded in; SiLU(gate)*up formed as the
// up rows complete), down (+ residual); lm_head (RMSNorm folded in, argmax
// partials); argmax.
static int build_phases(q8d_step* S, std::vector<MPhase>& ph, int& stage_bytes) {
  const q8d_step_desc& d = S->desc;
  const int qw = d.n_heads * d.head_dim, kvw = d.n_kv_heads * d.head_dim;
  auto mv = [&](int layer, int n, const float* X, int xmode, const float* xw, int acc,
                std::initializer_list<std::pair<const void*, std::pair<float*, int>>> segs) {
    MPhase F{};
    F.kind = kPhMatvec;
    F.layer = layer;
    F.n = n;
    F.X = X;
    F.xmode = xmode;
    F.xw = xw;
    F.accumulate = acc;
    int i = 0, tot = 0;
    for (auto& sg : segs) {
      F.w[i] = static_cast<const uint8_t*>(sg.first);
      F.y[i] = sg.second.first;
      F.vbegin[i] = tot;
      tot += sg.second.second;
      ++i;
    }
    F.nseg = i;
    F.vbegin[i] = tot;
    return F;
  };
  MPhase E{};
  E.kind = kPhEmbed;
  ph.push_back(E);
  for (int li = 0; li < d.n_layers; ++li) {
    const q8d_layer_desc& L = S->layers[li];
    ph.push_back(mv(li, d.hidden, S->x, kXRmsNorm, L.attn_norm, 0,
                    {{L.wq, {S->q, qw}}, {L.wk, {S->k, kvw}}, {L.wv, {S->v, kvw}}}));
    MPhase A{};
    A.kind = kPhAttn;
    A.layer = li;
    ph.push_back(A);
    MPhase Cb{};
    Cb.kind = kPhCombine;
    Cb.layer = li;
    ph.push_back(Cb);
    ph.push_back(mv(li, qw, S->attn, kXPlain, nullptr, 1, {{L.wo, {S->x, d.hidden}}}));
    MPhase GU = mv(li, d.hidden, S->x, kXRmsNorm, L.ffn_norm, 0,
                   {{L.wg, {S->gu, d.ffn}}, {L.wu, {S->gu + d.ffn, d.ffn}}});
    GU.glu = 1;  // writes h = silu(gate) * up over the gate half of gu
    ph.push_back(GU);
    ph.push_back(mv(li, d.ffn, S->gu, kXPlain, nullptr, 1, {{L.wd, {S->x, d.hidden}}}));
  }
  MPhase LM = mv(-1, d.hidden, S->x, kXRmsNorm, d.out_norm, 0, {{d.lm_head, {S->logits, d.vocab}}});
  LM.argmax = 1;
  ph.push_back(LM);
  MPhase AM{};
  AM.kind = kPhArgmax;
  ph.push_back(AM);
  // Stage size: the largest tensor-core tile (8 row slots) when any phase
  // takes the tensor cores, else about a third of the ring; every CUDA-core
  // phase takes the largest tile of whole rows that fits it.
  stage_bytes = 0;
  for (auto& F : ph)
    if (F.kind == kPhMatvec) stage_bytes = std::max(stage_bytes, megastep_plan_tc(F, S->grid));
  const int target = stage_bytes ? stage_bytes : (megastep_ring_bytes() / 3) & ~127;
  for (auto& F : ph) {
    if (F.kind != kPhMatvec || F.tc) continue;
    if (!megastep_plan_matvec(F, S->grid, target)) return Q8D_EUNSUPPORTED;
    const long long sb = ((F.R * F.row_bytes + 32 + 127) / 128) * 128;
    stage_bytes = (int)std::max<long long>(stage_bytes, sb);
  }
  return Q8D_OK;
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
  const int G = d.n_heads / d.n_kv_heads;
  S->grid = sm_count();
  const int nc = std::max(1, S->grid / d.n_kv_heads);  // attention chunks per KV head
  // (the combine's lanes hold at most 5 chunks each; the final argmax's
  // warp at most 8 CTAs a lane; the attention phase gives every KV head at
  // least one of the grid's CTAs)
  if (nc > 160 || S->grid > 256 || d.n_kv_heads > S->grid) {
    delete S;
    return Q8D_EUNSUPPORTED;
  }

  // carve one allocation (256-byte aligned pieces)
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t nphases = 3 + 6ull * d.n_layers;
  const size_t o_x = take(4ull * d.hidden), o_q = take(4ull * qw), o_k = take(4ull * kvw),
               o_v = take(4ull * kvw), o_attn = take(4ull * qw), o_gu = take(8ull * d.ffn),
               o_logits = d.d_logits ? 0 : take(4ull * d.vocab),
               o_cos = take(4ull * d.cap * half), o_sin = take(4ull * d.cap * half),
               o_amv = take(4ull * S->grid), o_ami = take(4ull * S->grid), o_bar = take(16),
               o_wm = take(4ull * d.n_kv_heads * nc * G), o_wl = take(4ull * d.n_kv_heads * nc * G),
               o_wo = take(4ull * d.n_kv_heads * nc * G * d.head_dim),
               o_ph = take(sizeof(MPhase) * nphases), o_ly = take(sizeof(MLayer) * d.n_layers);
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
  S->bar = reinterpret_cast<unsigned*>(base + o_bar);

  auto fail = [&](int code) {
    q8d_step_destroy(S);
    return code;
  };
  std::vector<MPhase> phases;
  int stage_bytes = 0;
  if ((rc = build_phases(S, phases, stage_bytes))) return fail(rc);
  std::vector<MLayer> mlayers(d.n_layers);
  for (int li = 0; li < d.n_layers; ++li) {
    const q8d_layer_desc& L = S->layers[li];
    mlayers[li] = {L.kcache, L.vcache, d.qkv_bias ? L.bq : nullptr, d.qkv_bias ? L.bk : nullptr,
                   d.qkv_bias ? L.bv : nullptr, d.qk_norm ? L.q_norm : nullptr,
                   d.qk_norm ? L.k_norm : nullptr};
  }
  MParams& P = S->mp;
  P = MParams{};
  P.phases = reinterpret_cast<const MPhase*>(base + o_ph);
  P.nphases = (int)phases.size();
  P.layers = reinterpret_cast<const MLayer*>(base + o_ly);
  P.hidden = d.hidden;
  P.vocab = d.vocab;
  P.n_heads = d.n_heads;
  P.n_kv_heads = d.n_kv_heads;
  P.cap = d.cap;
  P.head_dim = d.head_dim;
  P.kv_esize = d.kv_dtype == Q8D_KV_F16 ? 2 : 4;
  P.eps = d.rms_eps;
  P.scale = (float)(1.0 / std::sqrt((double)d.head_dim));
  P.embed = static_cast<const uint8_t*>(d.embed);
  P.d_token = d.d_token;
  P.d_pos = d.d_pos;
  P.d_err = d.d_err;
  P.x = S->x;
  P.q = S->q;
  P.k = S->k;
  P.v = S->v;
  P.attn = S->attn;
  P.logits = S->logits;
  P.am_val = S->am_val;
  P.am_idx = S->am_idx;
  P.rope_cos = S->rope_cos;
  P.rope_sin = S->rope_sin;
  P.ws_m = reinterpret_cast<float*>(base + o_wm);
  P.ws_l = reinterpret_cast<float*>(base + o_wl);
  P.ws_o = reinterpret_cast<float*>(base + o_wo);
  P.nc = nc;
  P.bar = S->bar;
  P.abort = reinterpret_cast<int*>(S->bar + 1);
  P.wait_limit = S->bar + 2;
  P.stage_bytes = stage_bytes;
  P.nstages = std::min(8, megastep_max_stages(stage_bytes));
  P.pf_permille = kGluPrefetchPermille;
  if (P.nstages < 2) return fail(Q8D_EUNSUPPORTED);

  if ((e = cudaMallocHost(&S->h_err, sizeof(int))) != cudaSuccess) return fail(record_cuda(e));
  if ((e = cudaEventCreateWithFlags(&S->ev, cudaEventDisableTiming)) != cudaSuccess)
    return fail(record_cuda(e));
  if ((e = cudaMemcpyAsync(base + o_ph, phases.data(), sizeof(MPhase) * phases.size(),
                           cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return fail(record_cuda(e));
  if ((e = cudaMemcpyAsync(base + o_ly, mlayers.data(), sizeof(MLayer) * mlayers.size(),
                           cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return fail(record_cuda(e));
  const unsigned polls = kStepWaitPolls;
  if ((e = cudaMemcpyAsync(S->bar + 2, &polls, sizeof(polls), cudaMemcpyHostToDevice, st)) !=
      cudaSuccess)
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

int q8d_step_launch_host(q8d_step* S, const int* h_token_pos, int* h_next_token, void* stream) {
  if (!S || !S->exec) return Q8D_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (h_token_pos) {
    if (S->desc.d_pos == S->desc.d_token + 1) {
      e = cudaMemcpyAsync(S->desc.d_token, h_token_pos, 2 * sizeof(int), cudaMemcpyHostToDevice, st);
    } else {
      e = cudaMemcpyAsync(S->desc.d_token, h_token_pos, sizeof(int), cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(S->desc.d_pos, h_token_pos + 1, sizeof(int), cudaMemcpyHostToDevice, st);
    }
    if (e != cudaSuccess) return record_cuda(e);
  }
  if ((e = cudaGraphLaunch(S->exec, st)) != cudaSuccess) return record_cuda(e);
  if (h_next_token &&
      (e = cudaMemcpyAsync(h_next_token, S->desc.d_token, sizeof(int), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess)
    return record_cuda(e);
  return Q8D_OK;
}

int q8d_step_status(q8d_step* S, void* stream, int timeout_ms, int* err) {
  if (!S || !err) return Q8D_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(S->h_err, S->desc.d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return record_cuda(e);
  if ((e = cudaEventRecord(S->ev, st)) != cudaSuccess) return record_cuda(e);
  return wait_event_bounded(S->ev, timeout_ms, S->h_err, err);
}

int q8d_step_set_wait_limit(q8d_step* S, unsigned polls, void* stream) {
  if (!S) return Q8D_EINVAL;
  const unsigned v = polls ? polls : kStepWaitPolls;
  // (a pageable source: the value is staged before the call returns)
  const cudaError_t e = cudaMemcpyAsync(S->bar + 2, &v, sizeof(v), cudaMemcpyHostToDevice,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q8D_OK : record_cuda(e);
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
