// The decode step as one persistent kernel: phase table and parameters.
//
// "IV.4: One command buffer per token" encodes every operation of a decode
// step once and submits them as one unit.  On GB300 the step is one
// cooperative kernel with one CTA per SM that walks a table of phases
// (embedding, per layer q|k|v, attention, combine, o, gate|up, down, then
// lm_head and the argmax), with a grid-wide barrier between phases.  A
// producer warp per CTA streams every weight tile of the CTA's rows of all
// matvec phases through a shared-memory ring in table order, so the weight
// stream does not stop at phase boundaries.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q8d {

enum MPhaseKind { kPhEmbed = 0, kPhMatvec = 1, kPhAttn = 2, kPhCombine = 3, kPhArgmax = 4 };

// Activations of a matvec phase: as stored, or RMSNorm-ed while staged
// (x * (1/sqrt(mean(x^2) + eps)) * xw).
enum MXMode { kXPlain = 0, kXRmsNorm = 1 };

constexpr int kMsWarps = 20;                  // consumer warps per CTA
constexpr int kMsThreads = (kMsWarps + 1) * 32;  // + the producer warp
constexpr int kMsRegion = 44 * 1024;           // shared region: window partials / attention

// One phase.  Matvec phases hold up to three matrices that share their
// activations (rows concatenated: q|k|v, gate|up).
struct alignas(16) MPhase {  // (whole 16-byte chunks: copied by cp.async)
  int kind;
  int layer;
  // matvec
  int nseg;
  int n, bpr, NS, RG, R, win, paired, xmode, accumulate, argmax;
  int glu;  // gate|up: each CTA owns the same rows of both matrices and
            // writes silu(gate) * up over the gate rows
  int tc;   // block dot products on the tensor cores: tiles of T sets of 8
            // whole rows, SR bytes apart; a set is 8 >> gsh groups of
            // 1 << gsh consecutive rows, each group 16 bytes after the
            // previous one's end; win = tiles per window
  int SR, gsh, T;
  int total_rows, rows_per_cta;
  int vbegin[4];  // first virtual row of each matrix; vbegin[nseg] = total_rows
  long long row_bytes;
  const uint8_t* w[3];
  float* y[3];
  const float* X;
  const float* xw;
};

struct MLayer {
  void* kcache;
  void* vcache;
  const float *bq, *bk, *bv, *q_norm, *k_norm;
};

struct MParams {
  const MPhase* phases;
  int nphases;
  const MLayer* layers;
  int hidden, vocab, n_heads, n_kv_heads, cap, head_dim, kv_esize;
  float eps, scale;
  const uint8_t* embed;
  int* d_token;
  int* d_pos;
  int* d_err;
  float *x, *q, *k, *v, *attn, *logits, *am_val;
  int* am_idx;
  const float *rope_cos, *rope_sin;
  float *ws_m, *ws_l, *ws_o;  // attention partials, [Hk][nc][G] (and [D])
  int nc;                     // most context chunks per KV head
  unsigned* bar;              // grid barrier counter, zero at launch
  int* abort;                 // set when a CTA gives up a wait, zero at launch
  const unsigned* wait_limit; // polls a grid barrier wait makes before the step gives up
  int stage_bytes, nstages;
  int pf_permille;  // share (1/1000) of a CTA's rows of a gate|up phase pulled into L2 ahead
};

// Tensor-core plan of one matvec phase (host): sets F.tc, F.SR, F.win and
// the row split when the phase suits the tensor-core path (n % 256 == 0,
// at least 32 blocks a row, fragments within the shared region); returns
// its tile bytes, or 0 (F.tc = 0) when it does not.
int megastep_plan_tc(MPhase& F, int grid);

// Rows per tile, window tiles and stage size of one matvec phase (host).
// Returns false when the rows are too long for the kernel (more than 20
// warps' worth of 32-block columns).
bool megastep_plan_matvec(MPhase& F, int grid, int stage_target);

// Dynamic shared memory of the kernel for P.stage_bytes / P.nstages.
size_t megastep_smem(const MParams& P);

// Largest nstages that fits for a given stage size.
int megastep_max_stages(int stage_bytes);

// Shared memory available to the ring of stages.
int megastep_ring_bytes();

// Launches the step kernel (cooperative, grid = one CTA per SM) on `st`.
int megastep_launch(const MParams& P, int head_dim, int kv_dtype, int grid, cudaStream_t st);

}  // namespace q8d
