/*
 * q8d — Q8_0 single-token decode hot path for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer named d_* or documented as "device" is a device
 * pointer owned by the caller (the library never frees it).  Every compute
 * entry point is asynchronous on the CUDA stream passed as `stream`
 * (a cudaStream_t cast to void*; NULL means the legacy default stream) and
 * returns an int status:
 *     0               success (work enqueued)
 *     Q8D_EINVAL      null pointer or impossible size/shape
 *     Q8D_EALIGN      a pointer or stride breaks the stated alignment
 *     Q8D_EUNSUPPORTED a valid shape this build does not run
 *                     (n % 32 != 0, head_dim not 64/128, H % Hk != 0, ...)
 *     Q8D_ERANGE      an index/length outside its buffer (host-visible args)
 *     Q8D_ECUDA       a CUDA call failed; q8d_last_cuda_error() has the code
 *     Q8D_ETIMEOUT    a bounded host wait ran out
 *     Q8D_ENOMEM      the library's own allocation failed (step create only)
 * On any non-zero status nothing was launched.  There is no fallback path:
 * an unsupported case is refused, never computed another way.
 *
 * Quantities that live in device memory (positions, lengths, token ids) are
 * checked on the device: a bad value sets a bit in the caller's int error
 * word (Q8D_DERR_*), the affected write is skipped and the affected outputs
 * are set to NaN, so a silent no-write cannot pass for a result.
 *
 * Formats (from "IV.4: One command buffer per token", sections "Eight
 * kernels" and "The decoder: kernels and helpers"):
 *   Q8_0 block  34 bytes: little-endian IEEE binary16 scale (bytes 0-1) then
 *               32 two's-complement int8 quants (bytes 2-33); value of quant
 *               j is scale * q_j.
 *   Q8_0 matrix [p][n], row-major, n % 32 == 0: row r is n/32 consecutive
 *               blocks starting at byte r * (n/32) * 34 (no padding).
 *               The base must be 16-byte aligned.
 *   KV cache    per layer [cap][n_kv_heads * head_dim] of f32 or f16
 *               (Q8D_KV_F32 / Q8D_KV_F16); KV head g occupies columns
 *               [g*head_dim, (g+1)*head_dim) of every row ("minfer Metal
 *               Backend Design" / "Metal Backend Optimizations", the
 *               [nkv][nk*hd] layout shared with llama.cpp).
 *   Packed KV   Q8D_KV_Q8_0 ("minfer Metal Backend Design", "Execution
 *               dispatch": packed q8_0 KV): the same [cap][kv_width] cache
 *               stored as a Q8_0 matrix, row t = kv_width/32 consecutive
 *               34-byte blocks starting at byte t * kv_width/32 * 34, so
 *               KV head g is blocks [g*head_dim/32, (g+1)*head_dim/32).
 *               Rows are written by the Q8_0 quantizer: per block
 *               d = max|x| / 127, q_j = x_j * (1/d) rounded to nearest with
 *               halves away from zero, scale = d rounded to binary16, all in
 *               f32 (an all-zero block stores zeros); inputs must be finite.
 */
#ifndef Q8D_H
#define Q8D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q8D_OK 0
#define Q8D_EINVAL (-1)
#define Q8D_EALIGN (-2)
#define Q8D_EUNSUPPORTED (-3)
#define Q8D_ERANGE (-4)
#define Q8D_ECUDA (-5)
#define Q8D_ETIMEOUT (-6)
#define Q8D_ENOMEM (-7)

#define Q8D_KV_F32 0
#define Q8D_KV_F16 1
#define Q8D_KV_Q8_0 2 /* packed: every cache row is kv_width/32 Q8_0 blocks */

/* Bits of the device-side error word. */
#define Q8D_DERR_POS_RANGE 0x1   /* append position outside [0, cap)          */
#define Q8D_DERR_LEN_RANGE 0x2   /* attended length outside [1, cap]          */
#define Q8D_DERR_TOKEN_RANGE 0x4 /* token id outside [0, vocab)               */
#define Q8D_DERR_WAIT 0x8        /* a bounded in-kernel wait gave up          */

/* Library version (major*10000 + minor*100 + patch). */
int q8d_version(void);

/* Static text for a status code. */
const char* q8d_strerror(int status);

/* The cudaError_t of the last Q8D_ECUDA returned on this thread (0 if none). */
int q8d_last_cuda_error(void);

/* ------------------------------------------------------------------------
 * q8d_matvec — Q8_0 dequantising matrix-vector product
 * ("IV.4: One command buffer per token", "Eight kernels": q8_matvec).
 *   out[r] = sum_{b < n/32} scale(r,b) * sum_{j < 32} q(r,b,j) * x[32b + j]
 * x: device f32[n]; w_q8: device Q8_0 [p][n] (16-byte aligned);
 * out: device f32[p], fully overwritten, must not overlap x or w.
 * n % 32 == 0 (else Q8D_EUNSUPPORTED); n == 0 writes zeros; p == 0 is a
 * no-op.  f32 accumulation; x is used as given (never quantised).
 * ---------------------------------------------------------------------- */
int q8d_matvec(const float* x, const void* w_q8, float* out, int n, int p, void* stream);

/* ------------------------------------------------------------------------
 * q8d_matmul_small_m — the same weight matrix applied to m activations
 * ("Metal Backend Optimizations": the nt in [2, 8] batched-matvec gap and
 * the quantised GEMM tier for nt >= 2).
 *   Y[i][r] = sum_k X[i][k] * W[r][k],   i < m, r < p
 * X: device f32, row i at X + i*ldx (ldx >= n); Y: device f32, row i at
 * Y + i*ldy (ldy >= p), only the first p entries of each row are written.
 * m <= 8: f32-accurate paths (within 1e-5 of sum|terms| per output): the
 * tensor-core matvec with up to four activation rows per pass sharing every
 * decoded weight block (exact f16 quants, activations split into f16 hi +
 * lo, f32 accumulation) where the shape suits it (n % 256 == 0, n >= 2048,
 * p >= 16 rows per SM, the rows' activation fragments in shared memory),
 * else CUDA cores with the weights read once for up to four rows.
 * m >= 9 and n % 256 == 0: tensor-core path (tcgen05.mma, f16 operands:
 * the weights as f16 of scale * q, rounded once; the activations as f16
 * under a power-of-two scale per row, rounded once; f32 accumulation):
 * relative accuracy ~2^-11 per product, i.e. within 2e-3 of sum|terms|
 * per output (plus 2^-25 * sum|x| where scale * q is below 2^-14).  Block
 * scales above 511.75 (scale * q beyond f16) make the outputs of their
 * 128-row tile NaN.  It first writes the activations, rounded to f16, into
 * a workspace laid out as the MMA's B operand, with the rows' scales
 * (q8d_matmul_small_m_workspace_bytes(m, n) bytes); this entry point takes
 * that workspace from the stream's memory pool (cudaMallocAsync) and frees
 * it stream-ordered behind the kernels; q8d_matmul_small_m_ws uses the
 * caller's.  Other m >= 9 shapes run the f32 CUDA-core path.
 * 1 <= m <= 256; n % 32 == 0; X and w_q8 16-byte aligned, ldx % 4 == 0,
 * Y 4-byte aligned (Q8D_EALIGN otherwise); Y must not overlap X or w_q8
 * (Q8D_EINVAL).  m == 0 or p == 0: Q8D_OK, nothing written.
 * ---------------------------------------------------------------------- */
int q8d_matmul_small_m(const float* X, int ldx, const void* w_q8, float* Y, int ldy, int m,
                       int n, int p, void* stream);

/* Bytes of the workspace q8d_matmul_small_m_ws needs for m activation rows of
 * n elements: 2 * n * (m rounded up to 16 per block of 128 rows) + 16 *
 * ceil(m / 4) when the tensor-core path takes the shape (9 <= m <= 256,
 * n % 256 == 0), else 0. */
size_t q8d_matmul_small_m_workspace_bytes(int m, int n);

/* q8d_matmul_small_m with a caller-owned workspace: device memory of at
 * least q8d_matmul_small_m_workspace_bytes(m, n) bytes, 16-byte aligned,
 * overlapping none of X, w_q8 and Y, not in use by other work until the
 * call's kernels on `stream` have completed (the call writes it, then
 * reads it).  Q8D_EINVAL if it is needed and null or too small, or
 * overlaps an operand; Q8D_EALIGN if misaligned.  Unused (may be null)
 * when the size is 0. */
int q8d_matmul_small_m_ws(const float* X, int ldx, const void* w_q8, float* Y, int ldy, int m,
                          int n, int p, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * q8d_kv_append — write one token's K and V rows into the caches
 * ("IV.4: One command buffer per token", "Eight kernels": append_kv).
 *   kcache[pos][i] = cvt(k[i]), vcache[pos][i] = cvt(v[i]), i < kv_width
 * cvt is the identity for an f32 cache, round-to-nearest-even to binary16
 * for an f16 cache and the Q8_0 quantizer of each 32-element block for a
 * packed cache (kv_width % 32 == 0, else Q8D_EUNSUPPORTED; the stored bytes
 * equal a scalar CPU quantizer's).  pos is read from device memory (*d_pos)
 * so a captured graph replays unchanged; pos outside [0, cap) sets
 * Q8D_DERR_POS_RANGE in *d_err and writes nothing.  k, v: device
 * f32[kv_width]; caches: device, cap rows (a packed cache 16-byte aligned,
 * else Q8D_EALIGN); d_err: device int (OR-ed into, never cleared).
 * ---------------------------------------------------------------------- */
int q8d_kv_append(const float* k, const float* v, void* kcache, void* vcache, int kv_dtype,
                  int kv_width, int cap, const int* d_pos, int* d_err, void* stream);

/* Bytes of scratch q8d_gqa_decode_attn needs for these sizes: the split-K
 * partials {m, l, O} of up to a fixed number of chunk slots per sequence
 * and query head (chunk CTAs are split over a batch in proportion to the
 * lengths, on the device).  Pass the cache capacity `cap` as max_len: the
 * call checks ws_bytes against the size for its cap. */
size_t q8d_gqa_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim, int max_len);

/* ------------------------------------------------------------------------
 * q8d_gqa_decode_attn — grouped-query attention of one query token per
 * sequence over a resident KV cache, split over the context ("IV.4: One
 * command buffer per token", "Eight kernels": attention_decode; "Metal
 * Backend Optimizations" 3.3, split-attention partial + combine).
 * For sequence s with length L = d_lens[s] (read on the device) and query
 * head h, KV head g = h / (n_heads / n_kv_heads):
 *   s_t = scale * q[s,h,:] . K[s][t][g*hd : (g+1)*hd],   t < L
 *   out[s,h,:] = sum_t softmax(s)_t * V[s][t][g*hd : (g+1)*hd]
 * If k_new/v_new are non-NULL, row L-1 of sequence s is first written with
 * cvt(k_new[s]), cvt(v_new[s]) (as q8d_kv_append) and the rounded values
 * are the ones attended to.
 *   q, out:  device f32 [batch][n_heads*head_dim]
 *   k_new, v_new: device f32 [batch][n_kv_heads*head_dim] or both NULL
 *   kcache, vcache: device; sequence s's cache starts at element
 *            s*cache_batch_stride, rows of n_kv_heads*head_dim elements,
 *            16-byte aligned, cap rows
 *   d_lens:  device int[batch]; 1 <= L <= cap, else Q8D_DERR_LEN_RANGE is
 *            set in *d_err and that sequence's outputs are NaN
 *   workspace: device scratch of at least
 *            q8d_gqa_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, cap)
 *            bytes (contents need no initialisation)
 * head_dim in {64, 128}; n_heads % n_kv_heads == 0; n_heads/n_kv_heads <= 16.
 * ---------------------------------------------------------------------- */
int q8d_gqa_decode_attn(const float* q, const float* k_new, const float* v_new, void* kcache,
                        void* vcache, int kv_dtype, float* out, int batch, int n_heads,
                        int n_kv_heads, int head_dim, int cap, long long cache_batch_stride,
                        const int* d_lens, float scale, void* workspace, size_t ws_bytes,
                        int* d_err, void* stream);

/* ------------------------------------------------------------------------
 * q8d_gqa_decode_attn_window — q8d_gqa_decode_attn over explicit KV windows
 * ("minfer Metal Backend Design", "Execution dispatch", window modes: an
 * explicit [lo, hi) span per query, or a map of up to four (cell, len) runs
 * per query, e.g. a prefix shared by several sequences plus a private run).
 * Sequence s attends exactly the cache rows of its runs, in run order:
 *   d_runs:  device int [batch][Q8D_MAX_RUNS][2], run r of sequence s is
 *            (cell, len) = (d_runs[s][r][0], d_runs[s][r][1]), the rows
 *            [cell, cell + len) of sequence s's cache; unused runs have
 *            len 0.  A span [lo, hi) is the single run (lo, hi - lo).
 *            Every run must lie in [0, cap) (0 <= cell, 0 <= len,
 *            cell + len <= cap) and the runs must hold at least one row in
 *            all, else Q8D_DERR_LEN_RANGE is set in *d_err and the
 *            sequence's outputs are NaN.
 *   cache_batch_stride: as for q8d_gqa_decode_attn, or 0: every sequence
 *            reads the same cache (shared cells, e.g. a common prefix).
 * With k_new/v_new the rounded new rows are first written at the LAST row
 * of each sequence's window (the last row of its last non-empty run) and
 * attended to; that row must not be read by another sequence of the same
 * call (the calls' writes and reads would race).
 * Other arguments, the workspace and the results are those of
 * q8d_gqa_decode_attn (f32, f16 and packed Q8_0 caches).
 * ---------------------------------------------------------------------- */
#define Q8D_MAX_RUNS 4
int q8d_gqa_decode_attn_window(const float* q, const float* k_new, const float* v_new,
                               void* kcache, void* vcache, int kv_dtype, float* out, int batch,
                               int n_heads, int n_kv_heads, int head_dim, int cap,
                               long long cache_batch_stride, const int* d_runs, float scale,
                               void* workspace, size_t ws_bytes, int* d_err, void* stream);

/* ------------------------------------------------------------------------
 * q8d_gqa_decode_attn_noalloc — q8d_gqa_decode_attn without a caller
 * workspace.  The pages have no counterpart to this entry point.
 * It exists for callers that cannot allocate device memory: code whose
 * device memory is owned by a host framework's allocator or pool that
 * forbids side allocations, and latency-sensitive loops that cannot afford
 * cudaMalloc's implicit device-wide synchronisation.  The split-K scratch
 * lives instead in one fixed array inside libq8d, of
 * q8d_noalloc_scratch_bytes() bytes (4 MiB) on every GPU that loads the
 * library, held until the process exits.  Arguments and results are those
 * of q8d_gqa_decode_attn (the caller still passes q, caches, out, lengths
 * and the error word); sizes whose scratch would exceed the array,
 * i.e. q8d_gqa_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, cap)
 * > q8d_noalloc_scratch_bytes(), are refused with Q8D_ERANGE.
 * The call allocates nothing.  Its first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current)
 * and caches it; make that first call before any stream capture.
 * All calls on a device share the one array, and it keeps the last call's
 * contents (nothing in it needs to start at zero): calls that overlap on the
 * GPU (different streams, or concurrent host threads) race on it.
 * ---------------------------------------------------------------------- */
size_t q8d_noalloc_scratch_bytes(void);
int q8d_gqa_decode_attn_noalloc(const float* q, const float* k_new, const float* v_new,
                                void* kcache, void* vcache, int kv_dtype, float* out, int batch,
                                int n_heads, int n_kv_heads, int head_dim, int cap,
                                long long cache_batch_stride, const int* d_lens, float scale,
                                int* d_err, void* stream);

/* ------------------------------------------------------------------------
 * Decode step graph ("IV.4: One command buffer per token", "One command
 * buffer": the whole step encoded once and submitted as one unit).
 * The step, per layer: RMSNorm -> q/k/v Q8_0 matvecs -> (q/k/v bias) ->
 * (per-head q/k RMSNorm) -> RoPE(q, k) -> KV append -> attention -> o
 * matvec -> residual add -> RMSNorm -> gate/up matvecs -> SiLU(gate)*up ->
 * down matvec -> residual add; then final RMSNorm -> lm_head -> argmax.
 * The token id and position are read from device memory at replay time,
 * the argmax is written back as the next token and the position advanced,
 * so consecutive launches decode consecutive tokens with no host work.
 * All pointers in the descriptors are device pointers owned by the caller
 * and must stay valid until q8d_step_destroy.  Weights, caches and RMSNorm
 * weights must be 16-byte aligned, the other f32 vectors 4-byte aligned
 * (Q8D_EALIGN otherwise).  head_dim in {64, 128}; n_heads % n_kv_heads ==
 * 0; n_heads/n_kv_heads <= 16 with an f32 cache, <= 12 with an f16 cache;
 * n_kv_heads at most the device's SM count (Q8D_EUNSUPPORTED otherwise).
 * ---------------------------------------------------------------------- */
typedef struct q8d_layer_desc {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd; /* Q8_0: [H*hd][hidden], [Hk*hd][hidden] x2,
                                                   [hidden][H*hd], [ffn][hidden] x2,
                                                   [hidden][ffn]                          */
  const float *attn_norm, *ffn_norm;            /* f32 [hidden], 16-byte aligned          */
  const float *q_norm, *k_norm;                 /* f32 [head_dim] (qk_norm) or NULL       */
  const float *bq, *bk, *bv;                    /* f32 biases (qkv_bias) or NULL          */
  void *kcache, *vcache;                        /* [cap][Hk*hd] of kv_dtype               */
} q8d_layer_desc;

typedef struct q8d_step_desc {
  int hidden, n_layers, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int qk_norm;  /* 1: Qwen3-style per-head RMSNorm of q and k after projection */
  int qkv_bias; /* 1: Qwen2-style bias add on q, k, v                          */
  int kv_dtype; /* Q8D_KV_F32 or Q8D_KV_F16                                    */
  int cap;      /* rows of every KV cache                                      */
  float rms_eps, rope_theta;
  const void* embed;      /* Q8_0 [vocab][hidden]                 */
  const float* out_norm;  /* f32 [hidden], 16-byte aligned        */
  const void* lm_head;    /* Q8_0 [vocab][hidden]                 */
  const q8d_layer_desc* layers; /* host array of n_layers (copied at create) */
  int* d_token;           /* device int: input token; receives the argmax     */
  int* d_pos;             /* device int: position of the input token; +1 after */
  int* d_err;             /* device int error word (OR-ed into)               */
  float* d_logits;        /* device f32 [vocab] or NULL (library-owned then)  */
} q8d_step_desc;

typedef struct q8d_step q8d_step;

/* Builds the step: allocates its activation workspace (the only allocation
 * the library makes), prepares per-step tables with kernels on `stream`,
 * captures the step into a CUDA graph and instantiates it.  Synchronises
 * `stream`. */
int q8d_step_create(const q8d_step_desc* desc, void* stream, q8d_step** out);

/* Enqueues one decode step (one graph launch) on `stream`. */
int q8d_step_launch(q8d_step* step, void* stream);

/* One decode step with its inputs and output in host memory, in one call:
 * copies h_token_pos[0] (token id) and h_token_pos[1] (position) to the
 * step's device token and position (one 8-byte copy when they are adjacent
 * in device memory, d_pos == d_token + 1), launches the step graph, and
 * copies the next token id to *h_next_token, all enqueued on `stream`
 * (asynchronous: read *h_next_token after synchronising the stream; pinned
 * host memory keeps the copies asynchronous).  Either pointer may be NULL
 * to skip that copy.  The same operation as the host copies around
 * q8d_step_launch ("IV.4: One command buffer per token": token and
 * position in, next token out), with one call per step instead of four. */
int q8d_step_launch_host(q8d_step* step, const int* h_token_pos, int* h_next_token, void* stream);

/* Copies the step's device error word into *err (synchronous; waits for
 * work already enqueued on `stream`, polling with a time limit of
 * timeout_ms milliseconds, <= 0 meaning 10 s).  Returns Q8D_ETIMEOUT if the
 * limit ran out. */
int q8d_step_status(q8d_step* step, void* stream, int timeout_ms, int* err);

/* Sets how many polls a grid-wide barrier wait inside the step kernel makes
 * before the step gives up (polls == 0 restores the default, 2^21 polls,
 * about a second).  On expiry the step sets Q8D_DERR_WAIT in the error
 * word, every CTA of the step leaves at its next barrier, the remaining
 * phases are skipped (the token and position are not advanced) and the
 * CUDA context stays usable.  The value is written in stream order on
 * `stream` and applies to later launches.  A small value is a way to check
 * that a caller's error handling sees an abandoned step. */
int q8d_step_set_wait_limit(q8d_step* step, unsigned polls, void* stream);

/* Number of kernel nodes one launch runs. */
int q8d_step_kernel_count(const q8d_step* step);

/* Device pointer of the step's logits buffer (f32 [vocab]). */
float* q8d_step_logits(q8d_step* step);

/* Releases the graph and the workspace (not the caller's buffers). */
void q8d_step_destroy(q8d_step* step);

#ifdef __cplusplus
}
#endif
#endif /* Q8D_H */
