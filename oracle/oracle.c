/*
 * Q8_0 decode-step oracle: plain, slow, scalar C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file.  It is used by the tests under tests/, by
 * __graft_entry__.smoke() and by the cpu_baseline / reference leg of bench.py.
 * It shares no code, header, table or constant generator with the CUDA
 * library under q8_block_quantized_matvec_gb300/csrc.
 *
 * Every function computes the plain definition of one step of the decode path
 * described on the pages
 *   [P3] "IV.4: One command buffer per token" (sections "Eight kernels",
 *        "One command buffer", "The correctness ladder"),
 *   [P1] "minfer Metal Backend Design",
 *   [P2] "Metal Backend Optimizations" (section 3.3 "Decode optimizations
 *        (GPU)", split-attention design),
 * accumulating in IEEE double and rounding once at the end.  There is no
 * blocking, chunking or reordering beyond what those definitions state.
 *
 * Parity status of each function is recorded next to it ("pinned by ...").
 * The whole decode step (orc_decode_step) is pinned only through its parts
 * and through invariants; for seeded full-size inputs the pages print no
 * output values, so its end-to-end numbers are parity unpinned by the pages.
 *
 * Compile with -ffp-contract=off so no multiply-add is fused behind our back.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_QBLOCK 32        /* quants per Q8_0 block                       */
#define ORC_QBLOCK_BYTES 34  /* 2-byte little-endian f16 scale + 32 int8     */

#define ORC_KV_F32 0
#define ORC_KV_F16 1
#define ORC_KV_Q8_0 2  /* packed: rows of kvw/32 Q8_0 blocks */

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32, written from the format's definition.    */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.       */
/* ------------------------------------------------------------------------ */

/* Exact widening of a binary16 bit pattern.  Normal numbers are
 * (1024 + frac) * 2^(exp - 25); subnormals are frac * 2^-24; exp == 31 is
 * infinity (frac == 0) or NaN.  Pinned by tests/test_oracle_pins.py
 * (exhaustive over all 65536 patterns against numpy's float16 and against
 * hand-decoded examples such as the pages' 0x2C00 = 0.0625 block scale). */
float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)frac, -24);
  } else if (e == 31) {
    if (frac == 0) {
      mag = INFINITY;
    } else {
      return sign ? -NAN : NAN;
    }
  } else {
    mag = ldexp((double)(1024 + frac), e - 25);
  }
  return (float)(sign ? -mag : mag);
}

/* Round a non-negative double that holds an integer plus a fraction to the
 * nearest integer, ties to even.  All operations are exact in double for the
 * magnitudes used here (< 2^25). */
static double orc_round_half_even(double r) {
  double fl = floor(r);
  double diff = r - fl;
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary32 -> binary16, round to nearest, ties to even (the IEEE default
 * rounding attribute).  Overflow goes to infinity, NaN becomes the quiet NaN
 * 0x7E00 with the input's sign, subnormal results are produced exactly.
 * Pinned by tests/test_oracle_pins.py (all binary16 values and midpoints
 * between neighbours, numpy's float16 cast on random and extreme values). */
uint16_t orc_f32_to_f16(float f) {
  uint32_t bits;
  memcpy(&bits, &f, 4);
  uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
  double a = fabs((double)f);
  if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
  if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: units of 2^-24; 1024 units is the smallest normal,
     * whose encoding 0x0400 follows directly from the subnormals. */
    double m = orc_round_half_even(a * ldexp(1.0, 24));
    return (uint16_t)(sign | (uint16_t)m);
  }
  int e2;
  frexp(a, &e2);             /* a = fr * 2^e2, fr in [0.5, 1)  */
  int e = e2 - 1;            /* a in [2^e, 2^(e+1))            */
  double m = orc_round_half_even(a * ldexp(1.0, 10 - e)); /* in [1024, 2048] */
  if (m >= 2048.0) {
    m = 1024.0;
    e += 1;
  }
  int biased = e + 15;
  if (biased >= 31) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)(m - 1024.0));
}

/* ------------------------------------------------------------------------ */
/* Q8_0 block: [P3] "Eight kernels" (decode_scale, q8_matvec) and           */
/* "The decoder: kernels and helpers" (embed_row): 34 bytes, bytes 0-1 the  */
/* little-endian f16 scale, bytes 2..33 the 32 signed quants; the value of  */
/* quant j is scale * q_j.  Rows of an [p][n] matrix are n/32 consecutive   */
/* blocks; row r starts at byte r * (n/32) * 34.                            */
/* ------------------------------------------------------------------------ */

static double orc_block_scale(const uint8_t* blk) {
  uint16_t bits = (uint16_t)(blk[0] | (blk[1] << 8));
  return (double)orc_f16_to_f32(bits);
}

static int orc_block_quant(const uint8_t* blk, int j) {
  int b = blk[2 + j];
  return b >= 128 ? b - 256 : b; /* two's complement int8 */
}

/* Dequantise row `row` of a [*][n] Q8_0 matrix into out[n] (exact). */
void orc_q8_dequant_row(const uint8_t* w, int64_t row, int n, double* out) {
  int bpr = n / ORC_QBLOCK;
  const uint8_t* wrow = w + row * (int64_t)bpr * ORC_QBLOCK_BYTES;
  for (int b = 0; b < bpr; ++b) {
    const uint8_t* blk = wrow + (int64_t)b * ORC_QBLOCK_BYTES;
    double s = orc_block_scale(blk);
    for (int j = 0; j < ORC_QBLOCK; ++j) out[b * ORC_QBLOCK + j] = s * orc_block_quant(blk, j);
  }
}

/* One output of the Q8_0 matrix-vector product ([P3] "Eight kernels",
 * q8_matvec; the exact float reference of "The correctness ladder"):
 *   out[r] = sum_b sum_j scale(r,b) * q(r,b,j) * x[32b + j]
 * in double; absterm = sum of |scale*q*x| for the tolerance
 * |gpu - oracle| <= 1e-5 * absterm.  x is used as given (never quantised). */
static void orc_q8_row_dot(const uint8_t* w, int64_t row, int n, const double* x,
                           double* sum_out, double* abs_out) {
  int bpr = n / ORC_QBLOCK;
  const uint8_t* wrow = w + row * (int64_t)bpr * ORC_QBLOCK_BYTES;
  double sum = 0.0, absum = 0.0;
  for (int b = 0; b < bpr; ++b) {
    const uint8_t* blk = wrow + (int64_t)b * ORC_QBLOCK_BYTES;
    double s = orc_block_scale(blk);
    for (int j = 0; j < ORC_QBLOCK; ++j) {
      double t = s * (double)orc_block_quant(blk, j) * x[b * ORC_QBLOCK + j];
      sum += t;
      absum += fabs(t);
    }
  }
  *sum_out = sum;
  *abs_out = absum;
}

/* ---- a tiny parallel-for over independent output rows ------------------ */
/* Each row is computed by exactly the same scalar code whichever thread runs
 * it; threads only split the index range. */
typedef struct {
  void (*fn)(void* ctx, int64_t i);
  void* ctx;
  int64_t begin, end;
} orc_range;

static void* orc_range_run(void* arg) {
  orc_range* r = (orc_range*)arg;
  for (int64_t i = r->begin; i < r->end; ++i) r->fn(r->ctx, i);
  return NULL;
}

static void orc_parallel_for(int64_t count, int nthreads, void (*fn)(void*, int64_t), void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads == 1 || count < 64) {
    for (int64_t i = 0; i < count; ++i) fn(ctx, i);
    return;
  }
  pthread_t th[256];
  orc_range rg[256];
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    rg[t].fn = fn;
    rg[t].ctx = ctx;
    rg[t].begin = count * t / nthreads;
    rg[t].end = count * (t + 1) / nthreads;
    if (pthread_create(&th[t], NULL, orc_range_run, &rg[t]) == 0) {
      started = t + 1;
    } else {
      orc_range_run(&rg[t]);
      started = t + 1;
      th[t] = 0;
    }
  }
  for (int t = 0; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

typedef struct {
  const uint8_t* w;
  int n;
  const double* x;
  double* sum;
  double* absum;
} orc_mv_ctx;

static void orc_mv_row(void* c, int64_t r) {
  orc_mv_ctx* m = (orc_mv_ctx*)c;
  orc_q8_row_dot(m->w, r, m->n, m->x, &m->sum[r], &m->absum[r]);
}

/* Matvec with double input and double outputs (used inside the decode step). */
static void orc_q8_matvec_d(const uint8_t* w, const double* x, int n, int p, double* out,
                            double* absum, int nthreads) {
  double* ab = absum ? absum : (double*)malloc(sizeof(double) * (size_t)p);
  orc_mv_ctx c = {w, n, x, out, ab};
  orc_parallel_for(p, nthreads, orc_mv_row, &c);
  if (!absum) free(ab);
}

/* f32 in, f32 out (rounded once from the double sum), absterm in double.
 * Pinned by tests/test_oracle_pins.py: sum(x) for all-ones quants with scale
 * 1, exact integer sums for x = 1, one-hot x (every (row, column) byte), the
 * pages' fabricated 0x2C00-scale test matrix, brute force on tiny shapes. */
void orc_q8_matvec(const uint8_t* w, const float* x, int n, int p, float* out, double* absterm,
                   int nthreads) {
  double* xd = (double*)malloc(sizeof(double) * (size_t)n);
  double* sd = (double*)malloc(sizeof(double) * (size_t)p);
  for (int i = 0; i < n; ++i) xd[i] = x[i];
  orc_q8_matvec_d(w, xd, n, p, sd, absterm, nthreads);
  for (int r = 0; r < p; ++r) out[r] = (float)sd[r];
  free(xd);
  free(sd);
}

/* Selected output rows only (for full-size matrices whose full product is
 * too slow): out[i], absterm[i] belong to row rows[i]. */
void orc_q8_matvec_rows(const uint8_t* w, const float* x, int n, const int64_t* rows, int nrows,
                        float* out, double* absterm) {
  double* xd = (double*)malloc(sizeof(double) * (size_t)n);
  for (int i = 0; i < n; ++i) xd[i] = x[i];
  for (int i = 0; i < nrows; ++i) {
    double s, a;
    orc_q8_row_dot(w, rows[i], n, xd, &s, &a);
    out[i] = (float)s;
    absterm[i] = a;
  }
  free(xd);
}

/* Small-M product: m independent matvecs sharing one weight matrix,
 *   Y[i][r] = sum_k X[i][k] * W[r][k]
 * ([P2] "Metal Backend Optimizations": the nt in [2, 8] batched matvec gap
 * and the nt >= 2 quantised GEMM tier).  X row i starts at X + i*ldx, Y row i
 * at Y + i*ldy.  absterm has m*p entries laid out like Y with ld p. */
void orc_q8_matmul(const uint8_t* w, const float* X, int ldx, int m, int n, int p, float* Y,
                   int ldy, double* absterm, int nthreads) {
  for (int i = 0; i < m; ++i)
    orc_q8_matvec(w, X + (int64_t)i * ldx, n, p, Y + (int64_t)i * ldy,
                  absterm ? absterm + (int64_t)i * p : NULL, nthreads);
}

/* ------------------------------------------------------------------------ */
/* KV cache: [P3] "Eight kernels" (append_kv) and [P1] on the KV layout:    */
/* per layer a [cap][n_kv_heads * head_dim] row-major cache; the step       */
/* writes row `pos`.  The f16 cache stores the f32 value rounded to nearest */
/* even.  Pinned by tests (row placement, untouched neighbours, RNE).       */
/* ------------------------------------------------------------------------ */

/* ------------------------------------------------------------------------ */
/* Packed Q8_0 KV cache ([P1] "Execution dispatch", packed q8_0 KV: a store */
/* byte-identical to the CPU quantizer, and attention that reads the 34-byte */
/* blocks natively).  A cache row of kvw elements is kvw/32 consecutive      */
/* Q8_0 blocks in the weight matrices' layout: row t starts at byte          */
/* t * (kvw/32) * 34, element i of the row is quant i%32 of block i/32.      */
/* The pages name the CPU quantizer without restating it; it is read as the  */
/* Q8_0 format's reference quantizer, computed in f32 as that quantizer is:  */
/*   amax = max_j |x_j|,  d = amax / 127,  id = (d != 0) ? 1 / d : 0,        */
/*   q_j = x_j * id rounded to the nearest integer, halves away from zero,   */
/*   stored scale = d rounded to binary16 (nearest even).                    */
/* Inputs are finite.  Pinned by tests: an all-zero block, exact multiples   */
/* of a power of two, halves rounding away from zero, the round-trip bound   */
/* and sign symmetry on random blocks.                                       */
/* ------------------------------------------------------------------------ */
void orc_q8_0_quantize_block(const float* x, uint8_t* blk) {
  float amax = 0.0f;
  for (int j = 0; j < ORC_QBLOCK; ++j) {
    float a = fabsf(x[j]);
    if (a > amax) amax = a;
  }
  float d = amax / 127.0f;
  float id = d != 0.0f ? 1.0f / d : 0.0f;
  uint16_t sb = orc_f32_to_f16(d);
  blk[0] = (uint8_t)(sb & 0xff);
  blk[1] = (uint8_t)(sb >> 8);
  for (int j = 0; j < ORC_QBLOCK; ++j) {
    float v = x[j] * id;          /* one f32 product (no contraction: -ffp-contract=off) */
    int q = (int)roundf(v);       /* nearest, halves away from zero */
    blk[2 + j] = (uint8_t)(int8_t)q;
  }
}

static size_t orc_kv_row_bytes(int kv_dtype, int kvw) {
  if (kv_dtype == ORC_KV_F32) return 4 * (size_t)kvw;
  if (kv_dtype == ORC_KV_F16) return 2 * (size_t)kvw;
  return (size_t)(kvw / ORC_QBLOCK) * ORC_QBLOCK_BYTES;
}

void orc_kv_append(const float* k, const float* v, void* kc, void* vc, int kv_dtype, int kvw,
                   int64_t pos) {
  if (kv_dtype == ORC_KV_Q8_0) {
    uint8_t* kb = (uint8_t*)kc + (size_t)pos * orc_kv_row_bytes(kv_dtype, kvw);
    uint8_t* vb = (uint8_t*)vc + (size_t)pos * orc_kv_row_bytes(kv_dtype, kvw);
    for (int b = 0; b < kvw / ORC_QBLOCK; ++b) {
      orc_q8_0_quantize_block(k + (int64_t)b * ORC_QBLOCK, kb + (size_t)b * ORC_QBLOCK_BYTES);
      orc_q8_0_quantize_block(v + (int64_t)b * ORC_QBLOCK, vb + (size_t)b * ORC_QBLOCK_BYTES);
    }
    return;
  }
  if (kv_dtype == ORC_KV_F32) {
    float* kf = (float*)kc + pos * kvw;
    float* vf = (float*)vc + pos * kvw;
    for (int i = 0; i < kvw; ++i) {
      kf[i] = k[i];
      vf[i] = v[i];
    }
  } else {
    uint16_t* kh = (uint16_t*)kc + pos * kvw;
    uint16_t* vh = (uint16_t*)vc + pos * kvw;
    for (int i = 0; i < kvw; ++i) {
      kh[i] = orc_f32_to_f16(k[i]);
      vh[i] = orc_f32_to_f16(v[i]);
    }
  }
}

/* Element idx = t * kvw + i of a cache (kvw a multiple of 32 for Q8_0:
 * block idx / 32 of the packed rows, which start at multiples of kvw/32). */
static double orc_kv_read(const void* c, int kv_dtype, int64_t idx) {
  if (kv_dtype == ORC_KV_F32) return (double)((const float*)c)[idx];
  if (kv_dtype == ORC_KV_Q8_0) {
    const uint8_t* blk = (const uint8_t*)c + (size_t)(idx / ORC_QBLOCK) * ORC_QBLOCK_BYTES;
    return orc_block_scale(blk) * (double)orc_block_quant(blk, (int)(idx % ORC_QBLOCK));
  }
  return (double)orc_f16_to_f32(((const uint16_t*)c)[idx]);
}

/* ------------------------------------------------------------------------ */
/* Grouped-query decode attention for one query token ([P3] "Eight kernels",*/
/* attention_decode): query head h reads KV head h / (H / Hk); over the L   */
/* cached rows t = 0..L-1                                                   */
/*   s_t = scale * q_h . K[t, g]                                            */
/*   p_t = exp(s_t - max s) / sum exp(s - max s)                            */
/*   o_h = sum_t p_t V[t, g]                                                */
/* Unchunked: [P2] section 3.3 states the split result is invariant to the  */
/* chunk count, so the oracle is the plain two-pass softmax in double.      */
/* absterm[h,d] = sum_t p_t |V[t,g,d]|.  Pinned by tests: L = 1 returns the */
/* V row exactly, identical keys and q = 0 give the mean of V, brute force  */
/* on the pages' 4/2-head, hd 16, seq 9 shape.                              */
/* ------------------------------------------------------------------------ */

int orc_gqa_decode_attn(const float* q, const void* kc, const void* vc, int kv_dtype, int n_heads,
                        int n_kv_heads, int head_dim, int L, float scale, float* out,
                        double* absterm) {
  if (n_kv_heads <= 0 || n_heads % n_kv_heads != 0 || L < 1) return -1;
  int group = n_heads / n_kv_heads;
  int64_t kvw = (int64_t)n_kv_heads * head_dim;
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  for (int h = 0; h < n_heads; ++h) {
    int g = h / group;
    const float* qh = q + (int64_t)h * head_dim;
    double mx = -INFINITY;
    for (int t = 0; t < L; ++t) {
      double d = 0.0;
      for (int j = 0; j < head_dim; ++j)
        d += (double)qh[j] * orc_kv_read(kc, kv_dtype, (int64_t)t * kvw + (int64_t)g * head_dim + j);
      s[t] = (double)scale * d;
      if (s[t] > mx) mx = s[t];
    }
    double z = 0.0;
    for (int t = 0; t < L; ++t) {
      s[t] = exp(s[t] - mx);
      z += s[t];
    }
    for (int j = 0; j < head_dim; ++j) {
      double o = 0.0, a = 0.0;
      for (int t = 0; t < L; ++t) {
        double pt = s[t] / z;
        double vv = orc_kv_read(vc, kv_dtype, (int64_t)t * kvw + (int64_t)g * head_dim + j);
        o += pt * vv;
        a += pt * fabs(vv);
      }
      out[(int64_t)h * head_dim + j] = (float)o;
      if (absterm) absterm[(int64_t)h * head_dim + j] = a;
    }
  }
  free(s);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Windowed decode attention ([P1] "Execution dispatch", window modes: an    */
/* explicit [lo, hi) span, or a map of up to four (cell, len) runs per       */
/* query, e.g. a shared prefix plus a private run).  The query attends to    */
/* exactly the cells of its runs: the plain definition is the attention     */
/* above over the cache rows of the runs gathered in run order (a softmax    */
/* over a set; the order changes rounding only).  runs: nruns (cell, len)   */
/* pairs; every run inside [0, cap) and at least one row in all, else -1.    */
/* Pinned by tests: one run [0, L) equals the causal attention bitwise, a   */
/* one-cell window returns that cell's V row bitwise, brute force over     */
/* gathered rows, and a window shifted by one cell changes the output.     */
/* ------------------------------------------------------------------------ */
int orc_gqa_decode_attn_runs(const float* q, const void* kc, const void* vc, int kv_dtype,
                             int n_heads, int n_kv_heads, int head_dim, int cap, const int* runs,
                             int nruns, float scale, float* out, double* absterm) {
  int kvw = n_kv_heads * head_dim;
  if (kv_dtype == ORC_KV_Q8_0 && kvw % ORC_QBLOCK) return -1;
  size_t rb = orc_kv_row_bytes(kv_dtype, kvw);
  int64_t total = 0;
  for (int r = 0; r < nruns; ++r) {
    int cell = runs[2 * r], len = runs[2 * r + 1];
    if (cell < 0 || len < 0 || (int64_t)cell + len > cap) return -1;
    total += len;
  }
  if (total < 1) return -1;
  uint8_t* kg = (uint8_t*)malloc(rb * (size_t)total);
  uint8_t* vg = (uint8_t*)malloc(rb * (size_t)total);
  int64_t w = 0;
  for (int r = 0; r < nruns; ++r)
    for (int t = 0; t < runs[2 * r + 1]; ++t, ++w) {
      memcpy(kg + (size_t)w * rb, (const uint8_t*)kc + (size_t)(runs[2 * r] + t) * rb, rb);
      memcpy(vg + (size_t)w * rb, (const uint8_t*)vc + (size_t)(runs[2 * r] + t) * rb, rb);
    }
  int rc = orc_gqa_decode_attn(q, kg, vg, kv_dtype, n_heads, n_kv_heads, head_dim, (int)total,
                               scale, out, absterm);
  free(kg);
  free(vg);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Decode-step glue ([P3] "Eight kernels": rms_norm_row, rope_row,           */
/* add_inplace, silu_hadamard, argmax_row; "The decoder": embed_row).       */
/* ------------------------------------------------------------------------ */

/* RMSNorm: out = x / sqrt(mean(x^2) + eps) * w. */
void orc_rmsnorm(const double* x, const float* w, int dim, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < dim; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / dim + eps);
  for (int i = 0; i < dim; ++i) out[i] = x[i] * inv * (double)w[i];
}

/* Non-interleaved rotary embedding of one head: pairs (i, i + d/2) rotate by
 * pos * theta^(-i / (d/2)). */
void orc_rope_head(double* x, int head_dim, int64_t pos, double theta) {
  int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    double freq = 1.0 / pow(theta, (double)i / (double)half);
    double ang = (double)pos * freq;
    double c = cos(ang), s = sin(ang);
    double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = a * s + b * c;
  }
}

/* SwiGLU gate: silu(g) * u with silu(g) = g / (1 + exp(-g)). */
double orc_silu_mul(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/* Index of the largest value; ties go to the lowest index ([P3] argmax_row
 * and its planted-tie test).  NaN never wins. */
int64_t orc_argmax(const float* x, int64_t n) {
  int64_t best = -1;
  float bv = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    if (isnan(x[i])) continue;
    if (best < 0 || x[i] > bv) {
      bv = x[i];
      best = i;
    }
  }
  return best;
}

/* ------------------------------------------------------------------------ */
/* Whole decode step ([P3] "One command buffer": per layer rms_norm, q/k/v  */
/* projections, QK-norm (Qwen3) or q/k/v bias (Qwen2, [P1] weight list),    */
/* RoPE, KV append, attention, o projection, residual add, rms_norm,        */
/* gate/up, SwiGLU, down, residual add; then final norm, lm_head, argmax).  */
/* Activations stay in double; the KV cache stores the f32-rounded k/v      */
/* (rounded again to f16 for an f16 cache).  Logits are rounded to f32 once */
/* and the argmax is taken over them.                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint8_t *wq, *wk, *wv, *wo, *wg, *wu, *wd; /* Q8_0 matrices            */
  const float *attn_norm, *ffn_norm;               /* [hidden]                 */
  const float *q_norm, *k_norm;                    /* [head_dim] (qk_norm)     */
  const float *bq, *bk, *bv;                       /* biases (qkv_bias)        */
  void *kcache, *vcache;                           /* [cap][n_kv*head_dim]     */
} orc_layer;

typedef struct {
  int hidden, n_layers, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int qk_norm, qkv_bias, kv_dtype, cap;
  float rms_eps, rope_theta;
  const uint8_t* embed;   /* Q8_0 [vocab][hidden] */
  const float* out_norm;  /* [hidden]             */
  const uint8_t* lm_head; /* Q8_0 [vocab][hidden] */
  const orc_layer* layers;
} orc_model;

int orc_decode_step(const orc_model* m, int64_t token, int64_t pos, float* logits,
                    int64_t* next_token, int nthreads) {
  if (pos < 0 || pos >= m->cap || token < 0 || token >= m->vocab) return -1;
  int h = m->hidden, H = m->n_heads, Hk = m->n_kv_heads, d = m->head_dim;
  int qw = H * d, kvw = Hk * d, F = m->ffn;
  double eps = m->rms_eps;
  double *x = calloc((size_t)h, 8), *xn = calloc((size_t)h, 8), *tmp = calloc((size_t)h, 8);
  double *q = calloc((size_t)qw, 8), *k = calloc((size_t)kvw, 8), *v = calloc((size_t)kvw, 8);
  double *g = calloc((size_t)F, 8), *u = calloc((size_t)F, 8);
  double* lg = calloc((size_t)m->vocab, 8);
  float *kf = calloc((size_t)kvw, 4), *vf = calloc((size_t)kvw, 4);
  double* att = calloc((size_t)qw, 8);
  double* hd = calloc((size_t)d, 8);

  orc_q8_dequant_row(m->embed, token, h, x);
  for (int li = 0; li < m->n_layers; ++li) {
    const orc_layer* L = &m->layers[li];
    orc_rmsnorm(x, L->attn_norm, h, eps, xn);
    orc_q8_matvec_d(L->wq, xn, h, qw, q, NULL, nthreads);
    orc_q8_matvec_d(L->wk, xn, h, kvw, k, NULL, nthreads);
    orc_q8_matvec_d(L->wv, xn, h, kvw, v, NULL, nthreads);
    if (m->qkv_bias) {
      for (int i = 0; i < qw; ++i) q[i] += L->bq[i];
      for (int i = 0; i < kvw; ++i) k[i] += L->bk[i];
      for (int i = 0; i < kvw; ++i) v[i] += L->bv[i];
    }
    if (m->qk_norm) {
      for (int hh = 0; hh < H; ++hh) {
        orc_rmsnorm(q + (int64_t)hh * d, L->q_norm, d, eps, hd);
        memcpy(q + (int64_t)hh * d, hd, sizeof(double) * (size_t)d);
      }
      for (int hh = 0; hh < Hk; ++hh) {
        orc_rmsnorm(k + (int64_t)hh * d, L->k_norm, d, eps, hd);
        memcpy(k + (int64_t)hh * d, hd, sizeof(double) * (size_t)d);
      }
    }
    for (int hh = 0; hh < H; ++hh) orc_rope_head(q + (int64_t)hh * d, d, pos, m->rope_theta);
    for (int hh = 0; hh < Hk; ++hh) orc_rope_head(k + (int64_t)hh * d, d, pos, m->rope_theta);
    for (int i = 0; i < kvw; ++i) {
      kf[i] = (float)k[i];
      vf[i] = (float)v[i];
    }
    orc_kv_append(kf, vf, L->kcache, L->vcache, m->kv_dtype, kvw, pos);
    /* attention in double with the double-precision query */
    {
      int group = H / Hk;
      int64_t Lrows = pos + 1;
      double* s = malloc(sizeof(double) * (size_t)Lrows);
      double scale = 1.0 / sqrt((double)d);
      for (int hh = 0; hh < H; ++hh) {
        int gg = hh / group;
        double mx = -INFINITY;
        for (int64_t t = 0; t < Lrows; ++t) {
          double acc = 0.0;
          for (int j = 0; j < d; ++j)
            acc += q[(int64_t)hh * d + j] *
                   orc_kv_read(L->kcache, m->kv_dtype, t * kvw + (int64_t)gg * d + j);
          s[t] = scale * acc;
          if (s[t] > mx) mx = s[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < Lrows; ++t) {
          s[t] = exp(s[t] - mx);
          z += s[t];
        }
        for (int j = 0; j < d; ++j) {
          double o = 0.0;
          for (int64_t t = 0; t < Lrows; ++t)
            o += s[t] / z * orc_kv_read(L->vcache, m->kv_dtype, t * kvw + (int64_t)gg * d + j);
          att[(int64_t)hh * d + j] = o;
        }
      }
      free(s);
    }
    orc_q8_matvec_d(L->wo, att, qw, h, tmp, NULL, nthreads);
    for (int i = 0; i < h; ++i) x[i] += tmp[i];
    orc_rmsnorm(x, L->ffn_norm, h, eps, xn);
    orc_q8_matvec_d(L->wg, xn, h, F, g, NULL, nthreads);
    orc_q8_matvec_d(L->wu, xn, h, F, u, NULL, nthreads);
    for (int i = 0; i < F; ++i) g[i] = orc_silu_mul(g[i], u[i]);
    orc_q8_matvec_d(L->wd, g, F, h, tmp, NULL, nthreads);
    for (int i = 0; i < h; ++i) x[i] += tmp[i];
  }
  orc_rmsnorm(x, m->out_norm, h, eps, xn);
  orc_q8_matvec_d(m->lm_head, xn, h, m->vocab, lg, NULL, nthreads);
  for (int i = 0; i < m->vocab; ++i) logits[i] = (float)lg[i];
  *next_token = orc_argmax(logits, m->vocab);

  free(x); free(xn); free(tmp); free(q); free(k); free(v); free(g); free(u); free(lg);
  free(kf); free(vf); free(att); free(hd);
  return 0;
}
