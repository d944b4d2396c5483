/*
 * fp8idx oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, obviously-correct CPU statement of the FP8 "lightning
 * indexer" logits that the GPU library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load this file's
 * shared object.  It shares no code, header, table or constant with the CUDA
 * path; it includes only the C standard library and OpenMP.
 *
 * Sources (web pages; cited by title and section):
 *   [DEC] aiter PR 5047 "[HIP] [JIT] fp8_paged_mqa_logits: hand-written gfx950
 *         decode indexer kernel"
 *   [PRE] aiter PR 5046 "[HIP] [JIT] fp8_mqa_logits: hand-written gfx950
 *         prefill indexer kernel"
 *   [ISS] aiter issue 5477 "gfx950 paged MQA logits: next_n spends the tile on
 *         program count, leaving the kernel's own M-efficiency curve unused"
 *   [OFP8] OCP 8-bit Floating Point Specification, E4M3 encoding.
 *
 * What is computed (the definition, [DEC §Motivation], [PRE §Motivation]):
 *
 *   logits[m, n] = sum_h relu(<Q[m,h,:], K[n,:]>) * kv_scale[n] * weights[m,h]
 *
 * Arithmetic: every e4m3 code is decoded to a double from the format
 * definition; each 128-term dot product of two e4m3 values is exact in double
 * (products are multiples of 2^-18 bounded by 448^2, so any sum of 128 of them
 * needs at most 43 significant bits); the per-head term and the head sum are
 * formed in double in the formula's literal order (scale inside the head sum).
 * Results are returned as doubles; -inf marks positions outside the window.
 *
 * Pins (tests that tie this file to something other than itself) live in the
 * test suite: an all-256-code decode check against the format and a library
 * cast, hand-worked cases, a non-negative closed form that reduces to a
 * matrix-vector product, the kv_scale hoist, linearity in the weights, the
 * zero contribution of negative-dot heads, exact window placement, block-table
 * permutation invariance and decode/prefill consistency.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- e4m3 decode, from the format definition [OFP8] -----------------------
 * bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * exponent 0: subnormal, value = m/8 * 2^(1-7).
 * otherwise: value = (1 + m/8) * 2^(e-7); S.1111.111 is NaN; no infinities. */
double oracle_e4m3_to_double(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int expo = (code >> 3) & 0xF;
  const int mant = code & 0x7;
  double mag;
  if (expo == 0xF && mant == 0x7) return NAN;
  if (expo == 0)
    mag = ldexp((double)mant / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
  return sign ? -mag : mag;
}

/* <a, b> over `dim` e4m3 codes, summed in double (exact, see header). */
static double dot_e4m3(const uint8_t* a, const uint8_t* b, int dim) {
  double s = 0.0;
  for (int d = 0; d < dim; ++d)
    s += oracle_e4m3_to_double(a[d]) * oracle_e4m3_to_double(b[d]);
  return s;
}

/* One logit: the literal formula for one query row and one K row.
 * q_row: [heads, dim] e4m3, w_row: [heads] f32, k_row: [dim] e4m3. */
static double logit_one(const uint8_t* q_row, const float* w_row,
                        const uint8_t* k_row, float kv_scale, int heads,
                        int dim) {
  double total = 0.0;
  for (int h = 0; h < heads; ++h) {
    const double d = dot_e4m3(q_row + (size_t)h * dim, k_row, dim);
    const double r = d > 0.0 ? d : 0.0; /* relu */
    total += r * (double)kv_scale * (double)w_row[h];
  }
  return total;
}

/* ---- decode: fp8_paged_mqa_logits ------------------------------------------
 * [DEC §Technical Details]: the decode op takes q_fp8, kv_cache_fp8, weights,
 * context_lens, block_tables, max_model_len and writes only the causal window
 * p <= context_lens[b] - next_n + n; the -inf outside it is the caller's
 * ([DEC §GLM-5.2-MXFP4 E2E]: the caller pre-fills -inf).  [ISS §The ask]: one
 * output row per speculative token, causal bound context_length - next_n +
 * pid_next_n.
 *
 * Layouts (the plainest reading; the pages do not print shapes):
 *   q            [batch, next_n, heads, dim]        e4m3
 *   weights      [batch * next_n, heads]            f32
 *   context_lens [batch]                            i32
 *   block_tables [batch, max_blocks]                i32 (physical block ids)
 *   kv_cache     [num_blocks, block_size*(dim+4)]   bytes: a block holds its
 *                block_size K rows of `dim` e4m3 bytes, then block_size f32
 *                scales.  For block_size 1 this is the plain co-packed cache
 *                ([DEC §Technical Details]: "1 reads the plain co-packed
 *                cache"): 128 K bytes then a 4-byte scale per token.
 *   output row r = b*next_n + n, column p in [0, max_model_len).
 *
 * Token p of request b lives in block block_tables[b][p / block_size], slot
 * p % block_size.  Returns 0, or -1 when a needed block id is out of range or
 * a context exceeds what the table or max_model_len can address (a caller
 * precondition). */
typedef struct {
  const uint8_t* q;
  const uint8_t* kv_cache;
  const float* weights;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int64_t num_blocks;
  int32_t block_size;
  int32_t max_blocks;
  int32_t batch, next_n, heads, dim;
  int32_t max_model_len;
} oracle_paged_args;

/* Window test for decode: position p of row (b, n) is written iff
 * 0 <= p <= ctx - next_n + n and p < max_model_len. */
static int decode_in_window(const oracle_paged_args* a, int b, int n, int64_t p) {
  const int64_t last = (int64_t)a->context_lens[b] - a->next_n + n;
  return p >= 0 && p <= last && p < a->max_model_len;
}

static int decode_precondition_ok(const oracle_paged_args* a, int b) {
  const int64_t ctx = a->context_lens[b];
  if (ctx < 0) return 1; /* an empty window is legal */
  if (ctx > a->max_model_len) return 0;
  if (ctx > (int64_t)a->max_blocks * a->block_size) return 0;
  return 1;
}

/* The logit at (row, p); caller guarantees p is inside the window. */
static int decode_logit(const oracle_paged_args* a, int b, int n, int64_t p,
                        double* value) {
  const int64_t blk = p / a->block_size;
  const int64_t slot = p % a->block_size;
  const int64_t page = a->block_tables[(int64_t)b * a->max_blocks + blk];
  if (page < 0 || page >= a->num_blocks) return -1;
  const int64_t page_bytes = (int64_t)a->block_size * (a->dim + 4);
  const uint8_t* base = a->kv_cache + page * page_bytes;
  const uint8_t* k_row = base + slot * a->dim;
  float scale;
  {
    const uint8_t* sp = base + (int64_t)a->block_size * a->dim + 4 * slot;
    /* bytes -> f32 (little-endian host, the same byte order as the device) */
    union { uint8_t u[4]; float f; } cvt;
    cvt.u[0] = sp[0]; cvt.u[1] = sp[1]; cvt.u[2] = sp[2]; cvt.u[3] = sp[3];
    scale = cvt.f;
  }
  const int64_t row = (int64_t)b * a->next_n + n;
  const uint8_t* q_row = a->q + row * a->heads * a->dim;
  const float* w_row = a->weights + row * a->heads;
  *value = logit_one(q_row, w_row, k_row, scale, a->heads, a->dim);
  return 0;
}

/* Rows [row_begin, row_end) of the decode output, dense, into
 * out[(row - row_begin) * max_model_len + p]; -inf outside each window. */
int oracle_paged_mqa_logits(const oracle_paged_args* a, int64_t row_begin,
                            int64_t row_end, double* out) {
  int bad = 0;
  const int64_t width = a->max_model_len;
  for (int b = 0; b < a->batch; ++b)
    if (!decode_precondition_ok(a, b)) return -1;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t row = row_begin; row < row_end; ++row) {
    const int b = (int)(row / a->next_n);
    const int n = (int)(row % a->next_n);
    double* dst = out + (row - row_begin) * width;
    for (int64_t p = 0; p < width; ++p) {
      if (!decode_in_window(a, b, n, p)) {
        dst[p] = -INFINITY;
        continue;
      }
      if (decode_logit(a, b, n, p, &dst[p]) != 0) bad = 1;
    }
  }
  return bad ? -1 : 0;
}

/* Individual elements (row[i], col[i]) of the decode output. */
int oracle_paged_mqa_logits_at(const oracle_paged_args* a, int64_t count,
                               const int64_t* rows, const int64_t* cols,
                               double* vals) {
  int bad = 0;
  for (int b = 0; b < a->batch; ++b)
    if (!decode_precondition_ok(a, b)) return -1;
#pragma omp parallel for schedule(dynamic, 64) reduction(| : bad)
  for (int64_t i = 0; i < count; ++i) {
    const int b = (int)(rows[i] / a->next_n);
    const int n = (int)(rows[i] % a->next_n);
    if (!decode_in_window(a, b, n, cols[i])) {
      vals[i] = -INFINITY;
      continue;
    }
    if (decode_logit(a, b, n, cols[i], &vals[i]) != 0) bad = 1;
  }
  return bad ? -1 : 0;
}

/* ---- prefill: fp8_mqa_logits -----------------------------------------------
 * [PRE §Motivation]: K is a contiguous [N, dim] e4m3 buffer with a separate
 * [N] f32 scale; row m is defined for n in [cu_seqlen_ks[m], cu_seqlen_ke[m])
 * and is -inf elsewhere.  [PRE §Test Plan] lists bounds below zero, below the
 * start, and past seq_len_kv as legal input; the window is therefore taken as
 * [max(ks, 0), min(ke, N)), empty when that is empty.
 *
 * Layouts: q [M, heads, dim] e4m3; k [N, dim] e4m3; kv_scale [N] f32;
 * weights [M, heads] f32; ks, ke [M] i32; output [M, N]. */
typedef struct {
  const uint8_t* q;
  const uint8_t* k;
  const float* kv_scale;
  const float* weights;
  const int32_t* ks;
  const int32_t* ke;
  int64_t rows; /* M */
  int64_t cols; /* N */
  int32_t heads, dim;
} oracle_prefill_args;

static int prefill_in_window(const oracle_prefill_args* a, int64_t m, int64_t n) {
  int64_t lo = a->ks[m], hi = a->ke[m];
  if (lo < 0) lo = 0;
  if (hi > a->cols) hi = a->cols;
  return n >= lo && n < hi;
}

static double prefill_logit(const oracle_prefill_args* a, int64_t m, int64_t n) {
  return logit_one(a->q + m * a->heads * a->dim, a->weights + m * a->heads,
                   a->k + n * a->dim, a->kv_scale[n], a->heads, a->dim);
}

/* Rows [row_begin, row_end), dense, into out[(m - row_begin) * N + n]. */
int oracle_mqa_logits(const oracle_prefill_args* a, int64_t row_begin,
                      int64_t row_end, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = row_begin; m < row_end; ++m) {
    double* dst = out + (m - row_begin) * a->cols;
    for (int64_t n = 0; n < a->cols; ++n)
      dst[n] = prefill_in_window(a, m, n) ? prefill_logit(a, m, n) : -INFINITY;
  }
  return 0;
}

int oracle_mqa_logits_at(const oracle_prefill_args* a, int64_t count,
                         const int64_t* rows, const int64_t* cols, double* vals) {
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t i = 0; i < count; ++i)
    vals[i] = prefill_in_window(a, rows[i], cols[i])
                  ? prefill_logit(a, rows[i], cols[i])
                  : -INFINITY;
  return 0;
}

/* Threads OpenMP will use for the loops above (reported with CPU timings). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
