/*
 * lp_oracle.c -- plain, slow, obviously-correct CPU oracle for grammar-constrained
 * logit masking and per-row sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the test suite, the package smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library: every conversion, the random-number generator and the sampling rule are
 * written out here again from their definitions.
 *
 * Sources (web pages, cited by title and section):
 *   [XG]  XGrammar docs, "Bitmask Operations": apply_token_bitmask_inplace
 *         (the double loop over rows and tokens, the "Padding" and "Indices" notes).
 *   [MAX] Modular MAX docs, "apply_packed_bitmask": out-of-place apply with fill_value;
 *         trailing bits beyond the vocabulary are never read.
 *   [LP]  Kernel Hub "logits-processor": "Ops" (sample: temperature <= 0 is greedy,
 *         top_k <= 0 / top_p >= 1 / min_p <= 0 disable a filter, the filters are
 *         intersected, the draw is keyed by (seed, row, offset)); "Correctness"
 *         (greedy and top_k = 1 return the argmax); "How it works" (a single
 *         keep-threshold, Gumbel-max draw over the kept set).
 *   [TRT] TensorRT-Edge-LLM "Guided Decoder": a mask row with no allowed token is
 *         unsatisfiable (rowHasAnyToken, unsatisfiableSlots).
 *   [PH]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
 *         (SC'11): the Philox-4x32 bijection with 10 rounds.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - filters are all evaluated on the same temperature-scaled softmax, and the
 *     kept set is every candidate whose probability is >= the largest of the three
 *     thresholds (ties at the threshold are all kept), clamped to p_max;
 *   - top-p keeps the shortest descending prefix whose mass reaches top_p (the
 *     crossing token is kept);
 *   - min-p is relative to the row maximum probability;
 *   - greedy is the argmax of the raw masked logits, lowest index on ties;
 *   - a row with no candidate returns -1;
 *   - Gumbel noise g = -log(-log u), u = ((x >> 9) + 0.5) * 2^-23, x = word (v & 3)
 *     of Philox4x32-10 at counter (v >> 2, row, lo32(offset), hi32(offset)) and key
 *     (lo32(seed), hi32(seed)).
 *
 * All floating-point work of the sampler is in double precision.  Inputs in
 * half or bfloat16 are decoded exactly to double from their bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { LPO_F32 = 0, LPO_F16 = 1, LPO_BF16 = 2 };

/* ---------------------------------------------------------------- decoding */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double lpo_f16_value(uint16_t h) {
  const int sign = h >> 15;
  const int ex = (h >> 10) & 0x1f;
  const int fr = h & 0x3ff;
  double v;
  if (ex == 0)
    v = ldexp((double)fr, -24); /* subnormal: fr * 2^(1-15-10) */
  else if (ex == 31)
    v = fr ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + fr), ex - 25); /* (1.fr) * 2^(ex-15) */
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
static double lpo_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double lpo_value(const void* base, int dtype, int64_t i) {
  if (dtype == LPO_F32) {
    float f;
    memcpy(&f, (const char*)base + 4 * i, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + 2 * i, 2);
  return dtype == LPO_F16 ? lpo_f16_value(h) : lpo_bf16_value(h);
}

/* ---------------------------------------------------------------- encoding */

/* Round x to the nearest value with a p-bit significand, ties to even, in a
   format whose smallest normal exponent is emin and largest is emax.  Values past
   the largest finite magnitude become infinity.  Written from the definition of
   IEEE round-to-nearest-even; rint() rounds to nearest, ties to even, in the
   default floating-point environment. */
static double lpo_round_format(double x, int p, int emin, int emax) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e2;
  (void)frexp(fabs(x), &e2); /* |x| = f * 2^e2, f in [0.5, 1) */
  int lead = e2 - 1;         /* exponent of the leading bit */
  if (lead < emin) lead = emin;
  const double quantum = ldexp(1.0, lead - (p - 1));
  const double r = rint(x / quantum) * quantum;
  const double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
  if (fabs(r) > max_finite) return x > 0 ? INFINITY : -INFINITY;
  return r;
}

static uint16_t lpo_f16_bits(double r) { /* r already representable */
  uint16_t s = signbit(r) ? 0x8000 : 0;
  double a = fabs(r);
  if (isnan(r)) return 0x7e00;
  if (isinf(a)) return s | 0x7c00;
  if (a < ldexp(1.0, -14)) return s | (uint16_t)(a / ldexp(1.0, -24)); /* subnormal */
  int e2;
  double f = frexp(a, &e2); /* a = f 2^e2, leading exponent e2-1 */
  int ex = e2 - 1 + 15;
  uint16_t fr = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
  return s | (uint16_t)(ex << 10) | fr;
}

static uint16_t lpo_bf16_bits(double r) { /* r already representable in bf16 */
  if (isnan(r)) return 0x7fc0;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Store value `fill` (a binary32) as one element of the given dtype,
   rounded to nearest-even where the dtype is narrower. */
static void lpo_store_fill(void* base, int dtype, int64_t i, float fill) {
  if (dtype == LPO_F32) {
    memcpy((char*)base + 4 * i, &fill, 4);
    return;
  }
  uint16_t h;
  if (dtype == LPO_F16)
    h = lpo_f16_bits(lpo_round_format((double)fill, 11, -14, 15));
  else
    h = lpo_bf16_bits(lpo_round_format((double)fill, 8, -126, 127));
  memcpy((char*)base + 2 * i, &h, 2);
}

/* Exposed for tests: encode one binary32 value to the dtype's bit pattern. */
uint32_t lpo_encode(float x, int dtype) {
  uint32_t out = 0;
  if (dtype == LPO_F32) {
    memcpy(&out, &x, 4);
  } else {
    uint16_t h = 0;
    lpo_store_fill(&h, dtype, 0, x);
    out = h;
  }
  return out;
}

/* Exposed for tests: decode one element's bit pattern to double. */
double lpo_decode(uint32_t bits, int dtype) {
  if (dtype == LPO_F32) {
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
  return dtype == LPO_F16 ? lpo_f16_value((uint16_t)bits) : lpo_bf16_value((uint16_t)bits);
}

static int lpo_elt_size(int dtype) { return dtype == LPO_F32 ? 4 : 2; }

/* ------------------------------------------------------------ bitmask bits */

/* [XG] get_bitmask_value(bitmask, i, j): bit (j mod 32) of word j / 32 of row i,
   the word read as an unsigned 32-bit pattern.  1 keeps the token, 0 masks it. */
static int lpo_bit(const int32_t* bitmask, int64_t bitmask_stride, int64_t row, int64_t j) {
  uint32_t w = (uint32_t)bitmask[row * bitmask_stride + j / 32];
  return (int)((w >> (j % 32)) & 1u);
}

/* [XG] Padding note: vocab_size defaults to min(logits width, words * 32). */
int64_t lpo_resolve_vocab(int64_t vocab_size, int64_t cols, int64_t bitmask_words) {
  if (vocab_size >= 0) return vocab_size;
  int64_t w = bitmask_words * 32;
  return cols < w ? cols : w;
}

/* ------------------------------------------------------------------- apply */

/* [XG] apply_token_bitmask_inplace and [MAX] apply_packed_bitmask in one routine.
   out receives a copy of logits (every row, every column of the first `cols`),
   then, for each selected row b and each j < vocab_size whose bit is 0,
   out[b, j] = fill.  When out == logits (same pointer and stride) this is the
   in-place op.  Selected rows are indices[0..num_indices) if indices != NULL,
   else 0..B-1; an index outside [0, min(B, bitmask_rows)) is skipped.
   Returns 0, or -1 for an inconsistent geometry. */
int lpo_apply(void* out, int64_t out_stride, const void* logits, int dtype, int64_t B,
              int64_t cols, int64_t logits_stride, const int32_t* bitmask,
              int64_t bitmask_rows, int64_t bitmask_words, int64_t bitmask_stride,
              float fill, int64_t vocab_size, const int32_t* indices, int64_t num_indices) {
  const int es = lpo_elt_size(dtype);
  vocab_size = lpo_resolve_vocab(vocab_size, cols, bitmask_words);
  if (vocab_size > cols || vocab_size > bitmask_words * 32) return -1;
  if (out != logits || out_stride != logits_stride) {
    for (int64_t b = 0; b < B; ++b)
      memcpy((char*)out + b * out_stride * es, (const char*)logits + b * logits_stride * es,
             (size_t)(cols * es));
  }
  const int64_t nrows = indices ? num_indices : B;
  const int64_t row_limit = B < bitmask_rows ? B : bitmask_rows;
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t b = indices ? (int64_t)indices[i] : i;
    if (b < 0 || b >= row_limit) continue;
    for (int64_t j = 0; j < vocab_size; ++j)
      if (lpo_bit(bitmask, bitmask_stride, b, j) == 0)
        lpo_store_fill(out, dtype, b * out_stride + j, fill);
  }
  return 0;
}

/* [TRT] Guided Decoder, struct Impl: the mask the apply kernel reads comes with a
   per-row flag (deviceRowNeedsMask), and a row whose flag is zero is left alone;
   rowHasAnyToken is true when the row's mask admits at least one token, and
   fillMasks reports a slot whose mask is all zero as unsatisfiable.  In place:
   for each row b with flags == NULL or flags[b] != 0 and each j < vocab_size
   whose bit is 0, logits[b, j] = -inf.  has_token (when not NULL) gets, per row,
   1 if some j < vocab_size is kept (every j of an unflagged row), else 0.
   Returns 0, or -1 for an inconsistent geometry (bitmask_rows < B included). */
int lpo_apply_rows(void* logits, int dtype, int64_t B, int64_t cols, int64_t logits_stride,
                   const int32_t* bitmask, int64_t bitmask_rows, int64_t bitmask_words,
                   int64_t bitmask_stride, int64_t vocab_size, const uint8_t* flags,
                   int32_t* has_token) {
  vocab_size = lpo_resolve_vocab(vocab_size, cols, bitmask_words);
  if (vocab_size > cols || vocab_size > bitmask_words * 32 || bitmask_rows < B) return -1;
  for (int64_t b = 0; b < B; ++b) {
    const int masked = flags == NULL || flags[b] != 0;
    int any = 0;
    for (int64_t j = 0; j < vocab_size; ++j) {
      if (!masked || lpo_bit(bitmask, bitmask_stride, b, j)) {
        any = 1;
      } else {
        lpo_store_fill(logits, dtype, b * logits_stride + j, -INFINITY);
      }
    }
    if (has_token) has_token[b] = any;
  }
  return 0;
}

/* ------------------------------------------------------------------ Philox */

/* [PH] Philox-4x32 with 10 rounds.  One round multiplies words 0 and 2 of the
   counter by the two round constants, then forms the new counter from the high
   and low product halves XORed with the other two words and the round key; the
   key is bumped by the two Weyl constants before each round after the first. */
void lpo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
    const uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
    const uint32_t y0 = (uint32_t)(prod1 >> 32) ^ x1 ^ k0;
    const uint32_t y1 = (uint32_t)prod1;
    const uint32_t y2 = (uint32_t)(prod0 >> 32) ^ x3 ^ k1;
    const uint32_t y3 = (uint32_t)prod0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Raw 32-bit word for token v of a row under (seed, offset). */
uint32_t lpo_random_word(uint64_t seed, uint64_t offset, uint64_t row, uint64_t v) {
  uint32_t ctr[4] = {(uint32_t)(v >> 2), (uint32_t)row, (uint32_t)offset,
                     (uint32_t)(offset >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  lpo_philox4x32_10(ctr, key, out);
  return out[v & 3];
}

/* Uniform in [2^-24, 1 - 2^-24]: the top 23 bits of the word, centred. */
double lpo_uniform(uint32_t x) { return ((double)(x >> 9) + 0.5) * ldexp(1.0, -23); }

double lpo_gumbel(uint32_t x) { return -log(-log(lpo_uniform(x))); }

/* ---------------------------------------------------------------- sampling */

typedef struct {
  double p;
  int64_t v;
} lpo_cand;

/* order: probability descending, then token index ascending */
static int lpo_cmp(const void* a, const void* b) {
  const lpo_cand* x = (const lpo_cand*)a;
  const lpo_cand* y = (const lpo_cand*)b;
  if (x->p > y->p) return -1;
  if (x->p < y->p) return 1;
  return (x->v > y->v) - (x->v < y->v);
}

/* One row.  l[0..V) are the row's logits as doubles; allowed[j] != 0 marks a
   token the mask keeps (NULL: every token).  Writes the drawn id; optionally the
   keep flags (keep_out[0..V)), the probabilities (p_out[0..V), 0 outside the
   candidates) and the threshold (thr_out; 0 when no filter is active, -1 for a
   greedy or empty row).  Returns 0, or -1 on allocation failure. */
static int lpo_row(const double* l, const uint8_t* allowed, int64_t V, uint64_t row,
                   double T, int32_t top_k, double top_p, double min_p, uint64_t seed,
                   uint64_t offset, int64_t* id_out, uint8_t* keep_out, double* p_out,
                   double* thr_out) {
  if (keep_out) memset(keep_out, 0, (size_t)V);
  if (p_out)
    for (int64_t j = 0; j < V; ++j) p_out[j] = 0.0;
  if (thr_out) *thr_out = -1.0;

  /* candidates: allowed by the mask and not -inf */
  int64_t n = 0;
  for (int64_t j = 0; j < V; ++j)
    if ((!allowed || allowed[j]) && l[j] > -INFINITY) ++n;
  if (n == 0) { /* [TRT] unsatisfiable row */
    *id_out = -1;
    return 0;
  }

  /* [LP] temperature <= 0 is greedy; greedy and top_k = 1 return the argmax */
  if (!(T > 0.0) || top_k == 1) {
    int64_t best = -1;
    for (int64_t j = 0; j < V; ++j) {
      if ((allowed && !allowed[j]) || !(l[j] > -INFINITY)) continue;
      if (best < 0 || l[j] > l[best]) best = j;
    }
    *id_out = best;
    if (keep_out) keep_out[best] = 1;
    return 0;
  }

  lpo_cand* c = (lpo_cand*)malloc((size_t)n * sizeof(lpo_cand));
  double* z = (double*)malloc((size_t)V * sizeof(double));
  if (!c || !z) {
    free(c);
    free(z);
    return -1;
  }

  /* softmax of z = l / T over the candidates */
  double zmax = -INFINITY;
  for (int64_t j = 0; j < V; ++j) {
    z[j] = l[j] / T;
    if ((!allowed || allowed[j]) && l[j] > -INFINITY && z[j] > zmax) zmax = z[j];
  }
  double S = 0.0;
  int64_t k = 0;
  for (int64_t j = 0; j < V; ++j) {
    if ((allowed && !allowed[j]) || !(l[j] > -INFINITY)) continue;
    c[k].p = exp(z[j] - zmax);
    c[k].v = j;
    S += c[k].p;
    ++k;
  }
  for (int64_t i = 0; i < n; ++i) c[i].p /= S;
  qsort(c, (size_t)n, sizeof(lpo_cand), lpo_cmp);
  const double p_max = c[0].p;

  /* [LP] the three filters, each a threshold on the same probabilities */
  double t_k = 0.0, t_p = 0.0, t_m = 0.0;
  if (top_k > 0) t_k = (top_k >= n) ? c[n - 1].p : c[top_k - 1].p;
  if (top_p < 1.0) {
    double cum = 0.0;
    int64_t cut = n - 1; /* no prefix reaches top_p: keep every candidate */
    for (int64_t i = 0; i < n; ++i) {
      cum += c[i].p;
      if (cum >= top_p) {
        cut = i;
        break;
      }
    }
    t_p = c[cut].p;
  }
  if (min_p > 0.0) t_m = min_p * p_max;
  double t = t_k;
  if (t_p > t) t = t_p;
  if (t_m > t) t = t_m;
  if (t > p_max) t = p_max;
  if (thr_out) *thr_out = t;

  /* [LP] Gumbel-max over the kept set, lowest index on ties */
  int64_t best = -1;
  double best_score = -INFINITY;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t j = c[i].v;
    if (p_out) p_out[j] = c[i].p;
    if (!(c[i].p >= t)) continue;
    if (keep_out) keep_out[j] = 1;
    const double score = z[j] + lpo_gumbel(lpo_random_word(seed, offset, row, (uint64_t)j));
    if (best < 0 || score > best_score || (score == best_score && j < best)) {
      best = j;
      best_score = score;
    }
  }
  *id_out = best;
  free(c);
  free(z);
  return 0;
}

/* Fused mask + sample over B rows (plain sample when bitmask == NULL).
   Row b of the arrays is logical row r = row_ids ? row_ids[b] : b: r keys the
   noise, and the row is masked by bitmask row r when indices == NULL (every row)
   or when r appears in indices[0..num_indices); other rows sample unmasked.  The
   bitmask is addressed by the logical row.  Per-row parameters are full arrays of
   length B.  Optional outputs (NULL to skip): keep_out [B, vocab_size],
   p_out [B, vocab_size], thr_out [B].
   Returns 0, or -1 for an inconsistent geometry / allocation failure. */
int lpo_mask_and_sample(const void* logits, int dtype, int64_t B, int64_t cols,
                        int64_t logits_stride, const int32_t* bitmask, int64_t bitmask_rows,
                        int64_t bitmask_words, int64_t bitmask_stride, int64_t vocab_size,
                        const int32_t* indices, int64_t num_indices, const float* temperature,
                        const int32_t* top_k, const float* top_p, const float* min_p,
                        uint64_t seed, uint64_t offset, const int64_t* row_ids,
                        int64_t* ids_out, uint8_t* keep_out, double* p_out, double* thr_out) {
  if (bitmask)
    vocab_size = lpo_resolve_vocab(vocab_size, cols, bitmask_words);
  else if (vocab_size < 0)
    vocab_size = cols;
  if (vocab_size > cols || (bitmask && vocab_size > bitmask_words * 32)) return -1;
  const int64_t V = vocab_size;
  double* l = (double*)malloc((size_t)(V > 0 ? V : 1) * sizeof(double));
  uint8_t* allowed = (uint8_t*)malloc((size_t)(V > 0 ? V : 1));
  if (!l || !allowed) {
    free(l);
    free(allowed);
    return -1;
  }
  int rc = 0;
  for (int64_t b = 0; b < B && rc == 0; ++b) {
    const int64_t r = row_ids ? row_ids[b] : b;
    int masked = 0;
    if (bitmask) {
      if (!indices) {
        masked = 1;
      } else {
        for (int64_t i = 0; i < num_indices; ++i)
          if ((int64_t)indices[i] == r) masked = 1;
      }
      if (r < 0 || r >= bitmask_rows) masked = 0;
    }
    for (int64_t j = 0; j < V; ++j) {
      l[j] = lpo_value(logits, dtype, b * logits_stride + j);
      allowed[j] = masked ? (uint8_t)lpo_bit(bitmask, bitmask_stride, r, j) : 1;
    }
    rc = lpo_row(l, allowed, V, (uint64_t)r, (double)temperature[b], top_k[b],
                 (double)top_p[b], (double)min_p[b], seed, offset, &ids_out[b],
                 keep_out ? keep_out + b * V : NULL, p_out ? p_out + b * V : NULL,
                 thr_out ? thr_out + b : NULL);
  }
  free(l);
  free(allowed);
  return rc;
}
