/*
 * oracle.c -- plain fp64 CPU oracle of the 4-bit (int4 or NVFP4)
 * mixture-of-experts layer and the 4-bit LM-head projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code with the CUDA path.
 *
 * What it computes (the plain definition, step by step, no blocking, fusion
 * or reordering):
 *   router logits   l[t,e] = sum_i x[t,i] * Wr[e,i] + b[e]        (fp64, i ascending)
 *   softmax         p[t,:] = exp(l - max l) / sum exp(l - max l)
 *   top-k           the k largest logits, descending, equal logits -> lower e
 *   gates           w[t,j] = p[ids_j] / sum_j' p[ids_j']   (or p[ids_j] unrenormalised)
 *   permutation     rows r = t*k + j grouped by expert, ascending r inside an expert
 *   expert FFN      a = Wg[e] x, u = Wu[e] x, h = silu(a) * u, y = Wd[e] h
 *   combine         out[t] = resid[t] + sum_j w[t,j] * y[t,j]   (j ascending)
 *   RMSNorm         xh = x / sqrt(mean(x^2) + eps)               (gain 1)
 *   LM head         z[t,v] = sum_i Wlm[v,i] * xh[t,i];  argmax, lowest v on ties
 * with every int4 weight dequantised exactly: W[n,i] = q[n,i] * s[n, i/32],
 * or, for NVFP4 banks, W[n,i] = e2m1(q[n,i]) * e4m3(s[n, i/16]) * ts (below).
 *
 * Sources.  "Flint 40B : Best Mid Sized LLM" (video transcript): 02:35 -- 256
 * routed experts per mixture layer, a small router picks a few per token;
 * 03:36 -- the output layer maps hidden states to a ~150k vocabulary;
 * 05:39 -- the output layer is quantised to four bits.  "Recursive_SI's First
 * Model Unveiled!", section "Quantization" -- 4-bit weights including the
 * output layer.  The pages give no formula: the steps above are the standard
 * top-k MoE with SwiGLU experts, group-32 symmetric int4 with fp16 scales, and
 * the readings listed in the design notes (softmax over all experts then top-k
 * then renormalise; bias used for selection and gates; stable permutation).
 *
 * Storage formats: bf16 and fp16 values are passed as raw uint16 bits and
 * widened to fp64 exactly.  int4 rows are packed two per byte, element 2b in
 * the low nibble of byte b, two's complement.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

/* ------------------------------------------------------------ formats */

/* bf16: sign, 8-bit exponent, 7-bit fraction -- the top half of an fp32. */
double oracle_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* fp16 (IEEE binary16): sign, 5-bit exponent (bias 15), 10-bit fraction. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1f;
  int fr = h & 0x3ff;
  double v;
  if (ex == 0)
    v = ldexp((double)fr, -24); /* subnormal: fr * 2^-14 * 2^-10 */
  else if (ex == 31)
    v = fr ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + fr), ex - 25); /* (1 + fr/1024) * 2^(ex-15) */
  return sign ? -v : v;
}

/* Round an fp64 value to bf16, nearest with ties to even. */
uint16_t oracle_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7fc0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1; bf16 normals: 2^-126 <= a */
  int unb = e - 1;          /* a = (2m) * 2^unb, 1 <= 2m < 2 */
  double r;
  if (unb < -126) {
    /* subnormal bf16: multiples of 2^-133 */
    r = nearbyint(ldexp(a, 133));
    uint32_t fr = (uint32_t)r; /* may carry into the smallest normal */
    return sign | (uint16_t)fr;
  }
  r = nearbyint(ldexp(m, 8)); /* 8 significant bits: 128 <= r <= 256 */
  if (r == 256.0) {
    r = 128.0;
    unb += 1;
  }
  if (unb > 127) return sign | 0x7f80; /* overflow to infinity */
  return sign | (uint16_t)(((unb + 127) << 7) | ((uint32_t)r - 128));
}

/* Signed value of element i of a packed int4 row. */
static int int4_at(const uint8_t* row, int64_t i) {
  uint8_t byte = row[i >> 1];
  int nib = (i & 1) ? (byte >> 4) : (byte & 0x0f);
  return nib >= 8 ? nib - 16 : nib;
}

/* Dequantise rows x K packed int4 values: out[n,i] = q[n,i] * s[n, i/group]. */
int oracle_dequant_int4(const uint8_t* q, const uint16_t* s, int64_t rows, int64_t K, int64_t group,
                        double* out) {
  if (!q || !s || !out || K % 2 || group <= 0 || K % group) return ORACLE_EINVAL;
  for (int64_t n = 0; n < rows; ++n)
    for (int64_t i = 0; i < K; ++i)
      out[n * K + i] = (double)int4_at(q + n * (K / 2), i) * oracle_f16_to_f64(s[n * (K / group) + i / group]);
  return ORACLE_OK;
}

/* sum_i W[n,i] * v[i] for one packed int4 row, i ascending. */
static double int4_row_dot(const uint8_t* qrow, const uint16_t* srow, int64_t K, int64_t group, const double* v) {
  double acc = 0.0;
  for (int64_t i = 0; i < K; ++i) {
    double w = (double)int4_at(qrow, i) * oracle_f16_to_f64(srow[i / group]);
    acc += w * v[i];
  }
  return acc;
}

/* ------------------------------------------------------------ NVFP4 */

/*
 * NVFP4, the "four-bit NVFP" builds of the model ("Flint 40B : Best Mid Sized
 * LLM", transcript 07:15; "Recursive_SI's First Model Unveiled!", section
 * "Quantization": the final NVFP4 model).  The pages name the format without
 * defining it; this is its public definition (4-bit floating-point elements in
 * 16-element blocks with an 8-bit floating-point scale, plus one fp32 scale
 * per tensor):
 *   element  FP4 E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 *            mantissa; exponent 0 is subnormal (0 or 0.5); no Inf or NaN, so
 *            the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 *   scale    FP8 E4M3 for every 16 consecutive elements along the reduction
 *            dimension: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 *            mantissa; exponent 0 is subnormal; exponent 15 with mantissa 7 is
 *            NaN; no Inf (largest 448);
 *   tensor   one fp32 scale per matrix;
 *   W[n,i] = e2m1(q[n,i]) * e4m3(s[n, i/16]) * ts.
 * Codes are stored two per byte like the int4 values: element 2b in the low
 * nibble of byte b.
 */
double oracle_e2m1_to_f64(uint8_t code) {
  int sign = (code >> 3) & 1;
  int ex = (code >> 1) & 3;
  int m = code & 1;
  double v = (ex == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
  return sign ? -v : v;
}

double oracle_e4m3_to_f64(uint8_t b) {
  int sign = (b >> 7) & 1;
  int ex = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (ex == 15 && m == 7)
    v = NAN;
  else if (ex == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(8.0 + m, ex - 10); /* (1 + m/8) * 2^(ex-7) */
  return sign ? -v : v;
}

#define NVFP4_BLOCK 16

static uint8_t nib_at(const uint8_t* row, int64_t i) {
  uint8_t byte = row[i >> 1];
  return (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0f);
}

/* Dequantise one NVFP4 matrix rows x K: out[n,i] = e2m1(q) * e4m3(s[n, i/16]) * ts. */
int oracle_dequant_nvfp4(const uint8_t* q, const uint8_t* s, float ts, int64_t rows, int64_t K, double* out) {
  if (!q || !s || !out || K % NVFP4_BLOCK) return ORACLE_EINVAL;
  for (int64_t n = 0; n < rows; ++n)
    for (int64_t i = 0; i < K; ++i)
      out[n * K + i] = oracle_e2m1_to_f64(nib_at(q + n * (K / 2), i)) *
                       oracle_e4m3_to_f64(s[n * (K / NVFP4_BLOCK) + i / NVFP4_BLOCK]) * (double)ts;
  return ORACLE_OK;
}

/* sum_i W[n,i] * v[i] for one NVFP4 row, i ascending. */
static double nvfp4_row_dot(const uint8_t* qrow, const uint8_t* srow, double ts, int64_t K, const double* v) {
  double acc = 0.0;
  for (int64_t i = 0; i < K; ++i) {
    double w = oracle_e2m1_to_f64(nib_at(qrow, i)) * oracle_e4m3_to_f64(srow[i / NVFP4_BLOCK]) * ts;
    acc += w * v[i];
  }
  return acc;
}

/* ------------------------------------------------------------ weight banks */

/*
 * A bank of n matrices of rows x K in one of the two 4-bit formats, so that
 * the layer and the LM head below are written once for both.
 *   int4:  q [n, rows, K/2], s16 [n, rows, K/group] fp16
 *   NVFP4: q [n, rows, K/2], s8 [n, rows, K/16] E4M3, ts [n] fp32
 */
typedef struct {
  int nvfp4;
  const uint8_t* q;
  const uint16_t* s16;
  const uint8_t* s8;
  const float* ts;
  int64_t rows, K, group;
} wbank;

static wbank int4_bank(const uint8_t* q, const uint16_t* s, int64_t rows, int64_t K, int64_t group) {
  wbank b = {0, q, s, NULL, NULL, rows, K, group};
  return b;
}

static wbank nvfp4_bank(const uint8_t* q, const uint8_t* s, const float* ts, int64_t rows, int64_t K) {
  wbank b = {1, q, NULL, s, ts, rows, K, NVFP4_BLOCK};
  return b;
}

static int bank_ok(const wbank* b) {
  if (!b->q || b->K % 2 || b->group <= 0 || b->K % b->group) return 0;
  return b->nvfp4 ? (b->s8 && b->ts) : (b->s16 != NULL);
}

/* sum_i W[row,i] * v[i] for row `row` of the bank (counted over all matrices). */
static double bank_row_dot(const wbank* b, int64_t row, const double* v) {
  if (b->nvfp4)
    return nvfp4_row_dot(b->q + row * (b->K / 2), b->s8 + row * (b->K / NVFP4_BLOCK), (double)b->ts[row / b->rows],
                         b->K, v);
  return int4_row_dot(b->q + row * (b->K / 2), b->s16 + row * (b->K / b->group), b->K, b->group, v);
}

/* ------------------------------------------------------------ routing */

/* Router logits l[t,e] = sum_i x[t,i] Wr[e,i] + b[e] (b may be NULL). */
int oracle_router_logits(const uint16_t* x, int64_t T, int64_t d, int64_t E, const float* Wr, const float* b,
                         double* logits) {
  if ((T && !x) || !Wr || !logits || d <= 0 || E <= 0) return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t i = 0; i < d; ++i) acc += oracle_bf16_to_f64(x[t * d + i]) * (double)Wr[e * d + i];
      logits[t * E + e] = acc + (b ? (double)b[e] : 0.0);
    }
  }
  return ORACLE_OK;
}

/* Softmax over the E experts of each token. */
int oracle_softmax(const double* logits, int64_t T, int64_t E, double* p) {
  if ((T && (!logits || !p)) || E <= 0) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    double m = l[0];
    for (int64_t e = 1; e < E; ++e)
      if (l[e] > m) m = l[e];
    double z = 0.0;
    for (int64_t e = 0; e < E; ++e) z += exp(l[e] - m);
    for (int64_t e = 0; e < E; ++e) p[t * E + e] = exp(l[e] - m) / z;
  }
  return ORACLE_OK;
}

typedef struct {
  double l;
  int64_t e;
} le_pair;

/* Descending logit, then ascending expert index. */
static int cmp_desc_logit(const void* a, const void* b) {
  const le_pair* x = (const le_pair*)a;
  const le_pair* y = (const le_pair*)b;
  if (x->l > y->l) return -1;
  if (x->l < y->l) return 1;
  return (x->e > y->e) - (x->e < y->e);
}

/* Top-k by a full sort of (-l, e); gap[t] = l_(k) - l_(k+1) (+inf when k == E). */
int oracle_topk(const double* logits, int64_t T, int64_t E, int64_t k, int32_t* ids, double* gap) {
  if ((T && (!logits || !ids)) || k <= 0 || k > E) return ORACLE_EINVAL;
  le_pair* buf = (le_pair*)malloc(sizeof(le_pair) * (size_t)E);
  if (!buf) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      buf[e].l = logits[t * E + e];
      buf[e].e = e;
    }
    qsort(buf, (size_t)E, sizeof(le_pair), cmp_desc_logit);
    for (int64_t j = 0; j < k; ++j) ids[t * k + j] = (int32_t)buf[j].e;
    if (gap) gap[t] = (k < E) ? buf[k - 1].l - buf[k].l : INFINITY;
  }
  free(buf);
  return ORACLE_OK;
}

/* Gate weights: p of the chosen experts, renormalised to sum 1 when renorm != 0. */
int oracle_gates(const double* p, const int32_t* ids, int64_t T, int64_t E, int64_t k, int renorm, double* w) {
  if ((T && (!p || !ids || !w)) || k <= 0 || k > E) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    double z = 0.0;
    for (int64_t j = 0; j < k; ++j) z += p[t * E + ids[t * k + j]];
    for (int64_t j = 0; j < k; ++j) {
      double v = p[t * E + ids[t * k + j]];
      w[t * k + j] = renorm ? v / z : v;
    }
  }
  return ORACLE_OK;
}

/* Router logits -> softmax -> top-k -> gates; logits/gap may be NULL. */
int oracle_route(const uint16_t* x, int64_t T, int64_t d, int64_t E, int64_t k, const float* Wr, const float* b,
                 int renorm, int32_t* ids, double* w, double* logits_out, double* gap) {
  if (k <= 0 || k > E) return ORACLE_EINVAL;
  double* l = (double*)malloc(sizeof(double) * (size_t)(T * E + 1));
  double* p = (double*)malloc(sizeof(double) * (size_t)(T * E + 1));
  int rc = ORACLE_EINVAL;
  if (l && p) {
    rc = oracle_router_logits(x, T, d, E, Wr, b, l);
    if (!rc) rc = oracle_softmax(l, T, E, p);
    if (!rc) rc = oracle_topk(l, T, E, k, ids, gap);
    if (!rc) rc = oracle_gates(p, ids, T, E, k, renorm, w);
    if (!rc && logits_out) memcpy(logits_out, l, sizeof(double) * (size_t)(T * E));
  }
  free(l);
  free(p);
  return rc;
}

/* ------------------------------------------------------------ permutation */

/*
 * Token -> expert grouping.  For e = 0..E-1, for r = 0..T*k-1 in order, rows
 * with ids[r] == e are appended: sorted_rows[pos] = r, inv[r] = pos.
 * offsets[e] is the position of expert e's first row, offsets[E] = T*k.
 */
int oracle_permute(const int32_t* ids, int64_t T, int64_t E, int64_t k, int32_t* offsets, int32_t* sorted_rows,
                   int32_t* inv) {
  if (!offsets || E <= 0 || k <= 0 || (T && (!ids || !sorted_rows || !inv))) return ORACLE_EINVAL;
  int64_t R = T * k;
  for (int64_t r = 0; r < R; ++r)
    if (ids[r] < 0 || ids[r] >= E) return ORACLE_EINVAL;
  int64_t pos = 0;
  for (int64_t e = 0; e < E; ++e) {
    offsets[e] = (int32_t)pos;
    for (int64_t r = 0; r < R; ++r) {
      if (ids[r] == e) {
        sorted_rows[pos] = (int32_t)r;
        inv[r] = (int32_t)pos;
        ++pos;
      }
    }
  }
  offsets[E] = (int32_t)pos;
  return ORACLE_OK;
}

/* ------------------------------------------------------------ experts */

/*
 * Expert FFN for every (t, j): e = ids[t,j];
 *   a[n] = sum_i Wg[e,n,i] x[t,i],  u[n] = sum_i Wu[e,n,i] x[t,i]   (n < I)
 *   h[n] = a[n] / (1 + exp(-a[n])) * u[n]
 *   y[c] = sum_n Wd[e,c,n] h[n]                                     (c < d)
 * Weight banks: gate/up q [E, I, d/2], s [E, I, d/group]; down q [E, d, I/2],
 * s [E, d, I/group].  y is [T*k, d] in (t, j) order; h [T*k, I] may be NULL.
 */
static int expert_ffn_banks(const uint16_t* x, int64_t T, int64_t d, int64_t I, int64_t E, int64_t k,
                            const wbank* gb, const wbank* ub, const wbank* db, const int32_t* ids, double* y,
                            double* h_out) {
  if (d % 2 || I % 2 || k <= 0 || E <= 0) return ORACLE_EINVAL;
  if (T && (!x || !bank_ok(gb) || !bank_ok(ub) || !bank_ok(db) || !ids || !y)) return ORACLE_EINVAL;
  if (gb->K != d || ub->K != d || db->K != I || gb->rows != I || ub->rows != I || db->rows != d) return ORACLE_EINVAL;
  int64_t R = T * k;
  for (int64_t r = 0; r < R; ++r)
    if (ids[r] < 0 || ids[r] >= E) return ORACLE_EINVAL;
  int bad = 0;
#pragma omp parallel
  {
    double* xv = (double*)malloc(sizeof(double) * (size_t)d);
    double* hv = (double*)malloc(sizeof(double) * (size_t)I);
    if (!xv || !hv) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t r = 0; r < R; ++r) {
        int64_t t = r / k;
        int64_t e = ids[r];
        for (int64_t i = 0; i < d; ++i) xv[i] = oracle_bf16_to_f64(x[t * d + i]);
        for (int64_t n = 0; n < I; ++n) {
          int64_t row = e * I + n;
          double a = bank_row_dot(gb, row, xv);
          double u = bank_row_dot(ub, row, xv);
          hv[n] = a / (1.0 + exp(-a)) * u;
        }
        if (h_out) memcpy(h_out + r * I, hv, sizeof(double) * (size_t)I);
        for (int64_t c = 0; c < d; ++c) y[r * d + c] = bank_row_dot(db, e * d + c, hv);
      }
    }
    free(xv);
    free(hv);
  }
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}

int oracle_expert_ffn(const uint16_t* x, int64_t T, int64_t d, int64_t I, int64_t E, int64_t k, int64_t group,
                      const uint8_t* gq, const uint16_t* gs, const uint8_t* uq, const uint16_t* us,
                      const uint8_t* dq, const uint16_t* ds, const int32_t* ids, double* y, double* h_out) {
  if (group <= 0 || d % group || I % group) return ORACLE_EINVAL;
  wbank gb = int4_bank(gq, gs, I, d, group), ub = int4_bank(uq, us, I, d, group), db = int4_bank(dq, ds, d, I, group);
  return expert_ffn_banks(x, T, d, I, E, k, &gb, &ub, &db, ids, y, h_out);
}

/* The same with NVFP4 banks: gate/up q [E, I, d/2], s [E, I, d/16], ts [E];
 * down q [E, d, I/2], s [E, d, I/16], ts [E]. */
int oracle_expert_ffn_nvfp4(const uint16_t* x, int64_t T, int64_t d, int64_t I, int64_t E, int64_t k,
                            const uint8_t* gq, const uint8_t* gs, const float* gts, const uint8_t* uq,
                            const uint8_t* us, const float* uts, const uint8_t* dq, const uint8_t* ds,
                            const float* dts, const int32_t* ids, double* y, double* h_out) {
  if (d % NVFP4_BLOCK || I % NVFP4_BLOCK) return ORACLE_EINVAL;
  wbank gb = nvfp4_bank(gq, gs, gts, I, d), ub = nvfp4_bank(uq, us, uts, I, d), db = nvfp4_bank(dq, ds, dts, d, I);
  return expert_ffn_banks(x, T, d, I, E, k, &gb, &ub, &db, ids, y, h_out);
}

/* out[t,c] = resid[t,c] + sum_{j=0}^{k-1} w[t,j] * y[t*k+j, c]. */
int oracle_combine(const double* y, const double* w, const uint16_t* resid, int64_t T, int64_t d, int64_t k,
                   double* out) {
  if (T && (!y || !w || !resid || !out)) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j) acc += w[t * k + j] * y[(t * k + j) * d + c];
      out[t * d + c] = oracle_bf16_to_f64(resid[t * d + c]) + acc;
    }
  return ORACLE_OK;
}

/*
 * Whole layer: route (or take forced ids / gates), expert FFNs, combine.
 * With n_shared = 1 the banks hold E + 1 experts and the last one is the
 * shared expert, which every token uses with gate weight 1 besides its k
 * routed experts (the router, Wr [E, d] and b [E], scores only the routed
 * ones): each token then has k + 1 rows, the shared one last
 * ("Flint 40B : Best Mid Sized LLM", transcript 02:35).  k = 0 with
 * n_shared = 1 is a dense SwiGLU layer (the same transcript: the stack opens
 * with two dense layers): no router, every token through bank entry 0.
 * forced_ids / forced_w ([T, k + n_shared]) may be NULL (then both must be
 * NULL).  ids_out, w_out ([T, k + n_shared]), gap_out may be NULL.  out [T, d].
 */
static int moe_forward_banks(const uint16_t* x, const uint16_t* resid, int64_t T, int64_t d, int64_t E, int64_t k,
                             int64_t n_shared, int64_t I, int renorm, const float* Wr, const float* b,
                             const wbank* gb, const wbank* ub, const wbank* db, const int32_t* forced_ids,
                             const double* forced_w, int32_t* ids_out, double* w_out, double* gap_out, double* out) {
  if ((forced_ids == NULL) != (forced_w == NULL)) return ORACLE_EINVAL;
  if (n_shared < 0 || n_shared > 1 || k < 0 || (k == 0 && n_shared == 0)) return ORACLE_EINVAL;
  const int64_t kt = k + n_shared;  // rows per token
  int64_t R = T * kt;
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R + 1));
  double* w = (double*)malloc(sizeof(double) * (size_t)(R + 1));
  double* y = (double*)malloc(sizeof(double) * (size_t)(R * d + 1));
  int32_t* rids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * k + 1));
  double* rw = (double*)malloc(sizeof(double) * (size_t)(T * k + 1));
  int rc = ORACLE_EINVAL;
  if (ids && w && y && rids && rw) {
    if (forced_ids) {
      memcpy(ids, forced_ids, sizeof(int32_t) * (size_t)R);
      memcpy(w, forced_w, sizeof(double) * (size_t)R);
      rc = ORACLE_OK;
      if (gap_out)
        for (int64_t t = 0; t < T; ++t) gap_out[t] = NAN;
    } else {
      if (k > 0) {
        rc = oracle_route(x, T, d, E, k, Wr, b, renorm, rids, rw, NULL, gap_out);
      } else {  // dense layer: nothing to route
        rc = ORACLE_OK;
        if (gap_out)
          for (int64_t t = 0; t < T; ++t) gap_out[t] = INFINITY;
      }
      for (int64_t t = 0; !rc && t < T; ++t) {
        for (int64_t j = 0; j < k; ++j) {
          ids[t * kt + j] = rids[t * k + j];
          w[t * kt + j] = rw[t * k + j];
        }
        if (n_shared) {  // the shared expert: bank entry E, weight 1
          ids[t * kt + k] = (int32_t)E;
          w[t * kt + k] = 1.0;
        }
      }
    }
    if (!rc) rc = expert_ffn_banks(x, T, d, I, E + n_shared, kt, gb, ub, db, ids, y, NULL);
    if (!rc) rc = oracle_combine(y, w, resid, T, d, kt, out);
    if (!rc && ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)R);
    if (!rc && w_out) memcpy(w_out, w, sizeof(double) * (size_t)R);
  }
  free(ids);
  free(w);
  free(y);
  free(rids);
  free(rw);
  return rc;
}

int oracle_moe_forward(const uint16_t* x, const uint16_t* resid, int64_t T, int64_t d, int64_t E, int64_t k,
                       int64_t n_shared, int64_t I, int64_t group, int renorm, const float* Wr, const float* b,
                       const uint8_t* gq, const uint16_t* gs, const uint8_t* uq, const uint16_t* us,
                       const uint8_t* dq, const uint16_t* ds, const int32_t* forced_ids, const double* forced_w,
                       int32_t* ids_out, double* w_out, double* gap_out, double* out) {
  if (group <= 0 || d % group || I % group) return ORACLE_EINVAL;
  wbank gb = int4_bank(gq, gs, I, d, group), ub = int4_bank(uq, us, I, d, group), db = int4_bank(dq, ds, d, I, group);
  return moe_forward_banks(x, resid, T, d, E, k, n_shared, I, renorm, Wr, b, &gb, &ub, &db, forced_ids, forced_w,
                           ids_out, w_out, gap_out, out);
}

/* The same layer with NVFP4 expert banks (tensor scales gts/uts/dts [E + n_shared]). */
int oracle_moe_forward_nvfp4(const uint16_t* x, const uint16_t* resid, int64_t T, int64_t d, int64_t E, int64_t k,
                             int64_t n_shared, int64_t I, int renorm, const float* Wr, const float* b,
                             const uint8_t* gq, const uint8_t* gs, const float* gts, const uint8_t* uq,
                             const uint8_t* us, const float* uts, const uint8_t* dq, const uint8_t* ds,
                             const float* dts, const int32_t* forced_ids, const double* forced_w, int32_t* ids_out,
                             double* w_out, double* gap_out, double* out) {
  if (d % NVFP4_BLOCK || I % NVFP4_BLOCK) return ORACLE_EINVAL;
  wbank gb = nvfp4_bank(gq, gs, gts, I, d), ub = nvfp4_bank(uq, us, uts, I, d), db = nvfp4_bank(dq, ds, dts, d, I);
  return moe_forward_banks(x, resid, T, d, E, k, n_shared, I, renorm, Wr, b, &gb, &ub, &db, forced_ids, forced_w,
                           ids_out, w_out, gap_out, out);
}

/* ------------------------------------------------------------ stack helpers */

/* RMSNorm with unit gain: y[t,i] = x[t,i] / sqrt(mean_i x[t,i]^2 + eps). */
int oracle_rmsnorm(const uint16_t* x, int64_t T, int64_t d, double eps, double* y) {
  if ((T && (!x || !y)) || d <= 0) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t i = 0; i < d; ++i) {
      double v = oracle_bf16_to_f64(x[t * d + i]);
      ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)d + eps);
    for (int64_t i = 0; i < d; ++i) y[t * d + i] = oracle_bf16_to_f64(x[t * d + i]) * r;
  }
  return ORACLE_OK;
}

/*
 * LM head: z[t,v] = sum_i Wlm[v,i] h[t,i] over V rows of a packed int4 bank
 * q [V, d/2], s [V, d/group]; argmax[t] = lowest v reaching max_v z[t,v];
 * gap[t] = top-1 minus top-2 logit.  logits [T, V] and gap may be NULL.
 */
static int lmhead_bank(const uint16_t* h, int64_t T, int64_t d, int64_t V, const wbank* wb, double* logits,
                       int32_t* argmax, double* gap) {
  if (d % 2 || V <= 0 || wb->K != d || (T && (!h || !bank_ok(wb) || !argmax))) return ORACLE_EINVAL;
  double* hv = (double*)malloc(sizeof(double) * (size_t)(T * d + 1));
  double* z = (double*)malloc(sizeof(double) * (size_t)(T * V + 1));
  if (!hv || !z) {
    free(hv);
    free(z);
    return ORACLE_EINVAL;
  }
  for (int64_t i = 0; i < T * d; ++i) hv[i] = oracle_bf16_to_f64(h[i]);
#pragma omp parallel for schedule(static)
  for (int64_t v = 0; v < V; ++v)
    for (int64_t t = 0; t < T; ++t)
      z[t * V + v] = bank_row_dot(wb, v, hv + t * d);
  for (int64_t t = 0; t < T; ++t) {
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
      if (z[t * V + v] > z[t * V + best]) best = v;
    double second = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
      if (v != best && z[t * V + v] > second) second = z[t * V + v];
    argmax[t] = (int32_t)best;
    if (gap) gap[t] = z[t * V + best] - second;
  }
  if (logits) memcpy(logits, z, sizeof(double) * (size_t)(T * V));
  free(hv);
  free(z);
  return ORACLE_OK;
}

int oracle_lmhead(const uint16_t* h, int64_t T, int64_t d, int64_t V, int64_t group, const uint8_t* q,
                  const uint16_t* s, double* logits, int32_t* argmax, double* gap) {
  if (group <= 0 || d % group) return ORACLE_EINVAL;
  wbank wb = int4_bank(q, s, V, d, group);
  return lmhead_bank(h, T, d, V, &wb, logits, argmax, gap);
}

/* The LM head with an NVFP4 matrix: q [V, d/2], s [V, d/16] E4M3, tensor scale ts. */
int oracle_lmhead_nvfp4(const uint16_t* h, int64_t T, int64_t d, int64_t V, const uint8_t* q, const uint8_t* s,
                        float ts, double* logits, int32_t* argmax, double* gap) {
  if (d % NVFP4_BLOCK) return ORACLE_EINVAL;
  wbank wb = nvfp4_bank(q, s, &ts, V, d);
  return lmhead_bank(h, T, d, V, &wb, logits, argmax, gap);
}

int oracle_num_threads(void) {
  int n = 1;
#ifdef _OPENMP
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
#endif
  return n;
}
