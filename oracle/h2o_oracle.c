/*
 * h2o_oracle.c -- plain, slow CPU oracle of the H2O budgeted KV-cache eviction step.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library. The product path never calls it; it shares no code with the CUDA path.
 *
 * What it restates (web pages on H2O, "Heavy-Hitter Oracle"; Zhang et al., NeurIPS 2023):
 *   [post]   the ttsmallhot.github.io H2O summary post:
 *            §2.1.1  attention weights are Softmax(QK^T / sqrt(d)) (the paper drops sqrt(d) for
 *                    brevity; the post states it, and so does this oracle);
 *            §2.1.2  a token's accumulated attention score = the sum of the attention it receives;
 *            §2.2    budget k split into k_local recent tokens and k_heavy heavy hitters; after each
 *                    new token its attention to every cached token is added to that token's running
 *                    score; when the cache is full the recent tokens are kept and the cached token
 *                    with the lowest accumulated score among the rest is evicted;
 *            §2.3    the new token's K/V is written into the evicted slot (no compaction).
 *   [note]   "H2O Heavy-Hitter Oracle 分析" (liuhc.cn):
 *            §3.1    scores are kept per head; heavy hitters = top-k of the cumulative attention
 *                    (argsort of the negated sums);
 *            §3.2    victim = argmin(score); the new token is always admitted.
 *
 * Readings where the pages leave a step open (each also listed in the design notes):
 *   - scale: logits are (q . k) / sqrt(D), in float64;
 *   - attended set of step t: the n = min(t, budget) cached slots plus the new token itself; the new
 *     token's own weight becomes its initial score (prefill column sums include the diagonal too);
 *   - order: scores are accumulated first, then the victim is chosen on the updated scores;
 *   - protection: after step t the positions t-k_local+1 .. t must be resident, so cached slots with
 *     position <= t - k_local are the eviction candidates (k_local <= 1 leaves every cached slot a
 *     candidate, which is the unprotected argmin of [note] §3.2; k_heavy = 0 is a sliding window);
 *   - ties: the lowest score is evicted, equal scores evict the lowest position; prefill keeps the
 *     top k_heavy column sums ranked (sum desc, position desc), i.e. the same order read backwards;
 *   - prefill selection = column sums of the full causal prompt softmax, then one top-k ([note] §3.1),
 *     with the last k_local prompt positions always kept; kept tokens fill slots 0.. in ascending
 *     position, unused slots get position -1, score 0 and zero K/V rows;
 *   - precision: float64 for dot products, softmax and column sums; the score table is float32 and
 *     each step adds float32(p) to it with one float32 addition (the storage the method keeps).
 *
 * Near ties. Another implementation computing in float32 may order two nearly equal scores the other
 * way. When the caller passes that implementation's choice ("prefer"), the oracle adopts it only if it
 * is a valid choice whose score is within tie_rel (reported as NEAR_TIE) or err_rel (ERROR_BOUND) of
 * the rule's choice, relative to the larger magnitude; an exact tie is always decided by position.
 * The adoption changes which slot is overwritten, never any arithmetic.
 */
#include "h2o_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- element access: exact widening of the stored values ---------------------------------- */

static size_t elem_bytes(int32_t dtype) { return dtype == H2O_ORACLE_F32 ? 4 : 2; }

static double elem(const void* base, int32_t dtype, size_t i) {
  if (dtype == H2O_ORACLE_F32) return (double)((const float*)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* (q . k_row) in float64, d = 0 .. D-1 in order. */
static double dot(const double* q, const void* rows, int32_t dtype, size_t row, int32_t D) {
  double acc = 0.0;
  for (int32_t d = 0; d < D; ++d) acc += q[d] * elem(rows, dtype, row * (size_t)D + (size_t)d);
  return acc;
}

/* ---- FP8 E4M3 cache rows -------------------------------------------------------------------
 * The OCP 8-bit floating-point format E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * no infinities; exponent 15 with mantissa 7 is NaN; the largest finite magnitude is 448. A cached
 * row of the quantised cache is D such codes and one float32 scale: scale = amax / 448 (amax = the
 * largest magnitude in the row; an all-zero row gets scale 1), code_d = E4M3(x_d / scale), each
 * float32 operation rounded once, the conversion to nearest with ties to even and saturating at
 * +-448. The cached value is scale * value(code). */

static double e4m3_value(uint8_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);        /* subnormal: (m / 8) x 2^-6 */
  else v = ldexp(8.0 + m, e - 10);              /* (1 + m / 8) x 2^(e - 7) */
  return (b & 0x80) ? -v : v;
}

static uint8_t e4m3_code(float f) {
  if (isnan(f)) return 0x7F;
  const uint8_t sign = signbit(f) ? 0x80 : 0x00;
  const double a = fabs((double)f);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);                                /* a in [2^(e2-1), 2^e2) */
  int binade = e2 - 1;
  if (binade < -6) binade = -6;                 /* the subnormal spacing continues below 2^-6 */
  const double quantum = ldexp(1.0, binade - 3);
  double r = nearbyint(a / quantum) * quantum;  /* to nearest, ties to even */
  if (r > 448.0) r = 448.0;                     /* saturate */
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
  frexp(r, &e2);
  const int e = e2 - 1;                         /* r in [2^e, 2^(e+1)) */
  const int m = (int)(r / ldexp(1.0, e - 3)) - 8;
  return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)m);
}

uint8_t h2o_oracle_e4m3_code(float f) { return e4m3_code(f); }
double h2o_oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }

/* One row of the quantised cache from D input values (float32 or bf16). Returns the scale. */
static float e4m3_quantise_row(const void* src, int32_t dtype, size_t row, int32_t D, uint8_t* codes) {
  float amax = 0.0f;
  for (int32_t d = 0; d < D; ++d) {
    const float x = fabsf((float)elem(src, dtype, row * (size_t)D + (size_t)d));
    if (x > amax) amax = x;
  }
  const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int32_t d = 0; d < D; ++d)
    codes[d] = e4m3_code((float)elem(src, dtype, row * (size_t)D + (size_t)d) / scale);
  return scale;
}

/* The cache of one unit: rows stored as the input dtype, or as E4M3 codes with per-row scales. */
typedef struct {
  int32_t fmt;       /* H2O_ORACLE_F32, H2O_ORACLE_BF16 or H2O_ORACLE_E4M3 */
  char* rows;        /* [budget][D] elements of fmt */
  float* scales;     /* E4M3: [budget] */
  int32_t D;
} cache_rows;

static size_t cache_row_bytes(int32_t fmt, int32_t D) {
  return (size_t)D * (fmt == H2O_ORACLE_E4M3 ? 1 : elem_bytes(fmt));
}

static double cached(const cache_rows* c, size_t j, int32_t d) {
  if (c->fmt == H2O_ORACLE_E4M3)
    return (double)c->scales[j] * e4m3_value((uint8_t)c->rows[j * (size_t)c->D + (size_t)d]);
  return elem(c->rows, c->fmt, j * (size_t)c->D + (size_t)d);
}

/* Write input row `src_row` of `src` (dtype) into cache slot j. */
static void store_row(cache_rows* c, size_t j, const void* src, int32_t dtype, size_t src_row) {
  if (c->fmt == H2O_ORACLE_E4M3) {
    c->scales[j] = e4m3_quantise_row(src, dtype, src_row, c->D, (uint8_t*)c->rows + j * (size_t)c->D);
    return;
  }
  const size_t row = cache_row_bytes(c->fmt, c->D);
  memcpy(c->rows + j * row, (const char*)src + src_row * row, row);
}

static void clear_row(cache_rows* c, size_t j) {
  memset(c->rows + j * cache_row_bytes(c->fmt, c->D), 0, cache_row_bytes(c->fmt, c->D));
  if (c->fmt == H2O_ORACLE_E4M3) c->scales[j] = 0.0f;
}

static int check_dims(int32_t units, int32_t D, int32_t budget, int32_t k_heavy, int32_t k_local,
                      int32_t dtype) {
  if (units < 0 || D < 1 || budget < 1 || k_heavy < 0 || k_local < 0) return -1;
  if (k_heavy + k_local != budget) return -2;
  if (dtype != H2O_ORACLE_F32 && dtype != H2O_ORACLE_BF16) return -3;
  return 0;
}

static double rel_gap(double lo, double hi) {
  double scale = fmax(fabs(lo), fabs(hi));
  if (scale == 0.0) return 0.0;
  return (hi - lo) / scale;
}

/* ---- prefill: column sums of the causal softmax, then the heavy-hitter selection ----------- */

typedef struct {
  double c;
  int32_t pos;
} ranked;

/* Rank for keeping: larger column sum first; on equal sums the later position first (so that the
 * dropped side is "lowest score, then lowest position", the decode eviction order). */
static int keep_order(const void* a, const void* b) {
  const ranked* x = (const ranked*)a;
  const ranked* y = (const ranked*)b;
  if (x->c > y->c) return -1;
  if (x->c < y->c) return 1;
  return (x->pos > y->pos) ? -1 : (x->pos < y->pos) ? 1 : 0;
}

/* c_j = sum over rows i >= j of softmax_i(j), softmax over the causal row i: j' = 0..i. If
 * last_row is given it receives softmax_{P-1}(j), the last prompt query's attention. */
static void causal_column_sums(int32_t D, int32_t dtype, int32_t P, const void* q, const void* k,
                               double scale, double* c, double* qrow, double* s, double* last_row) {
  for (int32_t j = 0; j < P; ++j) c[j] = 0.0;
  for (int32_t i = 0; i < P; ++i) {
    for (int32_t d = 0; d < D; ++d) qrow[d] = elem(q, dtype, (size_t)i * D + d);
    double m = -INFINITY;
    for (int32_t j = 0; j <= i; ++j) {
      s[j] = dot(qrow, k, dtype, (size_t)j, D) * scale;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int32_t j = 0; j <= i; ++j) l += exp(s[j] - m);
    for (int32_t j = 0; j <= i; ++j) c[j] += exp(s[j] - m) / l;
    if (last_row && i == P - 1)
      for (int32_t j = 0; j <= i; ++j) last_row[j] = exp(s[j] - m) / l;
  }
}

/* ---- policies ------------------------------------------------------------------------------ */

static int check_policy(const h2o_oracle_policy* pol, int32_t budget) {
  switch (pol->kind) {
    case H2O_ORACLE_POLICY_H2O:
    case H2O_ORACLE_POLICY_LOCAL:
    case H2O_ORACLE_POLICY_TOPK:
      return 0;
    case H2O_ORACLE_POLICY_SINK_WINDOW:
      return (pol->n_sink >= 0 && pol->n_sink < budget) ? 0 : -7;
    case H2O_ORACLE_POLICY_STRIDED:
      return pol->stride >= 1 ? 0 : -7;
  }
  return -7;
}

/* Policies that decide by position alone (no near ties to adopt). */
static int by_position(const h2o_oracle_policy* pol) {
  return pol->kind == H2O_ORACLE_POLICY_LOCAL || pol->kind == H2O_ORACLE_POLICY_SINK_WINDOW ||
         pol->kind == H2O_ORACLE_POLICY_STRIDED;
}

/* Eviction order of the position rules: smaller goes first. Local and sink + window evict the
 * oldest position; strided evicts positions off its grid (pos mod stride != 0) oldest first, and
 * grid positions only when no other candidate is left. */
static int64_t position_rank(const h2o_oracle_policy* pol, int32_t pos) {
  if (pol->kind == H2O_ORACLE_POLICY_STRIDED && pos % pol->stride == 0) return (int64_t)1 << 40 | pos;
  return pos;
}

/* Whether a cached position may be evicted at step t. */
static int eviction_candidate(const h2o_oracle_policy* pol, int32_t pos, int32_t t, int32_t k_local) {
  switch (pol->kind) {
    case H2O_ORACLE_POLICY_LOCAL: return 1;
    case H2O_ORACLE_POLICY_SINK_WINDOW: return pos >= pol->n_sink;
    default: return (int64_t)pos <= (int64_t)t - k_local;
  }
}

/* Decide whether a preferred kept set (slot_pos layout) may replace the rule's. */
static int32_t assess_prefill_preference(int32_t budget, int32_t k_local, int32_t P,
                                        const double* c, const unsigned char* keep_rule,
                                        const int32_t* prefer, double tie_rel, double err_rel,
                                        unsigned char* keep_pref) {
  memset(keep_pref, 0, (size_t)P);
  for (int32_t s = 0; s < budget; ++s) {
    int32_t p = prefer[s];
    if (p < 0 || p >= P || keep_pref[p]) return H2O_ORACLE_REJECTED;
    keep_pref[p] = 1;
  }
  for (int32_t p = P - k_local; p < P; ++p)
    if (!keep_pref[p]) return H2O_ORACLE_REJECTED;
  double max_dropped_by_pref = -INFINITY, min_added_by_pref = INFINITY;
  int differs = 0;
  for (int32_t p = 0; p < P - k_local; ++p) {
    if (keep_rule[p] && !keep_pref[p]) { differs = 1; if (c[p] > max_dropped_by_pref) max_dropped_by_pref = c[p]; }
    if (!keep_rule[p] && keep_pref[p]) { differs = 1; if (c[p] < min_added_by_pref) min_added_by_pref = c[p]; }
  }
  if (!differs) return H2O_ORACLE_RULE;
  if (max_dropped_by_pref == min_added_by_pref) return H2O_ORACLE_REJECTED; /* exact tie: by position */
  double g = rel_gap(min_added_by_pref, max_dropped_by_pref);
  if (g <= tie_rel) return H2O_ORACLE_NEAR_TIE;
  if (g <= err_rel) return H2O_ORACLE_ERROR_BOUND;
  return H2O_ORACLE_REJECTED;
}

int h2o_oracle_prefill_select(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                              int32_t k_local, int32_t dtype, int32_t P, const void* q,
                              const void* k, const void* v, void* k_cache, void* v_cache,
                              float* scores, int32_t* slot_pos, double* colsum,
                              const int32_t* prefer_pos, double tie_rel, double err_rel,
                              h2o_oracle_prefill_info* infos) {
  return h2o_oracle_prefill_select_policy(units, D, budget, k_heavy, k_local, dtype, P, q, k, v,
                                          k_cache, v_cache, scores, slot_pos, colsum, NULL,
                                          prefer_pos, tie_rel, err_rel, infos);
}

static int prefill_select(int32_t units, int32_t D, int32_t budget, int32_t k_heavy, int32_t k_local,
                          int32_t dtype, int32_t cache_fmt, int32_t P, const void* q, const void* k,
                          const void* v, void* k_cache, void* v_cache, float* k_scale,
                          float* v_scale, float* scores, int32_t* slot_pos, double* colsum,
                          const h2o_oracle_policy* policy, const int32_t* prefer_pos,
                          double tie_rel, double err_rel, h2o_oracle_prefill_info* infos) {
  const h2o_oracle_policy h2o_rule = {H2O_ORACLE_POLICY_H2O, 0, 0};
  const h2o_oracle_policy* pol = policy ? policy : &h2o_rule;
  int rc = check_dims(units, D, budget, k_heavy, k_local, dtype);
  if (rc) return rc;
  if (P < 1) return -4;
  rc = check_policy(pol, budget);
  if (rc) return rc;
  const size_t eb = elem_bytes(dtype);
  const size_t row = (size_t)D * eb;
  const double scale = 1.0 / sqrt((double)D);

  double* c = (double*)malloc(sizeof(double) * (size_t)P);
  double* a = (double*)malloc(sizeof(double) * (size_t)P);  /* last prompt row's attention */
  double* s = (double*)malloc(sizeof(double) * (size_t)P);
  double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
  ranked* cand = (ranked*)malloc(sizeof(ranked) * (size_t)P);
  unsigned char* keep = (unsigned char*)malloc((size_t)P);
  unsigned char* keep_pref = (unsigned char*)malloc((size_t)P);
  if (!c || !a || !s || !qrow || !cand || !keep || !keep_pref) {
    free(c); free(a); free(s); free(qrow); free(cand); free(keep); free(keep_pref);
    return -9;
  }

  for (int32_t u = 0; u < units; ++u) {
    const char* qu = (const char*)q + (size_t)u * P * row;
    const char* ku = (const char*)k + (size_t)u * P * row;
    const char* vu = (const char*)v + (size_t)u * P * row;
    const size_t crow = cache_row_bytes(cache_fmt, D);
    cache_rows kc = {cache_fmt, (char*)k_cache + (size_t)u * budget * crow,
                     k_scale ? k_scale + (size_t)u * budget : NULL, D};
    cache_rows vc = {cache_fmt, (char*)v_cache + (size_t)u * budget * crow,
                     v_scale ? v_scale + (size_t)u * budget : NULL, D};
    float* sc = scores + (size_t)u * budget;
    int32_t* sp = slot_pos + (size_t)u * budget;
    h2o_oracle_prefill_info info = {H2O_ORACLE_NO_EVICTION, 0, INFINITY};

    causal_column_sums(D, dtype, P, qu, ku, scale, c, qrow, s, a);
    if (colsum) memcpy(colsum + (size_t)u * P, c, sizeof(double) * (size_t)P);
    /* The value a kept token starts from: its accumulated attention over the prompt, or for
     * Top-K the attention the current (last) prompt token gives it. */
    const double* start = pol->kind == H2O_ORACLE_POLICY_TOPK ? a : c;

    /* Which prompt positions stay. */
    if (P <= budget) {
      memset(keep, 1, (size_t)P);
    } else if (pol->kind == H2O_ORACLE_POLICY_LOCAL || pol->kind == H2O_ORACLE_POLICY_SINK_WINDOW) {
      /* The most recent positions, plus the first n_sink ones for sink + window. */
      const int32_t sinks = pol->kind == H2O_ORACLE_POLICY_SINK_WINDOW ? pol->n_sink : 0;
      memset(keep, 0, (size_t)P);
      for (int32_t p = 0; p < sinks; ++p) keep[p] = 1;
      for (int32_t p = P - (budget - sinks); p < P; ++p) keep[p] = 1;
      info.kind = H2O_ORACLE_RULE;
      if (prefer_pos) {
        const int32_t* pp = prefer_pos + (size_t)u * budget;
        for (int32_t sl = 0; sl < budget; ++sl)
          if (pp[sl] < 0 || pp[sl] >= P || !keep[pp[sl]]) info.kind = H2O_ORACLE_REJECTED;
      }
    } else {
      memset(keep, 0, (size_t)P);
      for (int32_t p = P - k_local; p < P; ++p) keep[p] = 1;     /* the k_local most recent */
      int32_t nc = P - k_local;                                 /* older positions compete */
      /* Ranked by the start value (H2O, Top-K) or, for strided, grid membership. */
      for (int32_t p = 0; p < nc; ++p) {
        cand[p].c = pol->kind == H2O_ORACLE_POLICY_STRIDED ? (double)(p % pol->stride == 0) : start[p];
        cand[p].pos = p;
      }
      qsort(cand, (size_t)nc, sizeof(ranked), keep_order);
      for (int32_t r = 0; r < k_heavy; ++r) keep[cand[r].pos] = 1;
      info.kind = H2O_ORACLE_RULE;
      if (k_heavy > 0 && k_heavy < nc) info.gap_rel = rel_gap(cand[k_heavy].c, cand[k_heavy - 1].c);
      if (prefer_pos) {
        int32_t kind = assess_prefill_preference(budget, k_local, P, c, keep,
                                                prefer_pos + (size_t)u * budget, tie_rel, err_rel,
                                                keep_pref);
        if (pol->kind != H2O_ORACLE_POLICY_H2O) {
          /* Same assessment on the values this policy ranks by. */
          double* vals = s;  /* row scratch is free here */
          for (int32_t p = 0; p < P; ++p)
            vals[p] = pol->kind == H2O_ORACLE_POLICY_STRIDED ? (double)(p % pol->stride == 0) : a[p];
          kind = assess_prefill_preference(budget, k_local, P, vals, keep,
                                          prefer_pos + (size_t)u * budget, tie_rel, err_rel, keep_pref);
          if (by_position(pol) && kind != H2O_ORACLE_RULE) kind = H2O_ORACLE_REJECTED;
        }
        info.kind = kind;
        if (kind == H2O_ORACLE_NEAR_TIE || kind == H2O_ORACLE_ERROR_BOUND)
          memcpy(keep, keep_pref, (size_t)P);
      }
    }

    /* Kept tokens fill slots in ascending position; the rest of the slots are empty. */
    int32_t slot = 0;
    for (int32_t p = 0; p < P; ++p) {
      if (!keep[p]) continue;
      store_row(&kc, (size_t)slot, ku, dtype, (size_t)p);
      store_row(&vc, (size_t)slot, vu, dtype, (size_t)p);
      sc[slot] = (float)start[p];
      sp[slot] = p;
      ++slot;
    }
    info.kept = slot;
    for (; slot < budget; ++slot) {
      clear_row(&kc, (size_t)slot);
      clear_row(&vc, (size_t)slot);
      sc[slot] = 0.0f;
      sp[slot] = -1;
    }
    if (infos) infos[u] = info;
  }
  free(c); free(a); free(s); free(qrow); free(cand); free(keep); free(keep_pref);
  return 0;
}

int h2o_oracle_prefill_select_policy(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                     int32_t k_local, int32_t dtype, int32_t P, const void* q,
                                     const void* k, const void* v, void* k_cache, void* v_cache,
                                     float* scores, int32_t* slot_pos, double* colsum,
                                     const h2o_oracle_policy* policy, const int32_t* prefer_pos,
                                     double tie_rel, double err_rel, h2o_oracle_prefill_info* infos) {
  return prefill_select(units, D, budget, k_heavy, k_local, dtype, dtype, P, q, k, v, k_cache, v_cache,
                        NULL, NULL, scores, slot_pos, colsum, policy, prefer_pos, tie_rel, err_rel,
                        infos);
}

int h2o_oracle_prefill_select_e4m3(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                   int32_t k_local, int32_t P, const void* q, const void* k,
                                   const void* v, uint8_t* k_cache, uint8_t* v_cache,
                                   float* k_scale, float* v_scale, float* scores,
                                   int32_t* slot_pos, double* colsum,
                                   const h2o_oracle_policy* policy, const int32_t* prefer_pos,
                                   double tie_rel, double err_rel, h2o_oracle_prefill_info* infos) {
  if (!k_scale || !v_scale) return -8;
  return prefill_select(units, D, budget, k_heavy, k_local, H2O_ORACLE_BF16, H2O_ORACLE_E4M3, P, q, k, v,
                        k_cache, v_cache, k_scale, v_scale, scores, slot_pos, colsum, policy,
                        prefer_pos, tie_rel, err_rel, infos);
}

/* ---- decode: attend, accumulate, evict, overwrite in place --------------------------------- */

int h2o_oracle_decode_step(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                           int32_t k_local, int32_t dtype, int32_t t, const void* q,
                           const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           float* scores, int32_t* slot_pos, double* out, double* probs,
                           int32_t* evicted_slot, int32_t* evicted_pos,
                           const int32_t* prefer_victim, double tie_rel, double err_rel,
                           h2o_oracle_step_info* infos) {
  return h2o_oracle_decode_step_policy(units, D, budget, k_heavy, k_local, dtype, t, q, k_new, v_new,
                                       k_cache, v_cache, scores, slot_pos, out, probs, evicted_slot,
                                       evicted_pos, NULL, prefer_victim, tie_rel, err_rel, infos);
}

static int decode_step(int32_t units, int32_t D, int32_t budget, int32_t k_heavy, int32_t k_local,
                       int32_t dtype, int32_t cache_fmt, int32_t t, const void* q, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache, float* k_scale,
                       float* v_scale, float* scores, int32_t* slot_pos, double* out, double* probs,
                       int32_t* evicted_slot, int32_t* evicted_pos, const h2o_oracle_policy* policy,
                       const int32_t* prefer_victim, double tie_rel, double err_rel,
                       h2o_oracle_step_info* infos) {
  const h2o_oracle_policy h2o_rule = {H2O_ORACLE_POLICY_H2O, 0, 0};
  const h2o_oracle_policy* pol = policy ? policy : &h2o_rule;
  int rc = check_dims(units, D, budget, k_heavy, k_local, dtype);
  if (rc) return rc;
  if (t < 1) return -4;
  rc = check_policy(pol, budget);
  if (rc) return rc;
  const int32_t n = t < budget ? t : budget;   /* valid cached slots before this step */
  const size_t crow = cache_row_bytes(cache_fmt, D);
  const double scale = 1.0 / sqrt((double)D);

  /* Every unit's slot map must hold exactly n valid, distinct-looking entries. */
  for (int32_t u = 0; u < units; ++u) {
    const int32_t* sp = slot_pos + (size_t)u * budget;
    for (int32_t j = 0; j < budget; ++j) {
      if (j < n && (sp[j] < 0 || sp[j] >= t)) return -5;
      if (j >= n && sp[j] != -1) return -5;
    }
  }

  double* qv = (double*)malloc(sizeof(double) * (size_t)D);
  double* s = (double*)malloc(sizeof(double) * ((size_t)n + 1));
  double* p = (double*)malloc(sizeof(double) * ((size_t)n + 1));
  if (!qv || !s || !p) { free(qv); free(s); free(p); return -9; }

  for (int32_t u = 0; u < units; ++u) {
    const size_t ub = (size_t)u * budget;
    cache_rows kc = {cache_fmt, (char*)k_cache + ub * crow, k_scale ? k_scale + ub : NULL, D};
    cache_rows vc = {cache_fmt, (char*)v_cache + ub * crow, v_scale ? v_scale + ub : NULL, D};
    float* sc = scores + ub;
    int32_t* sp = slot_pos + ub;
    h2o_oracle_step_info info = {H2O_ORACLE_NO_EVICTION, -1, -1, -1, -1, 0, INFINITY};

    /* Logits over the n cached slots and the new token (index n): [post] §2.1.1. */
    for (int32_t d = 0; d < D; ++d) qv[d] = elem(q, dtype, (size_t)u * D + d);
    for (int32_t j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int32_t d = 0; d < D; ++d) acc += qv[d] * cached(&kc, (size_t)j, d);
      s[j] = acc * scale;
    }
    s[n] = dot(qv, k_new, dtype, (size_t)u, D) * scale;

    double m = -INFINITY;
    for (int32_t j = 0; j <= n; ++j) if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int32_t j = 0; j <= n; ++j) l += exp(s[j] - m);
    for (int32_t j = 0; j <= n; ++j) p[j] = exp(s[j] - m) / l;
    if (probs) memcpy(probs + (size_t)u * (budget + 1), p, sizeof(double) * ((size_t)n + 1));

    /* Output o = sum_j p_j v_j over the same n + 1 keys. */
    for (int32_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int32_t j = 0; j < n; ++j) acc += p[j] * cached(&vc, (size_t)j, d);
      acc += p[n] * elem(v_new, dtype, (size_t)u * D + d);
      out[(size_t)u * D + d] = acc;
    }

    /* Local statistic: every cached token's score grows by the attention it just received
     * ([post] §2.2, [note] §3.2), as one float32 addition of the float32 weight. */
    for (int32_t j = 0; j < n; ++j) {
      float add = (float)p[j];
      if (pol->kind == H2O_ORACLE_POLICY_TOPK) {
        sc[j] = add;  /* Top-K ranks by the current step's attention only */
        continue;
      }
      sc[j] = sc[j] + add;
    }

    int32_t target;
    if (n < budget) {
      target = n;                                           /* free slot: no eviction */
    } else {
      /* Greedy eviction: the recent tokens are protected; among the rest the lowest updated
       * score goes, equal scores evict the lowest position ([post] §2.2, [note] §3.2). */
      const int64_t last_candidate = (int64_t)t - k_local;
      int32_t best = -1, second = -1;
      if (!by_position(pol)) {
        for (int32_t j = 0; j < n; ++j) {
          if ((int64_t)sp[j] > last_candidate) continue;
          ++info.n_candidates;
          if (best < 0 || sc[j] < sc[best] || (sc[j] == sc[best] && sp[j] < sp[best])) {
            second = best;
            best = j;
          } else if (second < 0 || sc[j] < sc[second] || (sc[j] == sc[second] && sp[j] < sp[second])) {
            second = j;
          }
        }
      } else {
        /* Position rules (Local, sink + window, strided): the first eligible slot in their
         * eviction order goes; positions are distinct, so there are no ties. */
        for (int32_t j = 0; j < n; ++j) {
          if (!eviction_candidate(pol, sp[j], t, k_local)) continue;
          ++info.n_candidates;
          if (best < 0 || position_rank(pol, sp[j]) < position_rank(pol, sp[best])) best = j;
        }
      }
      if (best < 0) { free(qv); free(s); free(p); return -6; }  /* impossible when kl <= budget */
      info.rule_victim = best;
      if (second >= 0) info.gap_rel = rel_gap((double)sc[best], (double)sc[second]);
      info.kind = H2O_ORACLE_RULE;
      target = best;
      if (prefer_victim && prefer_victim[u] != best && by_position(pol)) {
        info.kind = H2O_ORACLE_REJECTED;  /* decided by position: nothing to adopt */
      } else if (prefer_victim && prefer_victim[u] != best) {
        int32_t w = prefer_victim[u];
        info.kind = H2O_ORACLE_REJECTED;
        if (w >= 0 && w < n && (int64_t)sp[w] <= last_candidate && sc[w] != sc[best]) {
          double g = rel_gap((double)sc[best], (double)sc[w]);
          if (g <= tie_rel) info.kind = H2O_ORACLE_NEAR_TIE;
          else if (g <= err_rel) info.kind = H2O_ORACLE_ERROR_BOUND;
          if (info.kind != H2O_ORACLE_REJECTED) target = w;
        }
      }
      info.victim = target;
      info.evicted_pos = sp[target];
    }

    /* In-place overwrite, no compaction ([post] §2.3): the new token takes the slot, starting
     * from its own attention weight as score. */
    store_row(&kc, (size_t)target, k_new, dtype, (size_t)u);
    store_row(&vc, (size_t)target, v_new, dtype, (size_t)u);
    sc[target] = (float)p[n];
    sp[target] = t;
    info.written_slot = target;

    if (evicted_slot) evicted_slot[u] = info.victim;
    if (evicted_pos) evicted_pos[u] = info.evicted_pos;
    if (infos) infos[u] = info;
  }
  free(qv); free(s); free(p);
  return 0;
}

int h2o_oracle_decode_step_policy(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                  int32_t k_local, int32_t dtype, int32_t t, const void* q,
                                  const void* k_new, const void* v_new, void* k_cache,
                                  void* v_cache, float* scores, int32_t* slot_pos, double* out,
                                  double* probs, int32_t* evicted_slot, int32_t* evicted_pos,
                                  const h2o_oracle_policy* policy, const int32_t* prefer_victim,
                                  double tie_rel, double err_rel, h2o_oracle_step_info* infos) {
  return decode_step(units, D, budget, k_heavy, k_local, dtype, dtype, t, q, k_new, v_new, k_cache,
                     v_cache, NULL, NULL, scores, slot_pos, out, probs, evicted_slot, evicted_pos,
                     policy, prefer_victim, tie_rel, err_rel, infos);
}

int h2o_oracle_decode_step_e4m3(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                int32_t k_local, int32_t t, const void* q, const void* k_new,
                                const void* v_new, uint8_t* k_cache, uint8_t* v_cache,
                                float* k_scale, float* v_scale, float* scores, int32_t* slot_pos,
                                double* out, double* probs, int32_t* evicted_slot,
                                int32_t* evicted_pos, const h2o_oracle_policy* policy,
                                const int32_t* prefer_victim, double tie_rel, double err_rel,
                                h2o_oracle_step_info* infos) {
  if (!k_scale || !v_scale) return -8;
  return decode_step(units, D, budget, k_heavy, k_local, H2O_ORACLE_BF16, H2O_ORACLE_E4M3, t, q, k_new,
                     v_new, k_cache, v_cache, k_scale, v_scale, scores, slot_pos, out, probs,
                     evicted_slot, evicted_pos, policy, prefer_victim, tie_rel, err_rel, infos);
}

/* Causal attention output of the prompt ([post] §2.1.1: the weights are Softmax(QK^T / sqrt(d)) over
 * the keys a row may see, here j <= i). Each row: float64 logits, their maximum, the exponentials and
 * their sum, then the weighted sum of the value rows in position order. */
int h2o_oracle_prefill_attention(int32_t units, int32_t D, int32_t dtype, int32_t P, const void* q,
                                 const void* k, const void* v, double* out) {
  if (units < 0 || D < 1 || P < 1) return -1;
  if (dtype != H2O_ORACLE_F32 && dtype != H2O_ORACLE_BF16) return -3;
  const double scale = 1.0 / sqrt((double)D);
  const size_t eb = elem_bytes(dtype);
  double* qrow = malloc(sizeof(double) * (size_t)D);
  double* w = malloc(sizeof(double) * (size_t)P);
  if (!qrow || !w) {
    free(qrow);
    free(w);
    return -4;
  }
  for (int32_t u = 0; u < units; ++u) {
    const size_t base = (size_t)u * P * D;
    const void* qu = (const char*)q + base * eb;
    const void* ku = (const char*)k + base * eb;
    const void* vu = (const char*)v + base * eb;
    for (int32_t i = 0; i < P; ++i) {
      for (int32_t d = 0; d < D; ++d) qrow[d] = elem(qu, dtype, (size_t)i * D + d);
      double m = -INFINITY;
      for (int32_t j = 0; j <= i; ++j) {
        w[j] = dot(qrow, ku, dtype, (size_t)j, D) * scale;
        if (w[j] > m) m = w[j];
      }
      double l = 0.0;
      for (int32_t j = 0; j <= i; ++j) {
        w[j] = exp(w[j] - m);
        l += w[j];
      }
      double* o = out + base + (size_t)i * D;
      for (int32_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int32_t j = 0; j <= i; ++j) acc += w[j] / l * elem(vu, dtype, (size_t)j * D + d);
        o[d] = acc;
      }
    }
  }
  free(qrow);
  free(w);
  return 0;
}

/* ---- timing driver: one unit's prefill and decode steps back to back ----------------------- */

int h2o_oracle_run_unit(int32_t D, int32_t budget, int32_t k_heavy, int32_t k_local, int32_t dtype,
                        int32_t P, int32_t steps, const void* q, const void* k, const void* v,
                        const void* q_dec, const void* k_dec, const void* v_dec, int64_t dec_stride,
                        void* k_cache, void* v_cache, float* scores, int32_t* slot_pos,
                        double* out) {
  int rc = h2o_oracle_prefill_select(1, D, budget, k_heavy, k_local, dtype, P, q, k, v, k_cache,
                                     v_cache, scores, slot_pos, NULL, NULL, 0.0, 0.0, NULL);
  if (rc) return rc;
  const size_t eb = elem_bytes(dtype);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)D);
  if (!tmp) return -9;
  for (int32_t s = 0; s < steps && rc == 0; ++s) {
    const size_t off = (size_t)s * (size_t)dec_stride * eb;
    rc = h2o_oracle_decode_step(1, D, budget, k_heavy, k_local, dtype, P + s,
                                (const char*)q_dec + off, (const char*)k_dec + off,
                                (const char*)v_dec + off, k_cache, v_cache, scores, slot_pos,
                                out ? out + (size_t)s * D : tmp, NULL, NULL, NULL, NULL, 0.0, 0.0,
                                NULL);
  }
  free(tmp);
  return rc;
}
