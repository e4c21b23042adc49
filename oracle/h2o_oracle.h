/*
 * h2o_oracle.h -- plain CPU oracle of the H2O budgeted KV-cache eviction step.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library. The product path (the CUDA kernels behind include/h2o.h) never calls it
 * and shares no code, header, table or helper with it.
 *
 * All buffers are host memory, row-major and contiguous. "Unit" = one (layer, sequence, head);
 * units are independent. dtype 0 = float32, 1 = bfloat16 (passed as uint16 bit patterns).
 * Every function returns 0 on success and a negative code on invalid arguments (nothing written).
 */
#ifndef H2O_ORACLE_H
#define H2O_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { H2O_ORACLE_F32 = 0, H2O_ORACLE_BF16 = 1, H2O_ORACLE_E4M3 = 2 /* cache rows only */ };

/* How one unit's eviction decision was reached (decode) or its kept set chosen (prefill). */
enum {
  H2O_ORACLE_NO_EVICTION = 0,   /* decode: cache not full; prefill: prompt fits the budget     */
  H2O_ORACLE_RULE = 1,          /* the rule's own choice (no preference, or preference agreed) */
  H2O_ORACLE_NEAR_TIE = 2,      /* preference adopted: within tie_rel of the rule's choice     */
  H2O_ORACLE_ERROR_BOUND = 3,   /* preference adopted: within err_rel (but not tie_rel)        */
  H2O_ORACLE_REJECTED = 4       /* preference not adopted: rule's choice kept                  */
};

/* Eviction policies. H2O is the method; the others are the baselines the pages compare it with,
 * run through the same state: see h2o_oracle.c for the exact rules. */
enum {
  H2O_ORACLE_POLICY_H2O = 0,          /* accumulated attention, k_local recent tokens protected   */
  H2O_ORACLE_POLICY_LOCAL = 1,        /* sliding window: the oldest cached position goes          */
  H2O_ORACLE_POLICY_SINK_WINDOW = 2,  /* the first n_sink positions never go, else the oldest     */
  H2O_ORACLE_POLICY_TOPK = 3,         /* like H2O but ranked by the current step's attention only */
  H2O_ORACLE_POLICY_STRIDED = 4       /* off-grid positions (pos % stride != 0) go first, oldest  */
};

typedef struct {
  int32_t kind;
  int32_t n_sink;   /* sink + window: 0 <= n_sink < budget */
  int32_t stride;   /* strided: >= 1 */
} h2o_oracle_policy;

typedef struct {
  int32_t kind;          /* one of the enum above                                              */
  int32_t rule_victim;   /* slot the rule picks (-1 if the cache was not full)                 */
  int32_t victim;        /* slot actually overwritten after eviction (-1 if none)              */
  int32_t evicted_pos;   /* position evicted (-1 if none)                                      */
  int32_t written_slot;  /* slot that received the new token                                   */
  int32_t n_candidates;  /* slots eligible for eviction                                        */
  double gap_rel;        /* (2nd lowest - lowest) / max(|.|) over candidate scores; inf if < 2 */
} h2o_oracle_step_info;

typedef struct {
  int32_t kind;          /* one of the enum above                                              */
  int32_t kept;          /* number of slots filled                                             */
  double gap_rel;        /* relative gap between the last kept and first dropped column sum    */
} h2o_oracle_prefill_info;

/*
 * Prefill score pass + selection for `units` independent units.
 *   q, k, v     [units, P, D]        prompt queries / keys / values
 *   k_cache,
 *   v_cache     [units, budget, D]   written: kept rows in ascending position, zero rows after
 *   scores      [units, budget]      written: float32(column sum) of kept tokens, 0 after
 *   slot_pos    [units, budget]      written: kept positions ascending, -1 after
 *   colsum      [units, P] or NULL   written: the float64 column sums c_j
 *   prefer_pos  [units, budget] or NULL: another implementation's slot_pos; adopted where its kept
 *               set differs from the rule's only by near-tied column sums (see h2o_oracle.c)
 *   infos       [units] or NULL
 */
int h2o_oracle_prefill_select(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                              int32_t k_local, int32_t dtype, int32_t P, const void* q,
                              const void* k, const void* v, void* k_cache, void* v_cache,
                              float* scores, int32_t* slot_pos, double* colsum,
                              const int32_t* prefer_pos, double tie_rel, double err_rel,
                              h2o_oracle_prefill_info* infos);

/*
 * One decode step at absolute position t (t >= 1) for `units` independent units; the caches hold
 * n = min(t, budget) valid slots in 0..n-1 and -1 positions after.
 *   q, k_new, v_new  [units, D]
 *   out              [units, D] float64 attention output
 *   probs            [units, budget + 1] or NULL: float64 softmax weights of slots 0..n-1, then the
 *                    new token at index n (entries past n untouched)
 *   evicted_slot,
 *   evicted_pos      [units] or NULL: victim slot / its old position, -1 when nothing was evicted
 *   prefer_victim    [units] or NULL: another implementation's victim, adopted on near-ties
 *   infos            [units] or NULL
 */
int h2o_oracle_decode_step(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                           int32_t k_local, int32_t dtype, int32_t t, const void* q,
                           const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           float* scores, int32_t* slot_pos, double* out, double* probs,
                           int32_t* evicted_slot, int32_t* evicted_pos,
                           const int32_t* prefer_victim, double tie_rel, double err_rel,
                           h2o_oracle_step_info* infos);

/* The same two operations under another eviction policy (NULL = H2O). Prefill: Local keeps the last
 * `budget` prompt positions; sink + window the first n_sink and the last budget - n_sink; Top-K the
 * last k_local plus the k_heavy older positions the last prompt token attends to most, its scores
 * starting from that attention; strided the last k_local plus the k_heavy newest older positions
 * on its grid (then off-grid ones). Decode: Top-K replaces each score by the step's weight instead
 * of adding it; Local, sink + window and strided evict by position (see h2o_oracle.c). */
int h2o_oracle_prefill_select_policy(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                     int32_t k_local, int32_t dtype, int32_t P, const void* q,
                                     const void* k, const void* v, void* k_cache, void* v_cache,
                                     float* scores, int32_t* slot_pos, double* colsum,
                                     const h2o_oracle_policy* policy, const int32_t* prefer_pos,
                                     double tie_rel, double err_rel, h2o_oracle_prefill_info* infos);
int h2o_oracle_decode_step_policy(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                  int32_t k_local, int32_t dtype, int32_t t, const void* q,
                                  const void* k_new, const void* v_new, void* k_cache,
                                  void* v_cache, float* scores, int32_t* slot_pos, double* out,
                                  double* probs, int32_t* evicted_slot, int32_t* evicted_pos,
                                  const h2o_oracle_policy* policy, const int32_t* prefer_victim,
                                  double tie_rel, double err_rel, h2o_oracle_step_info* infos);

/*
 * The same two operations with a quantised cache: q, k, v, k_new, v_new in bf16, cached rows as
 * FP8 E4M3 codes (k_cache, v_cache: [units, budget, D] bytes) with one float32 scale per row
 * (k_scale, v_scale: [units, budget]); see h2o_oracle.c for the quantisation. Attention reads the
 * cached rows as scale x value(code); the new token attends with its bf16 values and is stored
 * quantised. Everything else as the policy forms above. Returns -8 without scale arrays.
 */
int h2o_oracle_prefill_select_e4m3(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                   int32_t k_local, int32_t P, const void* q, const void* k,
                                   const void* v, uint8_t* k_cache, uint8_t* v_cache,
                                   float* k_scale, float* v_scale, float* scores,
                                   int32_t* slot_pos, double* colsum,
                                   const h2o_oracle_policy* policy, const int32_t* prefer_pos,
                                   double tie_rel, double err_rel, h2o_oracle_prefill_info* infos);
int h2o_oracle_decode_step_e4m3(int32_t units, int32_t D, int32_t budget, int32_t k_heavy,
                                int32_t k_local, int32_t t, const void* q, const void* k_new,
                                const void* v_new, uint8_t* k_cache, uint8_t* v_cache,
                                float* k_scale, float* v_scale, float* scores, int32_t* slot_pos,
                                double* out, double* probs, int32_t* evicted_slot,
                                int32_t* evicted_pos, const h2o_oracle_policy* policy,
                                const int32_t* prefer_victim, double tie_rel, double err_rel,
                                h2o_oracle_step_info* infos);
/* E4M3 code of a float32 (to nearest, ties to even, saturating) and the value of a code; exported
 * for the format pins. */
uint8_t h2o_oracle_e4m3_code(float f);
double h2o_oracle_e4m3_value(uint8_t code);

/*
 * Prompt pass of the attention layer: out[u][i] = sum over j <= i of softmax_j(q_i . k_j / sqrt(D))
 * v_j, the causal attention output of every prompt row, whose weights the prefill's column sums add
 * up. Inputs [units, P, D] in `dtype`; out [units, P, D] float64. Returns 0, or < 0 on bad sizes.
 */
int h2o_oracle_prefill_attention(int32_t units, int32_t D, int32_t dtype, int32_t P, const void* q,
                                 const void* k, const void* v, double* out);

/*
 * Convenience driver for timing: one unit's whole job, i.e. h2o_oracle_prefill_select on its prompt
 * followed by `steps` calls of h2o_oracle_decode_step at positions P, P+1, ... It adds no arithmetic.
 *   q, k, v                [P, D]         the unit's prompt
 *   q_dec, k_dec, v_dec    step s's row at offset s * dec_stride elements
 *   k_cache, v_cache       [budget, D];  scores, slot_pos [budget]   the unit's state (written)
 *   out                    [steps, D] float64 or NULL
 */
int h2o_oracle_run_unit(int32_t D, int32_t budget, int32_t k_heavy, int32_t k_local, int32_t dtype,
                        int32_t P, int32_t steps, const void* q, const void* k, const void* v,
                        const void* q_dec, const void* k_dec, const void* v_dec, int64_t dec_stride,
                        void* k_cache, void* v_cache, float* scores, int32_t* slot_pos,
                        double* out);

#ifdef __cplusplus
}
#endif

#endif /* H2O_ORACLE_H */
