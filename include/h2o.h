/*
 * h2o.h -- C ABI of libh2o.so, the GB300 (sm_103a) hot path of H2O ("Heavy-Hitter Oracle")
 * budgeted KV-cache eviction.
 *
 * The method (web pages on H2O, Zhang et al., NeurIPS 2023):
 *   - ttsmallhot.github.io H2O post, §2.1.1: attention weights are Softmax(QK^T / sqrt(d));
 *     §2.1.2: a token's accumulated attention score is the attention it has received;
 *     §2.2: the KV budget k is split into k_local recent tokens and k_heavy heavy hitters; after each
 *     new token its attention to every cached token is added to that token's score; when the cache is
 *     full the recent tokens are kept and the lowest-scoring other token is evicted;
 *     §2.3: the new token's K/V overwrites the evicted slot in place (no compaction);
 *   - "H2O Heavy-Hitter Oracle 分析" (liuhc.cn), §3.1: per-head cumulative attention, heavy hitters
 *     are its top-k; §3.2: victim = argmin(score), the new token is always admitted.
 *
 * Terms. A "unit" is one (layer, sequence, head); units are independent. dims.units_b counts
 * (layer, sequence) rows, so there are units_b * heads units, laid out [units_b][heads].
 * D = head_dim. Positions are absolute token indices (0-based); every unit has the same prompt
 * length and the same current position (fixed-length padded prompts, as in the post's §3.2.2).
 *
 * Readings of the pages used throughout (the pages leave these open):
 *   - logits are (q . k) / sqrt(D);
 *   - step t attends the n = min(t, budget) cached slots plus the new token; the new token's own
 *     weight is its initial score;
 *   - scores are accumulated first, then the victim is chosen among cached slots whose position is
 *     <= t - k_local (so positions t-k_local+1 .. t stay resident); the lowest updated score goes,
 *     equal scores evict the lowest position;
 *   - prefill keeps the last k_local prompt positions plus the k_heavy largest causal column sums of
 *     Softmax(QK^T/sqrt(D)) among the rest (equal sums keep the later position); kept tokens fill
 *     slots 0.. in ascending position, unused slots get position -1, score 0 and zero K/V rows.
 *
 * Memory. Every pointer argument is DEVICE memory owned by the caller, row-major and contiguous.
 * q, k, v, k_new, v_new, k_cache, v_cache and the workspace must be 16-byte aligned (they are read
 * with 16-byte vector and bulk copies; every row of D = 64 or 128 elements keeps that alignment);
 * scores, slot_pos, evicted_* and colsum 4-byte aligned; out aligned to its element. Element type
 * of q/k/v/out/caches is
 * dims.dtype (H2O_F32: float, H2O_BF16: bfloat16); scores are float32; positions and indices are
 * int32. The library allocates nothing per call; it keeps one 4-byte device error word per device,
 * created on first use.
 *
 * Streams and errors. `stream` is a cudaStream_t (NULL = the legacy default stream); every call only
 * enqueues work on it and returns without synchronising. Argument errors return
 * H2O_ERR_INVALID_ARG or H2O_ERR_UNSUPPORTED before anything is launched; a failed launch returns
 * H2O_ERR_CUDA. Conditions detected on the device (a bounded wait that ran out) are recorded in the
 * device error word and reported by h2o_get_device_error. No C++ exception crosses this ABI.
 * Calls that overlap on the GPU and touch the same cache race; order them on one stream.
 *
 * Decode steps are launched with programmatic dependent launch: a step may start while the kernel
 * before it on the stream finishes, and waits for it before reading anything that kernel may write.
 * When the library's previous launch on the same stream was a decode step that wrote none of this
 * call's cache arrays (one launch per layer: consecutive launches belong to different layers), the
 * step may load its cached K/V rows before that wait. Any other launch of the library on the stream
 * (a prefill call, the self-test) cancels this for the next decode step, which then waits before
 * its first read. Precondition for the early case: a kernel of the caller's that sits between two
 * decode calls on the stream and itself signals programmatic completion early must not write the
 * second call's cache (ordinary kernels, which do not signal early, are always safe).
 */
#ifndef H2O_H
#define H2O_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define H2O_API __attribute__((visibility("default")))
#else
#define H2O_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  H2O_OK = 0,
  H2O_ERR_INVALID_ARG = 1,  /* bad pointer, alignment, size or budget split                 */
  H2O_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement (e.g. D = 96)    */
  H2O_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed                          */
  H2O_ERR_DEVICE = 4        /* the device error word was set (see h2o_get_device_error)      */
} h2o_status;

typedef enum { H2O_F32 = 0, H2O_BF16 = 1 } h2o_dtype;

typedef struct {
  int32_t units_b;   /* layers * batch: (layer, sequence) rows; 0 makes every call a no-op     */
  int32_t heads;     /* heads per row, >= 1                                                   */
  int32_t head_dim;  /* D: 64 or 128                                                          */
  int32_t budget;    /* k: cached slots per unit, >= 1                                        */
  int32_t k_heavy;   /* heavy-hitter share of the budget, >= 0                                */
  int32_t k_local;   /* recent-token share, >= 0; k_heavy + k_local == budget                 */
  int32_t dtype;     /* h2o_dtype of q/k/v/out and the K/V caches                             */
} h2o_dims;

/* Eviction policies. H2O is the method; the others are the baselines the pages compare it with
 * (the ttsmallhot.github.io post's §3.1.1 "Local" and "Top-K", StreamingLLM's attention sinks named
 * in its §4, and a fixed-stride rule after its "Strided" sparse-attention baseline), run through the
 * same cache state so they can be compared under the same budget. */
typedef enum {
  H2O_POLICY_H2O = 0,          /* lowest accumulated score among positions <= t - k_local           */
  H2O_POLICY_LOCAL = 1,        /* the oldest cached position (sliding window of `budget` tokens)     */
  H2O_POLICY_SINK_WINDOW = 2,  /* the oldest position >= n_sink: the first n_sink positions stay     */
  H2O_POLICY_TOPK = 3,         /* like H2O, but each score is replaced by the step's weight instead
                                  of accumulated; the prefill ranks by the last prompt token's
                                  attention and seeds the scores with it                            */
  H2O_POLICY_STRIDED = 4       /* among positions <= t - k_local, the oldest with pos % stride != 0,
                                  else the oldest on the grid; the prefill keeps the newest grid
                                  positions among the older ones                                     */
} h2o_policy_kind;

typedef struct {
  int32_t kind;    /* h2o_policy_kind                                          */
  int32_t n_sink;  /* H2O_POLICY_SINK_WINDOW: 0 <= n_sink < budget; else 0     */
  int32_t stride;  /* H2O_POLICY_STRIDED: >= 1; else ignored                   */
} h2o_policy;

/* Device error word values. */
#define H2O_DEVERR_NONE 0
#define H2O_DEVERR_WAIT_TIMEOUT 1   /* a bounded wait on a copy or a peer block gave up       */
#define H2O_DEVERR_NO_CANDIDATE 2   /* no eviction candidate (cannot happen with valid state) */

/* Bytes of device workspace h2o_prefill_scores / h2o_prefill_select need for this shape:
 * three float32 arrays [units, prompt_len] (row max, row normaliser, column sums), each rounded
 * up to 256 bytes. Returns 0 for invalid dims. */
H2O_API size_t h2o_prefill_workspace_bytes(const h2o_dims* dims, int32_t prompt_len);

/*
 * Prefill score pass (the rows P1-P2 of the hot path): for every unit, the causal column sums
 *   colsum[j] = sum_{i >= j} softmax_i(j),  softmax_i over j' <= i of (q_i . k_j') / sqrt(D),
 * written as float32 [units, prompt_len] into `colsum` (device). Source: the post's §2.1.2 and §2.2
 * (accumulated attention) and "H2O Heavy-Hitter Oracle 分析" §3.1 (cum_attn per head).
 *   q, k        [units, prompt_len, D]  prompt queries and keys (device)
 *   workspace   >= h2o_prefill_workspace_bytes(dims, prompt_len) bytes of device memory; its
 *               contents on entry are ignored and on return are scratch
 * 1 <= prompt_len <= 16384.
 */
H2O_API h2o_status h2o_prefill_scores(const h2o_dims* dims, int32_t prompt_len, const void* q,
                              const void* k, float* colsum, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Prefill score pass + selection + gather (rows P1-P4): computes the column sums as
 * h2o_prefill_scores does, keeps min(prompt_len, budget) prompt tokens per unit (the last k_local
 * positions plus the k_heavy largest column sums among the older ones) and fills the caches:
 *   k_cache, v_cache   [units, budget, D]  kept K/V rows in ascending position, zero rows after
 *   scores             [units, budget]     float32 column sum of each kept token, 0 after
 *   slot_pos           [units, budget]     kept positions, ascending, -1 after
 * Afterwards the caches are ready for h2o_decode_step at position = prompt_len.
 * On return the workspace's column-sum array (offset 2 * round_up(4 * units * prompt_len, 256))
 * holds the float32 column sums.
 */
H2O_API h2o_status h2o_prefill_select(const h2o_dims* dims, int32_t prompt_len, const void* q,
                              const void* k, const void* v, void* k_cache, void* v_cache,
                              float* scores, int32_t* slot_pos, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Size of the device array h2o_prefill_select_static uses as its scratch (16 MiB). */
#define H2O_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * h2o_prefill_select without a workspace argument, for callers that cannot allocate device memory
 * (for example a serving engine that reserved all device memory for its own pool at start-up, or a
 * plugin running inside a host framework that owns the allocator and hands it only the tensors it
 * declared). The H2O pages have no counterpart: this is a deployment convenience. The scratch lives
 * in one device array of H2O_STATIC_SCRATCH_BYTES inside this library, which a GPU holds from the
 * moment the library's device code is loaded on it (see below) until the process exits; nothing is
 * allocated or freed by the call.
 *   - Same arguments, results and errors as h2o_prefill_select, minus the workspace.
 *   - Limit: h2o_prefill_workspace_bytes(dims, prompt_len) <= H2O_STATIC_SCRATCH_BYTES, i.e.
 *     units * prompt_len <= 1,398,080 (e.g. 2048 units with 512-token prompts); larger calls return
 *     H2O_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *     that device current); make that first call before any stream capture.
 *   - When its memory is taken: the array sits in the library's device code, which the CUDA runtime
 *     loads into a device's memory when that code is first needed there. Under the default lazy
 *     module loading that is the first h2o_prefill_select_static call on the device (the address
 *     lookup loads it), not the moment the library is loaded. A caller that is about to reserve
 *     all device memory for its own pool should therefore make one call (any valid shape) before
 *     reserving, or run with CUDA_MODULE_LOADING=EAGER so the array is placed when the CUDA context
 *     is created; otherwise that first call can fail with H2O_ERR_CUDA (out of memory, see
 *     h2o_last_cuda_error).
 *   - Every call on a device shares the one array, which keeps the last call's contents (no array
 *     has to start at zero: each is fully written before it is read). Calls that overlap on the
 *     GPU, on different streams or from different threads, race on it: order them on one stream.
 */
H2O_API h2o_status h2o_prefill_select_static(const h2o_dims* dims, int32_t prompt_len,
                                             const void* q, const void* k, const void* v,
                                             void* k_cache, void* v_cache, float* scores,
                                             int32_t* slot_pos, void* stream);

/*
 * One budgeted decode step (rows D1-D7) at absolute position `position` (>= 1) for every unit,
 * fused into one kernel launch. With n = min(position, budget) valid cached slots 0..n-1:
 *   D2-D4  attends q over the n cached keys plus k_new:  out = softmax(q.K^T/sqrt(D)) V  [units, D]
 *   D5     scores[j] += p_j (float32) for every cached slot j
 *   D6     if n == budget: victim = argmin over slots with slot_pos <= position - k_local of
 *          (updated score, position); evicted_slot = victim, evicted_pos = its old position;
 *          otherwise no eviction: evicted_slot = evicted_pos = -1 and the new token goes to slot n
 *   D7     the chosen slot gets K = k_new, V = v_new, score = p_new, slot_pos = position, in place
 *   q, k_new, v_new    [units, D]
 *   k_cache, v_cache   [units, budget, D]   read and updated in place
 *   scores, slot_pos   [units, budget]      read and updated in place
 *   out                [units, D]           written (dtype of q)
 *   evicted_slot,
 *   evicted_pos        [units] int32        written
 * The cache state must be the one left by h2o_prefill_select (prompt_len <= position) and the
 * previous decode steps, called with consecutive positions.
 */
H2O_API h2o_status h2o_decode_step(const h2o_dims* dims, int32_t position, const void* q,
                           const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           float* scores, int32_t* slot_pos, void* out, int32_t* evicted_slot,
                           int32_t* evicted_pos, void* stream);

/*
 * h2o_prefill_select and h2o_decode_step under another eviction policy (policy == NULL means
 * H2O_POLICY_H2O, i.e. the plain entry points). Same buffers, layouts and errors; an invalid policy
 * (unknown kind, n_sink outside [0, budget), stride < 1) returns H2O_ERR_INVALID_ARG. Prefill
 * selection per policy (prompt longer than the budget): Local keeps the last `budget` positions;
 * sink + window the first n_sink and the last budget - n_sink; Top-K the last k_local plus the
 * k_heavy older positions the last prompt token attends to most, with scores starting from that
 * attention (the workspace's column-sum array then holds it); strided the last k_local plus the
 * k_heavy newest older positions on its grid (then off it). A cache must be decoded under the policy
 * it was prefilled with.
 */
H2O_API h2o_status h2o_prefill_select_policy(const h2o_dims* dims, const h2o_policy* policy,
                                             int32_t prompt_len, const void* q, const void* k,
                                             const void* v, void* k_cache, void* v_cache,
                                             float* scores, int32_t* slot_pos, void* workspace,
                                             size_t workspace_bytes, void* stream);
H2O_API h2o_status h2o_decode_step_policy(const h2o_dims* dims, const h2o_policy* policy,
                                          int32_t position, const void* q, const void* k_new,
                                          const void* v_new, void* k_cache, void* v_cache,
                                          float* scores, int32_t* slot_pos, void* out,
                                          int32_t* evicted_slot, int32_t* evicted_pos, void* stream);

/*
 * The cache arrays of the decode call that will follow this one on the same stream: same dims and
 * layouts as this call's k_cache, v_cache, scores and slot_pos (e.g. the next layer's cache when a
 * model launches the step once per layer). All four non-NULL, k_cache and v_cache 16-byte aligned.
 */
typedef struct {
  const void* k_cache;
  const void* v_cache;
  const float* scores;
  const int32_t* slot_pos;
} h2o_next_cache;

/*
 * h2o_decode_step_policy with a hint: while this step runs, the kernel asks L2 for `next`'s rows
 * (prefetch only; nothing of `next` is read into a result or written), so that the next call's
 * cache reads hit L2 instead of waiting for HBM. The step's results are identical with and without
 * the hint, and next == NULL is the plain call. Honoured by the kernels that run one CTA per unit
 * (few units per SM, bf16, D = 128: one layer's batch x heads per launch); ignored by the others.
 * next's arrays must be device memory of the stated shape (an invalid address is undefined
 * behaviour, as for every pointer here); H2O_ERR_INVALID_ARG for a NULL or misaligned member.
 */
H2O_API h2o_status h2o_decode_step_prefetch(const h2o_dims* dims, const h2o_policy* policy,
                                            int32_t position, const void* q, const void* k_new,
                                            const void* v_new, void* k_cache, void* v_cache,
                                            float* scores, int32_t* slot_pos, void* out,
                                            int32_t* evicted_slot, int32_t* evicted_pos,
                                            const h2o_next_cache* next, void* stream);

/*
 * The same two operations over a quantised cache (the H2O post §3.3 discusses combining H2O with
 * KV-cache quantisation): q, k, v, k_new, v_new and out stay as dims->dtype, which must be
 * H2O_BF16 with head_dim 128 and budget <= 512 (else H2O_ERR_UNSUPPORTED); the caches hold FP8
 * E4M3 codes (OCP 8-bit float: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
 * finite 448) with one float32 scale per cached row:
 *   k_cache, v_cache  [units, budget, 128] uint8, device, 16-byte aligned
 *   k_scale, v_scale  [units, budget] float32, device, 4-byte aligned
 * A row x is stored as scale = amax(|x|) / 448 (1 for an all-zero row) and codes E4M3(x_d / scale),
 * each float32 operation rounded once, the conversion to nearest with ties to even, saturating;
 * attention reads scale * value(code). The new token attends with its bf16 values and is then stored
 * quantised into its slot; empty slots hold zero codes and scale 0. Everything else (selection,
 * scores, eviction, policies, errors) as h2o_prefill_select_policy / h2o_decode_step_policy. The
 * logits and the output run on the tensor cores straight from the 8-bit tiles: the query is split
 * exactly into two E4M3 rows after a power-of-two rescale, the weights into three (about 12
 * significant bits).
 */
H2O_API h2o_status h2o_prefill_select_e4m3(const h2o_dims* dims, const h2o_policy* policy,
                                           int32_t prompt_len, const void* q, const void* k,
                                           const void* v, void* k_cache, void* v_cache,
                                           float* k_scale, float* v_scale, float* scores,
                                           int32_t* slot_pos, void* workspace,
                                           size_t workspace_bytes, void* stream);
H2O_API h2o_status h2o_decode_step_e4m3(const h2o_dims* dims, const h2o_policy* policy,
                                        int32_t position, const void* q, const void* k_new,
                                        const void* v_new, void* k_cache, void* v_cache,
                                        float* k_scale, float* v_scale, float* scores,
                                        int32_t* slot_pos, void* out, int32_t* evicted_slot,
                                        int32_t* evicted_pos, void* stream);

/*
 * Prefill forward of one attention layer with the budgeted cache built in the same pass
 * (H2O post §2.1.1: the prompt's attention weights are Softmax(QK^T/sqrt(d)); their column sums are
 * the scores h2o_prefill_select keeps by). Everything h2o_prefill_select_policy does, plus
 *   out  [units, prompt_len, head_dim] dtype, device, caller-owned, 16-byte aligned: row i receives
 *        the causal attention output sum_{j<=i} softmax_j(q_i . k_j / sqrt(D)) v_j of prompt row i.
 * The bf16 path computes the probabilities in float32, rounds them to bf16 for the P V product
 * (float32 accumulation) and the result to bf16; float32 stays in float32. The output shares the
 * logits and exponentials of the row-statistics pass. NULL out: H2O_ERR_INVALID_ARG.
 */
H2O_API h2o_status h2o_prefill_forward(const h2o_dims* dims, const h2o_policy* policy,
                                       int32_t prompt_len, const void* q, const void* k,
                                       const void* v, void* out, void* k_cache, void* v_cache,
                                       float* scores, int32_t* slot_pos, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, reads the current device's error word into *code (if code != NULL) and
 * clears it. Returns H2O_OK when the word was H2O_DEVERR_NONE, H2O_ERR_DEVICE when it was set, and
 * H2O_ERR_CUDA if the synchronisation or copy failed.
 */
H2O_API h2o_status h2o_get_device_error(void* stream, int32_t* code);

/*
 * Self-test of the device-side bounded wait: launches one block that waits on a shared-memory
 * barrier nothing ever completes, with a 50 ms limit. The wait gives up, sets the device error word
 * to H2O_DEVERR_WAIT_TIMEOUT and the kernel returns normally; a following h2o_get_device_error
 * reports it (and clears it). Nothing else is touched. Returns H2O_ERR_CUDA if the launch fails.
 */
H2O_API h2o_status h2o_selftest_wait_timeout(void* stream);

/* Name of the CUDA error (e.g. "cudaErrorInvalidValue") behind the most recent H2O_ERR_CUDA
 * returned on the calling thread; "cudaSuccess" if there was none. Static string. */
H2O_API const char* h2o_last_cuda_error(void);

/* Static, human-readable name of a status. */
H2O_API const char* h2o_status_string(h2o_status status);

#ifdef __cplusplus
}
#endif

#endif /* H2O_H */
