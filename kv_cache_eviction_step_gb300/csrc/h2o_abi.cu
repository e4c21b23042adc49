// h2o_abi.cu -- the extern "C" entry points of libh2o.so (declared in include/h2o.h): argument
// validation, the per-device error word, workspace carving and the launches. Every check that can
// fail happens before the first launch, so a rejected call has no effect on the GPU.
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

__device__ int32_t g_error_word;

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// Device address of the error word for the current device (resolved once per device).
int32_t* error_word() {
  thread_local int last_dev = -1;
  thread_local int32_t* last_ptr = nullptr;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return nullptr;
  if (cur == last_dev && last_ptr != nullptr) return last_ptr;
  static std::mutex mu;
  static std::vector<std::pair<int, int32_t*>> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& c : cache)
    if (c.first == dev) {
      last_dev = dev;
      last_ptr = c.second;
      return c.second;
    }
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_error_word);
  if (e != cudaSuccess) {
    t_last_cuda_error = e;
    return nullptr;
  }
  cache.emplace_back(dev, static_cast<int32_t*>(ptr));
  last_dev = dev;
  last_ptr = static_cast<int32_t*>(ptr);
  return last_ptr;
}

int sm_count() {
  thread_local int dev_cached = -1, sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1 << 30;
  if (dev != dev_cached) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1 << 30;
    dev_cached = dev;
  }
  return sms;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned_to(const void* p, int bytes) {
  return (reinterpret_cast<uintptr_t>(p) & static_cast<uintptr_t>(bytes - 1)) == 0;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

h2o_status check_dims(const h2o_dims* d) {
  if (d == nullptr) return H2O_ERR_INVALID_ARG;
  if (d->units_b < 0 || d->heads < 1 || d->budget < 1 || d->k_heavy < 0 || d->k_local < 0)
    return H2O_ERR_INVALID_ARG;
  if (static_cast<int64_t>(d->k_heavy) + d->k_local != d->budget) return H2O_ERR_INVALID_ARG;
  if (d->dtype != H2O_F32 && d->dtype != H2O_BF16) return H2O_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return H2O_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->units_b) * d->heads > INT32_MAX / 16) return H2O_ERR_UNSUPPORTED;
  return H2O_OK;
}

int elem_bytes(const h2o_dims* d) { return d->dtype == H2O_F32 ? 4 : 2; }

h2o_status check_policy(const h2o_policy* pol, int32_t budget) {
  switch (pol->kind) {
    case H2O_POLICY_H2O:
    case H2O_POLICY_LOCAL:
    case H2O_POLICY_TOPK:
      return H2O_OK;
    case H2O_POLICY_SINK_WINDOW:
      return (pol->n_sink >= 0 && pol->n_sink < budget) ? H2O_OK : H2O_ERR_INVALID_ARG;
    case H2O_POLICY_STRIDED:
      return pol->stride >= 1 ? H2O_OK : H2O_ERR_INVALID_ARG;
  }
  return H2O_ERR_INVALID_ARG;
}

h2o_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return H2O_OK;
  t_last_cuda_error = e;
  (void)cudaGetLastError();  // clear the sticky-free launch error so later calls start clean
  return H2O_ERR_CUDA;
}

// Waits on an mbarrier that nothing ever arrives at, with a short limit: exercises the bounded-wait
// path (error word set, clean return) without any copy in flight.
__global__ void wait_timeout_probe_kernel(int32_t* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, err, limit_ns);
}

}  // namespace
}  // namespace h2o

using namespace h2o;

extern "C" {

const char* h2o_last_cuda_error(void) {
  return t_last_cuda_error == cudaSuccess ? "cudaSuccess" : cudaGetErrorName(t_last_cuda_error);
}

const char* h2o_status_string(h2o_status status) {
  switch (status) {
    case H2O_OK: return "ok";
    case H2O_ERR_INVALID_ARG: return "invalid argument";
    case H2O_ERR_UNSUPPORTED: return "unsupported shape";
    case H2O_ERR_CUDA: return "CUDA error";
    case H2O_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

size_t h2o_prefill_workspace_bytes(const h2o_dims* dims, int32_t prompt_len) {
  if (check_dims(dims) != H2O_OK || prompt_len < 1) return 0;
  const size_t units = static_cast<size_t>(dims->units_b) * dims->heads;
  return 3 * round256(units * static_cast<size_t>(prompt_len) * 4);
}

// Per (device, stream), the device memory the last launch of this library on that stream may
// write. A decode kernel may start its cache reads before waiting for the previous grid only if
// that grid writes none of them; with every decode kernel signalling its dependents after its own
// wait, all earlier launches have completed by then (launches that signal nothing let the next one
// start only when they complete). Any other launch of the library (a prefill, the self-test) marks
// all memory as possibly written, so the decode launch after it always waits before its first read.
struct Span {
  uintptr_t lo, hi;
};
struct LastDecode {
  int dev;
  void* stream;
  Span w[9];
};
static std::mutex g_decode_mu;
static std::vector<LastDecode> g_last_decode;

static Span span_of(const void* ptr, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
  return {a, ptr == nullptr ? a : a + bytes};
}

// Records that a launch other than a decode step was enqueued on `stream` of the current device.
static void note_other_launch(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    dev = -1;
  }
  std::lock_guard<std::mutex> lock(g_decode_mu);
  for (auto& l : g_last_decode) {
    if (l.stream != stream || (dev >= 0 && l.dev != dev)) continue;
    for (Span& w : l.w) w = Span{0, ~uintptr_t(0)};
  }
}

static h2o_status prefill_scores_impl(const h2o_dims* dims, int32_t prompt_len, const void* q,
                                      const void* k, float* colsum, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream,
                                      bool last_row_only = false, const void* v = nullptr,
                                      void* out = nullptr) {
  const int units = dims->units_b * dims->heads;
  const size_t arr = round256(static_cast<size_t>(units) * prompt_len * 4);
  PrefillParams p = {};
  p.q = q;
  p.k = k;
  p.row_max = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace));
  p.row_sum = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + arr);
  p.colsum = colsum;
  p.err = error_word();
  if (p.err == nullptr) return from_cuda(cudaGetLastError());
  p.units = units;
  p.P = prompt_len;
  p.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(dims->head_dim)));
  p.last_row_only = last_row_only ? 1 : 0;
  p.v = v;
  p.out = out;
  (void)workspace_bytes;
  note_other_launch(stream);
  // bf16: tcgen05 tensor cores (bf16 x bf16 products are exact in the fp32 accumulator); fp32 stays
  // on the CUDA cores, where the products are not rounded to tf32.
  if (dims->dtype == H2O_BF16) return from_cuda(launch_prefill_scores_tc(p, dims->head_dim, stream));
  return from_cuda(launch_prefill_scores_simt(p, dims->head_dim, dims->dtype, stream));
}

static h2o_status check_prefill(const h2o_dims* dims, int32_t prompt_len, const void* q,
                                const void* k, void* workspace, size_t workspace_bytes) {
  h2o_status st = check_dims(dims);
  if (st != H2O_OK) return st;
  if (prompt_len < 1) return H2O_ERR_INVALID_ARG;
  if (prompt_len > select_max_prompt()) return H2O_ERR_UNSUPPORTED;
  if (dims->units_b == 0) return H2O_OK;
  if (!q || !k || !workspace || !aligned16(q) || !aligned16(k) || !aligned16(workspace))
    return H2O_ERR_INVALID_ARG;
  if (workspace_bytes < h2o_prefill_workspace_bytes(dims, prompt_len)) return H2O_ERR_INVALID_ARG;
  return H2O_OK;
}

h2o_status h2o_prefill_scores(const h2o_dims* dims, int32_t prompt_len, const void* q,
                              const void* k, float* colsum, void* workspace,
                              size_t workspace_bytes, void* stream) {
  h2o_status st = check_prefill(dims, prompt_len, q, k, workspace, workspace_bytes);
  if (st != H2O_OK) return st;
  if (dims->units_b == 0) return H2O_OK;
  if (!colsum || !aligned4(colsum)) return H2O_ERR_INVALID_ARG;
  return prefill_scores_impl(dims, prompt_len, q, k, colsum, workspace, workspace_bytes,
                             static_cast<cudaStream_t>(stream));
}

static h2o_status prefill_select_impl(const h2o_dims* dims, const h2o_policy* policy,
                                      int32_t prompt_len, const void* q, const void* k,
                                      const void* v, void* k_cache, void* v_cache, float* scores,
                                      int32_t* slot_pos, void* workspace, size_t workspace_bytes,
                                      void* stream, void* out = nullptr, float* k_scale = nullptr,
                                      float* v_scale = nullptr) {
  h2o_status st = check_prefill(dims, prompt_len, q, k, workspace, workspace_bytes);
  if (st != H2O_OK) return st;
  const h2o_policy pol = policy ? *policy : h2o_policy{H2O_POLICY_H2O, 0, 1};
  st = check_policy(&pol, dims->budget);
  if (st != H2O_OK) return st;
  if (dims->budget > select_max_budget()) return H2O_ERR_UNSUPPORTED;
  if (dims->units_b == 0) return H2O_OK;
  if (!v || !k_cache || !v_cache || !scores || !slot_pos) return H2O_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(scores) ||
      !aligned4(slot_pos))
    return H2O_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int units = dims->units_b * dims->heads;
  const size_t arr = round256(static_cast<size_t>(units) * prompt_len * 4);
  float* colsum = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + 2 * arr);
  st = prefill_scores_impl(dims, prompt_len, q, k, colsum, workspace, workspace_bytes, s,
                           pol.kind == H2O_POLICY_TOPK, v, out);
  if (st != H2O_OK) return st;
  SelectParams p = {};
  p.colsum = colsum;
  p.k = k;
  p.v = v;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.scores = scores;
  p.slot_pos = slot_pos;
  p.units = units;
  p.P = prompt_len;
  p.budget = dims->budget;
  p.k_heavy = dims->k_heavy;
  p.k_local = dims->k_local;
  p.row_bytes = dims->head_dim * elem_bytes(dims);
  p.key_mode = 0;
  p.stride = 1;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  switch (pol.kind) {
    case H2O_POLICY_LOCAL:  // the last `budget` positions
      p.k_heavy = 0;
      p.k_local = dims->budget;
      break;
    case H2O_POLICY_SINK_WINDOW:  // the first n_sink positions and the last budget - n_sink
      p.k_heavy = pol.n_sink;
      p.k_local = dims->budget - pol.n_sink;
      p.key_mode = 2;
      break;
    case H2O_POLICY_STRIDED:
      p.key_mode = 1;
      p.stride = pol.stride;
      break;
    default:  // H2O ranks by column sums, Top-K by the last row's attention (same array)
      break;
  }
  return from_cuda(launch_select(p, s));
}

h2o_status h2o_prefill_select(const h2o_dims* dims, int32_t prompt_len, const void* q,
                              const void* k, const void* v, void* k_cache, void* v_cache,
                              float* scores, int32_t* slot_pos, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return prefill_select_impl(dims, nullptr, prompt_len, q, k, v, k_cache, v_cache, scores, slot_pos,
                             workspace, workspace_bytes, stream);
}

h2o_status h2o_prefill_select_policy(const h2o_dims* dims, const h2o_policy* policy,
                                     int32_t prompt_len, const void* q, const void* k,
                                     const void* v, void* k_cache, void* v_cache, float* scores,
                                     int32_t* slot_pos, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return prefill_select_impl(dims, policy, prompt_len, q, k, v, k_cache, v_cache, scores, slot_pos,
                             workspace, workspace_bytes, stream);
}

static h2o_status check_e4m3(const h2o_dims* dims, const float* k_scale, const float* v_scale) {
  h2o_status st = check_dims(dims);
  if (st != H2O_OK) return st;
  if (!decode_e4m3_supported(dims->head_dim, dims->dtype, dims->budget)) return H2O_ERR_UNSUPPORTED;
  if (dims->units_b > 0 && (!k_scale || !v_scale || !aligned4(k_scale) || !aligned4(v_scale)))
    return H2O_ERR_INVALID_ARG;
  return H2O_OK;
}

h2o_status h2o_prefill_select_e4m3(const h2o_dims* dims, const h2o_policy* policy,
                                   int32_t prompt_len, const void* q, const void* k, const void* v,
                                   void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                   float* scores, int32_t* slot_pos, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  const h2o_status st = check_e4m3(dims, k_scale, v_scale);
  if (st != H2O_OK) return st;
  return prefill_select_impl(dims, policy, prompt_len, q, k, v, k_cache, v_cache, scores, slot_pos,
                             workspace, workspace_bytes, stream, nullptr, k_scale, v_scale);
}


h2o_status h2o_prefill_forward(const h2o_dims* dims, const h2o_policy* policy, int32_t prompt_len,
                               const void* q, const void* k, const void* v, void* out,
                               void* k_cache, void* v_cache, float* scores, int32_t* slot_pos,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (dims != nullptr && dims->units_b > 0 && (out == nullptr || !aligned16(out))) return H2O_ERR_INVALID_ARG;
  return prefill_select_impl(dims, policy, prompt_len, q, k, v, k_cache, v_cache, scores, slot_pos,
                             workspace, workspace_bytes, stream, out);
}

// The launch of one decode step on the kernel its shape calls for.
static h2o_status dispatch_decode(DecodeParams& p, const h2o_dims* dims, void* stream) {
  // E4M3 caches: the tensor-core kernel over 8-bit tiles (bf16, D = 128, budgets up to 512).
  if (p.k_scale != nullptr) return from_cuda(launch_decode_e4m3(p, static_cast<cudaStream_t>(stream)));
  // Many bf16 units of D = 128 with budgets up to 512 slots: both contractions on tcgen05, persistent
  // over units. Other shapes (fp32, D = 64, caches beyond 8192 slots) use the CUDA-core kernel, each
  // unit split over a CTA cluster when units are few.
  if (decode_tc_supported(dims->head_dim, dims->dtype, dims->budget) && p.units >= 4 * sm_count())
    return from_cuda(launch_decode_tc(p, static_cast<cudaStream_t>(stream)));
  // At least one unit per SM but fewer than four (e.g. one layer's batch x heads per launch), bf16,
  // D = 128, caches of at most 208 slots: one CTA per unit with the unit's K and V resident in shared
  // memory and both contractions on the CUDA cores.
  if (decode_resident_supported(dims->head_dim, dims->dtype, dims->budget) && p.units >= sm_count())
    return from_cuda(launch_decode_resident(p, static_cast<cudaStream_t>(stream)));
  // Fewer bf16 units of D = 128 (or longer caches): the tensor-core step split over a CTA cluster.
  if (decode_tc_split_supported(dims->head_dim, dims->dtype, p.units, p.n))
    return from_cuda(launch_decode_tc_split(p, static_cast<cudaStream_t>(stream)));
  size_t smem = 0;
  if (!plan_decode(p.units, p.n, dims->head_dim, elem_bytes(dims), &p.splits, &p.chunk, &p.stages, &smem,
                   &p.grid))
    return H2O_ERR_UNSUPPORTED;
  return from_cuda(launch_decode(p, dims->head_dim, dims->dtype, static_cast<cudaStream_t>(stream)));
}

static h2o_status decode_step_impl(const h2o_dims* dims, const h2o_policy* policy,
                                   int32_t position, const void* q, const void* k_new,
                                   const void* v_new, void* k_cache, void* v_cache, float* scores,
                                   int32_t* slot_pos, void* out, int32_t* evicted_slot,
                                   int32_t* evicted_pos, void* stream, float* k_scale = nullptr,
                                   float* v_scale = nullptr, const h2o_next_cache* next = nullptr) {
  h2o_status st = check_dims(dims);
  if (st != H2O_OK) return st;
  if (next != nullptr && (next->k_cache == nullptr || next->v_cache == nullptr || next->scores == nullptr ||
                          next->slot_pos == nullptr || !aligned16(next->k_cache) ||
                          !aligned16(next->v_cache) || !aligned4(next->scores) || !aligned4(next->slot_pos)))
    return H2O_ERR_INVALID_ARG;
  const h2o_policy pol = policy ? *policy : h2o_policy{H2O_POLICY_H2O, 0, 1};
  st = check_policy(&pol, dims->budget);
  if (st != H2O_OK) return st;
  if (position < 1) return H2O_ERR_INVALID_ARG;
  if (dims->units_b == 0) return H2O_OK;
  const void* vec_ptrs[] = {q, k_new, v_new, k_cache, v_cache};  // 16-byte vector / bulk loads
  for (const void* ptr : vec_ptrs)
    if (ptr == nullptr || !aligned16(ptr)) return H2O_ERR_INVALID_ARG;
  const void* word_ptrs[] = {scores, slot_pos, evicted_slot, evicted_pos};
  for (const void* ptr : word_ptrs)
    if (ptr == nullptr || !aligned4(ptr)) return H2O_ERR_INVALID_ARG;
  if (out == nullptr || !aligned_to(out, elem_bytes(dims))) return H2O_ERR_INVALID_ARG;
  DecodeParams p = {};
  p.q = q;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.scores = scores;
  p.slot_pos = slot_pos;
  p.out = out;
  p.evicted_slot = evicted_slot;
  p.evicted_pos = evicted_pos;
  p.err = error_word();
  if (p.err == nullptr) return from_cuda(cudaGetLastError());
  p.units = dims->units_b * dims->heads;
  p.budget = dims->budget;
  p.k_local = dims->k_local;
  p.position = position;
  p.n = position < dims->budget ? position : dims->budget;
  p.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(dims->head_dim)));
  p.policy = pol.kind;
  p.n_sink = pol.n_sink;
  p.stride = pol.kind == H2O_POLICY_STRIDED ? pol.stride : 1;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  if (next != nullptr) {
    p.next_k_cache = next->k_cache;
    p.next_v_cache = next->v_cache;
    p.next_scores = next->scores;
    p.next_slot_pos = next->slot_pos;
  }

  // This call's cache arrays (read, and written in place) and its outputs.
  const size_t slots = static_cast<size_t>(p.units) * static_cast<size_t>(dims->budget);
  const size_t row_bytes = static_cast<size_t>(dims->head_dim) * (k_scale != nullptr ? 1 : elem_bytes(dims));
  const size_t units = static_cast<size_t>(p.units);
  LastDecode mine = {0, stream,
                     {span_of(k_cache, slots * row_bytes), span_of(v_cache, slots * row_bytes),
                      span_of(scores, slots * 4), span_of(slot_pos, slots * 4), span_of(k_scale, slots * 4),
                      span_of(v_scale, slots * 4), span_of(out, units * dims->head_dim * elem_bytes(dims)),
                      span_of(evicted_slot, units * 4), span_of(evicted_pos, units * 4)}};
  if (cudaGetDevice(&mine.dev) != cudaSuccess) return from_cuda(cudaGetLastError());
  std::lock_guard<std::mutex> lock(g_decode_mu);
  LastDecode* prev = nullptr;
  for (auto& l : g_last_decode)
    if (l.dev == mine.dev && l.stream == stream) prev = &l;
  p.early = 0;
  if (prev != nullptr) {
    bool disjoint = true;
    for (int i = 0; i < 6; ++i)  // the cache arrays
      for (const Span& w : prev->w)
        if (mine.w[i].lo < w.hi && w.lo < mine.w[i].hi) disjoint = false;
    p.early = disjoint ? 1 : 0;
  }
  const h2o_status st_launch = dispatch_decode(p, dims, stream);
  if (st_launch == H2O_OK) {
    if (prev != nullptr) *prev = mine;
    else g_last_decode.push_back(mine);
  } else if (prev != nullptr) {
    *prev = LastDecode{mine.dev, stream, {}};  // unknown: treat every range as possibly written
    for (Span& w : prev->w) w = Span{0, ~uintptr_t(0)};
  }
  return st_launch;
}

h2o_status h2o_decode_step(const h2o_dims* dims, int32_t position, const void* q,
                           const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           float* scores, int32_t* slot_pos, void* out, int32_t* evicted_slot,
                           int32_t* evicted_pos, void* stream) {
  return decode_step_impl(dims, nullptr, position, q, k_new, v_new, k_cache, v_cache, scores,
                          slot_pos, out, evicted_slot, evicted_pos, stream);
}

h2o_status h2o_decode_step_policy(const h2o_dims* dims, const h2o_policy* policy, int32_t position,
                                  const void* q, const void* k_new, const void* v_new,
                                  void* k_cache, void* v_cache, float* scores, int32_t* slot_pos,
                                  void* out, int32_t* evicted_slot, int32_t* evicted_pos,
                                  void* stream) {
  return decode_step_impl(dims, policy, position, q, k_new, v_new, k_cache, v_cache, scores,
                          slot_pos, out, evicted_slot, evicted_pos, stream);
}

h2o_status h2o_decode_step_prefetch(const h2o_dims* dims, const h2o_policy* policy, int32_t position,
                                    const void* q, const void* k_new, const void* v_new,
                                    void* k_cache, void* v_cache, float* scores, int32_t* slot_pos,
                                    void* out, int32_t* evicted_slot, int32_t* evicted_pos,
                                    const h2o_next_cache* next, void* stream) {
  return decode_step_impl(dims, policy, position, q, k_new, v_new, k_cache, v_cache, scores,
                          slot_pos, out, evicted_slot, evicted_pos, stream, nullptr, nullptr, next);
}

h2o_status h2o_decode_step_e4m3(const h2o_dims* dims, const h2o_policy* policy, int32_t position,
                                const void* q, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, float* k_scale, float* v_scale, float* scores,
                                int32_t* slot_pos, void* out, int32_t* evicted_slot,
                                int32_t* evicted_pos, void* stream) {
  const h2o_status st = check_e4m3(dims, k_scale, v_scale);
  if (st != H2O_OK) return st;
  return decode_step_impl(dims, policy, position, q, k_new, v_new, k_cache, v_cache, scores, slot_pos,
                          out, evicted_slot, evicted_pos, stream, k_scale, v_scale);
}

h2o_status h2o_selftest_wait_timeout(void* stream) {
  int32_t* word = error_word();
  if (word == nullptr) return from_cuda(cudaGetLastError());
  note_other_launch(stream);
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(word, 50000000ull);
  return from_cuda(cudaGetLastError());
}

h2o_status h2o_get_device_error(void* stream, int32_t* code) {
  int32_t* word = error_word();
  if (word == nullptr) return H2O_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess) return H2O_ERR_CUDA;
  if (cudaMemsetAsync(word, 0, sizeof host, s) != cudaSuccess) return H2O_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return H2O_ERR_CUDA;
  if (code) *code = host;
  return host == H2O_DEVERR_NONE ? H2O_OK : H2O_ERR_DEVICE;
}

}  // extern "C"
