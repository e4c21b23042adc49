// h2o_internal.cuh -- shared internals of libh2o.so: launch-parameter structs, launcher
// declarations and the small PTX helpers (mbarrier, bulk async copy, bounded waits) the sm_103a
// kernels use. Not part of the public ABI (include/h2o.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/h2o.h"

namespace h2o {

// ---- launch parameters --------------------------------------------------------------------

struct DecodeParams {
  const void* q;        // [units, D]
  const void* k_new;    // [units, D]
  const void* v_new;    // [units, D]
  void* k_cache;        // [units, budget, D]
  void* v_cache;        // [units, budget, D]
  float* scores;        // [units, budget]
  int32_t* slot_pos;    // [units, budget]
  void* out;            // [units, D]
  int32_t* evicted_slot;  // [units]
  int32_t* evicted_pos;   // [units]
  int32_t* err;         // device error word
  int32_t units;
  int32_t budget;
  int32_t k_local;
  int32_t position;     // t
  int32_t n;            // min(t, budget) valid cached slots
  int32_t splits;       // CTAs (one cluster) per unit
  int32_t chunk;        // cached slots per CTA
  int32_t stages;       // ring depth in tiles
  int32_t grid;         // CTAs launched
  float scale;          // 1/sqrt(D)
  int32_t policy;       // h2o_policy_kind
  int32_t n_sink;       // sink + window
  int32_t stride;       // strided
  float* k_scale;       // E4M3 caches: [units, budget] per-row scales
  float* v_scale;
  int32_t early;        // the previous decode launch on this stream wrote none of this call's cache
                        // arrays: their reads may start before griddepcontrol.wait
  const void* next_k_cache;      // the next decode call's cache arrays on this stream (same shape),
  const void* next_v_cache;      // for an L2 prefetch while this step runs; null: no hint
  const float* next_scores;
  const int32_t* next_slot_pos;
};

struct PrefillParams {
  const void* q;        // [units, P, D]
  const void* k;        // [units, P, D]
  float* row_max;       // [units, P]
  float* row_sum;       // [units, P]
  float* colsum;        // [units, P]
  int32_t* err;
  int32_t units;
  int32_t P;
  float scale;
  int32_t last_row_only;  // column-sum pass: write the last prompt row's attention instead
  const void* v;          // [units, P, D], with `out`
  void* out;              // [units, P, D] prompt attention output, or nullptr
};

struct SelectParams {
  const float* colsum;  // [units, P]
  const void* k;        // [units, P, D]
  const void* v;        // [units, P, D]
  void* k_cache;        // [units, budget, D]
  void* v_cache;
  float* scores;        // [units, budget]
  int32_t* slot_pos;    // [units, budget]
  int32_t units;
  int32_t P;
  int32_t budget;
  int32_t k_heavy;      // older positions kept by key (policy-adjusted)
  int32_t k_local;      // most recent positions kept (policy-adjusted)
  int32_t row_bytes;    // D * element size
  int32_t key_mode;     // 0: by colsum value, 1: stride grid, 2: lowest positions
  int32_t stride;
  float* k_scale;       // non-null: the caches hold E4M3 codes (D = 128, bf16 inputs) with
  float* v_scale;       // these per-row scales [units, budget]
};

// ---- launchers (host) ---------------------------------------------------------------------

// Launch `kernel(*params)` with programmatic stream serialization allowed (the kernel calls
// pdl_launch_dependents / pdl_wait), so consecutive decode steps overlap launch and prologue.
template <typename Params>
inline cudaError_t launch_pdl(const void* kernel, int grid, int threads, int smem, cudaStream_t stream,
                              Params* params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {params};
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

// Grid of the persistent decode kernels (bf16 and E4M3), whose CTAs take units
// u = blockIdx.x + k gridDim.x. A launch ends with its most loaded CTA; when every CTA runs many
// units (at least 8) the launch is bandwidth-bound, so its time goes as ceil(units / G) unit times,
// each inversely proportional to the bandwidth share of G SMs: proportional to ceil(units / G) * G.
// The G in [4/5 of the SMs, all of them] that minimises that is taken when it saves at least 3 %.
// Measured: 2048 units of 460 slots run on 128 CTAs of 16 units instead of 152 of 13-14, 77.4 ->
// 75.3 us (E4M3 cache: 43.3 -> 42.4 us); 1792 units of 307 slots, where 128 CTAs of 14 would save
// 1.75 % on paper, ran 5.8 % slower (fewer SMs, each with less in flight), which is what the 3 %
// margin keeps out; 8192 units keep all 152 SMs (0.2 %).
inline int balanced_grid(int units, int sms) {
  if (units < 8 * sms) return units < sms ? units : sms;
  const long long full = static_cast<long long>((units + sms - 1) / sms) * sms;
  int best = sms;
  long long best_cost = full;
  for (int g = sms - 1; g * 5 >= sms * 4; --g) {
    const long long cost = static_cast<long long>((units + g - 1) / g) * g;
    if (cost < best_cost) {
      best_cost = cost;
      best = g;
    }
  }
  return best_cost * 100 <= full * 97 ? best : sms;
}

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int dtype, cudaStream_t s);
cudaError_t launch_prefill_scores_simt(const PrefillParams& p, int head_dim, int dtype, cudaStream_t s);
cudaError_t launch_prefill_scores_tc(const PrefillParams& p, int head_dim, cudaStream_t s);  // bf16
cudaError_t launch_select(const SelectParams& p, cudaStream_t s);
// Tensor-core decode step (bf16, D = 128, budget <= 512), persistent over units.
bool decode_tc_supported(int head_dim, int dtype, int budget);
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s);
// Tensor-core decode step with each unit split over a CTA cluster (bf16, D = 128, few units).
bool decode_tc_split_supported(int head_dim, int dtype, int units, int n);
cudaError_t launch_decode_tc_split(const DecodeParams& p, cudaStream_t s);
// One CTA per unit with the unit's K and V resident in shared memory (bf16, D = 128, budget <= 208).
bool decode_resident_supported(int head_dim, int dtype, int budget);
cudaError_t launch_decode_resident(const DecodeParams& p, cudaStream_t s);
bool decode_e4m3_supported(int head_dim, int dtype, int budget);
cudaError_t launch_decode_e4m3(const DecodeParams& p, cudaStream_t s);  // E4M3 caches
int select_max_prompt();
int select_max_budget();

// Chooses how many CTAs (one thread-block cluster) share one unit's decode step and how many slots
// each CTA owns; also the ring depth, shared memory and grid. Returns false if no shape fits.
bool plan_decode(int units, int n, int head_dim, int elem_bytes, int* splits, int* chunk,
                 int* stages, size_t* smem_bytes, int* grid);

// ---- device helpers -----------------------------------------------------------------------

#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One bulk (TMA-engine) copy of `bytes` contiguous bytes global -> this CTA's shared memory;
// completion is signalled on `bar` as transaction bytes. Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns` of wall time (2 s by
// default): then the device error word is set and false is returned, so no wait in this library
// can hang the GPU. Each try_wait may suspend the thread (up to the hint, ~10 ms) until the phase
// completes, so waiting warps do not spin on the issue slots.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                          uint64_t limit_ns = 2000000000ull) {
  const uint32_t addr = smem_u32(bar);
  uint64_t start = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(10000000u)
        : "memory");
    if (done) return true;
    if ((it & 3u) == 0) {
      const uint64_t now = global_timer_ns();
      if (it == 0) start = now;
      else if (now - start > limit_ns) {
        atomicCAS(err, H2O_DEVERR_NONE, H2O_DEVERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// One arrival on `bar` (release semantics: this thread's prior shared-memory reads are ordered
// before the phase it helps complete).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Eviction order of one cached slot under a policy: `key` smaller = evicted first; `cand` = the
// slot may be evicted at all. score is the updated score (H2O: accumulated, Top-K: this step's).
__device__ __forceinline__ unsigned long long policy_key(int32_t policy, float score, int32_t pos,
                                                         int32_t last_candidate, int32_t n_sink,
                                                         int32_t stride, bool* cand) {
  switch (policy) {
    case H2O_POLICY_LOCAL:
      *cand = true;
      return static_cast<uint32_t>(pos);
    case H2O_POLICY_SINK_WINDOW:
      *cand = pos >= n_sink;
      return static_cast<uint32_t>(pos);
    case H2O_POLICY_STRIDED:
      *cand = pos <= last_candidate;
      return (static_cast<unsigned long long>(pos % stride == 0) << 32) | static_cast<uint32_t>(pos);
    default: {  // H2O, Top-K: (score, position), the score made order-preserving as unsigned bits
      *cand = pos <= last_candidate;
      uint32_t b = __float_as_uint(score);
      b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
      return (static_cast<unsigned long long>(b) << 32) | static_cast<uint32_t>(pos);
    }
  }
}

// Programmatic dependent launch: the next kernel in the stream may start its prologue once every
// CTA of this one has signalled; it waits for this grid's completion (and memory) before touching
// the data this grid writes. Every decode kernel signals only after its own wait has returned, so
// while a launch runs, every launch before its predecessor has completed: data that the predecessor
// does not write may be read before the wait.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of the same shared-memory object in the CTA of rank `rank` of this cluster.
template <typename T>
__device__ __forceinline__ const T* peer_ptr(const T* local, uint32_t rank) {
  uint64_t out;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
  return reinterpret_cast<const T*>(out);
}

// bf16 -> f32 of the low / high half of a 32-bit word (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

#endif  // __CUDACC__

}  // namespace h2o
