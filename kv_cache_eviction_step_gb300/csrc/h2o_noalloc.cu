// h2o_noalloc.cu -- h2o_prefill_select_static: the prefill score pass + selection with its scratch
// held in a fixed device array inside this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory for the workspace: a serving engine that reserved
// all device memory for its own pool at start-up (a cudaMalloc then fails, or takes memory the
// pool believes it owns), or code that runs as a plugin or callback of a host framework that owns
// the allocator and hands it only the tensors it declared. This entry point needs nothing beyond
// the inputs and outputs: the row max, row normaliser and column-sum arrays live in
// g_prefill_scratch, a file-scope device array of H2O_STATIC_SCRATCH_BYTES that every GPU which
// loads the library keeps until the process exits. It runs exactly the kernels h2o_prefill_select
// runs.
#include <mutex>
#include <utility>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[H2O_STATIC_SCRATCH_BYTES];

// Device address of g_prefill_scratch on the current device. In host code the array's name is a
// host-side stand-in, not a device address, so the address is looked up once per device (with that
// device current) and cached.
void* static_scratch(cudaError_t* err) {
  static std::mutex mu;
  static std::vector<std::pair<int, void*>> cache;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& c : cache)
    if (c.first == dev) return c.second;
  void* ptr = nullptr;
  *err = cudaGetSymbolAddress(&ptr, g_prefill_scratch);
  if (*err != cudaSuccess || ptr == nullptr) return nullptr;
  cache.emplace_back(dev, ptr);
  return ptr;
}

}  // namespace
}  // namespace h2o

extern "C" h2o_status h2o_prefill_select_static(const h2o_dims* dims, int32_t prompt_len,
                                                const void* q, const void* k, const void* v,
                                                void* k_cache, void* v_cache, float* scores,
                                                int32_t* slot_pos, void* stream) {
  const size_t need = h2o_prefill_workspace_bytes(dims, prompt_len);
  if (need == 0) {
    // Invalid arguments or no units: the regular entry point reports which, launching nothing.
    return h2o_prefill_select(dims, prompt_len, q, k, v, k_cache, v_cache, scores, slot_pos,
                              nullptr, 0, stream);
  }
  if (need > H2O_STATIC_SCRATCH_BYTES) return H2O_ERR_UNSUPPORTED;
  cudaError_t err = cudaSuccess;
  void* scratch = h2o::static_scratch(&err);
  if (scratch == nullptr) {
    (void)cudaGetLastError();
    return H2O_ERR_CUDA;
  }
  // Nothing in the scratch has to start at zero: every array is fully written before it is read.
  return h2o_prefill_select(dims, prompt_len, q, k, v, k_cache, v_cache, scores, slot_pos, scratch,
                            H2O_STATIC_SCRATCH_BYTES, stream);
}
