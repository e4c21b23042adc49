// h2o_select.cu -- prefill selection and gather (hot-path rows P3-P4).
//
//   P3  if the prompt is longer than the budget: keep the last k_local positions plus the k_heavy
//       largest column sums among the older positions (heavy hitters = top-k of the cumulative
//       attention: "H2O Heavy-Hitter Oracle 分析" §3.1; the budget split of the H2O post §2.2);
//       equal sums keep the later position, the decode step's eviction order read backwards
//   P4  kept tokens' K/V rows fill slots 0.. in ascending position, their scores start at the
//       column sums, their positions go into the slot map; unused slots are emptied
//
// One block of 256 threads per unit (several resident per SM). The candidates' 64-bit keys (column sum made order-
// preserving in the high half, position in the low half) are bitonic-sorted in shared memory, the
// k_heavy-th key is the keep threshold, a block scan over positions assigns the slots, and the
// K/V rows are copied with 16-byte accesses spread over the whole block.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>
#include <utility>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kThreads = 256;  // several units per SM: one sorts while another gathers
constexpr int kMaxPrompt = 16384;
constexpr int kMaxBudget = 16384;

__device__ __forceinline__ unsigned long long keep_key(float c, int32_t pos) {
  uint32_t b = __float_as_uint(c);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(b) << 32) | static_cast<uint32_t>(pos);
}

// Ranking key of an older prompt position (larger = kept first): by column-sum value (H2O, and Top-K
// whose array holds the last row's attention), by stride-grid membership then position (strided), or
// lowest position first (the sinks of sink + window).
__device__ __forceinline__ unsigned long long select_key(int mode, float c, int32_t pos, int32_t stride) {
  if (mode == 1) return (static_cast<unsigned long long>(pos % stride == 0) << 32) | static_cast<uint32_t>(pos);
  if (mode == 2) return 0xFFFFFFFFull - static_cast<uint32_t>(pos);
  return keep_key(c, pos);
}

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (kThreads / 32) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    if (lane < (kThreads / 32)) warp_tot[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  return warp_tot[warp] + incl - v;
}

// Four bf16 values (this lane's 8 bytes) of a 128-element row quantised to
// E4M3 against the row's scale (amax over the warp / 448, or 1 for an all-zero row); returns the
// scale and packs the four codes into *codes.
__device__ __forceinline__ float quantise4(uint2 raw, uint32_t* codes) {
  float x[4];
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  x[0] = __low2float(a);
  x[1] = __high2float(a);
  x[2] = __low2float(b);
  x[3] = __high2float(b);
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(x[i] / scale, __NV_SATFINITE, __NV_E4M3)) << (8 * i);
  *codes = w;
  return scale;
}

__global__ void __launch_bounds__(kThreads) prefill_select_kernel(const SelectParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int kept_total;
  __shared__ unsigned long long threshold;
  const int unit = blockIdx.x;
  const int tid = threadIdx.x;
  const int P = p.P;
  const float* c = p.colsum + static_cast<size_t>(unit) * P;
  const bool keep_all = P <= p.budget;
  const int ncand = P - p.k_local;  // older positions that compete (when !keep_all)
  int npad = 1;
  while (npad < ncand) npad <<= 1;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  int32_t* pos_of_slot = reinterpret_cast<int32_t*>(smem + (keep_all ? 0 : static_cast<size_t>(npad) * 8));

  if (tid == 0) threshold = ~0ull;
  if (!keep_all && p.k_heavy > 0) {
    for (int i = tid; i < npad; i += kThreads) keys[i] = i < ncand ? select_key(p.key_mode, c[i], i, p.stride) : 0ull;
    __syncthreads();
    for (int k = 2; k <= npad; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < npad; i += kThreads) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const unsigned long long a = keys[i], b = keys[ixj];
            const bool descending = (i & k) == 0;
            if (descending ? (a < b) : (a > b)) {
              keys[i] = b;
              keys[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }
    if (tid == 0) threshold = keys[p.k_heavy - 1];
  }
  __syncthreads();
  const unsigned long long thr = threshold;

  // Slot of each kept position: exclusive scan of keep flags over contiguous position segments.
  const int seg = (P + kThreads - 1) / kThreads;
  const int lo = min(P, tid * seg), hi = min(P, lo + seg);
  auto kept = [&](int j) {
    if (keep_all || j >= ncand) return true;
    return p.k_heavy > 0 && select_key(p.key_mode, c[j], j, p.stride) >= thr;
  };
  int cnt = 0;
  for (int j = lo; j < hi; ++j) cnt += kept(j) ? 1 : 0;
  int slot = block_exclusive_scan(cnt, warp_tot, &kept_total);
  for (int j = lo; j < hi; ++j)
    if (kept(j)) pos_of_slot[slot++] = j;
  __syncthreads();
  const int nk = kept_total;

  // Gather the kept rows and reset the unused slots.
  const size_t ub = static_cast<size_t>(unit) * p.budget;
  const int vecs = p.row_bytes / 16;
  const uint4* ksrc = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.k) +
                                                     static_cast<size_t>(unit) * P * p.row_bytes);
  const uint4* vsrc = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.v) +
                                                     static_cast<size_t>(unit) * P * p.row_bytes);
  uint4* kdst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.k_cache) + ub * p.row_bytes);
  uint4* vdst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.v_cache) + ub * p.row_bytes);
  if (p.k_scale != nullptr) {
    // E4M3 caches (D = 128): one warp per slot, four elements per lane; scale = amax / 448 over the
    // row, codes to nearest even, saturating; empty slots get zero codes and scale 0.
    const int warp = tid >> 5, lane = tid & 31;
    const uint2* k2 = reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(p.k) +
                                                     static_cast<size_t>(unit) * P * 256);
    const uint2* v2 = reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(p.v) +
                                                     static_cast<size_t>(unit) * P * 256);
    uint32_t* kc = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(p.k_cache) + ub * 128);
    uint32_t* vc = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(p.v_cache) + ub * 128);
    for (int s = warp; s < p.budget; s += kThreads / 32) {
      uint32_t kw = 0, vw = 0;
      float ks = 0.f, vs = 0.f;
      if (s < nk) {
        const size_t src = static_cast<size_t>(pos_of_slot[s]) * 32 + lane;  // 32 uint2 per row
        ks = quantise4(__ldg(k2 + src), &kw);
        vs = quantise4(__ldg(v2 + src), &vw);
      }
      kc[static_cast<size_t>(s) * 32 + lane] = kw;
      vc[static_cast<size_t>(s) * 32 + lane] = vw;
      if (lane == 0) {
        p.k_scale[ub + s] = ks;
        p.v_scale[ub + s] = vs;
      }
    }
  } else {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    // Four 16-byte rows pieces per thread per round, all loads issued before the stores, so each
    // thread keeps eight reads in flight.
    constexpr int kBatch = 4;
    const int total = p.budget * vecs;
    for (int e0 = tid; e0 < total; e0 += kBatch * kThreads) {
      uint4 kr[kBatch], vr[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int e = e0 + b * kThreads;
        kr[b] = zero;
        vr[b] = zero;
        if (e < total) {
          const int s = e / vecs;
          if (s < nk) {
            const size_t src = static_cast<size_t>(pos_of_slot[s]) * vecs + (e - s * vecs);
            kr[b] = __ldg(ksrc + src);
            vr[b] = __ldg(vsrc + src);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int e = e0 + b * kThreads;
        if (e < total) {
          kdst[e] = kr[b];
          vdst[e] = vr[b];
        }
      }
    }
  }
  for (int s = tid; s < p.budget; s += kThreads) {
    const bool used = s < nk;
    p.scores[ub + s] = used ? c[pos_of_slot[s]] : 0.f;
    p.slot_pos[ub + s] = used ? pos_of_slot[s] : -1;
  }
}

cudaError_t prepare_select() {
  static std::mutex mu;
  static std::vector<int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int d : done)
    if (d == dev) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_select_kernel);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin - static_cast<int>(fa.sharedSizeBytes));
  if (e != cudaSuccess) return e;
  done.push_back(dev);
  return cudaSuccess;
}

}  // namespace

int select_max_prompt() { return kMaxPrompt; }
int select_max_budget() { return kMaxBudget; }

cudaError_t launch_select(const SelectParams& p, cudaStream_t s) {
  cudaError_t e = prepare_select();
  if (e != cudaSuccess) return e;
  size_t smem = 0;
  if (p.P > p.budget) {
    int npad = 1;
    while (npad < p.P - p.k_local) npad <<= 1;
    smem = static_cast<size_t>(npad) * 8;
  }
  smem += static_cast<size_t>(p.budget) * 4;
  prefill_select_kernel<<<p.units, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace h2o
