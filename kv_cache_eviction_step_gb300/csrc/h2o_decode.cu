// h2o_decode.cu -- the fused H2O budgeted decode step for sm_103a (hot-path rows D1-D7).
//
// One launch does, for every unit (layer, sequence, head) and its n = min(t, budget) cached slots:
//   D2 logits s_j = (q . K_j) / sqrt(D) and s_new = (q . k_new) / sqrt(D)   (H2O post §2.1.1)
//   D3 softmax over the n + 1 keys; D4 out = sum_j p_j V_j + p_new v_new
//   D5 scores[j] += p_j in float32 (accumulated attention: H2O post §2.1.2 / §2.2,
//      "H2O Heavy-Hitter Oracle 分析" §3.2)
//   D6 victim = argmin over slots with position <= t - k_local of (updated score, position)
//      (greedy eviction outside the recent tokens: H2O post §2.2)
//   D7 k_new / v_new / p_new / t written into the victim slot in place (H2O post §2.3)
//
// Work decomposition. A unit is handled by `splits` CTAs forming one thread-block cluster; CTA r
// owns the contiguous slots [r*chunk, (r+1)*chunk). The step is HBM-bound (K and V are read once,
// 2*n*D*elem bytes), so each CTA streams its K rows and then its V rows through a ring of 8 KB
// shared-memory tiles filled by bulk asynchronous copies (cp.async.bulk, the TMA engine) and
// tracked with mbarriers; thread 0 refills a stage as soon as every thread has finished reading it.
// Logits stay in shared memory, so the softmax needs no rescaling: the K pass produces all logits,
// the block max and the weights w_j = exp(s_j - m_local) are formed, then the V pass accumulates
// sum_j w_j V_j. CTAs of a cluster exchange (m, l, o) through distributed shared memory, every CTA
// forms p_j = exp(s_j - m) / l for its slots, updates its scores and reduces a local argmin key; a
// second exchange picks the cluster-wide victim and the CTA that owns it writes the new token.
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>
#include <utility>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kConsumers = 256;                 // 8 consumer warps compute
constexpr int kWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 32;       // + 1 producer warp issues the bulk copies
constexpr int kTileBytes = 8192;
constexpr int kMaxSplits = 16;
constexpr int kDefaultStages = 6;

template <typename T, int D>
struct Shape {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kLanesPerRow = kRowBytes / 16;        // lanes sharing one K/V row
  static constexpr int kElems = 16 / static_cast<int>(sizeof(T));  // elements per lane
  static constexpr int kGroups = kConsumers / kLanesPerRow;  // rows processed side by side
  static constexpr int kTileRows = kTileBytes / kRowBytes;
  static_assert(kLanesPerRow >= 1 && kLanesPerRow <= 32, "row must span 1..32 lanes");
};

// Per-CTA values exchanged inside the cluster.
template <int D>
struct alignas(16) Publish {
  float m;                       // local max logit (-inf if the CTA owns no slot)
  float l;                       // local sum of exp(s - m)
  unsigned long long best_key;   // local eviction key, ~0 if no candidate
  int32_t best_slot;
  int32_t pad;
  float f[kMaxSplits];           // exp(m_c - m) per cluster rank (rank 0 only)
  float o[D];                    // local sum_j exp(s_j - m) V_j
};

// Reduction scratch: kWarps floats, then s_new, then kWarps argmin keys and kWarps slots.
constexpr int kRedKeys = 64;
constexpr int kRedSlots = kRedKeys + kWarps * 8;
constexpr int kRedBytes = kRedSlots + kWarps * 4 + 16;
static_assert(kWarps * 4 + 4 <= kRedKeys, "reduction floats overlap the keys");

struct Layout {
  int ring, bars, pub, red, logit, wgt, sc, sp, total;
};

template <int D>
__host__ __device__ inline Layout decode_layout(int stages, int chunk) {
  Layout L;
  auto up = [](int x, int a) { return (x + a - 1) / a * a; };
  L.ring = 0;
  L.bars = stages * kTileBytes;               // full[stages], then empty[stages]
  L.pub = up(L.bars + 2 * stages * 8, 16);
  L.red = up(L.pub + static_cast<int>(sizeof(Publish<D>)), 16);
  L.logit = up(L.red + kRedBytes, 16);
  L.wgt = L.logit + chunk * 4;
  L.sc = L.wgt + chunk * 4;
  L.sp = L.sc + chunk * 4;
  L.total = up(L.sp + chunk * 4, 128);
  return L;
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float* f) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_lo(w[i]);
      f[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
}

template <int LANES>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Barrier over the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int warp = threadIdx.x >> 5;
  consumer_sync();
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  consumer_sync();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5;
  consumer_sync();
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  consumer_sync();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r += red[w];
  return r;
}

template <typename T>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (sizeof(T) == 2) {
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<float*>(out)[idx] = v;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) h2o_decode_step_kernel(const DecodeParams p) {
  using S = Shape<T, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int splits = p.splits;
  const int rank = static_cast<int>(blockIdx.x) % splits;
  const int unit = static_cast<int>(blockIdx.x) / splits;
  const int c0 = rank * p.chunk;
  const int rows = max(0, min(p.n, c0 + p.chunk) - c0);
  const int tiles = (rows + S::kTileRows - 1) / S::kTileRows;
  const int total = 2 * tiles;
  const int stages = p.stages;

  const Layout L = decode_layout<D>(stages, p.chunk);
  unsigned char* ring = smem + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + stages;
  Publish<D>* pub = reinterpret_cast<Publish<D>*>(smem + L.pub);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* s_new_sh = red + kWarps;          // one float after the reduction slots
  float* logit = reinterpret_cast<float*>(smem + L.logit);
  float* wgt = reinterpret_cast<float*>(smem + L.wgt);
  float* sc = reinterpret_cast<float*>(smem + L.sc);
  int32_t* sp = reinterpret_cast<int32_t*>(smem + L.sp);
  const bool cache_full = p.n == p.budget;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();  // the last block-wide barrier: from here on producer and consumers split

  const size_t row0 = static_cast<size_t>(unit) * p.budget + c0;
  if (warp == kWarps) {
    // Producer warp: K tiles then V tiles, each into the next ring stage once every consumer warp
    // has released it.
    if (lane == 0) {
      const unsigned char* kbase = static_cast<const unsigned char*>(p.k_cache) + row0 * S::kRowBytes;
      const unsigned char* vbase = static_cast<const unsigned char*>(p.v_cache) + row0 * S::kRowBytes;
      for (int i = 0; i < total; ++i) {
        const int s = i % stages;
        if (i >= stages && !mbar_wait(&empty[s], static_cast<uint32_t>(i / stages - 1) & 1u, p.err)) break;
        const int tt = i < tiles ? i : i - tiles;
        const int r0 = tt * S::kTileRows;
        const int nr = min(S::kTileRows, rows - r0);
        const uint32_t bytes = static_cast<uint32_t>(nr) * S::kRowBytes;
        mbar_expect_tx(&full[s], bytes);
        bulk_g2s(ring + s * kTileBytes, (i < tiles ? kbase : vbase) + static_cast<size_t>(r0) * S::kRowBytes,
                 bytes, &full[s]);
      }
    }
    __syncwarp();
    // Join the cluster barriers the consumers pass through, then leave.
    if (splits > 1) {
      cluster_sync_all();
      if (cache_full) cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  // D1: the new token. Each lane keeps its 16-byte slice of q in registers.
  const int lig = tid % S::kLanesPerRow;
  const int grp = tid / S::kLanesPerRow;
  float qf[S::kElems];
  {
    const uint4 raw = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.q) +
                                                     static_cast<size_t>(unit) * S::kRowBytes)[lig];
    unpack16<T>(raw, qf);
  }
  if (warp == 0) {
    const uint4 raw = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.k_new) +
                                                     static_cast<size_t>(unit) * S::kRowBytes)[lig];
    float kf[S::kElems];
    unpack16<T>(raw, kf);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < S::kElems; ++e) acc = fmaf(qf[e], kf[e], acc);
    acc = row_sum<S::kLanesPerRow>(acc);
    if (lane == 0) *s_new_sh = acc * p.scale;
  }
  // Scores and positions of this CTA's slots, read while the first tiles are in flight.
  for (int r = tid; r < rows; r += kConsumers) {
    sc[r] = p.scores[row0 + r];
    sp[r] = p.slot_pos[row0 + r];
  }

  // D2: logits over the K tiles.
  bool ok = true;
  int i = 0;
  for (; i < tiles; ++i) {
    const int s = i % stages;
    if (ok) ok = mbar_wait(&full[s], static_cast<uint32_t>(i / stages) & 1u, p.err);
    const unsigned char* tile = ring + s * kTileBytes;
    const int r0 = i * S::kTileRows;
    const int nr = min(S::kTileRows, rows - r0);
    for (int rb = 0; rb < nr; rb += S::kGroups) {
      const int r = rb + grp;
      float acc = 0.f;
      if (r < nr && ok) {
        const uint4 raw = *reinterpret_cast<const uint4*>(tile + r * S::kRowBytes + lig * 16);
        float kf[S::kElems];
        unpack16<T>(raw, kf);
#pragma unroll
        for (int e = 0; e < S::kElems; ++e) acc = fmaf(qf[e], kf[e], acc);
      }
      acc = row_sum<S::kLanesPerRow>(acc);
      if (r < nr && lig == 0) logit[r0 + r] = acc * p.scale;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // D3 (local part): max and weights; rank 0 also carries the new token.
  consumer_sync();  // logits, s_new and the score/position prefetch are visible (also if tiles == 0)
  const float s_new = *s_new_sh;
  float mloc = -INFINITY;
  for (int r = tid; r < rows; r += kConsumers) mloc = fmaxf(mloc, logit[r]);
  if (rank == 0 && tid == 0) mloc = fmaxf(mloc, s_new);
  mloc = block_max(mloc, red);
  float lsum = 0.f;
  for (int r = tid; r < rows; r += kConsumers) {
    const float w = expf(logit[r] - mloc);
    wgt[r] = w;
    lsum += w;
  }
  const float w_new = (rank == 0) ? expf(s_new - mloc) : 0.f;
  if (rank == 0 && tid == 0) lsum += w_new;
  lsum = block_sum(lsum, red);  // its barrier also publishes wgt[]

  // D4 (local part): sum_j w_j V_j over the V tiles.
  float acc[S::kElems];
#pragma unroll
  for (int e = 0; e < S::kElems; ++e) acc[e] = 0.f;
  for (; i < total; ++i) {
    const int s = i % stages;
    if (ok) ok = mbar_wait(&full[s], static_cast<uint32_t>(i / stages) & 1u, p.err);
    const unsigned char* tile = ring + s * kTileBytes;
    const int r0 = (i - tiles) * S::kTileRows;
    const int nr = min(S::kTileRows, rows - r0);
    if (ok) {
      for (int r = grp; r < nr; r += S::kGroups) {
        const uint4 raw = *reinterpret_cast<const uint4*>(tile + r * S::kRowBytes + lig * 16);
        float vf[S::kElems];
        unpack16<T>(raw, vf);
        const float w = wgt[r0 + r];
#pragma unroll
        for (int e = 0; e < S::kElems; ++e) acc[e] = fmaf(w, vf[e], acc[e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // All tiles are consumed, so the ring is free: reduce the row groups' partial outputs there.
  float* part = reinterpret_cast<float*>(ring);
  consumer_sync();  // every warp is done with its last tile before the ring is reused
#pragma unroll
  for (int e = 0; e < S::kElems; ++e) part[grp * D + lig * S::kElems + e] = acc[e];
  consumer_sync();
  for (int d = tid; d < D; d += kConsumers) {
    float o = 0.f;
    for (int g = 0; g < S::kGroups; ++g) o += part[g * D + d];
    if (rank == 0) {
      float vn;
      if constexpr (sizeof(T) == 2) {
        vn = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.v_new)[static_cast<size_t>(unit) * D + d]);
      } else {
        vn = reinterpret_cast<const float*>(p.v_new)[static_cast<size_t>(unit) * D + d];
      }
      o = fmaf(w_new, vn, o);
    }
    pub->o[d] = o;
  }
  if (tid == 0) {
    pub->m = mloc;
    pub->l = lsum;
  }

  // D3 (global part): combine (m, l, o) across the cluster.
  if (splits > 1) cluster_sync_all();
  consumer_sync();
  if (tid == 0) {
    float m = -INFINITY;
    for (int c = 0; c < splits; ++c) m = fmaxf(m, (splits > 1 ? peer_ptr(pub, c) : pub)->m);
    float l = 0.f;
    for (int c = 0; c < splits; ++c) {
      const Publish<D>* pc = splits > 1 ? peer_ptr(pub, c) : pub;
      const float f = expf(pc->m - m);
      pub->f[c] = f;
      l = fmaf(pc->l, f, l);
    }
    red[0] = m;
    red[1] = l;
  }
  consumer_sync();
  const float mg = red[0];
  const float lg = red[1];
  if (rank == 0) {
    for (int d = tid; d < D; d += kConsumers) {
      float o = 0.f;
      for (int c = 0; c < splits; ++c) o = fmaf((splits > 1 ? peer_ptr(pub, c) : pub)->o[d], pub->f[c], o);
      store_out<T>(p.out, static_cast<size_t>(unit) * D + d, o / lg);
    }
  }

  // D5 + D6 (local part): p_j, updated scores, argmin key over the unprotected slots.
  const int32_t last_candidate = p.position - p.k_local;
  unsigned long long best = ~0ull;
  int32_t best_slot = -1;
  for (int r = tid; r < rows; r += kConsumers) {
    const float pr = expf(logit[r] - mg) / lg;
    const float ns = p.policy == H2O_POLICY_TOPK ? pr : sc[r] + pr;  // Top-K: this step's weight
    sc[r] = ns;
    bool cand = false;
    const unsigned long long key = policy_key(p.policy, ns, sp[r], last_candidate, p.n_sink, p.stride, &cand);
    if (cache_full && cand && key < best) {
      best = key;
      best_slot = c0 + r;
    }
  }
  const float p_new = expf(s_new - mg) / lg;

  int32_t victim = -1;
  unsigned long long vkey = ~0ull;
  if (cache_full) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long ok2 = __shfl_xor_sync(0xffffffffu, best, off);
      const int32_t os = __shfl_xor_sync(0xffffffffu, best_slot, off);
      if (ok2 < best) {
        best = ok2;
        best_slot = os;
      }
    }
    unsigned long long* kred = reinterpret_cast<unsigned long long*>(smem + L.red + kRedKeys);
    int32_t* sred = reinterpret_cast<int32_t*>(smem + L.red + kRedSlots);
    consumer_sync();
    if (lane == 0) {
      kred[warp] = best;
      sred[warp] = best_slot;
    }
    consumer_sync();
    if (tid == 0) {
      for (int w = 1; w < kWarps; ++w) {
        if (kred[w] < best) {
          best = kred[w];
          best_slot = sred[w];
        }
      }
      pub->best_key = best;
      pub->best_slot = best_slot;
    }
    // D6 (global part): cluster-wide minimum key; its owner holds the victim slot.
    if (splits > 1) cluster_sync_all();
    consumer_sync();
    if (tid == 0) {
      unsigned long long k = ~0ull;
      int32_t slot = -1;
      for (int c = 0; c < splits; ++c) {
        const Publish<D>* pc = splits > 1 ? peer_ptr(pub, c) : pub;
        if (pc->best_key < k) {
          k = pc->best_key;
          slot = pc->best_slot;
        }
      }
      if (slot < 0) atomicCAS(p.err, H2O_DEVERR_NONE, H2O_DEVERR_NO_CANDIDATE);
      kred[0] = k;
      sred[0] = slot;
    }
    consumer_sync();
    vkey = kred[0];
    victim = sred[0];
  }

  // D7: write back the score table and put the new token into its slot.
  for (int r = tid; r < rows; r += kConsumers) p.scores[row0 + r] = (c0 + r == victim) ? p_new : sc[r];
  const int32_t target = cache_full ? victim : p.n;
  const bool owner = cache_full ? (victim >= c0 && victim < c0 + rows) : (rank == 0);
  if (owner && target >= 0 && ok) {
    const size_t trow = static_cast<size_t>(unit) * p.budget + target;
    constexpr int kVec = S::kRowBytes / 16;
    if (tid < 2 * kVec) {
      const bool is_v = tid >= kVec;
      const int c = is_v ? tid - kVec : tid;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(is_v ? p.v_new : p.k_new) +
                                                        static_cast<size_t>(unit) * S::kRowBytes);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(is_v ? p.v_cache : p.k_cache) +
                                            trow * S::kRowBytes);
      dst[c] = src[c];
    }
    if (tid == 0) {
      p.slot_pos[trow] = p.position;
      if (!cache_full) p.scores[trow] = p_new;
    }
  }
  if (rank == 0 && tid == 0) {
    p.evicted_slot[unit] = cache_full ? victim : -1;
    p.evicted_pos[unit] = (cache_full && victim >= 0) ? static_cast<int32_t>(vkey & 0xffffffffu) : -1;
  }
  // Keep this CTA's shared memory alive until every peer has finished reading it.
  if (splits > 1) cluster_sync_all();
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 152;
  return sms;
}

// Opt one kernel into the device's full dynamic shared memory and into 16-CTA clusters, once per
// (kernel, device).
cudaError_t prepare_kernel(const void* fn) {
  thread_local const void* last_fn = nullptr;
  thread_local int last_dev = -1;
  int cur = 0;
  if (cudaGetDevice(&cur) == cudaSuccess && fn == last_fn && cur == last_dev) return cudaSuccess;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& d : done)
    if (d.first == fn && d.second == dev) {
      last_fn = fn;
      last_dev = dev;
      return cudaSuccess;
    }
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin - static_cast<int>(fa.sharedSizeBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  done.emplace_back(fn, dev);
  last_fn = fn;
  last_dev = dev;
  return cudaSuccess;
}

const void* kernel_of(int head_dim, int dtype) {
  if (dtype == H2O_BF16)
    return head_dim == 64 ? reinterpret_cast<const void*>(h2o_decode_step_kernel<__nv_bfloat16, 64>)
                          : reinterpret_cast<const void*>(h2o_decode_step_kernel<__nv_bfloat16, 128>);
  return head_dim == 64 ? reinterpret_cast<const void*>(h2o_decode_step_kernel<float, 64>)
                        : reinterpret_cast<const void*>(h2o_decode_step_kernel<float, 128>);
}

cudaLaunchConfig_t make_config(int units, int splits, size_t smem, cudaStream_t stream,
                               cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units) * static_cast<unsigned>(splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// True if at least one cluster of `splits` CTAs with `smem` bytes each fits on the device.
bool cluster_fits(const void* fn, int splits, size_t smem) {
  if (splits == 1) return true;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config(splits, splits, smem, nullptr, attr);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return clusters > 0;
}

}  // namespace

namespace {

bool plan_decode_uncached(int units, int n, int head_dim, int elem_bytes, int* splits_out,
                          int* chunk_out, int* stages_out, size_t* smem_out, int* grid_out);

struct PlanMemo {
  int dev = -1, units = -1, n = -1, head_dim = -1, elem_bytes = -1;
  int splits = 0, chunk = 0, stages = 0, grid = 0;
  size_t smem = 0;
  bool ok = false;
};

}  // namespace

// Decode steps of one workload repeat the same shape (n stops changing once the cache is full), so
// the plan of the previous call on this thread is reused when nothing changed.
bool plan_decode(int units, int n, int head_dim, int elem_bytes, int* splits_out, int* chunk_out,
                 int* stages_out, size_t* smem_out, int* grid_out) {
  thread_local PlanMemo memo;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (!(memo.dev == dev && memo.units == units && memo.n == n && memo.head_dim == head_dim &&
        memo.elem_bytes == elem_bytes)) {
    memo.ok = plan_decode_uncached(units, n, head_dim, elem_bytes, &memo.splits, &memo.chunk,
                                   &memo.stages, &memo.smem, &memo.grid);
    memo.dev = dev;
    memo.units = units;
    memo.n = n;
    memo.head_dim = head_dim;
    memo.elem_bytes = elem_bytes;
  }
  *splits_out = memo.splits;
  *chunk_out = memo.chunk;
  *stages_out = memo.stages;
  *smem_out = memo.smem;
  *grid_out = memo.grid;
  return memo.ok;
}

namespace {

bool plan_decode_uncached(int units, int n, int head_dim, int elem_bytes, int* splits_out,
                          int* chunk_out, int* stages_out, size_t* smem_out, int* grid_out) {
  const int dtype = elem_bytes == 2 ? H2O_BF16 : H2O_F32;
  const int row_bytes = head_dim * elem_bytes;
  const int tile_rows = kTileBytes / row_bytes;
  const int target_ctas = 4 * device_sm_count();
  int want = 1;
  if (units < target_ctas) want = (target_ctas + units - 1) / units;
  const int max_by_rows = (n + tile_rows - 1) / tile_rows;  // at least one tile per CTA
  want = max(1, min(want, min(kMaxSplits, max_by_rows)));

  // Each unit over `splits` CTAs of one cluster (one CTA when there are enough units). Fewest splits
  // whose shared memory fits, starting from the wanted parallelism; wider clusters are taken only if
  // the device can schedule them.
  const void* fn = kernel_of(head_dim, dtype);
  if (prepare_kernel(fn) != cudaSuccess) return false;
  for (int splits = want; splits <= kMaxSplits; ++splits) {
    const int chunk = (n + splits - 1) / splits;
    const int tiles = (chunk + tile_rows - 1) / tile_rows;
    const int stages = max(1, min(kDefaultStages, 2 * tiles));
    const Layout L = head_dim == 64 ? decode_layout<64>(stages, chunk) : decode_layout<128>(stages, chunk);
    if (L.total > 200 * 1024) continue;
    int s = splits;
    while (s > 1 && !cluster_fits(fn, s, static_cast<size_t>(L.total))) --s;
    if (s != splits) continue;
    *splits_out = splits;
    *chunk_out = chunk;
    *stages_out = stages;
    *smem_out = static_cast<size_t>(L.total);
    *grid_out = units * splits;
    return true;
  }
  return false;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int dtype, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(
      (head_dim == 64 ? decode_layout<64>(p.stages, p.chunk) : decode_layout<128>(p.stages, p.chunk)).total);
  const void* fn = kernel_of(head_dim, dtype);
  cudaError_t e = prepare_kernel(fn);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config(p.units, p.splits, smem, stream, attr);
  void* args[] = {const_cast<DecodeParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace h2o
