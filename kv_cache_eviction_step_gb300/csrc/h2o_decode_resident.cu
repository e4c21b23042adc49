// h2o_decode_resident.cu -- the decode step (D1-D7) for launches of few units with short caches,
// e.g. one layer of a model's batch x heads per launch: one CTA per unit that holds the unit's whole
// K and V in shared memory.
//
// Per unit and step (n = min(t, budget) cached slots; H2O post §2.1.1-§2.3, "H2O Heavy-Hitter
// Oracle 分析" §3.2): logits s_j = (q . K_j) / sqrt(D) and s_new, softmax over the n + 1 keys,
// out = sum_j p_j V_j + p_new v_new, scores[j] += p_j in fp32, victim = argmin over the slots with
// position <= t - k_local of (score, position), and the new token written into the victim slot.
//
// Why a kernel of its own. A launch of 256 units of 204 slots carries 27.8 MB, ~4 us of HBM time,
// so it is bound by what happens around the previous launch: when its CTAs can start, when their
// data arrives, and the chain of dependent steps once the query is there. Here:
//   - the unit's K and V (n rows each, <= 208 x 256 B) are fetched by bulk copies of 26 rows with one
//     mbarrier each, issued at CTA start (before griddepcontrol.wait when the previous launch on the
//     stream wrote none of this call's cache), and stay resident: no ring, no refill round trip;
//   - both contractions are GEMVs (one query row) on the CUDA cores. Warp w owns slots
//     [26 w, 26 w + 26) (so all 8 warps have slots at 204-208) and waits only for their copies; a
//     half-warp covers a 256-byte row, lane
//     (hl, li) = (lane / 16, lane % 16) reading columns [8 li, 8 li + 8) of the rows of parity hl
//     with one 16-byte shared load per row (conflict-free). The logits use fma.rn.f32.bf16 (bf16
//     operands, fp32 products and sums); the 13 partial dot products of a lane (padded to 16) are
//     reduced across its half-warp by a butterfly reduce-scatter (8 + 4 + 2 + 1 shuffles) that leaves
//     lane (hl, li), li < 13, holding slot 26 w + 2 li + hl's logit, the slot it keeps for the
//     softmax, the score update and the victim search. V^T w accumulates column pairs with fma.rn.f32x2;
//   - the softmax needs one block barrier: each warp publishes its (max, sum of exp) pair, and every
//     lane forms the normaliser from them with one exp and a 3-shuffle sum;
//   - with a next-call hint (h2o_decode_step_prefetch) the CTA asks L2 for the next call's rows of
//     its unit once its own critical reads have arrived, so the next launch's copies hit L2.
// Two CTAs fit on an SM (at most 109 KiB of shared memory each, at 208 slots), so the next launch's
// CTAs start, and fetch their cache, while this one runs.
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kD = 128;
constexpr int kRowBytes = kD * 2;            // one bf16 K or V row
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBlockRows = 26;               // slots per warp, per bulk copy and per mbarrier (26 x 8
                                             // warps = 208: every warp works at the largest budgets)
constexpr int kPairs = kBlockRows / 2;       // row pairs per warp (one per half-warp each)
constexpr int kMaxSlots = 208;
constexpr int kMaxBlocks = (kMaxSlots + kBlockRows - 1) / kBlockRows;
static_assert(kMaxBlocks <= kWarps, "one warp per block of slots");

// Shared memory: K rows [budget], V rows [budget], per-warp output partials [kWarps][kD] (f32),
// per-warp softmax pairs and eviction keys, the new token's rows, 2 x kWarps + 1 mbarriers.
struct Layout {
  int k, v, part, red, tok, bars, total;
};

__host__ __device__ inline Layout resident_layout(int budget) {
  Layout L;
  L.k = 0;
  L.v = budget * kRowBytes;
  L.part = 2 * budget * kRowBytes;
  L.red = L.part + kWarps * kD * 4;   // m[kWarps], l[kWarps] (f32), key[kWarps] (u64), slot[kWarps],
                                      // then a flag: some wait of this CTA gave up
  L.tok = L.red + kWarps * 20 + 16;   // the new token's q, k_new and v_new rows
  L.bars = L.tok + 3 * kRowBytes;
  L.total = L.bars + (2 * kWarps + 1) * 8;
  return L;
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_line_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ float dot4_bf16(uint2 k, unsigned short q0, unsigned short q1, unsigned short q2,
                                           unsigned short q3) {
  float r;
  asm("{\n .reg .b16 k0, k1, k2, k3;\n mov.b32 {k0, k1}, %1;\n mov.b32 {k2, k3}, %2;\n"
      " fma.rn.f32.bf16 %0, %3, k0, 0f00000000;\n fma.rn.f32.bf16 %0, %4, k1, %0;\n"
      " fma.rn.f32.bf16 %0, %5, k2, %0;\n fma.rn.f32.bf16 %0, %6, k3, %0;\n}"
      : "=f"(r)
      : "r"(k.x), "r"(k.y), "h"(q0), "h"(q1), "h"(q2), "h"(q3));
  return r;
}
// Two fp32 fmas in one instruction (each lane of the pair rounded as fmaf).
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float dot8_bf16(uint4 k, const unsigned short (&q)[8]) {
  return dot4_bf16(make_uint2(k.x, k.y), q[0], q[1], q[2], q[3]) + dot4_bf16(make_uint2(k.z, k.w), q[4], q[5], q[6], q[7]);
}

// Butterfly reduce-scatter over groups of N lanes (lane bits below N): on entry lane l holds v[i],
// its share of row i's sum (i < N); on exit v[0] of lane l is the group's sum for row l mod N. At
// step h each lane keeps the half of its rows whose index has bit h equal to its own lane bit h and
// adds the partner's share of those rows.
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
  for (int h = N / 2; h >= 1; h >>= 1) {
    const bool upper = (lane & h) != 0;
#pragma unroll
    for (int j = 0; j < h; ++j) {
      const float send = upper ? v[j] : v[j + h];
      const float keep = upper ? v[j + h] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, h);
    }
  }
  return v[0];
}

__global__ void __launch_bounds__(kThreads, 2) h2o_decode_resident_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int unit = static_cast<int>(blockIdx.x);
  const int B = p.budget, n = p.n;
  const int blocks = (n + kBlockRows - 1) / kBlockRows;
  const Layout L = resident_layout(B);
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* red_m = reinterpret_cast<float*>(smem + L.red);
  float* red_l = red_m + kWarps;
  unsigned long long* red_key = reinterpret_cast<unsigned long long*>(red_l + kWarps);
  int32_t* red_slot = reinterpret_cast<int32_t*>(red_key + kWarps);
  int32_t* gave_up = red_slot + kWarps;
  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* vbar = kbar + kWarps;
  uint64_t* tbar = vbar + kWarps;  // the new token's rows
  const uint32_t tok = smem_u32(smem + L.tok);
  const size_t row0 = static_cast<size_t>(unit) * B;
  // Lane (hl, li) = (lane / 16, lane % 16) works on columns [8 li, 8 li + 8) of its warp's rows with
  // parity hl, and holds slot j = 26 warp + 2 li + hl (if li < 13 and j < n).
  const int hl = lane >> 4, li = lane & 15;
  const int j = warp * kBlockRows + 2 * li + hl;
  const bool has_slot = li < kPairs && j < n;
  const bool mine = warp < blocks;  // this warp's block of slots holds cached rows
  const bool cache_full = n == B;

  // Without a next-call hint, the new token's rows are asked of L2 at once (a prefetch only: the read
  // after griddepcontrol.wait still sees whatever the previous kernel wrote), so that read is an L2
  // hit when they were in HBM (one layer of 256 units per launch: 6.18 -> 5.94 us). With a hint the
  // previous launch is prefetching this launch's cache rows at this moment, and this early read,
  // queued against them, measured slower (5.57 -> 5.71 us), so it is left out.
  if (warp == 2 && lane < 3 && p.next_k_cache == nullptr) {
    const void* src = lane == 0 ? p.q : lane == 1 ? p.k_new : p.v_new;
    bulk_prefetch_l2(static_cast<const unsigned char*>(src) + static_cast<size_t>(unit) * kRowBytes, kRowBytes);
  }
  if (tid == 0) {
    for (int b = 0; b < 2 * kWarps + 1; ++b) mbar_init(&kbar[b], 1);
    fence_mbar_init();
    *gave_up = 0;
  }
  __syncthreads();

  // The unit's K rows, then its V rows, 32 rows per copy; the scores and positions of slot j.
  auto fetch = [&]() {
    if (tid == 0) {
      const unsigned char* ksrc = static_cast<const unsigned char*>(p.k_cache) + row0 * kRowBytes;
      const unsigned char* vsrc = static_cast<const unsigned char*>(p.v_cache) + row0 * kRowBytes;
      for (int b = 0; b < blocks; ++b) {
        const uint32_t bytes = static_cast<uint32_t>(min(kBlockRows, n - b * kBlockRows) * kRowBytes);
        mbar_expect_tx(&kbar[b], bytes);
        bulk_g2s(smem + L.k + b * kBlockRows * kRowBytes, ksrc + b * kBlockRows * kRowBytes, bytes, &kbar[b]);
      }
      for (int b = 0; b < blocks; ++b) {
        const uint32_t bytes = static_cast<uint32_t>(min(kBlockRows, n - b * kBlockRows) * kRowBytes);
        mbar_expect_tx(&vbar[b], bytes);
        bulk_g2s(smem + L.v + b * kBlockRows * kRowBytes, vsrc + b * kBlockRows * kRowBytes, bytes, &vbar[b]);
      }
    }
  };
  float sc = 0.f;
  int32_t sp = 0;
  if (p.early != 0) {  // the previous launch on the stream wrote none of this call's cache arrays
    fetch();
    if (has_slot) {
      sc = p.scores[row0 + j];
      sp = p.slot_pos[row0 + j];
    }
    pdl_wait();
    pdl_launch_dependents();
  } else {
    pdl_wait();  // the previous step's cache, scores and slot map are complete from here on
    pdl_launch_dependents();
    fetch();
    if (has_slot) {
      sc = p.scores[row0 + j];
      sp = p.slot_pos[row0 + j];
    }
  }

  // D1: the new token's q, k_new and v_new rows, copied into shared memory (no warp waits on a
  // register load); every warp forms s_new = q . k_new itself. Once they have arrived, the next
  // call's rows of this unit are asked of L2 (a hint only: nothing here reads them): the new token's
  // rows are this step's critical read, and a prefetch issued earlier would queue other CTAs' reads
  // of them behind its 104 KB in HBM (measured on one OPT-6.7B layer of 256 units per launch: issued
  // right after the new token's copies 6.05 us per launch, after they arrived 5.90 us, after the
  // logits 6.07 us).
  if (tid == 0) {
    const size_t urow = static_cast<size_t>(unit) * kRowBytes;
    mbar_expect_tx(tbar, 3 * kRowBytes);
    bulk_g2s(smem + L.tok, static_cast<const unsigned char*>(p.q) + urow, kRowBytes, tbar);
    bulk_g2s(smem + L.tok + kRowBytes, static_cast<const unsigned char*>(p.k_new) + urow, kRowBytes, tbar);
    bulk_g2s(smem + L.tok + 2 * kRowBytes, static_cast<const unsigned char*>(p.v_new) + urow, kRowBytes, tbar);
  }
  if (warp == 1 && p.next_k_cache != nullptr) {
    for (int o = lane * 128; o < B * 4; o += 32 * 128) {
      prefetch_line_l2(reinterpret_cast<const unsigned char*>(p.next_scores + row0) + o);
      prefetch_line_l2(reinterpret_cast<const unsigned char*>(p.next_slot_pos + row0) + o);
    }
  }
  bool ok = mbar_wait(tbar, 0, p.err);
  if (tid == 0 && p.next_k_cache != nullptr) {
    const size_t off = row0 * kRowBytes;
    bulk_prefetch_l2(static_cast<const unsigned char*>(p.next_k_cache) + off, static_cast<uint32_t>(B * kRowBytes));
    bulk_prefetch_l2(static_cast<const unsigned char*>(p.next_v_cache) + off, static_cast<uint32_t>(B * kRowBytes));
  }
  const uint4 q_raw = *reinterpret_cast<const uint4*>(smem + L.tok + li * 16);
  const unsigned short q16[8] = {
      static_cast<unsigned short>(q_raw.x & 0xffffu), static_cast<unsigned short>(q_raw.x >> 16),
      static_cast<unsigned short>(q_raw.y & 0xffffu), static_cast<unsigned short>(q_raw.y >> 16),
      static_cast<unsigned short>(q_raw.z & 0xffffu), static_cast<unsigned short>(q_raw.z >> 16),
      static_cast<unsigned short>(q_raw.w & 0xffffu), static_cast<unsigned short>(q_raw.w >> 16)};
  float sn = dot8_bf16(*reinterpret_cast<const uint4*>(smem + L.tok + kRowBytes + li * 16), q16);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) sn += __shfl_xor_sync(0xffffffffu, sn, off);  // over the 16 lanes
  const float s_new = sn * p.scale;

  // D2: logits of this warp's 26 slots once their K rows have landed (row pairs past the 13th: none).
  // Rows past the block's last cached slot re-read that slot (no branch per row, every load stays
  // inside the copied rows); their logits are dropped and their weights are zero.
  const int rows = min(kBlockRows, n - warp * kBlockRows);  // >= 1 for this warp's block
  float s = -INFINITY;  // slot j's logit
  if (mine) {
    if (ok) ok = mbar_wait(&kbar[warp], 0, p.err);
    const uint4* krow = reinterpret_cast<const uint4*>(smem + L.k + warp * kBlockRows * kRowBytes) + li;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = 2 * i + hl;
      v[i] = i < kPairs ? dot8_bf16(krow[(r < rows ? r : rows - 1) * (kRowBytes / 16)], q16) : 0.f;
    }
    const float dot = reduce_scatter<16>(v, li);
    if (has_slot) s = dot * p.scale;
  }

  // D3: softmax over the n slots and the new token. Each warp publishes (its max, its sum of
  // exp(s - max)); every thread combines the pairs into the block's max m and normaliser l.
  float mw = warp_max(warp == 0 ? fmaxf(s, s_new) : s);
  float ew = has_slot ? expf(s - mw) : 0.f;
  if (warp == 0 && lane == 0) ew += expf(s_new - mw);
  ew = warp_sum(ew);
  if (lane == 0) {
    red_m[warp] = mw;
    red_l[warp] = ew;
  }
  __syncthreads();
  float m = red_m[0];
#pragma unroll
  for (int w2 = 1; w2 < kWarps; ++w2) m = fmaxf(m, red_m[w2]);
  // l = sum over warps of (their sum) exp(their max - m): lane k of each group of kWarps lanes takes
  // warp k's term and three shuffles add them, so each thread evaluates one exp instead of kWarps
  // (the sum is the same in every lane: each step adds the same pairs).
  float l = red_l[lane % kWarps] * expf(red_m[lane % kWarps] - m);
#pragma unroll
  for (int off = 1; off < kWarps; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const float wj = has_slot ? expf(s - m) : 0.f;  // slot j's unnormalised weight
  const float w_new = expf(s_new - m);

  // D4: this warp's share of sum_j w_j V_j: lane (hl, li) accumulates columns [8 li, 8 li + 8) over
  // the rows of parity hl (row 2 i + hl's weight is held by lane 16 hl + i), then the two halves add.
  if (mine) {
    unsigned long long a[4] = {0ull, 0ull, 0ull, 0ull};  // column pairs (8 li + 2 e, 8 li + 2 e + 1)
    if (ok) ok = mbar_wait(&vbar[warp], 0, p.err);
    const uint4* vrow = reinterpret_cast<const uint4*>(smem + L.v + warp * kBlockRows * kRowBytes) + li;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const int r = 2 * i + hl;
      const float wr = __shfl_sync(0xffffffffu, wj, 16 * hl + i);  // 0 for rows past the last cached slot
      const uint4 raw = vrow[(r < rows ? r : rows - 1) * (kRowBytes / 16)];
      const unsigned long long w2 = pack2(wr, wr);
      a[0] = ffma2(w2, pack2(bf16_lo(raw.x), bf16_hi(raw.x)), a[0]);
      a[1] = ffma2(w2, pack2(bf16_lo(raw.y), bf16_hi(raw.y)), a[1]);
      a[2] = ffma2(w2, pack2(bf16_lo(raw.z), bf16_hi(raw.z)), a[2]);
      a[3] = ffma2(w2, pack2(bf16_lo(raw.w), bf16_hi(raw.w)), a[3]);
    }
    float o8[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o8[2 * e] = __uint_as_float(static_cast<uint32_t>(a[e]));
      o8[2 * e + 1] = __uint_as_float(static_cast<uint32_t>(a[e] >> 32));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) o8[e] += __shfl_xor_sync(0xffffffffu, o8[e], 16);
    if (hl == 0) {
      float4* dst = reinterpret_cast<float4*>(part + warp * kD + li * 8);
      dst[0] = make_float4(o8[0], o8[1], o8[2], o8[3]);
      dst[1] = make_float4(o8[4], o8[5], o8[6], o8[7]);
    }
  }

  // D5 + D6: p_j, the updated score of slot j and the block's eviction key.
  const int32_t last_candidate = p.position - p.k_local;
  unsigned long long best = ~0ull;
  float ns = 0.f;
  if (has_slot) {
    const float pr = wj / l;
    ns = p.policy == H2O_POLICY_TOPK ? pr : sc + pr;  // Top-K: this step's weight
    bool cand = false;
    const unsigned long long key = policy_key(p.policy, ns, sp, last_candidate, p.n_sink, p.stride, &cand);
    if (cache_full && cand) best = key;
  }
  int32_t best_slot = best == ~0ull ? -1 : j;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, off);
    const int32_t os = __shfl_xor_sync(0xffffffffu, best_slot, off);
    if (ob < best) {
      best = ob;
      best_slot = os;
    }
  }
  if (lane == 0) {
    red_key[warp] = best;
    red_slot[warp] = best_slot;
  }
  if (!ok) *gave_up = 1;
  __syncthreads();  // output partials and eviction keys complete (and every wait of the CTA is over)
  // The smallest of the eight warp keys, as a 3-level tree over loads issued together.
  unsigned long long tk[kWarps];
  int32_t ts[kWarps];
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2) {
    tk[w2] = red_key[w2];
    ts[w2] = red_slot[w2];
  }
#pragma unroll
  for (int h = kWarps / 2; h >= 1; h >>= 1)
#pragma unroll
    for (int w2 = 0; w2 < h; ++w2)
      if (tk[w2 + h] < tk[w2]) {
        tk[w2] = tk[w2 + h];
        ts[w2] = ts[w2 + h];
      }
  unsigned long long vkey = tk[0];
  int32_t victim = ts[0];
  if (!cache_full) {
    victim = -1;
    vkey = ~0ull;
  } else if (tid == 0 && victim < 0) {
    atomicCAS(p.err, H2O_DEVERR_NONE, H2O_DEVERR_NO_CANDIDATE);
  }
  const float p_new = w_new / l;
  if (tid < kD) {  // output element tid: the warps' partials (zero past the last block), as a tree
    float o8[kWarps];
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) o8[w2] = w2 < blocks ? part[w2 * kD + tid] : 0.f;
#pragma unroll
    for (int h = kWarps / 2; h >= 1; h >>= 1)
#pragma unroll
      for (int w2 = 0; w2 < h; ++w2) o8[w2] += o8[w2 + h];
    float o = o8[0];
    const float vn = bf16_lo(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(smem + L.tok + 2 * kRowBytes + 2 * tid)));
    o = fmaf(w_new, vn, o);
    static_cast<__nv_bfloat16*>(p.out)[static_cast<size_t>(unit) * kD + tid] = __float2bfloat16_rn(o / l);
  }

  // D7: the score table written back, the new token in its slot (warp 0 writes K, warp 1 V).
  if (has_slot) p.scores[row0 + j] = (j == victim) ? p_new : ns;
  const int32_t target = cache_full ? victim : n;
  if (target >= 0 && ok) {
    const size_t trow = row0 + static_cast<size_t>(target);
    if (warp < 2)
      *reinterpret_cast<uint2*>(static_cast<unsigned char*>(warp == 0 ? p.k_cache : p.v_cache) + trow * kRowBytes + lane * 8) =
          lds64(tok + (1 + warp) * kRowBytes + lane * 8);
    if (tid == 0) {
      p.slot_pos[trow] = p.position;
      if (!cache_full) p.scores[trow] = p_new;
    }
  }
  if (tid == 0) {
    p.evicted_slot[unit] = cache_full ? victim : -1;
    p.evicted_pos[unit] = (cache_full && victim >= 0) ? static_cast<int32_t>(vkey & 0xffffffffu) : -1;
    // If a wait above gave up, a copy may still be landing in this CTA's shared memory: keep the CTA
    // until every copy it issued has completed (a second bounded window).
    if (*gave_up) {
      for (int b = 0; b < blocks; ++b) {
        (void)mbar_wait(&kbar[b], 0, p.err, 8000000000ull);
        (void)mbar_wait(&vbar[b], 0, p.err, 8000000000ull);
      }
      (void)mbar_wait(tbar, 0, p.err, 8000000000ull);
    }
  }
}

}  // namespace

bool decode_resident_supported(int head_dim, int dtype, int budget) {
  return head_dim == kD && dtype == H2O_BF16 && budget >= 1 && budget <= kMaxSlots;
}

cudaError_t launch_decode_resident(const DecodeParams& p, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(h2o_decode_resident_kernel);
  {  // opt in to more than 48 KB of dynamic shared memory, once per device
    static std::mutex mu;
    static std::vector<int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    bool found = false;
    for (int d : done) found = found || d == dev;
    if (!found) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, resident_layout(kMaxSlots).total);
      if (e != cudaSuccess) return e;
      done.push_back(dev);
    }
  }
  DecodeParams q = p;
  return launch_pdl(fn, p.units, kThreads, resident_layout(p.budget).total, stream, &q);
}

}  // namespace h2o
