// h2o_decode_tc.cu -- the fused H2O decode step (hot-path rows D1-D7) with both contractions on the
// 5th-generation tensor cores, for bf16 caches with D = 128 and budgets up to 512 slots.
//
// Per unit (layer, sequence, head) with n = min(t, budget) cached slots:
//   D2  logits: S = K q, K the unit's [n x 128] key rows (tiles of 128 rows) and q the new query,
//       as tcgen05.mma M = 128 (slots) x N = 16 (q in row 0, zeros after) x K = 128; the logit of
//       slot j lands in TMEM lane j % 128, column 16 (j / 128)          (H2O post §2.1.1)
//   D3  softmax over the n logits and the new token on the epilogue warps (one slot per thread per
//       tile)
//   D4  output: o = V^T w as tcgen05.mma M = 128 (d) x N = 16 x K = slots, V^T read straight from
//       the TMA-written V tile as an MN-major operand, w written by the epilogue as two bf16 rows
//       (w = hi + lo, so the weights keep ~16 significant bits); o lands in TMEM lane d
//   D5  scores[j] += p_j in fp32, p_j = exp(s_j - m) / l from the fp32 logits (not from hi/lo)
//                                                            (H2O post §2.2; 分析 §3.2)
//   D6  victim = argmin over slots with position <= t - k_local of (score, position)
//   D7  the new token's K/V row, score p_new and position go into the victim slot (H2O post §2.3)
//
// The kernel is persistent: each CTA walks units blockIdx.x, +gridDim.x, ... Warp roles: warps 0-3
// epilogue (one TMEM lane quarter each), warp 4 TMA producer (q rows, K tiles, V tiles of the
// successive units through one 5-stage ring of 32 KB tiles), warp 5 TMEM allocator + MMA issuer.
// Tensor memory holds two unit slots (logits + output accumulator each), so the producer and the
// tensor core run into the next unit while the epilogue finishes the current one. All waits are
// bounded (mbar_wait); every role stops at its first timeout and tensor memory is always freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kD = 128;                    // head dim of this path
constexpr int kTileRows = 128;             // cache rows per tile (MMA M for the logits)
constexpr int kBox = 128 * 128;            // one [128 rows x 64 cols] bf16 box: 16 KB
constexpr int kTileBytes = 2 * kBox;       // a 128-row tile, both 64-column halves
constexpr int kStages = 5;
constexpr int kMaxTiles = 4;               // budgets up to 512 slots
constexpr int kNRows = 16;                 // rows of the small operand (q, or w hi/lo): MMA N
constexpr int kSmallBox = kNRows * 128;    // [16 rows x 64 cols] bf16: 2 KB
constexpr int kQBytes = 2 * kSmallBox;     // q operand: both 64-column halves
constexpr int kWBytes = 2 * kMaxTiles * kSmallBox;  // w operand: 64 slots per 2 KB box
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kEpiWarps + 2);
constexpr int kTmaWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr uint32_t kTmemCols = 256;        // two unit slots of 128 columns
constexpr uint32_t kPvCol = 64;            // output accumulator column inside a unit slot
constexpr int kAlign = 1024;

// Shared-memory layout (offsets from a 1024-aligned base).
constexpr int kRingOff = 0;
constexpr int kQOff = kRingOff + kStages * kTileBytes;
constexpr int kWOff = kQOff + 2 * kQBytes;
constexpr int kCtrlOff = kWOff + 2 * kWBytes;
constexpr int kCtrlBytes = 1024;
constexpr int kSmem = kCtrlOff + kCtrlBytes + kAlign;

struct TcDecodeParams {
  CUtensorMap tm_k;        // K cache [units][budget][128] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap tm_v;        // V cache, same
  CUtensorMap tm_q;        // queries [units][128] bf16, box 64 x 1, 128-byte swizzle
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  float* scores;
  int32_t* slot_pos;
  __nv_bfloat16* out;
  int32_t* evicted_slot;
  int32_t* evicted_pos;
  int32_t* err;
  int32_t units, budget, k_local, position, n, tiles;
  float scale;
  int32_t policy, n_sink, stride;  // eviction policy (h2o_policy_kind)
  int32_t early;                   // cache reads may start before griddepcontrol.wait (DecodeParams)
  const unsigned char* next_k;     // the next decode call's caches (an L2 prefetch hint), or null
  const unsigned char* next_v;
};

// ---- PTX wrappers (same encodings as the prefill's tcgen05 path) -------------------------------

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes made visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 128-byte-swizzled operand descriptor. K-major: rows of 128 bytes, 8-row groups `sbo` apart.
// MN-major: 64-element MN groups `lbo` apart, 8-row K groups `sbo` apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// kind::f16 instruction descriptors, fp32 accumulate, bf16 A and B, M = 128, N = 16.
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((kNRows >> 3) << 17) | ((128 >> 4) << 24);
constexpr uint32_t kIdescQK = kIdescBase;              // A = K tile (K-major), B = q (K-major)
constexpr uint32_t kIdescPV = kIdescBase | (1u << 15); // A = V^T (MN-major), B = w (K-major)

__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}

__device__ __forceinline__ void tmem_ld2(uint32_t taddr, float& a, float& b) {
  uint32_t r0, r1;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1)
      : "r"(taddr)
      : "memory");
  a = __uint_as_float(r0);
  b = __uint_as_float(r1);
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 3, %0;" ::"n"(32 * kEpiWarps) : "memory"); }

// Byte offset of element j (0..n) of row `row` (0 = hi, 1 = lo) of the w operand: 64 slots per
// 2 KB box, 128-byte rows, 16-byte chunks swizzled by the row index.
__device__ __forceinline__ int w_offset(int j, int row) {
  const int box = j >> 6, jj = j & 63;
  return box * kSmallBox + row * 128 + ((((jj >> 3) ^ row) & 7) << 4) + ((jj & 7) << 1);
}

// kAnyPolicy = false compiles the H2O rule alone (the policy switch folds away); true reads it from p.
template <bool kAnyPolicy>
__global__ void __launch_bounds__(kThreads, 1) h2o_decode_tc_kernel(const __grid_constant__ TcDecodeParams p) {
  const int32_t policy = kAnyPolicy ? p.policy : static_cast<int32_t>(H2O_POLICY_H2O);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  unsigned char* ring = smem + kRingOff;
  unsigned char* qbuf = smem + kQOff;
  unsigned char* wbuf = smem + kWOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCtrlOff);
  uint64_t* full = bars;                     // [kStages]
  uint64_t* empty = full + kStages;          // [kStages]
  uint64_t* q_full = empty + kStages;        // [2]
  uint64_t* q_empty = q_full + 2;            // [2]
  uint64_t* s_full = q_empty + 2;            // [2] logits ready
  uint64_t* w_ready = s_full + 2;            // [2] weights written
  uint64_t* o_full = w_ready + 2;            // [2] output ready
  uint64_t* tm_free = o_full + 2;            // [2] unit slot of tensor memory free again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tm_free + 2);
  float* red = reinterpret_cast<float*>(smem + kCtrlOff + 512);          // [kEpiWarps] + 4
  unsigned long long* kred = reinterpret_cast<unsigned long long*>(smem + kCtrlOff + 640);  // [kEpiWarps]
  int32_t* sred = reinterpret_cast<int32_t*>(smem + kCtrlOff + 704);     // [kEpiWarps]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.tiles;
  const int n = p.n;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&q_full[r], 1);
      mbar_init(&q_empty[r], 1);
      mbar_init(&s_full[r], 1);
      mbar_init(&w_ready[r], 1);
      mbar_init(&o_full[r], 1);
      mbar_init(&tm_free[r], kEpiWarps);
    }
    fence_mbar_init();
  }
  // Rows 1..15 of the q operand stay zero (TMA writes row 0 only); the w operand is fully
  // rewritten per unit.
  for (int i = tid; i < 2 * kQBytes / 16; i += kThreads) reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  fence_async_smem();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the previous step's cache, scores and slot map are complete from here on
  pdl_launch_dependents();

  if (warp == kTmaWarp) {
    if (lane == 0) {
      uint32_t g = 0;
      int k = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++k) {
        const int r = k & 1;
        if (k >= 2 && !mbar_wait(&q_empty[r], static_cast<uint32_t>((k >> 1) - 1) & 1u, p.err)) break;
        mbar_expect_tx(&q_full[r], 2 * 128);
        tma_load_2d(qbuf + r * kQBytes, &p.tm_q, 0, u, &q_full[r]);
        tma_load_2d(qbuf + r * kQBytes + kSmallBox, &p.tm_q, 64, u, &q_full[r]);
        for (int i = 0; i < 2 * T; ++i, ++g) {
          const int s = static_cast<int>(g % kStages);
          if (g >= kStages && !mbar_wait(&empty[s], (g / kStages - 1) & 1u, p.err)) {
            ok = false;
            break;
          }
          const CUtensorMap* map = i < T ? &p.tm_k : &p.tm_v;
          const int row0 = (i < T ? i : i - T) * kTileRows;
          mbar_expect_tx(&full[s], kTileBytes);
          tma_load_3d(ring + s * kTileBytes, map, 0, row0, u, &full[s]);
          tma_load_3d(ring + s * kTileBytes + kBox, map, 64, row0, u, &full[s]);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      uint32_t g = 0;
      int k = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++k) {
        const int r = k & 1;
        const uint32_t ph = static_cast<uint32_t>(k >> 1) & 1u;
        const uint32_t slot = tmem + static_cast<uint32_t>(r) * 128;
        if (k >= 2 && !mbar_wait(&tm_free[r], ph ^ 1u, p.err)) break;
        if (!mbar_wait(&q_full[r], ph, p.err)) break;
        const uint32_t q_base = smem_u32(qbuf + r * kQBytes);
        // D2: logits of each 128-row K tile into columns 16 t of this unit's slot.
        for (int t = 0; t < T; ++t, ++g) {
          const int s = static_cast<int>(g % kStages);
          if (!mbar_wait(&full[s], (g / kStages) & 1u, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(ring + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off_a = (kk >> 2) * kBox + (kk & 3) * 32;
            const uint32_t off_b = (kk >> 2) * kSmallBox + (kk & 3) * 32;
            mma(slot + 16 * t, sw128_desc(a_base + off_a, 16, 1024), sw128_desc(q_base + off_b, 16, 1024),
                kIdescQK, kk > 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&q_empty[r]);
        mma_commit(&s_full[r]);
        // D4: o = V^T w over the V tiles, once the epilogue has written w.
        if (!mbar_wait(&w_ready[r], ph, p.err)) break;
        tc_fence_after();
        const uint32_t w_base = smem_u32(wbuf + r * kWBytes);
        for (int t = 0; t < T; ++t, ++g) {
          const int s = static_cast<int>(g % kStages);
          if (!mbar_wait(&full[s], (g / kStages) & 1u, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_base = smem_u32(ring + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk) {
            // V^T as MN-major A: 64-d groups one box apart, 8-slot groups 1024 bytes apart; 16 slots
            // (two groups) per instruction. w as K-major B: 64 slots per 2 KB box.
            const uint32_t off_a = kk * 2048;
            const int j0 = t * kTileRows + kk * 16;
            const uint32_t off_b = (j0 >> 6) * kSmallBox + ((j0 & 63) >> 3) * 16;
            mma(slot + kPvCol, sw128_desc(v_base + off_a, kBox, 1024), sw128_desc(w_base + off_b, 16, 1024),
                kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&o_full[r]);
      }
    }
    __syncwarp();
  } else {
    // Epilogue: thread (warp, lane) owns slot 128 t + 32 warp + lane of every tile t, and output
    // element d = tid.
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int32_t last_candidate = p.position - p.k_local;
    const bool cache_full = n == p.budget;
    int k = 0;
    bool ok = true;
    // A unit's new token and state are loaded one unit ahead, so their latency hides behind the
    // previous unit's epilogue.
    __nv_bfloat16 nq = __float2bfloat16_rn(0.f), nkn = nq, nvn = nq;
    float nsc[kMaxTiles];
    int32_t nsp[kMaxTiles];
    auto prefetch = [&](int u) {
      if (u >= p.units) return;
      const size_t row0 = static_cast<size_t>(u) * p.budget;
      const size_t ud = static_cast<size_t>(u) * kD + tid;
      nq = p.q[ud];
      nkn = p.k_new[ud];
      nvn = p.v_new[ud];
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        const int j = t * kTileRows + tid;
        const bool valid = t < T && j < n;
        nsc[t] = valid ? p.scores[row0 + j] : 0.f;
        nsp[t] = valid ? p.slot_pos[row0 + j] : 0;
      }
    };
    prefetch(blockIdx.x);
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++k) {
      const int r = k & 1;
      const uint32_t ph = static_cast<uint32_t>(k >> 1) & 1u;
      const size_t row0 = static_cast<size_t>(u) * p.budget;
      const size_t ud = static_cast<size_t>(u) * kD + tid;
      const float qd = __bfloat162float(nq);
      const __nv_bfloat16 kn = nkn;
      const __nv_bfloat16 vn = nvn;
      float sc[kMaxTiles];
      int32_t sp[kMaxTiles];
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        sc[t] = nsc[t];
        sp[t] = nsp[t];
      }
      prefetch(u + gridDim.x);
      // s_new = q . k_new / sqrt(D) across the 128 epilogue threads.
      float part = qd * __bfloat162float(kn);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0) red[warp] = part;

      if (!mbar_wait(&s_full[r], ph, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kMaxTiles];
      float m = -INFINITY;
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        s[t] = -INFINITY;
        if (t < T) {
          const float raw = tmem_ld1(lane_base + r * 128 + 16 * t);
          if (t * kTileRows + tid < n) s[t] = raw * p.scale;
        }
        m = fmaxf(m, s[t]);
      }
      epi_sync();  // red[] holds the s_new partials
      const float s_new = (red[0] + red[1] + red[2] + red[3]) * p.scale;
      m = fmaxf(m, s_new);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      epi_sync();
      if (lane == 0) red[warp] = m;
      epi_sync();
      m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      // D3: weights, and the bf16 hi/lo split of each weight into the w operand.
      float e[kMaxTiles];
      float lsum = 0.f;
      unsigned char* wb = wbuf + r * kWBytes;
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        if (t < T) {
          const int j = t * kTileRows + tid;
          e[t] = (s[t] == -INFINITY) ? 0.f : expf(s[t] - m);
          lsum += e[t];
          const __nv_bfloat16 hi = __float2bfloat16_rn(e[t]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(e[t] - __bfloat162float(hi));
          *reinterpret_cast<__nv_bfloat16*>(wb + w_offset(j, 0)) = hi;
          *reinterpret_cast<__nv_bfloat16*>(wb + w_offset(j, 1)) = lo;
        } else {
          e[t] = 0.f;
        }
      }
      fence_async_smem();
      const float w_new = expf(s_new - m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      epi_sync();  // every thread's w entries are written (and fenced); red[] free again
      if (tid == 0) mbar_arrive(&w_ready[r]);
      if (lane == 0) red[warp] = lsum;
      epi_sync();
      const float l = red[0] + red[1] + red[2] + red[3] + w_new;

      // D5 + D6 while the tensor core computes the output.
      unsigned long long best = ~0ull;
      int32_t best_slot = -1;
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        if (t < T && t * kTileRows + tid < n) {
          const float pr = e[t] / l;
          sc[t] = policy == H2O_POLICY_TOPK ? pr : sc[t] + pr;  // Top-K: this step's weight
          bool cand = false;
          const unsigned long long key =
              policy_key(policy, sc[t], sp[t], last_candidate, p.n_sink, p.stride, &cand);
          if (cache_full && cand && key < best) {
            best = key;
            best_slot = t * kTileRows + tid;
          }
        }
      }
      const float p_new = w_new / l;
      int32_t victim = -1;
      unsigned long long vkey = ~0ull;
      if (cache_full) {
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
          kred[warp] = best;
          sred[warp] = best_slot;
        }
        epi_sync();
        vkey = kred[0];
        victim = sred[0];
#pragma unroll
        for (int w = 1; w < kEpiWarps; ++w)
          if (kred[w] < vkey) {
            vkey = kred[w];
            victim = sred[w];
          }
        if (tid == 0 && victim < 0) atomicCAS(p.err, H2O_DEVERR_NONE, H2O_DEVERR_NO_CANDIDATE);
      }

      // D4 result: o[d] = (V^T w_hi + V^T w_lo + w_new v_new) / l.
      if (!mbar_wait(&o_full[r], ph, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float c0, c1;
      tmem_ld2(lane_base + r * 128 + kPvCol, c0, c1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tm_free[r]);
      p.out[ud] = __float2bfloat16_rn((c0 + c1 + w_new * __bfloat162float(vn)) / l);

      // D7: scores back, the new token into its slot, eviction indices.
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        const int j = t * kTileRows + tid;
        if (t < T && j < n) p.scores[row0 + j] = (j == victim) ? p_new : sc[t];
      }
      const int32_t target = cache_full ? victim : n;
      if (target >= 0) {
        p.k_cache[(row0 + target) * kD + tid] = kn;
        p.v_cache[(row0 + target) * kD + tid] = vn;
        if (tid == 0) {
          p.slot_pos[row0 + target] = p.position;
          if (!cache_full) p.scores[row0 + target] = p_new;
        }
      }
      if (tid == 0) {
        p.evicted_slot[u] = cache_full ? victim : -1;
        p.evicted_pos[u] = (cache_full && victim >= 0) ? static_cast<int32_t>(vkey & 0xffffffffu) : -1;
      }
      epi_sync();  // red / kred reuse by the next unit
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---- cluster-split variant: few units, long caches ---------------------------------------------
//
// When there are too few units to fill the GPU (e.g. 32 heads of one sequence with a 4096-slot
// budget), a unit is split over a cluster of `splits` CTAs, CTA r owning slots [r chunk, (r+1) chunk)
// with chunk <= 512. Each CTA computes its logits and V^T w on the tensor core as above, with the
// weights taken relative to its own logit max so the tensor core never waits for the cluster; the
// CTAs then exchange (1) their (max, normaliser) pairs, from which every CTA forms the common max m
// and normaliser l, and (2) their eviction key plus a 1/splits slice of their output partial,
// rescaled by exp(m_c - m), by asynchronous stores into the peers' shared memory (st.async), each
// counting its bytes against the receiving CTA's exchange mbarrier (complete_tx), which every CTA
// arms with the total it expects before the cluster barrier at the start lets any peer send; thread
// r of the sender serves peer r, so the stores to the peers go out side by side. Only the epilogue
// warps take part, so the TMA and MMA warps never wait on the cluster.
// CTA r finishes output elements [r 128/splits, (r+1) 128/splits); the CTA holding the victim writes
// the new token; rank 0 writes the eviction indices. With splits == 1 (one CTA per unit, e.g. one
// layer's 256 units per launch) there is nothing to exchange and the kernel skips both exchanges.

constexpr int kSplitStages = 3;
constexpr int kMaxSplitsTc = 16;
constexpr int kSplitMaxChunk = kMaxTiles * kTileRows;  // 512 slots per CTA
// The small operands keep only the rows that are read back (q: row 0; w: rows 0-1) in 1 KB boxes
// (one 8-row group) placed 1 KB apart. An operand's second 8-row group (rows 8-15) is then the next
// box, and those rows only feed accumulator columns 8-15, which are never read.
constexpr int kNarrowBox = 8 * 128;
constexpr int kSQOff = kSplitStages * kTileBytes;
constexpr int kSQBytes = 3 * kNarrowBox;
constexpr int kSWOff = kSQOff + kSQBytes;
constexpr int kSWBytes = (kSplitMaxChunk / 64 + 1) * kNarrowBox;
constexpr int kSXOff = kSWOff + kSWBytes;

struct SplitXchg {
  float2 ml_in[kMaxSplitsTc];  // (local max, local normaliser) of each rank (exchange 1, st.async)
  unsigned long long key_in[kMaxSplitsTc];
  int32_t slot_in[kMaxSplitsTc];
  float o_in[kD];  // [rank][128 / splits]: the senders' partials of this CTA's output slice
};
constexpr int kSCtrlOff = kSXOff + 1024;
constexpr int kSplitSmem = kSCtrlOff + 512 + kAlign;
static_assert(sizeof(SplitXchg) <= 1024, "exchange area");

struct TcSplitParams {
  TcDecodeParams d;
  int32_t splits, chunk;
};

__device__ __forceinline__ uint32_t peer_smem(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}
// Asynchronous store of (a, b) into a peer's shared memory; on completion it counts 8 bytes
// against the peer's mbarrier (complete_tx), which makes the data visible to the peer's waiters.
__device__ __forceinline__ void st_async_peer_f32x2(uint32_t addr, float a, float b, uint32_t bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(a), "f"(b), "r"(bar_addr)
               : "memory");
}
__device__ __forceinline__ void st_async_peer_f32(uint32_t addr, float v, uint32_t bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
               "r"(bar_addr)
               : "memory");
}
__device__ __forceinline__ void st_async_peer_u64(uint32_t addr, unsigned long long v, uint32_t bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(addr), "l"(v),
               "r"(bar_addr)
               : "memory");
}
__device__ __forceinline__ void st_async_peer_s32(uint32_t addr, int32_t v, uint32_t bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.s32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
               "r"(bar_addr)
               : "memory");
}

// Bounded wait with cluster-scope acquire: data that peers stored before their release-arrive on
// this barrier is visible afterwards.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int32_t* err,
                                                  uint64_t limit_ns = 2000000000ull) {
  const uint32_t addr = smem_u32(bar);
  uint64_t start = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
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

__device__ __forceinline__ int w_offset_narrow(int j, int row) {
  const int box = j >> 6, jj = j & 63;
  return box * kNarrowBox + row * 128 + ((((jj >> 3) ^ row) & 7) << 4) + ((jj & 7) << 1);
}

template <bool kAnyPolicy>
__global__ void __launch_bounds__(kThreads, 1) h2o_decode_tc_split_kernel(const __grid_constant__ TcSplitParams sp_) {
  const TcDecodeParams& p = sp_.d;
  const int32_t policy = kAnyPolicy ? p.policy : static_cast<int32_t>(H2O_POLICY_H2O);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  unsigned char* ring = smem;
  unsigned char* qbuf = smem + kSQOff;
  unsigned char* wbuf = smem + kSWOff;
  SplitXchg* xg = reinterpret_cast<SplitXchg*>(smem + kSXOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSCtrlOff);  // [kSplitStages]
  uint64_t* empty = full + kSplitStages;                             // [kSplitStages]
  uint64_t* q_full = empty + kSplitStages;
  uint64_t* s_full = q_full + 1;
  uint64_t* w_ready = s_full + 1;
  uint64_t* o_full = w_ready + 1;
  uint64_t* xbar = o_full + 1;                                        // [3] exchanges
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 3);
  float* red = reinterpret_cast<float*>(smem + kSCtrlOff + 256);
  unsigned long long* kred = reinterpret_cast<unsigned long long*>(smem + kSCtrlOff + 320);
  int32_t* sred = reinterpret_cast<int32_t*>(smem + kSCtrlOff + 384);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int splits = sp_.splits;
  const uint32_t rank = cluster_ctarank();
  const int unit = static_cast<int>(blockIdx.x) / splits;
  const int c0 = static_cast<int>(rank) * sp_.chunk;
  const int rows = max(0, min(p.n - c0, sp_.chunk));
  const int T = (rows + kTileRows - 1) / kTileRows;
  constexpr uint32_t kCols = 128;
  // One CTA per unit with a next-call hint: the next call's rows of this unit are asked of L2 first
  // (a prefetch only; nothing here reads them), so the next launch's tiles hit L2.
  if (splits == 1 && p.next_k != nullptr && warp == kTmaWarp && lane == 0) {
    const size_t off = static_cast<size_t>(unit) * p.budget * kD * 2;
    const uint32_t bytes = static_cast<uint32_t>(p.budget) * kD * 2;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.next_k + off), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.next_v + off), "r"(bytes) : "memory");
  }

  if (tid == 0) {
    for (int s = 0; s < kSplitStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(w_ready, 1);
    mbar_init(o_full, 1);
    // Both exchanges arrive as st.async bytes against one local arrival each, armed here, before the
    // cluster barrier below lets any peer send: exchange 1 (max, normaliser) 8 bytes per rank;
    // exchange 2 the 128 output elements (a slice from each rank) plus a key and a slot per rank.
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_mbar_init();
    if (splits > 1) {
      mbar_expect_tx(&xbar[0], static_cast<uint32_t>(8 * splits));
      mbar_expect_tx(&xbar[1], static_cast<uint32_t>(kD * 4 + 12 * splits));
    }
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (splits > 1) cluster_sync_all();  // every CTA's exchange barriers exist before any peer arrives
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // With p.early (the previous launch on the stream writes none of this call's cache) the producer's
  // first cache tiles go out, and the epilogue warps read the unit's scores and slot map, before the
  // wait; everything else waits for the previous grid.
  const bool early_tiles = p.early != 0 && warp == kTmaWarp && lane == 0;
  const bool early_epi = p.early != 0 && warp < kEpiWarps;
  if (!early_tiles && !early_epi) {
    pdl_wait();  // the previous step's cache, scores and slot map are complete from here on
    pdl_launch_dependents();
  }
  const size_t row0 = static_cast<size_t>(unit) * p.budget;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      auto tile = [&](int i) {  // ring tile i: K tiles 0..T-1, then V tiles
        const int s = i % kSplitStages;
        const CUtensorMap* map = i < T ? &p.tm_k : &p.tm_v;
        const int r0 = c0 + (i < T ? i : i - T) * kTileRows;
        mbar_expect_tx(&full[s], kTileBytes);
        tma_load_3d(ring + s * kTileBytes, map, 0, r0, unit, &full[s]);
        tma_load_3d(ring + s * kTileBytes + kBox, map, 64, r0, unit, &full[s]);
      };
      int i = 0;
      if (early_tiles) {
        for (; i < 2 * T && i < kSplitStages; ++i) tile(i);
        pdl_wait();
        pdl_launch_dependents();
      }
      mbar_expect_tx(q_full, 2 * 128);
      tma_load_2d(qbuf, &p.tm_q, 0, unit, q_full);
      tma_load_2d(qbuf + kNarrowBox, &p.tm_q, 64, unit, q_full);
      for (; i < 2 * T; ++i) {
        const int s = i % kSplitStages;
        if (i >= kSplitStages && !mbar_wait(&empty[s], static_cast<uint32_t>(i / kSplitStages - 1) & 1u, p.err)) break;
        tile(i);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && mbar_wait(q_full, 0, p.err)) {
      const uint32_t q_base = smem_u32(qbuf);
      bool ok = true;
      int i = 0;
      for (int t = 0; t < T && ok; ++t, ++i) {
        const int s = i % kSplitStages;
        if (!(ok = mbar_wait(&full[s], static_cast<uint32_t>(i / kSplitStages) & 1u, p.err))) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(ring + s * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off_a = (kk >> 2) * kBox + (kk & 3) * 32;
          const uint32_t off_b = (kk >> 2) * kNarrowBox + (kk & 3) * 32;
          mma(tmem + 16 * t, sw128_desc(a_base + off_a, 16, 1024), sw128_desc(q_base + off_b, 16, 1024),
              kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(s_full);
      if (ok && mbar_wait(w_ready, 0, p.err)) {
        tc_fence_after();
        const uint32_t w_base = smem_u32(wbuf);
        for (int t = 0; t < T; ++t, ++i) {
          const int s = i % kSplitStages;
          if (!mbar_wait(&full[s], static_cast<uint32_t>(i / kSplitStages) & 1u, p.err)) break;
          tc_fence_after();
          const uint32_t v_base = smem_u32(ring + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk) {
            const int j0 = t * kTileRows + kk * 16;
            const uint32_t off_b = (j0 >> 6) * kNarrowBox + ((j0 & 63) >> 3) * 16;
            mma(tmem + kPvCol, sw128_desc(v_base + kk * 2048, kBox, 1024), sw128_desc(w_base + off_b, 16, 1024),
                kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
      }
      mma_commit(o_full);
    }
    __syncwarp();
  } else {
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool cache_full = p.n == p.budget;
    const int32_t last_candidate = p.position - p.k_local;
    const size_t ud = static_cast<size_t>(unit) * kD + tid;
    float sc[kMaxTiles];
    int32_t sp[kMaxTiles];
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
      const int jl = t * kTileRows + tid;
      const bool valid = t < T && jl < rows;
      sc[t] = valid ? p.scores[row0 + c0 + jl] : 0.f;
      sp[t] = valid ? p.slot_pos[row0 + c0 + jl] : 0;
    }
    if (early_epi) {  // the new token's rows may be written by the previous grid: read after the wait
      pdl_wait();
      pdl_launch_dependents();
    }
    const float qd = __bfloat162float(p.q[ud]);
    const __nv_bfloat16 kn = p.k_new[ud];
    const __nv_bfloat16 vn = p.v_new[ud];
    const int slice = kD / splits;
    float vn_slice = 0.f;
    if (tid < slice) vn_slice = __bfloat162float(p.v_new[static_cast<size_t>(unit) * kD + rank * slice + tid]);
    float part = qd * __bfloat162float(kn);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) red[warp] = part;

    bool ok = mbar_wait(s_full, 0, p.err);
    tc_fence_after();
    float s[kMaxTiles];
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
      s[t] = -INFINITY;
      if (t < T) {
        const float raw = tmem_ld1(lane_base + 16 * t);
        if (ok && t * kTileRows + tid < rows) s[t] = raw * p.scale;
      }
      m = fmaxf(m, s[t]);
    }
    epi_sync();
    const float s_new = (red[0] + red[1] + red[2] + red[3]) * p.scale;
    if (rank == 0) m = fmaxf(m, s_new);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    epi_sync();
    if (lane == 0) red[warp] = m;
    epi_sync();
    const float mc = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));  // this CTA's max
    // Weights with respect to the local max, so the tensor core can start on V^T w at once; the
    // partial output is rescaled by exp(mc - m) once the cluster-wide max m is known.
    float lsum = 0.f;
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
      if (t < T) {
        const int jl = t * kTileRows + tid;
        const float e = (s[t] == -INFINITY) ? 0.f : expf(s[t] - mc);
        lsum += e;
        const __nv_bfloat16 hi = __float2bfloat16_rn(e);
        const __nv_bfloat16 lo = __float2bfloat16_rn(e - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16*>(wbuf + w_offset_narrow(jl, 0)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(wbuf + w_offset_narrow(jl, 1)) = lo;
      }
    }
    fence_async_smem();
    if (rank == 0 && tid == 0) lsum += expf(s_new - mc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    epi_sync();  // w written and fenced by every thread; red[] read by every thread
    if (tid == 0) mbar_arrive(w_ready);
    if (lane == 0) red[warp] = lsum;
    epi_sync();
    const float lc = red[0] + red[1] + red[2] + red[3];
    // Exchange 1: (local max, local normaliser) -> cluster-wide max and normaliser. One CTA per unit
    // (splits == 1) has both already: m = mc, l = lc (what the exchange would give: lc * exp(0)).
    float mg = mc, l = lc;
    if (splits > 1) {
      // Thread r serves peer r, so the stores and release-arrivals to the peers go out side by side
      // (one thread looping over them serialised one cluster-scope release per peer).
      if (tid < splits) st_async_peer_f32x2(peer_smem(&xg->ml_in[rank], tid), mc, lc, peer_smem(&xbar[0], tid));
      ok = mbar_wait_cluster(&xbar[0], 0, p.err) && ok;
      mg = -INFINITY;
      for (int r = 0; r < splits; ++r) mg = fmaxf(mg, xg->ml_in[r].x);
      l = 0.f;
      for (int r = 0; r < splits; ++r) l = fmaf(xg->ml_in[r].y, expf(xg->ml_in[r].x - mg), l);
    }
    const float w_new = expf(s_new - mg);

    unsigned long long best = ~0ull;
    int32_t best_slot = -1;
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
      const int jl = t * kTileRows + tid;
      if (t < T && jl < rows) {
        const float pr = expf(s[t] - mg) / l;
        sc[t] = policy == H2O_POLICY_TOPK ? pr : sc[t] + pr;  // Top-K: this step's weight
        bool cand = false;
        const unsigned long long key =
            policy_key(policy, sc[t], sp[t], last_candidate, p.n_sink, p.stride, &cand);
        if (cache_full && cand && key < best) {
          best = key;
          best_slot = c0 + jl;
        }
      }
    }
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
      kred[warp] = best;
      sred[warp] = best_slot;
    }
    const float p_new = w_new / l;

    // This CTA's output partial, rescaled to the common max, one slice to each rank.
    ok = mbar_wait(o_full, 0, p.err) && ok;
    tc_fence_after();
    float oc0 = 0.f, oc1 = 0.f;
    tmem_ld2(lane_base + kPvCol, oc0, oc1);
    const float opart = T > 0 ? (oc0 + oc1) * expf(mc - mg) : 0.f;
    int32_t victim = -1;
    unsigned long long vkey = ~0ull;
    float o_sum = 0.f;  // this thread's output element (tid < slice) before the new token's share
    if (splits == 1) {
      // One CTA per unit: the block's own argmin and output, no exchange.
      epi_sync();  // kred / sred complete
      for (int w = 0; w < kEpiWarps; ++w)
        if (kred[w] < vkey) {
          vkey = kred[w];
          victim = sred[w];
        }
      o_sum += opart;
    } else {
      // Exchange 2: output slices (each thread's element to the rank that finishes it) and eviction
      // keys (thread r to peer r, once every warp's key is in kred).
      st_async_peer_f32(peer_smem(&xg->o_in[rank * slice + tid % slice], tid / slice), opart,
                        peer_smem(&xbar[1], tid / slice));
      epi_sync();
      if (tid < splits) {
        unsigned long long kb = kred[0];
        int32_t sb = sred[0];
        for (int w = 1; w < kEpiWarps; ++w)
          if (kred[w] < kb) {
            kb = kred[w];
            sb = sred[w];
          }
        st_async_peer_u64(peer_smem(&xg->key_in[rank], tid), kb, peer_smem(&xbar[1], tid));
        st_async_peer_s32(peer_smem(&xg->slot_in[rank], tid), sb, peer_smem(&xbar[1], tid));
      }
      ok = mbar_wait_cluster(&xbar[1], 0, p.err) && ok;
      for (int r = 0; r < splits; ++r)
        if (xg->key_in[r] < vkey) {
          vkey = xg->key_in[r];
          victim = xg->slot_in[r];
        }
      if (tid < slice)
        for (int r = 0; r < splits; ++r) o_sum += xg->o_in[r * slice + tid];
    }
    if (!cache_full) {
      victim = -1;
      vkey = ~0ull;
    } else if (tid == 0 && rank == 0 && victim < 0) {
      atomicCAS(p.err, H2O_DEVERR_NONE, H2O_DEVERR_NO_CANDIDATE);
    }
    if (tid < slice) {
      const float o = fmaf(w_new, vn_slice, o_sum);
      p.out[static_cast<size_t>(unit) * kD + rank * slice + tid] = __float2bfloat16_rn(o / l);
    }
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
      const int jl = t * kTileRows + tid;
      if (t < T && jl < rows) p.scores[row0 + c0 + jl] = (c0 + jl == victim) ? p_new : sc[t];
    }
    const int32_t target = cache_full ? victim : p.n;
    const bool owner = cache_full ? (victim >= c0 && victim < c0 + rows) : (rank == 0);
    if (owner && target >= 0 && ok) {
      p.k_cache[(row0 + target) * kD + tid] = kn;
      p.v_cache[(row0 + target) * kD + tid] = vn;
      if (tid == 0) {
        p.slot_pos[row0 + target] = p.position;
        if (!cache_full) p.scores[row0 + target] = p_new;
      }
    }
    if (rank == 0 && tid == 0) {
      p.evicted_slot[unit] = cache_full ? victim : -1;
      p.evicted_pos[unit] = (cache_full && victim >= 0) ? static_cast<int32_t>(vkey & 0xffffffffu) : -1;
    }
    // Every peer stores into this CTA's exchange buffers before it arrives on xbar[1], and every
    // peer always reaches that arrival (its own waits are bounded). If a wait above gave up, a late
    // peer may still be on its way, so this CTA must not exit yet: thread 0 waits for all arrivals
    // on xbar[1] (a second, longer bounded window; an immediate return on the normal path), and
    // the block barrier below holds the whole CTA until then.
    if (tid == 0 && splits > 1) {
      (void)mbar_wait_cluster(&xbar[0], 0, p.err, 8000000000ull);
      (void)mbar_wait_cluster(&xbar[1], 0, p.err, 8000000000ull);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

// ---- host side ---------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps depend only on the buffers and the shape; a decode loop reuses them every step.
struct MapCache {
  const void *k = nullptr, *v = nullptr, *q = nullptr;
  int units = -1, budget = -1;
  CUtensorMap tm_k, tm_v, tm_q;
};

}  // namespace

namespace {

// Fills the tensor-core parameters shared by both variants (tensor maps cached per thread).
cudaError_t fill_params(const DecodeParams& dp, TcDecodeParams& p) {
  thread_local MapCache mc;
  const cuuint32_t tile_box[3] = {64, kTileRows, 1};
  if (mc.k != dp.k_cache || mc.units != dp.units || mc.budget != dp.budget) {
    const cuuint64_t dims[3] = {kD, static_cast<cuuint64_t>(dp.budget), static_cast<cuuint64_t>(dp.units)};
    const cuuint64_t strides[2] = {kD * 2, static_cast<cuuint64_t>(dp.budget) * kD * 2};
    if (!encode(&mc.tm_k, dp.k_cache, 3, dims, strides, tile_box)) return cudaErrorInvalidValue;
    mc.k = dp.k_cache;
  }
  if (mc.v != dp.v_cache || mc.units != dp.units || mc.budget != dp.budget) {
    const cuuint64_t dims[3] = {kD, static_cast<cuuint64_t>(dp.budget), static_cast<cuuint64_t>(dp.units)};
    const cuuint64_t strides[2] = {kD * 2, static_cast<cuuint64_t>(dp.budget) * kD * 2};
    if (!encode(&mc.tm_v, dp.v_cache, 3, dims, strides, tile_box)) return cudaErrorInvalidValue;
    mc.v = dp.v_cache;
  }
  if (mc.q != dp.q || mc.units != dp.units) {
    const cuuint64_t dims[2] = {kD, static_cast<cuuint64_t>(dp.units)};
    const cuuint64_t strides[1] = {kD * 2};
    const cuuint32_t box[2] = {64, 1};
    if (!encode(&mc.tm_q, dp.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
    mc.q = dp.q;
  }
  mc.units = dp.units;
  mc.budget = dp.budget;
  p.tm_k = mc.tm_k;
  p.tm_v = mc.tm_v;
  p.tm_q = mc.tm_q;
  p.q = static_cast<const __nv_bfloat16*>(dp.q);
  p.k_new = static_cast<const __nv_bfloat16*>(dp.k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(dp.v_new);
  p.k_cache = static_cast<__nv_bfloat16*>(dp.k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(dp.v_cache);
  p.scores = dp.scores;
  p.slot_pos = dp.slot_pos;
  p.out = static_cast<__nv_bfloat16*>(dp.out);
  p.evicted_slot = dp.evicted_slot;
  p.evicted_pos = dp.evicted_pos;
  p.err = dp.err;
  p.units = dp.units;
  p.budget = dp.budget;
  p.k_local = dp.k_local;
  p.position = dp.position;
  p.n = dp.n;
  p.tiles = (dp.n + kTileRows - 1) / kTileRows;
  p.scale = dp.scale;
  p.policy = dp.policy;
  p.n_sink = dp.n_sink;
  p.stride = dp.stride;
  p.early = dp.early;
  p.next_k = static_cast<const unsigned char*>(dp.next_k_cache);
  p.next_v = static_cast<const unsigned char*>(dp.next_v_cache);
  return cudaSuccess;
}

// The H2O-only and the any-policy instantiations of each kernel.
const void* const kSplitKernels[2] = {reinterpret_cast<const void*>(h2o_decode_tc_split_kernel<false>),
                                      reinterpret_cast<const void*>(h2o_decode_tc_split_kernel<true>)};
const void* const kTcKernels[2] = {reinterpret_cast<const void*>(h2o_decode_tc_kernel<false>),
                                   reinterpret_cast<const void*>(h2o_decode_tc_kernel<true>)};

struct SplitPlan {
  int dev = -1, units = -1, n = -1;
  int splits = 0, chunk = 0;
  bool ok = false;
};

cudaLaunchConfig_t split_config(int units, int splits, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units) * static_cast<unsigned>(splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSplitSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Power-of-two cluster size (so the 128 output elements split evenly) and a chunk of whole 128-slot
// tiles, at most 512 slots; more CTAs per unit (up to 8) while there are fewer than ~2 per SM and each
// would still get at least one full tile.
bool plan_split(int units, int n, int* splits_out, int* chunk_out) {
  thread_local SplitPlan memo;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (memo.dev == dev && memo.units == units && memo.n == n) {
    *splits_out = memo.splits;
    *chunk_out = memo.chunk;
    return memo.ok;
  }
  memo.dev = dev;
  memo.units = units;
  memo.n = n;
  memo.ok = false;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
  // Splitting for parallelism stops at 8 CTAs per cluster: a 16-CTA cluster has to fit inside one
  // GPC, which leaves too few of them resident at once; only caches over 4096 slots take 16.
  int splits = 1;
  while (splits < kMaxSplitsTc &&
         ((n + splits - 1) / splits > kSplitMaxChunk ||
          (splits < 8 && units * splits < 2 * sms && (n + 2 * splits - 1) / (2 * splits) >= kTileRows)))
    splits *= 2;
  int chunk = (n + splits - 1) / splits;
  chunk = (chunk + kTileRows - 1) / kTileRows * kTileRows;
  if (chunk > kSplitMaxChunk) return false;
  static std::mutex mu;
  static std::vector<int> ready;
  {
    std::lock_guard<std::mutex> lock(mu);
    bool found = false;
    for (int d : ready) found |= d == dev;
    if (!found) {
      for (const void* fn : kSplitKernels) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmem) != cudaSuccess ||
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
          (void)cudaGetLastError();
          return false;
        }
      }
      ready.push_back(dev);
    }
  }
  if (splits > 1) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = split_config(splits, splits, nullptr, attr);
    cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
    for (const void* fn : kSplitKernels) {
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess || clusters == 0) {
        (void)cudaGetLastError();
        return false;
      }
    }
  }
  memo.splits = splits;
  memo.chunk = chunk;
  memo.ok = true;
  *splits_out = splits;
  *chunk_out = chunk;
  return true;
}

}  // namespace

bool decode_tc_split_supported(int head_dim, int dtype, int units, int n) {
  int splits = 0, chunk = 0;
  return head_dim == kD && dtype == H2O_BF16 && n <= kMaxSplitsTc * kSplitMaxChunk && encode_fn() != nullptr &&
         plan_split(units, n, &splits, &chunk);
}

cudaError_t launch_decode_tc_split(const DecodeParams& dp, cudaStream_t stream) {
  TcSplitParams sp;
  cudaError_t e = fill_params(dp, sp.d);
  if (e != cudaSuccess) return e;
  if (!plan_split(dp.units, dp.n, &sp.splits, &sp.chunk)) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = split_config(dp.units, sp.splits, stream, attr);
  void* args[] = {&sp};
  return cudaLaunchKernelExC(&cfg, kSplitKernels[dp.policy != H2O_POLICY_H2O], args);
}

bool decode_tc_supported(int head_dim, int dtype, int budget) {
  return head_dim == kD && dtype == H2O_BF16 && budget <= kMaxTiles * kTileRows && encode_fn() != nullptr;
}

cudaError_t launch_decode_tc(const DecodeParams& dp, cudaStream_t stream) {
  TcDecodeParams p;
  cudaError_t fe = fill_params(dp, p);
  if (fe != cudaSuccess) return fe;

  static std::mutex mu;
  static std::vector<std::pair<int, int>> ready;  // (device, SM count)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto& d : ready)
      if (d.first == dev) sms = d.second;
    if (sms == 0) {
      for (const void* fn : kTcKernels) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
      }
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      ready.emplace_back(dev, sms);
    }
  }
  const int grid = balanced_grid(dp.units, sms);
  return launch_pdl(kTcKernels[dp.policy != H2O_POLICY_H2O], grid, kThreads, kSmem, stream, &p);
}

}  // namespace h2o
