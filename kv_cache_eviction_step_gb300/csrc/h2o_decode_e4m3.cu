// h2o_decode_e4m3.cu -- the fused H2O decode step (hot-path rows D1-D7) over a quantised cache: K/V
// rows stored as FP8 E4M3 codes with one float32 scale per row (the combination of H2O with KV-cache
// quantisation discussed in the H2O post §3.3), bf16 queries and new tokens, D = 128, budgets up to
// 512 slots. Both contractions run on the 5th-generation tensor cores straight from the 8-bit tiles
// (tcgen05.mma kind::f8f6f4), so a slot costs 2 x 128 bytes of K/V instead of 2 x 256.
//
// Per unit with n = min(t, budget) cached slots (code rows K8, V8, scales ks, vs):
//   D2  logits s_j = ks_j (q . K8_j) / sqrt(D). q is rescaled by 2^kq (max |q| into [128, 256)) and
//       split into two E4M3 rows, q' = q1 + q2, exact for bf16 values in the normal E4M3 range;
//       MMA M = 128 slots x N = 16 (q1, q2, zeros) x K = 128, the two columns summed in the
//       epilogue                                                           (H2O post §2.1.1)
//   D3  softmax over the n logits and the new token (bf16 k_new) on the epilogue warps, the logits
//       taken in log2 units so that each weight is one ex2
//   D4  o = (sum_j e_j vs_j V8_j) / l + p_new v_new: the weights w_j = e_j vs_j c (c = 2^kc puts the
//       largest scale below 256) split into three E4M3 rows (about 12 significant bits), V8^T read as
//       an MN-major operand straight from the TMA tile; MMA M = 128 (d) x N = 16 x K = slots
//   D5  scores[j] += p_j in fp32, p_j = e_j / l from the fp32 logits  (H2O post §2.2; 分析 §3.2)
//   D6  victim = argmin over slots with position <= t - k_local of the policy's key
//   D7  the new token quantised (scale = amax / 448, codes to nearest even, saturating) into the
//       victim slot with its score p_new and position                      (H2O post §2.3)
//
// Persistent like the bf16 kernel: each CTA walks units blockIdx.x, +gridDim.x, ... The first warps
// are the epilogue, four groups of four warps (one warp per TMEM lane quarter) that take units in
// turn, each with its own tensor-memory unit slot: with half the
// bytes per unit, one group's serial chain of reductions and barriers per unit would be slower than
// the memory system, and more warps hide more latency. The next warp is the producer (all lanes
// prepare the split query of each unit, lane 0 streams code tiles through a ring of 16 KB tiles in
// the order the tensor core consumes them), the last allocates tensor memory and issues the MMAs, the
// logits of unit k before the product of unit k - 2. Each group loads
// its units' tokens and state a unit ahead. All waits are bounded (mbar_wait); tensor memory is
// always freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kD = 128;                    // head dim of this path: one 128-byte code row
constexpr int kTileRows = 128;             // cache rows per tile (MMA M for the logits)
constexpr int kTileBytes = kTileRows * kD; // [128 rows x 128 codes]: 16 KB, 128-byte swizzle
constexpr int kMaxTiles = 4;               // budgets up to 512 slots
constexpr int kNRows = 16;                 // rows of the small operand (q split, or w split): MMA N
constexpr int kSmallBox = kNRows * 128;    // [16 rows x 128 codes]: 2 KB
constexpr int kGroupWarps = 4;             // one epilogue group: a warp per TMEM lane quarter
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr uint32_t kPvCol = 64;            // output accumulator column inside a unit slot
constexpr int kAlign = 1024;

// Epilogue groups take units in turn (unit k -> group and tensor-memory slot k % kGroups). One
// instantiation per largest cache served, NT 128-slot tiles (2 or 4): the smaller one sizes its
// buffers and register arrays for two tiles. Shared-memory offsets are from a 1024-aligned base.
constexpr int kGroups = 4;
template <int NT>
struct Layout {
  static constexpr int G = kGroups;
  static constexpr int kTiles = NT;                      // largest cache this instantiation serves
  static constexpr int kWBytes = kTiles * kSmallBox;     // w operand: 128 slots per 2 KB box
  static constexpr int kStages = 10;                     // streamed 16 KB tiles
  static constexpr int kEpiWarps = G * kGroupWarps;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static constexpr int kTmaWarp = kEpiWarps;
  static constexpr int kMmaWarp = kEpiWarps + 1;
  static constexpr uint32_t kTmemCols = 128 * G;     // one unit slot of 128 columns per group
  static constexpr int kQOff = kStages * kTileBytes;
  static constexpr int kWOff = kQOff + G * kSmallBox;
  static constexpr int kCtrlOff = kWOff + G * kWBytes;
  static constexpr int kCtrlBytes = 512 + 256 * G;   // mbarriers + TMEM slot, then per-group scratch
  static constexpr int kSmem = kCtrlOff + kCtrlBytes + kAlign;
};

struct Q8Params {
  CUtensorMap tm_k;        // K codes [units][budget][128] u8, box 128 x 128 x 1, 128-byte swizzle
  CUtensorMap tm_v;        // V codes, same
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  uint8_t* k_cache;
  uint8_t* v_cache;
  float* k_scale;          // [units][budget]
  float* v_scale;
  float* scores;
  int32_t* slot_pos;
  __nv_bfloat16* out;
  int32_t* evicted_slot;
  int32_t* evicted_pos;
  int32_t* err;
  int32_t units, budget, k_local, position, n, tiles;
  float scale;
  int32_t policy, n_sink, stride;
  int32_t early;  // the previous decode launch wrote none of this cache: tiles may load before the wait
};

// ---- PTX wrappers --------------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 128-byte-swizzled operand descriptor. K-major: rows of 128 bytes, 8-row groups `sbo` apart.
// MN-major: 128-byte MN groups `lbo` apart, 8-row K groups `sbo` apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// kind::f8f6f4 instruction descriptors: fp32 accumulate, E4M3 A and B (format code 0), M = 128,
// N = 16; K = 32 codes per instruction.
constexpr uint32_t kIdescQK = (1u << 4) | ((kNRows >> 3) << 17) | ((128 >> 4) << 24);  // A = K8 (K-major)
constexpr uint32_t kIdescPV = kIdescQK | (1u << 15);  // A = V8^T (MN-major), B = w (K-major)

__device__ __forceinline__ void mma8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
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

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float* v) {
  uint32_t r0, r1, r2, r3;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(taddr)
      : "memory");
  v[0] = __uint_as_float(r0);
  v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2);
  v[3] = __uint_as_float(r3);
}

// E4M3 code of x (to nearest, ties to even, saturating at +-448) and the value of a code.
__device__ __forceinline__ uint8_t e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_value(uint8_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(h));
}

// Power-of-two exponent that brings a positive maximum into [128, 256) (0 for an all-zero vector).
__device__ __forceinline__ int range_exp(float mx) { return mx > 0.f ? 7 - ilogbf(mx) : 0; }

// Byte offset of code j (0..127 within its 128-byte row) of row `row` in a 128-byte-swizzled box.
__device__ __forceinline__ int sw_offset(int row, int j) { return row * 128 + ((((j >> 4) ^ row) & 7) << 4) + (j & 15); }

template <bool kAnyPolicy, int kNT>
__global__ void __launch_bounds__(Layout<kNT>::kThreads, 1)
    h2o_decode_e4m3_kernel(const __grid_constant__ Q8Params p) {
  using L = Layout<kNT>;
  // Products issued kLag units behind the logits, so kLag + 1 epilogue groups run their softmax at
  // once; unit k's slot of tensor memory is reused by unit k + kGroups, whose logits follow product
  // k only if kLag < kGroups. The producer loads tiles in the order the tensor core consumes them
  // (unit k's K tiles, then unit k - kLag's V tiles), so ring slots free in order.
  constexpr int kLag = 2;
  static_assert(kLag < kGroups, "a unit's tensor-memory slot must be free before its logits");
  constexpr int kStages = L::kStages, kEpiWarps = L::kEpiWarps, kThreads = L::kThreads;
  constexpr int kTiles = L::kTiles, kWBytes = L::kWBytes;
  constexpr int kTmaWarp = L::kTmaWarp, kMmaWarp = L::kMmaWarp;
  constexpr uint32_t kTmemCols = L::kTmemCols;
  constexpr int kRingOff = 0, kQOff = L::kQOff, kWOff = L::kWOff, kCtrlOff = L::kCtrlOff;
  const int32_t policy = kAnyPolicy ? p.policy : static_cast<int32_t>(H2O_POLICY_H2O);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  unsigned char* ring = smem + kRingOff;
  (void)kEpiWarps;
  unsigned char* qbuf = smem + kQOff;
  unsigned char* wbuf = smem + kWOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCtrlOff);
  uint64_t* full = bars;                     // [kStages]
  uint64_t* empty = full + kStages;          // [kStages]
  uint64_t* q_full = empty + kStages;        // [kGroups] split query written
  uint64_t* s_full = q_full + kGroups;       // [kGroups] logits ready (and the q buffer free again)
  uint64_t* w_ready = s_full + kGroups;      // [kGroups] weights written
  uint64_t* o_full = w_ready + kGroups;      // [kGroups] output ready
  uint64_t* tm_free = o_full + kGroups;      // [kGroups] unit slot of tensor memory free again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tm_free + kGroups);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.tiles;
  const int n = p.n;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < kGroups; ++r) {
      mbar_init(&q_full[r], 1);
      mbar_init(&s_full[r], 1);
      mbar_init(&w_ready[r], 1);
      mbar_init(&o_full[r], 1);
      mbar_init(&tm_free[r], kGroupWarps);
    }
    fence_mbar_init();
  }
  // Rows 2..15 of the q operand and rows 3..15 of the w operand stay zero.
  for (int i = tid; i < (kGroups * kSmallBox + kGroups * kWBytes) / 16; i += kThreads)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
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
  // With p.early the producer's lane 0 loads the first ring tiles before the wait (the previous
  // launch on the stream writes none of this cache); everything else waits for the previous grid.
  const bool early_tiles = p.early != 0 && warp == kTmaWarp && lane == 0;
  if (!early_tiles) {
    pdl_wait();  // the previous step's cache, scales, scores and slot map are complete from here on
    pdl_launch_dependents();
  }

  if (warp == kTmaWarp) {
    // Producer: every lane splits four query elements (d = 4 lane .. 4 lane + 3); lane 0 streams.
    uint32_t g = 0;      // ring tiles issued (position in the consumption order)
    uint32_t g_pre = 0;  // tiles loaded before the wait
    if (early_tiles) {
      // The first unit's K tiles, the head of the consumption order (loading more of it before the
      // wait measured slower: it slows the previous launch's last units more than it saves).
      for (int t = 0; t < T; ++t, ++g_pre) {
        mbar_expect_tx(&full[g_pre], kTileBytes);
        tma_load_3d(ring + g_pre * kTileBytes, &p.tm_k, 0, t * kTileRows, blockIdx.x, &full[g_pre]);
      }
      pdl_wait();
      pdl_launch_dependents();
    }
    int k = 0;
    bool ok = true;
    uint2 qn = make_uint2(0, 0);  // the next unit's four bf16 query elements
    auto qload = [&](int u) {
      if (u < p.units) qn = *reinterpret_cast<const uint2*>(p.q + static_cast<size_t>(u) * kD + 4 * lane);
    };
    qload(blockIdx.x);
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++k) {
      const int r = k % kGroups;
      float x[4];
      {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&qn.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&qn.y);
        x[0] = __low2float(a);
        x[1] = __high2float(a);
        x[2] = __low2float(b);
        x[3] = __high2float(b);
      }
      qload(u + gridDim.x);
      float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const int kq = range_exp(mx);
      uint32_t w1 = 0, w2 = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float xs = ldexpf(x[i], kq);
        const uint8_t c1 = e4m3(xs);
        const uint8_t c2 = e4m3(xs - e4m3_value(c1));
        w1 |= static_cast<uint32_t>(c1) << (8 * i);
        w2 |= static_cast<uint32_t>(c2) << (8 * i);
      }
      if (lane == 0 && k >= kGroups)
        // the q buffer of this group is free once the logits of its previous unit are done
        ok = mbar_wait(&s_full[r], static_cast<uint32_t>(k / kGroups - 1) & 1u, p.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      unsigned char* qb = qbuf + r * kSmallBox;
      *reinterpret_cast<uint32_t*>(qb + sw_offset(0, 4 * lane)) = w1;
      *reinterpret_cast<uint32_t*>(qb + sw_offset(1, 4 * lane)) = w2;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&q_full[r]);
        // This unit's K tiles, then the V tiles of the unit kLag behind it (none for the first kLag).
        const int vu = u - kLag * static_cast<int>(gridDim.x);
        const int nt = k < kLag ? T : 2 * T;
        for (int i = 0; i < nt; ++i, ++g) {
          if (g < g_pre) continue;  // loaded before the wait
          const int s = static_cast<int>(g % kStages);
          if (g >= kStages && !mbar_wait(&empty[s], (g / kStages - 1) & 1u, p.err)) {
            ok = false;
            break;
          }
          const bool is_k = i < T;
          mbar_expect_tx(&full[s], kTileBytes);
          tma_load_3d(ring + s * kTileBytes, is_k ? &p.tm_k : &p.tm_v, 0, (is_k ? i : i - T) * kTileRows,
                      is_k ? u : vu, &full[s]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    // The V tiles of the last kLag units.
    for (int j = k - kLag < 0 ? 0 : k - kLag; lane == 0 && ok && j < k; ++j) {
      const int vu = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
      for (int t = 0; t < T; ++t, ++g) {
        if (g < g_pre) continue;  // loaded before the wait
        const int s = static_cast<int>(g % kStages);
        if (g >= kStages && !mbar_wait(&empty[s], (g / kStages - 1) & 1u, p.err)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&full[s], kTileBytes);
        tma_load_3d(ring + s * kTileBytes, &p.tm_v, 0, t * kTileRows, vu, &full[s]);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // The logits of unit k are issued before the product of unit k - kLag, so the epilogue finds
      // the next units' logits ready while the tensor core works on an earlier unit's output. Ring
      // tiles are consumed in the order the producer loads them.
      bool ok = true;
      uint32_t g = 0;  // ring tiles consumed
      auto wait_tile = [&](uint32_t pos) {
        return mbar_wait(&full[pos % kStages], (pos / kStages) & 1u, p.err);
      };
      auto product = [&](int k) {  // D4 of the k-th unit: o = V8^T w
        const int r = k % kGroups;
        const uint32_t ph = static_cast<uint32_t>(k / kGroups) & 1u;
        const uint32_t slot = tmem + static_cast<uint32_t>(r) * 128;
        if (!mbar_wait(&w_ready[r], ph, p.err)) return false;
        tc_fence_after();
        const uint32_t w_base = smem_u32(wbuf + r * kWBytes);
        for (int t = 0; t < T; ++t) {
          const uint32_t pos = g++;
          if (!wait_tile(pos)) return false;
          tc_fence_after();
          const uint64_t a0 = sw128_desc(smem_u32(ring + (pos % kStages) * kTileBytes), kTileBytes, 1024);
          const uint64_t b0 = sw128_desc(w_base + t * kSmallBox, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kTileRows / 32; ++kk) {
            // V8^T as MN-major A: the 128 codes of d form one MN group; 32 slots (four 8-row groups
            // of 1024 bytes) per instruction. w as K-major B: 128 slots per 2 KB box.
            mma8(slot + kPvCol, a0 + static_cast<uint64_t>(kk * (4096 >> 4)), b0 + static_cast<uint64_t>(kk * (32 >> 4)),
                 kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[pos % kStages]);
        }
        mma_commit(&o_full[r]);
        return true;
      };
      int k = 0;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++k) {
        const int r = k % kGroups;
        const uint32_t ph = static_cast<uint32_t>(k / kGroups) & 1u;
        const uint32_t slot = tmem + static_cast<uint32_t>(r) * 128;
        if (k >= kGroups && !mbar_wait(&tm_free[r], ph ^ 1u, p.err)) break;
        if (!mbar_wait(&q_full[r], ph, p.err)) break;
        tc_fence_after();
        const uint32_t q_base = smem_u32(qbuf + r * kSmallBox);
        // D2: logits of each 128-row K tile into columns 16 t, 16 t + 1 of this unit's slot.
        for (int t = 0; t < T; ++t) {
          const uint32_t pos = g++;
          if (!wait_tile(pos)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a0 = sw128_desc(smem_u32(ring + (pos % kStages) * kTileBytes), 16, 1024);
          const uint64_t b0 = sw128_desc(q_base, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 32; ++kk)  // 32 codes = 32 bytes of each row per instruction
            mma8(slot + 16 * t, a0 + static_cast<uint64_t>(kk * (32 >> 4)), b0 + static_cast<uint64_t>(kk * (32 >> 4)),
                 kIdescQK, kk > 0 ? 1u : 0u);
          mma_commit(&empty[pos % kStages]);
        }
        if (!ok) break;
        mma_commit(&s_full[r]);
        if (k >= kLag && !product(k - kLag)) {
          ok = false;
          break;
        }
      }
      for (int j = k - kLag < 0 ? 0 : k - kLag; ok && j < k; ++j) ok = product(j);
    }
    __syncwarp();
  } else {
    // Epilogue: kGroups groups of four warps take units in turn (group g the units k = g,
    // g + kGroups, ..., which use tensor-memory slot g). Thread (warp, lane) of a group owns slot 128 t + 32 (warp % 4)
    // + lane of every tile t, and output element d = its index in the group.
    const int grp = warp / kGroupWarps;
    const int gtid = tid - grp * kGroupThreads;
    const int gwarp = warp % kGroupWarps;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(gwarp * 32) << 16);
    // Per-group reduction scratch, one array per round, so that each round needs one barrier: a
    // round's array is rewritten only after the group has passed the next rounds' barriers.
    float* red = reinterpret_cast<float*>(smem + kCtrlOff + 512 + grp * 256);    // s_new partials [4]
    float* r1 = red + 4;                                                          // maxima [4][4]
    float* rm = red + 20;                                                         // logit max [4]
    float* rl = red + 24;                                                         // sums [4]
    unsigned long long* kred = reinterpret_cast<unsigned long long*>(smem + kCtrlOff + 640 + grp * 256);
    int32_t* sred = reinterpret_cast<int32_t*>(smem + kCtrlOff + 704 + grp * 256);
    auto gsync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(3 + grp), "n"(kGroupThreads) : "memory"); };
    const int32_t last_candidate = p.position - p.k_local;
    const bool cache_full = n == p.budget;
    bool ok = true;
    const int ustep = kGroups * gridDim.x;
    // This thread's w entries (slot gtid of each tile) in rows 0..2 of the swizzled w boxes.
    const int woff0 = sw_offset(0, gtid), woff1 = sw_offset(1, gtid), woff2 = sw_offset(2, gtid);
    // A unit's new token and state are loaded one unit (of this group) ahead.
    __nv_bfloat16 nq = __float2bfloat16_rn(0.f), nkn = nq, nvn = nq;
    float nsc[kTiles], nks[kTiles], nvs[kTiles];
    int32_t nsp[kTiles];
    auto prefetch = [&](int u) {
      if (u >= p.units) return;
      const size_t row0 = static_cast<size_t>(u) * p.budget;
      const size_t ud = static_cast<size_t>(u) * kD + gtid;
      nq = p.q[ud];
      nkn = p.k_new[ud];
      nvn = p.v_new[ud];
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const int j = t * kTileRows + gtid;
        const bool valid = t < T && j < n;
        nsc[t] = valid ? p.scores[row0 + j] : 0.f;
        nsp[t] = valid ? p.slot_pos[row0 + j] : 0;
        nks[t] = valid ? p.k_scale[row0 + j] : 0.f;
        nvs[t] = valid ? p.v_scale[row0 + j] : 0.f;
      }
    };
    prefetch(blockIdx.x + grp * gridDim.x);
    for (int u = blockIdx.x + grp * gridDim.x, k = grp; u < p.units && ok; u += ustep, k += kGroups) {
      const int r = grp;  // == k % kGroups
      const uint32_t ph = static_cast<uint32_t>(k / kGroups) & 1u;
      const size_t row0 = static_cast<size_t>(u) * p.budget;
      const size_t ud = static_cast<size_t>(u) * kD + gtid;
      const float qd = __bfloat162float(nq);
      const float knf = __bfloat162float(nkn), vnf = __bfloat162float(nvn);
      float sc[kTiles], ks[kTiles], vs[kTiles];
      int32_t sp[kTiles];
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        sc[t] = nsc[t];
        sp[t] = nsp[t];
        ks[t] = nks[t];
        vs[t] = nvs[t];
      }
      prefetch(u + ustep);
      // First reduction (one barrier): s_new partial, max |q| (the producer's split exponent), the largest
      // value scale, and the new row's max |k_new|, |v_new| for its quantisation.
      float part = qd * knf;
      float qm = fabsf(qd), vsm = vs[0];
#pragma unroll
      for (int t = 1; t < kTiles; ++t) vsm = fmaxf(vsm, vs[t]);
      float km = fabsf(knf), vm = fabsf(vnf);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        part += __shfl_xor_sync(0xffffffffu, part, off);
        qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, off));
        vsm = fmaxf(vsm, __shfl_xor_sync(0xffffffffu, vsm, off));
        km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, off));
        vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
      }
      if (lane == 0) {
        red[gwarp] = part;
        r1[gwarp] = qm;
        r1[4 + gwarp] = vsm;
        r1[8 + gwarp] = km;
        r1[12 + gwarp] = vm;
      }

      if (!mbar_wait(&s_full[r], ph, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      gsync();  // first-reduction partials visible
      const float s_new = (red[0] + red[1] + red[2] + red[3]) * p.scale;
      const float qmax = fmaxf(fmaxf(r1[0], r1[1]), fmaxf(r1[2], r1[3]));
      const float vsmax = fmaxf(fmaxf(r1[4], r1[5]), fmaxf(r1[6], r1[7]));
      const float kamax = fmaxf(fmaxf(r1[8], r1[9]), fmaxf(r1[10], r1[11]));
      const float vamax = fmaxf(fmaxf(r1[12], r1[13]), fmaxf(r1[14], r1[15]));
      // Logits: the tensor core's sum times ks_j 2^-kq (1/sqrt(D)).
      const float qinv = ldexpf(1.f, -range_exp(qmax)) * p.scale;
      float s[kTiles];
      float m = s_new;
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        s[t] = -INFINITY;
        if (t < T) {
          float c0, c1;
          tmem_ld2(lane_base + r * 128 + 16 * t, c0, c1);
          if (t * kTileRows + gtid < n) s[t] = (c0 + c1) * (qinv * ks[t]);
        }
        m = fmaxf(m, s[t]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) rm[gwarp] = m;
      gsync();
      m = fmaxf(fmaxf(rm[0], rm[1]), fmaxf(rm[2], rm[3]));
      // D3 + D4 weights: w_j = e_j vs_j 2^kc split into three E4M3 rows of the w operand.
      const float cw = ldexpf(1.f, range_exp(vsmax));
      float e[kTiles];
      float lsum = 0.f;
      unsigned char* wb = wbuf + r * kWBytes;
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        if (t < T) {
          e[t] = expf(s[t] - m);  // accurate exp (the score increments); 0 for slots past n
          lsum += e[t];
          const float w = e[t] * vs[t] * cw;
          const uint8_t c1 = e4m3(w);
          const float r1v = w - e4m3_value(c1);
          const uint8_t c2 = e4m3(r1v);
          const uint8_t c3 = e4m3(r1v - e4m3_value(c2));
          unsigned char* box = wb + t * kSmallBox;
          box[woff0] = c1;
          box[woff1] = c2;
          box[woff2] = c3;
        } else {
          e[t] = 0.f;
        }
      }
      fence_async_smem();
      const float w_new = expf(s_new - m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      if (lane == 0) rl[gwarp] = lsum;
      gsync();  // every thread's w entries are written (and fenced), and the sums
      if (gtid == 0) mbar_arrive(&w_ready[r]);
      const float l = rl[0] + rl[1] + rl[2] + rl[3] + w_new;

      // D5 + D6 while the tensor core computes the output.
      unsigned long long best = ~0ull;
      int32_t best_slot = -1;
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        if (t < T && t * kTileRows + gtid < n) {
          const float pr = e[t] / l;
          sc[t] = policy == H2O_POLICY_TOPK ? pr : sc[t] + pr;  // Top-K: this step's weight
          bool cand = false;
          const unsigned long long key =
              policy_key(policy, sc[t], sp[t], last_candidate, p.n_sink, p.stride, &cand);
          if (cache_full && cand && key < best) {
            best = key;
            best_slot = t * kTileRows + gtid;
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
          kred[gwarp] = best;
          sred[gwarp] = best_slot;
        }
        gsync();
        vkey = kred[0];
        victim = sred[0];
#pragma unroll
        for (int w = 1; w < kGroupWarps; ++w)
          if (kred[w] < vkey) {
            vkey = kred[w];
            victim = sred[w];
          }
        if (gtid == 0 && victim < 0) atomicCAS(p.err, H2O_DEVERR_NONE, H2O_DEVERR_NO_CANDIDATE);
      }

      // D4 result: o[d] = (sum_j w_j V8_j[d] / 2^kc + w_new v_new[d]) / l.
      if (!mbar_wait(&o_full[r], ph, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float c[4];
      tmem_ld4(lane_base + r * 128 + kPvCol, c);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tm_free[r]);
      p.out[ud] = __float2bfloat16_rn(((c[0] + c[1] + c[2]) / cw + w_new * vnf) / l);

      // D7: scores back, the new token quantised into its slot, eviction indices.
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const int j = t * kTileRows + gtid;
        if (t < T && j < n) p.scores[row0 + j] = (j == victim) ? p_new : sc[t];
      }
      const int32_t target = cache_full ? victim : n;
      if (target >= 0) {
        const float k_s = kamax > 0.f ? kamax / 448.f : 1.f;
        const float v_s = vamax > 0.f ? vamax / 448.f : 1.f;
        p.k_cache[(row0 + target) * kD + gtid] = e4m3(knf / k_s);
        p.v_cache[(row0 + target) * kD + gtid] = e4m3(vnf / v_s);
        if (gtid == 0) {
          p.k_scale[row0 + target] = k_s;
          p.v_scale[row0 + target] = v_s;
          p.slot_pos[row0 + target] = p.position;
          if (!cache_full) p.scores[row0 + target] = p_new;
        }
      }
      if (gtid == 0) {
        p.evicted_slot[u] = cache_full ? victim : -1;
        p.evicted_pos[u] = (cache_full && victim >= 0) ? static_cast<int32_t>(vkey & 0xffffffffu) : -1;
      }
    }
  }

  // Tensor memory is freed by the warp that allocated it, after every reader is done.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
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

// [units][budget][128] codes as a 3-D tensor; one box = 128 codes x 128 rows x 1 unit, 128-byte
// swizzle; rows past the budget read as zeros.
bool encode_codes(CUtensorMap* map, const void* base, int units, int budget) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {kD, static_cast<cuuint64_t>(budget), static_cast<cuuint64_t>(units)};
  const cuuint64_t strides[2] = {kD, static_cast<cuuint64_t>(budget) * kD};
  const cuuint32_t box[3] = {kD, kTileRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MapCache {
  const void *k = nullptr, *v = nullptr;
  int units = -1, budget = -1;
  CUtensorMap tm_k, tm_v;
};

// [groups == 4][any policy]
const void* const kKernels[2][2] = {
    {reinterpret_cast<const void*>(h2o_decode_e4m3_kernel<false, 2>),
     reinterpret_cast<const void*>(h2o_decode_e4m3_kernel<true, 2>)},
    {reinterpret_cast<const void*>(h2o_decode_e4m3_kernel<false, 4>),
     reinterpret_cast<const void*>(h2o_decode_e4m3_kernel<true, 4>)}};

}  // namespace

// Shapes this kernel serves (a driver without tensor-map encoding fails the launch instead).
bool decode_e4m3_supported(int head_dim, int dtype, int budget) {
  return head_dim == kD && dtype == H2O_BF16 && budget <= kMaxTiles * kTileRows;
}

cudaError_t launch_decode_e4m3(const DecodeParams& dp, cudaStream_t stream) {
  Q8Params p;
  thread_local MapCache mc;
  if (mc.k != dp.k_cache || mc.units != dp.units || mc.budget != dp.budget) {
    if (!encode_codes(&mc.tm_k, dp.k_cache, dp.units, dp.budget)) return cudaErrorInvalidValue;
    mc.k = dp.k_cache;
  }
  if (mc.v != dp.v_cache || mc.units != dp.units || mc.budget != dp.budget) {
    if (!encode_codes(&mc.tm_v, dp.v_cache, dp.units, dp.budget)) return cudaErrorInvalidValue;
    mc.v = dp.v_cache;
  }
  mc.units = dp.units;
  mc.budget = dp.budget;
  p.tm_k = mc.tm_k;
  p.tm_v = mc.tm_v;
  p.q = static_cast<const __nv_bfloat16*>(dp.q);
  p.k_new = static_cast<const __nv_bfloat16*>(dp.k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(dp.v_new);
  p.k_cache = static_cast<uint8_t*>(dp.k_cache);
  p.v_cache = static_cast<uint8_t*>(dp.v_cache);
  p.k_scale = dp.k_scale;
  p.v_scale = dp.v_scale;
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
      for (int t4 = 0; t4 < 2; ++t4)
        for (int any = 0; any < 2; ++any) {
          e = cudaFuncSetAttribute(kKernels[t4][any], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   t4 ? Layout<4>::kSmem : Layout<2>::kSmem);
          if (e != cudaSuccess) return e;
        }
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      ready.emplace_back(dev, sms);
    }
  }
  const int grid = balanced_grid(dp.units, sms);
  const bool any = dp.policy != H2O_POLICY_H2O;
  if (p.tiles <= 2) return launch_pdl(kKernels[0][any], grid, Layout<2>::kThreads, Layout<2>::kSmem, stream, &p);
  return launch_pdl(kKernels[1][any], grid, Layout<4>::kThreads, Layout<4>::kSmem, stream, &p);
}

}  // namespace h2o
