// h2o_prefill_tc.cu -- prefill score pass (hot-path rows P1-P2) for bf16 on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory, operands staged by TMA).
//
//   P1  m_i = max_{j<=i} s_ij and l_i = sum_{j<=i} exp(s_ij - m_i), s_ij = (q_i . k_j) / sqrt(D)
//       (causal Softmax(QK^T/sqrt(d)): H2O post §2.1.1)
//   P2  c_j = sum_{i>=j} exp(s_ij - m_i) / l_i: the attention each prompt token accumulates over the
//       prompt (H2O post §2.1.2 / §2.2; "H2O Heavy-Hitter Oracle 分析" §3.1)
//
//   P1+ with an output tensor, the row-stats pass is also the prompt's attention forward:
//       o_i = sum_{j<=i} exp(s_ij - m_i) / l_i v_j, sharing the logits and exponentials with P1.
//
// Both passes are the same kernel shape: one CTA keeps a 128-row "resident" tile of one operand and
// streams 128-row tiles of the other, so that S = A B^T lands in tensor memory with one TMEM lane
// (and so one epilogue thread) per resident row:
//   row stats   resident = Q tile i, streamed = K tiles 0..i    -> rows are queries, reduce along j
//   column sums resident = K tile j, streamed = Q tiles j..end  -> rows are keys, reduce along i,
//               recomputing S instead of storing the P x P probabilities.
// The output variant streams V tiles beside the K tiles; the epilogue writes exp(s - m) of each tile
// as a bf16 128 x 128 probability tile in shared memory (K-major, 128-byte swizzle) and the tensor
// core accumulates O += P V in a third tensor-memory region, with V read as an MN-major operand
// straight from its TMA tile. The running maximum is updated lazily: O and l are rescaled only when a
// tile's maximum exceeds the one in use by more than kLazyMax, so the probabilities stay below
// e^kLazyMax and a rescale (tcgen05.ld / st of the row's O) is rare.
// Warp roles: warps 0-3 are the epilogue (tcgen05.ld of their 32 TMEM lanes, masking, exp, running
// reductions), warp 4 issues the TMA tensor loads (128-byte swizzle, two 64-column boxes per tile for
// D = 128), warp 5 allocates tensor memory and one of its lanes issues tcgen05.mma (M = N = 128,
// K = 16 per instruction, bf16 x bf16 -> fp32) into two alternating 128-column accumulators, so the
// tensor core fills one while the epilogue drains the other. mbarriers link the roles: TMA ->
// b_full -> MMA -> (tcgen05.commit) b_empty / acc_full -> epilogue -> acc_empty -> MMA. Every wait is
// bounded (see mbar_wait); a CTA that gives up still frees its tensor memory before it exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kTile = 128;                 // rows per operand tile (TMEM lanes / MMA M and N)
constexpr int kBoxCols = 64;               // bf16 elements in one 128-byte swizzle row
constexpr int kBoxBytes = kTile * 128;     // one [128 rows x 64 cols] bf16 box: 16 KB
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kEpiWarps + 2);
constexpr int kTmaWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr uint32_t kTmemCols = 2 * kTile;  // two fp32 128 x 128 accumulators
constexpr int kCtrlBytes = 256;            // mbarriers + TMEM address slot
constexpr int kAlign = 1024;               // 128-byte swizzle atoms repeat every 1024 bytes
constexpr uint32_t kOCol = 2 * kTile;       // output variant: O accumulator columns [256, 256 + D)
constexpr uint32_t kTmemColsOut = 512;
constexpr int kPBytes = 2 * kBoxBytes;     // 128 x 128 bf16 probability tile (two 64-key boxes)
constexpr float kLazyMax = 8.f;            // rescale O only when the max grows by more than this

struct TcParams {
  CUtensorMap tm_a;        // resident operand: Q (row stats) or K (column sums), [units][P][D]
  CUtensorMap tm_b;        // streamed operand: K (row stats) or Q (column sums)
  CUtensorMap tm_v;        // output variant: V, [units][P][D]
  __nv_bfloat16* out;      // output variant: [units][P][D]
  const float* row_max_in; // column sums: m_i from the row-stats pass, [units][P]
  const float* row_sum_in; // column sums: l_i
  float* row_max;          // row stats output
  float* row_sum;
  float* colsum;           // column sums output
  int32_t* err;
  int32_t P;
  int32_t tiles;           // ceil(P / 128)
  float scale;
  int32_t last_row_only;   // column sums: only the last query's weight (Top-K prefill)
};

template <int D>
struct TcShape {
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStages = D == 128 ? 2 : 4;  // streamed-tile ring depth
  static constexpr int kSmem = (1 + kStages) * kTileBytes + kCtrlBytes + 4 * kTile * 4 + kAlign;
  // output variant: a V ring beside the K ring and the probability tile
  static constexpr int kSmemOut = (1 + 2 * kStages) * kTileBytes + kPBytes + kCtrlBytes + 4 * kTile * 4 + kAlign;
};

// ---- tcgen05 / TMA wrappers --------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with 128-byte swizzle:
// rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), descriptor version 1,
// layout type 2 = SWIZZLE_128B. Advancing along K inside the 128-byte row moves the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;              // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;      // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;              // descriptor version
  d |= static_cast<uint64_t>(2) << 61;              // SWIZZLE_128B
  return d;
}

// Descriptor of an MN-major operand tile written by TMA with 128-byte swizzle (V as the B operand of
// O += P V): 64-element MN groups `lbo` bytes apart (one box), 8-row K groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major, M = N = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kTile >> 3) << 17) |
                            (static_cast<uint32_t>(kTile >> 4) << 24);
// O += P V: A = P (K-major), B = V (MN-major, bit 16), M = 128 queries, N = D.
template <int D>
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                              (static_cast<uint32_t>(D >> 3) << 17) | (static_cast<uint32_t>(kTile >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate,
                                         uint32_t idesc = kIdesc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 accumulator columns of this warp's 32 TMEM lanes (one row per thread). The
// load and its wait sit in one asm statement, so no use of the registers can move above the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]);
}

// Store 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per thread) and wait.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Generic-proxy shared-memory writes made visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

template <int D, bool kColsum, bool kOut>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  static_assert(!(kColsum && kOut), "the output is produced by the row-statistics pass");
  using S = TcShape<D>;
  constexpr int kStages = S::kStages;
  constexpr int kRing = kStages * S::kTileBytes;
  constexpr int kCtrlOff = kOut ? S::kTileBytes + 2 * kRing + kPBytes : S::kTileBytes + kRing;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  unsigned char* sa = smem;                            // resident tile
  unsigned char* sb = smem + S::kTileBytes;            // streamed-tile ring
  unsigned char* sv = sb + kRing;                      // output variant: V-tile ring
  unsigned char* sp = sv + kRing;                      // output variant: probability tile
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + kCtrlOff);
  uint64_t* b_full = a_full + 1;
  uint64_t* b_empty = b_full + kStages;
  uint64_t* acc_full = b_empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* v_full = acc_empty + 2;                    // output variant only
  uint64_t* v_empty = v_full + kStages;
  uint64_t* p_full = v_empty + kStages;                // the epilogue wrote this tile's P
  uint64_t* o_prog = p_full + 1;                       // one completion per O += P V
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_prog + 1);
  // column sums: m_i and 1/l_i of the current query tile, double-buffered by tile parity
  float* sm_m = reinterpret_cast<float*>(smem + kCtrlOff + kCtrlBytes);
  float* sm_il = sm_m + 2 * kTile;
  constexpr uint32_t kCols = kOut ? kTmemColsOut : kTmemCols;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.x;
  const int at = blockIdx.y;                           // resident tile index
  // streamed tiles [t_begin, t_end); the last-row variant only needs the tile holding query P-1
  const int t_begin = kColsum ? (p.last_row_only ? p.tiles - 1 : at) : 0;
  const int t_end = kColsum ? p.tiles : at + 1;
  const int nt = t_end - t_begin;
  const int P = p.P;

  if (tid == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
      if constexpr (kOut) {
        mbar_init(&v_full[s], 1);
        mbar_init(&v_empty[s], 1);
      }
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    if constexpr (kOut) {
      mbar_init(p_full, kEpiWarps);
      mbar_init(o_prog, 1);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      mbar_expect_tx(a_full, S::kTileBytes);
      for (int b = 0; b < S::kBoxes; ++b)
        tma_load_3d(sa + b * kBoxBytes, &p.tm_a, b * kBoxCols, at * kTile, unit, a_full);
      for (int t = 0; t < nt; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !mbar_wait(&b_empty[s], static_cast<uint32_t>(t / kStages - 1) & 1u, p.err)) break;
        mbar_expect_tx(&b_full[s], S::kTileBytes);
        for (int b = 0; b < S::kBoxes; ++b)
          tma_load_3d(sb + s * S::kTileBytes + b * kBoxBytes, &p.tm_b, b * kBoxCols, (t_begin + t) * kTile,
                      unit, &b_full[s]);
        if constexpr (kOut) {
          if (t >= kStages && !mbar_wait(&v_empty[s], static_cast<uint32_t>(t / kStages - 1) & 1u, p.err)) break;
          mbar_expect_tx(&v_full[s], S::kTileBytes);
          for (int b = 0; b < S::kBoxes; ++b)
            tma_load_3d(sv + s * S::kTileBytes + b * kBoxBytes, &p.tm_v, b * kBoxCols, t * kTile, unit, &v_full[s]);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && mbar_wait(a_full, 0, p.err)) {
      const uint32_t a_base = smem_u32(sa);
      // Logits of tile t, then (output variant) O += P V of tile t-1 once the epilogue has written
      // its probabilities, so the epilogue of tile t overlaps the product of tile t-1.
      for (int t = 0; t < nt + (kOut ? 1 : 0); ++t) {
        if (t < nt) {
          const int s = t % kStages;
          const int a = t & 1;
          if (!mbar_wait(&b_full[s], static_cast<uint32_t>(t / kStages) & 1u, p.err)) break;
          if (t >= 2 && !mbar_wait(&acc_empty[a], static_cast<uint32_t>(t / 2 - 1) & 1u, p.err)) break;
          tc_fence_after();
          const uint32_t b_base = smem_u32(sb + s * S::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;  // 16 bf16 = 32 bytes per step
            mma_bf16(tmem + a * kTile, sw128_desc(a_base + off), sw128_desc(b_base + off), kk > 0 ? 1u : 0u);
          }
          mma_commit(&b_empty[s]);   // the streamed tile may be overwritten once these MMAs finish
          mma_commit(&acc_full[a]);  // and the accumulator may be read
        }
        if constexpr (kOut) {
          if (t >= 1) {
            const int u = t - 1;
            const int s = u % kStages;
            if (!mbar_wait(p_full, static_cast<uint32_t>(u) & 1u, p.err)) break;
            if (!mbar_wait(&v_full[s], static_cast<uint32_t>(u / kStages) & 1u, p.err)) break;
            tc_fence_after();
            const uint32_t p_base = smem_u32(sp);
            const uint32_t v_base = smem_u32(sv + s * S::kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              // P: K-major, 64 keys per box, 32 bytes per 16-key step; V: MN-major, 16 key rows of
              // 128 bytes per step, 64-column groups one box apart.
              const uint32_t off_p = (kk / 4) * kBoxBytes + (kk % 4) * 32;
              mma_bf16(tmem + kOCol, sw128_desc(p_base + off_p), sw128_desc_mn(v_base + kk * 2048, kBoxBytes),
                       (u > 0 || kk > 0) ? 1u : 0u, kIdescPV<D>);
            }
            mma_commit(&v_empty[s]);
            mma_commit(o_prog);  // P may be overwritten, O may be read or rescaled
          }
        }
      }
    }
    __syncwarp();
  } else {
    // Epilogue: thread r owns resident row `row` (a query for row stats, a key for column sums).
    const int r = tid;
    const int row = at * kTile + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const size_t ubase = static_cast<size_t>(unit) * P;
    float m = -INFINITY, l = 0.f, c = 0.f;
    float m_use = -INFINITY;  // output variant: the maximum the probabilities and O are taken against
    bool ok = true;
    float m_next = 0.f, il_next = 0.f;  // column sums: the next query tile's statistics, prefetched
    if constexpr (kColsum) {
      const int i = t_begin * kTile + r;
      if (i < P) {
        m_next = p.row_max_in[ubase + i];
        il_next = 1.f / p.row_sum_in[ubase + i];
      }
    }
    for (int t = 0; t < nt; ++t) {
      const int a = t & 1;
      const int col0 = (t_begin + t) * kTile;  // first key (row stats) or query (column sums)
      // Tiles strictly off the diagonal and inside the prompt need no causal or tail mask.
      const bool interior = (kColsum ? (t_begin + t > at) : (t_begin + t < at)) && col0 + kTile <= P &&
                            !p.last_row_only;
      const float* tm = sm_m + (t & 1) * kTile;
      const float* til = sm_il + (t & 1) * kTile;
      if constexpr (kColsum) {
        sm_m[(t & 1) * kTile + r] = m_next;
        sm_il[(t & 1) * kTile + r] = il_next;
        if (t + 1 < nt) {
          const int i = col0 + kTile + r;
          m_next = 0.f;
          il_next = 0.f;
          if (i < P) {
            m_next = p.row_max_in[ubase + i];
            il_next = 1.f / p.row_sum_in[ubase + i];
          }
        }
        epilogue_sync();  // this tile's statistics are visible (the buffer's previous readers finished
                          // before the last iteration's barrier)
      }
      if (ok) ok = mbar_wait(&acc_full[a], static_cast<uint32_t>(t / 2) & 1u, p.err);
      tc_fence_after();
      if constexpr (kOut) {
        // Sweep 1: the tile's maximum; the maximum in use moves only when exceeded by > kLazyMax.
        float tmax = -INFINITY;
#pragma unroll 1
        for (int ch = 0; ch < kTile / 32; ++ch) {
          float v[32];
          tmem_ld32(lane_addr + a * kTile + ch * 32, v);
          const int x0 = col0 + ch * 32;
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const bool valid = interior || (x0 + x <= row && x0 + x < P);
            tmax = fmaxf(tmax, valid ? v[x] * p.scale : -INFINITY);
          }
        }
        m = fmaxf(m, tmax);
        float alpha = 1.f;
        if (tmax > m_use + kLazyMax) {
          alpha = expf(m_use - tmax);  // 0 on the first tile
          l *= alpha;
          m_use = tmax;
        }
        // O += P V of the previous tile has finished: P may be overwritten and O rescaled.
        if (t > 0 && ok) ok = mbar_wait(o_prog, static_cast<uint32_t>(t - 1) & 1u, p.err);
        tc_fence_after();
        if (t > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float o[32];
            tmem_ld32(lane_addr + kOCol + ch * 32, o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            tmem_st32(lane_addr + kOCol + ch * 32, o);
          }
        }
        // Sweep 2: probabilities against m_use into row r of the P tile (bf16, 128-byte swizzle).
#pragma unroll 1
        for (int ch = 0; ch < kTile / 32; ++ch) {
          float v[32];
          tmem_ld32(lane_addr + a * kTile + ch * 32, v);
          const int x0 = col0 + ch * 32;
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const bool valid = interior || (x0 + x <= row && x0 + x < P);
            v[x] = valid ? expf(v[x] * p.scale - m_use) : 0.f;
            l += v[x];
          }
          unsigned char* box = sp + (ch >> 1) * kBoxBytes + r * 128;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int chunk = (ch & 1) * 4 + c4;  // 16-byte chunk (8 keys) within the 128-byte row
            uint4 w;
            w.x = pack_bf16(v[c4 * 8 + 0], v[c4 * 8 + 1]);
            w.y = pack_bf16(v[c4 * 8 + 2], v[c4 * 8 + 3]);
            w.z = pack_bf16(v[c4 * 8 + 4], v[c4 * 8 + 5]);
            w.w = pack_bf16(v[c4 * 8 + 6], v[c4 * 8 + 7]);
            *reinterpret_cast<uint4*>(box + ((chunk ^ (r & 7)) << 4)) = w;
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(p_full);
          mbar_arrive(&acc_empty[a]);
        }
      } else {
#pragma unroll 1
        for (int ch = 0; ch < kTile / 32; ++ch) {
          float v[32];
          tmem_ld32(lane_addr + a * kTile + ch * 32, v);
          const int x0 = col0 + ch * 32;
          if constexpr (!kColsum) {
            // running max / normaliser over the causal keys j <= row of this chunk
            float cm = -INFINITY;
            if (interior) {
#pragma unroll
              for (int x = 0; x < 32; ++x) {
                v[x] *= p.scale;
                cm = fmaxf(cm, v[x]);
              }
            } else {
#pragma unroll
              for (int x = 0; x < 32; ++x) {
                const int j = x0 + x;
                v[x] = (j <= row && j < P) ? v[x] * p.scale : -INFINITY;
                cm = fmaxf(cm, v[x]);
              }
            }
            if (cm > m) {
              l *= expf(m - cm);
              m = cm;
            }
            if (cm != -INFINITY) {
#pragma unroll
              for (int x = 0; x < 32; ++x) l += expf(v[x] - m);
            }
          } else {
            // probabilities of the queries i >= row of this chunk that attend this key
            if (interior) {
#pragma unroll
              for (int x = 0; x < 32; ++x) c += expf(v[x] * p.scale - tm[ch * 32 + x]) * til[ch * 32 + x];
            } else if (p.last_row_only) {
#pragma unroll
              for (int x = 0; x < 32; ++x)
                if (x0 + x == P - 1 && row <= P - 1) c += expf(v[x] * p.scale - tm[ch * 32 + x]) * til[ch * 32 + x];
            } else {
#pragma unroll
              for (int x = 0; x < 32; ++x) {
                const int i = x0 + x;
                if (i >= row && i < P) c += expf(v[x] * p.scale - tm[ch * 32 + x]) * til[ch * 32 + x];
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
      }
    }
    if constexpr (kOut) {
      // The last O += P V has finished: normalise the row and write it (bf16).
      if (ok) ok = mbar_wait(o_prog, static_cast<uint32_t>(nt - 1) & 1u, p.err);
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = p.out + (ubase + static_cast<size_t>(row)) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float o[32];
        tmem_ld32(lane_addr + kOCol + ch * 32, o);
        if (row < P) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint4 w;
            w.x = pack_bf16(o[c4 * 8 + 0] * inv_l, o[c4 * 8 + 1] * inv_l);
            w.y = pack_bf16(o[c4 * 8 + 2] * inv_l, o[c4 * 8 + 3] * inv_l);
            w.z = pack_bf16(o[c4 * 8 + 4] * inv_l, o[c4 * 8 + 5] * inv_l);
            w.w = pack_bf16(o[c4 * 8 + 6] * inv_l, o[c4 * 8 + 7] * inv_l);
            *reinterpret_cast<uint4*>(orow + ch * 32 + c4 * 8) = w;
          }
        }
      }
      l *= expf(m_use - m);  // the normaliser against the true maximum, for the column-sum pass
    }
    if (row < P) {
      if constexpr (!kColsum) {
        p.row_max[ubase + row] = m;
        p.row_sum[ubase + row] = l;
      } else {
        p.colsum[ubase + row] = c;
      }
    }
  }

  // Tensor memory is freed by the warp that allocated it, after every reader is done.
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

// [units][P][D] bf16 viewed as a 3-D tensor; boxes of 64 columns x 128 rows x 1 unit, 128-byte
// swizzle; rows past P read as zeros.
bool encode_operand(CUtensorMap* map, const void* base, int units, int P, int D) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(P),
                              static_cast<cuuint64_t>(units)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(P) * D * 2};
  const cuuint32_t box[3] = {kBoxCols, kTile, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kColsum, bool kOut = false>
cudaError_t launch_pass(const TcParams& p, int units, cudaStream_t s) {
  auto kernel = prefill_tc_kernel<D, kColsum, kOut>;
  constexpr int kSmem = kOut ? TcShape<D>::kSmemOut : TcShape<D>::kSmem;
  static std::mutex mu;
  static std::vector<int> ready;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    bool found = false;
    for (int d : ready) found |= d == dev;
    if (!found) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      ready.push_back(dev);
    }
  }
  kernel<<<dim3(units, p.tiles), kThreads, kSmem, s>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_typed(const PrefillParams& pp, cudaStream_t s) {
  TcParams p;
  if (!encode_operand(&p.tm_a, pp.q, pp.units, pp.P, D) || !encode_operand(&p.tm_b, pp.k, pp.units, pp.P, D))
    return cudaErrorInvalidValue;
  p.row_max_in = nullptr;
  p.row_sum_in = nullptr;
  p.row_max = pp.row_max;
  p.row_sum = pp.row_sum;
  p.colsum = pp.colsum;
  p.err = pp.err;
  p.P = pp.P;
  p.tiles = (pp.P + kTile - 1) / kTile;
  p.scale = pp.scale;
  p.last_row_only = 0;
  p.out = static_cast<__nv_bfloat16*>(pp.out);
  if (pp.out != nullptr && !encode_operand(&p.tm_v, pp.v, pp.units, pp.P, D)) return cudaErrorInvalidValue;
  // resident Q, streamed K (and V when the prompt's attention output is wanted)
  cudaError_t e = pp.out != nullptr ? launch_pass<D, false, true>(p, pp.units, s) : launch_pass<D, false>(p, pp.units, s);
  if (e != cudaSuccess) return e;
  const CUtensorMap q_map = p.tm_a;
  p.tm_a = p.tm_b;                                         // resident K, streamed Q
  p.tm_b = q_map;
  p.row_max_in = pp.row_max;
  p.row_sum_in = pp.row_sum;
  p.last_row_only = pp.last_row_only;
  return launch_pass<D, true>(p, pp.units, s);
}

}  // namespace

cudaError_t launch_prefill_scores_tc(const PrefillParams& p, int head_dim, cudaStream_t s) {
  return head_dim == 64 ? launch_typed<64>(p, s) : launch_typed<128>(p, s);
}

}  // namespace h2o
