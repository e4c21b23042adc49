// h2o_prefill_tc.cu -- prefill score pass (hot-path rows P1-P2) for bf16 on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory, operands staged by TMA), and the prompt's
// attention output when it is asked for.
//
//   P1  m_i = max_{j<=i} s_ij and l_i = sum_{j<=i} exp(s_ij - m_i), s_ij = (q_i . k_j) / sqrt(D)
//       (causal Softmax(QK^T/sqrt(d)): H2O post §2.1.1)
//   P2  c_j = sum_{i>=j} exp(s_ij - m_i) / l_i: the attention each prompt token accumulates over the
//       prompt (H2O post §2.1.2 / §2.2; "H2O Heavy-Hitter Oracle 分析" §3.1)
//   P1+ with an output tensor, the row-statistics pass is also the prompt's attention forward:
//       o_i = sum_{j<=i} exp(s_ij - m_i) / l_i v_j, sharing the logits and exponentials with P1.
//
// One persistent kernel shape serves the four passes. A work item is one 128-row "resident" tile of
// one unit; every CTA (one per SM) walks its items (whole units when there are many, see item_at) and
// streams, per item, 128-row tiles of the other operand, so that S = A B^T lands in tensor memory
// with one TMEM lane per resident row:
//   row stats    resident = Q tile i, streamed = K tiles 0..i   -> rows are queries, reduce along j
//   column sums  resident = K tile j, streamed = Q tiles j..end -> rows are keys, reduce along i,
//                recomputing S instead of storing the P x P probabilities.
// Warp roles: warp 16 issues the TMA loads (resident tiles double-buffered, so the next item's tile
// arrives while the current one is processed; streamed tiles through a ring), warp 17 allocates tensor
// memory and one of its lanes issues tcgen05.mma (M = N = 128, K = 16 per instruction, bf16 x bf16 ->
// fp32) into two alternating 128-column logit accumulators; warps 0-15 are the epilogue: warps q,
// q + 4, q + 8, q + 12 share TMEM lanes 32q..32q+31 (rows) and take 32 columns each of every tile, so
// sixteen warps keep the exponentials (the bound of this pass) busy; their partial row results are
// combined once per item. Each exponential is one fma and one ex2: the 1/sqrt(D) scale and log2(e)
// are folded into one multiplier.
// The output pass also streams V tiles (ring order K_t, V_{t-1}: the product of tile t-1 runs while
// the epilogue works on tile t). The epilogue writes exp(s - m) as a bf16 128 x 128 probability tile
// (two buffers, K-major, 128-byte swizzle) from which the tensor core accumulates O += P V into a
// third TMEM region, V read as an MN-major operand straight from its TMA tile. The maximum in use
// moves only when a tile's maximum exceeds it by more than kLazyMax (log2 units): O and l are rescaled
// then, rarely, and the probabilities stay below 2^kLazyMax. The warps of a row exchange their tile
// maxima and sums through spare tensor-memory columns (shared memory is full).
// One pass (prompts of at most four tiles, at least one unit per SM, no output tensor): the
// row-statistics shape with four logit accumulators, so that a query tile's logits against all of
// its key tiles sit in tensor memory at once; the epilogue takes the rows' statistics, overwrites the
// logits with their exponentials, then weights them by their row's normaliser and sums them across
// TMEM lanes for the column sums (onepass_epilogue). Every logit and exponential is computed once,
// against twice in the two passes above.
// Every wait is bounded (see mbar_wait); a CTA that gives up still frees its tensor memory.
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
constexpr int kSplit = 4;                  // epilogue warps per TMEM lane quarter
constexpr int kCols = kTile / kSplit;      // logit columns per epilogue warp and tile
constexpr int kEpiWarps = 4 * kSplit;
constexpr int kThreads = 32 * (kEpiWarps + 2);
constexpr int kTmaWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr uint32_t kTmemCols = 512;        // logits x2 [0, 256), output [256, 256 + D), exchange
constexpr uint32_t kOCol = 2 * kTile;
constexpr uint32_t kXCol = 448;            // output pass: [2][kSplit] max exchange, then [2][kSplit] l
constexpr int kPBytes = 2 * kBoxBytes;     // 128 x 128 bf16 probability tile (two 64-key boxes)
constexpr int kAlign = 1024;               // 128-byte swizzle atoms repeat every 1024 bytes
constexpr int kCtrlBytes = 384;            // mbarriers + TMEM address slot
constexpr int kRegions = 4;                // one-pass column sums: 128-column logit regions (all of TMEM)
constexpr int kQuarterRows = 32;           // one-pass column sums: rows per resident TMA box (a lane quarter)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyMax = 8.f;            // output pass: rescale only when the max grows by > 2^8

enum Mode { kRowStats = 0, kRowOut = 1, kColSums = 2, kOnePass = 3 };

struct TcParams {
  CUtensorMap tm_a;        // resident operand: Q (row stats) or K (column sums), [units][P][D]
  CUtensorMap tm_b;        // streamed operand: K (row stats) or Q (column sums)
  CUtensorMap tm_v;        // output pass: V
  const float* row_max_in; // column sums: m_i from the row-stats pass (log2 units), [units][P]
  const float* row_sum_in; // column sums: l_i, taken against m_i
  float* row_max;          // row stats output (log2 units: the largest s_ij log2(e) / sqrt(D))
  float* row_sum;
  float* colsum;           // column sums output
  __nv_bfloat16* out;      // output pass: [units][P][D]
  int32_t* err;
  int32_t units;
  int32_t P;
  int32_t tiles;           // ceil(P / 128)
  float sl;                // log2(e) / sqrt(D)
  int32_t last_row_only;   // column sums: only the last query's weight (Top-K prefill)
  int32_t unit_items;      // CTAs take whole units (see item_at)
};

template <int D, int kMode>
struct TcShape {
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  // Streamed ring depth. The output pass also holds V tiles and two probability tiles, so its ring
  // is shallower (it exchanges between warps through tensor memory); the other passes keep an
  // exchange area for the partial row results ([2][kSplit][128] float2) and, for column sums, each
  // warp's query statistics ([kEpiWarps][2][2][kCols] float: -m, 1/l); the one-pass column sums keep, instead,
  // each lane quarter's column partials of two units ([2][4][kRegions * 128] float).
  static constexpr int kStages = kMode == kRowOut ? (D == 128 ? 3 : 6) : (D == 128 ? 4 : 8);
  static constexpr int kXBytes = 2 * kSplit * kTile * 8;
  static constexpr int kPartBytes = 2 * 4 * kRegions * kTile * 4;
  static constexpr int kHeadBytes =
      kCtrlBytes + (kMode == kRowOut ? 0 : kXBytes + (kMode == kOnePass ? kPartBytes : kEpiWarps * 4 * kCols * 4));
  static constexpr int kBodyBytes = (2 + kStages) * kTileBytes + (kMode == kRowOut ? 2 * kPBytes : 0);
  static constexpr int kSmem = kHeadBytes + kAlign + kBodyBytes;
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

// Shared-memory matrix descriptor of a K-major operand tile written with 128-byte swizzle: rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), descriptor version 1, layout type
// 2 = SWIZZLE_128B. Advancing along K inside the 128-byte row moves the start address.
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
                                         uint32_t idesc) {
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

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v);
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float* v) {
  tmem_ld32(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int x = 0; x < 16; ++x) v[x] = __uint_as_float(r[x]);
}

template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v);
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const float* v) {
  tmem_st32(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// One value per thread (lane) into TMEM column `taddr`, and kSplit consecutive columns back.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\ntcgen05.wait::st.sync.aligned;" ::"r"(taddr),
               "r"(__float_as_uint(v))
               : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float* v) {
  uint32_t r0, r1, r2, r3;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\ntcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(taddr)
      : "memory");
  v[0] = __uint_as_float(r0);
  v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2);
  v[3] = __uint_as_float(r3);
}

// 2^x by the special-function unit (ex2.approx, relative error ~2^-22; results below 2^-126 flush to
// zero, far below what a softmax weight or a column sum can resolve next to its row's maximum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two-lane fp32 fma and add (packed instructions of this GPU generation): each lane rounds exactly
// like the scalar fmaf / + it stands for, so results do not change, at half the instructions.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
// Store 32 fp32 columns of this warp's 32 TMEM lanes without waiting for completion (tmem_wait_st
// orders them before a later read of the same columns).
__device__ __forceinline__ void tmem_st32_async(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
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
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 TMEM lanes x 32 columns of this warp's lane quarter in the 16x256b fragment shape (two loads of
// 16 lanes, four 256-bit column groups each), so that every thread holds 4 rows x 8 columns: for
// column group k (columns 8k..8k+7) and thread t, r[4k], r[4k+1] are row t/4, columns 8k + 2(t%4) and
// +1; r[4k+2], r[4k+3] row t/4 + 8, the same columns; r[16 + ...] likewise rows t/4 + 16 and t/4 + 24.
// tmem_ld_rows4_start starts the loads; tmem_wait_rows4 waits for them taking r as in/out operands,
// so that no use of r can move above the wait (work in between overlaps the loads).
__device__ __forceinline__ void tmem_ld_rows4_start(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%32];\n"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "r"(taddr + (16u << 16))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_rows4(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Sums over the 8 threads that share t % 4 (lane bits 2-4) of 8 column partials each: a butterfly
// reduce-scatter in which, at distance d, each thread keeps the half of its values selected by lane
// bit d, sends the other half to lane ^ d and adds what it receives. Thread t returns value
// (t >> 2) & 7 summed over the 8 threads (7 shuffles and 7 additions per thread).
__device__ __forceinline__ float column_sum8(float (&w)[8], int lane) {
#pragma unroll
  for (int half = 4, d = 16; half >= 1; half >>= 1, d >>= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? w[j] : w[j + half];
      const float keep = upper ? w[j + half] : w[j];
      w[j] = keep + __shfl_xor_sync(0xffffffffu, send, d);
    }
  }
  return w[0];
}

// The largest of three values in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float max32(const float* v) {
  float m[11];
#pragma unroll
  for (int x = 0; x < 10; ++x) m[x] = max3(v[3 * x], v[3 * x + 1], v[3 * x + 2]);
  m[10] = fmaxf(v[30], v[31]);
  const float a = max3(m[0], m[1], m[2]), b = max3(m[3], m[4], m[5]), c = max3(m[6], m[7], m[8]);
  return fmaxf(max3(a, b, c), fmaxf(m[9], m[10]));
}

// sum_x 2^(v[x] sl + nb[x]) over 32 values in four interleaved partial sums (x mod 4), combined as
// (s0 + s1) + (s2 + s3); lanes x < lo contribute nothing.
template <bool kMask>
__device__ __forceinline__ float exp2_sum32(const float* v, float2 sl2, const float* nb, int lo) {
  float2 s01 = make_float2(0.f, 0.f), s23 = s01;
#pragma unroll
  for (int x = 0; x < 32; x += 4) {
    const float2 e01 = fma2(make_float2(v[x], v[x + 1]), sl2, make_float2(nb[x], nb[x + 1]));
    const float2 e23 = fma2(make_float2(v[x + 2], v[x + 3]), sl2, make_float2(nb[x + 2], nb[x + 3]));
    if constexpr (kMask) {
      s01 = add2(s01, make_float2(x >= lo ? ex2(e01.x) : 0.f, x + 1 >= lo ? ex2(e01.y) : 0.f));
      s23 = add2(s23, make_float2(x + 2 >= lo ? ex2(e23.x) : 0.f, x + 3 >= lo ? ex2(e23.y) : 0.f));
    } else {
      s01 = add2(s01, make_float2(ex2(e01.x), ex2(e01.y)));
      s23 = add2(s23, make_float2(ex2(e23.x), ex2(e23.y)));
    }
  }
  return (s01.x + s01.y) + (s23.x + s23.y);
}

// sum_x 2^(v[x] sl + nb[x]) w[x] over 32 values, four interleaved partial sums as exp2_sum32; lanes
// x < lo contribute nothing. Column sums: nb = -m_i (the query's maximum, so that the argument is
// small where the weight matters) and w = 1 / l_i: the normaliser is applied as a factor rather than
// folded into the exponent, where its magnitude (log2 l plus a maximum of hundreds) would cost fp32
// bits of the argument.
template <bool kMask>
__device__ __forceinline__ float exp2_wsum32(const float* v, float2 sl2, const float4* nb4, const float4* w4, int lo) {
  float2 s01 = make_float2(0.f, 0.f), s23 = s01;
#pragma unroll
  for (int x = 0; x < 32; x += 4) {
    const float4 nb = nb4[x / 4], w = w4[x / 4];  // shared memory, read as needed
    const float2 e01 = fma2(make_float2(v[x], v[x + 1]), sl2, make_float2(nb.x, nb.y));
    const float2 e23 = fma2(make_float2(v[x + 2], v[x + 3]), sl2, make_float2(nb.z, nb.w));
    if constexpr (kMask) {
      s01 = fma2(make_float2(x >= lo ? ex2(e01.x) : 0.f, x + 1 >= lo ? ex2(e01.y) : 0.f), make_float2(w.x, w.y),
                 s01);
      s23 = fma2(make_float2(x + 2 >= lo ? ex2(e23.x) : 0.f, x + 3 >= lo ? ex2(e23.y) : 0.f), make_float2(w.z, w.w),
                 s23);
    } else {
      s01 = fma2(make_float2(ex2(e01.x), ex2(e01.y)), make_float2(w.x, w.y), s01);
      s23 = fma2(make_float2(ex2(e23.x), ex2(e23.y)), make_float2(w.z, w.w), s23);
    }
  }
  return (s01.x + s01.y) + (s23.x + s23.y);
}

// Generic-proxy shared-memory writes made visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The kSplit epilogue warps sharing TMEM lane quarter q (warps q, q + 4, ...): named barrier 1 + q.
__device__ __forceinline__ void quarter_sync(int q) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + q), "n"(32 * kSplit) : "memory");
}

// The n-th resident tile a CTA processes. With many units (unit_items) a CTA takes whole units, all
// their resident tiles in a row, so the tiles streamed for one resident tile are still in L2 for the
// next; with few units the (unit, resident tile) pairs are spread over the CTAs one by one, ordered
// tile-major and heaviest first so that the stride hands every CTA a similar mix.
struct Item {
  int unit, at, t_begin, nt;
};
template <int kMode>
__device__ __forceinline__ bool item_at(const TcParams& p, int n, Item* it) {
  int k;
  if (p.unit_items) {
    const int u = blockIdx.x + (n / p.tiles) * gridDim.x;
    if (u >= p.units) return false;
    it->unit = u;
    k = n % p.tiles;
  } else {
    const int i = blockIdx.x + n * gridDim.x;
    if (i >= p.units * p.tiles) return false;
    k = i / p.units;
    it->unit = i - k * p.units;
  }
  if constexpr (kMode == kColSums) {
    it->at = k;  // query tiles at..end
    it->t_begin = p.last_row_only ? p.tiles - 1 : it->at;
    it->nt = p.tiles - it->t_begin;
  } else {
    it->at = p.tiles - 1 - k;  // key tiles 0..at
    it->t_begin = 0;
    it->nt = it->at + 1;
  }
  return true;
}

// All 16 epilogue warps (named barrier 5).
__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 5, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

// Epilogue of the one-pass column sums (prompts of at most kRegions tiles; each CTA takes whole
// units, query tiles tiles - 1 down to 0). Item = query tile i of a unit; its logit tiles against key
// tiles 0..i stay in tensor-memory regions (g mod kRegions) until the item is done:
//   sweep 1, per key tile t: this warp's 32 columns of row r (one row per thread); the running
//            maximum m (log2 units) and sum l of 2^(s sl - m) over them; the logits are overwritten by
//            e = 2^(s sl - m_t), m_t the running maximum when tile t was read;
//   combine: the kSplit warps of the lane quarter exchange (m, l): the row's maximum M and sum L, and
//            each row's weight for tile t, f_t = 2^(m_t - M) / L (zero for rows past the prompt);
//   sweep 2, per key tile t: e back from tensor memory in the 16x256b shape (4 rows x 8 columns per
//            thread; the region is then released to the MMA lane); the thread sums its 4 rows weighted
//            by their f_t, and 8 threads add their partials per column (column_sum8).
// On the diagonal tile a warp whose 32 keys all lie past its 32 rows has nothing to add and skips the
// tile; one whose keys all lie before its rows needs no mask (unless the prompt ends inside them).
// That work differs between lane quarters, and the four warps of lane quarter q all run on SM
// sub-partition q, so the resident tile's 32-row blocks are rotated by the query tile index: lane
// quarter q holds rows 32 ((q + i) mod 4) .. of query tile i, and over a unit's items every
// sub-partition takes each block of the diagonal once.
// Each lane quarter's column sums go to its own shared-memory row (the unit's first item, which meets
// every key tile, writes; later items add), and once the unit's last item is done the four rows are
// added in a fixed order, so a column sum does not depend on warp timing.
template <int D>
__device__ __forceinline__ void onepass_epilogue(const TcParams& p, uint32_t tmem, int warp, int lane, float2* xh,
                                                 float* part, uint64_t* acc_full, uint64_t* acc_empty) {
  constexpr int kKeys = kRegions * kTile;
  const int q = warp & 3, h = warp >> 2;
  const int r = q * 32 + lane;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
  const float sl = p.sl;
  const int P = p.P;
  // sweep 2: this thread's column within the warp's 32 (column_sum8's output, see tmem_ld_rows4_start)
  const int vsel = (lane >> 2) & 7;
  const int col = 8 * (vsel >> 1) + 2 * (lane & 3) + (vsel & 1);
  bool ok = true;
  uint32_t g = 0;  // logit tiles consumed (over all items)
  Item it;
  for (int k = 0; item_at<kOnePass>(p, k, &it); ++k) {
    const int kt = k % p.tiles;       // item within the unit (0: query tile tiles - 1)
    const int ub = (k / p.tiles) & 1;  // the unit's buffer of column partials
    float* pq = part + (ub * 4 + q) * kKeys + h * kCols + col;
    const int sb = (q + it.at) & 3;  // the tile's 32-row block in this lane quarter (see the TMA loads)
    const int row = it.at * kTile + sb * kQuarterRows + lane;
    // The diagonal tile for this warp: no key before any of its rows (skip), or every key before all
    // of them and before the prompt's end (no mask).
    const bool diag_empty = h > sb;
    const bool diag_full = h < sb && P - 1 - (it.at * kTile + h * kCols) >= kCols - 1;
    float m2 = -INFINITY, l = 0.f;
    float mt[kRegions];
#pragma unroll
    for (int t = 0; t < kRegions; ++t) {
      mt[t] = -INFINITY;
      if (t < it.nt) {
        const uint32_t gt = g + t, a = gt % kRegions;
        if (ok) ok = mbar_wait(&acc_full[a], (gt / kRegions) & 1u, p.err);
        const bool diag = t == it.at;
        if (!(diag && diag_empty)) {
          tc_fence_after();
          const uint32_t taddr = lane_addr + a * kTile + h * kCols;
          float v[kCols];
          tmem_ld32(taddr, v);
          if (diag && !diag_full) {  // keys j <= row and j < P
            const int lim = min(row, P - 1) - (t * kTile + h * kCols);
#pragma unroll
            for (int x = 0; x < kCols; ++x) v[x] = x <= lim ? v[x] : -INFINITY;
          }
          const float cm = max32(v) * sl;
          if (cm > m2) {
            l *= ex2(m2 - cm);
            m2 = cm;
          }
          mt[t] = m2;
          if (m2 != -INFINITY) {
            const float2 sl2 = make_float2(sl, sl), nm = make_float2(-m2, -m2);
            float2 s01 = make_float2(0.f, 0.f), s23 = s01;
#pragma unroll
            for (int x = 0; x < kCols; x += 4) {
              const float2 e01 = fma2(make_float2(v[x], v[x + 1]), sl2, nm);
              const float2 e23 = fma2(make_float2(v[x + 2], v[x + 3]), sl2, nm);
              v[x] = ex2(e01.x);
              v[x + 1] = ex2(e01.y);
              v[x + 2] = ex2(e23.x);
              v[x + 3] = ex2(e23.y);
              s01 = add2(s01, make_float2(v[x], v[x + 1]));
              s23 = add2(s23, make_float2(v[x + 2], v[x + 3]));
            }
            l += (s01.x + s01.y) + (s23.x + s23.y);
          } else {
#pragma unroll
            for (int x = 0; x < kCols; ++x) v[x] = 0.f;
          }
          tmem_st32_async(taddr, v);
        }
      }
    }
    tmem_wait_st();
    // The row's maximum and normaliser over the quarter's kSplit warps (buffer by item parity: a warp
    // rewrites it two items later, after every warp of the quarter has passed the next exchange).
    float2* xk = xh + (k & 1) * kSplit * kTile;
    xk[h * kTile + r] = make_float2(m2, l);
    quarter_sync(q);
    float mm = xk[r].x;
#pragma unroll
    for (int j = 1; j < kSplit; ++j) mm = fmaxf(mm, xk[j * kTile + r].x);
    float lt = 0.f;
#pragma unroll
    for (int j = 0; j < kSplit; ++j) {
      const float2 o = xk[j * kTile + r];
      if (o.x != -INFINITY) lt += o.y * ex2(o.x - mm);
    }
    const float inv = row < P ? 1.f / lt : 0.f;
#pragma unroll
    for (int t = 0; t < kRegions; ++t) {
      if (t < it.nt) {
        const uint32_t a = (g + t) % kRegions;
        float cs = 0.f;
        if (t == it.at && diag_empty) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a]);
        } else {
          uint32_t rr[kCols];
          tmem_ld_rows4_start(lane_addr + a * kTile + h * kCols, rr);
          // row weights of the thread's four rows (lanes t/4 + 8i own them in sweep 1), while the
          // e values load
          const float f = mt[t] == -INFINITY ? 0.f : ex2(mt[t] - mm) * inv;
          float2 fr[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float fi = __shfl_sync(0xffffffffu, f, (lane >> 2) + 8 * i);
            fr[i] = make_float2(fi, fi);
          }
          tmem_wait_rows4(rr);
          float v[kCols];
#pragma unroll
          for (int x = 0; x < kCols; ++x) v[x] = __uint_as_float(rr[x]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a]);
          float w[8];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float2 acc = mul2(make_float2(v[4 * c4], v[4 * c4 + 1]), fr[0]);
            acc = fma2(make_float2(v[4 * c4 + 2], v[4 * c4 + 3]), fr[1], acc);
            acc = fma2(make_float2(v[16 + 4 * c4], v[16 + 4 * c4 + 1]), fr[2], acc);
            acc = fma2(make_float2(v[16 + 4 * c4 + 2], v[16 + 4 * c4 + 3]), fr[3], acc);
            w[2 * c4] = acc.x;
            w[2 * c4 + 1] = acc.y;
          }
          cs = column_sum8(w, lane);
        }
        float* dst = pq + t * kTile;
        *dst = kt == 0 ? cs : *dst + cs;
      }
    }
    g += it.nt;
    if (kt == p.tiles - 1) {  // the unit's last item: add the four quarters' partials
      epilogue_sync();
      const int key = warp * 32 + lane;
      if (key < P) {
        const float* pb = part + ub * 4 * kKeys + key;
        p.colsum[static_cast<size_t>(it.unit) * P + key] = (pb[0] + pb[kKeys]) + (pb[2 * kKeys] + pb[3 * kKeys]);
      }
    }
  }
}

template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  using S = TcShape<D, kMode>;
  constexpr int kStages = S::kStages;
  constexpr bool kOut = kMode == kRowOut;
  constexpr bool kCol = kMode == kColSums;
  // logit accumulators (the output pass keeps O at 256..; the one-pass column sums hold a query tile's
  // logits against all of its key tiles)
  constexpr uint32_t kNAcc = kOut ? 2u : (kMode == kOnePass ? static_cast<uint32_t>(kRegions) : 3u);
  extern __shared__ unsigned char smem_raw[];
  // head: mbarriers, TMEM slot, exchange areas; body (1024-aligned): resident x2, ring, P x2
  unsigned char* head = smem_raw;
  unsigned char* body = smem_raw + S::kHeadBytes;
  body += (kAlign - (smem_u32(body) & (kAlign - 1))) & (kAlign - 1);
  unsigned char* res = body;                                  // [2][kTileBytes]
  unsigned char* ring = body + 2 * S::kTileBytes;             // [kStages][kTileBytes]
  unsigned char* ptile = ring + kStages * S::kTileBytes;      // output pass: [2][kPBytes]
  uint64_t* res_full = reinterpret_cast<uint64_t*>(head);
  uint64_t* res_empty = res_full + 2;
  uint64_t* ring_full = res_empty + 2;
  uint64_t* ring_empty = ring_full + kStages;
  uint64_t* acc_full = ring_empty + kStages;
  uint64_t* acc_empty = acc_full + kRegions;
  uint64_t* p_full = acc_empty + kRegions;  // output pass: the epilogue wrote probability tile b
  uint64_t* p_free = p_full + 2;      // output pass: the product reading probability tile b finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_free + 2);
  float2* xh = reinterpret_cast<float2*>(head + kCtrlBytes);  // row stats / column sums: [2][kSplit][128]
  float* xq = reinterpret_cast<float*>(head + kCtrlBytes + S::kXBytes);  // column sums: [warps][2][kCols]
  float* part = xq;  // one-pass column sums: [2][4][kRegions * 128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.P;

  if (tid == 0) {
    for (int b = 0; b < kRegions; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&res_full[b], 1);
      mbar_init(&res_empty[b], 1);
      mbar_init(&p_full[b], kEpiWarps);
      mbar_init(&p_free[b], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    fence_mbar_init();
  }
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

  if (warp == kTmaWarp) {
    if (lane == 0) {
      uint32_t r = 0;  // streamed tiles issued so far
      bool ok = true;
      auto stream = [&](const CUtensorMap* map, int row, int unit) {
        const int s = static_cast<int>(r % kStages);
        if (r >= static_cast<uint32_t>(kStages) && !mbar_wait(&ring_empty[s], (r / kStages - 1) & 1u, p.err))
          return false;
        mbar_expect_tx(&ring_full[s], S::kTileBytes);
        for (int b = 0; b < S::kBoxes; ++b)
          tma_load_3d(ring + s * S::kTileBytes + b * kBoxBytes, map, b * kBoxCols, row, unit, &ring_full[s]);
        ++r;
        return true;
      };
      int prev_unit = -1, prev_last = 0;  // output pass: the previous item's last V tile
      int k = 0;
      Item it;
      for (; ok && item_at<kMode>(p, k, &it); ++k) {
        const int rb = k & 1;
        if (k >= 2 && !mbar_wait(&res_empty[rb], static_cast<uint32_t>(k / 2 - 1) & 1u, p.err)) break;
        mbar_expect_tx(&res_full[rb], S::kTileBytes);
        if constexpr (kMode == kOnePass) {
          // 32-row blocks, block j of query tile i at row block (j - i) mod 4, so that lane quarter q
          // holds rows 32 ((q + i) mod 4) .. of the tile (see onepass_epilogue)
          for (int b = 0; b < S::kBoxes; ++b)
            for (int j = 0; j < 4; ++j)
              tma_load_3d(res + rb * S::kTileBytes + b * kBoxBytes + ((j - it.at) & 3) * (kQuarterRows * 128),
                          &p.tm_a, b * kBoxCols, it.at * kTile + j * kQuarterRows, it.unit, &res_full[rb]);
        } else {
          for (int b = 0; b < S::kBoxes; ++b)
            tma_load_3d(res + rb * S::kTileBytes + b * kBoxBytes, &p.tm_a, b * kBoxCols, it.at * kTile, it.unit,
                        &res_full[rb]);
        }
        for (int t = 0; t < it.nt && ok; ++t) {
          ok = stream(&p.tm_b, (it.t_begin + t) * kTile, it.unit);
          if constexpr (kOut) {
            // V in the order the products consume it: V_{t-1} after K_t, and the previous item's
            // last V after this item's K_0
            if (ok && t > 0) ok = stream(&p.tm_v, (t - 1) * kTile, it.unit);
            else if (ok && prev_unit >= 0) ok = stream(&p.tm_v, prev_last * kTile, prev_unit);
          }
        }
        prev_unit = it.unit;
        prev_last = it.nt - 1;
      }
      if constexpr (kOut) {
        if (ok && prev_unit >= 0) stream(&p.tm_v, prev_last * kTile, prev_unit);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      uint32_t r = 0, g = 0, pv = 0;  // streamed tiles consumed, logit tiles, products issued
      bool ok = true;
      bool pending = false;           // output pass: a P V product waiting for its probabilities
      int pending_t = 0;              // its tile index within its item (0: overwrite O)
      auto product = [&]() {
        const uint32_t b = pv & 1u;
        const int s = static_cast<int>(r % kStages);
        if (!mbar_wait(&p_full[b], (pv / 2) & 1u, p.err)) return false;
        if (!mbar_wait(&ring_full[s], (r / kStages) & 1u, p.err)) return false;
        tc_fence_after();
        const uint32_t p_base = smem_u32(ptile + b * kPBytes);
        const uint32_t v_base = smem_u32(ring + s * S::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          // P: K-major, 64 keys per box, 32 bytes per 16-key step; V: MN-major, 16 key rows of 128
          // bytes per step, 64-column groups one box apart.
          const uint32_t off_p = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          mma_bf16(tmem + kOCol, sw128_desc(p_base + off_p), sw128_desc_mn(v_base + kk * 2048, kBoxBytes),
                   (pending_t > 0 || kk > 0) ? 1u : 0u, kIdescPV<D>);
        }
        mma_commit(&ring_empty[s]);
        mma_commit(&p_free[b]);  // probability tile b may be rewritten, O may be read or rescaled
        ++r;
        ++pv;
        return true;
      };
      int k = 0;
      Item it;
      for (; ok && item_at<kMode>(p, k, &it); ++k) {
        const int rb = k & 1;
        if (!mbar_wait(&res_full[rb], static_cast<uint32_t>(k / 2) & 1u, p.err)) break;
        const uint32_t a_base = smem_u32(res + rb * S::kTileBytes);
        for (int t = 0; t < it.nt; ++t, ++g) {
          const int s = static_cast<int>(r % kStages);
          const uint32_t a = g % kNAcc;
          if (!mbar_wait(&ring_full[s], (r / kStages) & 1u, p.err) ||
              (g >= kNAcc && !mbar_wait(&acc_empty[a], (g / kNAcc - 1) & 1u, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_base = smem_u32(ring + s * S::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;  // 16 bf16 = 32 bytes per step
            mma_bf16(tmem + a * kTile, sw128_desc(a_base + off), sw128_desc(b_base + off), kk > 0 ? 1u : 0u,
                     kIdesc);
          }
          mma_commit(&ring_empty[s]);  // the streamed tile may be overwritten once these MMAs finish
          mma_commit(&acc_full[a]);    // and the logits may be read
          if (t == it.nt - 1) mma_commit(&res_empty[rb]);
          ++r;
          if constexpr (kOut) {
            // the product of the previous logit tile (this item's, or the previous item's last)
            if (pending && !product()) {
              ok = false;
              break;
            }
            pending = true;
            pending_t = t;
          }
        }
      }
      if constexpr (kOut) {
        if (ok && pending) product();
      }
    }
    __syncwarp();
  } else if constexpr (kMode == kOnePass) {
    onepass_epilogue<D>(p, tmem, warp, lane, xh, part, acc_full, acc_empty);
  } else {
    // Epilogue: warp q + 4h owns TMEM lanes 32q.. (resident rows) and columns 32h..32h+31 of a tile.
    const int q = warp & 3, h = warp >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float sl = p.sl;
    bool ok = true;
    uint32_t g = 0;  // logit tiles consumed (over all items)
    int k = 0;
    float* xw = xq + warp * 4 * kCols;  // column sums: this warp's query statistics, [2][-m, 1/l][kCols]
    // column sums: a query's row statistics (m in log2 units), loaded one tile ahead of their use; its
    // weight is 2^(s sl - m) / l (queries past the prompt weigh nothing)
    float qm = 0.f, ql = 0.f;
    auto qload = [&](int unit, int i) {
      qm = INFINITY;
      ql = 1.f;
      if (i < P) {
        const size_t o = static_cast<size_t>(unit) * P + i;
        qm = p.row_max_in[o];
        ql = p.row_sum_in[o];
      }
    };
    Item it;
    for (; item_at<kMode>(p, k, &it); ++k) {
      const int row = it.at * kTile + r;
      const size_t ubase = static_cast<size_t>(it.unit) * P;
      float m2 = -INFINITY, l = 0.f, c = 0.f;  // this warp's partial statistics (log2 units)
      float mu = -INFINITY;  // output pass: the maximum the probabilities are taken against
      if constexpr (kCol) qload(it.unit, it.t_begin * kTile + h * kCols + lane);
      for (int t = 0; t < it.nt; ++t, ++g) {
        const uint32_t a = g % kNAcc;  // logit accumulator
        const uint32_t xa = g & 1u;    // query-statistics buffer
        const int x0 = (it.t_begin + t) * kTile + h * kCols;  // key (query) of this warp's column 0
        if constexpr (kCol) {
          // this tile's query statistics for this warp's columns; prefetch the next tile's
          xw[(2 * xa) * kCols + lane] = -qm;
          xw[(2 * xa + 1) * kCols + lane] = __frcp_rn(ql);
          if (t + 1 < it.nt) qload(it.unit, (it.t_begin + t + 1) * kTile + h * kCols + lane);
          __syncwarp();
        }
        if (ok) ok = mbar_wait(&acc_full[a], (g / kNAcc) & 1u, p.err);
        tc_fence_after();
        float v[kCols];
        tmem_ld32(lane_addr + a * kTile + h * kCols, v);
        if constexpr (!kCol) {
          // the diagonal tile: keys j <= row and j < P (earlier tiles lie wholly below the diagonal)
          if (t == it.at) {
            const int lim = min(row, P - 1) - x0;
#pragma unroll
            for (int x = 0; x < kCols; ++x) v[x] = x <= lim ? v[x] : -INFINITY;
          }
        }
        if constexpr (kMode == kRowStats) {
          const float cm = max32(v) * sl;
          if (cm > m2) {
            l *= ex2(m2 - cm);
            m2 = cm;
          }
          if (m2 != -INFINITY) {
            float nm[kCols];
#pragma unroll
            for (int x = 0; x < kCols; ++x) nm[x] = -m2;
            l += exp2_sum32<false>(v, make_float2(sl, sl), nm, 0);
          }
        } else if constexpr (kCol) {
          // this tile's -m and 1/l for this warp's columns (queries), in shared memory
          const float* nbs = xw + (2 * xa) * kCols;
          const float* ils = xw + (2 * xa + 1) * kCols;
          const float4* b4 = reinterpret_cast<const float4*>(nbs);
          const float4* w4 = reinterpret_cast<const float4*>(ils);
          const float2 sl2 = make_float2(sl, sl);
          if (p.last_row_only) {
            const int xl = P - 1 - x0;  // the last query's column, if this warp holds it
            if (xl >= 0 && xl < kCols) {
              float s0 = 0.f;
#pragma unroll
              for (int x = 0; x < kCols; ++x)
                if (x == xl && row <= P - 1) s0 += ex2(fmaf(v[x], sl, nbs[xl])) * ils[xl];
              c += s0;
            }
          } else if (it.t_begin + t > it.at) {  // queries all after the keys
            c += exp2_wsum32<false>(v, sl2, b4, w4, 0);
          } else {  // the diagonal tile: queries i >= row
            c += exp2_wsum32<true>(v, sl2, b4, w4, row - x0);
          }
        } else {
          // Output pass. Probability tile a was last read by the product of logit tile g - 2.
          if (g >= 2 && ok) ok = mbar_wait(&p_free[a], (g / 2 - 1) & 1u, p.err);
          // The tile's maximum over the quarter's kSplit warps, exchanged through TMEM columns.
          tmem_st1(lane_addr + kXCol + a * kSplit + h, max32(v));
          tc_fence_before();
          quarter_sync(q);
          tc_fence_after();
          float xm[4];
          tmem_ld4(lane_addr + kXCol + a * kSplit, xm);
          const float tmax = fmaxf(fmaxf(xm[0], xm[1]), fmaxf(xm[2], xm[3])) * sl;
          m2 = fmaxf(m2, tmax);
          float alpha = 1.f;
          if (tmax > mu + kLazyMax) {
            alpha = ex2(mu - tmax);  // 0 on the first tile
            l *= alpha;
            mu = tmax;
          }
          // Rescaling O needs the product of tile g - 1 finished.
          if (t > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
            if (ok) ok = mbar_wait(&p_free[a ^ 1u], ((g - 1) / 2) & 1u, p.err);
            tc_fence_after();
            constexpr int kOC = D / kSplit;  // output columns per warp
            float o[kOC];
            const uint32_t oaddr = lane_addr + kOCol + h * kOC;
            tmem_ld<kOC>(oaddr, o);
#pragma unroll
            for (int x = 0; x < kOC; ++x) o[x] *= alpha;
            tmem_st<kOC>(oaddr, o);
          }
          // Probabilities against mu (masked logits give 0) into this warp's 32 keys of tile a:
          // 16-byte chunks (h & 1) * 4 .. + 3 of box h >> 1, row r.
          {
            const float2 sl2 = make_float2(sl, sl), nmu = make_float2(-mu, -mu);
            float2 s01 = make_float2(0.f, 0.f), s23 = s01;
#pragma unroll
            for (int x = 0; x < kCols; x += 4) {
              const float2 e01 = fma2(make_float2(v[x], v[x + 1]), sl2, nmu);
              const float2 e23 = fma2(make_float2(v[x + 2], v[x + 3]), sl2, nmu);
              v[x] = ex2(e01.x);
              v[x + 1] = ex2(e01.y);
              v[x + 2] = ex2(e23.x);
              v[x + 3] = ex2(e23.y);
              s01 = add2(s01, make_float2(v[x], v[x + 1]));
              s23 = add2(s23, make_float2(v[x + 2], v[x + 3]));
            }
            l += (s01.x + s01.y) + (s23.x + s23.y);
          }
          unsigned char* rowp = ptile + a * kPBytes + (h >> 1) * kBoxBytes + r * 128;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int chunk = (h & 1) * 4 + c4;
            uint4 w;
            w.x = pack_bf16(v[c4 * 8 + 0], v[c4 * 8 + 1]);
            w.y = pack_bf16(v[c4 * 8 + 2], v[c4 * 8 + 3]);
            w.z = pack_bf16(v[c4 * 8 + 4], v[c4 * 8 + 5]);
            w.w = pack_bf16(v[c4 * 8 + 6], v[c4 * 8 + 7]);
            *reinterpret_cast<uint4*>(rowp + ((chunk ^ (r & 7)) << 4)) = w;
          }
          fence_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kOut) mbar_arrive(&p_full[a]);
          mbar_arrive(&acc_empty[a]);
        }
      }
      // Item end: combine the kSplit partial results of every row.
      if constexpr (kMode == kRowStats) {
        float2* xk = xh + (k & 1) * kSplit * kTile;  // by item parity: read before it is reused
        xk[h * kTile + r] = make_float2(m2, l);
        quarter_sync(q);
        if (h == 0 && row < P) {
          float mm = m2;
#pragma unroll
          for (int j = 1; j < kSplit; ++j) mm = fmaxf(mm, xk[j * kTile + r].x);
          float lt = 0.f;
#pragma unroll
          for (int j = 0; j < kSplit; ++j) {
            const float2 o = xk[j * kTile + r];
            if (o.x != -INFINITY) lt += o.y * ex2(o.x - mm);
          }
          p.row_max[ubase + row] = mm;
          p.row_sum[ubase + row] = lt;
        }
      } else if constexpr (kCol) {
        float2* xk = xh + (k & 1) * kSplit * kTile;
        xk[h * kTile + r] = make_float2(c, 0.f);
        quarter_sync(q);
        if (h == 0 && row < P) {
          float ct = 0.f;
#pragma unroll
          for (int j = 0; j < kSplit; ++j) ct += xk[j * kTile + r].x;
          p.colsum[ubase + row] = ct;
        }
      } else {
        // l over the quarter's warps (all taken against the same mu), through TMEM columns
        const uint32_t lcol = lane_addr + kXCol + 2 * kSplit + (k & 1) * kSplit;
        tmem_st1(lcol + h, l);
        tc_fence_before();
        quarter_sync(q);
        tc_fence_after();
        float xl[4];
        tmem_ld4(lcol, xl);
        const float lt = (xl[0] + xl[1]) + (xl[2] + xl[3]);
        // the last product of this item has finished: normalise and write this warp's columns
        if (ok) ok = mbar_wait(&p_free[(g - 1) & 1u], ((g - 1) / 2) & 1u, p.err);
        tc_fence_after();
        constexpr int kOC = D / kSplit;
        float o[kOC];
        tmem_ld<kOC>(lane_addr + kOCol + h * kOC, o);
        if (row < P) {
          const float inv_l = 1.f / lt;
          __nv_bfloat16* orow = p.out + (ubase + static_cast<size_t>(row)) * D + h * kOC;
#pragma unroll
          for (int c8 = 0; c8 < kOC / 8; ++c8) {
            uint4 w;
            w.x = pack_bf16(o[c8 * 8 + 0] * inv_l, o[c8 * 8 + 1] * inv_l);
            w.y = pack_bf16(o[c8 * 8 + 2] * inv_l, o[c8 * 8 + 3] * inv_l);
            w.z = pack_bf16(o[c8 * 8 + 4] * inv_l, o[c8 * 8 + 5] * inv_l);
            w.w = pack_bf16(o[c8 * 8 + 6] * inv_l, o[c8 * 8 + 7] * inv_l);
            *reinterpret_cast<uint4*>(orow + c8 * 8) = w;
          }
          if (h == 0) {
            p.row_max[ubase + row] = m2;
            p.row_sum[ubase + row] = lt * ex2(mu - m2);  // the normaliser against the true maximum
          }
        }
        tc_fence_before();  // the O reads are ordered before the next item's first product
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

// [units][P][D] bf16 viewed as a 3-D tensor; boxes of 64 columns x 128 rows x 1 unit, 128-byte
// swizzle; rows past P read as zeros.
bool encode_operand(CUtensorMap* map, const void* base, int units, int P, int D, int box_rows = kTile) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(P),
                              static_cast<cuuint64_t>(units)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(P) * D * 2};
  const cuuint32_t box[3] = {kBoxCols, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int kMode>
cudaError_t launch_pass(const TcParams& p, cudaStream_t s) {
  auto kernel = prefill_tc_kernel<D, kMode>;
  constexpr int kSmem = TcShape<D, kMode>::kSmem;
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
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      ready.emplace_back(dev, sms);
    }
  }
  // Whole units per CTA once there are at least 8 per SM (so the last round idles few CTAs).
  TcParams q = p;
  q.unit_items = (kMode == kOnePass || p.units >= 8 * sms) ? 1 : 0;
  const long long items = q.unit_items ? p.units : static_cast<long long>(p.units) * p.tiles;
  const int grid = items < sms ? static_cast<int>(items) : sms;
  kernel<<<grid, kThreads, kSmem, s>>>(q);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_typed(const PrefillParams& pp, cudaStream_t s) {
  TcParams p;
  if (!encode_operand(&p.tm_a, pp.q, pp.units, pp.P, D) || !encode_operand(&p.tm_b, pp.k, pp.units, pp.P, D))
    return cudaErrorInvalidValue;
  p.tm_v = p.tm_b;
  p.row_max_in = nullptr;
  p.row_sum_in = nullptr;
  p.row_max = pp.row_max;
  p.row_sum = pp.row_sum;
  p.colsum = pp.colsum;
  p.out = static_cast<__nv_bfloat16*>(pp.out);
  p.err = pp.err;
  p.units = pp.units;
  p.P = pp.P;
  p.tiles = (pp.P + kTile - 1) / kTile;
  p.sl = pp.scale * kLog2e;
  p.last_row_only = 0;
  p.unit_items = 0;
  cudaError_t e;
  // Prompts of at most kRegions tiles, at least one unit per SM and no output tensor: both rows in one
  // pass (each logit and exponential computed once; the column sums reduced across TMEM lanes).
  if (pp.out == nullptr && !pp.last_row_only && p.tiles <= kRegions) {
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (pp.units >= sms) {
      if (!encode_operand(&p.tm_a, pp.q, pp.units, pp.P, D, kQuarterRows)) return cudaErrorInvalidValue;
      return launch_pass<D, kOnePass>(p, s);
    }
  }
  // resident Q, streamed K (and V when the prompt's attention output is wanted)
  if (pp.out != nullptr) {
    if (!encode_operand(&p.tm_v, pp.v, pp.units, pp.P, D)) return cudaErrorInvalidValue;
    e = launch_pass<D, kRowOut>(p, s);
  } else {
    e = launch_pass<D, kRowStats>(p, s);
  }
  if (e != cudaSuccess) return e;
  const CUtensorMap q_map = p.tm_a;
  p.tm_a = p.tm_b;  // resident K, streamed Q
  p.tm_b = q_map;
  p.row_max_in = pp.row_max;
  p.row_sum_in = pp.row_sum;
  p.last_row_only = pp.last_row_only;
  return launch_pass<D, kColSums>(p, s);
}

}  // namespace

cudaError_t launch_prefill_scores_tc(const PrefillParams& p, int head_dim, cudaStream_t s) {
  return head_dim == 64 ? launch_typed<64>(p, s) : launch_typed<128>(p, s);
}

}  // namespace h2o
