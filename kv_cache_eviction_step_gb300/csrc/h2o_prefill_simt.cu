// h2o_prefill_simt.cu -- prefill score pass on the CUDA cores (hot-path rows P1-P2).
//
//   P1  for every prompt row i: m_i = max_{j<=i} s_ij and l_i = sum_{j<=i} exp(s_ij - m_i), with
//       s_ij = (q_i . k_j) / sqrt(D) (causal Softmax(QK^T/sqrt(d)), H2O post §2.1.1)
//   P2  column sums c_j = sum_{i>=j} exp(s_ij - m_i) / l_i: the attention each prompt token has
//       accumulated over the prompt (H2O post §2.1.2 / §2.2; "H2O Heavy-Hitter Oracle 分析" §3.1)
//   and, when asked for, the prompt's attention output o_i = sum_{j<=i} exp(s_ij - m_i) / l_i v_j.
//
// This is the float32 path (a tensor-core f32 contraction would round the products through tf32)
// and the plain reference-shaped path for bf16. A block of 128 threads owns 32 consecutive rows
// (P1) or columns (P2) of one unit; the 32 x D query/key tile it owns is staged in shared memory
// and the opposite operand is streamed in tiles of 32 rows, so every thread computes dot products
// from shared memory: thread (r, c) of a 32 x 4 grid takes row r against columns c, c+4, ...
#include <cuda_bf16.h>
#include <math.h>

#include "h2o_internal.cuh"

namespace h2o {
namespace {

constexpr int kTile = 32;       // rows (or columns) per block and per streamed tile
constexpr int kLanesX = 4;      // threads sharing one owned row
constexpr int kThreads = kTile * kLanesX;

template <typename T>
__device__ __forceinline__ float ld(const T* p, size_t i) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(p[i]);
  else return p[i];
}

// Copy a [rows, D] tile (rows beyond `valid` zero-filled) to shared memory as float.
template <typename T, int D>
__device__ __forceinline__ void stage(float (*dst)[D + 1], const T* src, int valid) {
  for (int e = threadIdx.x; e < kTile * D; e += kThreads) {
    const int r = e / D, d = e % D;
    dst[r][d] = r < valid ? ld(src, static_cast<size_t>(r) * D + d) : 0.f;
  }
}

template <int D>
__device__ __forceinline__ float dot_rows(const float (*a)[D + 1], int ra, const float (*b)[D + 1], int rb) {
  float acc = 0.f;
#pragma unroll 8
  for (int d = 0; d < D; ++d) acc = fmaf(a[ra][d], b[rb][d], acc);
  return acc;
}

// P1: row statistics. Block (x = unit, y = row tile).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_row_stats_kernel(const PrefillParams p) {
  __shared__ float qs[kTile][D + 1];
  __shared__ float ks[kTile][D + 1];
  __shared__ float red_m[kTile][kLanesX];
  __shared__ float red_l[kTile][kLanesX];
  const int unit = blockIdx.x;
  const int i0 = blockIdx.y * kTile;
  const int r = threadIdx.x / kLanesX, c = threadIdx.x % kLanesX;
  const size_t base = static_cast<size_t>(unit) * p.P;
  const T* q = static_cast<const T*>(p.q) + base * D;
  const T* k = static_cast<const T*>(p.k) + base * D;
  stage<T, D>(qs, q + static_cast<size_t>(i0) * D, p.P - i0);
  const int i = i0 + r;
  float m = -INFINITY, l = 0.f;  // online over this thread's columns
  for (int j0 = 0; j0 <= i0 + kTile - 1 && j0 < p.P; j0 += kTile) {
    __syncthreads();
    stage<T, D>(ks, k + static_cast<size_t>(j0) * D, p.P - j0);
    __syncthreads();
    for (int cc = c; cc < kTile; cc += kLanesX) {
      const int j = j0 + cc;
      if (j > i || i >= p.P) continue;
      const float s = dot_rows<D>(qs, r, ks, cc) * p.scale;
      if (s > m) {
        l = l * expf(m - s) + 1.f;
        m = s;
      } else {
        l += expf(s - m);
      }
    }
  }
  red_m[r][c] = m;
  red_l[r][c] = l;
  __syncthreads();
  if (c == 0 && i < p.P) {
    float mm = -INFINITY;
    for (int x = 0; x < kLanesX; ++x) mm = fmaxf(mm, red_m[r][x]);
    float ll = 0.f;
    for (int x = 0; x < kLanesX; ++x)
      if (red_l[r][x] > 0.f) ll += red_l[r][x] * expf(red_m[r][x] - mm);
    p.row_max[base + i] = mm;
    p.row_sum[base + i] = ll;
  }
}

// P2: column sums. Block (x = unit, y = column tile).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_colsum_kernel(const PrefillParams p) {
  __shared__ float ks[kTile][D + 1];
  __shared__ float qs[kTile][D + 1];
  __shared__ float mi[kTile], li[kTile];
  __shared__ float red[kTile][kLanesX];
  const int unit = blockIdx.x;
  const int j0 = blockIdx.y * kTile;
  const int r = threadIdx.x / kLanesX, c = threadIdx.x % kLanesX;
  const size_t base = static_cast<size_t>(unit) * p.P;
  const T* q = static_cast<const T*>(p.q) + base * D;
  const T* k = static_cast<const T*>(p.k) + base * D;
  stage<T, D>(ks, k + static_cast<size_t>(j0) * D, p.P - j0);
  const int j = j0 + r;
  float acc = 0.f;
  // The last-row variant (Top-K prefill) only needs the tile holding query P-1.
  const int i_first = p.last_row_only ? max(j0, (p.P - 1) / kTile * kTile) : j0;
  for (int i0 = i_first; i0 < p.P; i0 += kTile) {
    __syncthreads();
    stage<T, D>(qs, q + static_cast<size_t>(i0) * D, p.P - i0);
    if (threadIdx.x < kTile) {
      const int i = i0 + threadIdx.x;
      mi[threadIdx.x] = i < p.P ? p.row_max[base + i] : 0.f;
      li[threadIdx.x] = i < p.P ? p.row_sum[base + i] : 1.f;
    }
    __syncthreads();
    for (int cc = c; cc < kTile; cc += kLanesX) {
      const int i = i0 + cc;
      if (i < j || i >= p.P || j >= p.P || (p.last_row_only && i != p.P - 1)) continue;
      const float s = dot_rows<D>(ks, r, qs, cc) * p.scale;
      acc += expf(s - mi[cc]) / li[cc];
    }
  }
  red[r][c] = acc;
  __syncthreads();
  if (c == 0 && j < p.P) {
    float sum = 0.f;
    for (int x = 0; x < kLanesX; ++x) sum += red[r][x];
    p.colsum[base + j] = sum;
  }
}

// The prompt's attention output with the final row statistics of P1:
// o_i = sum_{j<=i} exp(s_ij - m_i) / l_i v_j. Block (x = unit, y = row tile); thread (r, c) computes
// the weights of row r against keys c, c+4, ... of each streamed tile into shared memory, then
// accumulates output elements c, c+4, ... of row r from the value tile staged in the same buffer.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_output_kernel(const PrefillParams p) {
  __shared__ float qs[kTile][D + 1];
  __shared__ float kv[kTile][D + 1];  // K tile, then V tile
  __shared__ float ps[kTile][kTile + 1];
  const int unit = blockIdx.x;
  const int i0 = blockIdx.y * kTile;
  const int r = threadIdx.x / kLanesX, c = threadIdx.x % kLanesX;
  const size_t base = static_cast<size_t>(unit) * p.P;
  const T* q = static_cast<const T*>(p.q) + base * D;
  const T* k = static_cast<const T*>(p.k) + base * D;
  const T* v = static_cast<const T*>(p.v) + base * D;
  stage<T, D>(qs, q + static_cast<size_t>(i0) * D, p.P - i0);
  const int i = i0 + r;
  const float mi = i < p.P ? p.row_max[base + i] : 0.f;
  const float il = i < p.P ? 1.f / p.row_sum[base + i] : 0.f;
  float acc[D / kLanesX];
#pragma unroll
  for (int e = 0; e < D / kLanesX; ++e) acc[e] = 0.f;
  for (int j0 = 0; j0 <= i0 + kTile - 1 && j0 < p.P; j0 += kTile) {
    __syncthreads();
    stage<T, D>(kv, k + static_cast<size_t>(j0) * D, p.P - j0);
    __syncthreads();
    for (int cc = c; cc < kTile; cc += kLanesX) {
      const int j = j0 + cc;
      ps[r][cc] = (j <= i && i < p.P && j < p.P) ? expf(dot_rows<D>(qs, r, kv, cc) * p.scale - mi) * il : 0.f;
    }
    __syncthreads();
    stage<T, D>(kv, v + static_cast<size_t>(j0) * D, p.P - j0);
    __syncthreads();
    for (int jj = 0; jj < kTile; ++jj) {
      const float w = ps[r][jj];
#pragma unroll
      for (int e = 0; e < D / kLanesX; ++e) acc[e] = fmaf(w, kv[jj][c + kLanesX * e], acc[e]);
    }
  }
  if (i < p.P) {
    T* o = static_cast<T*>(p.out) + (base + i) * D;
#pragma unroll
    for (int e = 0; e < D / kLanesX; ++e) {
      if constexpr (sizeof(T) == 2) o[c + kLanesX * e] = __float2bfloat16_rn(acc[e]);
      else o[c + kLanesX * e] = acc[e];
    }
  }
}

template <typename T, int D>
cudaError_t launch_typed(const PrefillParams& p, cudaStream_t s) {
  const dim3 grid(p.units, (p.P + kTile - 1) / kTile);
  prefill_row_stats_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.out != nullptr) {
    prefill_output_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  prefill_colsum_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_scores_simt(const PrefillParams& p, int head_dim, int dtype, cudaStream_t s) {
  if (dtype == H2O_BF16)
    return head_dim == 64 ? launch_typed<__nv_bfloat16, 64>(p, s) : launch_typed<__nv_bfloat16, 128>(p, s);
  return head_dim == 64 ? launch_typed<float, 64>(p, s) : launch_typed<float, 128>(p, s);
}

}  // namespace h2o
