// grad.cu -- the batched (non-recurrent) part of the backward pass: weight,
// bias, input and initial-state gradients from the deltas of every step.
//
// With delta_t = dL/da_t from the reverse recurrence (all T steps at once,
// K = T*B rows of [H]):
//   db  = column sums of delta                       (colsum_kernel)
//   dWh = delta^T [h0 ; y_0 .. y_{T-2}]              (gemm_tn_kernel)
//   dWx = delta^T x                                  (gemm_tn_kernel)
//   dx  = delta Wx,  dh0 = delta_0 Wh                (gemm_nn_kernel)
// For sparse Wh the weight gradient is needed only at the stored entries:
//   dvals[r][j] = sum_k delta[k][r] * Hprev[k][cols[r][j]]
// in fp32 as dot products of rows of the transposed delta and Hprev (each a
// contiguous T*B vector; sddmm_kernel), or for fp16 layers as the dense
// product on the tensor cores picked at the pattern (gather_pattern_kernel);
// dh0 = Wh^T delta_0 walks the rows of the padded Wh^T (sparse_dh0_kernel).
// They are the products the chain rule gives for the layer's two matrix
// products; like the forward projection they carry no dependence between
// steps and run as whole-sequence GEMMs ("Optimizing Performance of
// Recurrent Neural Networks on GPUs", Abstract: independent operations are
// batched rather than run step by step).  fp32 CUDA-core tiles (64 x 64 outputs per CTA, 16-deep K
// slices staged in shared memory, 4 x 4 outputs per thread): the gradients
// are kept in full fp32, and these GEMMs are a few percent of a training
// step next to the serial recurrences.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "prnn_internal.h"

namespace prnn {
namespace {

constexpr int kTile = 64, kBK = 16, kThreads = 256;

__device__ __forceinline__ float load_w(const void* w, size_t i, bool f16) {
  return f16 ? __half2float(static_cast<const __half*>(w)[i]) : static_cast<const float*>(w)[i];
}

// C[M][N] = sum_k A[k][m] * Brow(k)[n]; A row-major [K][lda]; row k of B is
// B0 + k*ldb for k < K0 (zeros when B0 is null) and B1 + (k-K0)*ldb after.
__global__ void __launch_bounds__(kThreads) gemm_tn_kernel(GemmTnArgs g) {
  __shared__ float As[kBK][kTile];
  __shared__ float Bs[kBK][kTile];
  const int tid = threadIdx.x;
  const int tm = tid / 16, tn = tid % 16;  // 16 x 16 threads, 4 x 4 outputs each
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += kBK) {
    for (int i = tid; i < kBK * kTile; i += kThreads) {
      const int kk = i / kTile, c = i % kTile;
      const int k = k0 + kk;
      float a = 0.f, b = 0.f;
      if (k < g.K) {
        if (m0 + c < g.M) a = g.A[(size_t)k * g.lda + m0 + c];
        if (n0 + c < g.N) {
          const float* row = k < g.K0 ? (g.B0 ? g.B0 + (size_t)k * g.ldb : nullptr)
                                      : g.B1 + (size_t)(k - g.K0) * g.ldb;
          if (row) b = row[n0 + c];
        }
      }
      As[kk][c] = a;
      Bs[kk][c] = b;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[kk][tm * 4 + i];
        bv[i] = Bs[kk][tn * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tn * 4 + j;
      if (n < g.N) g.C[(size_t)m * g.N + n] = acc[i][j];
    }
  }
}

// C[M][N] = sum_k A[m][k] * W[k][n]; A row-major [M][lda] fp32, W row-major
// [K][ldw] in fp32 or fp16.
__global__ void __launch_bounds__(kThreads) gemm_nn_kernel(GemmNnArgs g) {
  __shared__ float As[kBK][kTile];
  __shared__ float Ws[kBK][kTile];
  const int tid = threadIdx.x;
  const int tm = tid / 16, tn = tid % 16;
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += kBK) {
    for (int i = tid; i < kBK * kTile; i += kThreads) {
      const int kk = i % kBK, r = i / kBK;  // A: consecutive threads walk k
      const int k = k0 + kk;
      As[kk][r] = (k < g.K && m0 + r < g.M) ? g.A[(size_t)(m0 + r) * g.lda + k] : 0.f;
    }
    for (int i = tid; i < kBK * kTile; i += kThreads) {
      const int kk = i / kTile, c = i % kTile;
      const int k = k0 + kk;
      Ws[kk][c] = (k < g.K && n0 + c < g.N) ? load_w(g.W, (size_t)k * g.ldw + n0 + c, g.wf16)
                                            : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float av[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[kk][tm * 4 + i];
        wv[i] = Ws[kk][tn * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tn * 4 + j;
      if (n < g.N) g.C[(size_t)m * g.N + n] = acc[i][j];
    }
  }
}

// out[n] = sum_k A[k][n] for k < K (A row-major [K][N]): a block of 32 x 32
// threads owns 32 columns; thread (x, y) sums rows y, y + 32, ... of column
// x (coalesced over x), then the 32 partial sums of a column are added in
// shared memory in a fixed order.
__global__ void colsum_kernel(const float* A, int K, int N, float* out) {
  __shared__ float part[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int n = blockIdx.x * 32 + tx;
  float s = 0.f;
  if (n < N)
    for (int k = ty; k < K; k += 32) s += A[(size_t)k * N + n];
  part[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && n < N) {
    float t = 0.f;
    for (int i = 0; i < 32; ++i) t += part[i][tx];
    out[n] = t;
  }
}

// out[n][k] = Brow(k)[n] for k < K, n < N (Brow as in gemm_tn: B0 rows for
// k < K0, zeros if B0 is null, then B1 rows); 32 x 32 tiles through smem.
__global__ void transpose_rows_kernel(int K, int N, int K0, const float* B0, const float* B1,
                                      int ldb, float* out) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8 threads
  for (int i = ty; i < 32; i += 8) {
    const int k = k0 + i, n = n0 + tx;
    float v = 0.f;
    if (k < K && n < N) {
      const float* row = k < K0 ? (B0 ? B0 + (size_t)k * ldb : nullptr)
                                : B1 + (size_t)(k - K0) * ldb;
      if (row) v = row[n];
    }
    tile[i][tx] = v;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int n = n0 + i, k = k0 + tx;
    if (n < N && k < K) out[(size_t)n * K + k] = tile[tx][i];
  }
}

// One warp per row r of the padded forward layout: for each stored entry
// (r, cols[r][j]) the dot product of dT[r] and hT[cols[r][j]] (length K),
// written to out[caller_pos[r][j]] (padding entries are skipped).
__global__ void sddmm_kernel(int H, int kp, int K, const float* dT, const float* hT,
                             const uint16_t* cols, const int32_t* caller_pos, float* out) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= H) return;
  const int r = warp;
  const float* dr = dT + (size_t)r * K;
  for (int j = 0; j < kp; ++j) {
    const int pos = caller_pos[(size_t)r * kp + j];
    if (pos < 0) continue;
    const float* hc = hT + (size_t)cols[(size_t)r * kp + j] * K;
    float s = 0.f;
    for (int k = lane; k < K; k += 32) s = fmaf(dr[k], hc[k], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) out[pos] = s;
  }
}

// dh0[b][c] = sum_j valsT[c][j] * delta0[b][colsT[c][j]] (Wh^T padded rows).
__global__ void sparse_dh0_kernel(int B, int H, int kT, const uint16_t* valsT,
                                  const uint16_t* colsT, const float* delta0, float* dh0) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * H) return;
  const int b = i / H, c = i % H;
  float s = 0.f;
  for (int j = 0; j < kT; ++j) {
    const float v = __half2float(__ushort_as_half(valsT[(size_t)c * kT + j]));
    s = fmaf(v, delta0[(size_t)b * H + colsT[(size_t)c * kT + j]], s);
  }
  dh0[i] = s;
}

// out[n][k] = bf16(Brow(k)[n]) for k < K, 0 for K <= k < Kp (Brow as in
// transpose_rows_kernel): the K-major bf16 operands of the tensor-core
// gradient products.
__global__ void transpose_bf16_kernel(int K, int Kp, int N, int K0, const float* B0,
                                      const float* B1, int ldb, __nv_bfloat16* out) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8 threads
  for (int i = ty; i < 32; i += 8) {
    const int k = k0 + i, n = n0 + tx;
    float v = 0.f;
    if (k < K && n < N) {
      const float* row = k < K0 ? (B0 ? B0 + (size_t)k * ldb : nullptr)
                                : B1 + (size_t)(k - K0) * ldb;
      if (row) v = row[n];
    }
    tile[i][tx] = v;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int n = n0 + i, k = k0 + tx;
    if (n < N && k < Kp) out[(size_t)n * Kp + k] = __float2bfloat16_rn(tile[tx][i]);
  }
}

// out[m][k] = bf16(src[m][k]) for k < K, 0 for K <= k < Kp.
__global__ void rows_bf16_kernel(int M, int K, int Kp, const float* src, __nv_bfloat16* out) {
  const size_t total = (size_t)M * Kp;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / Kp), k = (int)(i % Kp);
    out[i] = __float2bfloat16_rn(k < K ? src[(size_t)m * K + k] : 0.f);
  }
}

// out[i] = y[i] > 0 ? dy[i] : kMaskedMarker: the ReLU mask folded into the
// reverse recurrence's P (see kMaskedMarker).
__global__ void fold_mask_kernel(const float* dy, const float* y, size_t n, float* out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = y[i] > 0.f ? dy[i] : __uint_as_float(kMaskedMarker);
}

// out[caller_pos[r][j]] = dense[r][cols[r][j]] for the stored entries: the
// sparse value gradients picked out of a dense dWh.
__global__ void gather_pattern_kernel(int H, int kp, const float* dense, const uint16_t* cols,
                                      const int32_t* caller_pos, float* out) {
  const size_t n = (size_t)H * kp;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int pos = caller_pos[i];
    if (pos >= 0) out[pos] = dense[(i / kp) * H + cols[i]];
  }
}

}  // namespace

cudaError_t launch_gather_pattern(int H, int kp, const float* dense, const uint16_t* cols,
                                  const int32_t* caller_pos, float* out, cudaStream_t s) {
  const size_t n = (size_t)H * kp;
  if (n == 0) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
  gather_pattern_kernel<<<blocks, 256, 0, s>>>(H, kp, dense, cols, caller_pos, out);
  return cudaGetLastError();
}

cudaError_t launch_fold_mask(const float* dy, const float* y, size_t n, float* out,
                             cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
  fold_mask_kernel<<<blocks, 256, 0, s>>>(dy, y, n, out);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(int K, int Kp, int N, int K0, const float* B0, const float* B1,
                                  int ldb, void* out, cudaStream_t s) {
  if (Kp <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + 31) / 32, (Kp + 31) / 32), block(32, 8);
  transpose_bf16_kernel<<<grid, block, 0, s>>>(K, Kp, N, K0, B0, B1, ldb,
                                               static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_rows_bf16(int M, int K, int Kp, const float* src, void* out, cudaStream_t s) {
  if (M <= 0 || Kp <= 0) return cudaSuccess;
  const size_t total = (size_t)M * Kp;
  const int blocks = (int)((total + 255) / 256 < 8192 ? (total + 255) / 256 : 8192);
  rows_bf16_kernel<<<blocks, 256, 0, s>>>(M, K, Kp, src, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_transpose_rows(int K, int N, int K0, const float* B0, const float* B1, int ldb,
                                  float* out, cudaStream_t s) {
  if (K <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
  transpose_rows_kernel<<<grid, block, 0, s>>>(K, N, K0, B0, B1, ldb, out);
  return cudaGetLastError();
}

cudaError_t launch_sddmm(int H, int kp, int K, const float* dT, const float* hT,
                         const uint16_t* cols, const int32_t* caller_pos, float* out,
                         cudaStream_t s) {
  if (H <= 0) return cudaSuccess;
  sddmm_kernel<<<(H * 32 + 255) / 256, 256, 0, s>>>(H, kp, K, dT, hT, cols, caller_pos, out);
  return cudaGetLastError();
}

cudaError_t launch_sparse_dh0(int B, int H, int kT, const uint16_t* valsT, const uint16_t* colsT,
                              const float* delta0, float* dh0, cudaStream_t s) {
  if (B * H <= 0) return cudaSuccess;
  sparse_dh0_kernel<<<(B * H + 255) / 256, 256, 0, s>>>(B, H, kT, valsT, colsT, delta0, dh0);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tn(const GemmTnArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  dim3 grid((g.N + kTile - 1) / kTile, (g.M + kTile - 1) / kTile);
  gemm_tn_kernel<<<grid, kThreads, 0, s>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nn(const GemmNnArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  dim3 grid((g.N + kTile - 1) / kTile, (g.M + kTile - 1) / kTile);
  gemm_nn_kernel<<<grid, kThreads, 0, s>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_colsum(const float* A, int K, int N, float* out, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  colsum_kernel<<<(N + 31) / 32, dim3(32, 32), 0, s>>>(A, K, N, out);
  return cudaGetLastError();
}

}  // namespace prnn
