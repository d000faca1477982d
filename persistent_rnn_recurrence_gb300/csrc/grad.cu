// grad.cu -- the batched (non-recurrent) part of the backward pass: weight,
// bias, input and initial-state gradients from the deltas of every step.
//
// With delta_t = dL/da_t from the reverse recurrence (all T steps at once,
// K = T*B rows of [H]):
//   db  = column sums of delta                       (colsum_kernel)
//   dWh = delta^T [h0 ; y_0 .. y_{T-2}]              (gemm_tn_kernel)
//   dWx = delta^T x                                  (gemm_tn_kernel)
//   dx  = delta Wx,  dh0 = delta_0 Wh                (gemm_nn_kernel)
// They are the products the chain rule gives for the layer's two matrix
// products; like the forward projection they carry no dependence between
// steps and run as whole-sequence GEMMs ("Optimizing Performance of
// Recurrent Neural Networks on GPUs", Abstract: exposing parallelism between
// operations).  fp32 CUDA-core tiles (64 x 64 outputs per CTA, 16-deep K
// slices staged in shared memory, 4 x 4 outputs per thread): the gradients
// are kept in full fp32, and these GEMMs are a few percent of a training
// step next to the serial recurrences.
#include <cuda_fp16.h>

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

// out[n] = sum_k A[k][n] for k < K (A row-major [K][N]).
__global__ void colsum_kernel(const float* A, int K, int N, float* out) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float s = 0.f;
  for (int k = 0; k < K; ++k) s += A[(size_t)k * N + n];
  out[n] = s;
}

}  // namespace

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
  colsum_kernel<<<(N + 255) / 256, 256, 0, s>>>(A, K, N, out);
  return cudaGetLastError();
}

}  // namespace prnn
