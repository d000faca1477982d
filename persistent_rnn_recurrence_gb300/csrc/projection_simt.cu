// projection_simt.cu -- fp32 CUDA-core input projection and the y sentinel fill.
//
// P[m][n] = bias[n] + sum_k x[m][k] * Wx[n][k] for all m = t*B + b at once:
// the input half of every step does not depend on h_{t-1}, so it is taken out
// of the serial loop as one matrix product (work independent of the previous
// step is batched across steps: Abstract of "Optimizing Performance of
// Recurrent Neural Networks on GPUs").  This kernel is the fp32 path (fp32 weights need full
// fp32 products; TF32 tensor cores would round x and Wx to 10-bit mantissas).
// It also serves fp16 weights when tensor cores are switched off.
#include "device_common.cuh"
#include "prnn_internal.h"

namespace prnn {

namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;

__device__ __forceinline__ float load_w(const void* W, size_t i, bool f16) {
  if (f16) return __half2float(__ushort_as_half(static_cast<const unsigned short*>(W)[i]));
  return static_cast<const float*>(W)[i];
}

// 64x64 output tile per CTA, 256 threads, 4x4 outputs per thread.
template <bool F16>
__global__ void __launch_bounds__(256) proj_simt_kernel(const ProjArgs a) {
  __shared__ float As[kTK][kTM + 4];
  __shared__ float Bs[kTK][kTN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.K; k0 += kTK) {
    // each thread stages 4 elements of A and 4 of B (row tid/4, k (tid%4)*4 + i)
    const int lr = tid >> 2, lk = (tid & 3) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = k0 + lk + i;
      const int m = m0 + lr, n = n0 + lr;
      As[lk + i][lr] = (m < a.M && k < a.K) ? __ldg(a.x + (size_t)m * a.K + k) : 0.f;
      Bs[lk + i][lr] = (n < a.N && k < a.K) ? load_w(a.Wx, (size_t)n * a.K + k, F16) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      a.P[(size_t)m * a.N + n] = acc[i][j] + __ldg(a.bias + n);
      if (a.y_fill) a.y_fill[(size_t)m * a.N + n] = __uint_as_float(kSentinel);
    }
  }
}

__global__ void fill_sentinel_kernel(float* y, size_t n) {
  const float s = __uint_as_float(kSentinel);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    y[i] = s;
}

}  // namespace

cudaError_t launch_projection_simt(const ProjArgs& a, bool wx_fp16, cudaStream_t s) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  dim3 grid((a.N + kTN - 1) / kTN, (a.M + kTM - 1) / kTM);
  if (wx_fp16)
    proj_simt_kernel<true><<<grid, 256, 0, s>>>(a);
  else
    proj_simt_kernel<false><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fill_sentinel(float* y, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  fill_sentinel_kernel<<<blocks, 256, 0, s>>>(y, n);
  return cudaGetLastError();
}

}  // namespace prnn
