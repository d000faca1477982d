// per_step.cu -- the non-persistent comparison path: one launch per step,
// y[t] = ReLU(P[t] + Wh h_{t-1}), with Wh read again from L2/HBM every step.
// This is the weights-re-read-every-step pattern that the persistent-rnn page
// contrasts with its register-cached kernel ("What This Project Does"),
// and the per-step dense / sparse matrix-product baselines of the sparse
// persistent RNN measurements.  The T launches are replayed as one CUDA graph.
#include "device_common.cuh"
#include "prnn_internal.h"

namespace prnn {

namespace {

constexpr int kRowsPerCta = 8;  // one warp per row

template <int V>
__device__ __forceinline__ void warp_sum_scatter(float (&v)[V], int lane) {
  warp_reduce_scatter<V>(v, lane);
}

// Dense: warp per row; lanes stride over 4-column chunks of the row (8 or 16
// byte weight loads, coalesced across the warp); h read through L1.
template <bool F16, int BMAX>
__global__ void __launch_bounds__(kRowsPerCta * 32) step_dense_kernel(const StepArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= a.H) return;
  const int H = a.H, B = a.B;
  float acc[BMAX];
#pragma unroll
  for (int b = 0; b < BMAX; ++b) acc[b] = 0.f;
  if (a.hprev != nullptr) {
    if ((H & 3) == 0) {
      for (int c = lane * 4; c < H; c += 128) {
        float w0, w1, w2, w3;
        if (F16) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(
              static_cast<const __half*>(a.W) + (size_t)row * H + c));
          const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
          const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
          w0 = f0.x; w1 = f0.y; w2 = f1.x; w3 = f1.y;
        } else {
          const float4 f = __ldg(reinterpret_cast<const float4*>(
              static_cast<const float*>(a.W) + (size_t)row * H + c));
          w0 = f.x; w1 = f.y; w2 = f.z; w3 = f.w;
        }
#pragma unroll
        for (int b = 0; b < BMAX; ++b) {
          if (b < B) {
            const float4 h = __ldg(reinterpret_cast<const float4*>(a.hprev + (size_t)b * H + c));
            float s = acc[b];
            s = fmaf(w0, h.x, s);
            s = fmaf(w1, h.y, s);
            s = fmaf(w2, h.z, s);
            s = fmaf(w3, h.w, s);
            acc[b] = s;
          }
        }
      }
    } else {  // ragged H: scalar loads
      for (int c = lane; c < H; c += 32) {
        const float wv = F16 ? __half2float(static_cast<const __half*>(a.W)[(size_t)row * H + c])
                             : static_cast<const float*>(a.W)[(size_t)row * H + c];
#pragma unroll
        for (int b = 0; b < BMAX; ++b)
          if (b < B) acc[b] = fmaf(wv, __ldg(a.hprev + (size_t)b * H + c), acc[b]);
      }
    }
  }
  warp_sum_scatter<BMAX>(acc, lane);
  constexpr int REP = (BMAX >= 32) ? 1 : 32 / BMAX;
  constexpr int NOUT = (BMAX >= 32) ? BMAX / 32 : 1;
  const float* Pt = a.P + (size_t)a.t * B * H;
  float* yt = a.y + (size_t)a.t * B * H;
  if (lane % REP == 0) {
#pragma unroll
    for (int i = 0; i < NOUT; ++i) {
      const int b = (BMAX >= 32) ? lane * NOUT + i : lane / REP;
      if (b < B) yt[(size_t)b * H + row] = relu(acc[i] + __ldg(Pt + (size_t)b * H + row));
    }
  }
}

// Sparse row-balanced: warp per row, lanes stride over the row's k packed
// entries (fp16 value | column << 16); h gathered through L1.
template <int BMAX>
__global__ void __launch_bounds__(kRowsPerCta * 32) step_sparse_kernel(const StepArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= a.H) return;
  const int H = a.H, B = a.B, k = a.kp;
  const uint32_t* W = static_cast<const uint32_t*>(a.W) + (size_t)row * k;
  float acc[BMAX];
#pragma unroll
  for (int b = 0; b < BMAX; ++b) acc[b] = 0.f;
  if (a.hprev != nullptr) {
    for (int j = lane; j < k; j += 32) {
      const uint32_t e = __ldg(W + j);
      const float val = __half2float(__ushort_as_half((unsigned short)(e & 0xffffu)));
      const int col = (int)(e >> 16);
#pragma unroll
      for (int b = 0; b < BMAX; ++b)
        if (b < B) acc[b] = fmaf(val, __ldg(a.hprev + (size_t)b * H + col), acc[b]);
    }
  }
  warp_sum_scatter<BMAX>(acc, lane);
  constexpr int REP = (BMAX >= 32) ? 1 : 32 / BMAX;
  constexpr int NOUT = (BMAX >= 32) ? BMAX / 32 : 1;
  const float* Pt = a.P + (size_t)a.t * B * H;
  float* yt = a.y + (size_t)a.t * B * H;
  if (lane % REP == 0) {
#pragma unroll
    for (int i = 0; i < NOUT; ++i) {
      const int b = (BMAX >= 32) ? lane * NOUT + i : lane / REP;
      if (b < B) yt[(size_t)b * H + row] = relu(acc[i] + __ldg(Pt + (size_t)b * H + row));
    }
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const dim3 grid((a.H + kRowsPerCta - 1) / kRowsPerCta), block(kRowsPerCta * 32);
  const int bmax = a.B <= 4 ? 4 : a.B <= 8 ? 8 : a.B <= 16 ? 16 : 32;
  if (a.B > 32) return cudaErrorInvalidValue;
#define PRNN_STEP(BM)                                                    \
  if (bmax == BM) {                                                      \
    if (a.sparse)                                                        \
      step_sparse_kernel<BM><<<grid, block, 0, s>>>(a);                  \
    else if (a.wfp16)                                                    \
      step_dense_kernel<true, BM><<<grid, block, 0, s>>>(a);             \
    else                                                                 \
      step_dense_kernel<false, BM><<<grid, block, 0, s>>>(a);            \
    return cudaGetLastError();                                           \
  }
  PRNN_STEP(4) PRNN_STEP(8) PRNN_STEP(16) PRNN_STEP(32)
#undef PRNN_STEP
  return cudaErrorInvalidValue;
}

}  // namespace prnn
