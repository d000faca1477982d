// noalloc.cu -- a forward entry point that allocates no device memory.
//
// prnn_forward (the handle API) allocates: packed weights, the projection
// workspace P, status words.  Some callers cannot do that: code that runs
// inside a latency-critical loop where cudaMalloc/cudaFree may synchronize the
// whole device, or a process whose device memory is entirely owned by another
// allocator (a framework's caching pool) or capped by a fixed budget.  For
// them, prnn_forward_dense_noalloc computes the same layer from the caller's
// own buffers, using as its only scratch a file-scope device array of fixed
// size that the CUDA module carries (reserved on each GPU when the module is
// loaded there, released at process exit).
//
// It runs the per-step path: the fp32 CUDA-core projection writes
// P = Wx x + b for all steps into the scratch array, then T step kernels each
// read Wh (row-major, the caller's buffer) and y[t-1] and write y[t].
#include "prnn.h"
#include "prnn_internal.h"

namespace {

// Scratch for P[T][B][H]: 4 Mi floats (16 MiB) per device.
constexpr size_t kScratchFloats = (size_t)1 << 22;
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

// Device address of the scratch array on the current device.  Host code may
// not use the symbol itself (it is a host-side stand-in), so the address is
// looked up with that device current -- on every call, not cached: a cached
// address would outlive a cudaDeviceReset (after which the module, and the
// array, are loaded again, possibly elsewhere).  The lookup is a host-side
// query; the first one on a device may load the library's module there.
cudaError_t scratch_on_current_device(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" prnn_status_t prnn_forward_dense_noalloc(int T, int B, int H, int I,
                                                    prnn_dtype_t wdtype, const float* x,
                                                    const void* Wx, const void* Wh,
                                                    const float* bias, const float* h0,
                                                    float* y, void* stream) {
  if (T < 0 || B < 0 || B > 32 || H < 1 || I < 1) return PRNN_ERR_INVALID_ARG;
  if (wdtype != PRNN_F32 && wdtype != PRNN_F16) return PRNN_ERR_INVALID_ARG;
  if (T == 0 || B == 0) return PRNN_OK;
  if (!x || !Wx || !Wh || !bias || !y) return PRNN_ERR_INVALID_ARG;
  if (!aligned16(y) || (h0 && !aligned16(h0)) || !aligned16(Wh)) return PRNN_ERR_INVALID_ARG;
  if ((size_t)T * B * H > kScratchFloats) return PRNN_ERR_INVALID_ARG;  // beyond the scratch
  float* P = nullptr;
  if (scratch_on_current_device(&P) != cudaSuccess) return PRNN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prnn::ProjArgs pa{T * B, H, I, x, Wx, bias, P, nullptr};
  if (prnn::launch_projection_simt(pa, wdtype == PRNN_F16, s) != cudaSuccess) return PRNN_ERR_CUDA;
  for (int t = 0; t < T; ++t) {
    prnn::StepArgs sa{};
    sa.t = t;
    sa.B = B;
    sa.H = H;
    sa.P = P;
    sa.hprev = t == 0 ? h0 : y + (size_t)(t - 1) * B * H;
    sa.y = y;
    sa.W = Wh;
    sa.wfp16 = wdtype == PRNN_F16;
    sa.sparse = 0;
    sa.kp = 0;
    if (prnn::launch_step(sa, s) != cudaSuccess) return PRNN_ERR_CUDA;
  }
  return PRNN_OK;
}
