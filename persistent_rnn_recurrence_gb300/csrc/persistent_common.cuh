// persistent_common.cuh -- pieces shared by the persistent recurrent kernels
// (dense, sparse and the sync-floor probe): the CTA's place in the grid, the
// grid barrier of the ablation mode, warp reductions, h staging and the
// cooperative launch helper.  Included by one translation unit each.
#pragma once

#include "device_common.cuh"
#include "prnn_internal.h"

namespace prnn {
namespace pk {


constexpr int kSparseThreads = 512;
constexpr int kCptMax = 4;          // 4-column chunks per thread of the dense kernel
constexpr int kRegQ = 4;            // sparse: uint4 weight groups held in registers
constexpr int kRegWThreads = 384;   // sparse register-weight build: threads per CTA at most
constexpr int kRegQWide = 6;        // ... and the uint4 weight groups it holds in registers

__device__ __forceinline__ unsigned ld_acquire_u(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The CTA's place in the grid: group gi (batch columns [b_lo, b_hi)) and the
// CTA's index lc within its group (rows row0 .. row0 + rows - 1).
struct Place {
  int lc, row0, rows, b_lo, b_hi;
};
__device__ __forceinline__ Place place_of(const RecurCommon& c) {
  Place p;
  const int gi = blockIdx.x / c.cpg;
  p.lc = blockIdx.x % c.cpg;
  p.row0 = p.lc * c.R;
  p.rows = max(0, min(c.R, c.H - p.row0));
  const int bl = (c.B + c.G - 1) / c.G;
  p.b_lo = min(c.B, gi * bl);
  p.b_hi = min(c.B, p.b_lo + bl);
  return p;
}

// Grid barrier (ablation only).  Counter is zeroed before the launch; the
// barrier after step t waits until it reaches (t+1)*n_cta.
__device__ __forceinline__ void grid_barrier(const RecurCommon& c, int t, Waiter& w,
                                             int* s_abort) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(c.bar, 1u);
    const unsigned target = (unsigned)(t + 1) * (unsigned)c.n_cta;
    uint32_t spins = 0;
    while (ld_acquire_u(c.bar) < target) {
      if (!w.still_ok(spins)) {
        report_timeout(c.status, t, blockIdx.x);
        *s_abort = 1;
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// Segmented reduce-scatter over groups of G lanes (G a power of two <= 32).
// After it, lane gl = lane % G holds value indices gl*V/G + i (V >= G) or
// gl/(G/V) (V < G, replicated).
template <int V, int G>
__device__ __forceinline__ void seg_reduce_scatter(float (&v)[V], int lane) {
  constexpr unsigned kFull = 0xffffffffu;
  int n = V;
#pragma unroll
  for (int o = G / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (lane & o) != 0;
      const int h = n >> 1;
#pragma unroll
      for (int i = 0; i < V / 2; ++i) {
        if (i < h) {
          float send = upper ? v[i] : v[i + h];
          float keep = upper ? v[i + h] : v[i];
          v[i] = keep + __shfl_xor_sync(kFull, send, o);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], o);
    }
  }
}

// ---------------------------------------------------------------------------
// Stage nb consecutive batch rows (from row b_start) of h_{t-1} (layout
// [b][H] in y) into smem with the same layout: a straight float4 copy,
// conflict-free.  A thread keeps up to UMAX float4 loads in flight; while any
// is still the sentinel it re-issues all of its stale loads together (one
// round trip per round) until every word is fresh.  Returns false if the wait
// gave up.  With rounds_out (the phase trace), the largest number of re-poll
// rounds any of the thread's load batches needed is recorded there.
// ---------------------------------------------------------------------------
template <int UMAX>
__device__ __forceinline__ bool stage_rows(const float* hprev, bool poll, int H, int b_start,
                                           int nb, float* hs, Waiter& w,
                                           uint32_t* rounds_out = nullptr) {
  const int NT = blockDim.x, tid = threadIdx.x;
  const int nf4 = (nb * H) >> 2;
  const float4* src = reinterpret_cast<const float4*>(hprev + (size_t)b_start * H);
  float4* dst = reinterpret_cast<float4*>(hs);
  for (int base = tid; base < nf4; base += UMAX * NT) {
    float4 v[UMAX];
#pragma unroll
    for (int u = 0; u < UMAX; ++u) {
      const int i = base + u * NT;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nf4 && hprev != nullptr)
        v[u] = poll ? ld_relaxed_f4(reinterpret_cast<const float*>(src + i)) : __ldg(src + i);
    }
    if (poll) {
      uint32_t spins = 0, round = 0;
      for (;;) {
        unsigned stale = 0;
#pragma unroll
        for (int u = 0; u < UMAX; ++u)
          if (base + u * NT < nf4 && !ready4(v[u])) stale |= 1u << u;
        if (stale == 0u) break;
        if (!w.still_ok(spins)) return false;
        w.pause(round);
#pragma unroll
        for (int u = 0; u < UMAX; ++u)
          if ((stale >> u) & 1u) v[u] = ld_relaxed_f4(reinterpret_cast<const float*>(src + base + u * NT));
      }
      if (rounds_out != nullptr && round > *rounds_out) *rounds_out = round;
    }
#pragma unroll
    for (int u = 0; u < UMAX; ++u)
      if (base + u * NT < nf4) dst[base + u * NT] = v[u];
  }
  return true;
}

// The same staging with 32-bit loads and stores: the "without wide memory
// loads" side of the ablation (four times the load instructions and poll
// checks for the same bytes).
template <int UMAX>
__device__ __forceinline__ bool stage_rows_narrow(const float* hprev, bool poll, int H,
                                                  int b_start, int nb, float* hs, Waiter& w) {
  const int NT = blockDim.x, tid = threadIdx.x;
  const int n = nb * H;
  const float* src = hprev + (size_t)b_start * H;
  for (int base = tid; base < n; base += UMAX * NT) {
    float v[UMAX];
#pragma unroll
    for (int u = 0; u < UMAX; ++u) {
      const int i = base + u * NT;
      v[u] = 0.f;
      if (i < n && hprev != nullptr) v[u] = poll ? ld_relaxed_f(src + i) : __ldg(src + i);
    }
    if (poll) {
      uint32_t spins = 0, round = 0;
      for (;;) {
        unsigned stale = 0;
#pragma unroll
        for (int u = 0; u < UMAX; ++u)
          if (base + u * NT < n && is_sentinel(v[u])) stale |= 1u << u;
        if (stale == 0u) break;
        if (!w.still_ok(spins)) return false;
        w.pause(round);
#pragma unroll
        for (int u = 0; u < UMAX; ++u)
          if ((stale >> u) & 1u) v[u] = ld_relaxed_f(src + base + u * NT);
      }
    }
#pragma unroll
    for (int u = 0; u < UMAX; ++u)
      if (base + u * NT < n) hs[base + u * NT] = v[u];
  }
  return true;
}

template <typename K>
cudaError_t coop_launch(K kernel, int grid, int block, size_t smem, cudaStream_t s, void** args) {
  // One CTA per SM: a persistent grid with fewer CTAs than SMs must not have
  // two CTAs share an SM (the block scheduler may pack them when registers and
  // shared memory allow, and the shared SM then sets every step's pace).
  // Asking for more than half of an SM's shared memory rules that out.
  int dev = 0, per_sm_smem = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const size_t one_per_sm = (size_t)per_sm_smem / 2 + 1024;
  if (smem < one_per_sm && one_per_sm <= (size_t)optin) smem = one_per_sm;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kernel), dim3(grid),
                                     dim3(block), args, smem, s);
}

}  // namespace pk
}  // namespace prnn
