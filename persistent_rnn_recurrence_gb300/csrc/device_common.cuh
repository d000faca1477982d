// device_common.cuh -- device helpers shared by the recurrent kernels:
// coherent (L1-bypassing) loads and stores of step data, the "not yet written"
// sentinel, bounded waiting with an error status, and warp reductions.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace prnn {

// A y word that has not been produced yet holds this bit pattern.  It is a
// NaN, and the ReLU used here (v > 0 ? v : +0) never returns a NaN, so no
// published value can be mistaken for it.
constexpr uint32_t kSentinel = 0xFFFFFFFFu;

// Status words in device memory (one int[4] per handle).
//   [0] error code (0 = ok, kStatusTimeout), [1] step, [2] CTA, [3] spare.
constexpr int kStatusTimeout = 6;

// In the backward pass a P word with this bit pattern (a quiet NaN other
// than the sentinel) marks an output whose forward value was 0: its delta is
// 0 (the ReLU derivative) whatever the sum.  Folding the mask into P keeps
// the reverse kernel at one early load per output, like the forward.
constexpr uint32_t kMaskedMarker = 0x7fc0beefu;

__device__ __forceinline__ bool is_sentinel(float v) {
  return __float_as_uint(v) == kSentinel;
}
__device__ __forceinline__ bool ready4(const float4& v) {
  return !(is_sentinel(v.x) | is_sentinel(v.y) | is_sentinel(v.z) | is_sentinel(v.w));
}

// Relaxed, gpu-scope accesses: each 32-bit element is single-copy atomic and
// bypasses the non-coherent L1, so a consumer polling a word eventually sees
// the producer's store.  The data word itself is the flag.
__device__ __forceinline__ float4 ld_relaxed_f4(const float* p) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_relaxed_f(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_f(float* p, float v) {
  asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_i(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Read-only load that the compiler may not move: used to issue the next step's
// projection value early so its latency hides behind the step exchange.
__device__ __forceinline__ float ld_nc_pinned(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float relu(float s) { return s > 0.f ? s : 0.f; }

// Busy-wait n SM cycles without touching memory.  The persistent kernels
// wait this long after publishing a step before their first poll of the
// next one: a first poll that reaches the L2 before the producers' stores
// have landed turns into re-poll rounds that contend with those stores, and
// on some GB300 machines the exchange then settles into a state 3x slower.
__device__ __forceinline__ void spin_cycles(int n) {
  if (n <= 0) return;
  const long long t0 = clock64();
  while (clock64() - t0 < (long long)n) {
  }
}

// Record the first failure; later ones keep the first record.
__device__ __forceinline__ void report_timeout(int* status, int step, int cta) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) {
    status[1] = step;
    status[2] = cta;
  }
}

// Bounded wait state.  The deadline (globaltimer ns) is armed lazily, on the
// first stale poll of a step, so steps whose data is already there never
// read the timer.  Call new_step() at the start of every step.
struct Waiter {
  uint64_t deadline;
  long long timeout_ns;
  const int* status;
  int backoff;  // SM cycles before re-polling stale data (0: none); x2 per round up to x4
  __device__ __forceinline__ void new_step() { deadline = 0; }
  // Pause (a clock64 busy-wait, no memory traffic) before re-issuing stale
  // polls.  Without it, many CTAs re-polling the lines a producer is about to
  // write can delay that write at the L2 long enough to need more rounds,
  // and the exchange settles into a state several times slower.
  __device__ __forceinline__ void pause(uint32_t& round) {
    if (backoff > 0) spin_cycles(backoff << (round < 2u ? round : 2u));
    ++round;
  }
  // true = keep waiting; false = give up (deadline passed or another CTA failed)
  __device__ __forceinline__ bool still_ok(uint32_t& spins) {
    if ((++spins & 63u) != 1u) return true;
    if (deadline == 0) {
      deadline = global_ns() + (uint64_t)timeout_ns;
      return true;
    }
    if (ld_relaxed_i(status) != 0) return false;
    return global_ns() < deadline;
  }
};

// Poll one float4 of step data until none of its words is the sentinel.
// Returns false if the wait gave up.
__device__ __forceinline__ bool poll_f4(const float* p, float4& v, Waiter& w) {
  uint32_t spins = 0;
  while (!ready4(v)) {
    if (!w.still_ok(spins)) return false;
    v = ld_relaxed_f4(p);
  }
  return true;
}
__device__ __forceinline__ bool poll_f(const float* p, float& v, Waiter& w) {
  uint32_t spins = 0;
  while (is_sentinel(v)) {
    if (!w.still_ok(spins)) return false;
    v = ld_relaxed_f(p);
  }
  return true;
}

// Warp reduce-scatter of V partial sums (V a power of two).  On return lane L
// holds, in v[0 .. max(V/32,1)-1], the warp-wide sums of value indices
// L*V/32 + i (V >= 32), or of index L / (32/V) (V < 32; replicated across
// 32/V lanes).  Costs V-1 shuffles for V <= 32.
template <int V>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[V], int lane) {
  constexpr unsigned kFull = 0xffffffffu;
  int n = V;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
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

}  // namespace prnn
