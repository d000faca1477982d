// cluster_probe.cu -- a diagnostic: the step exchange of h inside
// thread-block clusters, through distributed shared memory.
//
// The persistent kernels exchange h_{t-1} through L2 (flag in the data).  A
// cluster of up to 16 CTAs could exchange it through its members' shared
// memory instead.  This probe runs that exchange with no arithmetic, so the
// cost of the alternative can be measured on the device: each cluster
// exchanges a vector of `hidden` floats per step; CTA r owns rows
// [r * R, (r + 1) * R), R = hidden / cluster_size, and pushes them into every
// CTA of its cluster (its own included) with st.async, 16 bytes at a time,
// each completing transaction bytes on the receiver's mbarrier; a CTA waits
// until its whole vector of the step has arrived before it sends its rows of
// the next step.  Every received word is checked, one step late, while the
// next step's pushes are in flight, so the check stays off the exchange's
// critical path.  Three buffers (and mbarriers) rotate by step: a CTA can be
// at most one step ahead of a peer (its next step needs that peer's rows of
// this one), so a push of step t+2 never lands in the buffer of step t-1
// while it is being checked.
#include <vector>

#include "prnn.h"
#include "prnn_internal.h"
#include "device_common.cuh"
#include "tc_common.cuh"

namespace prnn {

namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeBufs = 3;
constexpr int kProbeMaxHidden = 16384;                    // three buffers of 64 KiB
constexpr uint64_t kProbeWaitNs = 1000ull * 1000 * 1000;  // 1 s per wait

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void push4(uint32_t dst, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(dst),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool probe_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(tc::smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// the value of row r at step t (exact in fp32)
__device__ __forceinline__ float probe_value(int t, int r) {
  return (float)((t * 131 + r) & 0xffff);
}

// ns[c]: globaltimer ns of cluster c's exchange (its rank 0); bad: wrong words
// received (all CTAs); status[0] = kStatusTimeout when a wait ran out.
__global__ void __launch_bounds__(kProbeThreads) cluster_exchange_kernel(int H, int T,
                                                                         unsigned long long* ns,
                                                                         unsigned int* bad,
                                                                         int* status) {
  extern __shared__ __align__(16) float hs[];  // [kProbeBufs][H]
  __shared__ __align__(8) uint64_t full[kProbeBufs];
  __shared__ int s_stop;
  const int tid = threadIdx.x, NT = blockDim.x;
  const uint32_t rank = cluster_rank(), ncl = cluster_ctas();
  const int R = H / (int)ncl, row0 = (int)rank * R, q4 = R / 4;
  if (tid == 0) {
    for (int i = 0; i < kProbeBufs; ++i) tc::mbar_init(&full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_stop = 0;
  }
  __syncthreads();
  cluster_barrier();  // every peer's mbarriers exist before the first push
  const uint64_t t0 = global_ns();
  uint64_t t_end = t0;
  unsigned int wrong = 0;
  for (int t = 0; t <= T; ++t) {
    const int b = t % kProbeBufs;
    if (t < T) {
      if (tid == 0) tc::mbar_arrive_expect_tx(&full[b], (uint32_t)H * 4u);
      // my rows of step t into every CTA of the cluster
      const uint32_t dst0 = tc::smem_u32(hs + (size_t)b * H + row0);
      const uint32_t bar0 = tc::smem_u32(&full[b]);
      for (int i = tid; i < (int)ncl * q4; i += NT) {
        const uint32_t peer = (uint32_t)(i / q4);
        const int q = i - (int)peer * q4, r = row0 + 4 * q;
        const float4 v = make_float4(probe_value(t, r), probe_value(t, r + 1),
                                     probe_value(t, r + 2), probe_value(t, r + 3));
        push4(peer_addr(dst0 + 16u * (uint32_t)q, peer), v, peer_addr(bar0, peer));
      }
    }
    if (t > 0) {  // the words of step t-1, while step t's pushes are in flight
      const float* prev = hs + (size_t)((t - 1) % kProbeBufs) * H;
      for (int i = tid; i < H; i += NT) wrong += prev[i] != probe_value(t - 1, i);
    }
    if (t == T) break;
    // the whole vector of step t
    const uint32_t parity = (uint32_t)(t / kProbeBufs) & 1u;
    if (!probe_try_wait(&full[b], parity)) {
      const uint64_t deadline = global_ns() + kProbeWaitNs;
      uint32_t n = 0;
      while (!probe_try_wait(&full[b], parity)) {
        if ((++n & 255u) == 0u && global_ns() > deadline) {
          if (atomicCAS(status, 0, kStatusTimeout) == 0) {
            status[1] = t;
            status[2] = blockIdx.x;
          }
          s_stop = 1;
          break;
        }
      }
    }
    if (t == T - 1) t_end = global_ns();
    __syncthreads();
    if (s_stop) break;
  }
  if (wrong) atomicAdd(bad, wrong);
  if (tid == 0 && rank == 0) ns[blockIdx.x / ncl] = t_end - t0;
  cluster_barrier();  // no CTA leaves while a peer may still push into it
}

}  // namespace

}  // namespace prnn

extern "C" prnn_status_t prnn_probe_cluster_exchange(int hidden, int cluster_size, int clusters,
                                                     int steps, double* ns_per_step,
                                                     long long* mismatches) {
  using namespace prnn;
  if (cluster_size != 2 && cluster_size != 4 && cluster_size != 8 && cluster_size != 16)
    return PRNN_ERR_INVALID_ARG;
  if (hidden < 4 * cluster_size || hidden > kProbeMaxHidden || hidden % (4 * cluster_size) != 0)
    return PRNN_ERR_INVALID_ARG;
  if (clusters < 1 || steps < 2 || !ns_per_step || !mismatches) return PRNN_ERR_INVALID_ARG;
  int dev = 0, cc = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&cc, cudaDevAttrClusterLaunch, dev) != cudaSuccess)
    return PRNN_ERR_CUDA;
  if (!cc) return PRNN_ERR_UNSUPPORTED;
  const size_t smem = (size_t)kProbeBufs * hidden * sizeof(float);
  if (cudaFuncSetAttribute(cluster_exchange_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) != cudaSuccess ||
      cudaFuncSetAttribute(cluster_exchange_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return PRNN_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cluster_size * clusters));
  cfg.blockDim = dim3(kProbeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = nullptr;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cluster_size;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // every cluster must be resident at once for a per-step time to mean anything
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, cluster_exchange_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return PRNN_ERR_UNSUPPORTED;
  }
  if (clusters > max_clusters) return PRNN_ERR_UNSUPPORTED;
  // device scratch: ns per cluster, the wrong-word count, a status block
  unsigned char* d = nullptr;
  const size_t bytes = (size_t)clusters * 8 + 8 + 16;
  if (cudaMalloc(&d, bytes) != cudaSuccess) {
    cudaGetLastError();
    return PRNN_ERR_OOM;
  }
  unsigned long long* d_ns = reinterpret_cast<unsigned long long*>(d);
  unsigned int* d_bad = reinterpret_cast<unsigned int*>(d + (size_t)clusters * 8);
  int* d_status = reinterpret_cast<int*>(d + (size_t)clusters * 8 + 8);
  prnn_status_t st = PRNN_OK;
  std::vector<unsigned long long> ns((size_t)clusters);
  unsigned int bad = 0;
  int status[4] = {0, 0, 0, 0};
  if (cudaMemset(d, 0, bytes) != cudaSuccess ||
      cudaLaunchKernelEx(&cfg, cluster_exchange_kernel, hidden, steps, d_ns, d_bad, d_status) !=
          cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(ns.data(), d_ns, ns.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&bad, d_bad, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(status, d_status, 16, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    st = PRNN_ERR_CUDA;
  }
  cudaFree(d);
  if (st != PRNN_OK) return st;
  if (status[0] != 0) return PRNN_ERR_TIMEOUT;
  double sum = 0.0;
  for (unsigned long long v : ns) sum += (double)v;
  *ns_per_step = sum / clusters / steps;
  *mismatches = (long long)bad;
  return PRNN_OK;
}
