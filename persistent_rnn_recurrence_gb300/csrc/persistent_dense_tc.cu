// persistent_dense_tc.cu -- the persistent dense recurrence on the tcgen05
// tensor cores, for batches wide enough that each step is a real (if small)
// matrix product: s = Wh h_{t-1} for Bl >= 8 batch columns per CTA group.
//
// Each CTA keeps its R rows of Wh (fp16, N = R rounded up to 16) on chip for
// the whole sequence as the B operand of tcgen05.mma (K-major, 128-byte
// swizzle, one 64-wide K slice after another).  Per step, eight filler warps
// poll h_{t-1} from L2 (flag in the data, as in the CUDA-core kernels; up to
// 16 float4 per thread in flight at once), round it to fp16 and write it, 64
// columns at a time, into a ring of 2-8 A tiles (M = 128 rows: the group's
// batch columns, zero beyond Bl); the
// control warp issues 4 MMAs (K = 16) per slice into a TMEM accumulator
// [128 lanes x N columns] and releases the slot with tcgen05.commit; after
// the last slice it reads its 32 lanes (batch rows) back, adds P_t, applies
// ReLU and publishes h_t into y.  The tensor cores make the per-step product
// cheap at B = 16-32 (a CUDA-core CTA would need R*H*Bl FMAs per step), and
// the exchange stays the same flag-in-data L2 broadcast.
//
// Measured on GB300 it is slower than the CUDA-core kernel at the batches
// this library serves (H=1152, B=16: 17-20 us/step against 3.8): every step
// is a chain of H/16 small MMAs (M=128, N<=32, K=16) into one accumulator,
// each waiting for the one before, plus a ring hand-off per 64 columns.  It
// is therefore opt-in (PRNN_OPT_RECURRENT_TC); splitting the chain over
// several TMEM accumulators is the next step for it.
//
// h is rounded to fp16 for the product (fp32 accumulation); the outputs
// stay fp32.  Every wait is bounded: on a timeout the CTA records the status,
// stops, waits (bounded) for its issued MMAs, frees its TMEM and returns.
#include "persistent_common.cuh"
#include "tc_common.cuh"

namespace prnn {

using namespace pk;
using namespace tc;

namespace {

constexpr int kRingMax = 8;                 // A slots (a.nring <= kRingMax)
constexpr int kSlotBytes = 128 * 128;       // 128 rows x 64 fp16
constexpr int kMaxV = 16;                   // float4 polls a filler keeps in flight
constexpr int kFillers = 256;               // threads of warps 1..8
constexpr int kTcThreads = 32 + kFillers;

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kTcThreads, 1) recur_dense_tc_kernel(const DenseTcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kRingMax];
  __shared__ __align__(8) uint64_t empty_bar[kRingMax];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ __align__(8) uint64_t fin_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = c.H, B = c.B, N = a.N, nsl = a.nslices, nring = a.nring;
  const Place pl = place_of(c);
  const int bl = pl.b_hi - pl.b_lo;  // <= 32
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t ring = base;
  const uint32_t wts = base + nring * kSlotBytes;
  const uint32_t tmem_cols = N <= 32 ? 32u : 64u;

  // weights image -> smem, ring -> zeros (rows >= bl of every A tile stay 0)
  {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.Wimg) +
                                                      (size_t)pl.lc * nsl * N * 128);
    uint4* wdst = reinterpret_cast<uint4*>(gbase + nring * kSlotBytes);
    const int nw = nsl * N * 128 / 16;
    for (int i = tid; i < nw; i += kTcThreads) wdst[i] = __ldg(src + i);
    uint4* rdst = reinterpret_cast<uint4*>(gbase);
    for (int i = tid; i < nring * kSlotBytes / 16; i += kTcThreads) rdst[i] = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  if (tid == 0) {
    for (int q = 0; q < nring; ++q) {
      mbar_init(&full_bar[q], kFillers / 32);  // one arrival per filler warp
      mbar_init(&empty_bar[q], 1);
    }
    mbar_init(&done_bar, 1);
    mbar_init(&fin_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = f16_idesc(128, N);
  volatile int* abort_flag = &s_abort;

  if (warp > 0) {
    // ---------------- fillers ----------------
    // Per step the h_{t-1} values of up to kMaxV float4 per thread are in
    // flight at once (a chunk of slices), then written slice by slice into
    // the ring as slots free up.  Item i of slice s: batch row i / 16, float4
    // i % 16 of the slice's 64 columns; thread ft takes i = ft, ft + 256, ...
    const int ft = tid - 32;
    // items per slice per thread (>= 1 even for a group with no batch
    // columns, so every index below stays defined)
    const int per_s = max(1, (bl * 16 + kFillers - 1) / kFillers);
    const int chunk = min(kMaxV / per_s, nring);  // slices per chunk (all in the ring at once)
    Waiter w;
    w.status = c.status;
    w.timeout_ns = c.timeout_ns;
    w.backoff = c.poll_backoff;
    // every decision below is warp-uniform (the filler warps use warp
    // collectives): the abort flag is read by lane 0 and broadcast
    auto aborted = [&]() { return __shfl_sync(0xffffffffu, *abort_flag, 0) != 0; };
    for (int t = 0; t < c.T && !aborted(); ++t) {
      const float* hprev = (t == 0) ? c.h0 : c.y + (size_t)(t - 1) * B * H;
      w.new_step();
      if (t > 0) spin_cycles(c.poll_delay);
      for (int s0 = 0; s0 < nsl && !aborted(); s0 += chunk) {
        const int ns = min(chunk, nsl - s0);
        float4 v[kMaxV];
        bool ok = true;
#pragma unroll
        for (int m = 0; m < kMaxV; ++m) {
          v[m] = make_float4(0.f, 0.f, 0.f, 0.f);
          const int sl = m / per_s, it = ft + (m % per_s) * kFillers;
          if (sl < ns && it < bl * 16 && hprev != nullptr) {
            const float* p = hprev + (size_t)(pl.b_lo + (it >> 4)) * H + (s0 + sl) * 64 + (it & 15) * 4;
            v[m] = (t == 0) ? __ldg(reinterpret_cast<const float4*>(p)) : ld_relaxed_f4(p);
          }
        }
        if (t > 0 && hprev != nullptr) {
          uint32_t spins = 0, round = 0;
          for (;;) {
            unsigned stale = 0;
#pragma unroll
            for (int m = 0; m < kMaxV; ++m) {
              const int sl = m / per_s, it = ft + (m % per_s) * kFillers;
              if (sl < ns && it < bl * 16 && !ready4(v[m])) stale |= 1u << m;
            }
            if (stale == 0u) break;
            if (!w.still_ok(spins)) {
              ok = false;
              break;
            }
            w.pause(round);
#pragma unroll
            for (int m = 0; m < kMaxV; ++m)
              if ((stale >> m) & 1u) {
                const int sl = m / per_s, it = ft + (m % per_s) * kFillers;
                v[m] = ld_relaxed_f4(hprev + (size_t)(pl.b_lo + (it >> 4)) * H + (s0 + sl) * 64 +
                                     (it & 15) * 4);
              }
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) report_timeout(c.status, t, blockIdx.x);
          *abort_flag = 1;
          break;
        }
        for (int sl = 0; sl < ns; ++sl) {
          const long g = (long)t * nsl + s0 + sl;
          const int q = (int)(g % nring);
          const long use = g / nring;
          bool free_ok = true;
          if (use > 0 && lane == 0)
            free_ok = mbar_wait(&empty_bar[q], (uint32_t)((use - 1) & 1), global_ns() + c.timeout_ns);
          free_ok = __shfl_sync(0xffffffffu, free_ok ? 1 : 0, 0) != 0;
          if (!free_ok) {
            if (lane == 0) report_timeout(c.status, t, blockIdx.x);
            *abort_flag = 1;
            ok = false;
            break;
          }
          unsigned char* slot = gbase + q * kSlotBytes;
#pragma unroll
          for (int m = 0; m < kMaxV; ++m) {
            const int it = ft + (m % per_s) * kFillers;
            if (m / per_s == sl && it < bl * 16) {
              const int rr = it >> 4, j = it & 15;
              // 128-byte-swizzled K-major row rr: 16-byte chunk j/2 at (j/2) ^ (rr & 7)
              const uint32_t off = rr * 128 + (((j >> 1) ^ (rr & 7)) << 4) + ((j & 1) << 3);
              *reinterpret_cast<uint2*>(slot + off) =
                  make_uint2(pack_half2(v[m].x, v[m].y), pack_half2(v[m].z, v[m].w));
            }
          }
        }
        if (!ok) break;
        // one proxy fence for the chunk's writes, then the chunk's slices are released
        fence_async_smem();
        __syncwarp();
        if (lane == 0)
          for (int sl = 0; sl < ns; ++sl) mbar_arrive(&full_bar[((long)t * nsl + s0 + sl) % nring]);
      }
    }
  } else {
    // ---------------- control warp: MMAs and the epilogue ----------------
    const uint32_t rows = (uint32_t)pl.rows;
    for (int t = 0; t < c.T && !*abort_flag; ++t) {
      const float* Pt = c.P + (size_t)t * B * H;
      float* yt = c.y + (size_t)t * B * H;
      // P for this lane's batch row, fetched before the step's wait
      float pv[32];
#pragma unroll
      for (int n = 0; n < 32; ++n)
        pv[n] = (lane < bl && n < (int)rows) ? __ldg(Pt + (size_t)(pl.b_lo + lane) * H + pl.row0 + n)
                                             : 0.f;
      bool ok = true;
      if (lane == 0) {
        for (int s = 0; s < nsl; ++s) {
          const long g = (long)t * nsl + s;
          const int q = (int)(g % nring);
          if (!mbar_wait(&full_bar[q], (uint32_t)((g / nring) & 1), global_ns() + c.timeout_ns) ||
              *abort_flag) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = sw128_kmajor_desc(ring + q * kSlotBytes + k * 32);
            const uint64_t bdesc = sw128_kmajor_desc(wts + (uint32_t)s * N * 128 + k * 32);
            umma_f16(tmem, adesc, bdesc, idesc, (s > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[q]);
        }
        if (ok) umma_commit(&done_bar);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (ok) ok = mbar_wait(&done_bar, (uint32_t)(t & 1), global_ns() + c.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          report_timeout(c.status, t, blockIdx.x);
          *abort_flag = 1;
        }
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      uint32_t r[32];
      tmem_load_32cols(tmem, r);  // lanes 0..31 = batch rows, columns 0..31 = rows
      if (lane < bl && !((int)blockIdx.x == c.drop_cta && t == c.drop_step)) {
        float* yrow = yt + (size_t)(pl.b_lo + lane) * H + pl.row0;
#pragma unroll
        for (int n = 0; n < 32; ++n)
          if (n < (int)rows) st_relaxed_f(yrow + n, relu(__uint_as_float(r[n]) + pv[n]));
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
    }
    // every issued MMA completes before the TMEM is freed
    if (lane == 0) {
      umma_commit(&fin_bar);
      mbar_wait(&fin_bar, 0, global_ns() + c.timeout_ns);
    }
    __syncwarp();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

}  // namespace

size_t recur_dense_tc_smem(int H, int N, int nring) {
  return 1024 + (size_t)nring * kSlotBytes + (size_t)(H / 64) * N * 128;
}

int recur_dense_tc_ring(int H, int N, size_t smem_optin) {
  const size_t fixed = 1024 + (size_t)(H / 64) * N * 128;
  if (fixed + 2 * (size_t)kSlotBytes > smem_optin) return 0;
  const int fit = (int)((smem_optin - fixed) / kSlotBytes);
  return fit < kRingMax ? fit : kRingMax;
}

int recur_dense_tc_threads() { return kTcThreads; }

cudaError_t launch_recur_dense_tc(const DenseTcArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<DenseTcArgs*>(&a)};
  return coop_launch(recur_dense_tc_kernel, a.c.n_cta, kTcThreads, a.c.smem, s, args);
}

}  // namespace prnn
