// persistent_dense_tc.cu -- the persistent dense recurrence on the tcgen05
// tensor cores, for batches wide enough that each step is a real (if small)
// matrix product: s = Wh h_{t-1} for Bl >= 8 batch columns per CTA group.
//
// Each CTA keeps its R rows of Wh (fp16, N = R rounded up to 16) on chip for
// the whole sequence as the B operand of tcgen05.mma (K-major, 128-byte
// swizzle, one 64-wide K slice after another).  Per step, eight filler warps
// poll h_{t-1} from L2 (flag in the data, as in the CUDA-core kernels),
// round it to fp16 and write it, 64 columns at a time, into a 4-slot ring of
// A tiles (M = 128 rows: the group's batch columns, zero beyond Bl); the
// control warp issues 4 MMAs (K = 16) per slice into a TMEM accumulator
// [128 lanes x N columns] and releases the slot with tcgen05.commit; after
// the last slice it reads its 32 lanes (batch rows) back, adds P_t, applies
// ReLU and publishes h_t into y.  The tensor cores make the per-step product
// cheap at B = 16-32 (a CUDA-core CTA would need R*H*Bl FMAs per step), and
// the exchange stays the same flag-in-data L2 broadcast.
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

constexpr int kRing = 4;                    // A slots
constexpr int kSlotBytes = 128 * 128;       // 128 rows x 64 fp16
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
  __shared__ __align__(8) uint64_t full_bar[kRing];
  __shared__ __align__(8) uint64_t empty_bar[kRing];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ __align__(8) uint64_t fin_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = c.H, B = c.B, N = a.N, nsl = a.nslices;
  const Place pl = place_of(c);
  const int bl = pl.b_hi - pl.b_lo;  // <= 32
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t ring = base;
  const uint32_t wts = base + kRing * kSlotBytes;
  const uint32_t tmem_cols = N <= 32 ? 32u : 64u;

  // weights image -> smem, ring -> zeros (rows >= bl of every A tile stay 0)
  {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.Wimg) +
                                                      (size_t)pl.lc * nsl * N * 128);
    uint4* wdst = reinterpret_cast<uint4*>(gbase + kRing * kSlotBytes);
    const int nw = nsl * N * 128 / 16;
    for (int i = tid; i < nw; i += kTcThreads) wdst[i] = __ldg(src + i);
    uint4* rdst = reinterpret_cast<uint4*>(gbase);
    for (int i = tid; i < kRing * kSlotBytes / 16; i += kTcThreads) rdst[i] = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  if (tid == 0) {
    for (int q = 0; q < kRing; ++q) {
      mbar_init(&full_bar[q], kFillers);
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
    const int ft = tid - 32;
    Waiter w;
    w.status = c.status;
    w.timeout_ns = c.timeout_ns;
    w.backoff = c.poll_backoff;
    for (int t = 0; t < c.T && !*abort_flag; ++t) {
      const float* hprev = (t == 0) ? c.h0 : c.y + (size_t)(t - 1) * B * H;
      w.new_step();
      if (t > 0) spin_cycles(c.poll_delay);
      for (int s = 0; s < nsl && !*abort_flag; ++s) {
        const long g = (long)t * nsl + s;
        const int q = (int)(g % kRing);
        const long use = g / kRing;
        if (use > 0 &&
            !mbar_wait(&empty_bar[q], (uint32_t)((use - 1) & 1), global_ns() + c.timeout_ns)) {
          report_timeout(c.status, t, blockIdx.x);
          *abort_flag = 1;
          break;
        }
        unsigned char* slot = gbase + q * kSlotBytes;
        bool ok = true;
        for (int i = ft; i < bl * 16; i += kFillers) {
          const int rr = i >> 4, j = i & 15;  // batch row, float4 within the 64-wide slice
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (hprev != nullptr) {
            const float* p = hprev + (size_t)(pl.b_lo + rr) * H + s * 64 + j * 4;
            if (t == 0) {
              v = __ldg(reinterpret_cast<const float4*>(p));
            } else {
              v = ld_relaxed_f4(p);
              uint32_t spins = 0, round = 0;
              while (!ready4(v)) {
                if (!w.still_ok(spins)) {
                  ok = false;
                  break;
                }
                w.pause(round);
                v = ld_relaxed_f4(p);
              }
            }
          }
          // 128-byte-swizzled K-major row rr: 16-byte chunk j/2 at (j/2) ^ (rr & 7)
          const uint32_t off = rr * 128 + (((j >> 1) ^ (rr & 7)) << 4) + ((j & 1) << 3);
          *reinterpret_cast<uint2*>(slot + off) = make_uint2(pack_half2(v.x, v.y), pack_half2(v.z, v.w));
          if (!ok) break;
        }
        if (!ok) {
          report_timeout(c.status, t, blockIdx.x);
          *abort_flag = 1;
        }
        fence_async_smem();
        mbar_arrive(&full_bar[q]);
        if (!ok) break;
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
          const int q = (int)(g % kRing);
          if (!mbar_wait(&full_bar[q], (uint32_t)((g / kRing) & 1), global_ns() + c.timeout_ns) ||
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

size_t recur_dense_tc_smem(int H, int N) {
  return 1024 + (size_t)kRing * kSlotBytes + (size_t)(H / 64) * N * 128;
}

int recur_dense_tc_threads() { return kTcThreads; }

cudaError_t launch_recur_dense_tc(const DenseTcArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<DenseTcArgs*>(&a)};
  return coop_launch(recur_dense_tc_kernel, a.c.n_cta, kTcThreads, a.c.smem, s, args);
}

}  // namespace prnn
