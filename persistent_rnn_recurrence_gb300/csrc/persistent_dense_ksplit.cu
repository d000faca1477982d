// persistent_dense_ksplit.cu -- the persistent dense recurrence for wide
// batches (fp16 weights, up to 32 batch columns) on the tcgen05 tensor cores,
// with each step's product split over K inside thread-block clusters.
//
// At B = 16-32 a step is a small matrix product s = Wh h_{t-1} (H x H by
// H x B).  On CUDA cores it is bound by instruction issue (the FMAs plus the
// fp16 conversions and shared loads that feed them).  On the tensor cores a
// tcgen05.mma with M = 128 and N <= 128 costs about the same whatever N is,
// so the count of MMAs per SM sets the time: a CTA that owned 128 rows for all
// of K would issue H / 16 of them in a chain.  Here each of the H / 128 row
// blocks gets a cluster of CS CTAs (CS <= 8, the largest for which all the
// clusters are resident at once), and CTA j of a cluster multiplies the
// block's rows by K slice j only: about H / (16 CS) MMAs of K = 16.
//
// Per step, in CTA j of a cluster:
//  1. all threads poll h_{t-1}[b][K slice j] for the batch columns (flag in
//     the data, relaxed loads, bounded) and split each fp32 value into
//     hi = fp16(h) and lo = fp16(h - hi), so hi + lo carries about 22 bits of
//     h; the two go side by side into the B operand: rows 0 .. BP-1 hold hi,
//     rows BP .. 2BP-1 lo (BP = the batch padded to 8, 16 or 32; N = 2 BP),
//     so one MMA per K step multiplies both;
//  2. two threads in different warps issue the slice's MMAs, half of the K
//     steps each (M = 128 rows of Wh, kept in shared memory for the whole
//     sequence as the A operand), into two TMEM accumulators [128 lanes x N
//     columns];
//  3. four warps read the accumulators back (lane = row), add the hi and lo
//     columns of both and stage the partial sums column by column; CTA o of
//     the cluster owns batch columns [o B / CS, (o + 1) B / CS), and lane
//     o / 4 of warp 4 + o % 4 sends owner o its columns with a bulk copy
//     into the owner's shared memory (cp.async.bulk shared::cta ->
//     shared::cluster, completing on the owner's mbarrier);
//  4. the owner waits for the CS - 1 blocks, sums the CS partials (slice
//     order) and P_t, applies ReLU and publishes its columns of the block's
//     128 rows of h_t into y, as the other persistent kernels do.
// Where a slice of Wh does not fit in shared memory beside the operand tiles
// (H above 2304), the A operand is not resident: each MMA issuer streams its
// atoms of the slice from the image in global memory, every step, through a
// ring of four 16 KB stages (bulk copies, full / empty mbarriers), for
// batches of up to 16 columns; the step is then bound by that stream.
// In reverse mode (the backward pass) the steps run T-1 .. 0 over Wh^T's
// image, h_prev is the next step's delta, and the output is P + sum, or 0
// where P holds the mask marker.
// The exchange of h between clusters stays the flag-in-data L2 broadcast;
// only the K reduction runs through distributed shared memory.
//
// h is fp32 in y.  A value of 2^15 or more would overflow the fp16 split: a
// step whose slice holds one is scaled by a power of two first (exact), and
// the partial sums are scaled back.  Every wait is bounded: on a timeout the
// CTA records the status; all CTAs leave the step loop together (the
// decisions are taken at CTA barriers), wait for their MMAs, free TMEM and
// meet their cluster peers once more before leaving, so no bulk copy targets
// the shared memory of a CTA that has left.
#include "persistent_common.cuh"
#include "tc_common.cuh"

namespace prnn {

using namespace pk;
using namespace tc;

namespace {

// 16 warps; warps 4..7 read TMEM lanes 0..127.  512 threads (6 polls each)
// measured 3-7 % faster than 256 (12 each): more warps hide the fill's latency
constexpr int kSplitThreads = 512;
constexpr int kSplitPollMax = 6;       // float4 polls a thread keeps in flight
static_assert(kSplitPollMax * kSplitThreads * 4 >= kKsplitMaxB * kKsplitMaxSlice,
              "one poll round covers the widest slice of the widest batch");
constexpr uint32_t kAtomA = 128 * 128;  // bytes of one A atom: 128 rows x 64 fp16
// Streamed A (layers whose weights do not fit beside the operand tiles): each
// MMA issuer has a ring of kNsq A stages refilled by bulk copies from the
// weight image in device memory, kNsq - 1 atoms ahead of its MMAs, across
// steps; 8 polls per thread cover a slice of up to kKsplitMaxSliceStream
// columns at B <= 16
constexpr int kNsq = 4;
constexpr int kStreamPollMax = 8;
static_assert(kStreamPollMax * kSplitThreads * 4 >= 16 * kKsplitMaxSliceStream,
              "one poll round covers the widest streamed slice at B <= 16");
constexpr int kSplitTmemCols = 128;    // two accumulators of N <= 64 columns
constexpr float kSplitLarge = 32768.f; // |h| from here on would overflow the fp16 split

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// bulk copy of `bytes` from this CTA's shared memory into a peer's, completing
// transaction bytes on the peer's mbarrier (both given as shared::cluster
// addresses)
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// bulk copy global -> this CTA's shared memory, completing on its mbarrier
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for an mbarrier phase.  The timer is read only once the phase
// is not complete at the first test; the wait also ends when another CTA has
// recorded a failure.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, long long limit_ns,
                                           const int* status) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t deadline = global_ns() + (uint64_t)limit_ns;
  uint32_t n = 0;
  while (!try_wait_cluster(bar, parity)) {
    if ((++n & 255u) == 0u && (global_ns() > deadline || ld_relaxed_i(status) != 0)) return false;
  }
  return true;
}
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Bounded wait for the MMAs this CTA issued, before TMEM is freed: by time
// only (another CTA's failure does not end it; the MMAs always complete).
__device__ __forceinline__ void wait_own_mmas(uint64_t* bar, uint32_t parity) {
  if (try_wait_cluster(bar, parity)) return;
  const uint64_t deadline = global_ns() + 100ull * 1000 * 1000;  // 100 ms
  uint32_t n = 0;
  while (!try_wait_cluster(bar, parity))
    if ((++n & 255u) == 0u && global_ns() > deadline) return;
}
// 2^e for |e| < 127, exactly
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// 16 consecutive 32-bit TMEM columns of the warp's 32 lanes (one per thread)
__device__ __forceinline__ void tmem_load_16cols(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Split four values (scaled by `scale`, a power of two) into their fp16 hi
// and lo parts and store them into the B operand at `hi` (4 consecutive K
// indices of one batch row n; lo goes to row BP + n, BP * 128 bytes on).
// Row n of an atom holds 128 bytes, its 16-byte chunk q at q ^ (n & 7).
template <int BP>
__device__ __forceinline__ void store_split(unsigned char* hi_dst, float4 v, float scale) {
  const float x[4] = {v.x * scale, v.y * scale, v.z * scale, v.w * scale};
  float hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half h = __float2half_rn(x[i]);
    hi[i] = __half2float(h);
    lo[i] = x[i] - hi[i];
  }
  *reinterpret_cast<uint2*>(hi_dst) = make_uint2(pack_half2(hi[0], hi[1]), pack_half2(hi[2], hi[3]));
  *reinterpret_cast<uint2*>(hi_dst + BP * 128) =
      make_uint2(pack_half2(lo[0], lo[1]), pack_half2(lo[2], lo[3]));
}

// TR: the phase-trace build (records per step and CTA in a.trace); STR: A
// streamed through per-issuer rings instead of resident
template <int BP, bool TR, bool STR>
__global__ void __launch_bounds__(kSplitThreads, 1) recur_dense_ksplit_kernel(const DenseSplitArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ __align__(8) uint64_t recv_bar[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_large[2];
  __shared__ float s_red[kSplitThreads / 32];
  __shared__ __align__(8) uint64_t a_full[2][kNsq];   // streamed A: stage loaded
  __shared__ __align__(8) uint64_t a_empty[2][kNsq];  // streamed A: its MMAs done
  constexpr int PM = STR ? kStreamPollMax : kSplitPollMax;  // polls per thread

  constexpr int N = 2 * BP;
  constexpr uint32_t kAtomB = (uint32_t)N * 128;  // bytes of one B atom: N rows x 64 fp16
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = c.H, B = c.B, T = c.T, cs = a.cs, nat = a.nat;
  {
    // launched in clusters of any other size (a launch that lost its cluster
    // shape), every peer address below would be wrong: record the failure
    // (step -1) and leave before touching TMEM or a peer
    uint32_t ncl;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncl));
    if ((int)ncl != cs || (int)gridDim.x != c.n_cta) {
      if (tid == 0) report_timeout(c.status, -1, blockIdx.x);
      return;
    }
  }
  const int j = (int)cluster_rank();                  // K slice of this CTA
  const int row0 = blockIdx.x / cs * 128;            // the cluster's row block
  const int k0 = ksplit_k0(H, cs, j), kl = ksplit_kl(H, cs, j);
  const int cb0 = j * B / cs, ncol = (j + 1) * B / cs - cb0;  // the batch columns it finalizes
  const int maxcol = (B + cs - 1) / cs;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - smem_u32(smem_raw));
  const int a_atoms = STR ? 2 * kNsq : nat;  // A in shared memory: all atoms, or the rings
  const uint32_t sA = base;
  const uint32_t sB = sA + (uint32_t)a_atoms * kAtomA;
  unsigned char* gB = gbase + (size_t)a_atoms * kAtomA;
  // partial sums out, [2][B][128] (column b of the block: 128 rows), and in,
  // [2][cs][maxcol][128] (slot i: CTA i's partials of this CTA's columns)
  float* stage = reinterpret_cast<float*>(gB + (size_t)nat * kAtomB);
  float* recv = stage + 2 * B * 128;
  const uint32_t in_bytes = (uint32_t)(cs - 1) * (uint32_t)ncol * 512u;

  // Wh rows of the block x K slice (the A operand, for the whole sequence);
  // the B operand zeroed: its rows past the batch stay zero
  {
    const uint4* src =
        reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.Wimg) +
                                       (size_t)blockIdx.x * nat * kAtomA);
    uint4* dst = reinterpret_cast<uint4*>(gbase);
    const int na = STR ? 0 : nat * (int)kAtomA / 16;
    for (int i = tid; i < na; i += kSplitThreads) dst[i] = __ldg(src + i);
    uint4* bz = reinterpret_cast<uint4*>(gB);
    for (int i = tid; i < nat * (int)kAtomB / 16; i += kSplitThreads) bz[i] = make_uint4(0, 0, 0, 0);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (tid == 0) {
    mbar_init(&mma_bar, 2);  // both MMA issuers commit
    mbar_init(&recv_bar[0], 1);
    mbar_init(&recv_bar[1], 1);
    s_large[0] = s_large[1] = 0;
    if constexpr (STR)
      for (int q = 0; q < 2; ++q)
        for (int st = 0; st < kNsq; ++st) {
          mbar_init(&a_full[q][st], 1);
          mbar_init(&a_empty[q][st], 1);
        }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the partial blocks of steps 0 and 1 (cs - 1 peers x ncol columns)
    if (T > 0) mbar_arrive_expect_tx(&recv_bar[0], in_bytes);
    if (T > 1) mbar_arrive_expect_tx(&recv_bar[1], in_bytes);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(kSplitTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  cluster_sync_all();  // every peer's mbarriers exist before the first copy

  // Streamed A: issuer q (threads 0 and 32) takes atoms [a_lo, a_lo + naq) of
  // the slice; its n-th atom overall (step n / naq) sits in ring stage
  // n % kNsq, loaded kNsq - 1 atoms ahead of the MMAs that read it
  const int qi = tid == 0 ? 0 : 1;
  const int na0 = (nat + 1) / 2;
  const int a_lo = qi == 0 ? 0 : na0, naq = qi == 0 ? na0 : nat - na0;
  const int n_total = STR && (tid == 0 || tid == 32) ? T * naq : 0;
  int n_issued = 0, n_cons = 0;
  const unsigned char* wimg =
      static_cast<const unsigned char*>(a.Wimg) + (size_t)blockIdx.x * nat * kAtomA;
  auto a_copy = [&](int n) {  // atom n of this issuer into its stage n % kNsq
    const int st = n % kNsq;
    mbar_arrive_expect_tx(&a_full[qi][st], kAtomA);
    bulk_g2s(sA + (uint32_t)(qi * kNsq + st) * kAtomA, wimg + (size_t)(a_lo + n % naq) * kAtomA,
             kAtomA, &a_full[qi][st]);
  };
  if constexpr (STR)
    for (; n_issued < kNsq - 1 && n_issued < n_total; ++n_issued) a_copy(n_issued);

  const uint32_t idesc = f16_idesc(128, N);
  const int nks = kl >> 4, nks_half = (nks + 1) >> 1;  // K steps: issuer 0 takes the first half
  const int q4 = kl >> 2;  // float4 per batch column of the slice
  const int nf4 = B * q4;
  const int nout = ncol * 128;  // outputs this CTA finalizes: column cb0 + o / 128, row o % 128
  // The thread's float4 items of the slice (at most PM: the plan keeps kl <=
  // kKsplitMaxSlice, or kKsplitMaxSliceStream at B <= 16, so B * kl / 4 <= PM *
  // kSplitThreads), with
  // their offsets in a step's h (floats) and in the B operand (bytes, hi),
  // computed once: dividing by the launch-time slice width in every step
  // measured slower than the step's whole arithmetic (dependent integer
  // chains with 8 warps per SM to hide them)
  int goff[PM];
  uint32_t soff[PM];
  unsigned items = 0;
#pragma unroll
  for (int u = 0; u < PM; ++u) {
    const int i = tid + u * kSplitThreads;
    goff[u] = 0;
    soff[u] = 0;
    if (i < nf4) {
      const int b = i / q4, k = 4 * (i % q4);
      goff[u] = b * H + k;
      soff[u] = (uint32_t)((k >> 6) * (int)kAtomB + b * 128 +
                           ((((k & 63) >> 3) ^ (b & 7)) << 4) + ((k & 7) << 1));
      items |= 1u << u;
    }
  }
  Waiter w;
  w.status = c.status;
  w.timeout_ns = c.timeout_ns;
  w.backoff = c.poll_backoff;
  constexpr int kOutMax = (kKsplitMaxB + 1) / 2 * 128 / kSplitThreads;  // cs >= 2
  // output o = tid + u * kSplitThreads (o < nout) sits at ooff[u] in a step of P and y
  int ooff[kOutMax];
#pragma unroll
  for (int u = 0; u < kOutMax; ++u) {
    const int o = tid + u * kSplitThreads;
    ooff[u] = (cb0 + (o >> 7)) * H + row0 + (o & 127);
  }
  const size_t step_floats = (size_t)B * H;
  float pn[kOutMax];  // projection values of the next step's outputs
  auto load_p = [&](int t) {
    const float* pt = c.P + (size_t)t * step_floats;
#pragma unroll
    for (int u = 0; u < kOutMax; ++u)
      pn[u] = tid + u * kSplitThreads < nout ? ld_nc_pinned(pt + ooff[u]) : 0.f;
  };
  // Reverse mode (the backward pass): steps run T-1 .. 0, the previous
  // step's h is y[ts + 1] (the deltas), P is the masked dy, and the output
  // is P + sum, or 0 where P holds the mask marker
  const bool rev = c.reverse != 0;
  if (T > 0) load_p(rev ? T - 1 : 0);
  bool bad = false;       // this thread saw a failed wait
  bool aborted = false;   // uniform: the CTA left the step loop early
  int last_mma = -1;      // threads 0 and 32: the last step whose MMAs they issued
  // trace build: thread 128 stores each stamp straight into the step's record
  // (a record held in registers until the step's end made every thread spill,
  // and the reloads inflated the phases they fell in)
  uint32_t* rec = nullptr;  // thread 128's record of the current step, else null
  auto stamp = [&](int k) {
    if constexpr (TR) {
      if (rec) rec[k] = (uint32_t)clock64();
    }
  };
  auto stamp_ns = [&](int k) {
    if constexpr (TR) {
      if (rec) {
        const uint64_t g = global_ns();
        rec[k] = (uint32_t)g;
        rec[k + 1] = (uint32_t)(g >> 32);
      }
    }
  };
  for (int t = 0; t < T; ++t) {
    const int par = t & 1;
    const int ts = rev ? T - 1 - t : t;  // the step computed (t counts the steps done)
    if constexpr (TR)
      rec = tid == 128 && a.trace ? a.trace + ((size_t)t * c.n_cta + blockIdx.x) * kTraceWords
                                  : nullptr;
    stamp(4);
    w.new_step();
    float pv[kOutMax];
#pragma unroll
    for (int u = 0; u < kOutMax; ++u) pv[u] = pn[u];
    if (t + 1 < T) load_p(rev ? ts - 1 : ts + 1);
    // ---- 1. h_{t-1} of the slice -> hi / lo fp16 in the B operand ----
    const float* src = (t == 0 ? a.h0_rows : c.y + (size_t)(rev ? ts + 1 : ts - 1) * B * H) + k0;
    const bool poll = t > 0;
    if (poll) spin_cycles(c.poll_delay);
    bool large = false;
    uint32_t round_max = 0;
    {
      float4 v[PM];
#pragma unroll
      for (int u = 0; u < PM; ++u)
        if ((items >> u) & 1u)
          v[u] = poll ? ld_relaxed_f4(src + goff[u])
                      : __ldg(reinterpret_cast<const float4*>(src + goff[u]));
      // each float4 is split and stored as soon as it is fresh, so the
      // conversions of early data overlap the loads still in flight (checking
      // all of them first and converting in one straight run measured slower:
      // H=1152 B=32 3.40 -> 4.24 us per step)
      unsigned pending = items;
      uint32_t spins = 0, round = 0;
      while (pending != 0u) {
#pragma unroll
        for (int u = 0; u < PM; ++u)
          if (((pending >> u) & 1u) && (!poll || ready4(v[u]))) {  // h0 is not polled
            large |= !(fabsf(v[u].x) < kSplitLarge) | !(fabsf(v[u].y) < kSplitLarge) |
                     !(fabsf(v[u].z) < kSplitLarge) | !(fabsf(v[u].w) < kSplitLarge);
            store_split<BP>(gB + soff[u], v[u], 1.f);
            pending &= ~(1u << u);
          }
        if (pending == 0u) break;
        if (!w.still_ok(spins)) {
          report_timeout(c.status, t, blockIdx.x);
          bad = true;
          break;
        }
        w.pause(round);
        if constexpr (TR) round_max = round > round_max ? round : round_max;
#pragma unroll
        for (int u = 0; u < PM; ++u)
          if ((pending >> u) & 1u) v[u] = ld_relaxed_f4(src + goff[u]);
      }
    }
    stamp(5);
    if constexpr (TR) {
      if (rec) rec[18] = round_max;
    }
    if (large) s_large[par] = 1;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (__syncthreads_or(bad)) {
      aborted = true;
      break;
    }
    stamp(6);
    stamp_ns(14);
    // a value too large for the fp16 split (rare): scale the slice by 2^-e
    int e = 0;
    if (s_large[par]) {
      float m = 0.f;
#pragma unroll
      for (int u = 0; u < PM; ++u)
        if ((items >> u) & 1u) {
          const float* q = src + goff[u];
          const float4 v = poll ? ld_relaxed_f4(q) : __ldg(reinterpret_cast<const float4*>(q));
          m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) s_red[warp] = m;
      __syncthreads();
      m = 0.f;
#pragma unroll
      for (int k = 0; k < kSplitThreads / 32; ++k) m = fmaxf(m, s_red[k]);
      // m * 2^-e < 2^15; an infinite value is left as it is
      if (m >= kSplitLarge && m <= 3.0e38f) e = ilogbf(m) - 14;
      const float scale = pow2i(-e);
#pragma unroll
      for (int u = 0; u < PM; ++u)
        if ((items >> u) & 1u) {
          const float* q = src + goff[u];
          const float4 v = poll ? ld_relaxed_f4(q) : __ldg(reinterpret_cast<const float4*>(q));
          store_split<BP>(gB + soff[u], v, scale);
        }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
    }
    // ---- 2. the block's partial product over the slice: kl / 16 MMAs ----
    // Two threads in different warps issue them, the first half of the K
    // steps into accumulator 0 (TMEM columns 0 ..) and the rest into
    // accumulator 1 (columns 64 ..): measured faster than one issuer where
    // the chain is long (H=2304, 24 K steps: B=16 3.82 -> 3.40 us per step)
    if (tid == 0 || tid == 32) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int ks_lo = tid == 0 ? 0 : nks_half, ks_hi = tid == 0 ? nks_half : nks;
      const uint32_t acc = tmem + (tid == 0 ? 0u : 64u);
      // K advances by 16 fp16 = 32 bytes inside the 128-byte swizzle atom:
      // the descriptors' start-address fields (bytes / 16) step by 2 within
      // an atom and by the atom size between atoms
      const uint64_t ad0 = sw128_kmajor_desc(sA), bd0 = sw128_kmajor_desc(sB);
      if constexpr (STR) {
        // the issuer's atoms from its ring, each released by a commit; then
        // the stage of the atom before it is refilled kNsq - 1 atoms ahead
        for (int ai = 0; ai < naq; ++ai) {
          const int n = n_cons, st = n % kNsq;
          if (!wait_phase(&a_full[qi][st], (uint32_t)(n / kNsq) & 1u, c.timeout_ns, c.status)) {
            report_timeout(c.status, t, blockIdx.x);
            bad = true;
            break;
          }
          ++n_cons;
          const uint32_t at = (uint32_t)(a_lo + ai);
          const uint64_t ad = sw128_kmajor_desc(sA + (uint32_t)(qi * kNsq + st) * kAtomA);
          const int k_hi = min(4, nks - 4 * (int)at);
          for (int s4 = 0; s4 < k_hi; ++s4)
            umma_f16(acc, ad + (((uint32_t)s4 * 32u) >> 4),
                     bd0 + ((at * kAtomB + (uint32_t)s4 * 32u) >> 4), idesc,
                     (ai > 0 || s4 > 0) ? 1u : 0u);
          umma_commit(&a_empty[qi][st]);
          const int nn = n + kNsq - 1;  // into the stage of atom n - 1
          if (nn < n_total && nn == n_issued) {
            if (nn >= kNsq &&
                !wait_phase(&a_empty[qi][(nn - kNsq) % kNsq], (uint32_t)((nn - kNsq) / kNsq) & 1u,
                            c.timeout_ns, c.status)) {
              report_timeout(c.status, t, blockIdx.x);
              bad = true;
              break;
            }
            a_copy(nn);
            ++n_issued;
          }
        }
      } else {
        for (int ks = ks_lo; ks < ks_hi; ++ks) {
          const uint32_t at = (uint32_t)(ks >> 2), s4 = (uint32_t)(ks & 3);
          umma_f16(acc, ad0 + ((at * kAtomA + s4 * 32u) >> 4), bd0 + ((at * kAtomB + s4 * 32u) >> 4),
                   idesc, ks > ks_lo ? 1u : 0u);
        }
      }
      umma_commit(&mma_bar);  // with no MMA of its own it arrives at once
      last_mma = t;
      if constexpr (TR) {
        const uint32_t ck = (uint32_t)clock64();
        if (a.trace && tid == 0) a.trace[((size_t)t * c.n_cta + blockIdx.x) * kTraceWords + 13] = ck;
      }
    }
    // ---- 3. warps 4..7: accumulator -> partial sums by column -> owners ----
    if (warp >= 4 && warp < 8) {
      const int wq = warp - 4;  // TMEM lanes (block rows) 32 wq .. 32 wq + 31
      if (!wait_phase(&mma_bar, (uint32_t)t & 1u, c.timeout_ns, c.status)) {
        report_timeout(c.status, t, blockIdx.x);
        bad = true;
      }
      // the TMEM loads below are warp-wide: one decision per warp
      bad = __any_sync(0xffffffffu, bad);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      stamp(7);
      float* dst = stage + (size_t)par * B * 128 + wq * 32 + lane;  // row wq * 32 + lane
      if (!bad) {
        // per column: (hi + lo of accumulator 0) + (hi + lo of accumulator
        // 1), 16 columns at a time
        const uint32_t lanes = tmem + ((uint32_t)(wq * 32) << 16);
        const float unscale = pow2i(e);
        constexpr int kChunk = BP < 16 ? BP : 16;
#pragma unroll
        for (int c0 = 0; c0 < BP; c0 += kChunk) {
          // accumulator 0, then accumulator 1 (fewer registers live at once)
          float sum[16];
          uint32_t hv[16], lv[16];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (q == 1 && (STR ? nat <= 1 : nks <= 1)) break;  // issuer 1 had no K step
            const uint32_t accq = lanes + 64u * (uint32_t)q;
            if constexpr (BP == 8) {  // hi and lo in one 16-column load
              tmem_load_16cols(accq, hv);
#pragma unroll
              for (int i = 0; i < 8; ++i) lv[i] = hv[8 + i];
            } else {
              tmem_load_16cols(accq + (uint32_t)c0, hv);
              tmem_load_16cols(accq + (uint32_t)(BP + c0), lv);
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
              const float pq = __uint_as_float(hv[i]) + __uint_as_float(lv[i]);
              sum[i] = q == 0 ? pq : sum[i] + pq;
            }
          }
#pragma unroll
          for (int i = 0; i < kChunk; ++i)
            if (c0 + i < B) dst[(c0 + i) * 128] = sum[i] * unscale;
        }
      }
      stamp(8);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("bar.sync 1, 128;" ::: "memory");
      // lane o / 4 of warp 4 + o % 4 sends owner o its columns (issue spread
      // over the four warps: H=1152 B=16 2.61 -> 2.54 us per step against
      // lanes 0 .. cs-1 of warp 4 alone)
      const int o_send = (lane << 2) | (warp - 4);
      if (lane < 2 && o_send < cs && o_send != j && !bad) {
        const int o = o_send, ob = o * B / cs, on = (o + 1) * B / cs - ob;
        if (on > 0)
          bulk_to_peer(peer_addr(smem_u32(recv + ((size_t)par * cs + j) * maxcol * 128), (uint32_t)o),
                       smem_u32(stage + ((size_t)par * B + ob) * 128), (uint32_t)on * 512u,
                       peer_addr(smem_u32(&recv_bar[par]), (uint32_t)o));
      }
      stamp(9);
    }
    if (__syncthreads_or(bad)) {
      aborted = true;
      break;
    }
    // ---- 4. owner: cs partials + P_t -> ReLU -> h_t ----
    stamp(10);
    if (!wait_phase(&recv_bar[par], (uint32_t)(t >> 1) & 1u, c.timeout_ns, c.status)) {
      report_timeout(c.status, t, blockIdx.x);
      bad = true;
    }
    stamp(11);
    if (!bad) {
      const bool publish = !(blockIdx.x == c.drop_cta && t == c.drop_step);
      const float* own = stage + ((size_t)par * B + cb0) * 128;
      const float* in = recv + (size_t)par * cs * maxcol * 128;
#pragma unroll
      for (int u = 0; u < kOutMax; ++u) {
        const int o = tid + u * kSplitThreads;
        if (o < nout) {
          // slices in order 0 .. cs-1 whichever CTA owns the column, so a
          // column's bits do not depend on the batch around it (the loads
          // first, all independent; adding the zeros past cs changes nothing)
          float part[kKsplitMaxCluster];
#pragma unroll
          for (int k = 0; k < kKsplitMaxCluster; ++k)
            part[k] = k >= cs ? 0.f : (k == j ? own[o] : in[(size_t)k * maxcol * 128 + o]);
          float sum = pv[u];
#pragma unroll
          for (int k = 0; k < kKsplitMaxCluster; ++k) sum += part[k];
          if (publish) {
            const float out =
                c.p_masked ? (__float_as_uint(pv[u]) == kMaskedMarker ? 0.f : sum) : relu(sum);
            const size_t yo = (size_t)ts * step_floats + ooff[u];
            st_relaxed_f(c.y + yo, out);
            if (c.y_mirror) c.y_mirror[yo] = out;
          }
        }
      }
    }
    if constexpr (TR) {
      if (rec) {
        stamp(12);
        stamp_ns(16);
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        rec[0] = smid;
        rec[1] = blockIdx.x;
        rec[2] = (uint32_t)cs;
        rec[3] = (uint32_t)j;
        rec[19] = 0;
      }
    }
    if (tid == 0) {
      // this parity's flag and mbarrier serve step t + 2 next (every thread
      // read the flag before the last barrier; no peer copies step t + 2's
      // blocks before this CTA has published all of step t).  The mbarrier is
      // armed again only once this thread has seen its phase complete: an
      // arrival on a phase that has none pending is not allowed
      s_large[par] = 0;
      if (t + 2 < T && !bad) mbar_arrive_expect_tx(&recv_bar[par], in_bytes);
    }
  }
  // ---- leave: MMAs retired, TMEM freed, then meet the cluster peers ----
  if ((tid == 0 || tid == 32) && last_mma >= 0) wait_own_mmas(&mma_bar, (uint32_t)last_mma & 1u);
  if constexpr (STR) {
    if (tid == 0 || tid == 32) {
      // every MMA this thread issued (its last commit covers them all), and
      // the A copies still in flight into its ring
      if (n_cons > 0) wait_own_mmas(&a_empty[qi][(n_cons - 1) % kNsq], (uint32_t)((n_cons - 1) / kNsq) & 1u);
      for (int n = n_cons; n < n_issued; ++n)
        wait_own_mmas(&a_full[qi][n % kNsq], (uint32_t)(n / kNsq) & 1u);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  // a wait that gave up in the last step counts as leaving early too
  aborted = __syncthreads_or(aborted || bad) != 0;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kSplitTmemCols)
                 : "memory");
  cluster_sync_all();  // every peer has issued its last copy
  if (aborted) {
    // a copy issued by a peer before it left may still be landing here
    const uint64_t until = global_ns() + 50000ull;
    while (global_ns() < until) {
    }
  }
}

}  // namespace

size_t recur_dense_ksplit_smem(int nat, int B, int cs, bool stream) {
  const int bp = B <= 8 ? 8 : (B <= 16 ? 16 : 32);
  const int maxcol = (B + cs - 1) / cs;
  return 1024 + (size_t)(stream ? 2 * kNsq : nat) * kAtomA + (size_t)nat * (2 * bp) * 128 +
         (size_t)2 * B * 128 * sizeof(float) + (size_t)2 * cs * maxcol * 128 * sizeof(float);
}

namespace {

template <int BP, bool TR, bool STR>
cudaError_t launch_bp(const DenseSplitArgs& a, cudaStream_t s, bool query_only, int* clusters_fit) {
  const size_t smem = recur_dense_ksplit_smem(a.nat, a.c.B, a.cs, STR);
  cudaError_t e = cudaFuncSetAttribute(recur_dense_ksplit_kernel<BP, TR, STR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.c.n_cta);
  cfg.blockDim = dim3(kSplitThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)a.cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.attrs = at;
  if (query_only) {
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters_fit, recur_dense_ksplit_kernel<BP, TR, STR>, &cfg);
  }
  // every CTA waits on CTAs of other clusters: the cooperative launch makes
  // the grid co-resident (or fails rather than run part of it)
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, recur_dense_ksplit_kernel<BP, TR, STR>, a);
}

}  // namespace

int recur_dense_ksplit_plan(int H, bool* stream) {
  *stream = false;
  if (H < 128 || H % 128 != 0) return 0;
  int dev = 0, cl = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&cl, cudaDevAttrClusterLaunch, dev) != cudaSuccess || !cl ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  const int nblk = H / 128;
  for (int cs = kKsplitMaxCluster; cs >= 2; --cs) {
    if (H / 16 < cs) continue;  // every slice holds at least one K step
    if ((H / 16 + cs - 1) / cs * 16 > kKsplitMaxSlice) continue;  // one poll round per thread
    DenseSplitArgs a{};
    a.c.B = kKsplitMaxB;  // the widest batch takes the most shared memory
    a.c.n_cta = nblk * cs;
    a.cs = cs;
    a.nat = ksplit_nat(H, cs);
    if (recur_dense_ksplit_smem(a.nat, kKsplitMaxB, cs, false) > (size_t)optin) continue;
    int fit = 0;
    if (launch_bp<32, false, false>(a, nullptr, true, &fit) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (fit >= nblk) return cs;
  }
  // the weights do not fit beside the operand tiles: A streamed from the
  // image through rings, for batches of up to 16 columns
  for (int cs = kKsplitMaxCluster; cs >= 2; --cs) {
    if (H / 16 < 2 * 4 * cs) continue;  // two atoms per slice at least
    if ((H / 16 + cs - 1) / cs * 16 > kKsplitMaxSliceStream) continue;
    DenseSplitArgs a{};
    a.c.B = 16;
    a.c.n_cta = nblk * cs;
    a.cs = cs;
    a.nat = ksplit_nat(H, cs);
    if (recur_dense_ksplit_smem(a.nat, 16, cs, true) > (size_t)optin) continue;
    int fit = 0;
    if (launch_bp<16, false, true>(a, nullptr, true, &fit) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (fit >= nblk) {
      *stream = true;
      return cs;
    }
  }
  return 0;
}

cudaError_t launch_recur_dense_ksplit(const DenseSplitArgs& a, cudaStream_t s) {
  const int B = a.c.B, H = a.c.H;
  if (B < 1 || B > kKsplitMaxB || H % 128 != 0 || a.cs < 2 || a.cs > kKsplitMaxCluster ||
      a.c.n_cta != H / 128 * a.cs || a.nat != ksplit_nat(H, a.cs))
    return cudaErrorInvalidValue;
  if (a.stream) {
    if (B > 16 || (H / 16 + a.cs - 1) / a.cs * 16 > kKsplitMaxSliceStream)
      return cudaErrorInvalidValue;
    if (a.trace)
      return B <= 8 ? launch_bp<8, true, true>(a, s, false, nullptr)
                    : launch_bp<16, true, true>(a, s, false, nullptr);
    return B <= 8 ? launch_bp<8, false, true>(a, s, false, nullptr)
                  : launch_bp<16, false, true>(a, s, false, nullptr);
  }
  if ((H / 16 + a.cs - 1) / a.cs * 16 > kKsplitMaxSlice) return cudaErrorInvalidValue;
  if (a.trace) {
    if (B <= 8) return launch_bp<8, true, false>(a, s, false, nullptr);
    if (B <= 16) return launch_bp<16, true, false>(a, s, false, nullptr);
    return launch_bp<32, true, false>(a, s, false, nullptr);
  }
  if (B <= 8) return launch_bp<8, false, false>(a, s, false, nullptr);
  if (B <= 16) return launch_bp<16, false, false>(a, s, false, nullptr);
  return launch_bp<32, false, false>(a, s, false, nullptr);
}

}  // namespace prnn
