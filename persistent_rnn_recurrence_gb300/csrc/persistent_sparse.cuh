// persistent_sparse.cuh -- the persistent recurrent kernel for row-balanced
// sparse Wh (a template over threads per row, batch columns per pass and the
// staging order of h) and its launch dispatch.  persistent_sparse.cu
// instantiates it with h staged in column order, persistent_sparse_placed.cu
// with each CTA's own bank-balancing order, so that neither set of kernels
// carries the other's staging code or registers.
//
// One cooperative launch runs all T steps of h_t = ReLU(P_t + Wh h_{t-1})
// (P_t = Wx x_t + b comes from the projection kernel).  Each CTA owns a block
// of R consecutive rows of Wh and loads them into shared memory / registers
// once, so the weights stay on chip for the whole sequence instead of being
// re-read every step (persistent-rnn page, "What This Project Does"; "Sparse
// Persistent RNNs: Squeezing Large Recurrent Networks On-Chip").
//
// CTA groups: the batch columns of the recurrence are independent, so the
// grid is split into G groups of cpg CTAs; group gi owns the contiguous batch
// columns [gi*Bl, gi*Bl + Bl) and holds its own on-chip copy of Wh.  A CTA
// only ever waits for the CTAs of its own group, and reads only its group's
// Bl columns of h_{t-1} per step, which cuts the data each SM pulls from L2
// per step by G.
//
// Step exchange: h_t is published by storing it into y[t] (pre-filled with a
// NaN sentinel); consumers poll y[t-1] with relaxed gpu-scope loads until no
// word is the sentinel.  The data word is its own "ready" flag, so there is no
// grid barrier between steps (the Lamport-timestamp row of the sparse
// persistent RNN ablation).  A grid-barrier mode is kept for that ablation.
//
// Every wait is bounded (globaltimer deadline); on expiry the kernel records
// a status word and every CTA leaves its time loop.
//
// Phase trace (opt-in, TRACE instantiations only): for the first batch pass
// of every step, each warp's lane 0 keeps SM-clock stamps in registers -- pass
// start, projection value requested, end of the pause before the first poll,
// the warp's last staging poll fresh, CTA barrier passed, gathers done,
// reduction done, publish issued -- the most re-poll rounds any lane of the
// warp needed, and globaltimer readings just after the barrier and just after
// the publish (one device-wide clock, 32 ns steps on GB300, so a producer's
// publish and a consumer's barrier can be compared across SMs), and writes
// them with four vector stores after its publish; warp 0 also writes a header
// (SM id, CTA, warps).  No shared memory and no atomics, so the trace
// disturbs the step little.  Layout: [T][n_cta][17][16] words, slot 0 the
// header, slot 1 + w warp w.
#pragma once
#include "persistent_common.cuh"

namespace prnn {

using namespace pk;

namespace {

// ---------------------------------------------------------------------------
// Staging into a per-CTA placement of h (the packer's bank-balancing order;
// opt-in): column 4g+j of batch row b goes to
//     b*H + 128*(g/32) + 32*j + byte j of place[g],
// four 32-bit stores per float4.  Each 32-column class's bytes are a
// permutation of the banks, so the 32 lanes of a warp hit 32 different banks
// per store.  Requires H % 128 == 0; every index stays inside its batch row
// for any table contents (bytes masked to 0..31, block start <= H - 128).
// Loads, polls and the bounded wait are those of stage_rows; the batch row and
// group of each load are stepped, not divided.
// ---------------------------------------------------------------------------
template <int UMAX>
__device__ __forceinline__ bool stage_rows_placed(const float* hprev, bool poll, int H,
                                                  int b_start, int nb, float* hs, Waiter& w,
                                                  const uint32_t* place) {
  const int NT = blockDim.x, tid = threadIdx.x;
  const int ng = H >> 2, nf4 = nb * ng;
  const float4* src = reinterpret_cast<const float4*>(hprev + (size_t)b_start * H);
  for (int base = tid; base < nf4; base += UMAX * NT) {
    float4 v[UMAX];
    uint32_t pw[UMAX];
    const int b0 = base / ng, g0 = base - b0 * ng;
    int b = b0, g = g0;
#pragma unroll
    for (int u = 0; u < UMAX; ++u) {
      const int i = base + u * NT;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      pw[u] = 0u;
      if (i < nf4) {
        pw[u] = __ldg(place + g);
        if (hprev != nullptr)
          v[u] = poll ? ld_relaxed_f4(reinterpret_cast<const float*>(src + i)) : __ldg(src + i);
      }
      g += NT;
      while (g >= ng) {
        g -= ng;
        ++b;
      }
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
    }
    b = b0;
    g = g0;
#pragma unroll
    for (int u = 0; u < UMAX; ++u) {
      if (base + u * NT < nf4) {
        float* blk = hs + b * H + ((g >> 5) << 7);
        blk[pw[u] & 31u] = v[u].x;
        blk[32 + ((pw[u] >> 8) & 31u)] = v[u].y;
        blk[64 + ((pw[u] >> 16) & 31u)] = v[u].z;
        blk[96 + ((pw[u] >> 24) & 31u)] = v[u].w;
      }
      g += NT;
      while (g >= ng) {
        g -= ng;
        ++b;
      }
    }
  }
  return true;
}

// stage_rows_narrow into the same placement (the ablation's 32-bit staging).
template <int UMAX>
__device__ __forceinline__ bool stage_rows_narrow_placed(const float* hprev, bool poll, int H,
                                                         int b_start, int nb, float* hs,
                                                         Waiter& w, const uint32_t* place) {
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
    for (int u = 0; u < UMAX; ++u) {
      const int i = base + u * NT;
      if (i < n) {
        const int b = i / H, c = i - b * H, g = c >> 2, j = c & 3;
        const uint32_t pw = __ldg(place + g);
        hs[(size_t)b * H + ((g >> 5) << 7) + 32 * j + ((pw >> (8 * j)) & 31u)] = v[u];
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// Sparse row-balanced kernel.  Thread (r, s) = (tid / TPR, tid % TPR) owns
// ept entries of row r, packed 4 to a uint4 (wide loads); entry = fp16 value
// | index << 16, padding entries have value 0.  The host places entries so
// that the 32 lanes of a warp gather from different banks in each slot.  The
// first REGQ uint4 groups live in registers, the rest in smem: kRegQ groups
// in the build for up to 512 threads, kRegQWide in the build for up to
// kRegWThreads threads (MAXT), whose larger register budget holds them
// without spilling and lets the compiler keep more gathers in flight.  The group's
// h_{t-1} columns are staged in smem as [b][H] per batch pass of BG columns
// (double-buffered when it fits, so one CTA barrier per pass); the index is
// the column's position in that staging, which is the column itself or, with
// a placement table, this CTA's bank-balancing order of the columns.
// ---------------------------------------------------------------------------
//
// Staging depth UM: the float4 loads of h_{t-1} a thread keeps in flight per
// round.  The launcher picks the smallest of 2, 6 or 12 (UM = 0: 12, and 8 or
// 4 for passes of 8 or more columns) that covers the thread's share of a pass
// in one round: a deeper unrolled staging than the pass needs costs
// registers and code on the step's critical path -- at the 10 % layer of
// 1792 units, 12 slots where 2 suffice cost 0.38 us of a 1.66 us step.
template <int TPR, int BG, bool PLACED, bool TRACE = false, int MAXT = kSparseThreads, int UM = 0>
__global__ void __launch_bounds__(MAXT, 1) recur_sparse_kernel(const SparseRecurArgs a) {
  extern __shared__ __align__(16) float smem_f[];
  __shared__ int s_abort;
  constexpr int UMAX = UM > 0 ? UM : ((BG >= 16) ? 4 : (BG == 8 ? 8 : 12));
  // the 32-bit staging of the ablation moves a quarter of the bytes per load
  constexpr int UNAR = UM > 0 ? (4 * UM < 12 ? 4 * UM : 12) : UMAX;
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, lane = tid & 31;
  const int NT = blockDim.x;
  const int cta = blockIdx.x;
  const int H = c.H, B = c.B, R = c.R;
  const Place pl = place_of(c);
  const int q4 = a.ept >> 2;
  const int nbuf = a.dbuf ? 2 : 1;

  // smem: packed weights (R*q4*TPR uint4), then nbuf staging buffers of BG*H floats
  uint4* Ws = reinterpret_cast<uint4*>(smem_f);
  const int hs_base = R * q4 * TPR * 4;  // float index of the first staging buffer

  {
    const size_t n16 = (size_t)R * q4 * TPR;
    const uint4* src = reinterpret_cast<const uint4*>(a.Wpk) + (size_t)pl.lc * n16;
    for (size_t i = tid; i < n16; i += NT) Ws[i] = __ldg(src + i);
  }
  if (tid == 0) s_abort = 0;
  __syncthreads();

  const int r = tid / TPR, s = tid % TPR;
  const bool has_row = r < pl.rows;
  const int row = pl.row0 + r;
  constexpr int REGQ = (BG >= 16) ? 2 : (MAXT <= kRegWThreads ? kRegQWide : kRegQ);
  uint4 wr[REGQ];
#pragma unroll
  for (int i = 0; i < REGQ; ++i) {
    wr[i] = make_uint4(0u, 0u, 0u, 0u);
    if (has_row && i < q4) wr[i] = Ws[((size_t)r * q4 + i) * TPR + s];
  }
  // output slots of this lane after the reduce-scatter
  constexpr int NOUT = (BG >= TPR) ? BG / TPR : 1;
  constexpr int REP = (BG >= TPR) ? 1 : TPR / BG;  // lanes holding copies of one sum
  const int gl = lane % TPR;

  Waiter w;
  w.status = c.status;
  w.timeout_ns = c.timeout_ns;
  w.backoff = c.poll_backoff;
  // trace state (registers of every lane; lane 0 of each warp writes it)
  uint32_t ts[9] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  uint64_t gt_bar = 0, gt_pub = 0;
  uint32_t rounds = 0;
  auto stamp = [&](int ph) {
    if (TRACE) ts[ph] = (uint32_t)clock64();
  };
  int seq = 0;
  for (int t = 0; t < c.T; ++t) {
    const int tt = c.reverse ? c.T - 1 - t : t;  // time index of this step
    const float* hprev = (t == 0) ? c.h0 : c.y + (size_t)(c.reverse ? tt + 1 : tt - 1) * B * H;
    const float* Pt = c.P + (size_t)tt * B * H;
    float* yt = c.y + (size_t)tt * B * H;
    w.new_step();
    for (int bs = pl.b_lo; bs < pl.b_hi; bs += BG, ++seq) {
      const int nbg = min(BG, pl.b_hi - bs);
      const bool tr = TRACE && bs == pl.b_lo;  // the trace records each step's first pass
      if (tr) {
        stamp(0);
        rounds = 0;
      }
      const int hs_off = hs_base + ((nbuf == 2) ? (seq & 1) : 0) * H * BG;
      // P for this lane's outputs, fetched before the wait
      float pv[NOUT];
      bool owns = false;
#pragma unroll
      for (int i = 0; i < NOUT; ++i) {
        pv[i] = 0.f;
        const int idx = (BG >= TPR) ? gl * NOUT + i : gl / REP;
        const bool mine = (gl % REP) == 0;
        if (has_row && mine && idx < nbg) {
          pv[i] = ld_nc_pinned(Pt + (size_t)(bs + idx) * H + row);
          owns = true;
        }
      }
      if (tr) stamp(1);
      if (t > 0 && bs == pl.b_lo) spin_cycles(c.poll_delay);
      if (tr) stamp(2);
      // the placed staging keeps fewer loads in flight (its table words take
      // registers of their own)
      constexpr int UPL = UMAX > 4 ? UMAX / 2 : UMAX;
      const bool ok =
          PLACED ? (a.narrow ? stage_rows_narrow_placed<UPL>(hprev, t > 0, H, bs, nbg,
                                                             smem_f + hs_off, w,
                                                             a.place + (size_t)pl.lc * (H >> 2))
                             : stage_rows_placed<UPL>(hprev, t > 0, H, bs, nbg, smem_f + hs_off,
                                                      w, a.place + (size_t)pl.lc * (H >> 2)))
                 : (a.narrow ? stage_rows_narrow<UNAR>(hprev, t > 0, H, bs, nbg, smem_f + hs_off, w)
                             : stage_rows<UMAX>(hprev, t > 0, H, bs, nbg, smem_f + hs_off, w,
                                                TRACE ? &rounds : nullptr));
      if (tr) {
        ts[3] = __reduce_max_sync(0xffffffffu, (uint32_t)clock64());
        ts[8] = __reduce_max_sync(0xffffffffu, rounds);
      }
      if (!ok) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;
      if (tr) {
        stamp(4);
        if (lane == 0) gt_bar = global_ns();
      }

      // gather-multiply: entry = fp16 value (low half) | column << 16.  Batch
      // columns past nbg read a zero-filled or stale row and are never stored.
      float acc[BG];
#pragma unroll
      for (int i = 0; i < BG; ++i) acc[i] = 0.f;
      if (has_row) {
        // groups past q4 hold zero words (value 0 at column 0): no guard needed
#pragma unroll
        for (int i = 0; i < REGQ; ++i) {
          const uint32_t ws4[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float val = __half2float(__ushort_as_half((unsigned short)(ws4[q] & 0xffffu)));
            const int hi = hs_off + (int)(ws4[q] >> 16);
#pragma unroll
            for (int b = 0; b < BG; ++b) acc[b] = fmaf(val, smem_f[hi + b * H], acc[b]);
          }
        }
        for (int i = REGQ; i < q4; ++i) {
          const uint4 e = Ws[((size_t)r * q4 + i) * TPR + s];
          const uint32_t ws4[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float val = __half2float(__ushort_as_half((unsigned short)(ws4[q] & 0xffffu)));
            const int hi = hs_off + (int)(ws4[q] >> 16);
#pragma unroll
            for (int b = 0; b < BG; ++b) acc[b] = fmaf(val, smem_f[hi + b * H], acc[b]);
          }
        }
      }
      if (tr) stamp(5);
      if (TPR > 1) seg_reduce_scatter<BG, TPR>(acc, lane);
      if (tr) stamp(6);
      if (owns && !(cta == c.drop_cta && t == c.drop_step)) {
#pragma unroll
        for (int i = 0; i < NOUT; ++i) {
          const int idx = (BG >= TPR) ? gl * NOUT + i : gl / REP;
          if (idx < nbg) {
            const float s = acc[i] + pv[i];
            const float out = c.p_masked ? (__float_as_uint(pv[i]) == kMaskedMarker ? 0.f : s)
                                         : relu(s);
            st_relaxed_f(yt + (size_t)(bs + idx) * H + row, out);
            if (c.y_mirror) c.y_mirror[(size_t)tt * B * H + (size_t)(bs + idx) * H + row] = out;
          }
        }
      }
      if (tr) {
        stamp(7);
        if (lane == 0 && a.trace != nullptr) {
          gt_pub = global_ns();
          uint32_t* rec = a.trace + ((size_t)t * c.n_cta + cta) * kTraceWords;
          uint4* wr4 = reinterpret_cast<uint4*>(rec + 16 * (1 + (tid >> 5)));
          wr4[0] = make_uint4(ts[0], ts[1], ts[2], ts[3]);
          wr4[1] = make_uint4(ts[4], ts[5], ts[6], ts[7]);
          wr4[2] = make_uint4(ts[8], (uint32_t)gt_bar, (uint32_t)(gt_bar >> 32), (uint32_t)gt_pub);
          wr4[3] = make_uint4((uint32_t)(gt_pub >> 32), (uint32_t)clock64(), 0u, 0u);
          if (tid == 0) {
            uint32_t sm;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
            reinterpret_cast<uint4*>(rec)[0] =
                make_uint4(sm, (uint32_t)cta, (uint32_t)(NT >> 5), 0u);
          }
        }
      }
      if (nbuf == 1) __syncthreads();  // hs is overwritten by the next staging
    }
    if (c.sync_mode == 1) {
      grid_barrier(c, t, w, &s_abort);
      if (s_abort) return;
    }
  }
}

}  // namespace

// One instantiation of the kernel, launched cooperatively; combinations that
// are never planned (the register-weight build or a chosen staging depth with
// passes of more than 4 columns) are never instantiated.
template <int T_, int BG_, bool PLACED, bool TRACE, int MAXT, int UM>
cudaError_t launch_sparse_case(int g, int nt, size_t sm, cudaStream_t s, void** args) {
  if constexpr ((MAXT > kRegWThreads && UM == 0) || BG_ <= 4)
    return coop_launch(recur_sparse_kernel<T_, BG_, PLACED, TRACE, MAXT, UM>, g, nt, sm, s, args);
  else
    return cudaErrorInvalidValue;
}

// Launch recur_sparse_kernel<tpr, bgroup, PLACED, TRACE, MAXT, UM> for the
// plan in a.  The register-weight build (MAXT = kRegWThreads) and the chosen
// staging depths (UM > 0) exist for batch passes of up to 4 columns.
template <bool PLACED, bool TRACE = false, int MAXT = kSparseThreads, int UM = 0>
cudaError_t launch_recur_sparse_impl(const SparseRecurArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<SparseRecurArgs*>(&a)};
  const int g = a.c.n_cta, nt = a.c.nthreads;
  const size_t sm = a.c.smem;
  const int bg = a.bgroup;
  if (nt > MAXT) return cudaErrorInvalidValue;
#define PRNN_SPARSE_CASE(T_, BG_) \
  if (a.tpr == T_ && bg == BG_)   \
    return launch_sparse_case<T_, BG_, PLACED, TRACE, MAXT, UM>(g, nt, sm, s, args);
#define PRNN_SPARSE_ROW(T_)                                                           \
  PRNN_SPARSE_CASE(T_, 1) PRNN_SPARSE_CASE(T_, 2) PRNN_SPARSE_CASE(T_, 4) PRNN_SPARSE_CASE(T_, 8) \
  PRNN_SPARSE_CASE(T_, 16) PRNN_SPARSE_CASE(T_, 32)
  PRNN_SPARSE_ROW(1) PRNN_SPARSE_ROW(2) PRNN_SPARSE_ROW(4) PRNN_SPARSE_ROW(8)
  PRNN_SPARSE_ROW(16) PRNN_SPARSE_ROW(32)
#undef PRNN_SPARSE_ROW
#undef PRNN_SPARSE_CASE
  return cudaErrorInvalidValue;
}

// The builds of one staging order, launch bound and trace setting, for each
// staging depth the launcher may choose (a.umax: 0, 2 or 6).
template <bool PLACED, bool TRACE, int MAXT>
cudaError_t launch_recur_sparse_depth(const SparseRecurArgs& a, cudaStream_t s) {
  switch (a.umax) {
    case 0: return launch_recur_sparse_impl<PLACED, TRACE, MAXT, 0>(a, s);
    case 2: return launch_recur_sparse_impl<PLACED, TRACE, MAXT, 2>(a, s);
    case 6: return launch_recur_sparse_impl<PLACED, TRACE, MAXT, 6>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace prnn
