// persistent_sparse.cu -- the persistent recurrent kernel for row-balanced
// sparse Wh, and the step-synchronisation floor probe.
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
#include "persistent_common.cuh"

namespace prnn {

using namespace pk;

namespace {

// ---------------------------------------------------------------------------
// Sparse row-balanced kernel.  Thread (r, s) = (tid / TPR, tid % TPR) owns
// ept entries of row r, packed 4 to a uint4 (wide loads); entry = fp16 value
// | column << 16, padding entries have value 0.  The host places entries so
// that the 32 lanes of a warp gather from different banks in each slot.  The
// first kRegQ uint4 groups live in registers, the rest in smem.  The group's
// h_{t-1} columns are staged in smem as [b][H] per batch pass of BG columns
// (double-buffered when it fits, so one CTA barrier per pass).
// ---------------------------------------------------------------------------
template <int TPR, int BG>
__global__ void __launch_bounds__(kSparseThreads, 1) recur_sparse_kernel(const SparseRecurArgs a) {
  extern __shared__ __align__(16) float smem_f[];
  __shared__ int s_abort;
  constexpr int UMAX = (BG >= 16) ? 4 : (BG == 8 ? 8 : 12);
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
  constexpr int REGQ = (BG >= 16) ? 2 : kRegQ;
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
  int seq = 0;
  for (int t = 0; t < c.T; ++t) {
    const int tt = c.reverse ? c.T - 1 - t : t;  // time index of this step
    const float* hprev = (t == 0) ? c.h0 : c.y + (size_t)(c.reverse ? tt + 1 : tt - 1) * B * H;
    const float* Pt = c.P + (size_t)tt * B * H;
    float* yt = c.y + (size_t)tt * B * H;
    w.new_step();
    for (int bs = pl.b_lo; bs < pl.b_hi; bs += BG, ++seq) {
      const int nbg = min(BG, pl.b_hi - bs);
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
      if (t > 0 && bs == pl.b_lo) spin_cycles(c.poll_delay);
      const bool ok = a.narrow
                          ? stage_rows_narrow<UMAX>(hprev, t > 0, H, bs, nbg, smem_f + hs_off, w)
                          : stage_rows<UMAX>(hprev, t > 0, H, bs, nbg, smem_f + hs_off, w);
      if (!ok) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;

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
      if (TPR > 1) seg_reduce_scatter<BG, TPR>(acc, lane);
      if (owns && !(cta == c.drop_cta && t == c.drop_step)) {
#pragma unroll
        for (int i = 0; i < NOUT; ++i) {
          const int idx = (BG >= TPR) ? gl * NOUT + i : gl / REP;
          if (idx < nbg) {
            const float s = acc[i] + pv[i];
            st_relaxed_f(yt + (size_t)(bs + idx) * H + row,
                         c.p_masked ? (__float_as_uint(pv[i]) == kMaskedMarker ? 0.f : s)
                                    : relu(s));
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

// ---------------------------------------------------------------------------
// Sync-floor probe: the sparse kernel's exchange (stage the group's columns of
// h_{t-1}, one CTA barrier, publish R rows of h_t) with no arithmetic.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSparseThreads, 1) sync_probe_kernel(const RecurCommon c, int BG) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  float* hs = reinterpret_cast<float*>(smem);
  const int tid = threadIdx.x, cta = blockIdx.x;
  const int H = c.H, B = c.B;
  const Place pl = place_of(c);
  if (tid == 0) s_abort = 0;
  __syncthreads();
  Waiter w;
  w.status = c.status;
  w.timeout_ns = c.timeout_ns;
  w.backoff = c.poll_backoff;
  for (int t = 0; t < c.T; ++t) {
    const float* hprev = (t == 0) ? nullptr : c.y + (size_t)(t - 1) * B * H;
    float* yt = c.y + (size_t)t * B * H;
    w.new_step();
    for (int bs = pl.b_lo; bs < pl.b_hi; bs += BG) {
      const int nbg = min(BG, pl.b_hi - bs);
      bool ok = true;
      if (t > 0 && bs == pl.b_lo) spin_cycles(c.poll_delay);
      if (t > 0) ok = stage_rows<8>(hprev, true, H, bs, nbg, hs, w);
      if (!ok) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;
      for (int i = tid; i < pl.rows * nbg; i += blockDim.x) {
        const int rr = i % pl.rows, bb = i / pl.rows;
        st_relaxed_f(yt + (size_t)(bs + bb) * H + pl.row0 + rr, (float)(t + 1));
      }
      __syncthreads();
    }
  }
}

}  // namespace

size_t recur_sparse_smem(int H, int R, int ept, int tpr, int bgroup, bool dbuf) {
  // weights: R rows x (ept * tpr) packed 4-byte entries; then the h staging buffers
  return (size_t)R * ept * tpr * 4 + (size_t)(dbuf ? 2 : 1) * H * bgroup * sizeof(float);
}

cudaError_t launch_recur_sparse(const SparseRecurArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<SparseRecurArgs*>(&a)};
  const int g = a.c.n_cta, nt = a.c.nthreads;
  const size_t sm = a.c.smem;
  const int bg = a.bgroup;
#define PRNN_SPARSE_CASE(T_, BG_) \
  if (a.tpr == T_ && bg == BG_) return coop_launch(recur_sparse_kernel<T_, BG_>, g, nt, sm, s, args);
#define PRNN_SPARSE_ROW(T_)                                                           \
  PRNN_SPARSE_CASE(T_, 1) PRNN_SPARSE_CASE(T_, 2) PRNN_SPARSE_CASE(T_, 4) PRNN_SPARSE_CASE(T_, 8) \
  PRNN_SPARSE_CASE(T_, 16) PRNN_SPARSE_CASE(T_, 32)
  PRNN_SPARSE_ROW(1) PRNN_SPARSE_ROW(2) PRNN_SPARSE_ROW(4) PRNN_SPARSE_ROW(8)
  PRNN_SPARSE_ROW(16) PRNN_SPARSE_ROW(32)
#undef PRNN_SPARSE_ROW
#undef PRNN_SPARSE_CASE
  return cudaErrorInvalidValue;
}

size_t sync_probe_smem(int H, int bgroup) { return (size_t)H * bgroup * sizeof(float); }

cudaError_t launch_sync_probe(const RecurCommon& c, int bgroup, cudaStream_t s) {
  int bg = bgroup;
  void* args[] = {const_cast<RecurCommon*>(&c), &bg};
  return coop_launch(sync_probe_kernel, c.n_cta, c.nthreads, c.smem, s, args);
}

}  // namespace prnn
