// persistent_dense.cu -- the persistent recurrent kernel for dense Wh.
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
// Dense kernel.  Thread i owns the 4-column chunks i, i+NT, ... (all R rows of
// the CTA for those columns), so each h value it loads is reused for R rows
// straight from registers; h_{t-1} goes from L2 into registers directly (no
// smem staging).  Weights: smem, [chunk slot j][row r][thread] of 4-weight
// vectors, so a warp's weight loads are consecutive 8/16-byte words
// (128-bit-friendly, bank-conflict-free).  Partial sums are reduced across the
// warp by a reduce-scatter and across warps through smem.  BW batch columns
// are processed per pass.
// ---------------------------------------------------------------------------
template <bool F16, int RMAX, int BW, int CPT>
__global__ void __launch_bounds__(dense_launch_bound(F16, RMAX, BW, CPT), 1)
    recur_dense_kernel(const DenseRecurArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NT = blockDim.x, nwarps = NT >> 5;
  const int cta = blockIdx.x;
  const int H = c.H, B = c.B, R = c.R;
  const Place pl = place_of(c);
  const int nchunks = H >> 2;
  constexpr int VB = F16 ? 8 : 16;
  constexpr int V = RMAX * BW;

  float* red = reinterpret_cast<float*>(smem + (size_t)CPT * R * NT * VB);

  {  // this CTA's weights, loaded once for the whole sequence
    const size_t bytes = (size_t)CPT * R * NT * VB;
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const unsigned char*>(a.Wpk) + (size_t)pl.lc * bytes);
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (size_t i = tid; i < bytes / 16; i += NT) dst[i] = __ldg(src + i);
  }
  if (tid == 0) s_abort = 0;
  __syncthreads();

  // No guards inside the unrolled loops (they stop the compiler from batching
  // the shared loads): chunk slots past the matrix read chunk 0 of h, rows
  // past R read row R-1's weights; both multiply zero-padded weights or feed
  // sums that are never stored.
  int chv[CPT];
  bool chok[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    chok[j] = tid + j * NT < nchunks;
    chv[j] = chok[j] ? tid + j * NT : 0;
  }

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
    for (int b0 = pl.b_lo; b0 < pl.b_hi; b0 += BW, ++seq) {
      const int nb = min(BW, pl.b_hi - b0);
      // P for the output this thread finalizes (index tid = r*BW + b)
      float pv = 0.f;
      int orow = -1, ob = -1;
      if (tid < V) {
        const int r = tid / BW, bb = tid % BW;
        if (r < pl.rows && bb < nb) {
          orow = pl.row0 + r;
          ob = b0 + bb;
          pv = ld_nc_pinned(Pt + (size_t)ob * H + orow);
        }
      }
      // issue every load of h_{t-1} this thread needs (batch columns past nb
      // reuse column b0), then wait on them
      if (t > 0 && b0 == pl.b_lo) spin_cycles(c.poll_delay);
      float4 hv[CPT][BW];
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
#pragma unroll
        for (int bb = 0; bb < BW; ++bb) {
          const int b = bb < nb ? b0 + bb : b0;
          hv[j][bb] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (hprev != nullptr) {
            const float* p = hprev + (size_t)b * H + chv[j] * 4;
            hv[j][bb] = (t == 0) ? __ldg(reinterpret_cast<const float4*>(p)) : ld_relaxed_f4(p);
          }
        }
      }
      // wait until every loaded chunk is fresh, re-issuing all stale loads each round
      bool ok = true;
      if (t > 0) {
        uint32_t spins = 0, round = 0;
        for (;;) {
          unsigned stale = 0;
#pragma unroll
          for (int j = 0; j < CPT; ++j)
#pragma unroll
            for (int bb = 0; bb < BW; ++bb)
              if (!ready4(hv[j][bb])) stale |= 1u << (j * BW + bb);
          if (stale == 0u) break;
          if (!w.still_ok(spins)) {
            ok = false;
            break;
          }
          w.pause(round);
#pragma unroll
          for (int j = 0; j < CPT; ++j)
#pragma unroll
            for (int bb = 0; bb < BW; ++bb)
              if ((stale >> (j * BW + bb)) & 1u)
                hv[j][bb] = ld_relaxed_f4(hprev + (size_t)(bb < nb ? b0 + bb : b0) * H + chv[j] * 4);
        }
      }
      float acc[RMAX][BW];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int bb = 0; bb < BW; ++bb) acc[r][bb] = 0.f;
      // rows in blocks of RB; between blocks the empty asm keeps the next
      // block's weight loads from being hoisted (bounds the registers in flight)
      constexpr int RB = dense_row_block(F16, RMAX, BW, CPT);
#pragma unroll
      for (int r0 = 0; r0 < RMAX; r0 += RB) {
        if (RB < RMAX) asm volatile("" ::: "memory");
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int wv = j * R * NT + tid;  // vector index of (slot j, row 0)
#pragma unroll
        for (int r = r0; r < (r0 + RB < RMAX ? r0 + RB : RMAX); ++r) {
          const int rr = r < R ? r : R - 1;
          float w0, w1, w2, w3;
          if constexpr (F16) {
            const uint2 u = reinterpret_cast<const uint2*>(smem)[wv + rr * NT];
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            w0 = fa.x; w1 = fa.y; w2 = fb.x; w3 = fb.y;
          } else {
            const float4 f = reinterpret_cast<const float4*>(smem)[wv + rr * NT];
            w0 = f.x; w1 = f.y; w2 = f.z; w3 = f.w;
          }
          if (!chok[j]) w0 = w1 = w2 = w3 = 0.f;  // slot past the matrix: chunk 0 was loaded
#pragma unroll
          for (int bb = 0; bb < BW; ++bb) {
            float s = acc[r][bb];
            s = fmaf(w0, hv[j][bb].x, s);
            s = fmaf(w1, hv[j][bb].y, s);
            s = fmaf(w2, hv[j][bb].z, s);
            s = fmaf(w3, hv[j][bb].w, s);
            acc[r][bb] = s;
          }
        }
      }
      }
      float v[V];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int bb = 0; bb < BW; ++bb) v[r * BW + bb] = acc[r][bb];
      seg_reduce_scatter<V, 32>(v, lane);
      float* rb = red + (size_t)(seq & 1) * nwarps * V;
      if (V >= 32) {
#pragma unroll
        for (int i = 0; i < (V >= 32 ? V / 32 : 1); ++i) rb[warp * V + lane * (V / 32) + i] = v[i];
      } else {
        constexpr int DREP = (V >= 32) ? 1 : 32 / V;
        if ((lane % DREP) == 0) rb[warp * V + lane / DREP] = v[0];
      }
      if (!ok) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;
      if (orow >= 0) {
        float s = pv;
        for (int ww = 0; ww < nwarps; ++ww) s += rb[ww * V + tid];
        if (!(cta == c.drop_cta && t == c.drop_step)) {
          const float out = c.p_masked ? (__float_as_uint(pv) == kMaskedMarker ? 0.f : s) : relu(s);
          st_relaxed_f(yt + (size_t)ob * H + orow, out);
          if (c.y_mirror) c.y_mirror[(size_t)tt * B * H + (size_t)ob * H + orow] = out;
        }
      }
    }
    if (c.sync_mode == 1) {
      grid_barrier(c, t, w, &s_abort);
      if (s_abort) return;
    }
  }
}

}  // namespace

int recur_dense_rmax(int R) {
  if (R <= 4) return 4;
  if (R <= 8) return 8;
  if (R <= 16) return 16;
  if (R <= 32) return 32;
  return 0;
}

int recur_dense_bw(int bl) { return bl <= 1 ? 1 : bl <= 2 ? 2 : 4; }

size_t recur_dense_smem(int R, int cpt, int nthreads, bool fp16, int bw) {
  const int rmax = recur_dense_rmax(R);
  return (size_t)cpt * R * nthreads * (fp16 ? 8 : 16) +
         (size_t)2 * (nthreads / 32) * rmax * bw * sizeof(float);
}

cudaError_t launch_recur_dense(const DenseRecurArgs& a, int bw, cudaStream_t s) {
  void* args[] = {const_cast<DenseRecurArgs*>(&a)};
  const int rmax = recur_dense_rmax(a.c.R);
  const int g = a.c.n_cta, nt = a.c.nthreads;
  const size_t sm = a.c.smem;
  const int cpt = a.cpt;
#define PRNN_DENSE_CASE(F, RM, BW_, CP) \
  if (a.wfp16 == F && rmax == RM && bw == BW_ && cpt == CP) \
    return coop_launch(recur_dense_kernel<F, RM, BW_, CP>, g, nt, sm, s, args);
#define PRNN_DENSE_CPT(F, RM, BW_) \
  PRNN_DENSE_CASE(F, RM, BW_, 1) PRNN_DENSE_CASE(F, RM, BW_, 2) \
  PRNN_DENSE_CASE(F, RM, BW_, 3) PRNN_DENSE_CASE(F, RM, BW_, 4)
#define PRNN_DENSE_ROW(F, RM) \
  PRNN_DENSE_CPT(F, RM, 1) PRNN_DENSE_CPT(F, RM, 2) PRNN_DENSE_CPT(F, RM, 4)
  PRNN_DENSE_ROW(1, 4) PRNN_DENSE_ROW(1, 8) PRNN_DENSE_ROW(1, 16) PRNN_DENSE_ROW(1, 32)
  PRNN_DENSE_ROW(0, 4) PRNN_DENSE_ROW(0, 8) PRNN_DENSE_ROW(0, 16) PRNN_DENSE_ROW(0, 32)
#undef PRNN_DENSE_ROW
#undef PRNN_DENSE_CPT
#undef PRNN_DENSE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace prnn
