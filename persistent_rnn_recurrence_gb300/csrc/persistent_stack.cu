// persistent_stack.cu -- a stack of L dense ReLU RNN layers in ONE persistent
// launch, pipelined across layers (a wavefront over (layer, step)).
//
// Layer l computes h^l_t = ReLU(b_l + Wx_l h^{l-1}_t + Wh_l h^l_{t-1}), with
// h^{-1}_t = x_t.  The grid is split into L slices of n_cta CTAs; slice l
// holds the rows of the concatenated matrix [Wx_l | Wh_l] on chip for the
// whole sequence and multiplies it with the concatenated vector
// [h^{l-1}_t ; h^l_{t-1}].  Both halves are polled straight from the layers'
// output sequences y_{l-1}[t] and y_l[t-1] (sentinel-prefilled, the data word
// is its own ready flag), so layer l starts step t as soon as layer l-1 has
// published step t: after a fill of L-1 steps all layers advance together,
// and the stack takes about T + L - 1 step times instead of L * T.  This is
// the multi-layer stage of "Optimizing Performance of Recurrent Neural
// Networks on GPUs" (Abstract: the network is optimized as a whole, with work
// of different layers overlapped) with the on-chip weights of the persistent-rnn
// page ("What This Project Does").
//
// The inner structure is that of the single-layer dense kernel: thread i owns
// 4-column chunks i, i+NT, ... of the concatenated vector for all R rows of
// its CTA; weights in shared memory as [slot][row][thread] 4-weight vectors;
// warp reduce-scatter plus a cross-warp shared-memory sum; CTA groups split
// the batch.  Every wait is bounded (globaltimer deadline, status word).
#include "persistent_common.cuh"

namespace prnn {

using namespace pk;

namespace {

template <bool F16, int RMAX, int BW, int CPT>
__global__ void __launch_bounds__(dense_launch_bound(F16, RMAX, BW, CPT), 1)
    recur_stack_kernel(const StackArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NT = blockDim.x, nwarps = NT >> 5;
  const int layer = blockIdx.x / c.n_cta;
  const int local = blockIdx.x % c.n_cta;
  const StackLayerArgs& L = a.layer[layer];
  const int H = c.H, B = c.B, R = c.R;
  const int I = L.I;
  const int ic = I >> 2;                 // chunks of the layer input
  const int nchunks = ic + (H >> 2);     // chunks of [input ; h]
  Place pl;
  {
    const int gi = local / c.cpg;
    pl.lc = local % c.cpg;
    pl.row0 = pl.lc * R;
    pl.rows = max(0, min(R, H - pl.row0));
    const int bl = (B + c.G - 1) / c.G;
    pl.b_lo = min(B, gi * bl);
    pl.b_hi = min(B, pl.b_lo + bl);
  }
  constexpr int VB = F16 ? 8 : 16;
  constexpr int V = RMAX * BW;

  float* red = reinterpret_cast<float*>(smem + (size_t)CPT * R * NT * VB);

  {  // this CTA's rows of [Wx_l | Wh_l], loaded once for the whole sequence
    const size_t bytes = (size_t)CPT * R * NT * VB;
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const unsigned char*>(L.Wpk) + (size_t)pl.lc * bytes);
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (size_t i = tid; i < bytes / 16; i += NT) dst[i] = __ldg(src + i);
  }
  if (tid == 0) s_abort = 0;
  __syncthreads();

  // chunk slot j of this thread: input chunk (offset into x_t / y_{l-1}[t])
  // or h chunk (offset into h_{t-1}); slots past the vector read chunk 0 of
  // the input and multiply zero weights.
  int off[CPT];
  bool in_src[CPT], chok[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int q = tid + j * NT;
    chok[j] = q < nchunks;
    in_src[j] = !chok[j] || q < ic;
    off[j] = !chok[j] ? 0 : (q < ic ? q * 4 : (q - ic) * 4);
  }

  Waiter w;
  w.status = c.status;
  w.timeout_ns = c.timeout_ns;
  w.backoff = c.poll_backoff;
  int seq = 0;
  for (int t = 0; t < c.T; ++t) {
    const float* xt = L.xin + (size_t)t * B * I;
    const float* hprev = (t == 0) ? L.h0 : L.y + (size_t)(t - 1) * B * H;
    float* yt = L.y + (size_t)t * B * H;
    w.new_step();
    for (int b0 = pl.b_lo; b0 < pl.b_hi; b0 += BW, ++seq) {
      const int nb = min(BW, pl.b_hi - b0);
      float pv = 0.f;
      int orow = -1, ob = -1;
      if (tid < V) {
        const int r = tid / BW, bb = tid % BW;
        if (r < pl.rows && bb < nb) {
          orow = pl.row0 + r;
          ob = b0 + bb;
          pv = __ldg(L.bias + orow);
        }
      }
      // issue every load; polled ones: the layer input when it is produced in
      // this launch, and h_{t-1} for t > 0
      if ((t > 0 || L.poll_in) && b0 == pl.b_lo) spin_cycles(c.poll_delay);
      float4 hv[CPT][BW];
      unsigned pollmask = 0;
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
#pragma unroll
        for (int bb = 0; bb < BW; ++bb) {
          const int b = bb < nb ? b0 + bb : b0;
          hv[j][bb] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (in_src[j]) {
            const float* p = xt + (size_t)b * I + off[j];
            if (L.poll_in) {
              hv[j][bb] = ld_relaxed_f4(p);
              pollmask |= 1u << (j * BW + bb);
            } else {
              hv[j][bb] = __ldg(reinterpret_cast<const float4*>(p));
            }
          } else if (hprev != nullptr) {
            const float* p = hprev + (size_t)b * H + off[j];
            if (t > 0) {
              hv[j][bb] = ld_relaxed_f4(p);
              pollmask |= 1u << (j * BW + bb);
            } else {
              hv[j][bb] = __ldg(reinterpret_cast<const float4*>(p));
            }
          }
        }
      }
      bool ok = true;
      if (pollmask != 0u) {
        uint32_t spins = 0, round = 0;
        for (;;) {
          unsigned stale = 0;
#pragma unroll
          for (int j = 0; j < CPT; ++j)
#pragma unroll
            for (int bb = 0; bb < BW; ++bb)
              if (!ready4(hv[j][bb])) stale |= 1u << (j * BW + bb);
          stale &= pollmask;
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
              if ((stale >> (j * BW + bb)) & 1u) {
                const int b = bb < nb ? b0 + bb : b0;
                const float* p = in_src[j] ? xt + (size_t)b * I + off[j]
                                           : hprev + (size_t)b * H + off[j];
                hv[j][bb] = ld_relaxed_f4(p);
              }
        }
      }
      float acc[RMAX][BW];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int bb = 0; bb < BW; ++bb) acc[r][bb] = 0.f;
      constexpr int RB = dense_row_block(F16, RMAX, BW, CPT);
#pragma unroll
      for (int r0 = 0; r0 < RMAX; r0 += RB) {
        if (RB < RMAX) asm volatile("" ::: "memory");
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int wv = j * R * NT + tid;
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
            if (!chok[j]) w0 = w1 = w2 = w3 = 0.f;
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
        report_timeout(c.status, t, blockIdx.x);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;
      if (orow >= 0) {
        float s = pv;
        for (int ww = 0; ww < nwarps; ++ww) s += rb[ww * V + tid];
        if (!((int)blockIdx.x == c.drop_cta && t == c.drop_step))
          st_relaxed_f(yt + (size_t)ob * H + orow, relu(s));
      }
    }
  }
}

}  // namespace

size_t recur_stack_smem(int R, int cpt, int nthreads, bool fp16, int bw) {
  const int rmax = recur_dense_rmax(R);
  return (size_t)cpt * R * nthreads * (fp16 ? 8 : 16) +
         (size_t)2 * (nthreads / 32) * rmax * bw * sizeof(float);
}

cudaError_t launch_recur_stack(const StackArgs& a, int bw, cudaStream_t s) {
  void* args[] = {const_cast<StackArgs*>(&a)};
  const int rmax = recur_dense_rmax(a.c.R);
  const int g = a.c.n_cta * a.L, nt = a.c.nthreads;
  const size_t sm = a.c.smem;
  const int cpt = a.cpt;
#define PRNN_STACK_CASE(F, RM, BW_, CP) \
  if (a.wfp16 == F && rmax == RM && bw == BW_ && cpt == CP) \
    return coop_launch(recur_stack_kernel<F, RM, BW_, CP>, g, nt, sm, s, args);
#define PRNN_STACK_CPT(F, RM, BW_) \
  PRNN_STACK_CASE(F, RM, BW_, 1) PRNN_STACK_CASE(F, RM, BW_, 2) \
  PRNN_STACK_CASE(F, RM, BW_, 3) PRNN_STACK_CASE(F, RM, BW_, 4)
#define PRNN_STACK_ROW(F, RM) \
  PRNN_STACK_CPT(F, RM, 1) PRNN_STACK_CPT(F, RM, 2) PRNN_STACK_CPT(F, RM, 4)
  PRNN_STACK_ROW(1, 8) PRNN_STACK_ROW(1, 16) PRNN_STACK_ROW(1, 32)
  PRNN_STACK_ROW(0, 8) PRNN_STACK_ROW(0, 16) PRNN_STACK_ROW(0, 32)
#undef PRNN_STACK_ROW
#undef PRNN_STACK_CPT
#undef PRNN_STACK_CASE
  return cudaErrorInvalidValue;
}

}  // namespace prnn
