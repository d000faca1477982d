// persistent.cu -- the persistent recurrent kernels.
//
// One cooperative launch runs all T steps of h_t = ReLU(P_t + Wh h_{t-1})
// (P_t = Wx x_t + b comes from the projection kernel).  Each CTA owns a block
// of R consecutive rows of Wh and loads them into shared memory / registers
// once, so the weights stay on chip for the whole sequence instead of being
// re-read every step (persistent-rnn page, "What This Project Does"; "Sparse
// Persistent RNNs: Squeezing Large Recurrent Networks On-Chip").
//
// Step exchange: h_t is published by storing it into y[t] (pre-filled with a
// NaN sentinel); consumers poll y[t-1] with relaxed gpu-scope loads until no
// word is the sentinel.  The data word is its own "ready" flag, so there is no
// grid barrier between steps (the Lamport-timestamp row of the sparse
// persistent RNN ablation).  A grid-barrier mode is kept for that ablation.
//
// Every wait is bounded (globaltimer deadline); on expiry the kernel records
// a status word and every CTA leaves its time loop.
#include <cstdio>

#include "device_common.cuh"
#include "prnn_internal.h"

namespace prnn {

namespace {

constexpr int kDenseThreads = 256;  // upper bound of blockDim for the dense kernel
constexpr int kSparseThreads = 512;
constexpr int kCptMax = 4;          // 4-column chunks per thread (H <= 4096 at 256 threads)
constexpr int kRegQ = 4;            // sparse: uint4 weight groups held in registers (BV < 8)

__device__ __forceinline__ unsigned ld_acquire_u(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
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

__device__ __forceinline__ void load_w4(const unsigned char* p, bool f16, float& w0,
                                        float& w1, float& w2, float& w3) {
  if (f16) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const __half2 a = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&u.y);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    w0 = fa.x; w1 = fa.y; w2 = fb.x; w3 = fb.y;
  } else {
    const float4 f = *reinterpret_cast<const float4*>(p);
    w0 = f.x; w1 = f.y; w2 = f.z; w3 = f.w;
  }
}

// ---------------------------------------------------------------------------
// Dense kernel.  Thread i owns the 4-column chunks i, i+NT, ... (all R rows of
// the CTA for those columns), so each h value it loads is reused for R rows
// straight from registers.  Weights: smem, [chunk slot j][row r][thread] of
// 4-weight vectors, so a warp's weight loads are consecutive 8/16-byte words
// (128-bit-friendly, bank-conflict-free).  Partial sums are reduced across the
// warp by a reduce-scatter and across warps through smem.
// ---------------------------------------------------------------------------
template <bool F16, int RMAX>
__global__ void __launch_bounds__(kDenseThreads, 1) recur_dense_kernel(const DenseRecurArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NT = blockDim.x, nwarps = NT >> 5;
  const int cta = blockIdx.x;
  const int H = c.H, B = c.B, R = c.R;
  const int row0 = cta * R;
  const int Rc = min(R, H - row0);
  const int nchunks = H >> 2;
  const int cpt = a.cpt;
  constexpr int VB = F16 ? 8 : 16;
  constexpr int V = RMAX * 4;

  unsigned char* Ws = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)cpt * R * NT * VB);

  {  // this CTA's weights, loaded once for the whole sequence
    const size_t bytes = (size_t)cpt * R * NT * VB;
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const unsigned char*>(a.Wpk) + (size_t)cta * bytes);
    uint4* dst = reinterpret_cast<uint4*>(Ws);
    for (size_t i = tid; i < bytes / 16; i += NT) dst[i] = __ldg(src + i);
  }
  if (tid == 0) s_abort = 0;
  __syncthreads();

  Waiter w;
  w.status = c.status;
  int seq = 0;
  for (int t = 0; t < c.T; ++t) {
    const float* hprev = (t == 0) ? c.h0 : c.y + (size_t)(t - 1) * B * H;
    const float* Pt = c.P + (size_t)t * B * H;
    float* yt = c.y + (size_t)t * B * H;
    w.deadline = global_ns() + (uint64_t)c.timeout_ns;
    for (int b0 = 0; b0 < B; b0 += 4, ++seq) {
      const int nb = min(4, B - b0);
      // P for the output this thread finalizes (index tid = r*4 + b)
      float pv = 0.f;
      int orow = -1, ob = -1;
      if (tid < RMAX * 4) {
        const int r = tid >> 2, bb = tid & 3;
        if (r < Rc && bb < nb) {
          orow = row0 + r;
          ob = b0 + bb;
          pv = __ldg(Pt + (size_t)ob * H + orow);
        }
      }
      // issue every load of h_{t-1} this thread needs, then wait on them
      float4 hv[kCptMax][4];
#pragma unroll
      for (int j = 0; j < kCptMax; ++j) {
        const int ch = tid + j * NT;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          hv[j][bb] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j < cpt && ch < nchunks && bb < nb && hprev != nullptr) {
            const float* p = hprev + (size_t)(b0 + bb) * H + ch * 4;
            hv[j][bb] = (t == 0) ? __ldg(reinterpret_cast<const float4*>(p)) : ld_relaxed_f4(p);
          }
        }
      }
      bool ok = true;
      float acc[RMAX][4];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) acc[r][bb] = 0.f;
#pragma unroll
      for (int j = 0; j < kCptMax; ++j) {
        const int ch = tid + j * NT;
        if (j < cpt && ch < nchunks) {
          if (t > 0) {
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
              if (bb < nb && ok)
                ok = poll_f4(hprev + (size_t)(b0 + bb) * H + ch * 4, hv[j][bb], w);
          }
          const unsigned char* wp = Ws + ((size_t)j * R * NT + tid) * VB;
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
              float w0, w1, w2, w3;
              load_w4(wp + (size_t)r * NT * VB, F16, w0, w1, w2, w3);
#pragma unroll
              for (int bb = 0; bb < 4; ++bb) {
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
      }
      float v[V];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) v[r * 4 + bb] = acc[r][bb];
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
        if (!(cta == c.drop_cta && t == c.drop_step))
          st_relaxed_f(yt + (size_t)ob * H + orow, relu(s));
      }
    }
    if (c.sync_mode == 1) {
      grid_barrier(c, t, w, &s_abort);
      if (s_abort) return;
    }
  }
}

// ---------------------------------------------------------------------------
// Stage h_{t-1}[b][:] for one batch group into smem as hs[col][BG] (BG = 4*BV
// batch columns per column; float4 groups XOR-swizzled by col so gathers of
// different columns spread over banks).  Items are (4-column chunk, batch
// quad); a thread issues the loads of up to 4 items before waiting on any.
// Returns false if a wait gave up.
// ---------------------------------------------------------------------------
template <int BV>
__device__ __forceinline__ bool stage_h(const float* hprev, bool poll, int H, int B, int g,
                                        float* hs, Waiter& w) {
  constexpr int BG = 4 * BV;
  constexpr int U = (BV >= 8) ? 2 : 4;  // items in flight per thread
  const int NT = blockDim.x, tid = threadIdx.x;
  const int nc4 = H >> 2;
  const int nitems = nc4 * BV;
  bool ok = true;
  for (int base = tid; base < nitems; base += U * NT) {
    float4 v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int id = base + u * NT;
      const int c4 = id % nc4, bq = id / nc4;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        v[u][bb] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int b = g * BG + bq * 4 + bb;
        if (id < nitems && b < B && hprev != nullptr) {
          const float* p = hprev + (size_t)b * H + c4 * 4;
          v[u][bb] = poll ? ld_relaxed_f4(p) : __ldg(reinterpret_cast<const float4*>(p));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int id = base + u * NT;
      if (id >= nitems) continue;
      const int c4 = id % nc4, bq = id / nc4;
      if (poll) {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int b = g * BG + bq * 4 + bb;
          if (b < B && ok) ok = poll_f4(hprev + (size_t)b * H + c4 * 4, v[u][bb], w);
        }
      }
      const float4 o0 = make_float4(v[u][0].x, v[u][1].x, v[u][2].x, v[u][3].x);
      const float4 o1 = make_float4(v[u][0].y, v[u][1].y, v[u][2].y, v[u][3].y);
      const float4 o2 = make_float4(v[u][0].z, v[u][1].z, v[u][2].z, v[u][3].z);
      const float4 o3 = make_float4(v[u][0].w, v[u][1].w, v[u][2].w, v[u][3].w);
      const int col = c4 * 4;
      *reinterpret_cast<float4*>(hs + (size_t)(col + 0) * BG + ((bq ^ ((col + 0) & (BV - 1))) << 2)) = o0;
      *reinterpret_cast<float4*>(hs + (size_t)(col + 1) * BG + ((bq ^ ((col + 1) & (BV - 1))) << 2)) = o1;
      *reinterpret_cast<float4*>(hs + (size_t)(col + 2) * BG + ((bq ^ ((col + 2) & (BV - 1))) << 2)) = o2;
      *reinterpret_cast<float4*>(hs + (size_t)(col + 3) * BG + ((bq ^ ((col + 3) & (BV - 1))) << 2)) = o3;
    }
  }
  return ok;
}

// ---------------------------------------------------------------------------
// Sparse row-balanced kernel.  Thread (r, s) = (tid / TPR, tid % TPR) owns
// ept = kp / TPR entries of row r, packed 4 to a uint4 (wide loads).  Entry =
// fp16 value | column << 16; padding entries have value 0.  The first kRegQ
// uint4 groups live in registers, the rest in smem.  h_{t-1} is staged in smem
// (double-buffered when it fits) and gathered per entry.
// ---------------------------------------------------------------------------
template <int TPR, int BV>
__global__ void __launch_bounds__(kSparseThreads, 1) recur_sparse_kernel(const SparseRecurArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  constexpr int BG = 4 * BV;
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, lane = tid & 31;
  const int NT = blockDim.x;
  const int cta = blockIdx.x;
  const int H = c.H, B = c.B, R = c.R;
  const int row0 = cta * R;
  const int Rc = min(R, H - row0);
  const int q4 = a.ept >> 2;
  const int nbuf = a.dbuf ? 2 : 1;

  uint4* Ws = reinterpret_cast<uint4*>(smem);
  float* hs0 = reinterpret_cast<float*>(Ws + (size_t)R * q4 * TPR);

  {
    const size_t n16 = (size_t)R * q4 * TPR;
    const uint4* src = reinterpret_cast<const uint4*>(a.Wpk) + (size_t)cta * n16;
    for (size_t i = tid; i < n16; i += NT) Ws[i] = __ldg(src + i);
  }
  if (tid == 0) s_abort = 0;
  __syncthreads();

  const int r = tid / TPR, s = tid % TPR;
  const bool has_row = r < Rc;
  constexpr int REGQ = (BV >= 8) ? 1 : kRegQ;
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
  int seq = 0;
  for (int t = 0; t < c.T; ++t) {
    const float* hprev = (t == 0) ? c.h0 : c.y + (size_t)(t - 1) * B * H;
    const float* Pt = c.P + (size_t)t * B * H;
    float* yt = c.y + (size_t)t * B * H;
    w.deadline = global_ns() + (uint64_t)c.timeout_ns;
    for (int g = 0; g * BG < B; ++g, ++seq) {
      const int nbg = min(BG, B - g * BG);
      float* hs = hs0 + (size_t)((nbuf == 2) ? (seq & 1) : 0) * H * BG;
      // P for this lane's outputs, fetched before the wait
      float pv[NOUT];
      bool owns = false;
#pragma unroll
      for (int i = 0; i < NOUT; ++i) {
        pv[i] = 0.f;
        const int idx = (BG >= TPR) ? gl * NOUT + i : gl / REP;
        const bool mine = (gl % REP) == 0;
        if (has_row && mine && idx < nbg) {
          pv[i] = __ldg(Pt + (size_t)(g * BG + idx) * H + row0 + r);
          owns = true;
        }
      }
      const bool ok = stage_h<BV>(hprev, t > 0, H, B, g, hs, w);
      if (!ok) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;

      float acc[BG];
#pragma unroll
      for (int i = 0; i < BG; ++i) acc[i] = 0.f;
      auto consume = [&](const uint4 e) {
        const uint32_t ws[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float val = __half2float(__ushort_as_half((unsigned short)(ws[q] & 0xffffu)));
          const int col = (int)(ws[q] >> 16);
          const float* hc = hs + (size_t)col * BG;
#pragma unroll
          for (int bq = 0; bq < BV; ++bq) {
            const float4 h4 = *reinterpret_cast<const float4*>(hc + ((bq ^ (col & (BV - 1))) << 2));
            acc[bq * 4 + 0] = fmaf(val, h4.x, acc[bq * 4 + 0]);
            acc[bq * 4 + 1] = fmaf(val, h4.y, acc[bq * 4 + 1]);
            acc[bq * 4 + 2] = fmaf(val, h4.z, acc[bq * 4 + 2]);
            acc[bq * 4 + 3] = fmaf(val, h4.w, acc[bq * 4 + 3]);
          }
        }
      };
      if (has_row) {
#pragma unroll
        for (int i = 0; i < REGQ; ++i)
          if (i < q4) consume(wr[i]);
        for (int i = REGQ; i < q4; ++i) consume(Ws[((size_t)r * q4 + i) * TPR + s]);
      }
      if (TPR > 1) seg_reduce_scatter<BG, TPR>(acc, lane);
      if (owns && !(cta == c.drop_cta && t == c.drop_step)) {
#pragma unroll
        for (int i = 0; i < NOUT; ++i) {
          const int idx = (BG >= TPR) ? gl * NOUT + i : gl / REP;
          if (idx < nbg)
            st_relaxed_f(yt + (size_t)(g * BG + idx) * H + row0 + r, relu(acc[i] + pv[i]));
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
// Sync-floor probe: the sparse kernel's exchange (stage all of h_{t-1}, one
// CTA barrier, publish R rows of h_t) with no arithmetic.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSparseThreads, 1) sync_probe_kernel(const RecurCommon c, int bv) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_abort;
  float* hs = reinterpret_cast<float*>(smem);
  const int tid = threadIdx.x, cta = blockIdx.x;
  const int H = c.H, B = c.B, R = c.R;
  const int row0 = cta * R;
  const int Rc = min(R, H - row0);
  if (tid == 0) s_abort = 0;
  __syncthreads();
  Waiter w;
  w.status = c.status;
  const int BG = 4 * bv;
  for (int t = 0; t < c.T; ++t) {
    const float* hprev = (t == 0) ? nullptr : c.y + (size_t)(t - 1) * B * H;
    float* yt = c.y + (size_t)t * B * H;
    w.deadline = global_ns() + (uint64_t)c.timeout_ns;
    for (int g = 0; g * BG < B; ++g) {
      bool ok = true;
      if (t > 0) {
        switch (bv) {
          case 1: ok = stage_h<1>(hprev, true, H, B, g, hs, w); break;
          case 2: ok = stage_h<2>(hprev, true, H, B, g, hs, w); break;
          case 4: ok = stage_h<4>(hprev, true, H, B, g, hs, w); break;
          default: ok = stage_h<8>(hprev, true, H, B, g, hs, w); break;
        }
      }
      if (!ok) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) return;
      const int nbg = min(BG, B - g * BG);
      for (int i = tid; i < Rc * nbg; i += blockDim.x) {
        const int rr = i / nbg, bb = i % nbg;
        st_relaxed_f(yt + (size_t)(g * BG + bb) * H + row0 + rr, (float)(t + 1));
      }
      __syncthreads();
    }
  }
}

template <typename K>
cudaError_t coop_launch(K kernel, int grid, int block, size_t smem, cudaStream_t s, void** args) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kernel), dim3(grid),
                                     dim3(block), args, smem, s);
}

}  // namespace

int recur_dense_rmax(int R) {
  if (R <= 4) return 4;
  if (R <= 8) return 8;
  if (R <= 16) return 16;
  if (R <= 32) return 32;
  return 0;
}

size_t recur_dense_smem(int R, int cpt, int nthreads, bool fp16) {
  const int rmax = recur_dense_rmax(R);
  return (size_t)cpt * R * nthreads * (fp16 ? 8 : 16) +
         (size_t)2 * (nthreads / 32) * rmax * 4 * sizeof(float);
}

cudaError_t launch_recur_dense(const DenseRecurArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<DenseRecurArgs*>(&a)};
  const int rmax = recur_dense_rmax(a.c.R);
  const int g = a.c.n_cta, nt = a.c.nthreads;
  const size_t sm = a.c.smem;
#define PRNN_DENSE_CASE(F, RM) \
  if (a.wfp16 == F && rmax == RM) return coop_launch(recur_dense_kernel<F, RM>, g, nt, sm, s, args);
  PRNN_DENSE_CASE(1, 4) PRNN_DENSE_CASE(1, 8) PRNN_DENSE_CASE(1, 16) PRNN_DENSE_CASE(1, 32)
  PRNN_DENSE_CASE(0, 4) PRNN_DENSE_CASE(0, 8) PRNN_DENSE_CASE(0, 16) PRNN_DENSE_CASE(0, 32)
#undef PRNN_DENSE_CASE
  return cudaErrorInvalidValue;
}

size_t recur_sparse_smem(int H, int R, int ept, int tpr, int bgroup, bool dbuf) {
  // weights: R rows x (ept * tpr) packed 4-byte entries; then the h staging buffers
  return (size_t)R * ept * tpr * 4 + (size_t)(dbuf ? 2 : 1) * H * bgroup * sizeof(float);
}

cudaError_t launch_recur_sparse(const SparseRecurArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<SparseRecurArgs*>(&a)};
  const int g = a.c.n_cta, nt = a.c.nthreads;
  const size_t sm = a.c.smem;
  const int bv = a.bgroup / 4;
#define PRNN_SPARSE_CASE(T_, BV_) \
  if (a.tpr == T_ && bv == BV_) return coop_launch(recur_sparse_kernel<T_, BV_>, g, nt, sm, s, args);
#define PRNN_SPARSE_ROW(T_) \
  PRNN_SPARSE_CASE(T_, 1) PRNN_SPARSE_CASE(T_, 2) PRNN_SPARSE_CASE(T_, 4) PRNN_SPARSE_CASE(T_, 8)
  PRNN_SPARSE_ROW(1) PRNN_SPARSE_ROW(2) PRNN_SPARSE_ROW(4) PRNN_SPARSE_ROW(8)
  PRNN_SPARSE_ROW(16) PRNN_SPARSE_ROW(32)
#undef PRNN_SPARSE_ROW
#undef PRNN_SPARSE_CASE
  return cudaErrorInvalidValue;
}

size_t sync_probe_smem(int H, int bgroup) { return (size_t)H * bgroup * sizeof(float); }

cudaError_t launch_sync_probe(const RecurCommon& c, int bgroup, cudaStream_t s) {
  int bv = bgroup / 4;
  void* args[] = {const_cast<RecurCommon*>(&c), &bv};
  return coop_launch(sync_probe_kernel, c.n_cta, c.nthreads, c.smem, s, args);
}

}  // namespace prnn
