// persistent_dense_wide.cu -- the persistent dense recurrence for wide
// batches: fp16 weights, 16 or more batch columns.
//
// The B <= 4 kernel (persistent_dense.cu) gives every thread all of the CTA's
// rows for a few 4-column chunks and one batch pass of up to 4 columns: at
// B = 32 that is 8 passes per step, each with its own poll of h and CTA
// barrier, and every weight is converted from fp16 for 4 columns only.  Here
// a step is a few passes of 8 batch columns, each a small matrix product
//     acc[R rows][8 columns] = W[R][H] . h_{t-1}[H][8 columns],
// register-tiled: thread (q, s) owns rows 4q .. 4q+3 and all 8 columns of
// the pass (32 accumulators) for the 4-column chunks s, s+S, s+2S, ... of the
// K dimension, so each weight it converts feeds 8 columns and each h value 4
// rows: 128 FMAs per chunk from 2 + 8 shared 128-bit loads and 16 fp16
// conversions.  R = 8 rows per CTA where H / 8 CTAs fit on the device, else
// 16; R / 4 x S threads.  The S partial sums of each output are reduced by a
// warp reduce-scatter and one exchange through shared memory.  The CTA's
// fp16 weights stay in shared memory for the whole sequence.
//
// h_{t-1} for a pass (8 batch rows of H floats, contiguous in y) is brought
// into shared memory by one bulk TMA copy (cp.async.bulk, mbarrier
// complete_tx), issued one pass ahead into a second buffer, so the copy of
// pass p+1 overlaps the arithmetic of pass p.  A prefetch can run ahead of a
// slow producer and bring the "not yet written" pattern.  With three or more
// passes a step the copy is issued long after its rows were published and is
// nearly always clean: the arithmetic runs at once, and a NaN in any thread's
// accumulators sends the whole CTA back to scan its staged rows, re-poll the
// stale float4s with relaxed loads (bounded, all of them together) and
// compute the pass again.  With two passes the copy is nearly always stale,
// so the scan and re-poll come before the arithmetic.  Results are published
// in y exactly as by the other persistent kernels (flag in the data).
#include "persistent_common.cuh"
#include "tc_common.cuh"

namespace prnn {

using namespace pk;

namespace {

constexpr int kWidePass = 8;     // batch columns per pass
constexpr int kWideMaxBufs = 3;  // h buffers: prefetch distance up to 2 passes
// Deepest prefetch the plan chooses.  Two passes ahead measured slower than
// one at every size tried (H = 640 .. 2304, B = 16, 32): a copy that far
// ahead of the slowest producer comes back stale and the pass is computed
// twice.
constexpr int kWideMaxDepth = 1;
// A copy issued at least this many passes after the CTA's own publish of the
// rows it reads is assumed clean: stale words are caught by the NaN check
// after the arithmetic (and the pass recomputed).  Closer copies are scanned
// and re-polled before the arithmetic.  Measured: with 4 passes a step
// (gap 3) checking after the arithmetic is 15 % faster than scanning first;
// with 2 (gap 1) nearly every copy is stale and scanning first wins.
constexpr int kWideCleanGap = 2;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

// Bounded wait for a bulk copy's mbarrier phase.  The timer is read only
// once the phase is not complete at the first test.
__device__ __forceinline__ bool wait_copy(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  return tc::mbar_wait(bar, parity, global_ns() + limit_ns);
}

// Re-poll the stale float4s among the n4 staged at hs (copied from src):
// each thread checks slots tid, tid + NT, ... and re-issues, together, the
// relaxed loads of up to 4 stale slots per round trip.  False if the wait
// gave up.  A thread that wrote into hs fences its writes against the async
// proxy, so a later bulk copy into the same buffer is ordered after them
// (with the CTA barrier that follows every call); the issuing thread fences
// again before each copy.
__device__ __forceinline__ bool fix_stale(const float* src, int n4, float* hs, Waiter& w) {
  const int NT = blockDim.x, tid = threadIdx.x;
  float4* h4 = reinterpret_cast<float4*>(hs);
  const float4* s4 = reinterpret_cast<const float4*>(src);
  bool wrote = false;
  bool ok = true;
  for (int base = tid; base < n4; base += 4 * NT) {
    float4 v[4];
    unsigned stale = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * NT;
      if (i < n4) {
        v[u] = h4[i];
        if (!ready4(v[u])) stale |= 1u << u;
      }
    }
    if (stale == 0u) continue;
    wrote = true;
    uint32_t spins = 0, round = 0;
    for (;;) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((stale >> u) & 1u) v[u] = ld_relaxed_f4(reinterpret_cast<const float*>(s4 + base + u * NT));
      unsigned still = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (((stale >> u) & 1u) && !ready4(v[u])) still |= 1u << u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (((stale & ~still) >> u) & 1u) h4[base + u * NT] = v[u];
      stale = still;
      if (stale == 0u) break;
      if (!w.still_ok(spins)) {
        ok = false;
        break;
      }
      w.pause(round);
    }
    if (!ok) break;
  }
  if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  return ok;
}

// 4-row x 4-column fp16 block -> fp32: lo holds rows 0, 1 and hi rows 2, 3
// (4 consecutive columns each)
__device__ __forceinline__ void unpack_rows(const uint4& lo, const uint4& hi, float (&w)[4][4]) {
  const uint32_t u[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u[2 * i]));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u[2 * i + 1]));
    w[i][0] = a.x;
    w[i][1] = a.y;
    w[i][2] = b.x;
    w[i][3] = b.y;
  }
}

// S threads per 4-row group (a multiple of 32 dividing H / 4), R rows per CTA.
template <int S, int R>
__global__ void __launch_bounds__(R / 4 * S, 1) recur_dense_wide_kernel(const DenseWideArgs a) {
  constexpr int QG = R / 4;        // 4-row groups
  constexpr int WPQ = S / 32;      // warps per group
  constexpr int NOUT = R * kWidePass;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kWideMaxBufs];
  __shared__ int s_abort;
  const RecurCommon& c = a.c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x;
  const int H = c.H, B = c.B;
  const Place pl = place_of(c);
  const int nch = H >> 2;
  const int C = nch / S;
  const int q = warp / WPQ;
  const int s = (warp % WPQ) * 32 + lane;
  const int NB = a.depth + 1;  // h buffers
  // shared memory: Wlo[QG][nch], Whi[QG][nch] (uint4), NB h buffers of
  // kWidePass rows of H floats, two reduction buffers [warps][32]
  uint4* Wlo = reinterpret_cast<uint4*>(smem);
  uint4* Whi = Wlo + QG * nch;
  float* hbuf = reinterpret_cast<float*>(Whi + QG * nch);
  float* red = hbuf + (size_t)NB * kWidePass * H;

  {  // this CTA's weights, loaded once for the whole sequence
    const int n16 = 2 * QG * nch;
    const uint4* src = reinterpret_cast<const uint4*>(a.Wpk) + (size_t)pl.lc * n16;
    for (int i = tid; i < n16; i += blockDim.x) Wlo[i] = __ldg(src + i);
  }
  if (tid == 0) {
    for (int i = 0; i < NB; ++i) tc::mbar_init(&full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  __syncthreads();

  const int bl = pl.b_hi - pl.b_lo;
  const int P = (bl + kWidePass - 1) / kWidePass;  // passes per step
  const int nseq = bl > 0 ? c.T * P : 0;
  // prefetch distance: two passes only when a step has three or more, so a
  // copy that crosses into the next step starts a pass after the CTA's own
  // publish of the columns it reads
  const int D = (P >= 3) ? a.depth : 1;
  auto pass_cols = [&](int seq, int* bs) {  // first column and width of pass seq
    const int p = seq % P;
    *bs = pl.b_lo + p * kWidePass;
    return min(kWidePass, pl.b_hi - *bs);
  };
  auto issue = [&](int seq) {  // issuer: bulk copy of pass seq into buffer seq % NB
    const int t = seq / P;
    int bs;
    const int nb = pass_cols(seq, &bs);
    // source rows: h0 (or zeros) at t = 0, else y[t-1]
    const float* base = (t == 0) ? a.h0_rows : c.y + (size_t)(t - 1) * B * H;
    const int buf = seq % NB;
    const uint32_t bytes = (uint32_t)nb * (uint32_t)H * 4u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::mbar_arrive_expect_tx(&full[buf], bytes);
    bulk_g2s(tc::smem_u32(hbuf + (size_t)buf * kWidePass * H), base + (size_t)bs * H, bytes,
             &full[buf]);
  };
  // the output this thread finalizes (tid < R x 8): row tid / 8 of the CTA,
  // column tid % 8 of the pass; its projection value is loaded a pass ahead
  const int orow = pl.row0 + (tid >> 3), oc = tid & 7;
  auto load_p = [&](int seq) {
    int bs;
    const int nb = pass_cols(seq, &bs);
    const bool outs = tid < NOUT && oc < nb && orow < H;
    return outs ? ld_nc_pinned(c.P + ((size_t)(seq / P) * B + bs + oc) * H + orow) : 0.f;
  };

  // The copies are issued by the last thread.  When the CTA has more threads
  // than outputs its warp has no output work after a pass's barrier, so it
  // reaches the next pass's copy wait first and starts the following copy
  // earlier than an output thread would (measured at H = 1792, B = 32:
  // 9.8 against 11.4 us per step with thread 0 issuing).
  const bool issuer = tid == (int)blockDim.x - 1;
  int issued = -1;  // issuer: last pass whose copy was issued
  if (issuer)
    for (int k = 0; k < D && k < nseq; ++k) issue(issued = k);
  float pv_next = nseq > 0 ? load_p(0) : 0.f;
  Waiter w;
  w.status = c.status;
  w.timeout_ns = c.timeout_ns;
  w.backoff = c.poll_backoff;
  const uint64_t copy_limit_ns = (uint64_t)c.timeout_ns;
  for (int seq = 0; seq < nseq; ++seq) {
    const int t = seq / P, p = seq - t * P;
    int bs;
    const int nb = pass_cols(seq, &bs);
    const int buf = seq % NB;
    if (p == 0) w.new_step();
    const float pv = pv_next;
    if (seq + 1 < nseq) pv_next = load_p(seq + 1);
    // wait for this pass's copy; then start the one D passes ahead (its
    // buffer was last read in pass seq + D - NB <= seq - 1, which every
    // thread has finished: the CTA barrier at the end of that pass)
    if (!wait_copy(&full[buf], (uint32_t)(seq / NB) & 1u, copy_limit_ns)) {
      report_timeout(c.status, t, cta);
      s_abort = 1;
    }
    if (issuer && seq + D < nseq && !s_abort) issue(issued = seq + D);
    float* hs = hbuf + (size_t)buf * kWidePass * H;
    float* rb = red + (size_t)(seq & 1) * QG * WPQ * 32;
    // the copy of pass seq was issued P - D passes after this CTA published
    // the rows it reads: when that gap is short, scan before the arithmetic
    if (t > 0 && P - D < kWideCleanGap) {
      if (!fix_stale(c.y + (size_t)(t - 1) * B * H + (size_t)bs * H, nb * H / 4, hs, w)) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
    }
    const float4* h4 = reinterpret_cast<const float4*>(hs);
    for (int attempt = 0;; ++attempt) {
      // rows past nb of the buffer hold stale words (finite or the NaN
      // pattern): their columns are never published
      float acc[4][kWidePass];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int b = 0; b < kWidePass; ++b) acc[i][b] = 0.f;
      for (int j = 0; j < C; ++j) {
        const int ch = s + S * j;
        float wr[4][4];
        unpack_rows(Wlo[q * nch + ch], Whi[q * nch + ch], wr);
#pragma unroll
        for (int b = 0; b < kWidePass; ++b) {
          const float4 hv = h4[b * nch + ch];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float sum = acc[i][b];
            sum = fmaf(wr[i][0], hv.x, sum);
            sum = fmaf(wr[i][1], hv.y, sum);
            sum = fmaf(wr[i][2], hv.z, sum);
            sum = fmaf(wr[i][3], hv.w, sum);
            acc[i][b] = sum;
          }
        }
      }
      // h is a ReLU output and the weights are finite, so a NaN sum means the
      // copy ran ahead of a producer and brought the "not yet written" pattern
      bool bad = false;
#pragma unroll
      for (int b = 0; b < kWidePass; ++b)
        if (b < nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) bad |= acc[i][b] != acc[i][b];
      // reduce the S partial sums of each of the group's 32 outputs: lane L
      // of each warp ends with output L (row 4q + L / 8, column L % 8)
      float v32[32];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int b = 0; b < kWidePass; ++b) v32[i * kWidePass + b] = acc[i][b];
      warp_reduce_scatter<32>(v32, lane);
      rb[warp * 32 + lane] = v32[0];
      const bool retry = __syncthreads_or(bad) && attempt == 0 && t > 0 && !s_abort;
      if (!retry) break;
      // once per stale pass: re-poll, all at once, the float4s of the staged
      // rows that still hold the pattern, then compute the pass again
      if (!fix_stale(c.y + (size_t)(t - 1) * B * H + (size_t)bs * H, nb * H / 4, hs, w)) {
        report_timeout(c.status, t, cta);
        s_abort = 1;
      }
      __syncthreads();
    }
    if (s_abort) {
      // let the copies in flight land before the CTA leaves
      if (issuer)
        for (int k = seq + 1; k <= issued; ++k)
          wait_copy(&full[k % NB], (uint32_t)(k / NB) & 1u, copy_limit_ns);
      return;
    }
    if (tid < NOUT && oc < nb && orow < H) {
      const int r = tid >> 3, oq = r >> 2, L = (r & 3) * kWidePass + oc;
      float sum = pv;
#pragma unroll
      for (int k = 0; k < WPQ; ++k) sum += rb[(oq * WPQ + k) * 32 + L];
      if (!(cta == c.drop_cta && t == c.drop_step)) {
        const float out = relu(sum);
        const size_t o = ((size_t)t * B + bs + oc) * H + orow;
        st_relaxed_f(c.y + o, out);
        if (c.y_mirror) c.y_mirror[o] = out;
      }
    }
  }
}

template <int R>
cudaError_t launch_rows(const DenseWideArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<DenseWideArgs*>(&a)};
  const int g = a.c.n_cta;
  const size_t sm = a.c.smem;
  if (a.S == 96) return coop_launch(recur_dense_wide_kernel<96, R>, g, R / 4 * 96, sm, s, args);
  if (a.S == 64) return coop_launch(recur_dense_wide_kernel<64, R>, g, R / 4 * 64, sm, s, args);
  if (a.S == 32) return coop_launch(recur_dense_wide_kernel<32, R>, g, R / 4 * 32, sm, s, args);
  return cudaErrorInvalidValue;
}

}  // namespace

bool recur_dense_wide_plan(int H, int sm_count, size_t smem_optin, int* R_out, int* S_out,
                           int* depth_out, size_t* smem_out) {
  if (H % 128 != 0) return false;
  const int nch = H / 4;
  const int S = (nch % 96 == 0) ? 96 : ((nch % 64 == 0) ? 64 : 32);
  int R = 0;
  if (H / 8 <= sm_count) R = 8;
  else if (H / 16 <= sm_count) R = 16;
  if (R == 0) return false;
  const int warps = R / 4 * S / 32;
  auto bytes = [&](int nbuf) {
    return (size_t)2 * (R / 4) * nch * 16 + (size_t)nbuf * kWidePass * H * 4 +
           (size_t)2 * warps * 32 * 4;
  };
  int depth = kWideMaxDepth;
  while (depth >= 1 && bytes(depth + 1) > smem_optin) --depth;
  if (depth < 1) return false;
  *R_out = R;
  *S_out = S;
  *depth_out = depth;
  *smem_out = bytes(depth + 1);
  return true;
}

cudaError_t launch_recur_dense_wide(const DenseWideArgs& a, cudaStream_t s) {
  if (a.c.H % 128 != 0 || (a.c.H / 4) % a.S != 0 || a.depth < 1 || a.depth >= kWideMaxBufs)
    return cudaErrorInvalidValue;
  if (a.c.R == 8) return launch_rows<8>(a, s);
  if (a.c.R == 16) return launch_rows<16>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace prnn
