// persistent_sparse.cu -- the persistent sparse kernels that stage h_{t-1} in
// column order (the kernel itself is in persistent_sparse.cuh), the launcher
// that picks them or the placed ones, and the step-synchronisation floor
// probe.
#include "persistent_sparse.cuh"

namespace prnn {

using namespace pk;

namespace {

// ---------------------------------------------------------------------------
// Sync-floor probe: the sparse kernel's exchange (stage the group's columns of
// h_{t-1}, one CTA barrier, publish R rows of h_t) with no arithmetic.
// ---------------------------------------------------------------------------
template <int UMAX>
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
      if (t > 0) ok = stage_rows<UMAX>(hprev, true, H, bs, nbg, hs, w);
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
  if (a.trace != nullptr) {
    if (a.place != nullptr || a.narrow) return cudaErrorNotSupported;
    return a.regw ? launch_recur_sparse_trace_regw(a, s) : launch_recur_sparse_trace(a, s);
  }
  if (a.place != nullptr) return launch_recur_sparse_placed(a, s);
  if (a.regw) return launch_recur_sparse_regw(a, s);
  if (a.umax != 0) return launch_recur_sparse_um(a, s);
  return launch_recur_sparse_impl<false>(a, s);
}

size_t sync_probe_smem(int H, int bgroup) { return (size_t)H * bgroup * sizeof(float); }

cudaError_t launch_sync_probe(const RecurCommon& c, int bgroup, int umax, cudaStream_t s) {
  int bg = bgroup;
  void* args[] = {const_cast<RecurCommon*>(&c), &bg};
  switch (umax) {
    case 0: return coop_launch(sync_probe_kernel<8>, c.n_cta, c.nthreads, c.smem, s, args);
    case 2: return coop_launch(sync_probe_kernel<2>, c.n_cta, c.nthreads, c.smem, s, args);
    case 6: return coop_launch(sync_probe_kernel<6>, c.n_cta, c.nthreads, c.smem, s, args);
  }
  return cudaErrorInvalidValue;
}

}  // namespace prnn
