// persistent_sparse_trace.cu -- the persistent sparse kernels with the phase
// trace compiled in (column-order staging only), in a translation unit of
// their own: the default kernels carry none of the trace's code or registers.
#include "persistent_sparse.cuh"

namespace prnn {

cudaError_t launch_recur_sparse_trace(const SparseRecurArgs& a, cudaStream_t s) {
  return launch_recur_sparse_impl<false, true>(a, s);
}

cudaError_t launch_recur_sparse_trace_regw(const SparseRecurArgs& a, cudaStream_t s) {
  return launch_recur_sparse_impl<false, true, kRegWThreads>(a, s);
}

}  // namespace prnn
