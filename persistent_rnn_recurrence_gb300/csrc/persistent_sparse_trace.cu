// persistent_sparse_trace.cu -- the persistent sparse kernels with the phase
// trace compiled in (column-order staging only, each staging depth), in a
// translation unit of their own: the default kernels carry none of the
// trace's code or registers.
#include "persistent_sparse.cuh"

namespace prnn {

cudaError_t launch_recur_sparse_trace(const SparseRecurArgs& a, cudaStream_t s) {
  return launch_recur_sparse_depth<false, true, kSparseThreads>(a, s);
}

}  // namespace prnn
