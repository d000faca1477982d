// persistent_sparse_trace_regw.cu -- the register-weight build of the
// persistent sparse kernel with the phase trace compiled in (each staging
// depth), in a translation unit of its own so that it compiles in parallel.
#include "persistent_sparse.cuh"

namespace prnn {

cudaError_t launch_recur_sparse_trace_regw(const SparseRecurArgs& a, cudaStream_t s) {
  return launch_recur_sparse_depth<false, true, kRegWThreads>(a, s);
}

}  // namespace prnn
