// persistent_sparse_placed.cu -- the persistent sparse kernels that stage
// h_{t-1} in each CTA's bank-balancing order (see the packer), in a
// translation unit of their own so that they compile in parallel with the
// column-order kernels.
#include "persistent_sparse.cuh"

namespace prnn {

cudaError_t launch_recur_sparse_placed(const SparseRecurArgs& a, cudaStream_t s) {
  return launch_recur_sparse_depth<true, false, kSparseThreads>(a, s);
}

}  // namespace prnn
