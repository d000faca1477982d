// persistent_sparse_um.cu -- the column-order persistent sparse kernels
// (launch bound 512 threads) with a staging depth matched to the plan, 2 or 6
// float4 loads in flight per thread instead of 12; in a translation unit of
// their own so that they compile in parallel with the default ones.
#include "persistent_sparse.cuh"

namespace prnn {

cudaError_t launch_recur_sparse_um(const SparseRecurArgs& a, cudaStream_t s) {
  switch (a.umax) {
    case 2: return launch_recur_sparse_impl<false, false, kSparseThreads, 2>(a, s);
    case 6: return launch_recur_sparse_impl<false, false, kSparseThreads, 6>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace prnn
