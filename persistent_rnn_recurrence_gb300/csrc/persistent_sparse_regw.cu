// persistent_sparse_regw.cu -- the register-weight build of the persistent
// sparse kernel (column-order staging): launch bound kRegWThreads (384)
// threads instead of 512, so each thread may use up to 168 registers and
// holds its first kRegQWide (6) uint4 weight groups -- 24 entries, all of a
// row's entries at the 10 % layer of 1792 units -- in registers.  Measured on
// GB300 at that layer: gathers 424 -> 341 ns per step, step 1.72 -> 1.64 us.
// In a translation unit of its own so that it compiles in parallel.
#include "persistent_sparse.cuh"

namespace prnn {

cudaError_t launch_recur_sparse_regw(const SparseRecurArgs& a, cudaStream_t s) {
  return launch_recur_sparse_depth<false, false, kRegWThreads>(a, s);
}

}  // namespace prnn
