// long.cu -- instantiations of the long-row kernels (long_kernel.cuh)
// without the fused residual add.
#include "long_kernel.cuh"

namespace gbn {

namespace {

template <int MODE, int K, bool CLUSTER>
const void *pick_long(bool bwd, bool e) {
  if (bwd)
    return e ? reinterpret_cast<const void *>(&norm_bwd_long_kernel<MODE, K, CLUSTER, true, false>)
             : reinterpret_cast<const void *>(&norm_bwd_long_kernel<MODE, K, CLUSTER, false, false>);
  return e ? reinterpret_cast<const void *>(&norm_fwd_long_kernel<MODE, K, CLUSTER, true, false>)
           : reinterpret_cast<const void *>(&norm_fwd_long_kernel<MODE, K, CLUSTER, false, false>);
}

template <int MODE, bool CLUSTER>
const void *pick_long_k(int K, bool bwd, bool e) {
  switch (K) {
    case 4: return pick_long<MODE, 4, CLUSTER>(bwd, e);
    case 8: return pick_long<MODE, 8, CLUSTER>(bwd, e);
    default: return nullptr;
  }
}

template <bool CLUSTER>
const void *pick_mode(int mode, int K, bool bwd, bool e) {
  return mode == kRMS ? pick_long_k<kRMS, CLUSTER>(K, bwd, e) : pick_long_k<kLayer, CLUSTER>(K, bwd, e);
}

}  // namespace

const void *long_kernel_ptr(int mode, int K, bool cluster, bool exact, bool bwd, bool resid) {
  if (resid) return long_resid_kernel_ptr(mode, K, cluster, exact, bwd);
  return cluster ? pick_mode<true>(mode, K, bwd, exact) : pick_mode<false>(mode, K, bwd, exact);
}

}  // namespace gbn
