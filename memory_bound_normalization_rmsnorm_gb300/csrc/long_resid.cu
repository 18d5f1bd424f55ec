// long_resid.cu -- instantiations of the long-row kernels (long_kernel.cuh)
// with the fused residual add: the forward reads x and r and writes h and y,
// the backward reads h, dy and dh.
#include "long_kernel.cuh"

namespace gbn {

namespace {

template <int MODE, int K, bool CLUSTER>
const void *pick_long(bool bwd, bool e) {
  if (bwd)
    return e ? reinterpret_cast<const void *>(&norm_bwd_long_kernel<MODE, K, CLUSTER, true, true>)
             : reinterpret_cast<const void *>(&norm_bwd_long_kernel<MODE, K, CLUSTER, false, true>);
  return e ? reinterpret_cast<const void *>(&norm_fwd_long_kernel<MODE, K, CLUSTER, true, true>)
           : reinterpret_cast<const void *>(&norm_fwd_long_kernel<MODE, K, CLUSTER, false, true>);
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

const void *long_resid_kernel_ptr(int mode, int K, bool cluster, bool exact, bool bwd) {
  return cluster ? pick_mode<true>(mode, K, bwd, exact) : pick_mode<false>(mode, K, bwd, exact);
}

}  // namespace gbn
