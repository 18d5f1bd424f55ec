// long_fp8.cu -- E4M3-output instantiations of the long-row forward kernel
// (long_kernel.cuh): MX block or per-row scaling, with or without a
// cluster; plain or fused-residual.  8 chunks per thread (the long-row
// planner's choice for the forward).
#include "long_kernel.cuh"

namespace gbn {

namespace {

template <int MODE, int K, bool CLUSTER, bool RESID, int OUT>
const void *pick_exact(bool e) {
  return e ? reinterpret_cast<const void *>(
                 &norm_fwd_long_kernel<MODE, K, CLUSTER, true, RESID, OUT>)
           : reinterpret_cast<const void *>(
                 &norm_fwd_long_kernel<MODE, K, CLUSTER, false, RESID, OUT>);
}

template <int MODE, int K>
const void *pick(bool cluster, bool e, bool r, int out) {
  if (out == kOutFp8Mx) {
    if (cluster) return r ? pick_exact<MODE, K, true, true, kOutFp8Mx>(e)
                          : pick_exact<MODE, K, true, false, kOutFp8Mx>(e);
    return r ? pick_exact<MODE, K, false, true, kOutFp8Mx>(e)
             : pick_exact<MODE, K, false, false, kOutFp8Mx>(e);
  }
  if (out == kOutFp8Row) {
    if (cluster) return r ? pick_exact<MODE, K, true, true, kOutFp8Row>(e)
                          : pick_exact<MODE, K, true, false, kOutFp8Row>(e);
    return r ? pick_exact<MODE, K, false, true, kOutFp8Row>(e)
             : pick_exact<MODE, K, false, false, kOutFp8Row>(e);
  }
  return nullptr;
}

}  // namespace

const void *long_fp8_kernel_ptr(int mode, int K, bool cluster, bool exact, bool resid, int out) {
  if (K != 8) return nullptr;
  return mode == kRMS ? pick<kRMS, 8>(cluster, exact, resid, out)
                      : pick<kLayer, 8>(cluster, exact, resid, out);
}

}  // namespace gbn
