// fwd.cu -- bf16-output instantiations of the forward kernel
// (fwd_kernel.cuh): plain and fused-residual, per mode, chunks per thread,
// cluster and exact-split variant.
#include "fwd_kernel.cuh"

namespace gbn {

namespace {

template <int MODE, int K, bool CLUSTER, bool RESID>
const void *pick_exact(bool e) {
  return e ? reinterpret_cast<const void *>(
                 &norm_fwd_kernel<MODE, K, CLUSTER, true, RESID, kOutBf16, false>)
           : reinterpret_cast<const void *>(
                 &norm_fwd_kernel<MODE, K, CLUSTER, false, RESID, kOutBf16, false>);
}

template <int MODE, int K, bool CLUSTER>
const void *pick_variant(bool e, bool r) {
  if (r) return CLUSTER ? nullptr : pick_exact<MODE, K, false, true>(e);  // no cluster variants
  return pick_exact<MODE, K, CLUSTER, false>(e);
}

template <int MODE, bool CLUSTER>
const void *pick_fwd(int K, bool e, bool r) {
  switch (K) {
    case 1: return pick_variant<MODE, 1, CLUSTER>(e, r);
    case 2: return pick_variant<MODE, 2, CLUSTER>(e, r);
    case 3: return pick_variant<MODE, 3, CLUSTER>(e, r);
    case 4: return pick_variant<MODE, 4, CLUSTER>(e, r);
    case 5: return pick_variant<MODE, 5, CLUSTER>(e, r);
    case 6: return pick_variant<MODE, 6, CLUSTER>(e, r);
    case 8: return pick_variant<MODE, 8, CLUSTER>(e, r);
    default: return nullptr;
  }
}

// Variants whose stage waits sleep (the plan's suspend hint): exact,
// single-CTA, plain, 2 or 4 chunks per thread.
template <int MODE>
const void *pick_sleep(int K) {
  switch (K) {
    case 2: return reinterpret_cast<const void *>(
        &norm_fwd_kernel<MODE, 2, false, true, false, kOutBf16, false, true>);
    case 4: return reinterpret_cast<const void *>(
        &norm_fwd_kernel<MODE, 4, false, true, false, kOutBf16, false, true>);
    default: return nullptr;
  }
}

}  // namespace

const void *fwd_kernel_ptr(int mode, int K, bool cluster, bool exact, bool resid, bool gsm,
                           bool sleep) {
  if (sleep) {
    if (cluster || !exact || resid || gsm) return nullptr;
    return mode == kRMS ? pick_sleep<kRMS>(K) : pick_sleep<kLayer>(K);
  }
  if (gsm) return (cluster || !exact) ? nullptr : fwd_gsm_kernel_ptr(mode, K, resid, kOutBf16);
  if (mode == kRMS)
    return cluster ? pick_fwd<kRMS, true>(K, exact, resid) : pick_fwd<kRMS, false>(K, exact, resid);
  return cluster ? pick_fwd<kLayer, true>(K, exact, resid)
                 : pick_fwd<kLayer, false>(K, exact, resid);
}

}  // namespace gbn
