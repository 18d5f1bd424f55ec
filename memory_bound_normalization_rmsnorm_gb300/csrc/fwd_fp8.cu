// fwd_fp8.cu -- E4M3-output instantiations of the forward kernel
// (fwd_kernel.cuh): per-row or MX block scaling, plain or fused-residual,
// register-resident rows only (no cluster variants).
#include "fwd_kernel.cuh"

namespace gbn {

namespace {

template <int MODE, int K, bool RESID, int OUT>
const void *pick_exact(bool e) {
  return e ? reinterpret_cast<const void *>(
                 &norm_fwd_kernel<MODE, K, false, true, RESID, OUT, false>)
           : reinterpret_cast<const void *>(
                 &norm_fwd_kernel<MODE, K, false, false, RESID, OUT, false>);
}

template <int MODE, int K>
const void *pick_variant(bool e, bool r, int out) {
  if (out == kOutFp8Row) return r ? pick_exact<MODE, K, true, kOutFp8Row>(e)
                                  : pick_exact<MODE, K, false, kOutFp8Row>(e);
  if (out == kOutFp8Mx) return r ? pick_exact<MODE, K, true, kOutFp8Mx>(e)
                                 : pick_exact<MODE, K, false, kOutFp8Mx>(e);
  return nullptr;
}

// Chunks per thread that the planner can pick for register-resident rows
// (at most 4 for LayerNorm and 6 for RMSNorm: the most that fit in
// registers without spilling); wider rows are refused for E4M3 output.
template <int MODE, int K>
const void *pick_k(bool e, bool r, int out) {
  if constexpr (K <= (MODE == kLayer ? 4 : 6)) return pick_variant<MODE, K>(e, r, out);
  return nullptr;
}

template <int MODE>
const void *pick_fp8(int K, bool e, bool r, int out) {
  switch (K) {
    case 1: return pick_k<MODE, 1>(e, r, out);
    case 2: return pick_k<MODE, 2>(e, r, out);
    case 3: return pick_k<MODE, 3>(e, r, out);
    case 4: return pick_k<MODE, 4>(e, r, out);
    case 5: return pick_k<MODE, 5>(e, r, out);
    case 6: return pick_k<MODE, 6>(e, r, out);
    default: return nullptr;
  }
}

}  // namespace

const void *fwd_fp8_kernel_ptr(int mode, int K, bool exact, bool resid, int out, bool gsm) {
  if (gsm) return exact ? fwd_gsm_kernel_ptr(mode, K, resid, out) : nullptr;
  return mode == kRMS ? pick_fp8<kRMS>(K, exact, resid, out)
                      : pick_fp8<kLayer>(K, exact, resid, out);
}

}  // namespace gbn
