// fwd_gsm.cu -- instantiations of the forward kernel (fwd_kernel.cuh) that
// stage gamma and beta in shared memory and read them per row, so a thread
// can hold 5, 6 or 8 chunks of the row in registers: fewer, fuller warps per
// row, which amortises each row's reduction rounds.  Exact splits only, no
// cluster; bf16 or E4M3 output, plain or fused-residual.
#include "fwd_kernel.cuh"

namespace gbn {

namespace {

template <int MODE, int K, bool RESID>
const void *pick_out(int out) {
  switch (out) {
    case kOutBf16:
      return reinterpret_cast<const void *>(&norm_fwd_kernel<MODE, K, false, true, RESID, kOutBf16, true>);
    case kOutFp8Row:
      return reinterpret_cast<const void *>(&norm_fwd_kernel<MODE, K, false, true, RESID, kOutFp8Row, true>);
    case kOutFp8Mx:
      return reinterpret_cast<const void *>(&norm_fwd_kernel<MODE, K, false, true, RESID, kOutFp8Mx, true>);
    default: return nullptr;
  }
}

template <int MODE, int K>
const void *pick_resid(bool r, int out) {
  return r ? pick_out<MODE, K, true>(out) : pick_out<MODE, K, false>(out);
}

template <int MODE>
const void *pick_k(int K, bool r, int out) {
  switch (K) {
    case 5: return pick_resid<MODE, 5>(r, out);
    case 6: return pick_resid<MODE, 6>(r, out);
    case 8: return pick_resid<MODE, 8>(r, out);
    default: return nullptr;
  }
}

}  // namespace

const void *fwd_gsm_kernel_ptr(int mode, int K, bool resid, int out) {
  return mode == kRMS ? pick_k<kRMS>(K, resid, out) : pick_k<kLayer>(K, resid, out);
}

}  // namespace gbn
