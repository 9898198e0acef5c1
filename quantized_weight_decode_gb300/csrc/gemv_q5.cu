// Kernel instances of the groupwise GEMV for 5-bit codes.
#include "gemv.cuh"

namespace nq {

const void* gemv_kernel_q5(int route, int ntok) {
  if (route == kRouteMma) {
    if (ntok == kNtokXreg) return reinterpret_cast<const void*>(&nq_gemv_kernel<5, kRouteMma, kNtokXreg>);
    if (ntok == kNtokXreg2) return reinterpret_cast<const void*>(&nq_gemv_kernel<5, kRouteMma, kNtokXreg2>);
    if (ntok == kNtokXregH) return reinterpret_cast<const void*>(&nq_gemv_kernel<5, kRouteMma, kNtokXregH>);
    return ntok == 1 ? reinterpret_cast<const void*>(&nq_gemv_kernel<5, kRouteMma, 1>)
                     : reinterpret_cast<const void*>(&nq_gemv_kernel<5, kRouteMma, 2>);
  }
  return reinterpret_cast<const void*>(&nq_gemv_kernel<5, kRouteFfma, 4>);
}

}  // namespace nq
