// Kernel instances of the groupwise GEMV for 8-bit codes (MMA route only).
#include "gemv.cuh"

namespace nq {

const void* gemv_kernel_q8(int route, int ntok) {
  if (route != kRouteMma) return nullptr;
  if (ntok == kNtokXreg) return reinterpret_cast<const void*>(&nq_gemv_kernel<8, kRouteMma, kNtokXreg>);
  if (ntok == kNtokXreg2) return reinterpret_cast<const void*>(&nq_gemv_kernel<8, kRouteMma, kNtokXreg2>);
  if (ntok == kNtokXregH) return reinterpret_cast<const void*>(&nq_gemv_kernel<8, kRouteMma, kNtokXregH>);
  return ntok == 1 ? reinterpret_cast<const void*>(&nq_gemv_kernel<8, kRouteMma, 1>)
                   : reinterpret_cast<const void*>(&nq_gemv_kernel<8, kRouteMma, 2>);
}

}  // namespace nq
