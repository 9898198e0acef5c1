// Kernel instances of the one-launch MLP layer (gate+up width, down width).
#include "gemv.cuh"

namespace nq {

const void* mlp_kernel(int bits_gu, int bits_down) {
  if (bits_gu == 4 && bits_down == 4) return reinterpret_cast<const void*>(&nq_mlp_kernel<4, 4>);
  if (bits_gu == 4 && bits_down == 5) return reinterpret_cast<const void*>(&nq_mlp_kernel<4, 5>);
  if (bits_gu == 6 && bits_down == 4) return reinterpret_cast<const void*>(&nq_mlp_kernel<6, 4>);
  if (bits_gu == 8 && bits_down == 8) return reinterpret_cast<const void*>(&nq_mlp_kernel<8, 8>);
  return nullptr;
}

}  // namespace nq
