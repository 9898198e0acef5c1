// Auxiliary device kernels: device packer, round-to-nearest encoder,
// dequantisation (test aid), the bounded-wait self-test, and the per-device
// status word that kernels use to report errors.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "gemv.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace nq {

__device__ int g_status_word;  // per device: first error a kernel recorded

int* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

// Per device: the activation counters of the one-launch MLP layer, two words
// per launch slot; zero at load, reset to zero by every launch that uses them.
__device__ unsigned g_sync_slots[2 * kSyncSlots];

unsigned* sync_slots_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_sync_slots) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

// ------------------------------------------------------------------ packer
// One thread per (row tile, group, lane): gathers the lane's 32 codes from the
// row-major code matrix and writes its words; lanes 0..15 also write the
// scale of row `lane` of the tile.
template <int BITS>
__global__ void nq_pack_kernel(const int8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                            long long K, long long N, int G, long long nthreads,
                            uint8_t* __restrict__ packed, uint16_t* __restrict__ scales_out) {
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (tid >= nthreads) return;
  const int lane = static_cast<int>(tid & 31);
  const long long blk = tid >> 5;  // rt * G + g
  const long long rt = blk / G;
  const int g = static_cast<int>(blk - rt * G);
  uint32_t u[32];
#pragma unroll
  for (int p = 0; p < 16; ++p) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int row, k;
      lane_code_coords(lane, p, h, &row, &k);
      const long long n = rt * kTileRows + row;
      const int c = n < N ? codes[n * K + static_cast<long long>(g) * kGroup + k] : 0;
      u[2 * p + h] = static_cast<uint32_t>(c + (1 << (BITS - 1)));
    }
  }
  uint32_t w[BITS];
  encode_lane(BITS, u, w);
  uint8_t* base = packed + blk * block_bytes(BITS);
#pragma unroll
  for (int i = 0; i < BITS; ++i)
    *reinterpret_cast<uint32_t*>(base + lane_word_offset(BITS, lane, i)) = w[i];
  if (lane < 16) {
    const int m = lane & 7, h = lane >> 3;
    const long long n = rt * kTileRows + lane;
    scales_out[blk * 16 + 2 * m + h] = n < N ? scales[n * G + g] : static_cast<uint16_t>(0);
  }
}

cudaError_t launch_pack_device(const int8_t* codes, const uint16_t* scales, long long K,
                               long long N, int bits, void* packed, uint16_t* scales_out,
                               cudaStream_t st) {
  const int G = static_cast<int>(K / kGroup);
  const long long nt = (N + kTileRows - 1) / kTileRows;
  const long long nthreads = nt * G * 32;
  const int block = 256;
  const long long grid = (nthreads + block - 1) / block;
  auto* out = static_cast<uint8_t*>(packed);
  switch (bits) {
    case 4: nq_pack_kernel<4><<<grid, block, 0, st>>>(codes, scales, K, N, G, nthreads, out, scales_out); break;
    case 5: nq_pack_kernel<5><<<grid, block, 0, st>>>(codes, scales, K, N, G, nthreads, out, scales_out); break;
    case 8: nq_pack_kernel<8><<<grid, block, 0, st>>>(codes, scales, K, N, G, nthreads, out, scales_out); break;
    default: nq_pack_kernel<6><<<grid, block, 0, st>>>(codes, scales, K, N, G, nthreads, out, scales_out); break;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dequant
// w = fp32(scale) * fp32(code), exact; uses the GEMV's own decode of a lane.
template <int BITS>
__global__ void nq_dequant_kernel(const uint8_t* __restrict__ packed,
                               const uint16_t* __restrict__ scales, long long K, long long N,
                               int G, long long nthreads, float* __restrict__ w) {
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (tid >= nthreads) return;
  const int lane = static_cast<int>(tid & 31);
  const long long blk = tid >> 5;
  const long long rt = blk / G;
  const int g = static_cast<int>(blk - rt * G);
  const uint8_t* base = packed + blk * block_bytes(BITS);
  uint32_t words[BITS];
#pragma unroll
  for (int i = 0; i < BITS; ++i)
    words[i] = *reinterpret_cast<const uint32_t*>(base + lane_word_offset(BITS, lane, i));
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    // bf16 codes from the GEMV's decode; 8-bit codes (wider than the bf16
    // trick) straight from their fields
    uint32_t c2;
    if constexpr (BITS == 8) c2 = pair_field<8>(words, p);
    else c2 = pair_codes_bf16<BITS>(words, p);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int row, k;
      lane_code_coords(lane, p, h, &row, &k);
      const long long n = rt * kTileRows + row;
      if (n >= N) continue;
      float c;
      if constexpr (BITS == 8) c = static_cast<float>(static_cast<int>((c2 >> (16 * h)) & 0xFFu) - 128);
      else c = __uint_as_float(h == 0 ? (c2 << 16) : (c2 & 0xFFFF0000u));
      const uint16_t sb = scales[blk * 16 + 2 * (row & 7) + (row >> 3)];
      const float s = __half2float(__ushort_as_half(sb));
      w[n * K + static_cast<long long>(g) * kGroup + k] = s * c;
    }
  }
}

cudaError_t launch_dequant(const void* packed, const uint16_t* scales, float* w, long long K,
                           long long N, int bits, cudaStream_t st) {
  const int G = static_cast<int>(K / kGroup);
  const long long nt = (N + kTileRows - 1) / kTileRows;
  const long long nthreads = nt * G * 32;
  const int block = 256;
  const long long grid = (nthreads + block - 1) / block;
  auto* in = static_cast<const uint8_t*>(packed);
  switch (bits) {
    case 4: nq_dequant_kernel<4><<<grid, block, 0, st>>>(in, scales, K, N, G, nthreads, w); break;
    case 5: nq_dequant_kernel<5><<<grid, block, 0, st>>>(in, scales, K, N, G, nthreads, w); break;
    case 8: nq_dequant_kernel<8><<<grid, block, 0, st>>>(in, scales, K, N, G, nthreads, w); break;
    default: nq_dequant_kernel<6><<<grid, block, 0, st>>>(in, scales, K, N, G, nthreads, w); break;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ RTN encoder
// One warp per 64-group: absmax by warp reduction (exact), scale = FP16
// round-to-nearest-even of the fp64 quotient absmax / qmax, codes
// = clamp(rint(w / s)) with the quotient in fp64 (IEEE, correctly rounded).
__global__ void nq_quantize_rtn_kernel(const float* __restrict__ w, long long K, long long ngroups,
                                    int G, int bits, int8_t* __restrict__ codes,
                                    uint16_t* __restrict__ scales, int* status) {
  const long long gw = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= ngroups) return;
  const long long n = gw / G;
  const int g = static_cast<int>(gw - n * G);
  const long long off = n * K + static_cast<long long>(g) * kGroup + 2 * lane;
  const float2 v = *reinterpret_cast<const float2*>(w + off);
  float a = fmaxf(fabsf(v.x), fabsf(v.y));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  const int qmax = (1 << (bits - 1)) - 1;
  const __half sh = __double2half(static_cast<double>(a) / static_cast<double>(qmax));
  const uint16_t sbits = __half_as_ushort(sh);
  if ((sbits & 0x7C00u) == 0x7C00u) {
    if (lane == 0) atomicCAS(status, 0, -3);
  }
  const double s = static_cast<double>(__half2float(sh));
  int c0 = 0, c1 = 0;
  if (s != 0.0) {
    const double lo = -static_cast<double>(qmax) - 1.0, hi = static_cast<double>(qmax);
    c0 = static_cast<int>(fmin(fmax(rint(static_cast<double>(v.x) / s), lo), hi));
    c1 = static_cast<int>(fmin(fmax(rint(static_cast<double>(v.y) / s), lo), hi));
  }
  char2 cc;
  cc.x = static_cast<signed char>(c0);
  cc.y = static_cast<signed char>(c1);
  *reinterpret_cast<char2*>(codes + off) = cc;
  if (lane == 0) scales[n * G + g] = sbits;
}

cudaError_t launch_quantize_rtn(const float* w, long long K, long long N, int bits, int8_t* codes,
                                uint16_t* scales, int* status, cudaStream_t st) {
  const int G = static_cast<int>(K / kGroup);
  const long long ngroups = N * G;
  const int block = 256;  // 8 groups per block
  const long long grid = (ngroups * 32 + block - 1) / block;
  nq_quantize_rtn_kernel<<<grid, block, 0, st>>>(w, K, ngroups, G, bits, codes, scales, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ searched encoder
// The "grouped_search" encoder of the page "Qwen3.8-27B for NInfer on the RTX
// 3090" (section "What is different from the upstream artifact"): each
// group's FP16 scale is the best of 50 candidates by importance-weighted
// squared error, importance q_k per channel (an imatrix); scales may be
// negative.  Candidates (the page gives none; our reading): with a = max|w|,
// h_i = fp16_rne(12 a / (12 (qmax + 1) - i)), i = 0..24, tried as +h_i
// (candidate 2i) and -h_i (2i + 1); codes clamp(rint(w / s)) (0 for a zero
// scale); error sum_k q_k (w_k - s c_k)^2 accumulated over k in order in fp64,
// every product and sum rounded on its own (no fused multiply-add), so the
// choice is reproducible bit for bit.  Smallest error wins, ties to the lower
// candidate; candidates whose scale overflows FP16 take no part (if all do,
// NQ_ERANGE).  One warp per group: lane l holds weights 2l, 2l + 1 and
// candidates l and l + 32.
__global__ void nq_quantize_search_kernel(const float* __restrict__ w, const float* __restrict__ imp,
                                       long long K, long long ngroups, int G, int bits,
                                       int8_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                       int* status) {
  const long long gw = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= ngroups) return;
  const long long n = gw / G;
  const int g = static_cast<int>(gw - n * G);
  const long long off = n * K + static_cast<long long>(g) * kGroup + 2 * lane;
  const float2 v = *reinterpret_cast<const float2*>(w + off);
  const float2 qv = imp ? *reinterpret_cast<const float2*>(imp + static_cast<long long>(g) * kGroup + 2 * lane)
                        : make_float2(1.f, 1.f);
  float a = fmaxf(fabsf(v.x), fabsf(v.y));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  const int qmax = (1 << (bits - 1)) - 1;
  const double lo = -static_cast<double>(qmax) - 1.0, hi = static_cast<double>(qmax);
  auto cand_bits = [&](int j) -> uint16_t {
    const int i = j >> 1;
    const __half h = __double2half((12.0 * static_cast<double>(a)) / (12.0 * (qmax + 1) - i));
    return static_cast<uint16_t>(__half_as_ushort(h) | ((j & 1) << 15));
  };
  auto code_of = [&](double x, double s) -> double {
    return s == 0.0 ? 0.0 : fmin(fmax(rint(x / s), lo), hi);
  };
  double sj[2], err[2] = {0.0, 0.0};
  bool valid[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int j = lane + 32 * c;
    const uint16_t b = j < 50 ? cand_bits(j) : 0x7C00u;
    valid[c] = j < 50 && (b & 0x7C00u) != 0x7C00u;
    sj[c] = valid[c] ? static_cast<double>(__half2float(__ushort_as_half(b))) : 0.0;
  }
  for (int k = 0; k < kGroup; ++k) {
    const double wk = __shfl_sync(0xffffffffu, (k & 1) ? v.y : v.x, k >> 1);
    const double qk = __shfl_sync(0xffffffffu, (k & 1) ? qv.y : qv.x, k >> 1);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const double d = __dsub_rn(wk, __dmul_rn(sj[c], code_of(wk, sj[c])));
      err[c] = __dadd_rn(err[c], __dmul_rn(qk, __dmul_rn(d, d)));
    }
  }
  double be = INFINITY;
  int bj = INT_MAX;
#pragma unroll
  for (int c = 0; c < 2; ++c)
    if (valid[c] && err[c] < be) {
      be = err[c];
      bj = lane + 32 * c;
    }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const double oe = __shfl_xor_sync(0xffffffffu, be, m);
    const int oj = __shfl_xor_sync(0xffffffffu, bj, m);
    if (oe < be || (oe == be && oj < bj)) {
      be = oe;
      bj = oj;
    }
  }
  uint16_t sbits = 0x7C00u;
  double s = 0.0;
  if (bj == INT_MAX) {
    if (lane == 0) atomicCAS(status, 0, -3);
  } else {
    sbits = cand_bits(bj);
    s = static_cast<double>(__half2float(__ushort_as_half(sbits)));
  }
  char2 cc;
  cc.x = static_cast<signed char>(code_of(v.x, s));
  cc.y = static_cast<signed char>(code_of(v.y, s));
  *reinterpret_cast<char2*>(codes + off) = cc;
  if (lane == 0) scales[n * G + g] = sbits;
}

cudaError_t launch_quantize_search(const float* w, const float* imatrix, long long K, long long N,
                                   int bits, int8_t* codes, uint16_t* scales, int* status,
                                   cudaStream_t st) {
  const int G = static_cast<int>(K / kGroup);
  const long long ngroups = N * G;
  const int block = 256;  // 8 groups per block
  const long long grid = (ngroups * 32 + block - 1) / block;
  nq_quantize_search_kernel<<<grid, block, 0, st>>>(w, imatrix, K, ngroups, G, bits, codes, scales,
                                                 status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ self-test
// Waits on a barrier that nothing completes; the bounded wait gives up after
// `limit_ns`, records NQ_ETIMEOUT and the kernel returns normally.
__global__ void nq_selftest_timeout_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(smem_addr(&bar), 1);
  abort_flag = 0;
  fence_mbar_init();
  const Waiter wt{&abort_flag, limit_ns, status};
  (void)wt.wait<false>(smem_addr(&bar), 0);
}

cudaError_t launch_selftest_timeout(unsigned long long limit_ns, int* status, cudaStream_t st) {
  nq_selftest_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace nq
