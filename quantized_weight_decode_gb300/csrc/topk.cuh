// Top-k of the fused verify head: keys, warp-level bitonic sort and merge.
//
// The candidate top-k of a speculative-verify round reads the output head's
// logits (page "Qwen3.8-27B for NInfer on the RTX 3090", section "Run it":
// the drafter's candidate top-k over the proposal head or the full head).
// Each logit y[t, n] becomes one 64-bit key whose unsigned order is the
// order of the result: the fp32 value mapped to an order-preserving 32-bit
// pattern in the high half (larger value, larger key; -0 just below +0), the
// complement of the row index in the low half (equal values: smaller index
// first).  Keys of distinct rows are distinct, so the top k are unique, and
// key 0 (never a real logit's: its index would be 2^32 - 1) marks an empty
// entry.
#pragma once

#include <cstdint>

namespace nq {

constexpr int kTopkMax = 32;  // largest k: one key per lane of a warp

__device__ __forceinline__ unsigned long long topk_key(float v, uint32_t idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(~idx);
}
__device__ __forceinline__ float topk_key_value(unsigned long long key) {
  const uint32_t h = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((h & 0x80000000u) ? (h & 0x7FFFFFFFu) : ~h);
}
__device__ __forceinline__ int topk_key_index(unsigned long long key) {
  return static_cast<int>(~static_cast<uint32_t>(key));
}

// 32 keys, one per lane, sorted in descending order across the lanes
// (bitonic sorting network: in each step the lower lane of a pair keeps the
// larger key where its block runs descending, the smaller where ascending).
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int d = size >> 1; d >= 1; d >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, d);
      const bool keep_max = ((lane & d) == 0) == ((lane & size) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// A bitonic sequence of 32 keys (one per lane) sorted descending.
__device__ __forceinline__ unsigned long long warp_bitonic_merge_desc(unsigned long long v,
                                                                      int lane) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, d);
    v = (lane & d) == 0 ? (v > o ? v : o) : (v < o ? v : o);
  }
  return v;
}

// The 32 largest of two descending 32-key lists a and b (lane j holds entry
// j of each): max(a[j], b[31 - j]) keeps exactly the 32 largest keys of the
// union as a bitonic sequence, which the merge then sorts.
__device__ __forceinline__ unsigned long long warp_top32_of_two(unsigned long long a,
                                                                unsigned long long b, int lane) {
  const unsigned long long br = __shfl_sync(0xffffffffu, b, 31 - lane);
  return warp_bitonic_merge_desc(a > br ? a : br, lane);
}

}  // namespace nq
