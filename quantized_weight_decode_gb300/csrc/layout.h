// Packed-code layout, version 2 (full description in include/nq.h).
//
// The groupwise encoding itself -- signed codes in 64-weight groups with one
// FP16 scale each, w = scale * code -- is the one on the page "Qwen3.8-27B
// for NInfer on the RTX 3090" (section "What is different from the upstream
// artifact").  The page gives no storage layout; this one is ours, built for
// the sm_103a kernels:
//   * a row tile of 16 rows x one 64-group is one 1024-code block, split over
//     the 32 lanes of a warp in the register order of the A operand of
//     mma.m16n8k16 (lane q*4+r: rows q and q+8), with the group's K order
//     permuted so that the 16 k of lane r are k = 16r .. 16r + 15 (K slice j
//     of the MMA takes k = 16r + 4j + {0,1} and 16r + 4j + 2 + {0,1}): a dot
//     product does not depend on the order of its terms, and this one makes
//     a lane's x fragments 32 contiguous bytes of x (two 16-byte loads);
//   * the two codes of an A-fragment register sit at the same bit offset in
//     the two 16-bit halves of a 32-bit word, so one mask-and-or turns them
//     into two bf16 values 128 + u (u <= 127 fills the 7-bit mantissa of
//     bf16 with exponent 2^7), and one bf16x2 FMA removes 128 + 2^(b-1);
//   * 5- and 6-bit fields are packed three (resp. two) per 16-bit half, with
//     the leftover bits of every half holding one (resp. four) extra pairs, so
//     no bits are wasted: 5.0 / 6.0 bits per code on top of the scales;
//   * 8-bit fields are the two bytes of each half (pair 2w + f at byte f of
//     word w's halves).
// This header is shared by the host packer, the device packer, the dequant
// kernel and the GEMV kernels, so all of them agree on the format.
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define NQ_HD __host__ __device__ __forceinline__
#else
#define NQ_HD inline
#endif

namespace nq {

constexpr int kTileRows = 16;           // rows per tile (MMA M)
constexpr int kGroup = 64;              // codes per group along K
constexpr int kLanes = 32;
constexpr int kScaleBytesPerBlock = 32; // 16 FP16 scales
constexpr int kLayoutVersion = 2;

NQ_HD int block_bytes(int bits) { return 128 * bits; }   // 32 lanes * bits words * 4 B

// Position of code (pair p, half h) of lane `lane` inside the block:
// row in the tile and k inside the group.
NQ_HD void lane_code_coords(int lane, int p, int h, int* row, int* k) {
  const int q = lane >> 2, r = lane & 3;
  const int j = p >> 2, i = p & 3;
  *row = q + 8 * (i & 1);
  *k = 16 * r + 4 * j + 2 * (i >> 1) + h;
}

// Byte offset, inside a block, of word w of lane `lane`.
NQ_HD int lane_word_offset(int bits, int lane, int w) {
  return w < 4 ? 16 * lane + 4 * w : 512 + 4 * (bits - 4) * lane + 4 * (w - 4);
}

// Encode: biased codes u[2p + h] (0 <= u < 2^bits) of one lane -> `bits` words.
NQ_HD void encode_lane(int bits, const uint32_t* u, uint32_t* w) {
  for (int i = 0; i < bits; ++i) w[i] = 0;
  for (int p = 0; p < 16; ++p) {
    for (int h = 0; h < 2; ++h) {
      const uint32_t v = u[2 * p + h];
      const int hs = 16 * h;
      if (bits == 4) {
        w[p >> 2] |= v << (4 * (p & 3) + hs);
      } else if (bits == 8) {
        w[p >> 1] |= v << (8 * (p & 1) + hs);
      } else if (bits == 5) {
        if (p < 15) {
          w[p / 3] |= v << (5 * (p % 3) + hs);
        } else {
          for (int m = 0; m < 5; ++m) w[m] |= ((v >> m) & 1u) << (15 + hs);
        }
      } else {  // 6
        if (p < 12) {
          w[p >> 1] |= v << (6 * (p & 1) + hs);
        } else {
          const int d = p - 12;
          w[d] |= (v & 15u) << (12 + hs);
          w[4 + (d >> 1)] |= (v >> 4) << (12 + 2 * (d & 1) + hs);
        }
      }
    }
  }
}

// Decode one pair of fields: the two biased codes of pair p placed at bits
// [0, bits) and [16, 16 + bits) of the result, everything else zero.
template <int BITS>
NQ_HD uint32_t pair_field(const uint32_t (&w)[BITS], int p) {
  if constexpr (BITS == 4) {
    return (w[p >> 2] >> (4 * (p & 3))) & 0x000F000Fu;
  } else if constexpr (BITS == 8) {
    return (w[p >> 1] >> (8 * (p & 1))) & 0x00FF00FFu;
  } else if constexpr (BITS == 5) {
    if (p < 15) return (w[p / 3] >> (5 * (p % 3))) & 0x001F001Fu;
    uint32_t t = (w[0] >> 15) & 0x00010001u;
    t |= (w[1] >> 14) & 0x00020002u;
    t |= (w[2] >> 13) & 0x00040004u;
    t |= (w[3] >> 12) & 0x00080008u;
    t |= (w[4] >> 11) & 0x00100010u;
    return t;
  } else {
    if (p < 12) return (w[p >> 1] >> (6 * (p & 1))) & 0x003F003Fu;
    const int d = p - 12;
    const uint32_t lo = (w[d] >> 12) & 0x000F000Fu;
    const uint32_t hi = (w[4 + (d >> 1)] >> (8 + 2 * (d & 1))) & 0x00300030u;
    return lo | hi;
  }
}

// bf16 patterns: 128 + u  (exponent 2^7, u in the mantissa), and the bias
// 128 + 2^(bits-1) that turns it back into the signed code.
constexpr uint32_t kBf16Magic2 = 0x43004300u;
NQ_HD uint32_t bf16_neg_bias2(int bits) {
  // -(128 + 2^(bits-1)) as bf16: sign | exponent 2^7 | mantissa 2^(bits-1)
  const uint32_t h = 0xC300u | (1u << (bits - 1));
  return h | (h << 16);
}
constexpr uint32_t kBf16One2 = 0x3F803F80u;

}  // namespace nq
