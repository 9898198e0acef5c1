// Groupwise-quantized small-T GEMV for sm_103a.
//
//   y[t, n] = sum_g s[n, g] * sum_{k in g} c[n, k] * x[t, k]
//
// The operation is the decode / speculative-verify product of the engine on
// the pages "Qwen3.8-27B for NInfer on the RTX 3090" (groupwise codes, 64-
// weight groups, FP16 scales; section "What is different from the upstream
// artifact") and "giveen/ninfer-ext" (K-split routes for the small batches of
// the verify rounds; group-level load pipelining; sections "Where ninfer-ext
// leads" and "Engineering").  The kernel structure is our own design for one
// GB300 SM:
//
//   warp 0..15 consumers : each owns a fixed K slice of the CTA's K range and
//                          streams its own chunks (several 64-groups of one
//                          16-row tile, plus their scales) with 1-D bulk copies
//                          (TMA engine, L2 evict-first) into a private ring of
//                          shared-memory slots; it decodes the codes in
//                          registers, contracts them with the x tile (bf16 MMA
//                          m16n8k16 or fp32 FMA) and scales each 64-wide
//                          partial by the group's FP16 scale;
//   warp 16    epilogue  : sums the 16 per-warp partials of a row tile in a
//                          fixed order, adds the partials of the other CTAs of
//                          its cluster (K split, distributed shared memory,
//                          rank order) and stores y.
//
// A warp refills a ring slot as soon as it has read it, so no CTA-wide
// handshake sits on the weight stream.  Work split: a persistent grid of
// clusters of KS CTAs; cluster c owns a contiguous range of 16-row tiles
// ("jobs"); rank q handles groups [q G / KS, (q+1) G / KS) of every job.  The
// x slice of a CTA is loaded once into shared memory, permuted into MMA
// B-fragment order.  Every wait is bounded by a time limit; on expiry the
// kernel records NQ_ETIMEOUT in the status word and winds down without
// hanging or leaving bulk copies in flight.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "layout.h"
#include "ptx.cuh"

namespace nq {

constexpr int kWarps = 16;                   // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;  // + the epilogue warp
constexpr int kEpilogueWarp = kWarps;
constexpr int kMaxWarpStages = 8;            // ring slots per consumer warp
constexpr int kMaxChunkGroups = 8;           // 64-groups per chunk
constexpr int kStatusTimeout = -5;
// MMA route kernel variants (template NTOK): 1 or 2 token blocks of 8 with x
// in shared memory, or kNtokXreg: one token block, x in registers, at most
// kXregMaxGroups groups per warp slice.
constexpr int kNtokXreg = 3;
constexpr int kXregMaxGroups = 6;

enum Route : int { kRouteMma = 1, kRouteFfma = 2 };

struct GemvArgs {
  const uint8_t* codes;    // packed codes
  const uint16_t* scales;  // packed scales
  const uint16_t* x;       // bf16 [T, K]
  float* y;                // fp32 [T, N]
  long long N;
  int K, T, G, Nt;
  int ksplit;              // CTAs per cluster splitting K
  int clusters;            // clusters in the grid
  int chunk_groups;        // 64-groups per chunk (one pair of bulk copies)
  int wstages;             // ring slots per consumer warp
  int wstage_bytes;        // bytes of one slot (codes + scales, 128-aligned)
  int off_ring, off_red, off_cl, off_x;  // shared-memory offsets
  unsigned long long wait_ns;
  int* status;
};

// Shared-memory map of the barrier region (first 2 KiB).
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int w, int s) const { return base + 8 * (w * kMaxWarpStages + s); }
  __device__ uint32_t red_full(int b) const { return base + 1024 + 8 * b; }
  __device__ uint32_t red_empty(int b) const { return base + 1040 + 8 * b; }
  __device__ uint32_t cl_full(int b) const { return base + 1056 + 8 * b; }
  __device__ uint32_t cl_empty(int b) const { return base + 1072 + 8 * b; }
};
constexpr int kAbortFlagOffset = 1152;
constexpr int kZeroAreaOffset = 1536;  // 32 zero bytes: x fragments of absent tokens
constexpr int kBarRegionBytes = 2048;
static_assert(8 * kWarps * kMaxWarpStages <= 1024, "barrier region");

struct Waiter {
  volatile int* abort;
  unsigned long long limit;
  int* status;

  // Bounded wait for the completion of the phase with parity `par`.
  template <bool kClusterScope>
  __device__ bool wait(uint32_t bar, uint32_t par) const {
    auto probe = [&]() {
      return kClusterScope ? mbar_try_wait_cluster(bar, par) : mbar_try_wait(bar, par);
    };
    if (probe()) return true;
    const uint64_t t0 = global_ns();
    while (true) {
      if (probe()) return true;
      if (*abort) return false;
      if (global_ns() - t0 > limit) {
        *abort = 1;
        atomicCAS(status, 0, kStatusTimeout);
        return false;
      }
    }
  }
  // Same, executed by a whole warp; the result is the same in every lane.
  template <bool kClusterScope>
  __device__ bool wait_warp(uint32_t bar, uint32_t par) const {
    const bool ok = wait<kClusterScope>(bar, par);
    return __all_sync(0xffffffffu, ok) != 0;
  }
};

struct Work {
  long long rt_begin;  // first row tile of this cluster
  int njobs;           // row tiles of this cluster
  int g_begin, g_end;  // this CTA's groups
  int rank;
};

__device__ __forceinline__ Work cta_work(const GemvArgs& a) {
  Work w;
  const int ks = a.ksplit;
  const int cl = blockIdx.x / ks;
  w.rank = (ks > 1) ? static_cast<int>(cluster_ctarank()) : 0;
  const long long nt = a.Nt;
  w.rt_begin = (static_cast<long long>(cl) * nt) / a.clusters;
  const long long rt_end = (static_cast<long long>(cl + 1) * nt) / a.clusters;
  w.njobs = static_cast<int>(rt_end - w.rt_begin);
  w.g_begin = (w.rank * a.G) / ks;
  w.g_end = ((w.rank + 1) * a.G) / ks;
  return w;
}

// The K slice of consumer warp `warp`: groups [gs, ge) of every job, cut into
// nch chunks of up to chunk_groups groups.
struct Slice {
  int gs, ge, nch;
};
__device__ __forceinline__ Slice warp_slice(const Work& wk, int warp, int cg) {
  const int gc = wk.g_end - wk.g_begin;
  Slice s;
  s.gs = wk.g_begin + (warp * gc) / kWarps;
  s.ge = wk.g_begin + ((warp + 1) * gc) / kWarps;
  s.nch = (s.ge - s.gs + cg - 1) / cg;
  return s;
}

// ------------------------------------------------------------------ chunk stream
// Lane 0 of a consumer warp: bulk copies of chunk c of its slice into `slot`.
template <int BITS>
__device__ __forceinline__ void issue_chunk(const GemvArgs& a, const Work& wk, const Slice& sl,
                                            int c, uint32_t slot, uint32_t bar, uint64_t policy) {
  constexpr int kBlock = 128 * BITS;
  const int j = c / sl.nch, ci = c - j * sl.nch;
  const int g0 = sl.gs + ci * a.chunk_groups;
  const int n = min(a.chunk_groups, sl.ge - g0);
  const long long blk = (wk.rt_begin + j) * a.G + g0;
  const uint32_t bc = static_cast<uint32_t>(n * kBlock);
  const uint32_t bs = static_cast<uint32_t>(n * kScaleBytesPerBlock);
  mbar_arrive_expect_tx(bar, bc + bs);
  bulk_g2s(slot, a.codes + blk * kBlock, bc, bar, policy);
  bulk_g2s(slot + a.chunk_groups * kBlock, a.scales + blk * 16, bs, bar, policy);
}

// ------------------------------------------------------------------ x tile
// MMA route: entry (g, tok, r) = 8 words = B fragments of the four 16-wide
// K slices j of group g for lane r: word 2j = x[tok][16j+2r .. +1],
// word 2j+1 = x[tok][16j+2r+8 .. +9] (bf16 pairs).
__device__ inline void stage_x_bf16(const GemvArgs& a, uint8_t* smem, const Work& wk, int ctid,
                             int nthreads) {
  const int gc = wk.g_end - wk.g_begin;
  const int total = gc * a.T * 4;
  uint8_t* xs = smem + a.off_x;
  for (int e = ctid; e < total; e += nthreads) {
    const int g = e / (a.T * 4);
    const int rem = e - g * a.T * 4;
    const int tok = rem >> 2, j = rem & 3;
    const long long k0 = 64LL * (wk.g_begin + g) + 16 * j;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<long long>(tok) * a.K + k0);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      uint2 o;
      o.x = w[r];
      o.y = w[4 + r];
      *reinterpret_cast<uint2*>(xs + ((g * a.T + tok) * 4 + r) * 32 + 8 * j) = o;
    }
  }
}

// FMA route: entry (g, tok, r) = 16 floats, [4j + m] = x[tok][16j + 2r + {0,1,8,9}[m]].
__device__ inline void stage_x_f32(const GemvArgs& a, uint8_t* smem, const Work& wk, int ctid,
                            int nthreads) {
  const int gc = wk.g_end - wk.g_begin;
  const int total = gc * a.T * 4;
  uint8_t* xs = smem + a.off_x;
  for (int e = ctid; e < total; e += nthreads) {
    const int g = e / (a.T * 4);
    const int rem = e - g * a.T * 4;
    const int tok = rem >> 2, j = rem & 3;
    const long long k0 = 64LL * (wk.g_begin + g) + 16 * j;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<long long>(tok) * a.K + k0);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float4 o;
      o.x = __uint_as_float(w[r] << 16);
      o.y = __uint_as_float(w[r] & 0xFFFF0000u);
      o.z = __uint_as_float(w[4 + r] << 16);
      o.w = __uint_as_float(w[4 + r] & 0xFFFF0000u);
      *reinterpret_cast<float4*>(xs + ((g * a.T + tok) * 4 + r) * 64 + 16 * j) = o;
    }
  }
}

// ------------------------------------------------------------------ decode
template <int BITS>
__device__ __forceinline__ void load_lane_words(const uint8_t* blk, int lane, uint32_t (&w)[BITS]) {
  const uint4 v = *reinterpret_cast<const uint4*>(blk + 16 * lane);
  w[0] = v.x;
  w[1] = v.y;
  w[2] = v.z;
  w[3] = v.w;
  if constexpr (BITS == 5) {
    w[4] = *reinterpret_cast<const uint32_t*>(blk + 512 + 4 * lane);
  } else if constexpr (BITS == 6) {
    const uint2 u = *reinterpret_cast<const uint2*>(blk + 512 + 8 * lane);
    w[4] = u.x;
    w[5] = u.y;
  }
}

// bf16x2 of the signed codes of pair p (exact small integers): the pair's
// two b-bit fields are moved to bits [0, b) and [16, 16 + b) of a word and
// OR-ed into the bf16 pattern 128 + u with one lop3 each (mask and exponent
// pattern in registers), then 128 + 2^(b-1) is subtracted in bf16x2.  The
// same field positions as pair_field() in layout.h, written so that every
// (shift, mask, or) step is one instruction.
template <int BITS>
__device__ __forceinline__ uint32_t pair_codes_bf16(const uint32_t (&w)[BITS], int p) {
  const uint32_t magic = kBf16Magic2;
  uint32_t v;
  if constexpr (BITS == 4) {
    const uint32_t m = 0x000F000Fu;
    v = lop3_and_or(w[p >> 2] >> (4 * (p & 3)), m, magic);
  } else if constexpr (BITS == 5) {
    const uint32_t m = 0x001F001Fu;
    if (p < 15) {
      v = lop3_and_or(w[p / 3] >> (5 * (p % 3)), m, magic);
    } else {
      v = lop3_and_or(w[0] >> 15, 0x00010001u, magic);
      v = lop3_and_or(w[1] >> 14, 0x00020002u, v);
      v = lop3_and_or(w[2] >> 13, 0x00040004u, v);
      v = lop3_and_or(w[3] >> 12, 0x00080008u, v);
      v = lop3_and_or(w[4] >> 11, 0x00100010u, v);
    }
  } else {
    const uint32_t m = 0x003F003Fu;
    if (p < 12) {
      v = lop3_and_or(w[p >> 1] >> (6 * (p & 1)), m, magic);
    } else {
      const int d = p - 12;
      v = lop3_and_or(w[d] >> 12, 0x000F000Fu, magic);
      v = lop3_and_or(w[4 + (d >> 1)] >> (8 + 2 * (d & 1)), 0x00300030u, v);
    }
  }
  constexpr uint32_t kBias = 0x4300u | (1u << (BITS - 1));  // 128 + 2^(BITS-1)
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                   __halves2bfloat162(__ushort_as_bfloat16(kBias),
                                                      __ushort_as_bfloat16(kBias)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// ------------------------------------------------------------------ per-group math
// One group of one row tile on the MMA route: decode the lane's 32 codes, four
// chained MMAs against the x fragments (the first starts from zero), scale,
// accumulate.  xp[nb]: x fragments of token block nb for this lane (zeros if
// the token is absent).
template <int BITS, int NT>
__device__ __forceinline__ void mma_group(const uint8_t* blk, const uint8_t* sc,
                                          const uint8_t* const (&xp)[NT], int lane, int q,
                                          float (&acc)[NT][4]) {
  uint32_t w[BITS];
  load_lane_words<BITS>(blk, lane, w);
  const __half2 sh = *reinterpret_cast<const __half2*>(sc + 4 * q);
  uint4 xa[NT], xb[NT];
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) {
    xa[nb] = *reinterpret_cast<const uint4*>(xp[nb]);
    xb[nb] = *reinterpret_cast<const uint4*>(xp[nb] + 16);
  }
  float d[NT][4];
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    const uint32_t a0 = pair_codes_bf16<BITS>(w, 4 * js + 0);
    const uint32_t a1 = pair_codes_bf16<BITS>(w, 4 * js + 1);
    const uint32_t a2 = pair_codes_bf16<BITS>(w, 4 * js + 2);
    const uint32_t a3 = pair_codes_bf16<BITS>(w, 4 * js + 3);
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      const uint32_t b0 = js == 0 ? xa[nb].x : js == 1 ? xa[nb].z : js == 2 ? xb[nb].x : xb[nb].z;
      const uint32_t b1 = js == 0 ? xa[nb].y : js == 1 ? xa[nb].w : js == 2 ? xb[nb].y : xb[nb].w;
      if (js == 0) {
        mma_16816_zc(d[nb], a0, a1, a2, a3, b0, b1);
      } else {
        mma_16816(d[nb], a0, a1, a2, a3, b0, b1);
      }
    }
  }
  const float2 s = __half22float2(sh);
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) {
    acc[nb][0] = fmaf(s.x, d[nb][0], acc[nb][0]);
    acc[nb][1] = fmaf(s.x, d[nb][1], acc[nb][1]);
    acc[nb][2] = fmaf(s.y, d[nb][2], acc[nb][2]);
    acc[nb][3] = fmaf(s.y, d[nb][3], acc[nb][3]);
  }
}

// One group on the FMA route: the lane's 32 codes times x[t, k] in fp32 for
// t < TMAX; acc[h][t] is the partial of row q + 8h over this lane's k.
template <int BITS, int TMAX>
__device__ __forceinline__ void ffma_group(const uint8_t* blk, const uint8_t* sc,
                                           const uint8_t* xg, int lane, int q, int T,
                                           float (&acc)[2][TMAX]) {
  uint32_t w[BITS];
  load_lane_words<BITS>(blk, lane, w);
  const float2 s = __half22float2(*reinterpret_cast<const __half2*>(sc + 4 * q));
  float part[2][TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) part[0][t] = part[1][t] = 0.f;
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    float xv[TMAX][4];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      const float4 v = t < T ? *reinterpret_cast<const float4*>(xg + 256 * t + 16 * js)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      xv[t][0] = v.x;
      xv[t][1] = v.y;
      xv[t][2] = v.z;
      xv[t][3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t c2 = pair_codes_bf16<BITS>(w, 4 * js + i);
      const float c_lo = __uint_as_float(c2 << 16);
      const float c_hi = __uint_as_float(c2 & 0xFFFF0000u);
      const int row = i & 1, kk = 2 * (i >> 1);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        part[row][t] = fmaf(c_lo, xv[t][kk], part[row][t]);
        part[row][t] = fmaf(c_hi, xv[t][kk + 1], part[row][t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    acc[0][t] = fmaf(s.x, part[0][t], acc[0][t]);
    acc[1][t] = fmaf(s.y, part[1][t], acc[1][t]);
  }
}

// Same as mma_group for one token block, with the lane's x fragments of the
// group held in registers: xr[2 js] / xr[2 js + 1] are B fragments b0 / b1 of
// K slice js.
template <int BITS>
__device__ __forceinline__ void mma_group_xr(const uint8_t* blk, const uint8_t* sc,
                                             const uint32_t (&xr)[8], int lane, int q,
                                             float (&acc)[4]) {
  uint32_t w[BITS];
  load_lane_words<BITS>(blk, lane, w);
  const float2 s = __half22float2(*reinterpret_cast<const __half2*>(sc + 4 * q));
  float d[4];
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    const uint32_t a0 = pair_codes_bf16<BITS>(w, 4 * js + 0);
    const uint32_t a1 = pair_codes_bf16<BITS>(w, 4 * js + 1);
    const uint32_t a2 = pair_codes_bf16<BITS>(w, 4 * js + 2);
    const uint32_t a3 = pair_codes_bf16<BITS>(w, 4 * js + 3);
    if (js == 0) {
      mma_16816_zc(d, a0, a1, a2, a3, xr[0], xr[1]);
    } else {
      mma_16816(d, a0, a1, a2, a3, xr[2 * js], xr[2 * js + 1]);
    }
  }
  acc[0] = fmaf(s.x, d[0], acc[0]);
  acc[1] = fmaf(s.x, d[1], acc[1]);
  acc[2] = fmaf(s.y, d[2], acc[2]);
  acc[3] = fmaf(s.y, d[3], acc[3]);
}

// Consumer warp of the register-resident-x variant (T <= 8): a chunk is the
// warp's whole slice of one job (at most GWM groups), and the warp's x
// fragments for that slice are loaded from global memory once per kernel.
template <int BITS, int GWM>
__device__ void consumer_xreg(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                              const Waiter& wt, const Work& wk, const Slice& sl, int warp,
                              int lane, int issued) {
  constexpr int kBlock = 128 * BITS;
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  const int S = a.wstages;
  const int n = sl.ge - sl.gs;  // groups of this warp's slice (<= GWM)
  const uint32_t ring = smem_addr(smem + a.off_ring) + warp * S * a.wstage_bytes;
  const uint8_t* ring_ptr = smem + a.off_ring + warp * S * a.wstage_bytes;
  const uint8_t* scales_off = ring_ptr + a.chunk_groups * kBlock;
  const uint64_t policy = l2_evict_first_policy();
  float* red = reinterpret_cast<float*>(smem + a.off_red);

  uint32_t xr[GWM][8];
#pragma unroll
  for (int i = 0; i < GWM; ++i) {
#pragma unroll
    for (int e = 0; e < 8; ++e) xr[i][e] = 0u;
    if (i < n && q < T) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(
          a.x + static_cast<long long>(q) * a.K + 64LL * (sl.gs + i) + 2 * r);
#pragma unroll
      for (int js = 0; js < 4; ++js) {
        xr[i][2 * js] = __ldg(src + 8 * js);
        xr[i][2 * js + 1] = __ldg(src + 8 * js + 4);
      }
    }
  }

  int stage = 0;
  uint32_t phase = 0;
  int j = 0;
  for (; j < wk.njobs; ++j) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (n > 0) {
      if (!wt.wait_warp<false>(bars.full(warp, stage), phase)) break;
      const uint8_t* slot = ring_ptr + stage * a.wstage_bytes;
      const uint8_t* scb = scales_off + stage * a.wstage_bytes;
#pragma unroll
      for (int i = 0; i < GWM; ++i)
        if (i < n) mma_group_xr<BITS>(slot + i * kBlock, scb + i * kScaleBytesPerBlock, xr[i], lane, q, acc);
      __syncwarp();
      if (lane == 0 && j + S < wk.njobs) {
        fence_proxy_async_smem();
        issue_chunk<BITS>(a, wk, sl, j + S, ring + stage * a.wstage_bytes, bars.full(warp, stage),
                          policy);
        ++issued;
      }
      if (++stage == S) { stage = 0; phase ^= 1; }
    }
    const int b = j & 1;
    const uint32_t nuse = static_cast<uint32_t>(j >> 1);
    if (!wt.wait_warp<false>(bars.red_empty(b), (nuse & 1u) ^ 1u)) break;
    float* slotp = red + (b * kWarps + warp) * 16 * T;
    const int t0 = 2 * r;
    if (t0 < T) {
      slotp[t0 * 16 + q] = acc[0];
      slotp[t0 * 16 + q + 8] = acc[2];
    }
    if (t0 + 1 < T) {
      slotp[(t0 + 1) * 16 + q] = acc[1];
      slotp[(t0 + 1) * 16 + q + 8] = acc[3];
    }
    mbar_arrive(bars.red_full(b));
  }
  // Wind down: drain chunks issued but not consumed (only after an error).
  const int consumed = (n > 0) ? j : 0;
  if (lane == 0 && issued > consumed) {
    volatile int no_abort = 0;
    const Waiter drain{&no_abort, wt.limit, wt.status};
    for (int cc = consumed; cc < issued; ++cc)
      (void)drain.wait<false>(bars.full(warp, cc % S), static_cast<uint32_t>((cc / S) & 1));
  }
}

// ------------------------------------------------------------------ consumer warps
// Streams the warp's chunks, runs the per-group math and hands one 16 x T
// partial per job to the epilogue.  Lane 0 issued chunks 0 .. wstages-1
// before the call (see the kernel body).
template <int BITS, int ROUTE, int NT>
__device__ void consumer(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                         const Work& wk, const Slice& sl, int warp, int lane, int issued) {
  constexpr int kBlock = 128 * BITS;
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  const int cg = a.chunk_groups;
  const int S = a.wstages;
  const int total = wk.njobs * sl.nch;
  const uint32_t ring = smem_addr(smem + a.off_ring) + warp * S * a.wstage_bytes;
  const uint8_t* ring_ptr = smem + a.off_ring + warp * S * a.wstage_bytes;
  const uint64_t policy = l2_evict_first_policy();
  float* red = reinterpret_cast<float*>(smem + a.off_red);

  // MMA route: x fragments of token 8 nb + q, or the zero area if absent.
  const uint8_t* xbase[NT];
  int xstep[NT];
  if constexpr (ROUTE == kRouteMma) {
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      const bool v = 8 * nb + q < T;
      xbase[nb] = v ? smem + a.off_x + 1024 * nb + 32 * lane : smem + kZeroAreaOffset;
      xstep[nb] = v ? T * 128 : 0;
    }
  }
  const uint8_t* xf = smem + a.off_x + 64 * r;  // FMA route: entry (g, t, r) at (g T + t) 256 + 64 r

  int c = 0, stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int j = 0; j < wk.njobs && ok; ++j) {
    float acc[NT][4];
    float facc[2][NT];
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
      facc[0][nb] = facc[1][nb] = 0.f;
    }
    for (int ci = 0; ci < sl.nch; ++ci, ++c) {
      if (!wt.wait_warp<false>(bars.full(warp, stage), phase)) { ok = false; break; }
      const uint8_t* slot = ring_ptr + stage * a.wstage_bytes;
      const uint8_t* scb = slot + cg * kBlock;
      const int g0 = sl.gs + ci * cg;
      const int n = min(cg, sl.ge - g0);
      const int gx0 = g0 - wk.g_begin;
      int i = 0;
      if constexpr (ROUTE == kRouteMma) {
        for (; i + 1 < n; i += 2) {
          const uint8_t* xp0[NT];
          const uint8_t* xp1[NT];
#pragma unroll
          for (int nb = 0; nb < NT; ++nb) {
            xp0[nb] = xbase[nb] + (gx0 + i) * xstep[nb];
            xp1[nb] = xbase[nb] + (gx0 + i + 1) * xstep[nb];
          }
          mma_group<BITS, NT>(slot + i * kBlock, scb + i * kScaleBytesPerBlock, xp0, lane, q, acc);
          mma_group<BITS, NT>(slot + (i + 1) * kBlock, scb + (i + 1) * kScaleBytesPerBlock, xp1,
                              lane, q, acc);
        }
        if (i < n) {
          const uint8_t* xp0[NT];
#pragma unroll
          for (int nb = 0; nb < NT; ++nb) xp0[nb] = xbase[nb] + (gx0 + i) * xstep[nb];
          mma_group<BITS, NT>(slot + i * kBlock, scb + i * kScaleBytesPerBlock, xp0, lane, q, acc);
        }
      } else {
        for (; i < n; ++i)
          ffma_group<BITS, NT>(slot + i * kBlock, scb + i * kScaleBytesPerBlock,
                               xf + (gx0 + i) * T * 256, lane, q, T, facc);
      }
      // Every lane has read the slot: refill it with the chunk S ahead.
      __syncwarp();
      if (lane == 0 && c + S < total) {
        fence_proxy_async_smem();
        issue_chunk<BITS>(a, wk, sl, c + S, ring + stage * a.wstage_bytes, bars.full(warp, stage),
                          policy);
        ++issued;
      }
      if (++stage == S) { stage = 0; phase ^= 1; }
    }
    if (!ok) break;
    if constexpr (ROUTE == kRouteFfma) {
      // Sum the four lanes of a row quad (fixed butterfly order).
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v = facc[h][t];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          facc[h][t] = v;
        }
      }
    }
    // Hand the 16 x T partial of this warp to the epilogue warp.
    const int b = j & 1;
    const uint32_t nuse = static_cast<uint32_t>(j >> 1);
    if (!wt.wait_warp<false>(bars.red_empty(b), (nuse & 1u) ^ 1u)) { ok = false; break; }
    float* slotp = red + (b * kWarps + warp) * 16 * T;
    if constexpr (ROUTE == kRouteMma) {
#pragma unroll
      for (int nb = 0; nb < NT; ++nb) {
        const int t0 = 8 * nb + 2 * r;
        if (t0 < T) {
          slotp[t0 * 16 + q] = acc[nb][0];
          slotp[t0 * 16 + q + 8] = acc[nb][2];
        }
        if (t0 + 1 < T) {
          slotp[(t0 + 1) * 16 + q] = acc[nb][1];
          slotp[(t0 + 1) * 16 + q + 8] = acc[nb][3];
        }
      }
    } else {
      if (r == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < T) {
            slotp[t * 16 + q] = facc[0][t];
            slotp[t * 16 + q + 8] = facc[1][t];
          }
        }
      }
    }
    mbar_arrive(bars.red_full(b));  // every lane: count = 32 per warp
  }
  // Wind down: never leave bulk copies in flight into this CTA's shared
  // memory.  In normal operation every issued chunk has been consumed.
  if (lane == 0 && issued > c) {
    volatile int no_abort = 0;
    const Waiter drain{&no_abort, wt.limit, wt.status};
    for (int cc = c; cc < issued; ++cc)
      (void)drain.wait<false>(bars.full(warp, cc % S), static_cast<uint32_t>((cc / S) & 1));
  }
}

// ------------------------------------------------------------------ epilogue
__device__ inline void epilogue(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                         const Work& wk, int lane) {
  const int T = a.T;
  const int nv = 16 * T;             // values per row tile
  const int ks = a.ksplit;
  const float* red = reinterpret_cast<const float*>(smem + a.off_red);
  float* cl = reinterpret_cast<float*>(smem + a.off_cl);
  for (int j = 0; j < wk.njobs; ++j) {
    const int b = j & 1;
    const uint32_t n = static_cast<uint32_t>(j >> 1);
    if (!wt.wait_warp<false>(bars.red_full(b), n & 1u)) return;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      float s = 0.f;
      if (e < nv) {
        const float* p = red + b * kWarps * nv + e;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += p[w * nv];
      }
      v[i] = s;
    }
    mbar_arrive(bars.red_empty(b));  // every lane: count 32
    if (ks > 1) {
      if (wk.rank != 0) {
        if (!wt.wait_warp<true>(bars.cl_empty(b), (n & 1u) ^ 1u)) return;
        const uint32_t dst0 =
            map_to_rank(smem_addr(cl + (b * (ks - 1) + (wk.rank - 1)) * nv), 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = lane + 32 * i;
          if (e < nv) st_cluster_f32(dst0 + 4 * e, v[i]);
        }
        mbar_arrive_remote(map_to_rank(bars.cl_full(b), 0));
        continue;
      }
      if (!wt.wait_warp<true>(bars.cl_full(b), n & 1u)) return;
      for (int p = 1; p < ks; ++p) {
        const float* src = cl + (b * (ks - 1) + (p - 1)) * nv;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = lane + 32 * i;
          if (e < nv) v[i] += src[e];
        }
      }
      for (int p = 1; p < ks; ++p) mbar_arrive_remote(map_to_rank(bars.cl_empty(b), p));
    }
    const long long row0 = (wk.rt_begin + j) * 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < nv) {
        const int tok = e >> 4, row = e & 15;
        if (row0 + row < a.N) a.y[static_cast<long long>(tok) * a.N + row0 + row] = v[i];
      }
    }
  }
}

// ------------------------------------------------------------------ kernel
template <int BITS, int ROUTE, int NTOK>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Bars bars{smem_addr(smem)};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortFlagOffset);
  const Waiter wt{abort_flag, a.wait_ns, a.status};
  const Work wk = cta_work(a);

  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int s = 0; s < a.wstages; ++s) mbar_init(bars.full(w, s), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.red_full(b), 32 * kWarps);
      mbar_init(bars.red_empty(b), 32);
      mbar_init(bars.cl_full(b), 32 * (a.ksplit > 1 ? a.ksplit - 1 : 1));
      mbar_init(bars.cl_empty(b), 32);
    }
    *abort_flag = 0;
    for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t*>(smem + kZeroAreaOffset)[i] = 0u;
    fence_mbar_init();
  }
  // Later kernels of the stream may start their weight streaming once every
  // CTA of this grid is running (they wait for our completion before
  // touching x or y).
  griddep_launch_dependents();
  if (a.ksplit > 1) cluster_sync_all(); else __syncthreads();

  if (warp < kWarps) {
    const Slice sl = warp_slice(wk, warp, a.chunk_groups);
    int issued = 0;
    // Packed weights are read-only for the whole stream, so the first chunks
    // may be requested before the previous kernel has finished.
    if (lane == 0) {
      const int total = wk.njobs * sl.nch;
      const uint64_t policy = l2_evict_first_policy();
      const uint32_t ring = smem_addr(smem + a.off_ring) + warp * a.wstages * a.wstage_bytes;
      for (; issued < a.wstages && issued < total; ++issued)
        issue_chunk<BITS>(a, wk, sl, issued, ring + issued * a.wstage_bytes,
                          bars.full(warp, issued), policy);
    }
    griddep_wait();
    if constexpr (ROUTE == kRouteMma && NTOK == kNtokXreg) {
      consumer_xreg<BITS, kXregMaxGroups>(a, smem, bars, wt, wk, sl, warp, lane, issued);
    } else {
      if constexpr (ROUTE == kRouteMma) {
        stage_x_bf16(a, smem, wk, threadIdx.x, kWarps * 32);
      } else {
        stage_x_f32(a, smem, wk, threadIdx.x, kWarps * 32);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
      consumer<BITS, ROUTE, NTOK>(a, smem, bars, wt, wk, sl, warp, lane, issued);
    }
  } else {
    griddep_wait();
    epilogue(a, smem, bars, wt, wk, lane);
  }
  // No CTA may leave while cluster peers can still write into its shared
  // memory or arrive on its barriers.
  __syncwarp();
  if (a.ksplit > 1) cluster_sync_all();
}

}  // namespace nq
