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
//   warp 0..7  consumers : decode the codes of one group per step, contract
//                          with the x tile (bf16 MMA m16n8k16 or fp32 FMA),
//                          scale the 64-wide partial by the group's FP16 scale;
//   warp 8     producer  : one thread streams the packed weight blocks and
//                          their scales with 1-D bulk copies (TMA engine) into
//                          a ring of shared-memory stages, L2 evict-first;
//   warp 9     epilogue  : sums the consumers' per-warp partials of a row tile
//                          in a fixed order, adds the partials of the other
//                          CTAs of its cluster (K split, distributed shared
//                          memory, rank order) and stores y.
//
// Work split: a persistent grid of clusters of KS CTAs.  Cluster c owns a
// contiguous range of 16-row tiles ("jobs"); rank q of the cluster handles
// groups [q G / KS, (q+1) G / KS) of every job.  The x slice of a CTA is
// loaded once into shared memory, permuted into MMA B-fragment order.
// Every wait is bounded by a time limit; on expiry the kernel records
// NQ_ETIMEOUT in the status word and winds down without hanging.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "layout.h"
#include "ptx.cuh"

namespace nq {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp = kConsumerWarps + 1;
constexpr int kMaxStages = 24;
constexpr int kStatusTimeout = -5;

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
  int stage_groups;        // groups per pipeline stage
  int stages;              // ring depth
  int stage_bytes;         // bytes of one stage (codes + scales, 128-aligned)
  int off_stage, off_red, off_cl, off_x;  // shared-memory offsets
  unsigned long long wait_ns;
  int* status;
};

// Shared-memory map of the barrier region (first 1 KiB).
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (kMaxStages + s); }
  __device__ uint32_t red_full(int b) const { return base + 8 * (2 * kMaxStages + b); }
  __device__ uint32_t red_empty(int b) const { return base + 8 * (2 * kMaxStages + 2 + b); }
  __device__ uint32_t cl_full(int b) const { return base + 8 * (2 * kMaxStages + 4 + b); }
  __device__ uint32_t cl_empty(int b) const { return base + 8 * (2 * kMaxStages + 6 + b); }
};
constexpr int kAbortFlagOffset = 8 * (2 * kMaxStages + 8);
constexpr int kBarRegionBytes = 1024;
static_assert(kAbortFlagOffset + 4 <= kBarRegionBytes, "barrier region");

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

// ------------------------------------------------------------------ producer
template <int BITS>
__device__ void producer(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                         const Work& wk) {
  constexpr int kBlock = 128 * BITS;
  const uint64_t policy = l2_evict_first_policy();
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, last_par = 0;  // per-stage bookkeeping for the wind-down
  bool ok = true;
  for (int j = 0; j < wk.njobs && ok; ++j) {
    const long long rt = wk.rt_begin + j;
    for (int g0 = wk.g_begin; g0 < wk.g_end; g0 += a.stage_groups) {
      const int ng = min(a.stage_groups, wk.g_end - g0);
      if (!wt.wait<false>(bars.empty(stage), phase ^ 1)) { ok = false; break; }
      const uint32_t bc = static_cast<uint32_t>(ng * kBlock);
      const uint32_t bs = static_cast<uint32_t>(ng * kScaleBytesPerBlock);
      const uint32_t dst = smem_addr(smem + a.off_stage + stage * a.stage_bytes);
      mbar_arrive_expect_tx(bars.full(stage), bc + bs);
      const long long blk = rt * a.G + g0;
      bulk_g2s(dst, a.codes + blk * kBlock, bc, bars.full(stage), policy);
      bulk_g2s(dst + a.stage_groups * kBlock, a.scales + blk * 16, bs, bars.full(stage), policy);
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
  }
  // Wind down: never leave the CTA with bulk copies in flight into its
  // shared memory.  In normal operation every stage is already complete.
  volatile int no_abort = 0;
  const Waiter drain{&no_abort, wt.limit, wt.status};
  for (int s = 0; s < a.stages; ++s)
    if (issued & (1u << s)) (void)drain.wait<false>(bars.full(s), (last_par >> s) & 1u);
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

// bf16x2 of the signed codes of pair p (exact small integers).
template <int BITS>
__device__ __forceinline__ uint32_t pair_codes_bf16(const uint32_t (&w)[BITS], int p) {
  return fma_bf16x2(pair_field<BITS>(w, p) | kBf16Magic2, kBf16One2, bf16_neg_bias2(BITS));
}

// ------------------------------------------------------------------ consumers
template <int BITS, int NT>
__device__ void consumer_mma(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                             const Work& wk, int warp, int lane) {
  constexpr int kBlock = 128 * BITS;
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  const uint8_t* xs = smem + a.off_x;
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  int stage = 0;
  uint32_t phase = 0;
  for (int j = 0; j < wk.njobs; ++j) {
    float acc[NT][4];
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    for (int g0 = wk.g_begin; g0 < wk.g_end; g0 += a.stage_groups) {
      const int ng = min(a.stage_groups, wk.g_end - g0);
      if (!wt.wait_warp<false>(bars.full(stage), phase)) return;
      const uint8_t* st = smem + a.off_stage + stage * a.stage_bytes;
      for (int gl = warp; gl < ng; gl += kConsumerWarps) {
        uint32_t w[BITS];
        load_lane_words<BITS>(st + gl * kBlock, lane, w);
        const uint32_t sp = *reinterpret_cast<const uint32_t*>(
            st + a.stage_groups * kBlock + gl * kScaleBytesPerBlock + 4 * q);
        const int gx = g0 - wk.g_begin + gl;
        uint4 xa[NT], xb[NT];
#pragma unroll
        for (int nb = 0; nb < NT; ++nb) {
          const int tok = 8 * nb + q;
          if (tok < T) {
            const uint8_t* e = xs + ((gx * T + tok) * 4 + r) * 32;
            xa[nb] = *reinterpret_cast<const uint4*>(e);
            xb[nb] = *reinterpret_cast<const uint4*>(e + 16);
          } else {
            xa[nb] = make_uint4(0, 0, 0, 0);
            xb[nb] = make_uint4(0, 0, 0, 0);
          }
        }
        float d[NT][4];
#pragma unroll
        for (int nb = 0; nb < NT; ++nb) d[nb][0] = d[nb][1] = d[nb][2] = d[nb][3] = 0.f;
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
            mma_16816(d[nb], a0, a1, a2, a3, b0, b1);
          }
        }
        const float s_lo = half_lo_to_float(sp), s_hi = half_hi_to_float(sp);
#pragma unroll
        for (int nb = 0; nb < NT; ++nb) {
          acc[nb][0] = fmaf(s_lo, d[nb][0], acc[nb][0]);
          acc[nb][1] = fmaf(s_lo, d[nb][1], acc[nb][1]);
          acc[nb][2] = fmaf(s_hi, d[nb][2], acc[nb][2]);
          acc[nb][3] = fmaf(s_hi, d[nb][3], acc[nb][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(stage));
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
    // Hand the 16 x T partial of this warp to the epilogue warp.
    const int b = j & 1;
    const uint32_t n = static_cast<uint32_t>(j >> 1);
    if (!wt.wait_warp<false>(bars.red_empty(b), (n & 1u) ^ 1u)) return;
    float* slot = red + (b * kConsumerWarps + warp) * 16 * T;
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      const int t0 = 8 * nb + 2 * r;
      if (t0 < T) {
        slot[t0 * 16 + q] = acc[nb][0];
        slot[t0 * 16 + q + 8] = acc[nb][2];
      }
      if (t0 + 1 < T) {
        slot[(t0 + 1) * 16 + q] = acc[nb][1];
        slot[(t0 + 1) * 16 + q + 8] = acc[nb][3];
      }
    }
    mbar_arrive(bars.red_full(b));  // every lane: count = 32 per warp
  }
}

template <int BITS, int TMAX>
__device__ void consumer_ffma(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                              const Work& wk, int warp, int lane) {
  constexpr int kBlock = 128 * BITS;
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  const uint8_t* xs = smem + a.off_x;
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  int stage = 0;
  uint32_t phase = 0;
  for (int j = 0; j < wk.njobs; ++j) {
    float acc[2][TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[0][t] = acc[1][t] = 0.f;
    for (int g0 = wk.g_begin; g0 < wk.g_end; g0 += a.stage_groups) {
      const int ng = min(a.stage_groups, wk.g_end - g0);
      if (!wt.wait_warp<false>(bars.full(stage), phase)) return;
      const uint8_t* st = smem + a.off_stage + stage * a.stage_bytes;
      for (int gl = warp; gl < ng; gl += kConsumerWarps) {
        uint32_t w[BITS];
        load_lane_words<BITS>(st + gl * kBlock, lane, w);
        const uint32_t sp = *reinterpret_cast<const uint32_t*>(
            st + a.stage_groups * kBlock + gl * kScaleBytesPerBlock + 4 * q);
        const int gx = g0 - wk.g_begin + gl;
        float part[2][TMAX];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) part[0][t] = part[1][t] = 0.f;
#pragma unroll
        for (int js = 0; js < 4; ++js) {
          float xv[TMAX][4];
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
              const float4 v =
                  *reinterpret_cast<const float4*>(xs + ((gx * T + t) * 4 + r) * 64 + 16 * js);
              xv[t][0] = v.x;
              xv[t][1] = v.y;
              xv[t][2] = v.z;
              xv[t][3] = v.w;
            } else {
              xv[t][0] = xv[t][1] = xv[t][2] = xv[t][3] = 0.f;
            }
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
        const float s_lo = half_lo_to_float(sp), s_hi = half_hi_to_float(sp);
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          acc[0][t] = fmaf(s_lo, part[0][t], acc[0][t]);
          acc[1][t] = fmaf(s_hi, part[1][t], acc[1][t]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(stage));
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
    // Sum the four lanes of a row quad (fixed butterfly order).
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v = acc[h][t];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        acc[h][t] = v;
      }
    }
    const int b = j & 1;
    const uint32_t n = static_cast<uint32_t>(j >> 1);
    if (!wt.wait_warp<false>(bars.red_empty(b), (n & 1u) ^ 1u)) return;
    float* slot = red + (b * kConsumerWarps + warp) * 16 * T;
    if (r == 0) {
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          slot[t * 16 + q] = acc[0][t];
          slot[t * 16 + q + 8] = acc[1][t];
        }
      }
    }
    mbar_arrive(bars.red_full(b));
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
        const float* p = red + b * kConsumerWarps * nv + e;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) s += p[w * nv];
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
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.red_full(b), 32 * kConsumerWarps);
      mbar_init(bars.red_empty(b), 32);
      mbar_init(bars.cl_full(b), 32 * (a.ksplit > 1 ? a.ksplit - 1 : 1));
      mbar_init(bars.cl_empty(b), 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Later kernels of the stream may start their weight streaming once every
  // CTA of this grid is running (they wait for our completion before
  // touching x or y).
  griddep_launch_dependents();
  if (a.ksplit > 1) cluster_sync_all(); else __syncthreads();

  if (warp == kProducerWarp) {
    // Packed weights are read-only for the whole stream, so streaming them
    // may overlap the tail of the previous kernel.
    if (lane == 0) producer<BITS>(a, smem, bars, wt, wk);
  } else if (warp == kEpilogueWarp) {
    griddep_wait();
    epilogue(a, smem, bars, wt, wk, lane);
  } else {
    griddep_wait();
    if constexpr (ROUTE == kRouteMma) {
      stage_x_bf16(a, smem, wk, threadIdx.x, kConsumerWarps * 32);
    } else {
      stage_x_f32(a, smem, wk, threadIdx.x, kConsumerWarps * 32);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if constexpr (ROUTE == kRouteMma) {
      consumer_mma<BITS, NTOK>(a, smem, bars, wt, wk, warp, lane);
    } else {
      consumer_ffma<BITS, NTOK>(a, smem, bars, wt, wk, warp, lane);
    }
  }
  // No CTA may leave while cluster peers can still write into its shared
  // memory or arrive on its barriers.
  __syncwarp();
  if (a.ksplit > 1) cluster_sync_all();
}

}  // namespace nq
