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
//   warp 0..15 consumers : decode the codes of their groups in registers,
//                          contract them with x (bf16 MMA m16n8k16, or fp32
//                          FMA) and scale each 64-wide partial by the group's
//                          FP16 scale;
//   warp 16    producer  : one thread streams the weight stream in large
//                          stages -- the CTA's whole K range of one 16-row
//                          tile when it fits -- with two 1-D bulk copies per
//                          stage (codes, scales; TMA engine, L2 evict-first)
//                          into a ring of shared-memory stages;
//   warp 17,18 epilogue  : taking jobs in turn, sum the 16 per-warp partials
//                          of a row tile in a fixed order, add the partials of
//                          the other CTAs of the cluster (K split,
//                          asynchronous distributed shared-memory stores, rank
//                          order) and store y.
//
// Few large copies matter: the bulk-copy engine of an SM serves a limited
// number of requests per microsecond, so small per-warp copies cap the
// stream well below the HBM rate.  Work split: a persistent grid of clusters
// of KS CTAs; cluster c owns a contiguous range of 16-row tiles ("jobs");
// rank q handles groups [q G / KS, (q+1) G / KS) of every job.  When the
// slices are short (up to 5 groups per warp for T <= 8, 3 for T <= 16) each
// consumer warp owns a fixed slice of those groups and keeps its x fragments
// in registers ("x in registers"); otherwise the CTA's x slice sits in shared
// memory in B-fragment order, and the warps take the groups of a
// stage in turn.  With x in registers, 4-bit codes take an fp16 route: x is
// staged once as fp16 scaled by a power of two per token (exact, checked;
// else the bf16 route), which lets the decode reach two nibbles per half
// without a shift.  Every wait is bounded by a time limit; on
// expiry the kernel records NQ_ETIMEOUT in the status word and winds down
// without hanging or leaving bulk copies in flight.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "layout.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace nq {

constexpr int kWarps = 16;                   // consumer warps
constexpr int kProducerWarp = kWarps;
constexpr int kEpilogueWarp = kWarps + 1;     // first of kEpiWarps epilogue warps
constexpr int kEpiWarps = 2;                  // epilogue warps, taking jobs in turn
constexpr int kThreads = (kWarps + 1 + kEpiWarps) * 32;
constexpr int kMaxStages = 16;               // stages of the shared-memory ring
constexpr int kMaxBufs = 8;                  // partial-sum buffers (warps -> epilogue, peers -> rank 0)
constexpr int kStatusTimeout = -5;
// Kernel variants (template NTOK): MMA route with 1 or 2 token blocks of 8 and
// x in shared memory, kNtokXreg (MMA, one token block, x in registers, at
// most kXregMaxGroups groups per warp slice), FMA route: NTOK = max tokens.
constexpr int kNtokXreg = 3;
constexpr int kXregMaxGroups = 5;  // (the slice-length dispatch covers 1..5)
// kNtokXreg2: two token blocks (T <= 16), x in registers, at most
// kXreg2MaxGroups groups per warp slice.
constexpr int kNtokXreg2 = 4;
constexpr int kXreg2MaxGroups = 3;
// kNtokXregH: two token blocks (8 < T <= 16) with the first block's x in
// registers (at most kXregMaxGroups groups per warp slice, as for T <= 8) and
// the second block's x in shared memory, read per group (two 16-byte loads):
// twice the groups per warp of kNtokXreg2 for the same registers, so a
// smaller K split.
constexpr int kNtokXregH = 5;
// Row tiles per hand-off: the x-in-register consumers with one token block
// (T <= 8) take the tiles of their cluster in pairs (two ring stages, two
// accumulator sets, one partial buffer), which halves the per-job bookkeeping
// of consumers and epilogue; the other variants hand over one tile at a time
// (with two token blocks a second accumulator set costs more registers and
// buffer space than it saves).  (Route 1 is the MMA route; the FMA route's
// NTOK is its token count.)
template <int ROUTE, int NTOK>
constexpr int kJobTiles = (ROUTE == 1 && NTOK == kNtokXreg) ? 2 : 1;

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
  int stage_groups;        // 64-groups per stage (x in registers: the CTA's whole K range)
  int stages;              // ring depth
  int stage_bytes;         // bytes of one stage (codes, then scales; 128-aligned)
  int off_ring, off_red, off_cl, off_x;  // shared-memory offsets
  int off_xh;              // fp16 x staging (4-bit codes, x in registers) at the ring's
                           // tail, or -1: no fp16 route
  int xh_stage0;           // first ring stage overlapping that staging area
  int nbuf;                // partial-sum buffers in flight (<= kMaxBufs)
  unsigned long long wait_ns;
  int* status;
  // Fused verify head (h_ws != nullptr): per token t the argmax, the maximum
  // and the logsumexp of y[t, 0..N), reduced through the workspace h_ws
  // (layout: kHeadCounterBytes of arrival counters -- [0] all groups, [1 + g]
  // group g -- then one kHeadStateBytes state per (unit, epilogue warp,
  // token), then one per (group of kHeadGroup units, token); a unit is a
  // cluster, or a CTA where the K split finalises by reduce-scatter).  y may then
  // be null (logits not stored).
  uint8_t* h_ws;
  int* h_argmax;
  float* h_max;
  float* h_lse;
  // SwiGLU epilogue (act != nullptr): the matrix is a gate+up matrix packed
  // with rows interleaved per 8 (tile r = gate rows 8r..8r+7, then up rows
  // 8r..8r+7), and act[t, i] = bf16(silu(gate) * up) replaces y
  // ([T, N / 2] bf16 bits, N a multiple of 16).
  uint16_t* act;
  // Top-k of the fused head (tk_k > 0, 1 <= tk_k <= kTopkMax): epilogue
  // warp w of unit c keeps, per token t, the 32 largest keys of the logits
  // it finalised in tk_lists[((c * kEpiWarps + w) * kHeadMaxT + t) * 32 ...]
  // (sorted descending; what the merge kernel reads), its candidate buffer in
  // tk_bufs (64 keys per list, same indexing), and the buffer counts in
  // shared memory at off_tk (kHeadMaxT ints per warp).
  int tk_k;
  int off_tk;
  unsigned long long* tk_lists;
  unsigned long long* tk_bufs;
  // One-launch MLP layer (nq_mlp_kernel): the gate+up phase's epilogue adds
  // the number of row tiles whose activations it has stored to sync[0]; the
  // down phase's consumers wait until sync[0] == sync_target (all of them),
  // then count themselves in sync[1], and the last CTA to pass resets both
  // words for the next launch that uses the pair.  Null for a plain GEMV.
  unsigned* sync;
  int sync_target;
};

// Position in the stage ring and the partial-buffer ring, carried from the
// gate+up phase to the down phase of the one-launch layer.
struct RingPos {
  int stage;
  uint32_t phase;
  int rb;
  uint32_t rn;
};
// Launch slots of the one-launch layer's activation counters (per device):
// launches issued while a stream is captured into a CUDA graph take slots of
// their own pool, so a graph's baked-in slots are never handed to ordinary
// launches; a slot is reused after kSyncSlotsEager (kSyncSlotsCapture) more
// launches of its pool.
constexpr int kSyncSlotsEager = 1024;
constexpr int kSyncSlotsCapture = 4096;
constexpr int kSyncSlots = kSyncSlotsEager + kSyncSlotsCapture;
constexpr int kHeadCounterBytes = 256;
constexpr int kHeadStateBytes = 16;
constexpr int kHeadMaxT = 16;
constexpr int kHeadGroup = 8;       // units (clusters or CTAs) merged per group (first level)
constexpr int kHeadMaxGroups = 32;  // groups the second level covers (256 units)

// Shared-memory map of the barrier region (first 1 KiB).
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (kMaxStages + s); }
  __device__ uint32_t red_full(int b) const { return base + 8 * (2 * kMaxStages + b); }
  __device__ uint32_t red_empty(int b) const { return base + 8 * (2 * kMaxStages + kMaxBufs + b); }
  __device__ uint32_t cl_full(int b) const { return base + 8 * (2 * kMaxStages + 2 * kMaxBufs + b); }
  __device__ uint32_t cl_empty(int b) const { return base + 8 * (2 * kMaxStages + 3 * kMaxBufs + b); }
};
constexpr int kAbortFlagOffset = 8 * (2 * kMaxStages + 4 * kMaxBufs);
constexpr int kZeroAreaOffset = kAbortFlagOffset + 32;  // 32 zero bytes: x of absent tokens
constexpr int kXFreeBarOffset = kZeroAreaOffset + 32;   // mbarrier: consumers done with x staging
// fp16 x staging statistics: [t] largest |x| bit pattern of token t, [16 + t]
// smallest nonzero one, [32] set when some token cannot take the fp16 route.
constexpr int kXStatOffset = kXFreeBarOffset + 64;
constexpr int kBarRegionBytes = 1024;
static_assert(kXStatOffset + 33 * 4 <= kBarRegionBytes, "barrier region");

struct Waiter {
  volatile int* abort;
  unsigned long long limit;
  int* status;

  // Bounded wait for the completion of the phase with parity `par`.
  // kPoll: probe without suspending (barriers completed by thread arrivals,
  // where a suspended waiter may be woken late); otherwise try_wait (bulk-copy
  // completion).
  template <bool kClusterScope, bool kPoll = false>
  __device__ bool wait(uint32_t bar, uint32_t par) const {
    auto probe = [&]() {
      if constexpr (kClusterScope) return mbar_test_wait_cluster(bar, par);
      else if constexpr (kPoll) return mbar_test_wait(bar, par);
      else return mbar_try_wait(bar, par);
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
  template <bool kClusterScope, bool kPoll = false>
  __device__ bool wait_warp(uint32_t bar, uint32_t par) const {
    const bool ok = wait<kClusterScope, kPoll>(bar, par);
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
  // Contiguous row tiles per cluster; the Nt mod clusters extra tiles go to
  // the lowest cluster indices.  The grid's CTAs come up in block-index
  // order over the first 2-4 us, so the first clusters also start first:
  // on GB300 this ends the launch 1-3 % sooner than spreading the extras
  // evenly (27B shapes; gate+up 18.55 -> 18.36 us at T = 1, down 13.24 ->
  // 12.85 us for 4-bit codes at T = 1).
  const long long nt = a.Nt, base = nt / a.clusters, rem = nt % a.clusters;
  w.rt_begin = cl * base + min(static_cast<long long>(cl), rem);
  w.njobs = static_cast<int>(base + (cl < rem ? 1 : 0));
  w.g_begin = (w.rank * a.G) / ks;
  w.g_end = ((w.rank + 1) * a.G) / ks;
  return w;
}

// The fixed K slice of consumer warp `warp` (x in registers): groups
// [gs, ge) of every job.  When the CTA's groups do not divide evenly, the
// last (gc mod 16) warps take one group more: consecutive warps sit on the
// four SM sub-partitions in turn (warp mod 4), so the extra groups spread
// evenly over them instead of piling up on one sub-partition.
struct Slice {
  int gs, ge;
};
__device__ __forceinline__ Slice warp_slice(const Work& wk, int warp) {
  const int gc = wk.g_end - wk.g_begin;
  const int base = gc / kWarps, first_extra = kWarps - gc % kWarps;
  Slice s;
  s.gs = wk.g_begin + warp * base + max(0, warp - first_extra);
  s.ge = s.gs + base + (warp >= first_extra ? 1 : 0);
  return s;
}

// ------------------------------------------------------------------ producer
// One thread: stage after stage, the codes and the scales of groups
// [g0, g0 + ng) of one job, two bulk copies per stage.
template <int BITS>
__device__ void producer(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                         const Work& wk) {
  constexpr int kBlock = 128 * BITS;
  const uint64_t policy = l2_evict_first_policy();
  const uint32_t ring = smem_addr(smem + a.off_ring);
  const int sg = a.stage_groups;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, last_par = 0;  // per-stage bookkeeping for the wind-down
  bool ok = true;
  // Stages from xh_stage0 on share their bytes with the consumers' fp16 x
  // staging: their first fill waits until every consumer warp has taken its
  // x fragments (the fence orders those generic accesses before the copies).
  bool x_pending = a.off_xh >= 0;
  for (int j = 0; j < wk.njobs && ok; ++j) {
    const long long blk_job = (wk.rt_begin + j) * a.G;
    for (int g0 = wk.g_begin; g0 < wk.g_end; g0 += sg) {
      const int ng = min(sg, wk.g_end - g0);
      if (!wt.wait<false>(bars.empty(stage), phase ^ 1)) { ok = false; break; }
      if (x_pending && stage >= a.xh_stage0) {
        if (!wt.wait<false>(smem_addr(smem + kXFreeBarOffset), 0)) { ok = false; break; }
        fence_proxy_async_smem();
        x_pending = false;
      }
      const uint32_t bc = static_cast<uint32_t>(ng * kBlock);
      const uint32_t bs = static_cast<uint32_t>(ng * kScaleBytesPerBlock);
      const uint32_t dst = ring + stage * a.stage_bytes;
      const long long blk = blk_job + g0;
      mbar_arrive_expect_tx(bars.full(stage), bc + bs);
      bulk_g2s(dst, a.codes + blk * kBlock, bc, bars.full(stage), policy);
      bulk_g2s(dst + sg * kBlock, a.scales + blk * 16, bs, bars.full(stage), policy);
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
// K slices j of group g for lane r: words 2j, 2j + 1 = x[tok][16r + 4j ..
// 16r + 4j + 3] (bf16 pairs, the layout's K order), i.e. the 32 bytes of x
// at k = 16r .. 16r + 15 of the group.  The entry's two halves (slices 0-1,
// slices 2-3) sit in two planes, 16 bytes per entry each, the second plane
// gc T 64 bytes after the first: a lane's 16-byte reads of one plane are then
// consecutive across lanes (32-byte entries would make every 16-byte read
// 2-way bank conflicted).
__device__ inline void stage_x_bf16(const GemvArgs& a, uint8_t* smem, const Work& wk, int ctid,
                             int nthreads) {
  const int gc = wk.g_end - wk.g_begin;
  const int total = gc * a.T * 4;
  uint8_t* xs = smem + a.off_x;
  const int hb = gc * a.T * 64;  // second plane
  for (int e = ctid; e < total; e += nthreads) {
    const int g = e / (a.T * 4);
    const int rem = e - g * a.T * 4;
    const int tok = rem >> 2, r = rem & 3;
    const uint4* src = reinterpret_cast<const uint4*>(
        a.x + static_cast<long long>(tok) * a.K + 64LL * (wk.g_begin + g) + 16 * r);
    const int off = ((g * a.T + tok) * 4 + r) * 16;
    *reinterpret_cast<uint4*>(xs + off) = __ldg(src);
    *reinterpret_cast<uint4*>(xs + hb + off) = __ldg(src + 1);
  }
}

// FMA route: entry (g, tok, r) = 16 floats, [4j + m] = x[tok][16r + 4j + m]
// (the layout's K order: pair i of K slice j multiplies [4j + 2 (i / 2) + c]).
__device__ inline void stage_x_f32(const GemvArgs& a, uint8_t* smem, const Work& wk, int ctid,
                            int nthreads) {
  const int gc = wk.g_end - wk.g_begin;
  const int total = gc * a.T * 4;
  uint8_t* xs = smem + a.off_x;
  for (int e = ctid; e < total; e += nthreads) {
    const int g = e / (a.T * 4);
    const int rem = e - g * a.T * 4;
    const int tok = rem >> 2, r = rem & 3;
    const uint4* src = reinterpret_cast<const uint4*>(
        a.x + static_cast<long long>(tok) * a.K + 64LL * (wk.g_begin + g) + 16 * r);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float4* dst = reinterpret_cast<float4*>(xs + ((g * a.T + tok) * 4 + r) * 64);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float4 o;
      o.x = __uint_as_float(w[2 * m] << 16);
      o.y = __uint_as_float(w[2 * m] & 0xFFFF0000u);
      o.z = __uint_as_float(w[2 * m + 1] << 16);
      o.w = __uint_as_float(w[2 * m + 1] & 0xFFFF0000u);
      dst[m] = o;
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
  } else if constexpr (BITS == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(blk + 512 + 16 * lane);
    w[4] = u.x;
    w[5] = u.y;
    w[6] = u.z;
    w[7] = u.w;
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

// fp16 route for 4-bit codes (x in registers, converted once to fp16): with
// exponent 2^10 the 10-bit fp16 mantissa holds a nibble at bits 0-3 or at
// bits 4-7 of each half as it lies: (w & 0x000F000F) | 1024 = 1024 + u and
// (w & 0x00F000F0) | 1024 = 1024 + 16 u.  One shift by 8 serves the other two
// nibbles of the word (the bf16 route needs three shifts per word).
// Subtracting 1024 + 8, resp. 1024 + 128, leaves c and 16 c, exact in fp16.
// The nibbles at offsets 4 and 12 are pairs 1 and 3 of the word -- rows q + 8
// of the tile -- so those rows leave the MMA multiplied by 16, which the warp
// undoes exactly (a power of two) when it hands its partial over.
__device__ __forceinline__ void q4_codes_f16(uint32_t w, uint32_t& a0, uint32_t& a1,
                                             uint32_t& a2, uint32_t& a3) {
  constexpr uint32_t kMagic = 0x64006400u;  // 1024
  constexpr uint32_t kLo = 0x64086408u;     // 1024 + 8
  constexpr uint32_t kHi = 0x64806480u;     // 1024 + 128
  const uint32_t w8 = w >> 8;
  a0 = sub_f16x2(lop3_and_or(w, 0x000F000Fu, kMagic), kLo);
  a1 = sub_f16x2(lop3_and_or(w, 0x00F000F0u, kMagic), kHi);
  a2 = sub_f16x2(lop3_and_or(w8, 0x000F000Fu, kMagic), kLo);
  a3 = sub_f16x2(lop3_and_or(w8, 0x00F000F0u, kMagic), kHi);
}

// 8-bit codes: bf16 has 7 mantissa bits, so each biased code u = c + 128 is
// split into its low nibble (0..15) and its high nibble minus 8 (-8..7):
// c = 16 (hi - 8) + lo.  Both planes decode like 4-bit codes (one lop3 and one
// bf16x2 subtract each); the group runs two MMA chains and combines them as
// 16 D_hi + D_lo before the scale.
__device__ __forceinline__ void q8_pair_planes(const uint32_t (&w)[8], int p, uint32_t& lo,
                                               uint32_t& hi) {
  const uint32_t x = w[p >> 1] >> (8 * (p & 1));
  const uint32_t xl = lop3_and_or(x, 0x000F000Fu, kBf16Magic2);        // 128 + lo
  const uint32_t xh = lop3_and_or(x >> 4, 0x000F000Fu, kBf16Magic2);   // 128 + hi
  const __nv_bfloat162 vlo =
      __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&xl),
              __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300)));  // - 128
  const __nv_bfloat162 vhi =
      __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&xh),
              __halves2bfloat162(__ushort_as_bfloat16(0x4308), __ushort_as_bfloat16(0x4308)));  // - 136
  lo = *reinterpret_cast<const uint32_t*>(&vlo);
  hi = *reinterpret_cast<const uint32_t*>(&vhi);
}

// ------------------------------------------------------------------ per-group math
// One group of one row tile on the MMA route: decode the lane's 32 codes, four
// chained MMAs against the x fragments (the first starts from zero), scale,
// accumulate.  xp[nb]: x fragments of K slices 0-1 of token block nb for this
// lane, xp[nb] + xh[nb] those of slices 2-3 (zeros if the token is absent).
template <int BITS, int NT>
__device__ __forceinline__ void mma_group(const uint8_t* blk, const uint8_t* sc,
                                          const uint8_t* const (&xp)[NT], const int (&xh)[NT],
                                          int lane, int q, float (&acc)[NT][4]) {
  uint32_t w[BITS];
  load_lane_words<BITS>(blk, lane, w);
  const __half2 sh = *reinterpret_cast<const __half2*>(sc + 4 * q);
  uint4 xa[NT], xb[NT];
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) {
    xa[nb] = *reinterpret_cast<const uint4*>(xp[nb]);
    xb[nb] = *reinterpret_cast<const uint4*>(xp[nb] + xh[nb]);
  }
  float d[NT][4], dh[NT][4];   // dh: high-nibble plane of 8-bit codes
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    uint32_t a0, a1, a2, a3, h0 = 0, h1 = 0, h2 = 0, h3 = 0;
    if constexpr (BITS == 8) {
      q8_pair_planes(w, 4 * js + 0, a0, h0);
      q8_pair_planes(w, 4 * js + 1, a1, h1);
      q8_pair_planes(w, 4 * js + 2, a2, h2);
      q8_pair_planes(w, 4 * js + 3, a3, h3);
    } else {
      a0 = pair_codes_bf16<BITS>(w, 4 * js + 0);
      a1 = pair_codes_bf16<BITS>(w, 4 * js + 1);
      a2 = pair_codes_bf16<BITS>(w, 4 * js + 2);
      a3 = pair_codes_bf16<BITS>(w, 4 * js + 3);
    }
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      const uint32_t b0 = js == 0 ? xa[nb].x : js == 1 ? xa[nb].z : js == 2 ? xb[nb].x : xb[nb].z;
      const uint32_t b1 = js == 0 ? xa[nb].y : js == 1 ? xa[nb].w : js == 2 ? xb[nb].y : xb[nb].w;
      if (js == 0) {
        mma_16816_zc(d[nb], a0, a1, a2, a3, b0, b1);
        if constexpr (BITS == 8) mma_16816_zc(dh[nb], h0, h1, h2, h3, b0, b1);
      } else {
        mma_16816(d[nb], a0, a1, a2, a3, b0, b1);
        if constexpr (BITS == 8) mma_16816(dh[nb], h0, h1, h2, h3, b0, b1);
      }
    }
  }
  if constexpr (BITS == 8) {
#pragma unroll
    for (int nb = 0; nb < NT; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) d[nb][e] = fmaf(16.f, dh[nb][e], d[nb][e]);
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

// Same as mma_group with the lane's x fragments of the group held in
// registers: xr[nb][2 js] / xr[nb][2 js + 1] are B fragments b0 / b1 of K
// slice js for token block nb.
template <int BITS, int NT>
__device__ __forceinline__ void mma_group_xr(const uint8_t* blk, const uint8_t* sc,
                                             const uint32_t (&xr)[NT][8], int lane, int q,
                                             float (&acc)[NT][4]) {
  uint32_t w[BITS];
  load_lane_words<BITS>(blk, lane, w);
  const float2 s = __half22float2(*reinterpret_cast<const __half2*>(sc + 4 * q));
  float d[NT][4], dh[NT][4];   // dh: high-nibble plane of 8-bit codes
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    uint32_t a0, a1, a2, a3, h0 = 0, h1 = 0, h2 = 0, h3 = 0;
    if constexpr (BITS == 8) {
      q8_pair_planes(w, 4 * js + 0, a0, h0);
      q8_pair_planes(w, 4 * js + 1, a1, h1);
      q8_pair_planes(w, 4 * js + 2, a2, h2);
      q8_pair_planes(w, 4 * js + 3, a3, h3);
    } else {
      a0 = pair_codes_bf16<BITS>(w, 4 * js + 0);
      a1 = pair_codes_bf16<BITS>(w, 4 * js + 1);
      a2 = pair_codes_bf16<BITS>(w, 4 * js + 2);
      a3 = pair_codes_bf16<BITS>(w, 4 * js + 3);
    }
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      if (js == 0) {
        mma_16816_zc(d[nb], a0, a1, a2, a3, xr[nb][0], xr[nb][1]);
        if constexpr (BITS == 8) mma_16816_zc(dh[nb], h0, h1, h2, h3, xr[nb][0], xr[nb][1]);
      } else {
        mma_16816(d[nb], a0, a1, a2, a3, xr[nb][2 * js], xr[nb][2 * js + 1]);
        if constexpr (BITS == 8)
          mma_16816(dh[nb], h0, h1, h2, h3, xr[nb][2 * js], xr[nb][2 * js + 1]);
      }
    }
  }
  if constexpr (BITS == 8) {
#pragma unroll
    for (int nb = 0; nb < NT; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) d[nb][e] = fmaf(16.f, dh[nb][e], d[nb][e]);
  }
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) {
    acc[nb][0] = fmaf(s.x, d[nb][0], acc[nb][0]);
    acc[nb][1] = fmaf(s.x, d[nb][1], acc[nb][1]);
    acc[nb][2] = fmaf(s.y, d[nb][2], acc[nb][2]);
    acc[nb][3] = fmaf(s.y, d[nb][3], acc[nb][3]);
  }
}

// mma_group_xr on the fp16 route (4-bit codes; xr holds fp16 x * 2^e).
template <int NT>
__device__ __forceinline__ void mma_group_xr_f16(const uint8_t* blk, const uint8_t* sc,
                                                 const uint32_t (&xr)[NT][8], int lane, int q,
                                                 float (&acc)[NT][4]) {
  uint32_t w[4];
  load_lane_words<4>(blk, lane, w);
  const float2 s = __half22float2(*reinterpret_cast<const __half2*>(sc + 4 * q));
  float d[NT][4];
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    uint32_t a0, a1, a2, a3;
    q4_codes_f16(w[js], a0, a1, a2, a3);
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      if (js == 0) {
        mma_16816_f16_zc(d[nb], a0, a1, a2, a3, xr[nb][0], xr[nb][1]);
      } else {
        mma_16816_f16(d[nb], a0, a1, a2, a3, xr[nb][2 * js], xr[nb][2 * js + 1]);
      }
    }
  }
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) {
    acc[nb][0] = fmaf(s.x, d[nb][0], acc[nb][0]);
    acc[nb][1] = fmaf(s.x, d[nb][1], acc[nb][1]);
    acc[nb][2] = fmaf(s.y, d[nb][2], acc[nb][2]);
    acc[nb][3] = fmaf(s.y, d[nb][3], acc[nb][3]);
  }
}

// ------------------------------------------------------------------ consumers
// Hand a warp's 16 x T partial of job j to the epilogue (MMA accumulator
// layout: lane q*4+r holds rows q, q+8 and tokens 8 nb + 2r, +1).
// Buffer b = job % nbuf, nuse = job / nbuf (kept incrementally by the caller).
template <int NT>
__device__ __forceinline__ bool hand_partial_mma(const GemvArgs& a, uint8_t* smem,
                                                 const Bars& bars, const Waiter& wt, int warp,
                                                 int lane, int b, uint32_t nuse,
                                                 const float (&acc)[NT][4]) {
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  if (!wt.wait_warp<false>(bars.red_empty(b), (nuse & 1u) ^ 1u)) return false;
  float* slot = reinterpret_cast<float*>(smem + a.off_red) + (b * kWarps + warp) * 16 * T;
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
  return true;
}

// Hand over the partials of JT consecutive tiles (tile jt at offset jt 16 T
// of the slot); tiles past the cluster's last are zero.
template <int NT, int JT>
__device__ __forceinline__ bool hand_partials_mma(const GemvArgs& a, uint8_t* smem,
                                                  const Bars& bars, const Waiter& wt, int warp,
                                                  int lane, int b, uint32_t nuse,
                                                  const float (&acc)[JT][NT][4]) {
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  if (!wt.wait_warp<false>(bars.red_empty(b), (nuse & 1u) ^ 1u)) return false;
  float* slot = reinterpret_cast<float*>(smem + a.off_red) + (b * kWarps + warp) * JT * 16 * T;
#pragma unroll
  for (int jt = 0; jt < JT; ++jt) {
    float* st = slot + jt * 16 * T;
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      const int t0 = 8 * nb + 2 * r;
      if (t0 < T) {
        st[t0 * 16 + q] = acc[jt][nb][0];
        st[t0 * 16 + q + 8] = acc[jt][nb][2];
      }
      if (t0 + 1 < T) {
        st[(t0 + 1) * 16 + q] = acc[jt][nb][1];
        st[(t0 + 1) * 16 + q + 8] = acc[jt][nb][3];
      }
    }
  }
  mbar_arrive(bars.red_full(b));  // every lane: count = 32 per warp
  return true;
}

// NG consecutive groups of a warp slice, unrolled without branches.
template <int BITS, int NT, int GWM, int NG, bool F16>
__device__ __forceinline__ void slice_xr(const uint8_t* codes, const uint8_t* scales,
                                         const uint32_t (&xr)[GWM][NT][8], int lane, int q,
                                         float (&acc)[NT][4]) {
  if constexpr (NG <= GWM) {
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      if constexpr (F16) {
        mma_group_xr_f16<NT>(codes + i * (128 * BITS), scales + i * kScaleBytesPerBlock, xr[i],
                             lane, q, acc);
      } else {
        mma_group_xr<BITS, NT>(codes + i * (128 * BITS), scales + i * kScaleBytesPerBlock, xr[i],
                               lane, q, acc);
      }
    }
  }
}

// The lane's x fragments of the warp slice (groups i < n, tokens < T; zeros
// elsewhere), as bf16 pairs straight from x.
template <int GWM, int NT, bool CG = false>
__device__ __forceinline__ void load_x_frags(const GemvArgs& a, const Slice& sl, int n, int lane,
                                             uint32_t (&xr)[GWM][NT][8]) {
  const int q = lane >> 2, r = lane & 3;
#pragma unroll
  for (int i = 0; i < GWM; ++i) {
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
#pragma unroll
      for (int e = 0; e < 8; ++e) xr[i][nb][e] = 0u;
      const int tok = 8 * nb + q;
      if (i < n && tok < a.T) {
        // the layout's K order: the lane's fragments are x at k = 16r .. 16r + 15
        const uint4* src = reinterpret_cast<const uint4*>(
            a.x + static_cast<long long>(tok) * a.K + 64LL * (sl.gs + i) + 16 * r);
        // CG: x was written earlier in the same kernel (the layer's
        // activations), so it is read through L2, not the read-only path.
        const uint4 v0 = CG ? __ldcg(src) : __ldg(src), v1 = CG ? __ldcg(src + 1) : __ldg(src + 1);
        xr[i][nb][0] = v0.x; xr[i][nb][1] = v0.y; xr[i][nb][2] = v0.z; xr[i][nb][3] = v0.w;
        xr[i][nb][4] = v1.x; xr[i][nb][5] = v1.y; xr[i][nb][6] = v1.z; xr[i][nb][7] = v1.w;
      }
    }
  }
}

// fp16 route of 4-bit codes (taken for T <= 2, where staging x costs less
// than the shorter decode saves): the consumer warps stage the CTA's x range
// once, as fp16 pairs of x * 2^e_t with one power of two e_t per token t, in
// B-fragment order at off_xh (entry (g, t, r): 32 bytes, x at k = 16r ..
// 16r + 15 of group g for token t; the layout's K order).  e_t puts the
// token's largest |x| in [2^14, 2^15); every bf16 value then converts
// exactly when none lies more than 31 binades below it (fp16 keeps 11
// significant bits down to 2^-14 and steps of 2^-24 below), the maximum lies
// in [2^-100, 2^101) and nothing is subnormal, infinite or NaN.  Pass 1
// gathers each token's largest and smallest nonzero |x|, pass 2 converts.
// Returns, the same in every consumer thread, whether every token qualified;
// if not, the caller takes the bf16 route and the staging area is unused.
__device__ __forceinline__ int f16_exponent(uint32_t max_bits) {
  return max_bits == 0 ? 0 : 141 - static_cast<int>(max_bits >> 7);
}
__device__ inline bool stage_x_f16(const GemvArgs& a, uint8_t* smem, const Work& wk, int warp,
                                   int lane) {
  const int gc = wk.g_end - wk.g_begin;
  const int T = a.T;
  uint32_t* stat = reinterpret_cast<uint32_t*>(smem + kXStatOffset);
  const int per_tok = gc * 4;        // units of 16 values per token
  const int units = T * per_tok;     // unit u: token u / per_tok, group g, slice j
  auto src_of = [&](int u, int& tok, int& g, int& j) {
    tok = u / per_tok;
    const int rem = u - tok * per_tok;
    g = rem >> 2;
    j = rem & 3;
    return reinterpret_cast<const uint4*>(a.x + static_cast<long long>(tok) * a.K +
                                          64LL * (wk.g_begin + g) + 16 * j);
  };
  // Pass 1: per token, the largest and the smallest nonzero magnitude
  // (bf16 magnitudes order like unsigned integers; zeros count as 0x7FFF).
  for (int base = warp * 32; base < units; base += kWarps * 32) {
    const int u = base + lane;
    uint32_t mx = 0, mn = 0x7FFF7FFFu;
    int tok = T;
    if (u < units) {
      int g, j;
      const uint4* src = src_of(u, tok, g, j);
      const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t m = w[k] & 0x7FFF7FFFu;
        mx = __vmaxu2(mx, m);
        mn = __vminu2(mn, m | (__vcmpeq2(m, 0u) & 0x7FFF7FFFu));
      }
    }
    mx = max(mx & 0xFFFFu, mx >> 16);
    mn = min(mn & 0xFFFFu, mn >> 16);
    const unsigned same = __match_any_sync(0xffffffffu, tok);
    mx = __reduce_max_sync(same, mx);
    mn = __reduce_min_sync(same, mn);
    if (tok < T && lane == __ffs(same) - 1) {
      atomicMax(stat + tok, mx);
      atomicMin(stat + 16 + tok, mn);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
  // Pass 2: qualify each token, convert (the reloads hit L1).
  uint8_t* xs = smem + a.off_xh;
  for (int u = warp * 32 + lane; u < units; u += kWarps * 32) {
    int tok, g, j;
    const uint4* src = src_of(u, tok, g, j);
    const uint32_t mxb = stat[tok], mnb = stat[16 + tok];
    const int E = static_cast<int>(mxb >> 7), Emin = static_cast<int>(mnb >> 7);
    const bool ok = mxb == 0 || (E >= 27 && E <= 227 && Emin >= 1 && Emin >= E - 31);
    if (!ok) {
      stat[32] = 1u;
      continue;
    }
    const float sc = __int_as_float((127 + f16_exponent(mxb)) << 23);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      h[k] = cvt_f16x2(__uint_as_float(w[k] << 16) * sc, __uint_as_float(w[k] & 0xFFFF0000u) * sc);
    // unit j (k = 16j .. 16j + 15) is lane j's whole fragment entry
    uint4* dst = reinterpret_cast<uint4*>(xs + ((g * T + tok) * 4 + j) * 32);
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
  return stat[32] == 0u;
}

// The job loop of the x-in-registers consumer, for a slice of NG groups (one
// straight-line body, so the compiler can overlap one group's decode with the
// previous group's MMAs): per pair of row tiles (one tile with two token
// blocks), wait for each tile's stage, run the slice, release the stage; then
// hand the partials over at once.
// F16: fp16 route; the partials are brought back to the scale of x (inv) and
// rows q + 8 divided by 16 before they are handed over.
template <int BITS, int GWM, int NT, bool F16, int NG, bool CONT = false>
__device__ void xreg_jobs(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                          const Work& wk, int warp, int lane, int codes_off, int scales_off,
                          const uint32_t (&xr)[GWM][NT][8], const float (&inv)[NT][2],
                          RingPos* pos = nullptr) {
  constexpr int JT = NT == 1 ? 2 : 1;   // = kJobTiles of the kernel
  const int q = lane >> 2;
  const uint8_t* ring = smem + a.off_ring;
  float inv16[NT][2];
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) {
    inv16[nb][0] = inv[nb][0] * 0.0625f;
    inv16[nb][1] = inv[nb][1] * 0.0625f;
  }
  int stage = 0;
  uint32_t phase = 0;
  int rb = 0;        // partial buffer of this pair
  uint32_t rn = 0;   // uses of that buffer so far
  if constexpr (CONT) {  // continue where the previous phase left the rings
    stage = pos->stage;
    phase = pos->phase;
    rb = pos->rb;
    rn = pos->rn;
  }
  for (int j = 0; j < wk.njobs; j += JT) {
    float acc[JT][NT][4];
#pragma unroll
    for (int jt = 0; jt < JT; ++jt)
#pragma unroll
      for (int nb = 0; nb < NT; ++nb)
        acc[jt][nb][0] = acc[jt][nb][1] = acc[jt][nb][2] = acc[jt][nb][3] = 0.f;
#pragma unroll
    for (int jt = 0; jt < JT; ++jt) {
      if (jt > 0 && j + jt >= wk.njobs) break;
      if (!wt.wait_warp<false>(bars.full(stage), phase)) return;
      const uint8_t* st = ring + stage * a.stage_bytes;
      slice_xr<BITS, NT, GWM, NG, F16>(st + codes_off, st + scales_off, xr, lane, q, acc[jt]);
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(stage));
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
    if constexpr (F16) {
#pragma unroll
      for (int jt = 0; jt < JT; ++jt)
#pragma unroll
        for (int nb = 0; nb < NT; ++nb) {
          acc[jt][nb][0] *= inv[nb][0];
          acc[jt][nb][1] *= inv[nb][1];
          acc[jt][nb][2] *= inv16[nb][0];
          acc[jt][nb][3] *= inv16[nb][1];
        }
    }
    if (!hand_partials_mma<NT, JT>(a, smem, bars, wt, warp, lane, rb, rn, acc)) return;
    if (++rb == a.nbuf) { rb = 0; ++rn; }
  }
  if constexpr (CONT) *pos = RingPos{stage, phase, rb, rn};
}

// One group of the hybrid kernel: token block 0 against the x fragments in
// registers (xr), token block 1 against fragments read from the shared x tile
// (xs: this lane's entry of the group, xh: offset of the second plane; the
// zero area for lanes whose token is absent).
template <int BITS>
__device__ __forceinline__ void mma_group_xrh(const uint8_t* blk, const uint8_t* sc,
                                              const uint32_t (&xr)[8], const uint8_t* xs, int xh,
                                              int lane, int q, float (&acc)[2][4]) {
  uint32_t w[BITS];
  load_lane_words<BITS>(blk, lane, w);
  const float2 s = __half22float2(*reinterpret_cast<const __half2*>(sc + 4 * q));
  const uint4 xa = *reinterpret_cast<const uint4*>(xs);
  const uint4 xb = *reinterpret_cast<const uint4*>(xs + xh);
  float d[2][4], dh[2][4];   // dh: high-nibble plane of 8-bit codes
#pragma unroll
  for (int js = 0; js < 4; ++js) {
    uint32_t a0, a1, a2, a3, h0 = 0, h1 = 0, h2 = 0, h3 = 0;
    if constexpr (BITS == 8) {
      q8_pair_planes(w, 4 * js + 0, a0, h0);
      q8_pair_planes(w, 4 * js + 1, a1, h1);
      q8_pair_planes(w, 4 * js + 2, a2, h2);
      q8_pair_planes(w, 4 * js + 3, a3, h3);
    } else {
      a0 = pair_codes_bf16<BITS>(w, 4 * js + 0);
      a1 = pair_codes_bf16<BITS>(w, 4 * js + 1);
      a2 = pair_codes_bf16<BITS>(w, 4 * js + 2);
      a3 = pair_codes_bf16<BITS>(w, 4 * js + 3);
    }
    const uint32_t b0 = js == 0 ? xa.x : js == 1 ? xa.z : js == 2 ? xb.x : xb.z;
    const uint32_t b1 = js == 0 ? xa.y : js == 1 ? xa.w : js == 2 ? xb.y : xb.w;
    if (js == 0) {
      mma_16816_zc(d[0], a0, a1, a2, a3, xr[0], xr[1]);
      mma_16816_zc(d[1], a0, a1, a2, a3, b0, b1);
      if constexpr (BITS == 8) {
        mma_16816_zc(dh[0], h0, h1, h2, h3, xr[0], xr[1]);
        mma_16816_zc(dh[1], h0, h1, h2, h3, b0, b1);
      }
    } else {
      mma_16816(d[0], a0, a1, a2, a3, xr[2 * js], xr[2 * js + 1]);
      mma_16816(d[1], a0, a1, a2, a3, b0, b1);
      if constexpr (BITS == 8) {
        mma_16816(dh[0], h0, h1, h2, h3, xr[2 * js], xr[2 * js + 1]);
        mma_16816(dh[1], h0, h1, h2, h3, b0, b1);
      }
    }
  }
  if constexpr (BITS == 8) {
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) d[nb][e] = fmaf(16.f, dh[nb][e], d[nb][e]);
  }
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) {
    acc[nb][0] = fmaf(s.x, d[nb][0], acc[nb][0]);
    acc[nb][1] = fmaf(s.x, d[nb][1], acc[nb][1]);
    acc[nb][2] = fmaf(s.y, d[nb][2], acc[nb][2]);
    acc[nb][3] = fmaf(s.y, d[nb][3], acc[nb][3]);
  }
}

// The hybrid kernel's job loop for a slice of NG groups (one row tile per
// hand-off).  xs0: this lane's entry of the slice's first group in the shared
// x tile; xstep: bytes between groups; xh: the second plane's offset.
template <int BITS, int NG>
__device__ void xregh_jobs(const GemvArgs& a, uint8_t* smem, const Bars& bars, const Waiter& wt,
                           const Work& wk, int warp, int lane, int codes_off, int scales_off,
                           const uint32_t (&xr)[kXregMaxGroups][1][8], const uint8_t* xs0,
                           int xstep, int xh) {
  const int q = lane >> 2;
  const uint8_t* ring = smem + a.off_ring;
  int stage = 0;
  uint32_t phase = 0;
  int rb = 0;
  uint32_t rn = 0;
  for (int j = 0; j < wk.njobs; ++j) {
    float acc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    if (!wt.wait_warp<false>(bars.full(stage), phase)) return;
    const uint8_t* st = ring + stage * a.stage_bytes;
#pragma unroll
    for (int i = 0; i < NG; ++i)
      mma_group_xrh<BITS>(st + codes_off + i * (128 * BITS), st + scales_off + i * kScaleBytesPerBlock,
                          xr[i][0], xs0 + i * xstep, xh, lane, q, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.empty(stage));
    if (++stage == a.stages) { stage = 0; phase ^= 1; }
    if (!hand_partial_mma<2>(a, smem, bars, wt, warp, lane, rb, rn, acc)) return;
    if (++rb == a.nbuf) { rb = 0; ++rn; }
  }
}

// Hybrid consumer: token block 0's x fragments of the warp's fixed slice in
// registers, token block 1's (tokens 8 ..) in the shared x tile, which the
// consumer warps stage once in B-fragment order (stage_x_bf16's layout over
// tokens 8 .. T-1, as if x started at token 8).
template <int BITS>
__device__ void consumer_xregh(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                               const Waiter& wt, const Work& wk, int warp, int lane) {
  constexpr int kBlock = 128 * BITS;
  const Slice sl = warp_slice(wk, warp);
  const int n = sl.ge - sl.gs;  // <= kXregMaxGroups
  const int rel = sl.gs - wk.g_begin;
  const int codes_off = rel * kBlock;
  const int scales_off = a.stage_groups * kBlock + rel * kScaleBytesPerBlock;
  uint32_t xr[kXregMaxGroups][1][8];
  load_x_frags<kXregMaxGroups, 1>(a, sl, n, lane, xr);
  // Stage tokens 8 .. T-1 (T2 = T - 8 of them).
  GemvArgs b2 = a;
  b2.x = a.x + 8LL * a.K;
  b2.T = a.T - 8;
  stage_x_bf16(b2, smem, wk, threadIdx.x, kWarps * 32);
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
  const int q = lane >> 2;
  const int T2 = a.T - 8;
  const bool v = q < T2;
  const uint8_t* xs0 = v ? smem + a.off_x + ((rel * T2 + q) * 4 + (lane & 3)) * 16
                         : smem + kZeroAreaOffset;
  const int xstep = v ? T2 * 64 : 0;
  const int xh = v ? (wk.g_end - wk.g_begin) * T2 * 64 : 16;  // the zero area holds 32 bytes
#define NQ_XREGH_CASE(k)                                                                   \
  case k:                                                                                  \
    xregh_jobs<BITS, k>(a, smem, bars, wt, wk, warp, lane, codes_off, scales_off, xr, xs0, \
                        xstep, xh);                                                        \
    break;
  switch (n) {
    NQ_XREGH_CASE(1)
    NQ_XREGH_CASE(2)
    NQ_XREGH_CASE(3)
    NQ_XREGH_CASE(4)
    NQ_XREGH_CASE(5)
    default:
      xregh_jobs<BITS, 0>(a, smem, bars, wt, wk, warp, lane, codes_off, scales_off, xr, xs0,
                          xstep, xh);
      break;
  }
#undef NQ_XREGH_CASE
}

// The slice length n (uniform per warp, <= GWM) picks the job loop once.
template <int BITS, int GWM, int NT, bool F16, bool CONT = false>
__device__ __forceinline__ void run_xreg_jobs(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                                              const Waiter& wt, const Work& wk, int warp,
                                              int lane, int n, int codes_off, int scales_off,
                                              const uint32_t (&xr)[GWM][NT][8],
                                              const float (&inv)[NT][2],
                                              RingPos* pos = nullptr) {
  static_assert(GWM <= 5, "slice-length dispatch covers 1..5 groups");
#define NQ_XREG_CASE(k)                                                                      \
  case k:                                                                                    \
    if constexpr (k <= GWM)                                                                  \
      xreg_jobs<BITS, GWM, NT, F16, k, CONT>(a, smem, bars, wt, wk, warp, lane, codes_off,   \
                                             scales_off, xr, inv, pos);                      \
    break;
  switch (n) {
    NQ_XREG_CASE(1)
    NQ_XREG_CASE(2)
    NQ_XREG_CASE(3)
    NQ_XREG_CASE(4)
    NQ_XREG_CASE(5)
    default:
      // A warp without groups still takes part in every hand-off (zeros).
      xreg_jobs<BITS, GWM, NT, F16, 0, CONT>(a, smem, bars, wt, wk, warp, lane, codes_off,
                                             scales_off, xr, inv, pos);
      break;
  }
#undef NQ_XREG_CASE
}

// x in registers: a stage holds the CTA's whole K range of one job; the warp
// decodes its fixed slice of it (at most GWM groups) against x fragments of
// NT token blocks loaded once per kernel.  4-bit codes take the fp16 route
// when x converts exactly (see stage_x_f16), every other case the bf16 route.
template <int BITS, int GWM, int NT, bool CONT = false>
__device__ void consumer_xreg(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                              const Waiter& wt, const Work& wk, int warp, int lane,
                              RingPos* pos = nullptr) {
  constexpr int kBlock = 128 * BITS;
  const Slice sl = warp_slice(wk, warp);
  const int n = sl.ge - sl.gs;  // <= GWM
  const int rel = sl.gs - wk.g_begin;
  const int codes_off = rel * kBlock;
  const int scales_off = a.stage_groups * kBlock + rel * kScaleBytesPerBlock;

  uint32_t xr[GWM][NT][8];
  float inv[NT][2];
  if constexpr (BITS == 4 && NT == 1) {   // (the planner takes it for T <= 2 only)
    if (a.off_xh >= 0) {
      const bool f16 = stage_x_f16(a, smem, wk, warp, lane);
      if (f16) {
        // Fragments from the staging area; inv: 2^-e_t of this lane's
        // accumulator columns (tokens 8 nb + 2r + c).
        const int q = lane >> 2, r = lane & 3;
        const uint32_t* stat = reinterpret_cast<const uint32_t*>(smem + kXStatOffset);
#pragma unroll
        for (int nb = 0; nb < NT; ++nb) {
          const int tok = 8 * nb + q;
#pragma unroll
          for (int i = 0; i < GWM; ++i) {
            uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
            if (i < n && tok < a.T) {
              const uint8_t* p = smem + a.off_xh + (((rel + i) * a.T + tok) * 4 + r) * 32;
              v0 = *reinterpret_cast<const uint4*>(p);
              v1 = *reinterpret_cast<const uint4*>(p + 16);
            }
            xr[i][nb][0] = v0.x; xr[i][nb][1] = v0.y; xr[i][nb][2] = v0.z; xr[i][nb][3] = v0.w;
            xr[i][nb][4] = v1.x; xr[i][nb][5] = v1.y; xr[i][nb][6] = v1.z; xr[i][nb][7] = v1.w;
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int t = 8 * nb + 2 * r + c;
            const int e = t < a.T ? f16_exponent(stat[t]) : 0;
            inv[nb][c] = __int_as_float((127 - e) << 23);
          }
        }
      } else {
        load_x_frags<GWM, NT>(a, sl, n, lane, xr);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(smem + kXFreeBarOffset));
      if (f16) {
        run_xreg_jobs<BITS, GWM, NT, true, CONT>(a, smem, bars, wt, wk, warp, lane, n, codes_off,
                                                 scales_off, xr, inv, pos);
        return;
      }
#pragma unroll
      for (int nb = 0; nb < NT; ++nb) inv[nb][0] = inv[nb][1] = 1.f;
      run_xreg_jobs<BITS, GWM, NT, false, CONT>(a, smem, bars, wt, wk, warp, lane, n, codes_off,
                                                scales_off, xr, inv, pos);
      return;
    }
  }
  // (A continuing phase reads x that this kernel wrote: through L2.)
  load_x_frags<GWM, NT, CONT>(a, sl, n, lane, xr);
#pragma unroll
  for (int nb = 0; nb < NT; ++nb) inv[nb][0] = inv[nb][1] = 1.f;
  run_xreg_jobs<BITS, GWM, NT, false, CONT>(a, smem, bars, wt, wk, warp, lane, n, codes_off,
                                            scales_off, xr, inv, pos);
}

// x in shared memory: the warps take the groups of each stage in turn
// (warp, warp + 16, ...).
template <int BITS, int ROUTE, int NT>
__device__ void consumer_xsmem(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                               const Waiter& wt, const Work& wk, int warp, int lane) {
  constexpr int kBlock = 128 * BITS;
  const int q = lane >> 2, r = lane & 3;
  const int T = a.T;
  const int sg = a.stage_groups;
  const uint8_t* ring = smem + a.off_ring;
  // MMA route: x fragments of token 8 nb + q, or the zero area if absent.
  const uint8_t* xbase[NT];
  int xstep[NT], xhalf[NT];
  if constexpr (ROUTE == kRouteMma) {
    const int hb = (wk.g_end - wk.g_begin) * T * 64;  // second x plane (stage_x_bf16)
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      const bool v = 8 * nb + q < T;
      xbase[nb] = v ? smem + a.off_x + 512 * nb + 16 * lane : smem + kZeroAreaOffset;
      xstep[nb] = v ? T * 64 : 0;
      xhalf[nb] = v ? hb : 16;   // the zero area holds 32 bytes
    }
  }
  const uint8_t* xf = smem + a.off_x + 64 * r;  // FMA route: entry (g, t, r) at (g T + t) 256 + 64 r

  int stage = 0;
  uint32_t phase = 0;
  int rb = 0;        // partial buffer of this job
  uint32_t rn = 0;   // uses of that buffer so far
  for (int j = 0; j < wk.njobs; ++j) {
    float acc[NT][4];
    float facc[2][NT];
#pragma unroll
    for (int nb = 0; nb < NT; ++nb) {
      acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
      facc[0][nb] = facc[1][nb] = 0.f;
    }
    for (int g0 = wk.g_begin; g0 < wk.g_end; g0 += sg) {
      const int ng = min(sg, wk.g_end - g0);
      if (!wt.wait_warp<false>(bars.full(stage), phase)) return;
      const uint8_t* st = ring + stage * a.stage_bytes;
      const uint8_t* scb = st + sg * kBlock;
      const int gx0 = g0 - wk.g_begin;
      for (int gl = warp; gl < ng; gl += kWarps) {
        if constexpr (ROUTE == kRouteMma) {
          const uint8_t* xp[NT];
#pragma unroll
          for (int nb = 0; nb < NT; ++nb) xp[nb] = xbase[nb] + (gx0 + gl) * xstep[nb];
          mma_group<BITS, NT>(st + gl * kBlock, scb + gl * kScaleBytesPerBlock, xp, xhalf, lane, q,
                              acc);
        } else {
          ffma_group<BITS, NT>(st + gl * kBlock, scb + gl * kScaleBytesPerBlock,
                               xf + (gx0 + gl) * T * 256, lane, q, T, facc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(stage));
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
    if constexpr (ROUTE == kRouteMma) {
      if (!hand_partial_mma<NT>(a, smem, bars, wt, warp, lane, rb, rn, acc)) return;
    } else {
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
      if (!wt.wait_warp<false>(bars.red_empty(rb), (rn & 1u) ^ 1u)) return;
      float* slot = reinterpret_cast<float*>(smem + a.off_red) + (rb * kWarps + warp) * 16 * T;
      if (r == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < T) {
            slot[t * 16 + q] = facc[0][t];
            slot[t * 16 + q + 8] = facc[1][t];
          }
        }
      }
      mbar_arrive(bars.red_full(rb));
    }
    if (++rb == a.nbuf) { rb = 0; ++rn; }
  }
}

// ------------------------------------------------------------------ epilogue
// Per job: sum the 16 warps' partials in warp order; with a K split, ranks
// 1.. send their sums to rank 0 with asynchronous cluster stores whose bytes
// complete rank 0's barrier, and rank 0 adds them in rank order and stores y.
// No cluster-scope fence is needed: the peers' data is published by the
// transaction count of st.async, and rank 0's "slot free" signal back to a
// peer only orders rank 0's reads, which have completed once their values
// have been added.  Lane l handles the four consecutive values 4 l + 128 i,
// i < SLOTS, of the 16 x T tile (value e = 16 t + row); only slots that hold
// values are touched, so nothing is issued for tokens that do not exist.
// Epilogue warp `ew` handles jobs ew, ew + kEpiWarps, ...; nbuf is a multiple
// of kEpiWarps, so each partial buffer always belongs to the same warp.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, const float4& v,
                                            uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(cluster_addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cluster_bar)
               : "memory");
}
// silu(g) * u in fp32: g / (1 + exp(-g)) * u (expf; -0 for very negative g).
__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.f + expf(-g)) * u;
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}
// ------------------------------------------------------------------ fused head
// Running state of a softmax over logits seen so far: maximum m, sum of
// exp(y - m), argmax a (smallest index among equal maxima).  An empty state is
// (-inf, 0, INT_MAX).  head_merge is commutative bit for bit, so the butterfly
// merges below leave every lane with the same state.
__device__ __forceinline__ void head_push(float& m, float& s, int& a, float v, int idx) {
  if (v > m) {
    s = s * __expf(m - v) + 1.f;
    m = v;
    a = idx;
  } else if (v == -INFINITY) {
    // contributes exp(-inf) = 0 (and leaves an empty state empty)
  } else if (v == m) {
    s += 1.f;  // exp(0); also keeps a second +inf logit from forming inf - inf
  } else {
    s += __expf(v - m);
  }
}
// The same after the four logits of rows idx0 .. idx0 + 3: the batch's
// maximum first (one rescale at most), then one term per logit without
// branches.  Rows arrive in increasing order, so on equal maxima the state's
// index is the smaller one.
__device__ __forceinline__ void head_push4(float& m, float& s, int& a, const float4& v, int idx0) {
  const float x[4] = {v.x, v.y, v.z, v.w};
  float mb = -INFINITY;  // (NaN never becomes the maximum)
  int ib = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (x[c] > mb) {
      mb = x[c];
      ib = c;
    }
  if (mb > m) {
    s *= __expf(m - mb);  // 0 for the empty state (m = -inf, s = 0)
    m = mb;
    a = idx0 + ib;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
    s += x[c] == -INFINITY ? 0.f : x[c] == m ? 1.f : __expf(x[c] - m);
}
__device__ __forceinline__ void head_merge(float& m, float& s, int& a, float mo, float so, int ao) {
  if (mo == -INFINITY && so == 0.f) return;
  if (m == -INFINITY && s == 0.f) {
    m = mo;
    s = so;
    a = ao;
    return;
  }
  if (mo == m) {  // equal maxima (both +inf included): the factor is exactly 1
    s = s + so;
    a = min(a, ao);
  } else if (mo > m) {
    s = s * __expf(m - mo) + so;
    m = mo;
    a = ao;
  } else {
    s = s + so * __expf(mo - m);
  }
}
__device__ __forceinline__ void head_merge_lanes(float& m, float& s, int& a, int xor_mask) {
  const float mo = __shfl_xor_sync(0xffffffffu, m, xor_mask);
  const float so = __shfl_xor_sync(0xffffffffu, s, xor_mask);
  const int ao = __shfl_xor_sync(0xffffffffu, a, xor_mask);
  head_merge(m, s, a, mo, so, ao);
}

// End of a CTA's epilogue warp on the fused head: merge, per token, every
// lane's states of that token (slot i of a lane holds token vtok[i]) with a
// butterfly over the warp, and publish the warp's per-token states; then a
// two-level merge, each
// level done by the last warp to arrive and costing one round of loads:
// the last warp of a group of kHeadGroup clusters merges the group's
// 2 kHeadGroup states per token in (cluster, warp) order, and the last group
// to finish merges the groups in order and writes argmax, maximum and
// logsumexp.  Lanes 2t and 2t + 1 take token t, one half of the entries each.
template <int NMAX>
__device__ __forceinline__ void head_merge_entries(const uint8_t* base, int first, int count,
                                                   int tok, float& m, float& s, int& am) {
  float4 st[NMAX];
#pragma unroll
  for (int k = 0; k < NMAX; ++k)
    st[k] = k < count ? __ldcg(reinterpret_cast<const float4*>(
                            base + (static_cast<size_t>(first + k) * kHeadMaxT + tok) * kHeadStateBytes))
                      : make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
#pragma unroll
  for (int k = 0; k < NMAX; ++k) head_merge(m, s, am, st[k].x, st[k].y, __float_as_int(st[k].z));
}

template <int SLOTS>
__device__ void head_finish(const GemvArgs& a, const Work& wk, int ew, int lane,
                            const float (&hm)[SLOTS], const float (&hs)[SLOTS],
                            const int (&ha)[SLOTS], const int (&vtok)[SLOTS]) {
  const int T = a.T;
  const int cl = blockIdx.x / a.ksplit;
  const int grp = cl / kHeadGroup;
  const int ngroups = (a.clusters + kHeadGroup - 1) / kHeadGroup;
  const int gcl0 = grp * kHeadGroup;                              // first cluster of the group
  const int gcls = min(kHeadGroup, a.clusters - gcl0);           // clusters in the group
  unsigned* counters = reinterpret_cast<unsigned*>(a.h_ws);
  uint8_t* states = a.h_ws + kHeadCounterBytes;                  // (cluster, warp, token)
  uint8_t* gstates = states + static_cast<size_t>(a.clusters) * kEpiWarps * kHeadMaxT * kHeadStateBytes;
  for (int t = 0; t < T; ++t) {
    float m = -INFINITY, s = 0.f;
    int am = INT_MAX;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (vtok[i] == t) head_merge(m, s, am, hm[i], hs[i], ha[i]);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) head_merge_lanes(m, s, am, d);
    if (lane == 0) {
      const int me = cl * kEpiWarps + ew;
      *reinterpret_cast<float4*>(states + (static_cast<size_t>(me) * kHeadMaxT + t) * kHeadStateBytes) =
          make_float4(m, s, __int_as_float(am), 0.f);
    }
  }
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0)
    last = atomicAdd(counters + 1 + grp, 1u) == static_cast<unsigned>(gcls * kEpiWarps - 1);
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  // First level: this group's states.
  const int tok = lane >> 1, half = lane & 1;
  {
    constexpr int kHalf = kHeadGroup * kEpiWarps / 2;
    float m = -INFINITY, s = 0.f;
    int am = INT_MAX;
    if (tok < T) {
      const int n = gcls * kEpiWarps;
      const int first = half * kHalf;
      head_merge_entries<kHalf>(states, gcl0 * kEpiWarps + first, max(0, min(kHalf, n - first)),
                                tok, m, s, am);
    }
    head_merge_lanes(m, s, am, 1);
    if (half == 0 && tok < T)
      *reinterpret_cast<float4*>(gstates + (static_cast<size_t>(grp) * kHeadMaxT + tok) * kHeadStateBytes) =
          make_float4(m, s, __int_as_float(am), 0.f);
    if (lane == 0) *reinterpret_cast<volatile unsigned*>(counters + 1 + grp) = 0u;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) last = atomicAdd(counters, 1u) == static_cast<unsigned>(ngroups - 1);
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  // Second level: every group, in order.
  {
    constexpr int kHalf = kHeadMaxGroups / 2;
    float m = -INFINITY, s = 0.f;
    int am = INT_MAX;
    if (tok < T) {
      const int first = half * kHalf;
      head_merge_entries<kHalf>(gstates, first, max(0, min(kHalf, ngroups - first)), tok, m, s,
                                am);
    }
    head_merge_lanes(m, s, am, 1);
    if (half == 0 && tok < T) {
      a.h_argmax[tok] = am == INT_MAX ? -1 : am;
      a.h_max[tok] = m;
      a.h_lse[tok] = m + __logf(s);
    }
    if (lane == 0) *reinterpret_cast<volatile unsigned*>(counters) = 0u;
  }
}

// head_finish for epilogue_rs: every CTA publishes states (the ranks of a
// cluster finalise different slots), so the merge runs over CTAs.
template <int SLOTS>
__device__ void head_finish_cta(const GemvArgs& a, const Work& wk, int ew, int lane,
                            const float (&hm)[SLOTS], const float (&hs)[SLOTS],
                            const int (&ha)[SLOTS], const int (&vtok)[SLOTS]) {
  const int T = a.T;
  const int units = a.clusters * a.ksplit;  // CTAs publishing states
  const int cl = static_cast<int>(blockIdx.x);
  const int grp = cl / kHeadGroup;
  const int ngroups = (units + kHeadGroup - 1) / kHeadGroup;
  const int gcl0 = grp * kHeadGroup;                              // first unit of the group
  const int gcls = min(kHeadGroup, units - gcl0);                // units in the group
  unsigned* counters = reinterpret_cast<unsigned*>(a.h_ws);
  uint8_t* states = a.h_ws + kHeadCounterBytes;                  // (unit, warp, token)
  uint8_t* gstates = states + static_cast<size_t>(units) * kEpiWarps * kHeadMaxT * kHeadStateBytes;
  for (int t = 0; t < T; ++t) {
    float m = -INFINITY, s = 0.f;
    int am = INT_MAX;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (vtok[i] == t) head_merge(m, s, am, hm[i], hs[i], ha[i]);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) head_merge_lanes(m, s, am, d);
    if (lane == 0) {
      const int me = cl * kEpiWarps + ew;
      *reinterpret_cast<float4*>(states + (static_cast<size_t>(me) * kHeadMaxT + t) * kHeadStateBytes) =
          make_float4(m, s, __int_as_float(am), 0.f);
    }
  }
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0)
    last = atomicAdd(counters + 1 + grp, 1u) == static_cast<unsigned>(gcls * kEpiWarps - 1);
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  // First level: this group's states.
  const int tok = lane >> 1, half = lane & 1;
  {
    constexpr int kHalf = kHeadGroup * kEpiWarps / 2;
    float m = -INFINITY, s = 0.f;
    int am = INT_MAX;
    if (tok < T) {
      const int n = gcls * kEpiWarps;
      const int first = half * kHalf;
      head_merge_entries<kHalf>(states, gcl0 * kEpiWarps + first, max(0, min(kHalf, n - first)),
                                tok, m, s, am);
    }
    head_merge_lanes(m, s, am, 1);
    if (half == 0 && tok < T)
      *reinterpret_cast<float4*>(gstates + (static_cast<size_t>(grp) * kHeadMaxT + tok) * kHeadStateBytes) =
          make_float4(m, s, __int_as_float(am), 0.f);
    if (lane == 0) *reinterpret_cast<volatile unsigned*>(counters + 1 + grp) = 0u;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) last = atomicAdd(counters, 1u) == static_cast<unsigned>(ngroups - 1);
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  // Second level: every group, in order.
  {
    constexpr int kHalf = kHeadMaxGroups / 2;
    float m = -INFINITY, s = 0.f;
    int am = INT_MAX;
    if (tok < T) {
      const int first = half * kHalf;
      head_merge_entries<kHalf>(gstates, first, max(0, min(kHalf, ngroups - first)), tok, m, s,
                                am);
    }
    head_merge_lanes(m, s, am, 1);
    if (half == 0 && tok < T) {
      a.h_argmax[tok] = am == INT_MAX ? -1 : am;
      a.h_max[tok] = m;
      a.h_lse[tok] = m + __logf(s);
    }
    if (lane == 0) *reinterpret_cast<volatile unsigned*>(counters) = 0u;
  }
}

// Shared-memory bytes of the top-k buffer counts (all epilogue warps).
constexpr int kTopkSmemBytes = kEpiWarps * kHeadMaxT * 4;

// Folds the candidate buffer of token t (n keys, n < 64) into its list: at
// most two rounds of sort 32 + merge.  Whole warp; list and buf are this
// warp's own (global memory, written and read by this warp only).
__device__ __forceinline__ void topk_flush(unsigned long long* list, unsigned long long* buf,
                                           int* cnt, int t, int lane) {
  const int n = cnt[t];
  unsigned long long* lt = list + t * 32;
  unsigned long long m = lt[lane];
  for (int base = 0; base < n; base += 32) {
    unsigned long long c = base + lane < n ? buf[t * 64 + base + lane] : 0ull;
    c = warp_sort_desc(c, lane);
    m = warp_top32_of_two(m, c, lane);
  }
  __syncwarp();
  lt[lane] = m;
  if (lane == 0) cnt[t] = 0;
  __syncwarp();
}

// One hand-off's logits into the warp's top-k state (the selection scheme of
// warp-level k-selection: cheap filtering against a threshold, sorting only
// in batches).  A logit whose key beats the k-th key of its token's list
// (a lower bound of the warp's k-th largest so far) is appended to the
// token's buffer; a buffer holding 32 or more keys after the hand-off is
// folded into the list.  A hand-off adds at most JT x 16 <= 32 keys per
// token, so a buffer (64 keys) never overflows.  ok[i]: slot i holds logits
// (rows rbase[i] .. rbase[i] + 3, those below N) of token vtok[i].
template <int SLOTS>
__device__ __forceinline__ void topk_update(const GemvArgs& a, unsigned long long* list,
                                            unsigned long long* buf, int* cnt, int lane,
                                            const float4 (&v)[SLOTS], const bool (&ok)[SLOTS],
                                            const long long (&rbase)[SLOTS],
                                            const int (&vtok)[SLOTS]) {
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    if (!ok[i]) continue;
    const int t = vtok[i];
    const unsigned long long thr = list[t * 32 + a.tk_k - 1];
    const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const unsigned long long key = topk_key(vv[c], static_cast<uint32_t>(rbase[i] + c));
      if (rbase[i] + c < a.N && key > thr) buf[t * 64 + atomicAdd(cnt + t, 1)] = key;
    }
  }
  __syncwarp();
  unsigned full = __ballot_sync(0xffffffffu, lane < a.T && cnt[lane] >= 32);
  while (full) {
    const int t = __ffs(full) - 1;
    full &= full - 1;
    topk_flush(list, buf, cnt, t, lane);
  }
}

// topk_flush and topk_update for epilogue_rs (which keeps each slot's
// threshold in registers).  Folds the candidate buffer of token t into its list: at
// most two rounds of sort 32 + merge.  Whole warp; list and buf are this
// warp's own (global memory, written and read by this warp only).  Returns,
// in every lane, the list's new k-th key.
__device__ __forceinline__ unsigned long long topk_flush_kth(unsigned long long* list,
                                                         unsigned long long* buf, int* cnt, int t,
                                                         int lane, int k) {
  const int n = cnt[t];
  unsigned long long* lt = list + t * 32;
  unsigned long long m = lt[lane];
  for (int base = 0; base < n; base += 32) {
    unsigned long long c = base + lane < n ? buf[t * 64 + base + lane] : 0ull;
    c = warp_sort_desc(c, lane);
    m = warp_top32_of_two(m, c, lane);
  }
  __syncwarp();
  lt[lane] = m;
  if (lane == 0) cnt[t] = 0;
  __syncwarp();
  return __shfl_sync(0xffffffffu, m, k - 1);
}

// One hand-off's logits into the warp's top-k state (the selection scheme of
// warp-level k-selection: cheap filtering against a threshold, sorting only
// in batches).  A logit whose key beats the k-th key of its token's list
// (a lower bound of the warp's k-th largest so far) is appended to the
// token's buffer; a buffer holding 32 or more keys after the hand-off is
// folded into the list.  A hand-off adds at most JT x 16 <= 32 keys per
// token, so a buffer (64 keys) never overflows.  ok[i]: slot i holds logits
// (rows rbase[i] .. rbase[i] + 3, those below N) of token vtok[i]; thr[i]:
// the k-th key of that token's list, kept in registers (a lane's slots keep
// their tokens) and refreshed when the list changes.
template <int SLOTS>
__device__ __forceinline__ void topk_update_thr(const GemvArgs& a, unsigned long long* list,
                                            unsigned long long* buf, int* cnt, int lane,
                                            const float4 (&v)[SLOTS], const bool (&ok)[SLOTS],
                                            const long long (&rbase)[SLOTS],
                                            const int (&vtok)[SLOTS],
                                            unsigned long long (&thr)[SLOTS]) {
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    if (!ok[i]) continue;
    const int t = vtok[i];
    const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const unsigned long long key = topk_key(vv[c], static_cast<uint32_t>(rbase[i] + c));
      if (rbase[i] + c < a.N && key > thr[i]) buf[t * 64 + atomicAdd(cnt + t, 1)] = key;
    }
  }
  __syncwarp();
  unsigned full = __ballot_sync(0xffffffffu, lane < a.T && cnt[lane] >= 32);
  while (full) {
    const int t = __ffs(full) - 1;
    full &= full - 1;
    const unsigned long long kth = topk_flush_kth(list, buf, cnt, t, lane, a.tk_k);
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (vtok[i] == t) thr[i] = kth;
  }
}

// K-split exchange as a reduce-scatter (the fused head with two token blocks
// in registers): slot i of a hand-off (values 128 i .. 128 i + 127, those
// below nv) is finalised by rank i mod ks; every other rank sends its
// partials of that slot to that rank.  With one slot in use everything stays
// on rank 0.  Halves the per-logit softmax work of rank 0 at T = 16 (the
// fused head 266 -> 252 us, with top-8 385 -> 349 us on GB300); the plain
// products keep the gather to rank 0, which measured faster for them.
__device__ __forceinline__ int slot_values(int nv, int i) { return max(0, min(128, nv - 128 * i)); }
template <int SLOTS>
__device__ __forceinline__ unsigned slot_owners(int ks, int nv) {
  unsigned m = 0u;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i)
    if (slot_values(nv, i) > 0) m |= 1u << (i % ks);
  return m;
}

// Arrivals that complete one use of a rank's exchange-release barrier: one
// from every other rank that finalises slots (at least 1; unused then).
template <int SLOTS>
__device__ __forceinline__ unsigned cl_empty_count(int ks, int nv, int rank) {
  return max(1, __popc(slot_owners<SLOTS>(ks, nv) & ~(1u << rank)));
}

// The epilogue of the fused head whose K split finalises by reduce-scatter
// (two token blocks in registers, ksplit > 1; see slot_owners).  Besides the
// exchange it differs from epilogue() in the softmax update (head_push4), in
// keeping the top-k thresholds in registers and in publishing head states and
// top-k lists per CTA; a separate function, so that the other kernels' code
// stays as it is.
template <int SLOTS, int JT>
__device__ inline void epilogue_rs(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                                   const Waiter& wt, const Work& wk, int ew, int lane) {
  const int T = a.T;
  const int nvt = 16 * T;            // values per row tile (a multiple of 16)
  const int nv = JT * nvt;           // values per hand-off (JT consecutive tiles)
  const int ks = a.ksplit;
  const float* red = reinterpret_cast<const float*>(smem + a.off_red);
  float* cl = reinterpret_cast<float*>(smem + a.off_cl);
  // mine[i]: this rank finalises slot i; in_bytes: what its peers send it per
  // hand-off; sends: some other rank finalises a slot in use.
  bool mine[SLOTS];
  uint32_t in_bytes = 0;
  bool any_mine = false;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    mine[i] = i % ks == wk.rank;
    any_mine = any_mine || mine[i];
    if (mine[i]) in_bytes += static_cast<uint32_t>((ks - 1) * slot_values(nv, i) * 4);
  }
  const bool sends = (slot_owners<SLOTS>(ks, nv) & ~(1u << wk.rank)) != 0u;
  auto has = [&](int i) { return 4 * lane + 128 * i < nv; };
  float hm[SLOTS], hs[SLOTS];
  int ha[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    hm[i] = -INFINITY;
    hs[i] = 0.f;
    ha[i] = INT_MAX;
  }
  // Tile, token and row of this lane's four values in slot i (fixed per lane).
  int vt[SLOTS], vtok[SLOTS], vrow[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = 4 * lane + 128 * i;
    vt[i] = e / nvt;
    const int rest = e - vt[i] * nvt;
    vtok[i] = rest >> 4;
    vrow[i] = rest & 15;
  }
  const int njt = (wk.njobs + JT - 1) / JT;  // hand-offs of this CTA
  const bool topk = a.tk_k > 0;
  unsigned long long* tk_list = nullptr;
  unsigned long long* tk_buf = nullptr;
  int* tk_cnt = nullptr;
  unsigned long long tk_thr[SLOTS];  // k-th key of each slot's token list (empty: key 0)
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) tk_thr[i] = 0ull;
  if (topk) {
    const size_t me = static_cast<size_t>(blockIdx.x) * kEpiWarps + ew;  // one list per CTA
    tk_list = a.tk_lists + me * kHeadMaxT * 32;
    tk_buf = a.tk_bufs + me * kHeadMaxT * 64;
    tk_cnt = reinterpret_cast<int*>(smem + a.off_tk) + ew * kHeadMaxT;
    for (int t = 0; t < T; ++t) tk_list[t * 32 + lane] = 0ull;  // empty keys
    if (lane < T) tk_cnt[lane] = 0;
    __syncwarp();
  }
  int b = ew;        // buffer of hand-off j (j % nbuf), also its exchange buffer
  uint32_t n = 0;    // uses of that buffer so far (j / nbuf)
  for (int j = ew; j < njt; j += kEpiWarps) {
    if (in_bytes != 0u && lane == 0) mbar_arrive_expect_tx_relaxed(bars.cl_full(b), in_bytes);
    if (!wt.wait_warp<false>(bars.red_full(b), n & 1u)) return;
    float4 v[SLOTS];
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (has(i)) {
        const float* p = red + b * kWarps * nv + 4 * lane + 128 * i;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) add4(v[i], *reinterpret_cast<const float4*>(p + w * nv));
      }
    }
    mbar_arrive_relaxed(bars.red_empty(b));  // every lane: count 32
    if (sends) {
      // Partials of the slots other ranks finalise: peer r of slot i's owner
      // o writes area r - (r > o) of o's exchange buffer.
      if (!wt.wait_warp<false>(bars.cl_empty(b), (n & 1u) ^ 1u)) return;
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) {
        if (mine[i] || !has(i)) continue;
        const int o = i % ks;
        const int area = wk.rank - (wk.rank > o ? 1 : 0);
        st_async_v4(map_to_rank(smem_addr(cl + (b * (ks - 1) + area) * nv + 4 * lane + 128 * i), o),
                    v[i], map_to_rank(bars.cl_full(b), o));
      }
    }
    if (in_bytes != 0u) {
      // Finalise this rank's slots: the ranks' partials added in rank order
      // (this rank's own from registers), then release the buffer to every
      // peer.
      if (!wt.wait_warp<false>(bars.cl_full(b), n & 1u)) return;
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) {
        if (!mine[i] || !has(i)) continue;
        const float* src = cl + b * (ks - 1) * nv + 4 * lane + 128 * i;
        float4 acc = wk.rank == 0 ? v[i] : *reinterpret_cast<const float4*>(src);
        for (int r = 1; r < ks; ++r)
          add4(acc, r == wk.rank ? v[i]
                                 : *reinterpret_cast<const float4*>(src + (r - (r > wk.rank ? 1 : 0)) * nv));
        v[i] = acc;
      }
      __syncwarp();
      if (lane == 0) {
        for (int r = 0; r < ks; ++r)
          if (r != wk.rank) mbar_arrive_remote_relaxed(map_to_rank(bars.cl_empty(b), r));
      }
    }
    if (any_mine) {
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) {
        if (mine[i] && has(i) && j * JT + vt[i] < wk.njobs) {
          const long long row0 = (wk.rt_begin + j * JT + vt[i]) * 16;
          const int tok = vtok[i], row = vrow[i];
          const long long nrow = a.N - (row0 + row);  // rows left in y from this one
          const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
          if (a.y != nullptr) {
            float* yp = a.y + static_cast<long long>(tok) * a.N + row0 + row;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (c < nrow) yp[c] = vv[c];
          }
          if (nrow >= 4) {
            head_push4(hm[i], hs[i], ha[i], v[i], static_cast<int>(row0 + row));
          } else {
#pragma unroll
            for (int c = 0; c < 3; ++c)
              if (c < nrow) head_push(hm[i], hs[i], ha[i], vv[c], static_cast<int>(row0 + row + c));
          }
        }
      }
      if (topk) {
        bool ok[SLOTS];
        long long rbase[SLOTS];
#pragma unroll
        for (int i = 0; i < SLOTS; ++i) {
          ok[i] = mine[i] && has(i) && j * JT + vt[i] < wk.njobs;
          rbase[i] = (wk.rt_begin + j * JT + vt[i]) * 16 + vrow[i];
        }
        topk_update_thr<SLOTS>(a, tk_list, tk_buf, tk_cnt, lane, v, ok, rbase, vtok, tk_thr);
      }
    }
    b += kEpiWarps;
    if (b >= a.nbuf) { b -= a.nbuf; ++n; }
  }
  if (topk) {
    for (int t = 0; t < T; ++t)
      if (tk_cnt[t] > 0) (void)topk_flush_kth(tk_list, tk_buf, tk_cnt, t, lane, a.tk_k);
  }
  head_finish_cta<SLOTS>(a, wk, ew, lane, hm, hs, ha, vtok);
}

// CONT: a phase of the one-launch layer; its hand-offs continue the CTA's
// sequence after `h0` hand-offs of the previous phase (hand-off g uses
// buffer g % nbuf and belongs to epilogue warp g % kEpiWarps).
template <int SLOTS, int JT, bool CONT = false>
__device__ inline void epilogue(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                                const Waiter& wt, const Work& wk, int ew, int lane, int h0 = 0) {
  const int T = a.T;
  const int nvt = 16 * T;            // values per row tile (a multiple of 16)
  const int nv = JT * nvt;           // values per hand-off (JT consecutive tiles)
  const int ks = a.ksplit;
  const float* red = reinterpret_cast<const float*>(smem + a.off_red);
  float* cl = reinterpret_cast<float*>(smem + a.off_cl);
  const uint32_t cl_bytes = static_cast<uint32_t>((ks - 1) * nv * 4);
  auto has = [&](int i) { return 4 * lane + 128 * i < nv; };
  const bool head = a.h_ws != nullptr;
  float hm[SLOTS], hs[SLOTS];
  int ha[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    hm[i] = -INFINITY;
    hs[i] = 0.f;
    ha[i] = INT_MAX;
  }
  // Tile, token and row of this lane's four values in slot i (fixed per lane).
  int vt[SLOTS], vtok[SLOTS], vrow[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = 4 * lane + 128 * i;
    vt[i] = e / nvt;
    const int rest = e - vt[i] * nvt;
    vtok[i] = rest >> 4;
    vrow[i] = rest & 15;
  }
  const int njt = (wk.njobs + JT - 1) / JT;  // hand-offs of this CTA
  const bool topk = head && a.tk_k > 0 && (ks == 1 || wk.rank == 0);
  unsigned long long* tk_list = nullptr;
  unsigned long long* tk_buf = nullptr;
  int* tk_cnt = nullptr;
  if (topk) {
    const size_t me = static_cast<size_t>(blockIdx.x / ks) * kEpiWarps + ew;
    tk_list = a.tk_lists + me * kHeadMaxT * 32;
    tk_buf = a.tk_bufs + me * kHeadMaxT * 64;
    tk_cnt = reinterpret_cast<int*>(smem + a.off_tk) + ew * kHeadMaxT;
    for (int t = 0; t < T; ++t) tk_list[t * 32 + lane] = 0ull;  // empty keys
    if (lane < T) tk_cnt[lane] = 0;
    __syncwarp();
  }
  int b = ew;        // buffer of hand-off j (j % nbuf)
  uint32_t n = 0;    // uses of that buffer so far (j / nbuf)
  int j = ew;
  if constexpr (CONT) {
    j = (ew - h0 % kEpiWarps + kEpiWarps) % kEpiWarps;  // first local hand-off of this warp
    b = (h0 + j) % a.nbuf;
    n = static_cast<uint32_t>((h0 + j) / a.nbuf);
  }
  for (; j < njt; j += kEpiWarps) {
    // Cluster-exchange buffer of this hand-off: its position among this
    // launch's K-split hand-offs, the same on every rank (a continuing phase
    // starts its own count; its red buffers continue the CTA's count).
    const int cb = CONT ? j % a.nbuf : b;
    const uint32_t cn = CONT ? static_cast<uint32_t>(j / a.nbuf) : n;
    if (ks > 1 && wk.rank == 0 && lane == 0)
      mbar_arrive_expect_tx_relaxed(bars.cl_full(cb), cl_bytes);
    if (!wt.wait_warp<false>(bars.red_full(b), n & 1u)) return;
    float4 v[SLOTS];
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (has(i)) {
        const float* p = red + b * kWarps * nv + 4 * lane + 128 * i;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) add4(v[i], *reinterpret_cast<const float4*>(p + w * nv));
      }
    }
    // Every lane has consumed its loads of the slot (the sums above); a
    // release here would also wait for the previous job's y stores.
    mbar_arrive_relaxed(bars.red_empty(b));  // every lane: count 32
    bool store = true;
    if (ks > 1) {
      if (wk.rank != 0) {
        if (!wt.wait_warp<false>(bars.cl_empty(cb), (cn & 1u) ^ 1u)) return;
        const uint32_t dst0 =
            map_to_rank(smem_addr(cl + (cb * (ks - 1) + (wk.rank - 1)) * nv + 4 * lane), 0);
        const uint32_t bar0 = map_to_rank(bars.cl_full(cb), 0);
#pragma unroll
        for (int i = 0; i < SLOTS; ++i)
          if (has(i)) st_async_v4(dst0 + 512 * i, v[i], bar0);
        store = false;
      } else {
        if (!wt.wait_warp<false>(bars.cl_full(cb), cn & 1u)) return;
        for (int p = 1; p < ks; ++p) {
          const float* src = cl + (cb * (ks - 1) + (p - 1)) * nv + 4 * lane;
#pragma unroll
          for (int i = 0; i < SLOTS; ++i)
            if (has(i)) add4(v[i], *reinterpret_cast<const float4*>(src + 128 * i));
        }
        __syncwarp();
        if (lane == 0) {
          for (int p = 1; p < ks; ++p) mbar_arrive_remote_relaxed(map_to_rank(bars.cl_empty(cb), p));
        }
      }
    }
    if (store && a.act != nullptr) {
      // Lanes 4m + {0, 1} hold gate rows 0..7 of their tile and token, lanes
      // 4m + {2, 3} the up rows of the same indices (rows 8..15).
      const long long ni = a.N >> 1;
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) {
        float4 up;
        up.x = __shfl_down_sync(0xffffffffu, v[i].x, 2);
        up.y = __shfl_down_sync(0xffffffffu, v[i].y, 2);
        up.z = __shfl_down_sync(0xffffffffu, v[i].z, 2);
        up.w = __shfl_down_sync(0xffffffffu, v[i].w, 2);
        if (has(i) && (vrow[i] & 8) == 0 && j * JT + vt[i] < wk.njobs) {
          const long long idx = (wk.rt_begin + j * JT + vt[i]) * 8 + vrow[i];
          const __nv_bfloat162 lo = __floats2bfloat162_rn(silu_mul(v[i].x, up.x), silu_mul(v[i].y, up.y));
          const __nv_bfloat162 hi = __floats2bfloat162_rn(silu_mul(v[i].z, up.z), silu_mul(v[i].w, up.w));
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(a.act + vtok[i] * ni + idx) = pk;
        }
      }
      if (a.sync != nullptr) {
        // One-launch layer: publish this hand-off's activations (every
        // lane's stores, then one count) to the down phase's consumers.
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(a.sync, static_cast<unsigned>(min(JT, wk.njobs - j * JT)));
      }
    } else if (store) {
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) {
        if (has(i) && j * JT + vt[i] < wk.njobs) {
          const long long row0 = (wk.rt_begin + j * JT + vt[i]) * 16;
          const int tok = vtok[i], row = vrow[i];
          const long long nrow = a.N - (row0 + row);  // rows left in y from this one
          const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
          if (a.y != nullptr) {
            float* yp = a.y + static_cast<long long>(tok) * a.N + row0 + row;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (c < nrow) yp[c] = vv[c];
          }
          if (head) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (c < nrow) head_push(hm[i], hs[i], ha[i], vv[c], static_cast<int>(row0 + row + c));
          }
        }
      }
      if (topk) {
        bool ok[SLOTS];
        long long rbase[SLOTS];
#pragma unroll
        for (int i = 0; i < SLOTS; ++i) {
          ok[i] = has(i) && j * JT + vt[i] < wk.njobs;
          rbase[i] = (wk.rt_begin + j * JT + vt[i]) * 16 + vrow[i];
        }
        topk_update<SLOTS>(a, tk_list, tk_buf, tk_cnt, lane, v, ok, rbase, vtok);
      }
    }
    b += kEpiWarps;
    if (b >= a.nbuf) { b -= a.nbuf; ++n; }
  }
  if (topk) {
    for (int t = 0; t < T; ++t)
      if (tk_cnt[t] > 0) topk_flush(tk_list, tk_buf, tk_cnt, t, lane);
  }
  if (head && (ks == 1 || wk.rank == 0)) head_finish<SLOTS>(a, wk, ew, lane, hm, hs, ha, vtok);
}

// ------------------------------------------------------------------ kernel
template <int BITS, int ROUTE, int NTOK>
__global__ void __launch_bounds__(kThreads, 1) nq_gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Bars bars{smem_addr(smem)};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortFlagOffset);
  const Waiter wt{abort_flag, a.wait_ns, a.status};
  const Work wk = cta_work(a);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), kWarps);
    }
    if constexpr (NTOK == kNtokXreg2) {
      // The fused head with a K split finalises by reduce-scatter
      // (epilogue_rs): each other finalising rank releases the buffer.
      constexpr int kJt = kJobTiles<ROUTE, NTOK>;
      const unsigned rel = (a.h_ws != nullptr && a.ksplit > 1)
                               ? cl_empty_count<2 * kJt>(a.ksplit, kJt * 16 * a.T, wk.rank)
                               : 1u;
      for (int b = 0; b < a.nbuf; ++b) {
        mbar_init(bars.red_full(b), 32 * kWarps);
        mbar_init(bars.red_empty(b), 32);
        mbar_init(bars.cl_full(b), 1);  // the finalising rank's expect_tx; peers' bytes
        mbar_init(bars.cl_empty(b), rel);
      }
    } else {
      for (int b = 0; b < a.nbuf; ++b) {
        mbar_init(bars.red_full(b), 32 * kWarps);
        mbar_init(bars.red_empty(b), 32);
        mbar_init(bars.cl_full(b), 1);   // rank 0's expect_tx; peers' bytes
        mbar_init(bars.cl_empty(b), 1);  // rank 0, once per job
      }
    }
    *abort_flag = 0;
    for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t*>(smem + kZeroAreaOffset)[i] = 0u;
    mbar_init(smem_addr(smem + kXFreeBarOffset), kWarps);
    uint32_t* stat = reinterpret_cast<uint32_t*>(smem + kXStatOffset);
    for (int t = 0; t < 16; ++t) {
      stat[t] = 0u;
      stat[16 + t] = 0x7FFFu;
    }
    stat[32] = 0u;
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
  } else if (warp >= kEpilogueWarp) {
    const int ew = warp - kEpilogueWarp;
    griddep_wait();
    // Value slots per lane: 16 x T values over 32 lanes.
    // Value slots per lane: JT x 16 x T values over 32 lanes, four each.
    constexpr int JT = kJobTiles<ROUTE, NTOK>;
    constexpr int kTokBlocks =
        (ROUTE == kRouteMma && (NTOK == 2 || NTOK == kNtokXreg2 || NTOK == kNtokXregH)) ? 2 : 1;
    if constexpr (NTOK == kNtokXreg2) {
      if (a.h_ws != nullptr && a.ksplit > 1)
        epilogue_rs<JT * kTokBlocks, JT>(a, smem, bars, wt, wk, ew, lane);
      else
        epilogue<JT * kTokBlocks, JT>(a, smem, bars, wt, wk, ew, lane);
    } else {
      epilogue<JT * kTokBlocks, JT>(a, smem, bars, wt, wk, ew, lane);
    }
  } else {
    griddep_wait();
    if constexpr (ROUTE == kRouteMma && NTOK == kNtokXreg) {
      consumer_xreg<BITS, kXregMaxGroups, 1>(a, smem, bars, wt, wk, warp, lane);
    } else if constexpr (ROUTE == kRouteMma && NTOK == kNtokXreg2) {
      consumer_xreg<BITS, kXreg2MaxGroups, 2>(a, smem, bars, wt, wk, warp, lane);
    } else if constexpr (ROUTE == kRouteMma && NTOK == kNtokXregH) {
      consumer_xregh<BITS>(a, smem, bars, wt, wk, warp, lane);
    } else {
      if constexpr (ROUTE == kRouteMma) {
        stage_x_bf16(a, smem, wk, threadIdx.x, kWarps * 32);
      } else {
        stage_x_f32(a, smem, wk, threadIdx.x, kWarps * 32);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
      consumer_xsmem<BITS, ROUTE, NTOK>(a, smem, bars, wt, wk, warp, lane);
    }
  }
  // No CTA may leave while cluster peers can still write into its shared
  // memory or arrive on its barriers.
  __syncwarp();
  if (a.ksplit > 1) cluster_sync_all();
}

// ------------------------------------------------------------------ one-launch MLP layer
// The decoder layer's MLP in one launch (pages "giveen/ninfer-ext", section
// "Where ninfer-ext leads", and "Qwen3.8-27B for NInfer on the RTX 3090",
// section "What is different from the upstream artifact": gate and up as one
// matrix, then the down projection).  Phase A is the gate+up product with the
// SwiGLU epilogue, every CTA working alone (no K split); phase B is the down
// projection over the activations phase A wrote, in clusters of b.ksplit.
// Both phases share the stage ring and the partial-buffer ring, so the
// producer streams phase B's weights while phase A finishes, and phase B's
// consumers start on full stages once every activation is published.

// Issues the bulk copies of one phase's jobs (the loop body of producer()).
template <int BITS>
__device__ __forceinline__ bool producer_phase(const GemvArgs& a, uint8_t* smem, const Bars& bars,
                                               const Waiter& wt, const Work& wk, uint64_t policy,
                                               int& stage, uint32_t& phase, uint32_t& issued,
                                               uint32_t& last_par, bool& x_pending) {
  constexpr int kBlock = 128 * BITS;
  const uint32_t ring = smem_addr(smem + a.off_ring);
  const int sg = a.stage_groups;
  for (int j = 0; j < wk.njobs; ++j) {
    const long long blk_job = (wk.rt_begin + j) * a.G;
    for (int g0 = wk.g_begin; g0 < wk.g_end; g0 += sg) {
      const int ng = min(sg, wk.g_end - g0);
      if (!wt.wait<false>(bars.empty(stage), phase ^ 1)) return false;
      if (x_pending && stage >= a.xh_stage0) {
        if (!wt.wait<false>(smem_addr(smem + kXFreeBarOffset), 0)) return false;
        fence_proxy_async_smem();
        x_pending = false;
      }
      const uint32_t bc = static_cast<uint32_t>(ng * kBlock);
      const uint32_t bs = static_cast<uint32_t>(ng * kScaleBytesPerBlock);
      const uint32_t dst = ring + stage * a.stage_bytes;
      const long long blk = blk_job + g0;
      mbar_arrive_expect_tx(bars.full(stage), bc + bs);
      bulk_g2s(dst, a.codes + blk * kBlock, bc, bars.full(stage), policy);
      bulk_g2s(dst + sg * kBlock, a.scales + blk * 16, bs, bars.full(stage), policy);
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
  }
  return true;
}

template <int BITS_A, int BITS_B>
__device__ void producer_layer(const GemvArgs& a, const GemvArgs& b, uint8_t* smem, const Bars& bars,
                               const Waiter& wt, const Work& wa, const Work& wb) {
  const uint64_t policy = l2_evict_first_policy();
  int stage = 0;
  uint32_t phase = 0, issued = 0, last_par = 0;
  bool x_pending = a.off_xh >= 0;
  if (producer_phase<BITS_A>(a, smem, bars, wt, wa, policy, stage, phase, issued, last_par, x_pending))
    (void)producer_phase<BITS_B>(b, smem, bars, wt, wb, policy, stage, phase, issued, last_par,
                                 x_pending);
  volatile int no_abort = 0;
  const Waiter drain{&no_abort, wt.limit, wt.status};
  for (int s = 0; s < a.stages; ++s)
    if (issued & (1u << s)) (void)drain.wait<false>(bars.full(s), (last_par >> s) & 1u);
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Consumer warps: wait until every activation of phase A is published.  Warp
// 0 polls (bounded); the others wait at a barrier of the consumer warps.
// The last CTA to pass resets the pair for the next launch that uses it.
__device__ __forceinline__ bool wait_activations(const GemvArgs& b, const Waiter& wt, int warp,
                                                 int lane) {
  if (warp == 0 && lane == 0) {
    const uint64_t t0 = global_ns();
    while (ld_acquire_gpu(b.sync) < static_cast<unsigned>(b.sync_target)) {
      if (*wt.abort) break;
      if (global_ns() - t0 > wt.limit) {
        *wt.abort = 1;
        atomicCAS(wt.status, 0, kStatusTimeout);
        break;
      }
      __nanosleep(32);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
  if (*wt.abort) return false;
  (void)ld_acquire_gpu(b.sync);  // orders this lane's loads of the activations
  if (warp == 0 && lane == 0 && atomicAdd(b.sync + 1, 1u) == gridDim.x - 1) {
    atomicExch(b.sync, 0u);
    atomicExch(b.sync + 1, 0u);
  }
  return true;
}

template <int BITS_A, int BITS_B>
__global__ void __launch_bounds__(kThreads, 1)
    nq_mlp_kernel(const __grid_constant__ GemvArgs a, const __grid_constant__ GemvArgs b) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Bars bars{smem_addr(smem)};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortFlagOffset);
  const Waiter wt{abort_flag, a.wait_ns, a.status};
  const Work wa = cta_work(a);  // phase A: every CTA alone (a.ksplit == 1)
  const Work wb = cta_work(b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), kWarps);
    }
    for (int i = 0; i < a.nbuf; ++i) {
      mbar_init(bars.red_full(i), 32 * kWarps);
      mbar_init(bars.red_empty(i), 32);
      mbar_init(bars.cl_full(i), 1);
      mbar_init(bars.cl_empty(i), 1);
    }
    *abort_flag = 0;
    for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t*>(smem + kZeroAreaOffset)[i] = 0u;
    mbar_init(smem_addr(smem + kXFreeBarOffset), kWarps);
    uint32_t* stat = reinterpret_cast<uint32_t*>(smem + kXStatOffset);
    for (int t = 0; t < 16; ++t) {
      stat[t] = 0u;
      stat[16 + t] = 0x7FFFu;
    }
    stat[32] = 0u;
    fence_mbar_init();
  }
  griddep_launch_dependents();
  if (b.ksplit > 1) cluster_sync_all(); else __syncthreads();

  if (warp == kProducerWarp) {
    if (lane == 0) producer_layer<BITS_A, BITS_B>(a, b, smem, bars, wt, wa, wb);
  } else if (warp >= kEpilogueWarp) {
    const int ew = warp - kEpilogueWarp;
    griddep_wait();
    epilogue<2, 2, true>(a, smem, bars, wt, wa, ew, lane, 0);
    epilogue<2, 2, true>(b, smem, bars, wt, wb, ew, lane, (wa.njobs + 1) / 2);
  } else {
    griddep_wait();
    RingPos pos{0, 0u, 0, 0u};
    consumer_xreg<BITS_A, kXregMaxGroups, 1, true>(a, smem, bars, wt, wa, warp, lane, &pos);
    if (wait_activations(b, wt, warp, lane))
      consumer_xreg<BITS_B, kXregMaxGroups, 1, true>(b, smem, bars, wt, wb, warp, lane, &pos);
  }
  __syncwarp();
  if (b.ksplit > 1) cluster_sync_all();
}

}  // namespace nq
