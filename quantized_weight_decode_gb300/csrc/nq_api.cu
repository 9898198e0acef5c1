// Host side of the C ABI declared in include/nq.h: argument validation, the
// host packer, launch planning and kernel launches.  Every step of the
// computation runs in the kernels of gemv_q*.cu and aux_kernels.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <climits>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "gemv.cuh"
#include "layout.h"
#include "nq.h"

namespace nq {
const void* gemv_kernel_q4(int route, int ntok);
const void* gemv_kernel_q5(int route, int ntok);
const void* gemv_kernel_q6(int route, int ntok);
const void* gemv_kernel_q8(int route, int ntok);
cudaError_t launch_pack_device(const int8_t*, const uint16_t*, long long, long long, int, void*,
                               uint16_t*, cudaStream_t);
cudaError_t launch_dequant(const void*, const uint16_t*, float*, long long, long long, int,
                           cudaStream_t);
cudaError_t launch_quantize_rtn(const float*, long long, long long, int, int8_t*, uint16_t*, int*,
                                cudaStream_t);
cudaError_t launch_quantize_search(const float*, const float*, long long, long long, int, int8_t*,
                                   uint16_t*, int*, cudaStream_t);
cudaError_t launch_selftest_timeout(unsigned long long, int*, cudaStream_t);
cudaError_t launch_topk_merge(const unsigned long long*, int, int, int, int32_t*, float*, bool,
                              cudaStream_t);
int* device_status_ptr();
unsigned* sync_slots_ptr();
const void* mlp_kernel(int bits_gu, int bits_down);

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxT = 16;
constexpr int kFfmaMaxT = 4;

struct DevInfo {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
  int* status = nullptr;
  unsigned* sync = nullptr;  // activation counters of the one-launch layer (kSyncSlots pairs)
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
std::map<std::tuple<int, const void*>, bool> g_func_ready;
std::map<std::tuple<int, const void*, int, int>, int> g_clusters;
// Streams whose last launch by this library wrote packed weights
// (nq_pack_device): the next GEMV on such a stream is launched without
// programmatic dependent launch, because the GEMV's producer starts reading
// weights before it waits for the preceding kernel.
std::map<cudaStream_t, bool> g_weights_written;
std::atomic<unsigned> g_sync_eager{0};
std::atomic<unsigned> g_sync_capture{0};

void mark_weights_written(cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_weights_written[st] = true;
}
// True if the preceding launch of this library on `st` wrote packed weights
// (and forgets it: the GEMV about to launch orders everything after it).
bool take_weights_written(cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_weights_written.find(st);
  if (it == g_weights_written.end() || !it->second) return false;
  it->second = false;
  return true;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  if (*dev < 0 || *dev >= kMaxDevices) return NQ_ECUDA;
  return NQ_OK;
}

int dev_info(DevInfo** out) {
  int dev;
  if (int rc = current_device(&dev)) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      (void)cudaGetLastError();
      return NQ_ECUDA;
    }
    d.status = device_status_ptr();
    d.sync = sync_slots_ptr();
    if (!d.status || !d.sync) {
      (void)cudaGetLastError();
      return NQ_ECUDA;
    }
    d.ready = true;
  }
  *out = &d;
  return NQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int64_t K, int64_t N, int bits) {
  if (K <= 0 || N <= 0 || K % kGroup != 0) return NQ_EINVAL;
  if (bits < 4 || bits > 8 || bits == 7) return NQ_EINVAL;
  // The kernels index groups and row tiles with 32-bit integers.
  if (K / kGroup > (1LL << 30) || (N + kTileRows - 1) / kTileRows > INT_MAX) return NQ_EINVAL;
  return NQ_OK;
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::atoi(v);
}

int env_route() {
  const char* v = std::getenv("NQ_ROUTE");
  if (!v || !*v) return NQ_ROUTE_AUTO;
  if (!std::strcmp(v, "mma")) return NQ_ROUTE_MMA;
  if (!std::strcmp(v, "ffma")) return NQ_ROUTE_FFMA;
  return NQ_ROUTE_AUTO;
}

const void* kernel_for(int bits, int route, int ntok) {
  switch (bits) {
    case 4: return gemv_kernel_q4(route, ntok);
    case 5: return gemv_kernel_q5(route, ntok);
    case 8: return gemv_kernel_q8(route, ntok);
    default: return gemv_kernel_q6(route, ntok);
  }
}

int align_up(int v, int a) { return (v + a - 1) / a * a; }

constexpr int kF16MaxT = 2;  // largest T that takes the fp16 route of 4-bit codes

struct Plan {
  int route = 0, ntok = 0, ks = 1, clusters = 0, sg = 1, stages = 0, stage_bytes = 0, nbuf = 2;
  int smem = 0, off_ring = 0, off_red = 0, off_cl = 0, off_x = 0;
  int off_xh = -1, xh_stage0 = 0;  // fp16 x staging of the 4-bit x-in-register kernels
  int off_tk = 0;                  // top-k lists of the fused head's epilogue warps
  const void* func = nullptr;
  double est_us = 0;
};

// Shared-memory layout for a K-split, a stage size (64-groups per stage) and a
// number of partial-sum buffers; false if fewer than `min_stages` stages fit.
bool layout_nbuf(const Plan& base, int G, int T, int bits, int ks, int sg, int min_stages,
                 int smem_optin, int extra, int nbuf, Plan* out) {
  Plan p = base;
  p.ks = ks;
  p.sg = sg;
  p.nbuf = nbuf;
  const int gc_max = (G + ks - 1) / ks;
  const bool x_in_regs = p.route == NQ_ROUTE_MMA &&
                         (p.ntok == kNtokXreg || p.ntok == kNtokXreg2 || p.ntok == kNtokXregH);
  // The hybrid kernel keeps the second token block's x in shared memory.
  const long long x_bytes =
      p.ntok == kNtokXregH ? 1LL * gc_max * (T - 8) * 128
      : x_in_regs          ? 0
                           : 1LL * gc_max * T * (p.route == NQ_ROUTE_MMA ? 128 : 256);
  const int jt = (x_in_regs && p.ntok == kNtokXreg) ? 2 : 1;   // the kernel's kJobTiles
  const int red_bytes = p.nbuf * kWarps * jt * 16 * T * 4;
  const int cl_bytes = ks > 1 ? p.nbuf * (ks - 1) * jt * 16 * T * 4 : 0;
  p.stage_bytes = align_up(sg * (block_bytes(bits) + kScaleBytesPerBlock), 128);
  p.off_red = kBarRegionBytes;
  p.off_cl = p.off_red + align_up(red_bytes, 128);
  p.off_x = p.off_cl + align_up(cl_bytes, 128);
  p.off_tk = p.off_x + align_up(static_cast<int>(std::min<long long>(x_bytes, 1 << 30)), 128);
  const long long fixed = p.off_tk + align_up(extra, 128);
  if (fixed >= smem_optin) return false;
  p.off_ring = static_cast<int>(fixed);
  p.stages = static_cast<int>(std::min<long long>(kMaxStages, (smem_optin - fixed) / p.stage_bytes));
  if (p.stages < min_stages) return false;
  p.smem = p.off_ring + p.stages * p.stage_bytes;
  // 4-bit codes with x in registers, T <= kF16MaxT: the consumers stage x
  // once as fp16 at the tail of the ring (T x 64 values x 2 B per group),
  // before the producer's first fill of the stages there; at least one stage
  // stays clear of it so the stream starts at once.  (Staging costs grow
  // with T; from T = 4 on they exceed what the shorter decode saves.)
  p.off_xh = -1;
  p.xh_stage0 = p.stages;
  if (x_in_regs && p.ntok == kNtokXreg && bits == 4 && T <= kF16MaxT &&
      env_int("NQ_X_F16", 1) != 0) {
    const int xh_bytes = align_up(gc_max * T * 128, 128);
    const int off = (p.smem - xh_bytes) / 128 * 128;
    if (off >= p.off_ring + p.stage_bytes) {
      p.off_xh = off;
      p.xh_stage0 = (off - p.off_ring) / p.stage_bytes;
    }
  }
  *out = p;
  return true;
}

// The layout with the deepest partial-sum buffering that still leaves three
// ring stages, else the standard depth.  Buffers in flight between the warps,
// the epilogue and the cluster's rank 0: deep for small T (cheap), shallower
// for large T; the x-in-register kernels with one token block hand over two
// row tiles per buffer (JT = 2), so they need half as many for the same
// slack.  Measured on GB300 (27B shapes): one step deeper than standard is
// 2-3 % faster at T = 8 and 16 where three stages remain (gate+up 23.1 ->
// 22.6 us at T = 8, 33.5 -> 32.3 us at T = 16; down 17.4 -> 17.0 us at
// T = 8; head 213.7 -> 206.7 us at T = 16), and slower where it costs the
// third stage (the head at T = 8: 152 -> 160 us).  Counts are multiples of
// kEpiWarps: each buffer belongs to one epilogue warp.
bool layout_for(const Plan& base, int G, int T, int bits, int ks, int sg, int min_stages,
                int smem_optin, int extra, Plan* out) {
  const bool x_in_regs = base.route == NQ_ROUTE_MMA && (base.ntok == kNtokXreg ||
                                                        base.ntok == kNtokXreg2 ||
                                                        base.ntok == kNtokXregH);
  const int jt = (x_in_regs && base.ntok == kNtokXreg) ? 2 : 1;
  int std_nbuf, deep_nbuf;
  if (jt == 2) {
    std_nbuf = T <= 2 ? 4 : 2;
    // T <= 4: eight pair buffers (at T = 1 a whole CTA's share of the
    // 34,816-row gate+up product), so the consumers hardly ever wait for the
    // epilogue: gate+up 19.1 -> 18.7 us at T = 1 and 20.1 -> 19.8 us at T = 4,
    // down 15.1 -> 14.8 us at T = 4, even at one ring stage less; the same at
    // T = 2 within noise; the head keeps its third stage (and its depth).
    deep_nbuf = T <= 4 ? kMaxBufs : 4;
  } else {
    std_nbuf = T <= 2 ? kMaxBufs : T <= 4 ? 6 : T <= 8 ? 4 : 2;
    deep_nbuf = T <= 8 ? std_nbuf : 6;
  }
  static_assert(kMaxBufs % kEpiWarps == 0 && 6 % kEpiWarps == 0 && 4 % kEpiWarps == 0 &&
                    2 % kEpiWarps == 0,
                "buffer counts must be multiples of the epilogue warps");
  if (deep_nbuf > std_nbuf &&
      layout_nbuf(base, G, T, bits, ks, sg, std::max(3, min_stages), smem_optin, extra, deep_nbuf,
                  out))
    return true;
  return layout_nbuf(base, G, T, bits, ks, sg, min_stages, smem_optin, extra, std_nbuf, out);
}

int prepare_func(int dev, const void* func, int smem_optin) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, func);
  if (g_func_ready.count(key)) return NQ_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  g_func_ready[key] = true;
  return NQ_OK;
}

// Clusters of `ks` CTAs (one CTA per SM) that can be resident at once.
int max_clusters(int dev, const DevInfo& d, const void* func, int ks, int smem) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_clusters.find(std::make_tuple(dev, func, ks, smem));
    if (it != g_clusters.end()) return it->second;
  }
  int n = 0;
  if (ks == 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, kThreads, smem) != cudaSuccess)
      per_sm = 1;
    n = std::max(1, per_sm) * d.sms;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ks * std::max(1, d.sms / ks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = ks;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = d.sms / ks;
    }
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_clusters[std::make_tuple(dev, func, ks, smem)] = n;
  return n;
}

// Rough time model: the weight stream at the HBM rate while every SM is busy,
// the last partial wave at the per-SM rate of the SMs that still have work.
// The per-SM rate is capped by the bytes a CTA keeps in flight (Little's law
// with ~1 us of memory latency) and by the bulk-copy requests it issues
// (~60 ns each, two per stage).
double estimate_us(const Plan& p, long long Nt, int G, int bits) {
  const double bw = 6.5e12, bw_sm_max = 1.1e11, latency_s = 1.0e-6, request_s = 60e-9;
  const double group_bytes = block_bytes(bits) + kScaleBytesPerBlock;
  const double inflight = static_cast<double>(p.stages) * p.sg * group_bytes;
  const double stage_rate = p.sg * group_bytes / (2 * request_s);
  const double bw_sm = std::min(std::min(bw_sm_max, inflight / latency_s), stage_rate);
  const int gc_max = (G + p.ks - 1) / p.ks;
  const double job_bytes = gc_max * group_bytes;
  const long long C = p.clusters;
  const long long rounds = Nt / C, rem = Nt % C;
  const double act = static_cast<double>(C) * p.ks;
  double t = rounds * act * job_bytes / std::min(bw, act * bw_sm);
  if (rem) {
    const double ract = static_cast<double>(rem) * p.ks;
    t += ract * job_bytes / std::min(bw, ract * bw_sm);
  }
  t *= 1e6;
  t += (p.ks > 1 ? 0.5 * p.ks : 0.0);
  return t;
}

// extra: shared-memory bytes the epilogue needs besides the plain GEMV's (the
// fused head's top-k lists), placed at Plan::off_tk.
int make_plan(int64_t K, int64_t N, int T, int bits, int route, int ksplit, Plan* out,
              int extra = 0) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (T < 1 || T > kMaxT) return NQ_EINVAL;
  if (route == NQ_ROUTE_AUTO) route = env_route();
  if (route == NQ_ROUTE_AUTO) route = NQ_ROUTE_MMA;
  if (route != NQ_ROUTE_MMA && route != NQ_ROUTE_FFMA) return NQ_EINVAL;
  if (route == NQ_ROUTE_FFMA && T > kFfmaMaxT) return NQ_EINVAL;
  if (route == NQ_ROUTE_FFMA && bits == 8) return NQ_EINVAL;  // 8-bit codes: MMA route only
  if (ksplit == 0) ksplit = env_int("NQ_KSPLIT", 0);
  if (ksplit != 0 && ksplit != 1 && ksplit != 2 && ksplit != 4 && ksplit != 8) return NQ_EINVAL;

  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  int dev;
  if (int rc = current_device(&dev)) return rc;

  Plan base;
  base.route = route;
  base.ntok = route == NQ_ROUTE_MMA ? (T <= 8 ? 1 : 2) : kFfmaMaxT;
  base.func = kernel_for(bits, route, base.ntok);
  if (int rc = prepare_func(dev, base.func, d->smem_optin)) return rc;
  // x-in-register variants, in order of preference at one K split: one
  // token block (T <= 8, warp slices of up to kXregMaxGroups groups); for two
  // blocks (T <= 16) both in registers (up to kXreg2MaxGroups), else the
  // hybrid with the second block in shared memory (up to kXregMaxGroups).
  // NQ_XREGH=0 leaves the hybrid out, NQ_XREGH=1 takes only the hybrid.
  struct XregVariant {
    Plan plan;
    int max_groups;
  };
  XregVariant xv[2];
  int nxv = 0;
  if (route == NQ_ROUTE_MMA) {
    const int hyb = env_int("NQ_XREGH", -1);
    const int ntoks[2] = {T <= 8 ? kNtokXreg : (hyb == 1 ? 0 : kNtokXreg2),
                          T <= 8 || hyb == 0 ? 0 : kNtokXregH};
    for (int ntok : ntoks) {
      if (ntok == 0) continue;
      Plan xr = base;
      xr.ntok = ntok;
      xr.func = kernel_for(bits, route, ntok);
      if (int rc = prepare_func(dev, xr.func, d->smem_optin)) return rc;
      xv[nxv].plan = xr;
      xv[nxv].max_groups = ntok == kNtokXreg2 ? kXreg2MaxGroups : kXregMaxGroups;
      ++nxv;
    }
  }

  const int G = static_cast<int>(K / kGroup);
  const long long Nt = (N + kTileRows - 1) / kTileRows;
  const int cands[4] = {1, 2, 4, 8};
  bool have = false;
  Plan best;
  // The x-in-register kernel at the smallest K split (up to 4) that allows
  // it beats every other candidate on GB300 -- measured on the 27B shapes
  // (T <= 8, K = 5120: KS 1; K = 17408: KS 4, 7-15 % ahead of KS 1/2 with x
  // in shared memory; T = 12 and 16, K = 5120: KS 2, 205 / 213 us on the
  // 248,320-row head against 230 / 372 us at KS 1 with x in shared memory) --
  // because its consumers issue the fewest instructions per weight, and the
  // split's per-job overhead grows with KS.  For T > 8 the hybrid's smaller
  // split pays (gate+up T = 16: KS 1, 27.3 us against 29.0 us with both
  // blocks in registers at KS 2; 5-bit down T = 16: KS 4, 19.1 us against
  // 24.1 us; head T = 12: KS 1, 170.7 against 194.6 us), but at an equal
  // split both blocks in registers are faster (head T = 16, KS 2: 197.0
  // against 203.8 us).  No such candidate: the time model below decides.
  bool have_xreg = false;
  Plan best_xreg;
  for (int ks : cands) {
    if (ksplit != 0 && ks != ksplit) continue;
    if (ks > G) continue;
    const int gc_max = (G + ks - 1) / ks;
    const int gw_max = (gc_max + kWarps - 1) / kWarps;
    Plan p;
    bool fit = false;
    for (int v = 0; v < nxv && !fit; ++v) {
      // x held in registers; a stage is the CTA's whole K range of one job.
      if (gw_max <= xv[v].max_groups)
        fit = layout_for(xv[v].plan, G, T, bits, ks, gc_max, 2, d->smem_optin, extra, &p);
    }
    const bool is_xreg = fit;
    // Otherwise x in shared memory; a stage is the job's K range cut into
    // `parts` equal pieces, the fewest that leave at least 3 stages (2 when
    // a piece is down to one group per warp).
    for (int parts = 1; !fit && parts <= gc_max; ++parts) {
      const int sg = (gc_max + parts - 1) / parts;
      fit = layout_for(base, G, T, bits, ks, sg, sg <= kWarps ? 2 : 3, d->smem_optin, extra, &p);
      if (sg <= kWarps) break;
    }
    if (!fit) continue;
    const int mc = max_clusters(dev, *d, p.func, ks, p.smem);
    if (mc <= 0) continue;
    p.clusters = static_cast<int>(std::min<long long>(mc, Nt));
    p.est_us = estimate_us(p, Nt, G, bits);
    if (!have || p.est_us < best.est_us - 1e-3) {
      best = p;
      have = true;
    }
    if (!have_xreg && ks <= 4 && is_xreg) {
      best_xreg = p;
      have_xreg = true;
    }
  }
  if (!have) return NQ_EUNSUPPORTED;
  *out = have_xreg ? best_xreg : best;
  return NQ_OK;
}

// Outputs of the fused verify head (all null for a plain GEMV).
struct HeadOut {
  void* ws = nullptr;
  int32_t* argmax = nullptr;
  float* maxval = nullptr;
  float* lse = nullptr;
  int tk_k = 0;                           // top-k (0: none)
  unsigned long long* tk_lists = nullptr;
  unsigned long long* tk_bufs = nullptr;
};

int launch_plan(const Plan& p, const void* packed, const uint16_t* scales, const void* x, float* y,
                int64_t K, int64_t N, int T, cudaStream_t st, const HeadOut& head = HeadOut(),
                uint16_t* act = nullptr) {
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  GemvArgs a = {};  // every field not set below is zero (null sync: a plain product)
  a.codes = static_cast<const uint8_t*>(packed);
  a.scales = scales;
  a.x = static_cast<const uint16_t*>(x);
  a.y = y;
  a.N = N;
  a.K = static_cast<int>(K);
  a.T = T;
  a.G = static_cast<int>(K / kGroup);
  a.Nt = static_cast<int>((N + kTileRows - 1) / kTileRows);
  a.ksplit = p.ks;
  a.clusters = p.clusters;
  a.stage_groups = p.sg;
  a.stages = p.stages;
  a.stage_bytes = p.stage_bytes;
  a.off_ring = p.off_ring;
  a.off_red = p.off_red;
  a.off_cl = p.off_cl;
  a.off_x = p.off_x;
  a.off_xh = p.off_xh;
  a.xh_stage0 = p.xh_stage0;
  a.nbuf = p.nbuf;
  a.wait_ns = static_cast<unsigned long long>(std::max(1, env_int("NQ_WAIT_MS", 2000))) * 1000000ULL;
  a.status = d->status;
  a.h_ws = static_cast<uint8_t*>(head.ws);
  a.h_argmax = head.argmax;
  a.h_max = head.maxval;
  a.h_lse = head.lse;
  a.tk_k = head.tk_k;
  a.off_tk = p.off_tk;
  a.tk_lists = head.tk_lists;
  a.tk_bufs = head.tk_bufs;
  a.act = act;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.clusters * p.ks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (p.ks > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = p.ks;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  const bool after_pack = take_weights_written(st);
  if (env_int("NQ_PDL", 1) != 0 && !after_pack) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, p.func, args) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

// ---------------------------------------------------------------- one-launch MLP layer
struct MlpPlan {
  Plan p;                // shared layout: ring, partial buffers, fp16 staging of phase A
  int ks = 1;            // K split of the down phase (cluster size)
  int sg_a = 0, sg_b = 0;
};

// The layer runs in one launch when both phases fit the x-in-register kernel
// with one token block (T <= 8): the gate+up phase without a K split (at
// most 5 x 16 groups of K), the down phase at the K split nq_gemv would use.
// Anything else is NQ_EUNSUPPORTED, and nq_mlp takes two launches.
int make_mlp_plan(int64_t H, int64_t I, int64_t H_out, int T, int bits_gu, int bits_down,
                  MlpPlan* out) {
  if (T < 1 || T > 8) return NQ_EUNSUPPORTED;
  const void* func = mlp_kernel(bits_gu, bits_down);
  if (!func) return NQ_EUNSUPPORTED;
  if (int rc = check_shape(H, 2 * I, bits_gu)) return rc;
  if (int rc = check_shape(I, H_out, bits_down)) return rc;
  const int G_a = static_cast<int>(H / kGroup);
  if ((G_a + kWarps - 1) / kWarps > kXregMaxGroups) return NQ_EUNSUPPORTED;
  Plan pb;
  if (int rc = make_plan(I, H_out, T, bits_down, NQ_ROUTE_MMA, 0, &pb)) return rc;
  if (pb.ntok != kNtokXreg) return NQ_EUNSUPPORTED;
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  int dev;
  if (int rc = current_device(&dev)) return rc;
  if (int rc = prepare_func(dev, func, d->smem_optin)) return rc;
  const int ks = pb.ks;
  const int G_b = static_cast<int>(I / kGroup);
  const int gc_b = (G_b + ks - 1) / ks;
  const int sb_a = align_up(G_a * (block_bytes(bits_gu) + kScaleBytesPerBlock), 128);
  const int sb_b = align_up(gc_b * (block_bytes(bits_down) + kScaleBytesPerBlock), 128);
  const int stage_bytes = std::max(sb_a, sb_b);
  // Partial buffers as layout_for() sets them for the pair-of-tiles kernel:
  // the deep count where three ring stages remain, else the standard one.
  const int std_nbuf = T <= 2 ? 4 : 2, deep_nbuf = T <= 4 ? kMaxBufs : 4;
  Plan p;
  bool fit = false;
  for (int nbuf : {deep_nbuf, std_nbuf}) {
    const int red_bytes = nbuf * kWarps * 2 * 16 * T * 4;
    const int cl_bytes = ks > 1 ? nbuf * (ks - 1) * 2 * 16 * T * 4 : 0;
    p = Plan();
    p.route = NQ_ROUTE_MMA;
    p.ntok = kNtokXreg;
    p.ks = ks;
    p.nbuf = nbuf;
    p.stage_bytes = stage_bytes;
    p.off_red = kBarRegionBytes;
    p.off_cl = p.off_red + align_up(red_bytes, 128);
    p.off_x = p.off_cl + align_up(cl_bytes, 128);
    p.off_tk = p.off_x;
    p.off_ring = p.off_x;
    p.stages = std::min(kMaxStages, (d->smem_optin - p.off_ring) / stage_bytes);
    const int min_stages = (nbuf == deep_nbuf && deep_nbuf > std_nbuf) ? 3 : 2;
    if (p.stages >= min_stages) {
      fit = true;
      break;
    }
  }
  if (!fit) return NQ_EUNSUPPORTED;
  p.smem = p.off_ring + p.stages * stage_bytes;
  // Phase A's fp16 staging of x (4-bit gate+up, T <= 2) at the ring's tail,
  // as for the single product.
  p.off_xh = -1;
  p.xh_stage0 = p.stages;
  if (bits_gu == 4 && T <= kF16MaxT && env_int("NQ_X_F16", 1) != 0) {
    const int xh_bytes = align_up(G_a * T * 128, 128);
    const int off = (p.smem - xh_bytes) / 128 * 128;
    if (off >= p.off_ring + stage_bytes) {
      p.off_xh = off;
      p.xh_stage0 = (off - p.off_ring) / stage_bytes;
    }
  }
  p.func = func;
  const int mc = max_clusters(dev, *d, func, ks, p.smem);
  if (mc <= 0) return NQ_EUNSUPPORTED;
  p.clusters = mc;
  out->p = p;
  out->ks = ks;
  out->sg_a = G_a;
  out->sg_b = gc_b;
  return NQ_OK;
}

int launch_mlp(const MlpPlan& mp, const void* packed_gu, const uint16_t* scales_gu,
               const void* packed_down, const uint16_t* scales_down, const void* x, void* act,
               float* y, int64_t H, int64_t I, int64_t H_out, int T, cudaStream_t st) {
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  const Plan& p = mp.p;
  // This launch's activation counters: a slot of the eager pool, or of the
  // capture pool while the stream is being captured into a graph.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    cs = cudaStreamCaptureStatusNone;
  }
  const unsigned slot = cs == cudaStreamCaptureStatusActive
                            ? kSyncSlotsEager + g_sync_capture.fetch_add(1) % kSyncSlotsCapture
                            : g_sync_eager.fetch_add(1) % kSyncSlotsEager;
  GemvArgs a = {};
  a.codes = static_cast<const uint8_t*>(packed_gu);
  a.scales = scales_gu;
  a.x = static_cast<const uint16_t*>(x);
  a.y = nullptr;
  a.act = static_cast<uint16_t*>(act);
  a.N = 2 * I;
  a.K = static_cast<int>(H);
  a.T = T;
  a.G = static_cast<int>(H / kGroup);
  a.Nt = static_cast<int>((2 * I + kTileRows - 1) / kTileRows);
  a.ksplit = 1;                     // every CTA alone
  a.clusters = p.clusters * mp.ks;  // = CTAs
  a.stage_groups = mp.sg_a;
  a.stages = p.stages;
  a.stage_bytes = p.stage_bytes;
  a.off_ring = p.off_ring;
  a.off_red = p.off_red;
  a.off_cl = p.off_cl;
  a.off_x = p.off_x;
  a.off_xh = p.off_xh;
  a.xh_stage0 = p.xh_stage0;
  a.nbuf = p.nbuf;
  a.wait_ns = static_cast<unsigned long long>(std::max(1, env_int("NQ_WAIT_MS", 2000))) * 1000000ULL;
  a.status = d->status;
  a.sync = d->sync + 2 * static_cast<size_t>(slot);
  a.sync_target = 0;
  GemvArgs b = a;
  b.codes = static_cast<const uint8_t*>(packed_down);
  b.scales = scales_down;
  b.x = static_cast<const uint16_t*>(act);
  b.y = y;
  b.act = nullptr;
  b.N = H_out;
  b.K = static_cast<int>(I);
  b.G = static_cast<int>(I / kGroup);
  b.Nt = static_cast<int>((H_out + kTileRows - 1) / kTileRows);
  b.ksplit = mp.ks;
  b.clusters = p.clusters;
  b.stage_groups = mp.sg_b;
  // Phase B has no fp16 staging of its own, but its first fills of the stages
  // that overlap phase A's staging area must still wait until phase A's
  // consumers have taken their x (the producer's check uses xh_stage0).
  b.off_xh = -1;
  b.xh_stage0 = p.xh_stage0;
  b.sync_target = a.Nt;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.clusters * mp.ks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (mp.ks > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = mp.ks;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  const bool after_pack = take_weights_written(st);
  if (env_int("NQ_PDL", 1) != 0 && !after_pack) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  void* args[] = {&a, &b};
  if (cudaLaunchKernelExC(&cfg, p.func, args) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

// Identity row map: packed row n is row n of the inputs.
struct PlainRows {
  const int8_t* codes;
  const uint16_t* scales;
  const int8_t* code_row(int64_t n, int64_t K) const { return codes + n * K; }
  const uint16_t* scale_row(int64_t n, int64_t G) const { return scales + n * G; }
};
// Gate/up interleaving of nq_pack_gate_up: packed row 16 r + m is gate row
// 8 r + m and packed row 16 r + 8 + m is up row 8 r + m (m < 8).
struct GateUpRows {
  const int8_t *cg, *cu;
  const uint16_t *sg, *su;
  static int64_t src(int64_t n) { return (n >> 4) * 8 + (n & 7); }
  const int8_t* code_row(int64_t n, int64_t K) const { return ((n & 8) ? cu : cg) + src(n) * K; }
  const uint16_t* scale_row(int64_t n, int64_t G) const { return ((n & 8) ? su : sg) + src(n) * G; }
};

template <int BITS, class Rows>
void pack_host(const Rows& rows, int64_t K, int64_t N, uint8_t* out, uint16_t* sout) {
  const int64_t G = K / kGroup, Nt = (N + kTileRows - 1) / kTileRows;
  constexpr uint32_t bias = 1u << (BITS - 1);
  for (int64_t rt = 0; rt < Nt; ++rt) {
    for (int64_t g = 0; g < G; ++g) {
      const int64_t blk = rt * G + g;
      uint8_t* base = out + blk * block_bytes(BITS);
      for (int lane = 0; lane < kLanes; ++lane) {
        uint32_t u[32], w[8];
        for (int p = 0; p < 16; ++p) {
          for (int h = 0; h < 2; ++h) {
            int row, k;
            lane_code_coords(lane, p, h, &row, &k);
            const int64_t n = rt * kTileRows + row;
            const int c = n < N ? rows.code_row(n, K)[g * kGroup + k] : 0;
            u[2 * p + h] = static_cast<uint32_t>(c + static_cast<int>(bias));
          }
        }
        encode_lane(BITS, u, w);
        for (int i = 0; i < BITS; ++i) {
          std::memcpy(base + lane_word_offset(BITS, lane, i), &w[i], 4);
        }
      }
      for (int row = 0; row < kTileRows; ++row) {
        const int64_t n = rt * kTileRows + row;
        sout[blk * 16 + 2 * (row & 7) + (row >> 3)] = n < N ? rows.scale_row(n, G)[g] : 0;
      }
    }
  }
}

template <int BITS>
void unpack_host(const uint8_t* in, const uint16_t* sin, int64_t K, int64_t N, int8_t* codes,
                 uint16_t* scales) {
  const int64_t G = K / kGroup, Nt = (N + kTileRows - 1) / kTileRows;
  constexpr int bias = 1 << (BITS - 1);
  constexpr uint32_t mask = (1u << BITS) - 1;
  for (int64_t rt = 0; rt < Nt; ++rt) {
    for (int64_t g = 0; g < G; ++g) {
      const int64_t blk = rt * G + g;
      const uint8_t* base = in + blk * block_bytes(BITS);
      for (int lane = 0; lane < kLanes; ++lane) {
        uint32_t w[BITS];
        for (int i = 0; i < BITS; ++i) std::memcpy(&w[i], base + lane_word_offset(BITS, lane, i), 4);
        for (int p = 0; p < 16; ++p) {
          const uint32_t f = pair_field<BITS>(w, p);
          for (int h = 0; h < 2; ++h) {
            int row, k;
            lane_code_coords(lane, p, h, &row, &k);
            const int64_t n = rt * kTileRows + row;
            if (n >= N) continue;
            codes[n * K + g * kGroup + k] =
                static_cast<int8_t>(static_cast<int>((f >> (16 * h)) & mask) - bias);
          }
        }
      }
      for (int row = 0; row < kTileRows; ++row) {
        const int64_t n = rt * kTileRows + row;
        if (n < N) scales[n * G + g] = sin[blk * 16 + 2 * (row & 7) + (row >> 3)];
      }
    }
  }
}

}  // namespace
}  // namespace nq

using namespace nq;

extern "C" {

const char* nq_status_string(int status) {
  switch (status) {
    case NQ_OK: return "ok";
    case NQ_EINVAL: return "invalid argument (size, width, T, route or null pointer)";
    case NQ_EALIGN: return "device pointer not 16-byte aligned";
    case NQ_ERANGE: return "code out of range or scale not finite / overflowing FP16";
    case NQ_ECUDA: return "CUDA error";
    case NQ_ETIMEOUT: return "a kernel's bounded wait gave up";
    case NQ_EUNSUPPORTED: return "shape does not fit the shared-memory x tile";
    default: return "unknown status";
  }
}

int nq_layout_version(void) { return kLayoutVersion; }

int nq_packed_bytes(int64_t K, int64_t N, int bits, size_t* codes_bytes, size_t* scales_bytes) {
  if (int rc = check_shape(K, N, bits)) return rc;
  const int64_t G = K / kGroup, Nt = (N + kTileRows - 1) / kTileRows;
  if (codes_bytes) *codes_bytes = static_cast<size_t>(Nt * G * block_bytes(bits));
  if (scales_bytes) *scales_bytes = static_cast<size_t>(Nt * G * kScaleBytesPerBlock);
  return NQ_OK;
}

int nq_pack(const int8_t* codes, const uint16_t* scales, int64_t K, int64_t N, int bits,
            void* packed_out, uint16_t* scales_out) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (!codes || !scales || !packed_out || !scales_out) return NQ_EINVAL;
  const int lo = -(1 << (bits - 1)), hi = (1 << (bits - 1)) - 1;
  const int64_t total = K * N;
  for (int64_t i = 0; i < total; ++i)
    if (codes[i] < lo || codes[i] > hi) return NQ_ERANGE;
  const int64_t ns = N * (K / kGroup);
  for (int64_t i = 0; i < ns; ++i)
    if ((scales[i] & 0x7C00u) == 0x7C00u) return NQ_ERANGE;
  auto* out = static_cast<uint8_t*>(packed_out);
  const PlainRows rows{codes, scales};
  switch (bits) {
    case 4: pack_host<4>(rows, K, N, out, scales_out); break;
    case 5: pack_host<5>(rows, K, N, out, scales_out); break;
    case 8: pack_host<8>(rows, K, N, out, scales_out); break;
    default: pack_host<6>(rows, K, N, out, scales_out); break;
  }
  return NQ_OK;
}

int nq_pack_gate_up(const int8_t* codes_gate, const uint16_t* scales_gate, const int8_t* codes_up,
                    const uint16_t* scales_up, int64_t K, int64_t I, int bits, void* packed_out,
                    uint16_t* scales_out) {
  if (I <= 0 || I % 8 != 0) return NQ_EINVAL;
  if (int rc = check_shape(K, 2 * I, bits)) return rc;
  if (!codes_gate || !scales_gate || !codes_up || !scales_up || !packed_out || !scales_out)
    return NQ_EINVAL;
  const int lo = -(1 << (bits - 1)), hi = (1 << (bits - 1)) - 1;
  for (const int8_t* c : {codes_gate, codes_up})
    for (int64_t i = 0; i < K * I; ++i)
      if (c[i] < lo || c[i] > hi) return NQ_ERANGE;
  for (const uint16_t* sc : {scales_gate, scales_up})
    for (int64_t i = 0; i < I * (K / kGroup); ++i)
      if ((sc[i] & 0x7C00u) == 0x7C00u) return NQ_ERANGE;
  auto* out = static_cast<uint8_t*>(packed_out);
  const GateUpRows rows{codes_gate, codes_up, scales_gate, scales_up};
  switch (bits) {
    case 4: pack_host<4>(rows, K, 2 * I, out, scales_out); break;
    case 5: pack_host<5>(rows, K, 2 * I, out, scales_out); break;
    case 8: pack_host<8>(rows, K, 2 * I, out, scales_out); break;
    default: pack_host<6>(rows, K, 2 * I, out, scales_out); break;
  }
  return NQ_OK;
}

int nq_unpack(const void* packed, const uint16_t* scales_packed, int64_t K, int64_t N, int bits,
              int8_t* codes_out, uint16_t* scales_out) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (!packed || !scales_packed || !codes_out || !scales_out) return NQ_EINVAL;
  auto* in = static_cast<const uint8_t*>(packed);
  switch (bits) {
    case 4: unpack_host<4>(in, scales_packed, K, N, codes_out, scales_out); break;
    case 5: unpack_host<5>(in, scales_packed, K, N, codes_out, scales_out); break;
    case 8: unpack_host<8>(in, scales_packed, K, N, codes_out, scales_out); break;
    default: unpack_host<6>(in, scales_packed, K, N, codes_out, scales_out); break;
  }
  return NQ_OK;
}

int nq_pack_device(const int8_t* codes, const uint16_t* scales, int64_t K, int64_t N, int bits,
                   void* packed_out, uint16_t* scales_out, nq_stream_t stream) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (!codes || !scales || !packed_out || !scales_out) return NQ_EINVAL;
  if (!aligned16(codes) || !aligned16(packed_out) || !aligned16(scales_out)) return NQ_EALIGN;
  if (launch_pack_device(codes, scales, K, N, bits, packed_out, scales_out,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  mark_weights_written(reinterpret_cast<cudaStream_t>(stream));
  return NQ_OK;
}

int nq_quantize_rtn(const float* w, int64_t K, int64_t N, int bits, int8_t* codes_out,
                    uint16_t* scales_out, nq_stream_t stream) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (!w || !codes_out || !scales_out) return NQ_EINVAL;
  if (!aligned16(w) || !aligned16(codes_out)) return NQ_EALIGN;
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  if (launch_quantize_rtn(w, K, N, bits, codes_out, scales_out, d->status,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

int nq_quantize_search(const float* w, const float* imatrix, int64_t K, int64_t N, int bits,
                       int8_t* codes_out, uint16_t* scales_out, nq_stream_t stream) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (!w || !codes_out || !scales_out) return NQ_EINVAL;
  if (!aligned16(w) || !aligned16(codes_out) || (imatrix && !aligned16(imatrix))) return NQ_EALIGN;
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  if (launch_quantize_search(w, imatrix, K, N, bits, codes_out, scales_out, d->status,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

int nq_gemv_ex(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
               int64_t K, int64_t N, int T, int bits, int route, int ksplit, nq_stream_t stream) {
  if (!packed || !scales || !x_bf16 || !y) return NQ_EINVAL;
  if (int rc = check_shape(K, N, bits)) return rc;
  if (T < 1 || T > kMaxT) return NQ_EINVAL;
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(x_bf16) || !aligned16(y))
    return NQ_EALIGN;
  Plan p;
  if (int rc = make_plan(K, N, T, bits, route, ksplit, &p)) return rc;
  return launch_plan(p, packed, scales, x_bf16, y, K, N, T, reinterpret_cast<cudaStream_t>(stream));
}

int nq_gemv(const void* packed, const uint16_t* scales, const void* x_bf16, float* y, int64_t K,
            int64_t N, int T, int bits, nq_stream_t stream) {
  return nq_gemv_ex(packed, scales, x_bf16, y, K, N, T, bits, NQ_ROUTE_AUTO, 0, stream);
}

int nq_head_workspace_bytes(size_t* bytes) {
  if (!bytes) return NQ_EINVAL;
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  // one state per (CTA, epilogue warp, token) and per (group of
  // kHeadGroup CTAs, token); CTAs <= SMs
  const size_t groups = (static_cast<size_t>(d->sms) + kHeadGroup - 1) / kHeadGroup;
  *bytes = static_cast<size_t>(kHeadCounterBytes) +
           (static_cast<size_t>(d->sms) * kEpiWarps + groups) * kHeadMaxT * kHeadStateBytes;
  return NQ_OK;
}

// Shared by the fused head entry points: validation, the arrival counter
// clear, the head GEMV, and (k > 0) the top-k merge.
static int head_launch(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                       int64_t K, int64_t N, int T, int bits, int32_t* argmax, float* maxval,
                       float* lse, int k, int32_t* topk_idx, float* topk_val, void* workspace,
                       size_t workspace_bytes, nq_stream_t stream) {
  if (!packed || !scales || !x_bf16 || !argmax || !maxval || !lse || !workspace) return NQ_EINVAL;
  if (k < 0 || k > kTopkMax || (k > 0 && (!topk_idx || !topk_val))) return NQ_EINVAL;
  if (int rc = check_shape(K, N, bits)) return rc;
  if (T < 1 || T > kMaxT) return NQ_EINVAL;
  if (N > INT32_MAX) return NQ_EINVAL;  // row indices are int32
  {
    DevInfo* d;
    if (int rc = dev_info(&d)) return rc;
    if (d->sms > kHeadGroup * kHeadMaxGroups) return NQ_EUNSUPPORTED;  // merge covers 256 CTAs
  }
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(x_bf16) || !aligned16(workspace) ||
      (y && !aligned16(y)))
    return NQ_EALIGN;
  size_t need = 0;
  if (int rc = (k > 0 ? nq_head_topk_workspace_bytes(&need) : nq_head_workspace_bytes(&need)))
    return rc;
  if (workspace_bytes < need) return NQ_EINVAL;
  Plan p;
  if (int rc = make_plan(K, N, T, bits, NQ_ROUTE_AUTO, 0, &p,
                         k > 0 ? kTopkSmemBytes : 0))
    return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The arrival counter must start at zero on every call (a call that gave up
  // on a bounded wait leaves it behind).
  if (cudaMemsetAsync(workspace, 0, kHeadCounterBytes, st) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  HeadOut h;
  h.ws = workspace;
  h.argmax = argmax;
  h.maxval = maxval;
  h.lse = lse;
  size_t head_bytes = 0;
  if (k > 0) {
    if (int rc = nq_head_workspace_bytes(&head_bytes)) return rc;
    h.tk_k = k;
    h.tk_lists = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) +
                                                       align_up(static_cast<int>(head_bytes), 256));
    DevInfo* d;
    if (int rc = dev_info(&d)) return rc;
    h.tk_bufs = h.tk_lists + static_cast<size_t>(d->sms) * kEpiWarps * kHeadMaxT * 32;
  }
  if (int rc = launch_plan(p, packed, scales, x_bf16, y, K, N, T, st, h)) return rc;
  // one list per (unit, epilogue warp): per CTA where the kernel finalises by
  // reduce-scatter (two token blocks in registers, K split), else per cluster
  const int units = p.clusters * (p.ntok == kNtokXreg2 && p.ks > 1 ? p.ks : 1);
  if (k > 0 && launch_topk_merge(h.tk_lists, units * kEpiWarps, T, k, topk_idx, topk_val,
                                 env_int("NQ_PDL", 1) != 0, st) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

int nq_gemv_head(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                 int64_t K, int64_t N, int T, int bits, int32_t* argmax, float* maxval, float* lse,
                 void* workspace, size_t workspace_bytes, nq_stream_t stream) {
  return head_launch(packed, scales, x_bf16, y, K, N, T, bits, argmax, maxval, lse, 0, nullptr,
                     nullptr, workspace, workspace_bytes, stream);
}

int nq_head_topk_workspace_bytes(size_t* bytes) {
  if (!bytes) return NQ_EINVAL;
  size_t head_bytes = 0;
  if (int rc = nq_head_workspace_bytes(&head_bytes)) return rc;
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  // then per (CTA, epilogue warp, token) a list of 32 keys, then a
  // candidate buffer of 64 keys; CTAs <= SMs
  *bytes = static_cast<size_t>(align_up(static_cast<int>(head_bytes), 256)) +
           static_cast<size_t>(d->sms) * kEpiWarps * kHeadMaxT * (32 + 64) * sizeof(unsigned long long);
  return NQ_OK;
}

int nq_gemv_head_topk(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                      int64_t K, int64_t N, int T, int bits, int k, int32_t* topk_idx,
                      float* topk_val, int32_t* argmax, float* maxval, float* lse,
                      void* workspace, size_t workspace_bytes, nq_stream_t stream) {
  if (k < 1) return NQ_EINVAL;
  return head_launch(packed, scales, x_bf16, y, K, N, T, bits, argmax, maxval, lse, k, topk_idx,
                     topk_val, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- fused head, no allocation
// The scratch of nq_gemv_head_noalloc: one file-scope device array, present on
// every GPU that loads the library until the process exits.  Host code only
// sees a stand-in for it; the device address comes from cudaGetSymbolAddress,
// taken once per device with that device current.
static_assert(NQ_HEAD_SCRATCH_BYTES ==
                  kHeadCounterBytes + (256 * kEpiWarps + 256 / kHeadGroup) * kHeadMaxT * kHeadStateBytes,
              "the no-allocation scratch covers devices of up to 256 SMs");
static __device__ __align__(256) unsigned char g_head_scratch[NQ_HEAD_SCRATCH_BYTES];
void* g_head_scratch_addr[kMaxDevices] = {};

int nq_gemv_head_noalloc(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                         int64_t K, int64_t N, int T, int bits, int32_t* argmax, float* maxval,
                         float* lse, nq_stream_t stream) {
  size_t need = 0;
  if (int rc = nq_head_workspace_bytes(&need)) return rc;
  if (need > NQ_HEAD_SCRATCH_BYTES) return NQ_EUNSUPPORTED;  // more SMs than the scratch covers
  int dev;
  if (int rc = current_device(&dev)) return rc;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_head_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || !p) {
        (void)cudaGetLastError();
        return NQ_ECUDA;
      }
      g_head_scratch_addr[dev] = p;
    }
    ws = g_head_scratch_addr[dev];
  }
  // nq_gemv_head clears the arrival counter (the part that must start at
  // zero) on the stream before its launch.
  return nq_gemv_head(packed, scales, x_bf16, y, K, N, T, bits, argmax, maxval, lse, ws,
                      NQ_HEAD_SCRATCH_BYTES, stream);
}

int nq_gemv_swiglu(const void* packed_gu, const uint16_t* scales_gu, const void* x_bf16,
                   void* act_bf16, int64_t K, int64_t N, int T, int bits, nq_stream_t stream) {
  if (!packed_gu || !scales_gu || !x_bf16 || !act_bf16) return NQ_EINVAL;
  if (int rc = check_shape(K, N, bits)) return rc;
  if (T < 1 || T > kMaxT || N % 16 != 0) return NQ_EINVAL;
  if (!aligned16(packed_gu) || !aligned16(scales_gu) || !aligned16(x_bf16) || !aligned16(act_bf16))
    return NQ_EALIGN;
  Plan p;
  if (int rc = make_plan(K, N, T, bits, NQ_ROUTE_AUTO, 0, &p)) return rc;
  return launch_plan(p, packed_gu, scales_gu, x_bf16, nullptr, K, N, T,
                     reinterpret_cast<cudaStream_t>(stream), HeadOut(),
                     static_cast<uint16_t*>(act_bf16));
}

int nq_mlp_ex(const void* packed_gu, const uint16_t* scales_gu, int bits_gu,
              const void* packed_down, const uint16_t* scales_down, int bits_down,
              const void* x_bf16, void* act_bf16, float* y, int64_t H, int64_t I, int64_t H_out,
              int T, int launches, nq_stream_t stream) {
  if (!packed_down || !scales_down || !y) return NQ_EINVAL;
  if (I <= 0 || I % 64 != 0) return NQ_EINVAL;
  if (launches < 0 || launches > 2) return NQ_EINVAL;
  if (int rc = check_shape(I, H_out, bits_down)) return rc;
  if (!aligned16(packed_down) || !aligned16(scales_down) || !aligned16(y)) return NQ_EALIGN;
  if (!packed_gu || !scales_gu || !x_bf16 || !act_bf16) return NQ_EINVAL;
  if (int rc = check_shape(H, 2 * I, bits_gu)) return rc;
  if (T < 1 || T > kMaxT) return NQ_EINVAL;
  if (!aligned16(packed_gu) || !aligned16(scales_gu) || !aligned16(x_bf16) || !aligned16(act_bf16))
    return NQ_EALIGN;
  // The library's choice is two launches: measured faster on GB300 (the
  // one-launch kernel runs its gate+up phase on the down phase's clusters of
  // four, which leave 8 of the 152 SMs idle).  NQ_MLP_FUSED=1 changes it.
  if (launches == 0) launches = env_int("NQ_MLP_FUSED", 0) != 0 ? 1 : 2;
  if (launches == 1) {
    MlpPlan mp;
    if (int rc = make_mlp_plan(H, I, H_out, T, bits_gu, bits_down, &mp)) return rc;
    return launch_mlp(mp, packed_gu, scales_gu, packed_down, scales_down, x_bf16, act_bf16, y, H,
                      I, H_out, T, reinterpret_cast<cudaStream_t>(stream));
  }
  if (int rc = nq_gemv_swiglu(packed_gu, scales_gu, x_bf16, act_bf16, H, 2 * I, T, bits_gu, stream))
    return rc;
  return nq_gemv(packed_down, scales_down, act_bf16, y, I, H_out, T, bits_down, stream);
}

int nq_mlp(const void* packed_gu, const uint16_t* scales_gu, int bits_gu, const void* packed_down,
           const uint16_t* scales_down, int bits_down, const void* x_bf16, void* act_bf16,
           float* y, int64_t H, int64_t I, int64_t H_out, int T, nq_stream_t stream) {
  return nq_mlp_ex(packed_gu, scales_gu, bits_gu, packed_down, scales_down, bits_down, x_bf16,
                   act_bf16, y, H, I, H_out, T, 0, stream);
}

int nq_mlp_one_launch_ok(int64_t H, int64_t I, int64_t H_out, int T, int bits_gu, int bits_down,
                         int* ok_out) {
  if (!ok_out) return NQ_EINVAL;
  if (I <= 0 || I % 64 != 0 || T < 1 || T > kMaxT) return NQ_EINVAL;
  if (int rc = check_shape(H, 2 * I, bits_gu)) return rc;
  if (int rc = check_shape(I, H_out, bits_down)) return rc;
  MlpPlan mp;
  *ok_out = make_mlp_plan(H, I, H_out, T, bits_gu, bits_down, &mp) == NQ_OK ? 1 : 0;
  return NQ_OK;
}

int nq_gemv_plan(int64_t K, int64_t N, int T, int bits, int route, int ksplit, int* route_out,
                 int* ksplit_out, int* clusters_out, int* stages_out, int* smem_out) {
  Plan p;
  if (int rc = make_plan(K, N, T, bits, route, ksplit, &p)) return rc;
  if (route_out) *route_out = p.route;
  if (ksplit_out) *ksplit_out = p.ks;
  if (clusters_out) *clusters_out = p.clusters;
  if (stages_out) *stages_out = p.stages;
  if (smem_out) *smem_out = p.smem;
  return NQ_OK;
}

int nq_gemv_plan_x(int64_t K, int64_t N, int T, int bits, int route, int ksplit, int* x_out) {
  if (!x_out) return NQ_EINVAL;
  Plan p;
  if (int rc = make_plan(K, N, T, bits, route, ksplit, &p)) return rc;
  *x_out = p.route != NQ_ROUTE_MMA ? NQ_X_SMEM
           : p.ntok == kNtokXreg   ? NQ_X_REGS
           : p.ntok == kNtokXreg2  ? NQ_X_REGS2
           : p.ntok == kNtokXregH  ? NQ_X_HYBRID
                                   : NQ_X_SMEM;
  return NQ_OK;
}

int nq_dequant(const void* packed, const uint16_t* scales, float* w, int64_t K, int64_t N, int bits,
               nq_stream_t stream) {
  if (int rc = check_shape(K, N, bits)) return rc;
  if (!packed || !scales || !w) return NQ_EINVAL;
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(w)) return NQ_EALIGN;
  if (launch_dequant(packed, scales, w, K, N, bits, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

int nq_last_device_error(nq_stream_t stream) {
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  // A layer that gave up on a bounded wait may have left its activation
  // counters behind: clear every slot (nothing of this device may run).
  if (v != 0 && cudaMemset(d->sync, 0, 2 * sizeof(unsigned) * kSyncSlots) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return v;
}

int nq_selftest_wait_timeout(int limit_us, nq_stream_t stream) {
  if (limit_us <= 0 || limit_us > 10000000) return NQ_EINVAL;
  DevInfo* d;
  if (int rc = dev_info(&d)) return rc;
  if (launch_selftest_timeout(static_cast<unsigned long long>(limit_us) * 1000ULL, d->status,
                              reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return NQ_ECUDA;
  }
  return NQ_OK;
}

}  // extern "C"
