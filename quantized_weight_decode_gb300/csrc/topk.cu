// Second step of the fused head's top-k: one CTA per token merges the
// per-warp lists that the head GEMV's epilogue warps left in the workspace.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gemv.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace nq {

constexpr int kMergeWarps = 32;

// lists: [nlists][kHeadMaxT][32] keys, each list sorted descending.  Warp w
// folds lists w, w + 32, ... into one running top 32; the 32 warp results
// are then merged pairwise in a tree.  Selection only, so the result does
// not depend on the merge order.
__global__ void __launch_bounds__(kMergeWarps * 32)
    nq_topk_merge_kernel(const unsigned long long* __restrict__ lists, int nlists, int k,
                      int32_t* __restrict__ idx, float* __restrict__ val) {
  __shared__ unsigned long long part[kMergeWarps][32];
  griddep_wait();  // the lists are complete once the head GEMV has finished
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long acc = 0ull;
#pragma unroll 4
  for (int l = warp; l < nlists; l += kMergeWarps) {
    const unsigned long long b =
        __ldcg(lists + (static_cast<size_t>(l) * kHeadMaxT + t) * 32 + lane);
    acc = warp_top32_of_two(acc, b, lane);
  }
  part[warp][lane] = acc;
  __syncthreads();
#pragma unroll
  for (int n = kMergeWarps / 2; n >= 1; n >>= 1) {
    if (warp < n) part[warp][lane] = warp_top32_of_two(part[warp][lane], part[warp + n][lane], lane);
    __syncthreads();
  }
  if (warp == 0 && lane < k) {
    const unsigned long long key = part[0][lane];
    idx[t * k + lane] = key == 0ull ? -1 : topk_key_index(key);
    val[t * k + lane] = key == 0ull ? -INFINITY : topk_key_value(key);
  }
}

cudaError_t launch_topk_merge(const unsigned long long* lists, int nlists, int T, int k,
                              int32_t* idx, float* val, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, nq_topk_merge_kernel, lists, nlists, k, idx, val);
}

}  // namespace nq
