/*
 * nq.h -- C ABI of the groupwise-quantized small-T GEMV library (libnq.so).
 *
 * Operation (page "Qwen3.8-27B for NInfer on the RTX 3090", section "What is
 * different from the upstream artifact"): a weight matrix W[N, K] is stored as
 * signed integer codes c in groups of 64 consecutive weights along K, with one
 * FP16 scale s per group, and w = s * c.  Code widths: 4 bits [-8, 7],
 * 5 bits [-16, 15], 6 bits [-32, 31], and 8 bits [-128, 127] (the 8-bit
 * head and projections of the same engine: that page's section
 * "Measurements" and page "jabbatheduck/ninfer-ext-models", table
 * "Representation").  Scales may be negative.  The library
 * computes
 *
 *        y[t, n] = sum_k x[t, k] * s[n, k / 64] * c[n, k]      t < T <= 16
 *
 * with x in bf16 and y in fp32: the decode and speculative-verify matrix
 * products of the engine described on that page and on "giveen/ninfer-ext"
 * (sections "Where ninfer-ext leads" and "Engineering": small-batch K-split
 * routes for the verify rounds of speculative decoding).
 *
 * Conventions shared by every entry point
 *   - Return value: NQ_OK (0) or a negative nq_status.  Validation happens on
 *     the host before any launch; a failed validation launches nothing and
 *     writes nothing.
 *   - The caller owns every buffer; no call allocates memory.
 *   - "device" pointers are CUDA device pointers (current device); "host"
 *     pointers are ordinary CPU memory.  Device pointers must be 16-byte
 *     aligned (NQ_EALIGN otherwise).
 *   - Device entry points are asynchronous on `stream` (0 = legacy default
 *     stream).  A launch failure is reported as NQ_ECUDA (the CUDA error is
 *     consumed).  Errors found by a running kernel (a bounded wait that gave
 *     up, a scale that overflowed) are recorded in a per-device status word
 *     that nq_last_device_error() reads and clears.
 *   - Thread-safe: no state besides the per-device status word and cached
 *     per-device launch settings.
 *   - Ordering of weight writes.  The GEMV entry points launch with
 *     programmatic dependent launch (NQ_PDL=1, the default): the kernel may
 *     start while the preceding kernel on the stream is still finishing, and
 *     it reads x only after that kernel has completed, but it starts
 *     streaming the packed weights and scales at once.  So the packed
 *     weights and scales must not be written by the kernel launched
 *     immediately before the GEMV on the same stream.  The library orders its
 *     own writer: a GEMV that directly follows nq_pack_device on a stream is
 *     launched without programmatic dependent launch.  A caller that writes
 *     weights with a kernel of its own (a copy kernel, its own packer) must
 *     put another launch or a stream-ordered memcpy/event between that kernel
 *     and the GEMV, or set NQ_PDL=0.  (Weights are read-only in the decode
 *     loop, where the early start hides the weight stream's start-up latency:
 *     3 to 6 % per launch, measured.)
 *   - Environment switches, read at each call (for experiments; the defaults
 *     are the measured best): NQ_ROUTE (auto | mma | ffma), NQ_KSPLIT (0 =
 *     the planner's K split, else 1, 2, 4 or 8), NQ_X_F16 (1: fp16 route of
 *     4-bit codes at T <= 2; 0: bf16 route), NQ_XREGH (T > 8: unset = the
 *     planner's choice between both token blocks in registers and the hybrid,
 *     0 = never the hybrid, 1 = only the hybrid), NQ_MLP_FUSED (1: nq_mlp in
 *     one launch where it can), NQ_PDL (1: programmatic dependent launch),
 *     NQ_WAIT_MS (bound of every in-kernel wait, default 2000).
 *
 * PACKED LAYOUT (version 2)
 * -------------------------
 *   Rows are taken in tiles of 16 (Nt = ceil(N/16) tiles; rows >= N of the
 *   last tile are padding with code 0 and scale +0), groups of 64 along K
 *   (G = K/64).  One "block" holds the codes of one row tile and one group,
 *   1024 codes, split among 32 lanes: lane L (q = L/4, r = L%4) owns 32 codes,
 *   16 pairs p = 4*j + i (j = 0..3 sixteen-wide K slices, i = 0..3):
 *       i = 0: row q,     k = 16r + 4j + {0, 1}
 *       i = 1: row q + 8, k = 16r + 4j + {0, 1}
 *       i = 2: row q,     k = 16r + 4j + 2 + {0, 1}
 *       i = 3: row q + 8, k = 16r + 4j + 2 + {0, 1}
 *   (k relative to the group: the group's K order is permuted so that the
 *   x values lane r multiplies, k = 16r .. 16r + 15, are contiguous).  Every code is stored biased, u = c + 2^(b-1),
 *   as an unsigned b-bit field.  The first code of a pair sits in the low
 *   16-bit half of a 32-bit word, the second at the same offset + 16.
 *   A lane's words (W = b 32-bit words) are:
 *     4 bits: word j holds pairs 4j..4j+3; pair i at bit offset 4i.
 *     5 bits: 5 words; each half has three 5-bit fields at offsets 0, 5, 10
 *             holding pairs p = 3w + f (w word, f field) for p < 15; pair 15
 *             is spread over bit 15 of each half: bit m of its code is bit 15
 *             of word m (low code) / bit 31 of word m (high code).
 *     6 bits: 6 words; each half has two 6-bit fields at offsets 0 and 6
 *             holding pairs p = 2w + f for p < 12; pairs 12..15 (d = p - 12)
 *             take bits 0..3 of their code from bits 12..15 of word d and
 *             bits 4..5 from bits 12 + 2(d%2) .. 13 + 2(d%2) of word
 *             4 + d/2 (same offsets + 16 for the high code).
 *     8 bits: word j holds pairs 2j, 2j+1; pair i at bit offset 8i.
 *   Inside a block, words 0..3 of all lanes come first (lane L at byte
 *   16 L), then the remaining words (lane L at 512 + 4(W-4) L).  Block size:
 *   512 / 640 / 768 / 1024 bytes for 4 / 5 / 6 / 8 bits.  Blocks are ordered
 *   [row tile][group]; codes bytes = Nt * G * block size.
 *   Scales: [row tile][group][8][2] FP16, entry (m, h) = row m + 8h of the
 *   tile; 32 bytes per block; scales bytes = Nt * G * 32.
 */
#ifndef NQ_H
#define NQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* nq_stream_t;

typedef enum {
  NQ_OK = 0,
  NQ_EINVAL = -1,        /* bad size, width, T, route, or null pointer */
  NQ_EALIGN = -2,        /* device pointer not 16-byte aligned */
  NQ_ERANGE = -3,        /* code outside its range, non-finite or overflowing scale */
  NQ_ECUDA = -4,         /* CUDA launch or runtime error */
  NQ_ETIMEOUT = -5,      /* a kernel's bounded wait gave up (reported by nq_last_device_error) */
  NQ_EUNSUPPORTED = -6   /* shape needs more shared memory than one cluster provides */
} nq_status;

/* Kernel route of nq_gemv_ex. */
typedef enum {
  NQ_ROUTE_AUTO = 0,     /* library choice (see NQ_ROUTE environment variable) */
  NQ_ROUTE_MMA = 1,      /* warp-level bf16 tensor-core MMA, fp32 accumulate, T <= 16 */
  NQ_ROUTE_FFMA = 2      /* CUDA-core fp32 FMA, T <= 4, 4 to 6 bits */
} nq_route;

/* Byte sizes of the packed codes and packed scales of a W[N, K] tensor.
 * K % 64 == 0, K > 0, N > 0, bits in {4, 5, 6, 8}; outputs are host pointers.
 * Every entry point rejects K / 64 > 2^30 or more than 2^31 - 1 row tiles
 * (N > 16 (2^31 - 1)) with NQ_EINVAL: the kernels index groups and row tiles
 * with 32-bit integers. */
int nq_packed_bytes(int64_t K, int64_t N, int bits, size_t* codes_bytes, size_t* scales_bytes);

/* Host packer.  codes: host int8 [N, K] row-major, values in the signed range
 * of `bits`; scales: host FP16 bit patterns [N, K/64] row-major, finite.
 * Writes packed_out (codes_bytes) and scales_out (scales_bytes / 2 entries),
 * both host, caller-allocated.  NQ_ERANGE on an out-of-range code or a
 * non-finite scale (nothing is written in that case). */
int nq_pack(const int8_t* codes, const uint16_t* scales, int64_t K, int64_t N, int bits,
            void* packed_out, uint16_t* scales_out);

/* Host packer of a gate+up matrix for nq_gemv_swiglu / nq_mlp: gate and up
 * (host int8 codes [I, K] and host FP16 scale bits [I, K/64] each, row-major)
 * packed as one matrix of N = 2 I rows interleaved per 8 -- packed row
 * 16 r + m is gate row 8 r + m and packed row 16 r + 8 + m is up row 8 r + m
 * (m < 8) -- so that a C caller needs no row permutation of its own.  I must
 * be a multiple of 8 (NQ_EINVAL); outputs as nq_pack with N = 2 I.  Same
 * range checks as nq_pack (NQ_ERANGE, nothing written). */
int nq_pack_gate_up(const int8_t* codes_gate, const uint16_t* scales_gate, const int8_t* codes_up,
                    const uint16_t* scales_up, int64_t K, int64_t I, int bits, void* packed_out,
                    uint16_t* scales_out);

/* Host inverse of nq_pack (test and inspection aid).  All pointers host. */
int nq_unpack(const void* packed, const uint16_t* scales_packed, int64_t K, int64_t N, int bits,
              int8_t* codes_out, uint16_t* scales_out);

/* Device packer: same layout as nq_pack, for tensors already in device memory.
 * codes, scales, packed_out, scales_out are device pointers.  Range errors
 * are not checked here (use nq_pack or check beforehand). */
int nq_pack_device(const int8_t* codes, const uint16_t* scales, int64_t K, int64_t N, int bits,
                   void* packed_out, uint16_t* scales_out, nq_stream_t stream);

/* Device round-to-nearest encoder (the "upstream" encoder of the page named
 * above): per 64-group, scale = FP16 round-to-nearest-even of max|w| / qmax
 * (qmax = 7 / 15 / 31) and code = round-half-even(w / scale) clamped to the
 * code range; an all-zero group gives scale +0 and codes 0.
 * w: device fp32 [N, K]; codes_out: device int8 [N, K]; scales_out: device
 * FP16 bits [N, K/64].  A scale that overflows FP16 sets NQ_ERANGE in the
 * device status word. */
int nq_quantize_rtn(const float* w, int64_t K, int64_t N, int bits,
                    int8_t* codes_out, uint16_t* scales_out, nq_stream_t stream);

/* Device searched encoder (the "grouped_search" encoder of the page named
 * above): per 64-group, the FP16 scale is the best of 50 candidates by
 * importance-weighted squared error sum_k q_k (w_k - s c_k)^2, q the
 * per-channel importance (an imatrix, mean squared input activation).  The
 * page does not list the candidates; this library's: with a = max|w| and
 * qmax = 7 / 15 / 31, h_i = FP16 round-to-nearest-even of
 * 12 a / (12 (qmax + 1) - i), i = 0..24 (a / L for L from qmax + 1 down to
 * qmax - 1), each tried as +h_i and -h_i (negative scales let the group's
 * largest weight use code -2^(bits-1)).  Codes are round-half-even(w / s)
 * clamped to the range; the error is accumulated in fp64 over the group in
 * order; ties go to the lower candidate (+h_0, -h_0, +h_1, ...).  i = 12 is
 * the round-to-nearest scale, so the result is never worse than
 * nq_quantize_rtn under the same importance.
 * w: device fp32 [N, K]; imatrix: device fp32 [K] (>= 0), or NULL for all
 * ones; codes_out: device int8 [N, K]; scales_out: device FP16 bits [N, K/64]
 * (same outputs as nq_quantize_rtn).  A group whose every candidate overflows
 * FP16 sets NQ_ERANGE in the device status word. */
int nq_quantize_search(const float* w, const float* imatrix, int64_t K, int64_t N, int bits,
                       int8_t* codes_out, uint16_t* scales_out, nq_stream_t stream);

/* y[T, N] (fp32, device, row-major, overwritten) = x[T, K] (bf16 bit
 * patterns, device, row-major) times dequant(W)^T, W given by its packed codes
 * and packed scales (device, layout above).  1 <= T <= 16.
 * NQ_EUNSUPPORTED if K * T is too large for the shared-memory x tile
 * (K * T <= 327680 is always supported). */
int nq_gemv(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
            int64_t K, int64_t N, int T, int bits, nq_stream_t stream);

/* nq_gemv with an explicit kernel route and K-split (cluster size).
 * route: nq_route; ksplit: 0 = automatic, else 1, 2, 4 or 8 CTAs per cluster
 * splitting K.  NQ_EINVAL if the route does not support T. */
int nq_gemv_ex(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
               int64_t K, int64_t N, int T, int bits, int route, int ksplit, nq_stream_t stream);

/* Gate+up product with the SwiGLU activation in its epilogue: the first half
 * of the decoder layer's MLP (pages "giveen/ninfer-ext", section "Where
 * ninfer-ext leads": the fused gate+up matrix; "Qwen3.8-27B for NInfer on the
 * RTX 3090": Q4 gate/up projections), act[t, i] = bf16(silu(g) * u) with
 * g = (x W_gate^T)[t, i], u = (x W_up^T)[t, i], silu(g) = g / (1 + exp(-g)),
 * computed in fp32 and rounded to nearest-even bf16 (the input of the down
 * projection).  The gate+up matrix must be packed (nq_pack / nq_pack_device)
 * with its N = 2 I rows interleaved per 8: packed row 16 r + m is gate row
 * 8 r + m and packed row 16 r + 8 + m is up row 8 r + m (m < 8), so gate and
 * up of an index finish in the same row tile; N must be a multiple of 16.
 * x_bf16: device [T, K]; act_bf16: device bf16 bit patterns [T, N / 2],
 * written; the fp32 gate and up outputs never leave the chip. */
int nq_gemv_swiglu(const void* packed_gu, const uint16_t* scales_gu, const void* x_bf16,
                   void* act_bf16, int64_t K, int64_t N, int T, int bits, nq_stream_t stream);

/* The decoder layer's MLP on the stream: act = the nq_gemv_swiglu product
 * of x, then y[T, H_out] = act W_down^T.  H = K of gate+up, I = intermediate
 * size (gate+up has 2 I rows, interleaved as above; down has H_out rows and
 * K = I, a multiple of 64); act_bf16: device scratch [T, I] bf16 owned by the
 * caller (the intermediate, 2 I T bytes), written.  The library's choice of
 * launches (see nq_mlp_ex): two, nq_gemv_swiglu then nq_gemv, the second
 * overlapping the first's tail by programmatic dependent launch. */
int nq_mlp(const void* packed_gu, const uint16_t* scales_gu, int bits_gu, const void* packed_down,
           const uint16_t* scales_down, int bits_down, const void* x_bf16, void* act_bf16,
           float* y, int64_t H, int64_t I, int64_t H_out, int T, nq_stream_t stream);

/* nq_mlp with the number of launches chosen by the caller: launches = 0
 * (the library's choice: 2, or 1 with NQ_MLP_FUSED=1), 1 or 2.  One launch
 * runs the whole layer in one kernel: its gate+up phase publishes the
 * activations through a per-device counter, and its down phase starts on
 * weights the kernel streamed while the gate+up phase finished; the results
 * equal the two-launch path's bit for bit.  It supports T <= 8, H <= 5120
 * and the code widths (gate+up, down) = (4, 4), (4, 5), (6, 4), (8, 8)
 * (nq_mlp_one_launch_ok tells; NQ_EUNSUPPORTED otherwise).  It is measured
 * 2 to 6 % slower than two launches on GB300, whose clusters of four CTAs
 * (the down phase's K split) leave 8 of the 152 SMs without work in the
 * gate+up phase.  One-launch layers whose launches overlap on the GPU in
 * number beyond 1024 (4096 while capturing graphs) would share counters:
 * keep fewer layers in flight at once. */
int nq_mlp_ex(const void* packed_gu, const uint16_t* scales_gu, int bits_gu,
              const void* packed_down, const uint16_t* scales_down, int bits_down,
              const void* x_bf16, void* act_bf16, float* y, int64_t H, int64_t I, int64_t H_out,
              int T, int launches, nq_stream_t stream);

/* Whether nq_mlp_ex(launches = 1) supports this layer shape on the current
 * device: *ok_out (host) = 1 or 0.  Same shape checks as nq_mlp. */
int nq_mlp_one_launch_ok(int64_t H, int64_t I, int64_t H_out, int T, int bits_gu, int bits_down,
                         int* ok_out);

/* Fused verify head: the product of nq_gemv (y may be NULL: logits not
 * stored) and, per token t < T, over the N outputs y[t, 0..N):
 *   argmax[t] = the smallest n with y[t, n] maximal (int32; -1 if every
 *               output is -inf), maxval[t] = that maximum,
 *   lse[t]    = log(sum_n exp(y[t, n])), one pass (running maximum).
 * These are the greedy-acceptance and normalisation values of a
 * speculative-verify round over the output head: the pages "giveen/ninfer-ext"
 * (section "Engineering", single-pass logsumexp) and "Qwen3.8-27B for NInfer
 * on the RTX 3090" (section "Run it": candidate top-k over the full head).
 * argmax, maxval, lse: device arrays of T entries, written when the stream
 * reaches the end of the call.  workspace: device scratch of at least
 * nq_head_workspace_bytes() bytes, 16-byte aligned, owned by the caller, any
 * contents on entry; calls sharing a workspace must be ordered (one stream).
 * The result is deterministic: states are merged in a fixed order, and ties
 * of the maximum go to the smallest index.  N <= 2^31 - 1; devices of up to
 * 256 SMs (NQ_EUNSUPPORTED beyond). */
int nq_gemv_head(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                 int64_t K, int64_t N, int T, int bits, int32_t* argmax, float* maxval,
                 float* lse, void* workspace, size_t workspace_bytes, nq_stream_t stream);

/* Bytes of workspace nq_gemv_head needs on the current device (any T, N). */
int nq_head_workspace_bytes(size_t* bytes);

/* nq_gemv_head plus the top k logits of every token: the drafter's candidate
 * top-k over the output head of a speculative-verify round (page
 * "Qwen3.8-27B for NInfer on the RTX 3090", section "Run it": the
 * candidate top-k reads the proposal head or the full head; the pages do not
 * fix k).  For t < T and j < k, topk_idx[t * k + j] / topk_val[t * k + j] is
 * the j-th logit of token t in the order: larger fp32 value first, -0 just
 * below +0, equal values by smaller row index (so the answer is unique; NaN
 * logits rank by their bit pattern).  Entries beyond N (k > N) are index -1,
 * value -inf.  The logits are not stored unless y is given; each epilogue
 * warp keeps its own per-token top 32 while the product runs and a second
 * kernel merges those lists, launched on the same stream.  1 <= k <= 32;
 * topk_idx (int32) and topk_val (fp32): device arrays [T, k], row-major;
 * workspace: device scratch of at least nq_head_topk_workspace_bytes()
 * bytes, 16-byte aligned, owned by the caller, any contents on entry; calls
 * sharing a workspace must be ordered.  argmax, maxval and lse as in
 * nq_gemv_head.  Selection only: the result is deterministic. */
int nq_gemv_head_topk(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                      int64_t K, int64_t N, int T, int bits, int k, int32_t* topk_idx,
                      float* topk_val, int32_t* argmax, float* maxval, float* lse,
                      void* workspace, size_t workspace_bytes, nq_stream_t stream);

/* Bytes of workspace nq_gemv_head_topk needs on the current device (any T, N, k). */
int nq_head_topk_workspace_bytes(size_t* bytes);

/* nq_gemv_head for callers that cannot allocate device memory: a library
 * plugged into a host runtime that owns every device allocation and hands it
 * only the tensors it works on, or a latency-critical loop where a
 * cudaMalloc / cudaFree (which synchronise the device) is not acceptable.
 * No counterpart in the pages: it is an interface convenience, not part of
 * the method.  Same arguments and results as nq_gemv_head, without the
 * workspace: the scratch is one file-scope device array of
 * NQ_HEAD_SCRATCH_BYTES, held by every GPU that loads the library until the
 * process exits, enough for devices of up to 256 SMs (NQ_EUNSUPPORTED on a
 * larger one).  The call allocates nothing.  The first call on a device looks
 * up the array's device address (once per device, with that device current);
 * make that first call before any stream capture.  Every call shares the
 * array and finds the previous call's contents in it; the call clears the
 * part that must start at zero (the arrival counter) on its stream before
 * launching.  Calls that overlap on the GPU (other streams, other host
 * threads without ordering) race on the array and give wrong results: order
 * them on one stream.  The looked-up address stays cached for the life of
 * the process: after cudaDeviceReset (or anything else that destroys the
 * device's primary context) the library must be unloaded and loaded again,
 * or the process restarted, before this entry point is used on that device. */
#define NQ_HEAD_SCRATCH_BYTES 139520
int nq_gemv_head_noalloc(const void* packed, const uint16_t* scales, const void* x_bf16, float* y,
                         int64_t K, int64_t N, int T, int bits, int32_t* argmax, float* maxval,
                         float* lse, nq_stream_t stream);

/* Dequantised weights w[N, K] fp32 (device, row-major) = scale * code, exact.
 * Test aid: lets the decode path be checked bit for bit. */
int nq_dequant(const void* packed, const uint16_t* scales, float* w, int64_t K, int64_t N,
               int bits, nq_stream_t stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: NQ_OK, NQ_ETIMEOUT, NQ_ERANGE, or NQ_ECUDA if the synchronisation
 * itself failed. */
int nq_last_device_error(nq_stream_t stream);

/* Launch plan nq_gemv_ex would use (for tests and benchmarks): writes the
 * route, the K-split, the number of clusters, the pipeline stages and the
 * dynamic shared memory in bytes to the non-null host pointers.  Needs a
 * current CUDA device. */
int nq_gemv_plan(int64_t K, int64_t N, int T, int bits, int route, int ksplit,
                 int* route_out, int* ksplit_out, int* clusters_out, int* stages_out,
                 int* smem_out);

/* Where the kernel of that plan keeps x (test and benchmark aid). */
typedef enum {
  NQ_X_SMEM = 0,     /* a shared-memory x tile, staged once per CTA */
  NQ_X_REGS = 1,     /* one token block (T <= 8): x fragments in registers */
  NQ_X_REGS2 = 2,    /* two token blocks (T <= 16), both in registers */
  NQ_X_HYBRID = 3    /* two token blocks: tokens 0-7 in registers, 8.. in shared memory */
} nq_x_place;

/* Writes the nq_x_place of the plan nq_gemv_plan reports for the same
 * arguments to *x_out (host pointer, not null).  Needs a current CUDA device. */
int nq_gemv_plan_x(int64_t K, int64_t N, int T, int bits, int route, int ksplit, int* x_out);

/* Self-test of the bounded waits: launches one CTA that waits on a barrier
 * nothing will ever complete, with a limit of `limit_us` microseconds; the
 * kernel then gives up, records NQ_ETIMEOUT in the status word and returns.
 * The caller reads the result with nq_last_device_error(stream). */
int nq_selftest_wait_timeout(int limit_us, nq_stream_t stream);

/* Static description of a status code. */
const char* nq_status_string(int status);

/* Packed-layout version implemented by this library (2). */
int nq_layout_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NQ_H */
