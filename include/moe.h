/*
 * moe.h -- C interface of the GB300 (sm_103a) routed Mixture-of-Experts expert FFN
 * with MXFP4 expert weights and online FP8 activations.
 *
 * The method is the MoE expert path of "Pushing the Limits of Serving
 * DeepSeek-V4-Pro" (LMSYS, H20): MXFP4 expert weights with FP8 activations
 * quantised online (§2.2), W13 and W2 as two grouped GEMMs shaped by the routing
 * histogram (§3.3), SwiGLU fused with the FP8 quantisation that emits W2's operand
 * and scales (§4.3), and the top-k reduction merged with the shared-expert add
 * (§3.2); plus the GB10 "Optimization progress report", Optimization 14 (tokens
 * packed by expert before the MoE launch) and Optimization 06 (small-M expert GEMM
 * without padding the few tokens to large tiles).
 *
 * Conventions for every entry point
 *   - All tensors are caller-owned, row-major, contiguous DEVICE pointers, unless
 *     stated otherwise.  Pointers must be 16-byte aligned (the weight code tensors
 *     32-byte aligned).  bf16 tensors are passed as uint16_t storage.
 *   - Nothing allocates device memory.  Scratch comes from the caller's workspace,
 *     sized by the matching *_workspace_size() query.  Workspace must be 256-byte
 *     aligned.  (moe_host_pipeline_create creates CUDA streams and events, and a
 *     small host-side handle; see there.)
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and never synchronises the host, except moe_check_status,
 *     moe_route_static_status and moe_host_pipeline_sync / moe_host_pipeline_destroy.
 *   - Return value: MOE_OK or an MOE_ERR_* code.  Shapes and pointers are checked
 *     on the host before any launch; nothing is launched when a check fails.
 *     Launch failures return MOE_ERR_CUDA.  Data-dependent device checks (an index
 *     out of range, an expired wait inside a kernel) never trap: they set bits of
 *     a status word in the workspace, read back by moe_check_status.
 *
 * Formats (the pages do not define them; these are the OCP MX v1.0 / OFP8 formats)
 *   - MXFP4 weights: E2M1 codes, two per byte, the even K index in the low nibble,
 *     shape [G][N][K/2]; one E8M0 scale byte (2^(b-127)) per 32 consecutive K
 *     elements, shape [G][N][K/32].
 *   - FP8 activations: E4M3 ("FN": bias 7, max 448) codes [rows][cols]; one scale
 *     byte per row per 128 columns [rows][cols/128] holding e + 127, where e is the
 *     smallest integer with amax <= 448 * 2^e; codes = round-to-nearest-even of
 *     x * 2^-e.  A block of zeros gets scale byte 127 and zero codes.
 *
 * Shapes supported (else MOE_ERR_UNSUPPORTED_SHAPE): H % 128 == 0, I % 128 == 0,
 * 1 <= k <= min(E, 16), 1 <= E <= 1024, T >= 1, T * k < 2^31.
 */
#ifndef MOE_GB300_MOE_H_
#define MOE_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null / misaligned pointer, bad enum value        */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* dims outside the supported set above             */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,
  MOE_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed             */
  MOE_ERR_DEVICE_CHECK = 5        /* moe_check_status found a device status bit set   */
};

/* T tokens, hidden size H, per-expert intermediate size I, E routed experts, top-k,
 * has_shared = 1 adds one always-on shared expert stored as group E of the weight
 * tensors.  G = E + has_shared groups; R = T*k routed rows; Rs = R + T*has_shared
 * packed rows (routed rows grouped by expert, then one shared row per token). */
typedef struct moe_dims {
  int32_t T, H, I, E, k, has_shared;
} moe_dims;

/* MXFP4 expert weights, G groups each: w13 [G][2I][H/2] + w13_s [G][2I][H/32]
 * (rows 0..I-1 gate projection, rows I..2I-1 up projection), w2 [G][H][I/2] +
 * w2_s [G][H][I/32]. */
typedef struct moe_weights {
  const uint8_t* w13;
  const uint8_t* w13_s;
  const uint8_t* w2;
  const uint8_t* w2_s;
} moe_weights;

/* Optional outputs of moe_forward's intermediates (any member may be NULL). */
typedef struct moe_debug_out {
  int32_t* idx;      /* [T][k]              */
  float* w;          /* [T][k]              */
  int32_t* counts;   /* [E]                 */
  int32_t* offsets;  /* [G+1]               */
  int32_t* perm_src; /* [R]                 */
  int32_t* inv;      /* [R]                 */
  uint8_t* xq;       /* [T][H]              */
  uint8_t* xs;       /* [T][H/128]          */
  uint16_t* y13;     /* [Rs][2I] bf16       */
  uint8_t* hq;       /* [Rs][I]             */
  uint8_t* hs;       /* [Rs][I/128]         */
  uint16_t* y2;      /* [Rs][H] bf16        */
} moe_debug_out;

/* Text of a status code (static storage). */
const char* moe_error_string(int status);

/* Workspace bytes needed by moe_forward / moe_route / the two grouped GEMMs at
 * these dims (0 for unsupported dims). */
size_t moe_workspace_size(const moe_dims* d);
size_t moe_route_workspace_size(const moe_dims* d);
size_t moe_gemm_workspace_size(const moe_dims* d);

/* a1 + a2: top-k routing, token->expert histogram, exclusive scan and permutation.
 * Pages: LMSYS-H20 §3.2 (TopK) and §3.3 (per-expert M from the routing histogram);
 * GB10 report Optimization 14 (route preplan, tokens packed by expert).
 *   logits [T][E] fp32.  Per token: the k largest logits (equal logits -> lower
 *   expert index first), in that order -> idx [T][k]; weights softmax-renormalised
 *   over the selected k -> w [T][k] (sum 1).
 *   counts [E] tokens per expert; offsets [G+1] exclusive scan over groups
 *   (offsets[E+1] = Rs when has_shared); perm_src [R]: packed row -> routed row t*k+j,
 *   rows of a group in ascending token order; inv [R]: routed row -> packed row.
 *   Bit-exact and deterministic (no order-dependent atomics).
 *   ws: moe_route_workspace_size(d) bytes. */
int moe_route(const moe_dims* d, const float* logits, int32_t* idx, float* w, int32_t* counts,
              int32_t* offsets, int32_t* perm_src, int32_t* inv, void* ws, size_t ws_bytes,
              void* stream);

/* moe_route without a workspace argument, for callers that cannot allocate device
 * memory (a host framework whose pool owns every device byte, or a latency-critical
 * loop that cannot afford cudaMalloc/cudaFree and their implicit synchronisation).
 * The pages have no counterpart: this is an interface convenience, not a step of
 * the method.  Same arguments and results as moe_route minus ws / ws_bytes; logits
 * and the six outputs must be 4-byte aligned (else MOE_ERR_INVALID_ARG).
 *   - Scratch lives in a fixed device array of 256 KiB + 256 bytes inside the
 *     library, held on every GPU that loads it until the process exits.  Limit:
 *     ceil(T/256) * E <= 32768 (T <= 8192 at E = 1024, T <= 21760 at E = 384);
 *     larger inputs return MOE_ERR_UNSUPPORTED_SHAPE.
 *   - The first call in each CUDA context (per device, and again after
 *     cudaDeviceReset) looks up the array's device address with that context
 *     current; make that first call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents; calls that
 *     overlap on the GPU (other streams, other host threads) race on it and must be
 *     serialised by the caller.  Nothing is allocated.
 *   - Device-side checks (an expert index out of range) set bits in a status word
 *     at the start of the array, cleared by each call's first kernel; read it with
 *     moe_route_static_status. */
int moe_route_static(const moe_dims* d, const float* logits, int32_t* idx, float* w,
                     int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv,
                     void* stream);

/* Debug helper for moe_route_static (synchronises `stream`): reads the status word of
 * its fixed array as moe_check_status reads a workspace's.  Returns MOE_OK if no bit
 * is set, else MOE_ERR_DEVICE_CHECK and the bits in *bits_out (if not NULL); the
 * bits are those of the last moe_route_static call in the current context. */
int moe_route_static_status(void* stream, uint32_t* bits_out);

/* f4: router gate projection in front of moe_route:
 *     logits[t][e] = sum_h x[t][h] * wg[e][h],  fp32 products and fp32 sums,
 * for x bf16 [T][H] (the token hidden states) and wg fp32 [E][H] (the gate weight),
 * logits fp32 [T][E].  Pages: LMSYS-H20 §3.2 (the TopK step ranks these per-expert
 * scores; the gate itself is not printed, so it is read as this plain projection).
 * Each logit's H products are summed in one fixed order (run-to-run identical);
 * against an exactly rounded sum the error stays within fp32 accumulation bounds.
 * Requires T >= 1, E >= 1, H >= 16, H % 16 == 0 (MOE_ERR_UNSUPPORTED_SHAPE), x and wg
 * 16-byte aligned, logits 4-byte aligned (MOE_ERR_INVALID_ARG).  Caller-owned
 * device buffers; no workspace; asynchronous on `stream`. */
int moe_router_logits(int32_t T, int32_t H, int32_t E, const uint16_t* x, const float* wg,
                      float* logits, void* stream);

/* f4 on the tensor cores.  The gate weight is split once (weight preprocessing, like
 * loading a checkpoint) into three bf16 matrices with wg == hi + mid + lo exactly
 * (8 + 8 + 8 significant bits; exact unless a piece falls below bf16's normal range,
 * i.e. for weights under about 2^-110 in magnitude): moe_router_split writes them to
 * wg3 [3][E][H] (moe_router_split_bytes(E, H) bytes, 16-byte aligned, caller-owned).
 * moe_router_logits_split then computes the same logits as moe_router_logits with
 * tcgen05 MMAs: each product x * piece is exact in fp32 and the three pieces' products
 * of every 16-column step are accumulated in fp32 (a fixed order: run-to-run
 * identical; within the same fp32 accumulation bound).  The pages' TopK step
 * (LMSYS-H20 §3.2) ranks these scores.  Shapes and alignment as moe_router_logits; no
 * workspace; device-side wait failures of this call are not reported (it has no status
 * word).  Its tiles are 128 tokens x 128 experts, so it pays off from a few hundred
 * tokens (on GB300 at H = 7168, E = 384: 0.40 ms vs 4.2 ms at 32K tokens, 0.08 vs 0.10
 * ms at 256); decode-sized batches are faster through moe_router_logits. */
size_t moe_router_split_bytes(int32_t E, int32_t H);
int moe_router_split(int32_t E, int32_t H, const float* wg, uint16_t* wg3, void* stream);
int moe_router_logits_split(int32_t T, int32_t H, int32_t E, const uint16_t* x,
                            const uint16_t* wg3, float* logits, void* stream);

/* a3: online FP8 E4M3 quantisation of bf16 x [rows][cols] with one power-of-two
 * scale per row per 128 columns (rule above) -> q [rows][cols], s [rows][cols/128].
 * Pages: LMSYS-H20 §2.2 (online FP8 activations), §3.2 (fused FP8 quantisation).
 * cols % 128 == 0, rows >= 0 (rows == 0 is a no-op). */
int moe_quant_act(int32_t rows, int32_t cols, const uint16_t* x, uint8_t* q, uint8_t* s,
                  void* stream);

/* a4: W13 grouped GEMM (LMSYS-H20 §3.3).  For every group g and packed row r in
 * [group_offsets[g], group_offsets[g+1]):
 *     y13[r][n] = bf16( sum_k deq(xq)[tok(r)][k] * deq(w13[g])[n][k] ),  n < 2I,
 * FP8 x MXFP4 products accumulated in fp32 on the tensor cores (tcgen05 block-
 * scaled MMA).  tok(r) = perm_src[r] / k for r < R and r - R for shared rows; with
 * perm_src == NULL the activations are already packed (xq has Rs rows, tok(r) = r).
 * xq [T][H] (or [Rs][H]), xs [T][H/128]; group_offsets [G+1] device int32,
 * non-decreasing, group_offsets[G] <= Rs; y13 [Rs][2I] bf16 (rows outside every
 * group are not written).  ws: moe_gemm_workspace_size(d) bytes. */
int moe_grouped_gemm_w13(const moe_dims* d, const uint8_t* xq, const uint8_t* xs,
                         const int32_t* perm_src, const int32_t* group_offsets,
                         const uint8_t* w13, const uint8_t* w13_s, uint16_t* y13, void* ws,
                         size_t ws_bytes, void* stream);

/* a5: SwiGLU fused with FP8 requantisation (LMSYS-H20 §4.3): for each row,
 * h = silu(g) * u with g = y13[r][0:I], u = y13[r][I:2I], silu(g) = g / (1 + e^-g),
 * in fp32, then quantised per 128 columns with the activation rule -> hq [rows][I],
 * hs [rows][I/128] (W2's operand and scales).  I % 128 == 0. */
int moe_swiglu_quant(int32_t rows, int32_t I, const uint16_t* y13, uint8_t* hq, uint8_t* hs,
                     void* stream);

/* a6: W2 grouped GEMM (LMSYS-H20 §3.3): y2[r][n] = bf16( sum_i deq(hq)[r][i] *
 * deq(w2[g])[n][i] ), n < H, for r in group g.  hq [Rs][I], hs [Rs][I/128],
 * y2 [Rs][H].  ws: moe_gemm_workspace_size(d) bytes. */
int moe_grouped_gemm_w2(const moe_dims* d, const uint8_t* hq, const uint8_t* hs,
                        const int32_t* group_offsets, const uint8_t* w2, const uint8_t* w2_s,
                        uint16_t* y2, void* ws, size_t ws_bytes, void* stream);

/* a7: weighted top-k unpermute-combine plus shared-expert add (LMSYS-H20 §3.2):
 *     out[t] = bf16( sum_{j<k} w[t][j] * y2[inv[t*k+j]]  (+ y2[R+t] if has_shared) ),
 * summed in fp32 in j order, the shared row last.  y2 [Rs][H], inv [R], w [T][k],
 * out [T][H] bf16. */
int moe_combine(const moe_dims* d, const uint16_t* y2, const int32_t* inv, const float* w,
                uint16_t* out, void* stream);

/* The whole layer a1..a7 on one stream, no host synchronisation: x [T][H] bf16,
 * logits [T][E] fp32, weights W (G groups), out [T][H] bf16.  dbg may be NULL.
 * ws: moe_workspace_size(d) bytes. */
int moe_forward(const moe_dims* d, const uint16_t* x, const float* logits,
                const moe_weights* W, uint16_t* out, const moe_debug_out* dbg, void* ws,
                size_t ws_bytes, void* stream);

/* The whole layer from and to host memory, for callers whose activations live on the
 * host: copies x_host [T][H] bf16 and logits_host [T][E] fp32 to device staging in
 * the workspace, runs moe_forward, and copies the output back to out_host [T][H] bf16
 * -- two host->device copies, the layer's kernels and one device->host copy, all
 * asynchronous on `stream` (host buffers should be pinned for the copies to be
 * asynchronous; the caller synchronises before reading out_host).  The pages have no
 * counterpart (their layers run inside a serving engine with device-resident
 * activations); this is the end-to-end form of moe_forward.  Weights as for
 * moe_forward (device).  ws: moe_host_workspace_size(d) bytes, 256-byte aligned. */
size_t moe_host_workspace_size(const moe_dims* d);
int moe_forward_host(const moe_dims* d, const uint16_t* x_host, const float* logits_host,
                     const moe_weights* W, uint16_t* out_host, void* ws, size_t ws_bytes,
                     void* stream);

/* ---------------------------------------------------------------------------------
 * f3: NVFP4 expert weights (GB10 "Optimization progress report", Optimization 05,
 * native NVFP4 MoE: the expert weights stay NVFP4 in memory and the expert GEMMs read
 * them as such).  The page names the format without defining it; read as NVIDIA's
 * NVFP4: E2M1 codes packed as for MXFP4 ([G][N][K/2], even K index in the low
 * nibble), one FP8 E4M3 scale byte per 16 consecutive K elements ([G][N][K/16]), and
 * one fp32 scale per weight tensor.  Activations stay online FP8 (same codes and
 * scales as the MXFP4 path); the GEMMs multiply in bf16, where a weight (E2M1 x E4M3,
 * at most 6 significant bits) and an activation (E4M3 code x 2^e) are both exact
 * (activations below bf16's subnormal floor excepted: a 128-block with amax under
 * about 2^-116), and accumulate in fp32; the tensor scale multiplies the fp32 sum
 * before the bf16 rounding.  Requires H % 256 == 0 and I % 256 == 0 in addition to
 * the shapes above (else MOE_ERR_UNSUPPORTED_SHAPE). */
typedef struct moe_weights_nvfp4 {
  const uint8_t* w13;    /* [G][2I][H/2]  E2M1 codes (rows 0..I-1 gate, I..2I-1 up)   */
  const uint8_t* w13_s;  /* [G][2I][H/16] E4M3 block scales                          */
  const float* w13_gs;   /* [G][2] fp32 tensor scales (gate rows, up rows); NULL = 1 */
  const uint8_t* w2;     /* [G][H][I/2]                                              */
  const uint8_t* w2_s;   /* [G][H][I/16]                                             */
  const float* w2_gs;    /* [G] fp32 tensor scales; NULL = 1                         */
} moe_weights_nvfp4;

/* Workspace bytes of moe_forward_nvfp4 and of the two NVFP4 grouped GEMMs. */
size_t moe_workspace_size_nvfp4(const moe_dims* d);
size_t moe_gemm_workspace_size_nvfp4(const moe_dims* d);

/* moe_forward with NVFP4 expert weights: the same stages and results' definition, the
 * W13 / W2 GEMMs reading NVFP4 weights (y = bf16(gs * sum_k deq(a) * e2m1 * e4m3)).
 * The quantisation stages also write the bf16 values of their FP8 codes, the NVFP4
 * GEMMs' operand form.  dbg as for moe_forward.  ws: moe_workspace_size_nvfp4(d). */
int moe_forward_nvfp4(const moe_dims* d, const uint16_t* x, const float* logits,
                      const moe_weights_nvfp4* W, uint16_t* out, const moe_debug_out* dbg,
                      void* ws, size_t ws_bytes, void* stream);

/* moe_forward_nvfp4 with the stage events of moe_forward_timed. */
int moe_forward_nvfp4_timed(const moe_dims* d, const uint16_t* x, const float* logits,
                            const moe_weights_nvfp4* W, uint16_t* out, const moe_debug_out* dbg,
                            void* const* events, void* ws, size_t ws_bytes, void* stream);

/* a4 / a6 with NVFP4 weights: as moe_grouped_gemm_w13 / moe_grouped_gemm_w2 (same
 * operands, FP8 codes + per-128 scales, same row mapping), weights w [G][N][K/2] codes,
 * w_s [G][N][K/16] E4M3 scales, w_gs the fp32 tensor scales ([G][2] for W13, [G] for
 * W2; NULL = 1, 4-byte aligned).  The FP8 operand is first expanded to bf16 rows in
 * the workspace.  ws: moe_gemm_workspace_size_nvfp4(d). */
int moe_grouped_gemm_w13_nvfp4(const moe_dims* d, const uint8_t* xq, const uint8_t* xs,
                               const int32_t* perm_src, const int32_t* group_offsets,
                               const uint8_t* w13, const uint8_t* w13_s, const float* w13_gs,
                               uint16_t* y13, void* ws, size_t ws_bytes, void* stream);
int moe_grouped_gemm_w2_nvfp4(const moe_dims* d, const uint8_t* hq, const uint8_t* hs,
                              const int32_t* group_offsets, const uint8_t* w2,
                              const uint8_t* w2_s, const float* w2_gs, uint16_t* y2, void* ws,
                              size_t ws_bytes, void* stream);

/* Host-buffer pipeline: a sequence of layer steps whose inputs and outputs live in
 * host memory, with the copies of one step overlapping the kernels of its neighbours.
 * The library owns three CUDA streams (host->device copies, the layer, device->host
 * copy) and 3 x depth events, created by moe_host_pipeline_create and released by
 * moe_host_pipeline_destroy (the only calls here that create anything, and neither
 * allocates device memory).  Step i uses staging slot i % depth of the caller's
 * workspace: its two host->device copies wait until step i - depth has finished
 * reading that slot, its kernels run in submission order on the pipeline's compute
 * stream (so one forward workspace serves every step) once its copies landed and
 * step i - depth's output left the slot, and its device->host copy follows its
 * kernels.  Same results as moe_forward_host, step by step.  The pages have no
 * counterpart (their layers run inside a serving engine with device-resident
 * activations).
 *   depth: 1..8 staging slots (2 overlaps each step's copies with its neighbours).
 *   ws: moe_host_pipeline_workspace_size(d, depth) bytes, 256-byte aligned, owned
 *       by the caller and not touched by anything else until destroy; the status
 *       word moe_check_status reads is at its start.
 *   W: copied (the pointers), the weights must stay valid until destroy.
 *   submit: x_host [T][H] bf16, logits_host [T][E] fp32, out_host [T][H] bf16, host
 *       pointers (pinned, or the copies are not asynchronous).  Returns after
 *       enqueueing; the caller must not modify x_host / logits_host or read out_host
 *       until moe_host_pipeline_sync returns (or until depth later submits were
 *       made and synchronised).
 *   sync: blocks until every submitted step's output is in host memory; MOE_ERR_CUDA
 *       if a stream reported an error.
 *   destroy: synchronises, then releases the streams, events and the handle.
 * A pipeline is driven by one host thread at a time.  After a call returns an error
 * other than MOE_ERR_INVALID_ARG, sync and destroy it rather than submit again. */
typedef struct moe_host_pipeline moe_host_pipeline;
size_t moe_host_pipeline_workspace_size(const moe_dims* d, int depth);
int moe_host_pipeline_create(const moe_dims* d, const moe_weights* W, int depth, void* ws,
                             size_t ws_bytes, moe_host_pipeline** out);
int moe_host_pipeline_submit(moe_host_pipeline* p, const uint16_t* x_host,
                             const float* logits_host, uint16_t* out_host);
int moe_host_pipeline_sync(moe_host_pipeline* p);
int moe_host_pipeline_destroy(moe_host_pipeline* p);

/* moe_forward with per-stage timing.  events points to 8 cudaEvent_t handles created
 * by the caller (cudaEventCreate); the call records events[0] before the first stage
 * and events[i] after stage i: 1 route + histogram/scan/permute + tile plan, 2
 * activation quantisation with the packed-row scatter, 3 (empty: the plan runs in
 * stage 1 and the gather in stage 2; kept so that the indices stay fixed), 4 W13
 * grouped GEMM, 5 SwiGLU + quantisation, 6 W2 grouped GEMM, 7 combine.  Same results
 * as moe_forward. */
int moe_forward_timed(const moe_dims* d, const uint16_t* x, const float* logits,
                      const moe_weights* W, uint16_t* out, const moe_debug_out* dbg,
                      void* const* events, void* ws, size_t ws_bytes, void* stream);

/* Options of moe_forward_ex (zero-initialise; every field 0 = moe_forward).
 *   fuse_swiglu (f1): 1 = the W13 grouped GEMM's epilogue performs a5 (LMSYS-H20 §4.3,
 *     SwiGLU fused with the quantisation that emits W2's data and scales): each tile
 *     of an SM pair (a cluster of two CTAs sharing each cta_group::2 MMA) holds 64
 *     gate + the same 64 up rows per CTA, i.e. one 128-feature quantisation block per
 *     pair; h = silu(gate) * up is formed from the bf16-rounded accumulators, the two
 *     CTAs swap per-token amaxes, and the FP8 codes and scales are written directly
 *     with the stand-alone SwiGLU kernel's arithmetic, without y13 (the dbg->y13
 *     buffer is not written) and without that kernel.  The pair tile sums K in one
 *     accumulator where the stand-alone small tiles use two (even / odd stages), so a
 *     rare y13 element -- and so an FP8 code -- can differ from the stand-alone path
 *     at large K; within the float contract.  Needs H % 512 == 0.
 *   pair_tiles: 1 = the mid and large tile lists (groups of more than 64 rows) run on
 *     SM pairs (one cta_group::2 MMA per 256 weight rows, half the token tile per SM)
 *     instead of one SM per tile (when N % 256 == 0 and K % 512 == 0); the same
 *     accumulation order as the one-SM tiles of those lists.
 *   fuse_combine (f2): 1 = the W2 grouped GEMM's epilogue performs a7 (LMSYS-H20 §3.2,
 *     the TopK reduction merged with the shared-expert add): once a tile has stored its
 *     y2 rows, each row bumps its (token, 128-column block) arrival counter, and the
 *     tile that brings a block to k + has_shared arrivals sums that token's rows for
 *     those 128 columns in the stand-alone combine's order (fp32, j order, shared row
 *     last) -- the same out bit for bit, deterministic, no float atomics -- and the
 *     separate combine kernel is not launched.
 *   large_chunk_rows: the tile plan (a8) cuts every group of more than 64 rows into
 *     ceil(M / C) near-equal chunks of at most C rows, C = large_chunk_rows (0: 224;
 *     else a multiple of 16 in [144, 224], MOE_ERR_INVALID_ARG otherwise); chunks of
 *     <= 128 rows run on the mid tiles, larger ones on the large tiles.  The knob of
 *     LMSYS-H20 §3.3's exact-shape tuning: the best C depends on the routing histogram
 *     (the binding's tune_chunk_rows times candidates on a recorded batch).  Results
 *     are the same bit for bit for every C (each output element's K sum runs in the
 *     same order on the mid and large tiles).
 * The fusion and pair options take MXFP4 weights (MOE_ERR_INVALID_ARG otherwise). */
typedef struct moe_options {
  int32_t fuse_combine;
  int32_t fuse_swiglu;
  int32_t pair_tiles;
  int32_t large_chunk_rows;
} moe_options;

/* moe_forward_timed with options (opt may be NULL: all zero; events may be NULL).
 * Returns MOE_ERR_INVALID_ARG for an option value other than 0 / 1. */
int moe_forward_ex(const moe_dims* d, const uint16_t* x, const float* logits,
                   const moe_weights* W, const moe_options* opt, uint16_t* out,
                   const moe_debug_out* dbg, void* const* events, void* ws, size_t ws_bytes,
                   void* stream);

/* Debug helper (synchronises `stream`): reads the device status word at the start of
 * a workspace used by the calls above.  Returns MOE_OK if no bit is set, else
 * MOE_ERR_DEVICE_CHECK and the bits in *bits_out (if not NULL).  The word is
 * cleared by moe_forward / moe_route / the GEMMs at their start. */
int moe_check_status(const void* ws, void* stream, uint32_t* bits_out);

/* Failure-path self-test; the pages have no counterpart.  Launches one CTA whose
 * mbarrier wait can never complete (nothing arrives), so the library's bounded wait
 * (kWaitLimitNs = 2 s of the GPU's global timer) gives up, sets STATUS_WAIT_TIMEOUT
 * (bit 0) in the status word at the start of ws and returns: the path every GEMM wait
 * takes if a TMA copy or MMA never completes.  moe_check_status(ws) then returns
 * MOE_ERR_DEVICE_CHECK with bit 0 set, and the context stays usable.  About 2 s of GPU
 * time.  ws: >= 256 bytes, 256-byte aligned (its status word is overwritten). */
int moe_selftest_wait_timeout(void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H_ */
