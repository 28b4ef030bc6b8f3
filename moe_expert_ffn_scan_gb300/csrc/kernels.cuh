// Launch interfaces between the C-ABI layer (capi.cu) and the kernels.
#pragma once

#include "common.cuh"

namespace moe {

// Launch with programmatic dependent launch enabled or not (see pdl_wait in
// common.cuh; without it, pdl_wait returns at once because the stream has already
// ordered the launch after its predecessor).
template <typename... KArgs, typename... Args>
cudaError_t launch_k_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args... args) {
  return launch_k_pdl(true, kern, grid, block, smem, st, args...);
}

// GEMM variants, chosen per group by its row count M (the tile plan):
//   small  M <= 16: N = 16 tokens, 2 CTAs per SM, 3 stages of two 128-K sub-tiles;
//   medium M <= 64: N <= 64, 2 CTAs per SM, 2 stages;
//   larger M is cut into ceil(M / 224) near-equal chunks (multiples of 16 rows):
//   mid    chunks of <= 128 rows: N <= 128, 1 CTA per SM, 3 stages;
//   large  chunks of 129..224 rows: N <= 224, 1 CTA per SM, 2 stages (all the shared
//          memory).
// With K/128 odd the stages hold one sub-tile (the *KO1 stage counts).
constexpr int kSmallBN = 16;
constexpr int kSmallStages = 3;
constexpr int kSmallStagesKO1 = 5;
constexpr int kSmallOcc = 2;
constexpr int kMediumBN = 64;
constexpr int kMediumStages = 2;
constexpr int kMediumStagesKO1 = 4;
constexpr int kMediumOcc = 2;
constexpr int kMidBN = 128;
constexpr int kMidStages = 3;
constexpr int kMidStagesKO1 = 5;
constexpr int kLargeBN = 224;
constexpr int kLargeStages = 2;
constexpr int kLargeStagesKO1 = 2;
// Mid and large tiles on SM pairs (when N % 256 == 0 and K % 512 == 0): 224-token tiles
// (112 per SM), three stages of two 128-K sub-tiles.
constexpr int kPairBN = 224;
constexpr int kPairStages = 3;
constexpr int kPairSfSlots = 5;    // scale-factor ring (its own barriers)
constexpr int kPairSfSlotsF1 = 4;  // with the fused SwiGLU epilogue's scratch


// The tile plan's work lists, one per variant (0 small, 1 medium, 2 mid, 3 large),
// each {group, row0, rows, 0} in group order (the decode path's one-CTA plan lists
// the shared expert's items first), and their lengths.
constexpr int kNumVariants = 4;
struct PlanOut {
  int4* items[kNumVariants];
  int32_t* counts;                 // [kNumVariants]
  int32_t capacity[kNumVariants];  // list lengths; items past them are not written
  int32_t chunk_rows;              // groups above kMediumBN rows are cut into chunks of at
                                   // most this many rows (0: kLargeBN; else a multiple of
                                   // 16 in [kMinChunkRows, kLargeBN])
  int32_t* share_cnt;              // [kShareSlots] arrival counters of the tiles whose K
                                   // range the NVFP4 GEMM's last partial wave splits
                                   // among CTAs; zeroed by the plan kernel, left zero by
                                   // each GEMM
};
// Slots for the split tiles of the NVFP4 GEMM's last partial wave (at most one per CTA:
// the split applies when the grid has at most kShareSlots CTAs).
constexpr int kShareSlots = 256;
// Smallest chunk size the plan accepts: every chunk but a group's last then has more
// than kMediumBN rows, which the mid list's capacity assumes.
constexpr int kMinChunkRows = 144;

// Token count up to which route + histogram + permute + plan run as one CTA.
constexpr int kPrepMaxT = 128;

cudaError_t launch_prep_small(const float* logits, int T, int E, int k, int has_shared,
                              int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                              int32_t* perm_src, int32_t* inv, PlanOut plan, uint32_t* status,
                              cudaStream_t st);
// cnt (nullable): [T][H/128] arrival counters of a combine-fused W2 GEMM, zeroed here.
cudaError_t launch_quant_scatter(const uint16_t* x, int T, int H, int k, int has_shared,
                                 const int32_t* inv, uint8_t* xq, uint8_t* xs, uint8_t* xg,
                                 uint8_t* xsg, int32_t* cnt, uint32_t* status, cudaStream_t st);
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         uint32_t* clear_status, cudaStream_t st);
int perm_blocks(int T);
cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int has_shared,
                           int32_t* blockcnt, int32_t* blockbase, int32_t* counts,
                           int32_t* offsets, int32_t* perm_src, int32_t* inv, uint32_t* status,
                           cudaStream_t st);
cudaError_t launch_plan(const int32_t* offsets, int G, PlanOut plan, uint32_t* status,
                        cudaStream_t st);

cudaError_t launch_quant_act(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* s,
                             cudaStream_t st);

// Router gate projection: token count up to which the W_g-streaming kernel runs (it
// re-reads W_g, from L2, once per 16 tokens); above it the register-tiled kernel,
// which has too few tiles to fill the GPU below ~1K tokens.
constexpr int kRouterGemvMaxT = 1024;
cudaError_t launch_router_logits(const uint16_t* x, const float* wg, float* logits, int T, int H,
                                 int E, cudaStream_t st);
// The router projection on the tensor cores: W_g split into three bf16 pieces
// [3][E][H] (hi, mid, lo; hi + mid + lo == W_g), then logits from x and the pieces.
cudaError_t launch_router_split(const float* wg, int E, int H, uint16_t* wg3, cudaStream_t st);
cudaError_t launch_router_logits_split(const uint16_t* x, const uint16_t* wg3, float* logits,
                                       int T, int H, int E, uint32_t* status, cudaStream_t st);
cudaError_t launch_swiglu_quant(const uint16_t* y13, int rows, int I, uint8_t* hq, uint8_t* hs,
                                cudaStream_t st);
cudaError_t launch_gather_rows(const uint8_t* xq, const uint8_t* xs, const int32_t* perm_src,
                               int T, int k, int R, int Rs, int H, uint8_t* xg, uint8_t* xsg,
                               uint32_t* status, cudaStream_t st);
cudaError_t launch_combine(const uint16_t* y2, const int32_t* inv, const float* w, int T, int k,
                           int H, int has_shared, uint16_t* out, uint32_t* status,
                           cudaStream_t st);

struct GemmLaunch {
  const uint8_t* w_codes;     // [G][N][K/2]
  const uint8_t* w_scales;    // [G][N][K/32]
  const uint8_t* act;         // [rows_total][K] packed FP8 rows
  const uint8_t* act_scales;  // [rows_total][K/128]
  uint16_t* y;                // [rows_total][N]
  int G, N, K, rows_total;
  const int4* items[kNumVariants];
  const int32_t* item_counts;  // [kNumVariants]
  int max_items[kNumVariants];
  int max_group_rows;          // upper bound on any group's row count
  uint32_t* status;
  // 1 when the tile plan was complete before the launch preceding this GEMM started
  // (its producer ran two or more launches earlier): the weight loads of each CTA's
  // first stages then go out before the wait for the preceding kernel.
  int early_plan;
  // f2 (the W2 GEMM only): with out non-null the epilogue also performs the weighted
  // top-k combine + shared add into out [T][N]; cnt [T][N/128] must be zero.
  uint16_t* out = nullptr;
  const int32_t* perm_src = nullptr;
  const int32_t* inv = nullptr;
  const float* cw = nullptr;
  int32_t* cnt = nullptr;
  int T = 0, k = 0, has_shared = 0;
  // f1 (the W13 GEMM only): with hq non-null the epilogue performs SwiGLU + FP8
  // quantisation into hq [rows_total][N/2] and hs [rows_total][N/256] (y is not written).
  uint8_t* hq = nullptr;
  uint8_t* hs = nullptr;
  // 1: the mid and large lists on the SM-pair kernel (when N % 256 == 0 and K % 512 ==
  // 0), else on the one-SM mid and large variants
  int pair_tiles = 0;
};
cudaError_t launch_grouped_gemm(const GemmLaunch& a, cudaStream_t st);

// f3: the NVFP4-weight grouped GEMM (gemm_nv.cu).  Activations arrive as bf16 rows
// holding the exact values of their FP8 codes (code x 2^e).
struct NvGemmLaunch {
  const uint8_t* w_codes;     // [G][N][K/2] E2M1 codes
  const uint8_t* w_scales;    // [G][N][K/16] E4M3 block scales
  const float* gs;            // [G][gs_segments] fp32 tensor scales, or null (1.0)
  int gs_segments;            // equal row segments of N, each with its tensor scale
  const uint16_t* act;        // [rows_total][K] bf16
  uint16_t* y;                // [rows_total][N] bf16
  int G, N, K, rows_total;
  const int4* items[kNumVariants];
  const int32_t* item_counts;
  int max_items[kNumVariants];
  int max_group_rows;
  uint32_t* status;
  int32_t* share_cnt;  // the plan's counters (PlanOut::share_cnt)
  float* share_part;   // [kShareSlots][2][kSmallBN][128]: fp32 partials of split tiles
};
cudaError_t launch_grouped_gemm_nv(const NvGemmLaunch& a, cudaStream_t st);
int nv_encode_maps(const NvGemmLaunch& a, int ks, int bn, CUtensorMap* tmC, CUtensorMap* tmS,
                   CUtensorMap* tmX);

// cuTensorMapEncodeTiled through the runtime's driver entry point (null if absent).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled_fn();

// FP8 codes -> bf16 rows of their exact values (code x 2^e), for the NVFP4 GEMMs:
// the quant-scatter writes xe (the packed rows) directly; the stand-alone GEMM calls
// expand their FP8 operand with launch_expand_rows (row r of xe from row tok(r) of
// xq when perm_src is given, else from row r).
cudaError_t launch_quant_scatter_bf16(const uint16_t* x, int T, int H, int k, int has_shared,
                                      const int32_t* inv, uint8_t* xq, uint8_t* xs,
                                      uint16_t* xe, uint32_t* status, cudaStream_t st);
cudaError_t launch_swiglu_quant_bf16(const uint16_t* y13, int rows, int I, uint8_t* hq,
                                     uint8_t* hs, uint16_t* he, cudaStream_t st);
cudaError_t launch_expand_rows(const uint8_t* xq, const uint8_t* xs, const int32_t* perm_src,
                               int T, int k, int R, int rows, int K, uint16_t* xe,
                               uint32_t* status, cudaStream_t st);

// Unique id of the calling thread's current CUDA context (cuCtxGetId), 0 when no
// context is current or the driver entry points are unavailable.  Host-side caches of
// per-context state (a function attribute, a symbol's device address) are keyed on it:
// a context created after cudaDeviceReset has a new id, so the state is set up again.
unsigned long long current_context_id();

// Transaction bytes one 128 x 128 weight-tile TMA load reports to its mbarrier: the
// packed global size (128 rows x 64 bytes), not the 16-byte-aligned shared-memory
// footprint (which is twice that).
constexpr uint32_t kWeightTileTxBytes = 128 * 64;

}  // namespace moe
