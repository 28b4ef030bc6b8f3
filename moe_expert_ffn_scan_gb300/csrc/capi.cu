// C interface (include/moe.h): argument checks, workspace carving and launches.
// No allocation, no host synchronisation (except moe_check_status).
#include <stdio.h>

#include <mutex>
#include <new>

#include "kernels.cuh"

using namespace moe;

namespace moe {

unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuCtxGetCurrent", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPoint("cuCtxGetId", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  // a destroyed context that still reads as current makes cuCtxGetId fail: report 0
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace moe

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Bump allocator over a caller-provided workspace (or a size counter when base is null).
struct Carver {
  uint8_t* base;
  size_t used = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    size_t off = used;
    used = align_up(used + count * sizeof(T));
    return base ? reinterpret_cast<T*>(base + off) : nullptr;
  }
};

bool dims_ok(const moe_dims* d) {
  if (!d) return false;
  if (d->T < 1 || d->H < 128 || d->I < 128 || d->E < 1 || d->E > 1024 || d->k < 1) return false;
  if (d->k > 16 || d->k > d->E) return false;
  if (d->H % 128 || d->I % 128) return false;
  if (d->has_shared != 0 && d->has_shared != 1) return false;
  long long R = static_cast<long long>(d->T) * d->k;
  if (R + d->T >= (1LL << 31)) return false;
  if (static_cast<long long>(2) * d->I * d->H >= (1LL << 40)) return false;
  return true;
}

long long rows_R(const moe_dims* d) { return static_cast<long long>(d->T) * d->k; }
long long rows_Rs(const moe_dims* d) { return rows_R(d) + (d->has_shared ? d->T : 0); }
int groups_G(const moe_dims* d) { return d->E + d->has_shared; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct RouteWs {
  uint32_t* status;
  int32_t* blockcnt;
  int32_t* blockbase;
};

RouteWs carve_route(Carver& c, const moe_dims* d) {
  RouteWs w;
  w.status = c.take<uint32_t>(64);
  const size_t nb = static_cast<size_t>(perm_blocks(d->T)) * d->E;
  w.blockcnt = c.take<int32_t>(nb);
  w.blockbase = c.take<int32_t>(nb);
  return w;
}

struct PlanWs {
  PlanOut out;                    // per-variant item lists and their lengths
  int max_items[kNumVariants];
};

PlanWs carve_plan(Carver& c, const moe_dims* d) {
  PlanWs p;
  const int G = groups_G(d);
  const long long Rs = rows_Rs(d);
  p.max_items[0] = G;                                         // one item per group
  p.max_items[1] = G;
  p.max_items[2] = static_cast<int>(Rs / (kMediumBN + 1) + G + 1);  // chunks of > 64 rows
  p.max_items[3] = static_cast<int>(Rs / (kMidBN + 1) + G + 1);     // chunks of > 128 rows
  for (int v = 0; v < kNumVariants; ++v) {
    p.out.items[v] = c.take<int4>(p.max_items[v]);
    p.out.capacity[v] = p.max_items[v];
  }
  p.out.counts = c.take<int32_t>(kNumVariants);
  p.out.chunk_rows = 0;  // kLargeBN
  p.out.share_cnt = c.take<int32_t>(kShareSlots);
  return p;
}

// Expert weight formats (moe.h): the MXFP4 path moves FP8 codes into the GEMMs, the
// NVFP4 path bf16 rows holding the codes' exact values.
enum WeightFormat { kMxfp4 = 0, kNvfp4 = 1 };

struct LayerWeights {
  WeightFormat fmt;
  const uint8_t *w13, *w13_s, *w2, *w2_s;
  const float *w13_gs, *w2_gs;  // NVFP4 tensor scales (null: 1.0)
};

struct GemmWs {
  uint32_t* status;
  PlanWs plan;
  uint8_t* xg;   // MXFP4: packed FP8 rows for W13 [Rs][H]
  uint8_t* xsg;  // their scales [Rs][H/128]
  uint16_t* xe;  // NVFP4: packed bf16 rows for W13 (or W2's operand) [Rs][max(H, I)]
  float* share_part;  // NVFP4: partials of the tiles two CTAs share
};

GemmWs carve_gemm(Carver& c, const moe_dims* d, WeightFormat fmt) {
  GemmWs g{};
  g.status = c.take<uint32_t>(64);
  g.plan = carve_plan(c, d);
  const size_t Rs = static_cast<size_t>(rows_Rs(d));
  if (fmt == kMxfp4) {
    g.xg = c.take<uint8_t>(Rs * d->H);
    g.xsg = c.take<uint8_t>(Rs * (d->H / 128));
  } else {
    g.xe = c.take<uint16_t>(Rs * static_cast<size_t>(d->H > d->I ? d->H : d->I));
    g.share_part = c.take<float>(static_cast<size_t>(kShareSlots) * 2 * kSmallBN * 128);
  }
  return g;
}

struct ForwardWs {
  RouteWs route;
  GemmWs gemm;
  int32_t *idx, *counts, *offsets, *perm_src, *inv;
  float* w;
  uint8_t *xq, *xs, *hq, *hs;
  uint16_t *y13, *y2;
  uint16_t* he;  // NVFP4: W2's operand as bf16 rows [Rs][I]
  int32_t* cnt;  // f2: (token, 128-column block) arrival counters [T][H/128]
};

ForwardWs carve_forward(Carver& c, const moe_dims* d, WeightFormat fmt = kMxfp4) {
  ForwardWs f{};
  f.route = carve_route(c, d);  // status word first
  f.gemm = carve_gemm(c, d, fmt);
  f.gemm.status = f.route.status;
  const size_t T = d->T, R = rows_R(d), Rs = rows_Rs(d), H = d->H, I = d->I;
  f.idx = c.take<int32_t>(R);
  f.w = c.take<float>(R);
  f.counts = c.take<int32_t>(d->E);
  f.offsets = c.take<int32_t>(groups_G(d) + 1);
  f.perm_src = c.take<int32_t>(R);
  f.inv = c.take<int32_t>(R);
  f.xq = c.take<uint8_t>(T * H);
  f.xs = c.take<uint8_t>(T * (H / 128));
  f.y13 = c.take<uint16_t>(Rs * 2 * I);
  if (fmt == kMxfp4) {
    f.hq = c.take<uint8_t>(Rs * I);
    f.hs = c.take<uint8_t>(Rs * (I / 128));
  } else {
    f.he = c.take<uint16_t>(Rs * I);
  }
  f.y2 = c.take<uint16_t>(Rs * H);
  f.cnt = c.take<int32_t>(T * (H / 128));
  return f;
}

// The NVFP4 GEMMs need K % 256 == 0 (their scale rows are TMA rows of K/16 bytes,
// which must be whole 16-byte units).
bool nv_dims_ok(const moe_dims* d) { return dims_ok(d) && d->H % 256 == 0 && d->I % 256 == 0; }

// Device staging of the host-buffer forward, after the forward workspace.
struct HostStagingWs {
  uint16_t* x;
  float* logits;
  uint16_t* out;
};

HostStagingWs carve_host_staging(Carver& c, const moe_dims* d) {
  HostStagingWs h;
  const size_t T = d->T, H = d->H, E = d->E;
  h.x = c.take<uint16_t>(T * H);
  h.logits = c.take<float>(T * E);
  h.out = c.take<uint16_t>(T * H);
  return h;
}

// early_plan: the plan's producer ran at least two launches before this GEMM (see
// GemmLaunch).
// Fusions and tile choices of one GEMM launch (see GemmLaunch): f2, the combine in the
// W2 epilogue; f1, SwiGLU + quantisation in the W13 epilogue; SM-pair tiles.
struct FusedCombine {
  uint16_t* out = nullptr;
  const int32_t* perm_src = nullptr;
  const int32_t* inv = nullptr;
  const float* w = nullptr;
  int32_t* cnt = nullptr;
  uint8_t* hq = nullptr;
  uint8_t* hs = nullptr;
  int pair_tiles = 0;
};

int run_gemm(const moe_dims* d, const uint8_t* act, const uint8_t* act_s, const int32_t* offsets,
             const uint8_t* w, const uint8_t* w_s, int N, int K, uint16_t* y, const PlanWs& plan,
             int max_group_rows, uint32_t* status, cudaStream_t st, int early_plan,
             const FusedCombine& fc = FusedCombine{}) {
  GemmLaunch a{};
  a.out = fc.out;
  a.perm_src = fc.perm_src;
  a.inv = fc.inv;
  a.cw = fc.w;
  a.cnt = fc.cnt;
  a.hq = fc.hq;
  a.hs = fc.hs;
  a.pair_tiles = fc.pair_tiles;
  a.T = d->T;
  a.k = d->k;
  a.has_shared = d->has_shared;
  a.w_codes = w;
  a.w_scales = w_s;
  a.act = act;
  a.act_scales = act_s;
  a.y = y;
  a.G = groups_G(d);
  a.N = N;
  a.K = K;
  a.rows_total = static_cast<int>(rows_Rs(d));
  for (int v = 0; v < kNumVariants; ++v) {
    a.items[v] = plan.out.items[v];
    a.max_items[v] = plan.max_items[v];
  }
  a.item_counts = plan.out.counts;
  a.max_group_rows = max_group_rows;
  a.status = status;
  a.early_plan = early_plan;
  return cuda_rc(launch_grouped_gemm(a, st));
}

int run_gemm_nv(const moe_dims* d, const uint16_t* act, const uint8_t* w, const uint8_t* w_s,
                const float* gs, int gs_segments, int N, int K, uint16_t* y, const PlanWs& plan,
                int max_group_rows, uint32_t* status, float* share_part, cudaStream_t st) {
  NvGemmLaunch a{};
  a.w_codes = w;
  a.w_scales = w_s;
  a.gs = gs;
  a.gs_segments = gs_segments;
  a.act = act;
  a.y = y;
  a.G = groups_G(d);
  a.N = N;
  a.K = K;
  a.rows_total = static_cast<int>(rows_Rs(d));
  for (int v = 0; v < kNumVariants; ++v) {
    a.items[v] = plan.out.items[v];
    a.max_items[v] = plan.max_items[v];
  }
  a.item_counts = plan.out.counts;
  a.max_group_rows = max_group_rows;
  a.status = status;
  a.share_cnt = plan.out.share_cnt;
  a.share_part = share_part;
  return cuda_rc(launch_grouped_gemm_nv(a, st));
}

// One CTA, one waiting thread: an mbarrier that nothing arrives at.  The bounded wait
// must give up (STATUS_WAIT_TIMEOUT) and raise the CTA's abort flag; anything else is
// reported as STATUS_BAD_PLAN.
__global__ void k_selftest_wait(uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* ab = &abort_flag;
    const bool completed = mbar_wait(&bar, 0, status, ab);
    if (completed || *ab == 0) set_status(status, STATUS_BAD_PLAN);
  }
}

bool weights_ok(const uint8_t* c, const uint8_t* s) {
  return c && s && aligned(c, 32) && aligned(s, 16);
}

}  // namespace

extern "C" {

const char* moe_error_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_CHECK: return "device-side check failed (see status bits)";
    default: return "unknown status";
  }
}

size_t moe_route_workspace_size(const moe_dims* d) {
  if (!dims_ok(d)) return 0;
  Carver c(nullptr);
  carve_route(c, d);
  return c.used;
}

size_t moe_gemm_workspace_size(const moe_dims* d) {
  if (!dims_ok(d)) return 0;
  Carver c(nullptr);
  carve_gemm(c, d, kMxfp4);
  return c.used;
}

size_t moe_workspace_size(const moe_dims* d) {
  if (!dims_ok(d)) return 0;
  Carver c(nullptr);
  carve_forward(c, d);
  return c.used;
}

int moe_route(const moe_dims* d, const float* logits, int32_t* idx, float* w, int32_t* counts,
              int32_t* offsets, int32_t* perm_src, int32_t* inv, void* ws, size_t ws_bytes,
              void* stream) {
  if (!dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!logits || !idx || !w || !counts || !offsets || !perm_src || !inv || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign) || !aligned(logits, 4) || !aligned(idx, 4) || !aligned(w, 4) ||
      !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm_src, 4) || !aligned(inv, 4))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_route_workspace_size(d)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carver c(ws);
  RouteWs rw = carve_route(c, d);
  cudaError_t e = launch_route(logits, d->T, d->E, d->k, idx, w, rw.status, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_permute(idx, d->T, d->E, d->k, d->has_shared, rw.blockcnt, rw.blockbase, counts,
                     offsets, perm_src, inv, rw.status, st);
  return cuda_rc(e);
}

int moe_router_logits(int32_t T, int32_t H, int32_t E, const uint16_t* x, const float* wg,
                      float* logits, void* stream) {
  if (T < 1 || E < 1 || H < 16 || H % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x || !wg || !logits || !aligned(x, 16) || !aligned(wg, 16) || !aligned(logits, 4))
    return MOE_ERR_INVALID_ARG;
  return cuda_rc(
      launch_router_logits(x, wg, logits, T, H, E, static_cast<cudaStream_t>(stream)));
}

size_t moe_router_split_bytes(int32_t E, int32_t H) {
  if (E < 1 || H < 16 || H % 16) return 0;
  return static_cast<size_t>(3) * E * H * sizeof(uint16_t);
}

int moe_router_split(int32_t E, int32_t H, const float* wg, uint16_t* wg3, void* stream) {
  if (E < 1 || H < 16 || H % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!wg || !wg3 || !aligned(wg, 4) || !aligned(wg3, 16)) return MOE_ERR_INVALID_ARG;
  return cuda_rc(launch_router_split(wg, E, H, wg3, static_cast<cudaStream_t>(stream)));
}

int moe_router_logits_split(int32_t T, int32_t H, int32_t E, const uint16_t* x,
                            const uint16_t* wg3, float* logits, void* stream) {
  if (T < 1 || E < 1 || H < 16 || H % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x || !wg3 || !logits || !aligned(x, 16) || !aligned(wg3, 16) || !aligned(logits, 4))
    return MOE_ERR_INVALID_ARG;
  return cuda_rc(launch_router_logits_split(x, wg3, logits, T, H, E, nullptr,
                                            static_cast<cudaStream_t>(stream)));
}

int moe_quant_act(int32_t rows, int32_t cols, const uint16_t* x, uint8_t* q, uint8_t* s,
                  void* stream) {
  if (rows < 0 || cols <= 0 || cols % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !s || !aligned(x, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  return cuda_rc(launch_quant_act(x, rows, cols, q, s, static_cast<cudaStream_t>(stream)));
}

int moe_grouped_gemm_w13(const moe_dims* d, const uint8_t* xq, const uint8_t* xs,
                         const int32_t* perm_src, const int32_t* group_offsets,
                         const uint8_t* w13, const uint8_t* w13_s, uint16_t* y13, void* ws,
                         size_t ws_bytes, void* stream) {
  if (!dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!xq || !xs || !group_offsets || !y13 || !ws || !weights_ok(w13, w13_s))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(xs, 4) || !aligned(ws, kAlign) || !aligned(y13, 16))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_gemm_workspace_size(d)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carver c(ws);
  GemmWs g = carve_gemm(c, d, kMxfp4);
  if (cudaMemsetAsync(g.status, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e = launch_plan(group_offsets, groups_G(d), g.plan.out, g.status, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const uint8_t* act = xq;
  const uint8_t* act_s = xs;
  if (perm_src) {
    e = launch_gather_rows(xq, xs, perm_src, d->T, d->k, static_cast<int>(rows_R(d)),
                           static_cast<int>(rows_Rs(d)), d->H, g.xg, g.xsg, g.status, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    act = g.xg;
    act_s = g.xsg;
  }
  return run_gemm(d, act, act_s, group_offsets, w13, w13_s, 2 * d->I, d->H, y13, g.plan,
                  static_cast<int>(rows_Rs(d)), g.status, st, /*early_plan=*/0);
}

int moe_swiglu_quant(int32_t rows, int32_t I, const uint16_t* y13, uint8_t* hq, uint8_t* hs,
                     void* stream) {
  if (rows < 0 || I <= 0 || I % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!y13 || !hq || !hs || !aligned(y13, 16) || !aligned(hq, 16)) return MOE_ERR_INVALID_ARG;
  return cuda_rc(launch_swiglu_quant(y13, rows, I, hq, hs, static_cast<cudaStream_t>(stream)));
}

int moe_grouped_gemm_w2(const moe_dims* d, const uint8_t* hq, const uint8_t* hs,
                        const int32_t* group_offsets, const uint8_t* w2, const uint8_t* w2_s,
                        uint16_t* y2, void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!hq || !hs || !group_offsets || !y2 || !ws || !weights_ok(w2, w2_s))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(hq, 16) || !aligned(hs, 4) || !aligned(ws, kAlign) || !aligned(y2, 16))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_gemm_workspace_size(d)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carver c(ws);
  GemmWs g = carve_gemm(c, d, kMxfp4);
  if (cudaMemsetAsync(g.status, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e = launch_plan(group_offsets, groups_G(d), g.plan.out, g.status, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return run_gemm(d, hq, hs, group_offsets, w2, w2_s, d->H, d->I, y2, g.plan,
                  static_cast<int>(rows_Rs(d)), g.status, st, /*early_plan=*/0);
}

int moe_combine(const moe_dims* d, const uint16_t* y2, const int32_t* inv, const float* w,
                uint16_t* out, void* stream) {
  if (!dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!y2 || !inv || !w || !out || !aligned(y2, 16) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  return cuda_rc(launch_combine(y2, inv, w, d->T, d->k, d->H, d->has_shared, out, nullptr,
                                static_cast<cudaStream_t>(stream)));
}

int moe_forward(const moe_dims* d, const uint16_t* x, const float* logits,
                const moe_weights* W, uint16_t* out, const moe_debug_out* dbg, void* ws,
                size_t ws_bytes, void* stream) {
  return moe_forward_timed(d, x, logits, W, out, dbg, nullptr, ws, ws_bytes, stream);
}

size_t moe_host_workspace_size(const moe_dims* d) {
  if (!dims_ok(d)) return 0;
  Carver c(nullptr);
  carve_forward(c, d);
  carve_host_staging(c, d);
  return c.used;
}

int moe_forward_host(const moe_dims* d, const uint16_t* x_host, const float* logits_host,
                     const moe_weights* W, uint16_t* out_host, void* ws, size_t ws_bytes,
                     void* stream) {
  if (!dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x_host || !logits_host || !W || !out_host || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_host_workspace_size(d)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carver c(ws);
  carve_forward(c, d);  // the forward's own workspace comes first
  const size_t fwd_bytes = c.used;
  HostStagingWs h = carve_host_staging(c, d);
  const size_t xb = static_cast<size_t>(d->T) * d->H * sizeof(uint16_t);
  const size_t lb = static_cast<size_t>(d->T) * d->E * sizeof(float);
  if (cudaMemcpyAsync(h.x, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(h.logits, logits_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  int rc = moe_forward_timed(d, h.x, h.logits, W, h.out, nullptr, nullptr, ws, fwd_bytes, st);
  if (rc != MOE_OK) return rc;
  if (cudaMemcpyAsync(out_host, h.out, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"

namespace {
constexpr int kMaxPipelineDepth = 8;
}  // namespace

struct moe_host_pipeline {
  moe_dims d;
  moe_weights W;
  int depth;
  void* ws;
  size_t fwd_bytes;  // the forward's workspace, at the start of ws
  HostStagingWs slot[kMaxPipelineDepth];
  cudaStream_t s_in, s_comp, s_out;
  cudaEvent_t in_done[kMaxPipelineDepth], comp_done[kMaxPipelineDepth],
      out_done[kMaxPipelineDepth];
  long long submitted;
};

namespace {
void pipeline_release(moe_host_pipeline* p) {
  for (int j = 0; j < kMaxPipelineDepth; ++j) {
    if (p->in_done[j]) cudaEventDestroy(p->in_done[j]);
    if (p->comp_done[j]) cudaEventDestroy(p->comp_done[j]);
    if (p->out_done[j]) cudaEventDestroy(p->out_done[j]);
  }
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_comp) cudaStreamDestroy(p->s_comp);
  if (p->s_out) cudaStreamDestroy(p->s_out);
  delete p;
}
}  // namespace

extern "C" {

size_t moe_host_pipeline_workspace_size(const moe_dims* d, int depth) {
  if (!dims_ok(d) || depth < 1 || depth > kMaxPipelineDepth) return 0;
  Carver c(nullptr);
  carve_forward(c, d);
  for (int j = 0; j < depth; ++j) carve_host_staging(c, d);
  return c.used;
}

int moe_host_pipeline_create(const moe_dims* d, const moe_weights* W, int depth, void* ws,
                             size_t ws_bytes, moe_host_pipeline** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!W || !ws || depth < 1 || depth > kMaxPipelineDepth) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(W->w13, W->w13_s) || !weights_ok(W->w2, W->w2_s)) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_host_pipeline_workspace_size(d, depth)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_host_pipeline* p = new (std::nothrow) moe_host_pipeline{};
  if (!p) return MOE_ERR_CUDA;
  p->d = *d;
  p->W = *W;
  p->depth = depth;
  p->ws = ws;
  Carver c(ws);
  carve_forward(c, d);
  p->fwd_bytes = c.used;
  for (int j = 0; j < depth; ++j) p->slot[j] = carve_host_staging(c, d);
  bool ok = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess;
  for (int j = 0; ok && j < depth; ++j)
    ok = cudaEventCreateWithFlags(&p->in_done[j], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->comp_done[j], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->out_done[j], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    pipeline_release(p);
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}

int moe_host_pipeline_submit(moe_host_pipeline* p, const uint16_t* x_host,
                             const float* logits_host, uint16_t* out_host) {
  if (!p || !x_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
  const moe_dims* d = &p->d;
  const int j = static_cast<int>(p->submitted % p->depth);
  const bool reuse = p->submitted >= p->depth;  // slot j held step submitted - depth
  const HostStagingWs& h = p->slot[j];
  const size_t xb = static_cast<size_t>(d->T) * d->H * sizeof(uint16_t);
  const size_t lb = static_cast<size_t>(d->T) * d->E * sizeof(float);
  // inputs: once the previous user of the slot has consumed its inputs
  if (reuse && cudaStreamWaitEvent(p->s_in, p->comp_done[j], 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(h.x, x_host, xb, cudaMemcpyHostToDevice, p->s_in) != cudaSuccess ||
      cudaMemcpyAsync(h.logits, logits_host, lb, cudaMemcpyHostToDevice, p->s_in) !=
          cudaSuccess ||
      cudaEventRecord(p->in_done[j], p->s_in) != cudaSuccess)
    return MOE_ERR_CUDA;
  // the layer: once the inputs landed and the slot's previous output was copied out
  if (cudaStreamWaitEvent(p->s_comp, p->in_done[j], 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (reuse && cudaStreamWaitEvent(p->s_comp, p->out_done[j], 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  int rc = moe_forward_timed(d, h.x, h.logits, &p->W, h.out, nullptr, nullptr, p->ws,
                             p->fwd_bytes, p->s_comp);
  if (rc != MOE_OK) return rc;
  if (cudaEventRecord(p->comp_done[j], p->s_comp) != cudaSuccess) return MOE_ERR_CUDA;
  // output
  if (cudaStreamWaitEvent(p->s_out, p->comp_done[j], 0) != cudaSuccess ||
      cudaMemcpyAsync(out_host, h.out, xb, cudaMemcpyDeviceToHost, p->s_out) != cudaSuccess ||
      cudaEventRecord(p->out_done[j], p->s_out) != cudaSuccess)
    return MOE_ERR_CUDA;
  ++p->submitted;
  return MOE_OK;
}

int moe_host_pipeline_sync(moe_host_pipeline* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  const bool ok = cudaStreamSynchronize(p->s_in) == cudaSuccess &&
                  cudaStreamSynchronize(p->s_comp) == cudaSuccess &&
                  cudaStreamSynchronize(p->s_out) == cudaSuccess;
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

int moe_host_pipeline_destroy(moe_host_pipeline* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  const int rc = moe_host_pipeline_sync(p);
  pipeline_release(p);
  return rc;
}

}  // extern "C"

namespace {

// The layer a1..a7 on one stream for either weight format (see moe_forward_timed).
int forward_impl(const moe_dims* d, const uint16_t* x, const float* logits,
                 const LayerWeights& W, uint16_t* out, const moe_debug_out* dbg,
                 void* const* events, void* ws, size_t ws_bytes, cudaStream_t st,
                 const moe_options* opt = nullptr) {
  if (!(W.fmt == kMxfp4 ? dims_ok(d) : nv_dims_ok(d))) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x || !logits || !out || !ws) return MOE_ERR_INVALID_ARG;
  const bool fuse_combine = opt && opt->fuse_combine;
  const bool fuse_swiglu = opt && opt->fuse_swiglu;
  const int pair_tiles = opt ? opt->pair_tiles : 0;
  const int chunk_rows = opt ? opt->large_chunk_rows : 0;
  if (opt && ((opt->fuse_combine != 0 && opt->fuse_combine != 1) ||
              (opt->fuse_swiglu != 0 && opt->fuse_swiglu != 1) ||
              (opt->pair_tiles != 0 && opt->pair_tiles != 1) ||
              ((fuse_combine || fuse_swiglu || pair_tiles) && W.fmt != kMxfp4)))
    return MOE_ERR_INVALID_ARG;
  if (chunk_rows != 0 &&
      (chunk_rows < kMinChunkRows || chunk_rows > kLargeBN || chunk_rows % 16 != 0))
    return MOE_ERR_INVALID_ARG;
  // the fused W13 epilogue runs on SM pairs: 2I % 256 == 0 always, H % 512 needed
  if (fuse_swiglu && d->H % 512 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!weights_ok(W.w13, W.w13_s) || !weights_ok(W.w2, W.w2_s)) return MOE_ERR_INVALID_ARG;
  if (!aligned(W.w13_gs, 4) || !aligned(W.w2_gs, 4)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ws, kAlign) || !aligned(logits, 4))
    return MOE_ERR_INVALID_ARG;
  Carver c(ws);
  ForwardWs f = carve_forward(c, d, W.fmt);
  if (ws_bytes < c.used) return MOE_ERR_WORKSPACE_TOO_SMALL;
  f.gemm.plan.out.chunk_rows = chunk_rows;
  // caller-visible intermediates replace the workspace buffers
  uint8_t* dbg_hq = nullptr;
  uint8_t* dbg_hs = nullptr;
  if (dbg) {
#define MOE_DBG(field) \
  if (dbg->field) f.field = dbg->field;
    MOE_DBG(idx) MOE_DBG(w) MOE_DBG(counts) MOE_DBG(offsets) MOE_DBG(perm_src) MOE_DBG(inv)
    MOE_DBG(xq) MOE_DBG(xs) MOE_DBG(y13) MOE_DBG(hq) MOE_DBG(hs) MOE_DBG(y2)
#undef MOE_DBG
    dbg_hq = dbg->hq;
    dbg_hs = dbg->hs;
    if (!aligned(f.xq, 16) || !aligned(f.y13, 16) || !aligned(f.hq, 16) || !aligned(f.y2, 16) ||
        !aligned(f.hs, 4) || !aligned(f.xs, 4))
      return MOE_ERR_INVALID_ARG;
  }
  const int T = d->T, H = d->H, I = d->I, E = d->E, k = d->k;
  const int Rs = static_cast<int>(rows_Rs(d));
  uint32_t* status = f.route.status;  // cleared by the first kernel below
  auto mark = [&](int i) -> bool {
    return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };
  cudaError_t e;
#define MOE_TRY(call)                     \
  e = (call);                             \
  if (e != cudaSuccess) return MOE_ERR_CUDA;
#define MOE_MARK(i) \
  if (!mark(i)) return MOE_ERR_CUDA;
  MOE_MARK(0)
  if (T <= kPrepMaxT) {
    // decode: route + histogram + permute + tile plan in one CTA
    MOE_TRY(launch_prep_small(logits, T, E, k, d->has_shared, f.idx, f.w, f.counts, f.offsets,
                              f.perm_src, f.inv, f.gemm.plan.out, status, st))
  } else {
    MOE_TRY(launch_route(logits, T, E, k, f.idx, f.w, status, st))
    MOE_TRY(launch_permute(f.idx, T, E, k, d->has_shared, f.route.blockcnt, f.route.blockbase,
                           f.counts, f.offsets, f.perm_src, f.inv, status, st))
    // the tile plan before the quant-scatter, as in the one-CTA path, so that the
    // plan is complete two launches before W13
    MOE_TRY(launch_plan(f.offsets, groups_G(d), f.gemm.plan.out, status, st))
  }
  MOE_MARK(1)
  // quantise each token once, writing its codes (MXFP4 path) or their exact bf16
  // values (NVFP4 path) straight into its packed rows
  uint8_t* xq_out = dbg && dbg->xq ? f.xq : nullptr;
  uint8_t* xs_out = dbg && dbg->xs ? f.xs : nullptr;
  if (W.fmt == kMxfp4) {
    MOE_TRY(launch_quant_scatter(x, T, H, k, d->has_shared, f.inv, xq_out, xs_out, f.gemm.xg,
                                 f.gemm.xsg, fuse_combine ? f.cnt : nullptr, status, st))
  } else {
    MOE_TRY(launch_quant_scatter_bf16(x, T, H, k, d->has_shared, f.inv, xq_out, xs_out,
                                      f.gemm.xe, status, st))
  }
  MOE_MARK(2)
  MOE_MARK(3)  // (stage 3, the plan, now runs inside stage 1)
  // every group (a routed expert or the shared expert) holds at most T rows; W13
  // follows the quant-scatter, and the plan was written before it
  int rc;
  if (W.fmt == kMxfp4) {
    FusedCombine fs;
    fs.pair_tiles = pair_tiles;
    if (fuse_swiglu) {
      fs.hq = f.hq;
      fs.hs = f.hs;
    }
    rc = run_gemm(d, f.gemm.xg, f.gemm.xsg, f.offsets, W.w13, W.w13_s, 2 * I, H, f.y13,
                  f.gemm.plan, T, status, st, /*early_plan=*/1, fs);
  } else {
    rc = run_gemm_nv(d, f.gemm.xe, W.w13, W.w13_s, W.w13_gs, 2, 2 * I, H, f.y13, f.gemm.plan, T,
                     status, f.gemm.share_part, st);
  }
  if (rc != MOE_OK) return rc;
  MOE_MARK(4)
  if (W.fmt == kMxfp4) {
    if (!fuse_swiglu) MOE_TRY(launch_swiglu_quant(f.y13, Rs, I, f.hq, f.hs, st))
  } else {
    MOE_TRY(launch_swiglu_quant_bf16(f.y13, Rs, I, dbg_hq, dbg_hs, f.he, st))
  }
  MOE_MARK(5)
  if (W.fmt == kMxfp4) {
    FusedCombine fc;
    fc.pair_tiles = pair_tiles;
    if (fuse_combine) {
      fc.out = out;
      fc.perm_src = f.perm_src;
      fc.inv = f.inv;
      fc.w = f.w;
      fc.cnt = f.cnt;
    }
    rc = run_gemm(d, f.hq, f.hs, f.offsets, W.w2, W.w2_s, H, I, f.y2, f.gemm.plan, T, status,
                  st, /*early_plan=*/1, fc);  // follows SwiGLU; the plan preceded W13
  } else {
    rc = run_gemm_nv(d, f.he, W.w2, W.w2_s, W.w2_gs, 1, H, I, f.y2, f.gemm.plan, T, status,
                     f.gemm.share_part, st);
  }
  if (rc != MOE_OK) return rc;
  MOE_MARK(6)
  if (!fuse_combine)
    MOE_TRY(launch_combine(f.y2, f.inv, f.w, T, k, H, d->has_shared, out, status, st))
  MOE_MARK(7)
#undef MOE_TRY
#undef MOE_MARK
  return MOE_OK;
}

LayerWeights mx_weights(const moe_weights* W) {
  return LayerWeights{kMxfp4, W->w13, W->w13_s, W->w2, W->w2_s, nullptr, nullptr};
}

LayerWeights nv_weights(const moe_weights_nvfp4* W) {
  return LayerWeights{kNvfp4, W->w13, W->w13_s, W->w2, W->w2_s, W->w13_gs, W->w2_gs};
}

// Stand-alone NVFP4 GEMM: plan, FP8 operand expanded to bf16 rows, GEMM.
int gemm_nv_call(const moe_dims* d, const uint8_t* q, const uint8_t* qs, const int32_t* perm_src,
                 const int32_t* group_offsets, const uint8_t* w, const uint8_t* w_s,
                 const float* gs, int gs_segments, int N, int K, uint16_t* y, void* ws,
                 size_t ws_bytes, cudaStream_t st) {
  Carver c(ws);
  GemmWs g = carve_gemm(c, d, kNvfp4);
  if (ws_bytes < c.used) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (cudaMemsetAsync(g.status, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_plan(group_offsets, groups_G(d), g.plan.out, g.status, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int Rs = static_cast<int>(rows_Rs(d));
  if (launch_expand_rows(q, qs, perm_src, d->T, d->k, static_cast<int>(rows_R(d)), Rs, K, g.xe,
                         g.status, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return run_gemm_nv(d, g.xe, w, w_s, gs, gs_segments, N, K, y, g.plan, Rs, g.status,
                     g.share_part, st);
}

}  // namespace

extern "C" {

int moe_forward_timed(const moe_dims* d, const uint16_t* x, const float* logits,
                      const moe_weights* W, uint16_t* out, const moe_debug_out* dbg,
                      void* const* events, void* ws, size_t ws_bytes, void* stream) {
  if (!W) return dims_ok(d) ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  return forward_impl(d, x, logits, mx_weights(W), out, dbg, events, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream));
}

int moe_forward_ex(const moe_dims* d, const uint16_t* x, const float* logits,
                   const moe_weights* W, const moe_options* opt, uint16_t* out,
                   const moe_debug_out* dbg, void* const* events, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!W) return dims_ok(d) ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  return forward_impl(d, x, logits, mx_weights(W), out, dbg, events, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream), opt);
}

size_t moe_workspace_size_nvfp4(const moe_dims* d) {
  if (!nv_dims_ok(d)) return 0;
  Carver c(nullptr);
  carve_forward(c, d, kNvfp4);
  return c.used;
}

size_t moe_gemm_workspace_size_nvfp4(const moe_dims* d) {
  if (!nv_dims_ok(d)) return 0;
  Carver c(nullptr);
  carve_gemm(c, d, kNvfp4);
  return c.used;
}

int moe_forward_nvfp4(const moe_dims* d, const uint16_t* x, const float* logits,
                      const moe_weights_nvfp4* W, uint16_t* out, const moe_debug_out* dbg,
                      void* ws, size_t ws_bytes, void* stream) {
  return moe_forward_nvfp4_timed(d, x, logits, W, out, dbg, nullptr, ws, ws_bytes, stream);
}

int moe_forward_nvfp4_timed(const moe_dims* d, const uint16_t* x, const float* logits,
                            const moe_weights_nvfp4* W, uint16_t* out, const moe_debug_out* dbg,
                            void* const* events, void* ws, size_t ws_bytes, void* stream) {
  if (!W) return nv_dims_ok(d) ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  return forward_impl(d, x, logits, nv_weights(W), out, dbg, events, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream));
}

int moe_grouped_gemm_w13_nvfp4(const moe_dims* d, const uint8_t* xq, const uint8_t* xs,
                               const int32_t* perm_src, const int32_t* group_offsets,
                               const uint8_t* w13, const uint8_t* w13_s, const float* w13_gs,
                               uint16_t* y13, void* ws, size_t ws_bytes, void* stream) {
  if (!nv_dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!xq || !xs || !group_offsets || !y13 || !ws || !weights_ok(w13, w13_s))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(ws, kAlign) || !aligned(y13, 16) || !aligned(w13_gs, 4))
    return MOE_ERR_INVALID_ARG;
  return gemm_nv_call(d, xq, xs, perm_src, group_offsets, w13, w13_s, w13_gs, 2, 2 * d->I, d->H,
                      y13, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

int moe_grouped_gemm_w2_nvfp4(const moe_dims* d, const uint8_t* hq, const uint8_t* hs,
                              const int32_t* group_offsets, const uint8_t* w2,
                              const uint8_t* w2_s, const float* w2_gs, uint16_t* y2, void* ws,
                              size_t ws_bytes, void* stream) {
  if (!nv_dims_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!hq || !hs || !group_offsets || !y2 || !ws || !weights_ok(w2, w2_s))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(hq, 16) || !aligned(ws, kAlign) || !aligned(y2, 16) || !aligned(w2_gs, 4))
    return MOE_ERR_INVALID_ARG;
  return gemm_nv_call(d, hq, hs, nullptr, group_offsets, w2, w2_s, w2_gs, 1, d->H, d->I, y2, ws,
                      ws_bytes, static_cast<cudaStream_t>(stream));
}

int moe_selftest_wait_timeout(void* ws, void* stream) {
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_rc(launch_k(k_selftest_wait, 1, 32, 0, st, status));
}

int moe_check_status(const void* ws, void* stream, uint32_t* bits_out) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  uint32_t bits = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&bits, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  return bits ? MOE_ERR_DEVICE_CHECK : MOE_OK;
}

}  // extern "C"
