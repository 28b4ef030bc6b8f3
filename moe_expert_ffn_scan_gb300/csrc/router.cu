// f4: router gate projection, logits[t][e] = sum_h x[t][h] * W_g[e][h] in fp32.
//
// The TopK step of "Pushing the Limits of Serving DeepSeek-V4-Pro" (LMSYS, H20), §3.2,
// ranks per-expert router scores; this is the projection that produces them, kept in
// fp32 (x is the bf16 hidden state, W_g the fp32 gate weight).  A plain fp32
// contraction on the CUDA cores: two shapes of it matter.
//   * Decode and mid T (T <= 1024): HBM- / latency-bound on W_g (E x H x 4 bytes, 11 MB at E=384,
//     H=7168).  k_router_gemv: a CTA owns kRgExperts experts and up to 8 or 16
//     tokens; its 8 warps split H, each lane issues a round of W_g and x loads
//     together and keeps experts x tokens partial sums; warp sums, then the 8 warp
//     partials are added in warp order (deterministic, no atomics).
//   * Prefill (T > 1024): 2*T*E*H flops, compute-bound.  k_router_tiled: classic
//     register-tiled SGEMM, 128 tokens x 64 experts per CTA, 8 x 4 outputs per
//     thread, K staged 16 columns at a time in shared memory (x converted to fp32).
// Both accumulate each logit's H products in one fixed order, so results are
// reproducible run to run.
#include "kernels.cuh"

namespace moe {

// Experts per CTA: 2 measured best (1: x re-read too often; 4: too few CTAs at mid T).
constexpr int kRgExperts = 2;
constexpr int kRgWarps = 8;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// TT tokens per CTA (blockIdx.y walks token groups of TT); U 4-column steps per lane
// whose W_g and x loads are all issued before any of their FMAs.  Loads past the
// warp's slice read a valid column with W_g = 0 (adds +0, leaving sums unchanged), and
// token rows past T read row T-1 into sums that are never written, so the loop body
// is straight-line code.
template <int TT, int U>
__global__ void __launch_bounds__(256) k_router_gemv(const uint16_t* __restrict__ x,
                                                     const float* __restrict__ wg,
                                                     float* __restrict__ logits, int T, int H,
                                                     int E) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kRgWarps][kRgExperts][TT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * kRgExperts;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  // this warp's slice of H, in 4-column steps (H % 16 == 0: slices are whole steps)
  const int steps = H / 4;
  const int per = (steps + kRgWarps - 1) / kRgWarps;
  const int s0 = warp * per, s1 = min(steps, s0 + per);
  const float* wrow[kRgExperts];
#pragma unroll
  for (int j = 0; j < kRgExperts; ++j)
    wrow[j] = wg + static_cast<size_t>(min(e0 + j, E - 1)) * H;  // clamped rows: unused
  const uint16_t* xrow[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) xrow[t] = x + static_cast<size_t>(t0 + min(t, nt - 1)) * H;
  float acc[kRgExperts][TT];
#pragma unroll
  for (int j = 0; j < kRgExperts; ++j)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[j][t] = 0.f;
  for (int sb = s0 + lane; sb < s1; sb += 32 * U) {
    float4 w[U][kRgExperts];
    uint2 xv[U][TT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = sb + 32 * u;
      const bool ok = s < s1;
      const int sl = ok ? s : s1 - 1;
#pragma unroll
      for (int j = 0; j < kRgExperts; ++j)
        w[u][j] = ok ? __ldg(reinterpret_cast<const float4*>(wrow[j] + sl * 4))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int t = 0; t < TT; ++t)
        xv[u][t] = __ldg(reinterpret_cast<const uint2*>(xrow[t] + sl * 4));
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float x0 = bf16_lo(xv[u][t].x), x1 = bf16_hi(xv[u][t].x),
                    x2 = bf16_lo(xv[u][t].y), x3 = bf16_hi(xv[u][t].y);
#pragma unroll
        for (int j = 0; j < kRgExperts; ++j) {
          float a = acc[j][t];
          a = fmaf(x0, w[u][j].x, a);
          a = fmaf(x1, w[u][j].y, a);
          a = fmaf(x2, w[u][j].z, a);
          a = fmaf(x3, w[u][j].w, a);
          acc[j][t] = a;
        }
      }
  }
#pragma unroll
  for (int j = 0; j < kRgExperts; ++j)
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float v = acc[j][t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (lane == 0) red[warp][j][t] = v;
    }
  __syncthreads();
  if (threadIdx.x < kRgExperts * TT) {
    const int j = threadIdx.x / TT, t = threadIdx.x % TT;
    if (t < nt && e0 + j < E) {
      float v = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < kRgWarps; ++w8) v += red[w8][j][t];
      logits[static_cast<size_t>(t0 + t) * E + e0 + j] = v;
    }
  }
}

constexpr int kRtBM = 128;  // tokens per CTA
constexpr int kRtBN = 64;   // experts per CTA
constexpr int kRtBK = 16;   // H columns per shared-memory stage

__global__ void __launch_bounds__(256) k_router_tiled(const uint16_t* __restrict__ x,
                                                      const float* __restrict__ wg,
                                                      float* __restrict__ logits, int T, int H,
                                                      int E) {
  pdl_wait();
  pdl_trigger();
  // k-major tiles; +4 floats of padding per row keeps the 16-byte reads aligned
  __shared__ __align__(16) float As[2][kRtBK][kRtBM + 4];
  __shared__ __align__(16) float Bs[2][kRtBK][kRtBN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;  // thread computes tokens ty*8.., experts tx*4..
  const int m0 = blockIdx.y * kRtBM, n0 = blockIdx.x * kRtBN;
  // global -> register staging: x row (tid / 2), 8 bf16 at column (tid % 2) * 8;
  // W_g row (tid / 4), 4 floats at column (tid % 4) * 4
  const int xr = tid >> 1, xc = (tid & 1) * 8;
  const int wr = tid >> 2, wc = (tid & 3) * 4;
  const bool x_ok = m0 + xr < T, w_ok = n0 + wr < E;
  const uint16_t* xp = x + static_cast<size_t>(x_ok ? m0 + xr : 0) * H + xc;
  const float* wp = wg + static_cast<size_t>(w_ok ? n0 + wr : 0) * H + wc;
  uint4 xv = x_ok ? __ldg(reinterpret_cast<const uint4*>(xp)) : make_uint4(0, 0, 0, 0);
  float4 wv = w_ok ? __ldg(reinterpret_cast<const float4*>(wp)) : make_float4(0.f, 0.f, 0.f, 0.f);
  auto stash = [&](int buf) {
    const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      As[buf][xc + 2 * i][xr] = bf16_lo(u[i]);
      As[buf][xc + 2 * i + 1][xr] = bf16_hi(u[i]);
    }
    Bs[buf][wc + 0][wr] = wv.x;
    Bs[buf][wc + 1][wr] = wv.y;
    Bs[buf][wc + 2][wr] = wv.z;
    Bs[buf][wc + 3][wr] = wv.w;
  };
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  stash(0);
  __syncthreads();
  const int nk = H / kRtBK;
  for (int kb = 0; kb < nk; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nk) {  // next tile's loads in flight during this tile's FMAs
      const int off = (kb + 1) * kRtBK;
      xv = x_ok ? __ldg(reinterpret_cast<const uint4*>(xp + off)) : make_uint4(0, 0, 0, 0);
      wv = w_ok ? __ldg(reinterpret_cast<const float4*>(wp + off))
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kRtBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    if (kb + 1 < nk) stash(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = m0 + ty * 8 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = n0 + tx * 4 + j;
      if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[i][j];
    }
  }
}

cudaError_t launch_router_logits(const uint16_t* x, const float* wg, float* logits, int T, int H,
                                 int E, cudaStream_t st) {
  if (T <= 8) {
    dim3 grid((E + kRgExperts - 1) / kRgExperts, 1);
    return launch_k(k_router_gemv<8, 4>, grid, 256, 0, st, x, wg, logits, T, H, E);
  }
  if (T <= kRouterGemvMaxT) {
    dim3 grid((E + kRgExperts - 1) / kRgExperts, (T + 15) / 16);
    return launch_k(k_router_gemv<16, 2>, grid, 256, 0, st, x, wg, logits, T, H, E);
  }
  dim3 grid((E + kRtBN - 1) / kRtBN, (T + kRtBM - 1) / kRtBM);
  return launch_k(k_router_tiled, grid, 256, 0, st, x, wg, logits, T, H, E);
}


// ---------------------------------------------------------------- tensor cores ------
// The same projection on the tcgen05 tensor cores, for prefill-sized T.  W_g is split
// once into three bf16 matrices with W_g = hi + mid + lo exactly (hi = bf16(W_g), mid =
// bf16(W_g - hi), lo = W_g - hi - mid: 8 + 8 + 8 significant bits, the fp32 weight's 24;
// exact unless a piece falls below bf16's normal range, i.e. for weights under about
// 2^-110).  x is bf16, so every product x * piece is exact in fp32, and kind::f16 MMAs
// with fp32 accumulation sum x . hi, x . mid and x . lo of each 16-column step into one
// accumulator: the fp32 contraction, on the tensor cores.
//
// k_router_tc: a CTA owns tiles of 128 tokens x 128 experts (persistent), K staged 64
// columns at a time (one 128-byte swizzle row) by TMA -- x's tile and the three
// pieces' tiles -- three stages; warp 0 issues the TMA, warp 1 the MMAs (12 per stage:
// 4 K-steps x 3 pieces, into a double-buffered TMEM accumulator), warps 4-7 store the
// fp32 logits.  Every wait is bounded.

namespace {

constexpr int kRtStages = 3;
constexpr int kRtTile = 128;                     // tokens and experts per tile
constexpr int kRtXBytes = kRtTile * 128;          // [128 rows][64 bf16]
constexpr int kRtStageBytes = 4 * kRtXBytes;      // x + three pieces
constexpr int kRtOffBar = kRtStages * kRtStageBytes;
constexpr int kRtSmem = kRtOffBar + (2 * kRtStages + 4) * 8 + 16;

__global__ void __launch_bounds__(256) k_router_split(const float* __restrict__ wg, size_t n,
                                                      uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float w = wg[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);  // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));  // exact
    out[i] = *reinterpret_cast<const uint16_t*>(&hi);
    out[n + i] = *reinterpret_cast<const uint16_t*>(&mid);
    out[2 * n + i] = *reinterpret_cast<const uint16_t*>(&lo);
  }
}

__device__ __forceinline__ uint32_t idesc_bf16_m128(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

__global__ void __launch_bounds__(256, 1)
    k_router_tc(const __grid_constant__ CUtensorMap tmXr, const __grid_constant__ CUtensorMap tmWr,
                float* __restrict__ logits, int T, int H, int E, uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRtOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + kRtStages;
  uint64_t* acc_full = empty + kRtStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kRtOffBar + (2 * kRtStages + 4) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool misaligned = (smem_u32(smem) & 1023u) != 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    *abort_flag = misaligned ? 1 : 0;
    if (misaligned) set_status(status, STATUS_BAD_PLAN);
    fence_mbar_init();
    tma_prefetch_desc(&tmXr);
    tma_prefetch_desc(&tmWr);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;
  const int ttiles = (T + kRtTile - 1) / kRtTile, etiles = (E + kRtTile - 1) / kRtTile;
  const long long total = static_cast<long long>(ttiles) * etiles;
  const int nk = (H + 63) / 64;
  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
        const int t0 = static_cast<int>(L / etiles) * kRtTile;
        const int e0 = static_cast<int>(L % etiles) * kRtTile;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kRtStages;
          if (it >= kRtStages &&
              !mbar_wait(&empty[s], ((it / kRtStages) & 1u) ^ 1u, status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kRtStageBytes;
          mbar_arrive_expect_tx(&full[s], kRtStageBytes);
          tma_load_2d(st, &tmXr, &full[s], kb * 64, t0);
#pragma unroll
          for (int pc = 0; pc < 3; ++pc)
            tma_load_3d(st + (1 + pc) * kRtXBytes, &tmWr, &full[s], kb * 64, e0, pc);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      const uint32_t idesc = idesc_bf16_m128(kRtTile);
      for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
        const uint32_t b = tc & 1u, use = tc >> 1;
        if (tc >= 2 && !mbar_wait(&acc_empty[b], (use - 1) & 1u, status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * kRtTile;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kRtStages;
          if (!mbar_wait(&full[s], (it / kRtStages) & 1u, status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = smem_u32(smem + s * kRtStageBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(base + kk * 32, 0, 1024, kLayoutSw128);
#pragma unroll
            for (int pc = 0; pc < 3; ++pc) {
              const uint64_t bd =
                  smem_desc(base + (1 + pc) * kRtXBytes + kk * 32, 0, 1024, kLayoutSw128);
              mma_bf16_ss(d, ad, bd, idesc, kb > 0 || kk > 0 || pc > 0);
            }
          }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&acc_full[b]);
        ++tc;
      }
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    uint32_t tc = 0;
    for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
      const int t0 = static_cast<int>(L / etiles) * kRtTile;
      const int e0 = static_cast<int>(L % etiles) * kRtTile;
      const uint32_t b = tc & 1u, use = tc >> 1;
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&acc_full[b], use & 1u, status, abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, w_ok, 0)) break;
      tc_fence_after();
      const int t = t0 + q * 32 + lane;  // this thread's token row (TMEM lane)
      const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * kRtTile;
      float* out = logits + static_cast<size_t>(t < T ? t : 0) * E;
      for (int c0 = 0; c0 < kRtTile && e0 + c0 < E; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(acc + c0, r);
        tmem_ld_wait();
        if (t < T) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (e0 + c0 + i < E) out[e0 + c0 + i] = __uint_as_float(r[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++tc;
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

cudaError_t launch_router_split(const float* wg, int E, int H, uint16_t* wg3, cudaStream_t st) {
  const size_t n = static_cast<size_t>(E) * H;
  if (n == 0) return cudaSuccess;
  const long long blocks = static_cast<long long>((n + 255) / 256);
  const unsigned grid = static_cast<unsigned>(blocks < 4096 ? blocks : 4096);
  return launch_k(k_router_split, grid, 256, 0, st, wg, n, wg3);
}

cudaError_t launch_router_logits_split(const uint16_t* x, const uint16_t* wg3, float* logits,
                                       int T, int H, int E, uint32_t* status, cudaStream_t st) {
  EncodeTiledFn enc = get_encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmX, tmW;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, kRtTile};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(E), 3};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * 2,
                             static_cast<cuuint64_t>(E) * static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[3] = {64, kRtTile, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(wg3), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static unsigned long long attr_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || attr_ctx[dev] != ctx) {
    e = cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (e != cudaSuccess) return e;
    attr_ctx[dev] = current_context_id();
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>((T + kRtTile - 1) / kRtTile) *
                          ((E + kRtTile - 1) / kRtTile);
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  return launch_k(k_router_tc, grid, 256, kRtSmem, st, tmX, tmW, logits, T, H, E, status);
}

}  // namespace moe
