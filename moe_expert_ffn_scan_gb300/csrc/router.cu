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

}  // namespace moe
