// Memory-bound stages: a3 online FP8 activation quantisation, a5 SwiGLU fused with
// FP8 requantisation, the packed-row gather in front of W13, and a7 the weighted
// top-k combine with the shared-expert add.
//
// Pages: "Pushing the Limits of Serving DeepSeek-V4-Pro" (LMSYS, H20) -- §2.2 online
// FP8 activations, §3.2 fused FP8 quantisation and TopK reduction + shared-expert
// add, §4.3 SwiGLU fused with the quantisation that emits W2's data and scales.
//
// All of them move 16 bytes per thread per access (128-bit loads and stores).
#include "kernels.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Quantise the 16 values one lane of an 8-lane group holds; the group covers one
// 128-column block.  Returns the 16 codes packed little-endian and the block's scale
// exponent (the same in every lane of the group).  All 32 lanes must call it.
__device__ __forceinline__ uint4 quant16(const float (&f)[16], int& e) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int off = 4; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  e = fp8_scale_exponent(amax);
  const float s = pow2_neg(e);
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = e4m3x2(f[2 * i] * s, f[2 * i + 1] * s);
  return make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16),
                    c[6] | (c[7] << 16));
}

__device__ __forceinline__ void load_bf16x16(const uint16_t* p, float (&f)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  float lo[8], hi[8];
  bf16x8_to_f32(q[0], lo);
  bf16x8_to_f32(q[1], hi);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[i] = lo[i];
    f[8 + i] = hi[i];
  }
}

// Thread -> (row, 128-column block, lane in the block's 8-lane group).  Idx is the
// index type: 32-bit whenever 8 x rows x blocks-per-row fits (one 32-bit division per
// thread), 64-bit otherwise.
template <typename Idx>
struct BlockLane {
  Idx r, b;
  int sub;
  bool live;
  __device__ __forceinline__ BlockLane(int rows, int nblk) {
    const Idx gid = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x;
    const Idx blk = gid >> 3;
    sub = static_cast<int>(gid & 7);
    live = blk < static_cast<Idx>(rows) * static_cast<Idx>(nblk);
    r = live ? blk / static_cast<Idx>(nblk) : 0;
    b = live ? blk - r * static_cast<Idx>(nblk) : 0;
  }
};

// 2^e as a float, exact for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
}

// 16 E4M3 codes (byte j = element j) of a block with scale exponent e -> the 16 exact
// values code x 2^e as bf16 (element j at position j of lo:hi).  Exact whenever the
// value is a bf16 value: always, except below bf16's subnormal floor (a block whose
// amax is under about 2^-116 can lose its smallest codes there).
__device__ __forceinline__ void fp8x16_expand(const uint4& c, int e, uint4& lo, uint4& hi) {
  const float s = pow2f(e);
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * half)) & 0xFFFFu), __NV_E4M3);
      const float2 f = __half22float2(__half2(hr));
      __nv_bfloat162 b = __floats2bfloat162_rn(f.x * s, f.y * s);
      o[2 * i + half] = *reinterpret_cast<uint32_t*>(&b);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace

// a3.  Eight lanes per 128-column block, 16 values (two 16-byte loads) per lane.
template <typename Idx>
__global__ void __launch_bounds__(256) k_quant_act(const uint16_t* __restrict__ x, int rows,
                                                   int cols, uint8_t* __restrict__ q,
                                                   uint8_t* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int nblk = cols / 128;
  const BlockLane<Idx> L(rows, nblk);
  float f[16];
  if (L.live) {
    load_bf16x16(x + static_cast<size_t>(L.r) * cols + L.b * 128 + L.sub * 16, f);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = 0.f;
  }
  int e;
  const uint4 c = quant16(f, e);
  if (!L.live) return;
  *reinterpret_cast<uint4*>(q + static_cast<size_t>(L.r) * cols + L.b * 128 + L.sub * 16) = c;
  if (L.sub == 0) s[static_cast<size_t>(L.r) * nblk + L.b] = static_cast<uint8_t>(e + 127);
}

// a3 fused with the packed-row gather: token t's codes and scales go to xq / xs
// (when given) and straight to its k routed rows inv[t*k + j] and its shared row R + t
// of the packed activations, so no separate gather pass re-reads them.
template <typename Idx>
__global__ void __launch_bounds__(256) k_quant_scatter(const uint16_t* __restrict__ x, int T,
                                                       int H, int k, int has_shared,
                                                       const int32_t* __restrict__ inv,
                                                       uint8_t* __restrict__ xq,
                                                       uint8_t* __restrict__ xs,
                                                       uint8_t* __restrict__ xg,
                                                       uint8_t* __restrict__ xsg,
                                                       int32_t* __restrict__ cnt,
                                                       uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int nblk = H / 128;
  const BlockLane<Idx> L(T, nblk);
  // the (token, 128-column block) arrival counters of a W2 GEMM that performs the
  // combine in its epilogue start at zero
  if (cnt && L.live && L.sub == 0) cnt[static_cast<size_t>(L.r) * nblk + L.b] = 0;
  float f[16];
  if (L.live) {
    load_bf16x16(x + static_cast<size_t>(L.r) * H + L.b * 128 + L.sub * 16, f);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = 0.f;
  }
  int e;
  const uint4 c = quant16(f, e);
  if (!L.live) return;
  const uint8_t scale = static_cast<uint8_t>(e + 127);
  const size_t t = static_cast<size_t>(L.r);
  const int col = static_cast<int>(L.b) * 128 + L.sub * 16;
  if (xq) *reinterpret_cast<uint4*>(xq + t * H + col) = c;
  if (xs && L.sub == 0) xs[t * nblk + L.b] = scale;
  const long long R = static_cast<long long>(T) * k;
  for (int j = 0; j <= k; ++j) {
    long long r;
    if (j < k) {
      r = inv[t * k + j];
      if (r < 0 || r >= R) {
        if (L.sub == 0) set_status(status, STATUS_BAD_INDEX);
        continue;
      }
    } else {
      if (!has_shared) break;
      r = R + static_cast<long long>(t);
    }
    *reinterpret_cast<uint4*>(xg + r * H + col) = c;
    if (L.sub == 0) xsg[r * nblk + L.b] = scale;
  }
}

// a5.  Row r of y13 holds [gate(I) | up(I)] in bf16; h = silu(gate) * up in fp32.
template <typename Idx>
__global__ void __launch_bounds__(256) k_swiglu_quant(const uint16_t* __restrict__ y13,
                                                      int rows, int I,
                                                      uint8_t* __restrict__ hq,
                                                      uint8_t* __restrict__ hs) {
  pdl_wait();
  pdl_trigger();
  const int nblk = I / 128;
  const BlockLane<Idx> L(rows, nblk);
  float h[16];
  if (L.live) {
    const uint16_t* g_at = y13 + static_cast<size_t>(L.r) * (2 * static_cast<size_t>(I)) +
                           L.b * 128 + L.sub * 16;
    float g[16], u[16];
    load_bf16x16(g_at, g);
    load_bf16x16(g_at + I, u);
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = 0.f;
  }
  int e;
  const uint4 c = quant16(h, e);
  if (!L.live) return;
  *reinterpret_cast<uint4*>(hq + static_cast<size_t>(L.r) * I + L.b * 128 + L.sub * 16) = c;
  if (L.sub == 0) hs[static_cast<size_t>(L.r) * nblk + L.b] = static_cast<uint8_t>(e + 127);
}

// Packed-row gather: row r of the packed activations is token tok(r)'s row.
// tok(r) = perm_src[r] / k for routed rows, r - R for shared rows.  One warp per row.
__global__ void __launch_bounds__(256) k_gather_rows(const uint8_t* __restrict__ xq,
                                                     const uint8_t* __restrict__ xs,
                                                     const int32_t* __restrict__ perm_src,
                                                     int T, int k, int R, int Rs, int H,
                                                     uint8_t* __restrict__ xg,
                                                     uint8_t* __restrict__ xsg,
                                                     uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= Rs) return;
  int tok = r < R ? perm_src[r] / k : static_cast<int>(r - R);
  if (tok < 0 || tok >= T) {
    if (lane == 0) set_status(status, STATUS_BAD_INDEX);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<long long>(tok) * H);
  uint4* dst = reinterpret_cast<uint4*>(xg + r * H);
  for (int i = lane; i < H / 16; i += 32) dst[i] = src[i];
  const int ns = H / 128;
  for (int i = lane; i < ns; i += 32) xsg[r * ns + i] = xs[static_cast<long long>(tok) * ns + i];
}

// a7.  CTA (token t, 1024-column chunk); each thread owns 8 consecutive columns.
// fp32 sum in j order, shared row last, one rounding to bf16.
__global__ void __launch_bounds__(128) k_combine(const uint16_t* __restrict__ y2,
                                                 const int32_t* __restrict__ inv,
                                                 const float* __restrict__ w, int T, int k,
                                                 int H, int has_shared, int R, int Rs,
                                                 uint16_t* __restrict__ out,
                                                 uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  __shared__ int32_t s_row[16];
  __shared__ float s_w[16];
  if (threadIdx.x < k) {
    int32_t r = inv[static_cast<long long>(t) * k + threadIdx.x];
    if (r < 0 || r >= Rs) {
      set_status(status, STATUS_BAD_INDEX);
      r = -1;
    }
    s_row[threadIdx.x] = r;
    s_w[threadIdx.x] = w[static_cast<long long>(t) * k + threadIdx.x];
  }
  __syncthreads();
  const int c = blockIdx.y * (blockDim.x * 8) + threadIdx.x * 8;
  if (c < H) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    // issue the loads of up to 8 routed rows before consuming any
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int32_t r = j0 + jj < k ? s_row[j0 + jj] : -1;
        v[jj] = r >= 0 ? *reinterpret_cast<const uint4*>(y2 + static_cast<long long>(r) * H + c)
                       : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (j0 + jj >= k || s_row[j0 + jj] < 0) continue;
        const float wj = s_w[j0 + jj];
        float f[8];
        bf16x8_to_f32(v[jj], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
      }
    }
    if (has_shared) {
      float f[8];
      bf16x8_to_f32(
          *reinterpret_cast<const uint4*>(y2 + static_cast<long long>(R + t) * H + c), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      o[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    *reinterpret_cast<uint4*>(out + static_cast<long long>(t) * H + c) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// a3 for the NVFP4 path: quantise each token once (codes and scales to xq / xs when
// given) and write the exact bf16 values of its codes (code x 2^e) straight into its
// k routed rows and its shared row of the packed bf16 activations xe.
template <typename Idx>
__global__ void __launch_bounds__(256) k_quant_scatter_bf16(const uint16_t* __restrict__ x,
                                                            int T, int H, int k, int has_shared,
                                                            const int32_t* __restrict__ inv,
                                                            uint8_t* __restrict__ xq,
                                                            uint8_t* __restrict__ xs,
                                                            uint16_t* __restrict__ xe,
                                                            uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int nblk = H / 128;
  const BlockLane<Idx> L(T, nblk);
  float f[16];
  if (L.live) {
    load_bf16x16(x + static_cast<size_t>(L.r) * H + L.b * 128 + L.sub * 16, f);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = 0.f;
  }
  int e;
  const uint4 c = quant16(f, e);
  if (!L.live) return;
  const size_t t = static_cast<size_t>(L.r);
  const int col = static_cast<int>(L.b) * 128 + L.sub * 16;
  if (xq) *reinterpret_cast<uint4*>(xq + t * H + col) = c;
  if (xs && L.sub == 0) xs[t * nblk + L.b] = static_cast<uint8_t>(e + 127);
  uint4 lo, hi;
  fp8x16_expand(c, e, lo, hi);
  const long long R = static_cast<long long>(T) * k;
  for (int j = 0; j <= k; ++j) {
    long long r;
    if (j < k) {
      r = inv[t * k + j];
      if (r < 0 || r >= R) {
        if (L.sub == 0) set_status(status, STATUS_BAD_INDEX);
        continue;
      }
    } else {
      if (!has_shared) break;
      r = R + static_cast<long long>(t);
    }
    uint4* dst = reinterpret_cast<uint4*>(xe + r * H + col);
    dst[0] = lo;
    dst[1] = hi;
  }
}

// a5 for the NVFP4 path: as k_swiglu_quant (codes and scales to hq / hs when given),
// plus the exact bf16 values of the codes in he, W2's operand.
template <typename Idx>
__global__ void __launch_bounds__(256) k_swiglu_quant_bf16(const uint16_t* __restrict__ y13,
                                                           int rows, int I,
                                                           uint8_t* __restrict__ hq,
                                                           uint8_t* __restrict__ hs,
                                                           uint16_t* __restrict__ he) {
  pdl_wait();
  pdl_trigger();
  const int nblk = I / 128;
  const BlockLane<Idx> L(rows, nblk);
  float h[16];
  if (L.live) {
    const uint16_t* g_at = y13 + static_cast<size_t>(L.r) * (2 * static_cast<size_t>(I)) +
                           L.b * 128 + L.sub * 16;
    float g[16], u[16];
    load_bf16x16(g_at, g);
    load_bf16x16(g_at + I, u);
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = 0.f;
  }
  int e;
  const uint4 c = quant16(h, e);
  if (!L.live) return;
  const size_t off = static_cast<size_t>(L.r) * I + L.b * 128 + L.sub * 16;
  if (hq) *reinterpret_cast<uint4*>(hq + off) = c;
  if (hs && L.sub == 0) hs[static_cast<size_t>(L.r) * nblk + L.b] = static_cast<uint8_t>(e + 127);
  uint4 lo, hi;
  fp8x16_expand(c, e, lo, hi);
  uint4* dst = reinterpret_cast<uint4*>(he + off);
  dst[0] = lo;
  dst[1] = hi;
}

// FP8 rows -> bf16 rows of their exact values.  Thread -> (row, 16-column chunk); row r
// reads row tok(r) of xq (perm_src[r] / k for r < R, r - R above) or row r itself.
__global__ void __launch_bounds__(256) k_expand_rows(const uint8_t* __restrict__ xq,
                                                     const uint8_t* __restrict__ xs,
                                                     const int32_t* __restrict__ perm_src,
                                                     int T, int k, int R, int rows, int K,
                                                     uint16_t* __restrict__ xe,
                                                     uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int chunks = K / 16;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<long long>(rows) * chunks) return;
  const long long r = gid / chunks;
  const int c = static_cast<int>(gid - r * chunks);
  long long src = r;
  if (perm_src) {
    src = r < R ? perm_src[r] / k : r - R;
    if (src < 0 || src >= T) {
      if (c == 0) set_status(status, STATUS_BAD_INDEX);
      return;
    }
  }
  const uint4 code = *reinterpret_cast<const uint4*>(xq + src * K + c * 16);
  const int e = static_cast<int>(xs[src * (K / 128) + c / 8]) - 127;
  uint4 lo, hi;
  fp8x16_expand(code, e, lo, hi);
  uint4* dst = reinterpret_cast<uint4*>(xe + r * K + c * 16);
  dst[0] = lo;
  dst[1] = hi;
}

// ---------------------------------------------------------------- launchers -------

// Eight threads per 128-column block, 256 threads per CTA; the 32-bit-index kernel
// runs whenever every thread index fits in 32 bits.
template <typename... KArgs, typename... Args>
static cudaError_t launch_blocks(void (*k32)(KArgs...), void (*k64)(KArgs...),
                                 long long nblocks128, cudaStream_t st, Args... args) {
  if (nblocks128 == 0) return cudaSuccess;
  const long long grid = (nblocks128 + 31) / 32;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  return launch_k(grid * 256 <= 0xFFFFFFFFLL ? k32 : k64, static_cast<unsigned>(grid), 256, 0,
                  st, args...);
}

cudaError_t launch_quant_act(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* s,
                             cudaStream_t st) {
  return launch_blocks(k_quant_act<uint32_t>, k_quant_act<unsigned long long>,
                       static_cast<long long>(rows) * (cols / 128), st, x, rows, cols, q, s);
}

cudaError_t launch_quant_scatter(const uint16_t* x, int T, int H, int k, int has_shared,
                                 const int32_t* inv, uint8_t* xq, uint8_t* xs, uint8_t* xg,
                                 uint8_t* xsg, int32_t* cnt, uint32_t* status, cudaStream_t st) {
  return launch_blocks(k_quant_scatter<uint32_t>, k_quant_scatter<unsigned long long>,
                       static_cast<long long>(T) * (H / 128), st, x, T, H, k, has_shared, inv, xq,
                       xs, xg, xsg, cnt, status);
}

cudaError_t launch_quant_scatter_bf16(const uint16_t* x, int T, int H, int k, int has_shared,
                                      const int32_t* inv, uint8_t* xq, uint8_t* xs,
                                      uint16_t* xe, uint32_t* status, cudaStream_t st) {
  return launch_blocks(k_quant_scatter_bf16<uint32_t>, k_quant_scatter_bf16<unsigned long long>,
                       static_cast<long long>(T) * (H / 128), st, x, T, H, k, has_shared, inv,
                       xq, xs, xe, status);
}

cudaError_t launch_swiglu_quant_bf16(const uint16_t* y13, int rows, int I, uint8_t* hq,
                                     uint8_t* hs, uint16_t* he, cudaStream_t st) {
  return launch_blocks(k_swiglu_quant_bf16<uint32_t>, k_swiglu_quant_bf16<unsigned long long>,
                       static_cast<long long>(rows) * (I / 128), st, y13, rows, I, hq, hs, he);
}

cudaError_t launch_expand_rows(const uint8_t* xq, const uint8_t* xs, const int32_t* perm_src,
                               int T, int k, int R, int rows, int K, uint16_t* xe,
                               uint32_t* status, cudaStream_t st) {
  const long long n = static_cast<long long>(rows) * (K / 16);
  if (n == 0) return cudaSuccess;
  const long long grid = (n + 255) / 256;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  return launch_k(k_expand_rows, static_cast<unsigned>(grid), 256, 0, st, xq, xs, perm_src, T, k,
                  R, rows, K, xe, status);
}

cudaError_t launch_swiglu_quant(const uint16_t* y13, int rows, int I, uint8_t* hq, uint8_t* hs,
                                cudaStream_t st) {
  return launch_blocks(k_swiglu_quant<uint32_t>, k_swiglu_quant<unsigned long long>,
                       static_cast<long long>(rows) * (I / 128), st, y13, rows, I, hq, hs);
}

cudaError_t launch_gather_rows(const uint8_t* xq, const uint8_t* xs, const int32_t* perm_src,
                               int T, int k, int R, int Rs, int H, uint8_t* xg, uint8_t* xsg,
                               uint32_t* status, cudaStream_t st) {
  if (Rs == 0) return cudaSuccess;
  unsigned grid = static_cast<unsigned>((static_cast<long long>(Rs) + 7) / 8);
  return launch_k(k_gather_rows, grid, 256, 0, st, xq, xs, perm_src, T, k, R, Rs, H, xg, xsg,
                  status);
}

cudaError_t launch_combine(const uint16_t* y2, const int32_t* inv, const float* w, int T, int k,
                           int H, int has_shared, uint16_t* out, uint32_t* status,
                           cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int R = T * k, Rs = R + (has_shared ? T : 0);
  const int threads = 128;
  dim3 grid(T, (H + threads * 8 - 1) / (threads * 8));
  return launch_k(k_combine, grid, threads, 0, st, y2, inv, w, T, k, H, has_shared, R, Rs, out,
                  status);
}

}  // namespace moe
