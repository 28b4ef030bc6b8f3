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

// Quantise 8 values held by one lane of a 16-lane group that covers a 128-column
// block.  Returns the 8 codes packed little-endian; writes the scale byte via lane 0
// of the group.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], uint8_t* scale_out, int sublane) {
  // every lane of the 16-lane group gets the same scale; lane `sublane == 0` stores it
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int off = 8; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const int e = fp8_scale_exponent(amax);
  const float s = pow2_neg(e);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e4m3x2(f[2 * i] * s, f[2 * i + 1] * s);
  if (sublane == 0) *scale_out = static_cast<uint8_t>(e + 127);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

}  // namespace

// a3.  One warp per two 128-column blocks; 16 lanes x 8 values per block.
__global__ void __launch_bounds__(256) k_quant_act(const uint16_t* __restrict__ x, int rows,
                                                   int cols, uint8_t* __restrict__ q,
                                                   uint8_t* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int nblk = cols / 128;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
  const long long blk = gw * 2 + half;  // global 128-block id
  const long long total = static_cast<long long>(rows) * nblk;
  const bool live = blk < total;
  const long long r = live ? blk / nblk : 0, b = live ? blk % nblk : 0;
  float f[8];
  if (live) {
    uint4 u = *reinterpret_cast<const uint4*>(x + r * cols + b * 128 + sub * 8);
    bf16x8_to_f32(u, f);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = 0.f;
  }
  uint8_t dummy;
  uint2 c = quant8(f, live ? s + r * nblk + b : &dummy, sub);
  if (live) *reinterpret_cast<uint2*>(q + r * cols + b * 128 + sub * 8) = c;
}

// a3 fused with the packed-row gather: token t's codes and scales go to xq / xs
// (when given) and straight to its k routed rows inv[t*k + j] and its shared row R + t
// of the packed activations, so no separate gather pass re-reads them.
__global__ void __launch_bounds__(256) k_quant_scatter(const uint16_t* __restrict__ x, int T,
                                                       int H, int k, int has_shared,
                                                       const int32_t* __restrict__ inv,
                                                       uint8_t* __restrict__ xq,
                                                       uint8_t* __restrict__ xs,
                                                       uint8_t* __restrict__ xg,
                                                       uint8_t* __restrict__ xsg,
                                                       uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int nblk = H / 128;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
  const long long blk = gw * 2 + half;
  const long long total = static_cast<long long>(T) * nblk;
  const bool live = blk < total;
  const long long t = live ? blk / nblk : 0, b = live ? blk % nblk : 0;
  float f[8];
  if (live) {
    uint4 u = *reinterpret_cast<const uint4*>(x + t * H + b * 128 + sub * 8);
    bf16x8_to_f32(u, f);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = 0.f;
  }
  uint8_t scale;
  uint2 c = quant8(f, &scale, 0);
  if (!live) return;
  const long long R = static_cast<long long>(T) * k;
  if (xq) *reinterpret_cast<uint2*>(xq + t * H + b * 128 + sub * 8) = c;
  if (xs && sub == 0) xs[t * nblk + b] = scale;
  for (int j = 0; j <= k; ++j) {
    long long r;
    if (j < k) {
      r = inv[t * k + j];
      if (r < 0 || r >= R) {
        if (sub == 0) set_status(status, STATUS_BAD_INDEX);
        continue;
      }
    } else {
      if (!has_shared) break;
      r = R + t;
    }
    *reinterpret_cast<uint2*>(xg + r * H + b * 128 + sub * 8) = c;
    if (sub == 0) xsg[r * nblk + b] = scale;
  }
}

// a5.  Row r of y13 holds [gate(I) | up(I)] in bf16; h = silu(gate) * up in fp32.
__global__ void __launch_bounds__(256) k_swiglu_quant(const uint16_t* __restrict__ y13,
                                                      int rows, int I,
                                                      uint8_t* __restrict__ hq,
                                                      uint8_t* __restrict__ hs) {
  pdl_wait();
  pdl_trigger();
  const int nblk = I / 128;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
  const long long blk = gw * 2 + half;
  const long long total = static_cast<long long>(rows) * nblk;
  const bool live = blk < total;
  const long long r = live ? blk / nblk : 0, b = live ? blk % nblk : 0;
  float h[8];
  if (live) {
    const uint16_t* row = y13 + r * (2LL * I);
    uint4 ug = *reinterpret_cast<const uint4*>(row + b * 128 + sub * 8);
    uint4 uu = *reinterpret_cast<const uint4*>(row + I + b * 128 + sub * 8);
    float g[8], u[8];
    bf16x8_to_f32(ug, g);
    bf16x8_to_f32(uu, u);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = 0.f;
  }
  uint8_t dummy;
  uint2 c = quant8(h, live ? hs + r * nblk + b : &dummy, sub);
  if (live) *reinterpret_cast<uint2*>(hq + r * I + b * 128 + sub * 8) = c;
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

// ---------------------------------------------------------------- launchers -------

static unsigned grid_for_blocks(long long nblocks128) {
  // two 128-column blocks per warp, 8 warps per CTA
  long long warps = (nblocks128 + 1) / 2;
  return static_cast<unsigned>((warps + 7) / 8);
}

cudaError_t launch_quant_act(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* s,
                             cudaStream_t st) {
  long long nb = static_cast<long long>(rows) * (cols / 128);
  if (nb == 0) return cudaSuccess;
  return launch_k(k_quant_act, grid_for_blocks(nb), 256, 0, st, x, rows, cols, q, s);
}

cudaError_t launch_quant_scatter(const uint16_t* x, int T, int H, int k, int has_shared,
                                 const int32_t* inv, uint8_t* xq, uint8_t* xs, uint8_t* xg,
                                 uint8_t* xsg, uint32_t* status, cudaStream_t st) {
  long long nb = static_cast<long long>(T) * (H / 128);
  if (nb == 0) return cudaSuccess;
  return launch_k(k_quant_scatter, grid_for_blocks(nb), 256, 0, st, x, T, H, k, has_shared, inv,
                  xq, xs, xg, xsg, status);
}

cudaError_t launch_swiglu_quant(const uint16_t* y13, int rows, int I, uint8_t* hq, uint8_t* hs,
                                cudaStream_t st) {
  long long nb = static_cast<long long>(rows) * (I / 128);
  if (nb == 0) return cudaSuccess;
  return launch_k(k_swiglu_quant, grid_for_blocks(nb), 256, 0, st, y13, rows, I, hq, hs);
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
