// a4 / a6: grouped GEMM with MXFP4 expert weights and FP8 activations on the
// tcgen05 tensor cores (block-scaled MMA, kind::mxf8f6f4, one E8M0 scale per 32 K).
//
// Pages: "Pushing the Limits of Serving DeepSeek-V4-Pro" (LMSYS, H20), §2.2 (MXFP4
// expert weights x online FP8 activations) and §3.3 (W13 and W2 as separate grouped
// GEMMs whose shapes come from the routing histogram, tuned per effective M); GB10
// "Optimization progress report", Optimization 06 (a small-M path for a handful of
// tokens, no padding to large row tiles).
//
// Design (GB300-first, not a port of the Hopper/GB10 kernels the pages describe):
//   * Swap-AB: the MMA's M=128 side is a tile of 128 weight rows (output features),
//     its N side is the group's tokens, padded only to the next multiple of 16.  A
//     decode group with 1-2 tokens costs one N=16 MMA per K step while the weights
//     stream from HBM at full rate.
//   * Weights are loaded by TMA straight from the packed MXFP4 layout into the
//     16-byte-aligned FP4 shared-memory layout the MMA reads (16 codes in 8 bytes
//     followed by an 8-byte gap), 128B-swizzled, so HBM traffic stays at 0.5 byte per
//     weight.  Tokens' FP8 rows are loaded by TMA from the packed activations.
//   * Scale factors (weights: 4 per row per 128-K stage; activations: one per row per
//     128-K stage, replicated over the four 32-blocks) are rearranged by one warp
//     into the 128-row scale-factor atom and copied to TMEM with tcgen05.cp.
//   * Warp-specialised, persistent CTAs: warp 0 issues TMA, warp 1 issues MMAs, warp
//     2 stages scale factors, warps 4-7 drain the double-buffered TMEM accumulator
//     (fp32 -> bf16) while the next tile's MMAs run.
//   * Every wait is bounded; an expired wait sets a status bit and the CTA unwinds.
#include <mutex>

#include "kernels.cuh"

namespace moe {

struct GemmParams {
  const uint8_t* w_scales;    // [G][N][K/32]
  const uint8_t* x_scales;    // [rows_total][K/128]
  const int4* items;          // {group, row0, rows, 0}
  const int32_t* item_count;  // device
  int max_items;
  uint16_t* y;                // [rows_total][N]
  int N, K, G, rows_total;
  uint32_t a_tx_bytes;        // transaction bytes of one weight-tile TMA load (packed size)
  uint32_t* status;
};

template <int BN_MAX, int STAGES>
struct GemmCfg {
  static constexpr int kABytes = 128 * 128;       // 128 rows x 128 FP4 (16B-aligned form)
  static constexpr int kBBytes = BN_MAX * 128;    // BN_MAX rows x 128 FP8
  static constexpr int kSfBytes = 512;            // one 128-row scale atom
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffSfa = kOffB + STAGES * kBBytes;
  static constexpr int kOffSfb = kOffSfa + STAGES * kSfBytes;
  static constexpr int kOffBar = kOffSfb + STAGES * kSfBytes;
  static constexpr int kNumBars = 2 * STAGES + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr int kTmemNeed = 2 * BN_MAX + 8 * STAGES;
  static constexpr int kTmemCols =
      kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
  static_assert(BN_MAX % 16 == 0 && BN_MAX <= 128, "token tile");
  static_assert(kTmemNeed <= 512, "TMEM");
};

// Instruction descriptor, kind::mxf8f6f4 block-scaled: A = E2M1 (5), B = E4M3 (0),
// both K-major, scale type E8M0, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_mxf4_e4m3(int n) {
  uint32_t d = 0;
  d |= 5u << 7;                               // A format: E2M1
  d |= 0u << 10;                              // B format: E4M3
  d |= static_cast<uint32_t>(n >> 3) << 17;   // N >> 3
  d |= 1u << 23;                              // scale factor type: E8M0
  d |= static_cast<uint32_t>(128 >> 4) << 24; // M >> 4
  return d;
}

template <int BN_MAX, int STAGES>
__global__ void __launch_bounds__(256, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const GemmParams p) {
  using C = GemmCfg<BN_MAX, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = bars + 2 * STAGES + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);   // TMA arrive(+tx) and the scale-factor warp
      mbar_init(&empty[s], 1);  // tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // four epilogue warps
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles = p.N / 128;
  const int nk = p.K / 128;
  int count = *p.item_count;
  if (count > p.max_items) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    count = p.max_items;
  }
  const long long total = static_cast<long long>(count) * n_tiles;

  // Reads and validates one work item; every role sees the same result.
  auto load_item = [&](long long L, int& g, int& row0, int& rows, int& nt) -> bool {
    int4 it = p.items[L / n_tiles];
    nt = static_cast<int>(L % n_tiles);
    g = it.x;
    row0 = it.y;
    rows = it.z;
    if (rows <= 0) return false;
    if (g < 0 || g >= p.G || row0 < 0 || rows > BN_MAX || row0 + rows > p.rows_total) {
      if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
      return false;
    }
    return true;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
        int g, row0, rows, nt;
        if (!load_item(L, g, row0, rows, nt)) continue;
        const int bn = (rows + 15) & ~15;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1u, p.status, abort_flag)) break;
          mbar_arrive_expect_tx(&full[s], p.a_tx_bytes + bn * 128);
          tma_load_3d(smem + C::kOffA + s * C::kABytes, &tmW, &full[s], kb * 128, nt * 128, g);
          for (int i = 0; i < bn; i += 16)
            tma_load_2d(smem + C::kOffB + s * C::kBBytes + i * 128, &tmX, &full[s], kb * 128,
                        row0 + i);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
        int g, row0, rows, nt;
        if (!load_item(L, g, row0, rows, nt)) continue;
        const int bn = (rows + 15) & ~15;
        const uint32_t b = tc & 1u, use = tc >> 1;
        if (tc >= 2 && !mbar_wait(&acc_empty[b], (use - 1) & 1u, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * BN_MAX;
        const uint32_t idesc = idesc_mxf4_e4m3(bn);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + 2 * BN_MAX + s * 8;
          const uint32_t sfb_t = sfa_t + 4;
          tc_cp_32x128b_x4(sfa_t, smem_desc(smem_u32(smem + C::kOffSfa + s * C::kSfBytes), 0,
                                            128, kLayoutNone));
          tc_cp_32x128b_x4(sfb_t, smem_desc(smem_u32(smem + C::kOffSfb + s * C::kSfBytes), 0,
                                            128, kLayoutNone));
          const uint32_t a0 = smem_u32(smem + C::kOffA + s * C::kABytes);
          const uint32_t b0 = smem_u32(smem + C::kOffB + s * C::kBBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(a0 + kk * 32, 0, 1024, kLayoutSw128);
            const uint64_t bd = smem_desc(b0 + kk * 32, 0, 1024, kLayoutSw128);
            const uint32_t id = idesc | (static_cast<uint32_t>(kk) << 29) |
                                (static_cast<uint32_t>(kk) << 4);
            mma_mxf8f6f4(d_tmem, ad, bd, id, sfa_t, sfb_t, (kb | kk) != 0);
          }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&acc_full[b]);
        ++tc;
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- scale factors
    uint32_t it = 0;
    const int kw = p.K / 32, kx = p.K / 128;
    for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
      int g, row0, rows, nt;
      if (!load_item(L, g, row0, rows, nt)) continue;
      const uint8_t* ws = p.w_scales + (static_cast<size_t>(g) * p.N + nt * 128) * kw;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        if (it >= STAGES) {
          int w_ok = 1;
          if (lane == 0) w_ok = mbar_wait(&empty[s], ph ^ 1u, p.status, abort_flag);
          if (!__shfl_sync(0xFFFFFFFFu, w_ok, 0)) {
            ok = false;
            break;
          }
        }
        uint32_t va[4], vb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = j * 32 + lane;
          va[j] = __ldg(reinterpret_cast<const uint32_t*>(ws + static_cast<size_t>(r) * kw + kb * 4));
          uint32_t sb = 127u;
          if (r < rows) sb = __ldg(p.x_scales + static_cast<size_t>(row0 + r) * kx + kb);
          vb[j] = sb * 0x01010101u;
        }
        *reinterpret_cast<uint4*>(smem + C::kOffSfa + s * C::kSfBytes + lane * 16) =
            make_uint4(va[0], va[1], va[2], va[3]);
        *reinterpret_cast<uint4*>(smem + C::kOffSfb + s * C::kSfBytes + lane * 16) =
            make_uint4(vb[0], vb[1], vb[2], vb[3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
      if (!ok) break;
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp - 4;
    uint32_t tc = 0;
    for (long long L = blockIdx.x; L < total && !*abort_flag; L += gridDim.x) {
      int g, row0, rows, nt;
      if (!load_item(L, g, row0, rows, nt)) continue;
      const uint32_t b = tc & 1u, use = tc >> 1;
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, w_ok, 0)) break;
      tc_fence_after();
      const int n = nt * 128 + q * 32 + lane;
      uint16_t* ycol = p.y + static_cast<size_t>(row0) * p.N + n;
      for (int c0 = 0; c0 < rows; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN_MAX + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (c0 + i < rows) {
            __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(r[i]));
            ycol[static_cast<size_t>(c0 + i) * p.N] = *reinterpret_cast<uint16_t*>(&h);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++tc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side -------

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &ptr, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct DevInfo {
  int sms = 0;
};

DevInfo& dev_info() {
  static DevInfo info[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (info[dev].sms == 0) cudaDeviceGetAttribute(&info[dev].sms, cudaDevAttrMultiProcessorCount, dev);
  return info[dev];
}

template <int BN_MAX, int STAGES>
cudaError_t launch_one(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p,
                       int max_items, cudaStream_t st) {
  using C = GemmCfg<BN_MAX, STAGES>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_mx<BN_MAX, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long tiles = static_cast<long long>(max_items) * (p.N / 128);
  if (tiles == 0) return cudaSuccess;
  const int sms = dev_info().sms;
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  GemmParams q = p;
  q.max_items = max_items;
  k_gemm_mx<BN_MAX, STAGES><<<grid, 256, C::kSmemBytes, st>>>(tmW, tmX, q);
  return cudaGetLastError();
}

}  // namespace

int gemm_encode_maps(const uint8_t* w_codes, int G, int N, int K, const uint8_t* act,
                     int rows_total, CUtensorMap* tmW, CUtensorMap* tmX) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return MOE_ERR_CUDA;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K / 2),
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(w_codes), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K),
                          static_cast<cuuint64_t>(rows_total > 0 ? rows_total : 1)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t es[2] = {1, 1};
    if (enc(tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(act), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}


cudaError_t launch_grouped_gemm(const GemmLaunch& a, cudaStream_t st) {
  CUtensorMap tmW, tmX;
  int rc = gemm_encode_maps(a.w_codes, a.G, a.N, a.K, a.act, a.rows_total, &tmW, &tmX);
  if (rc != MOE_OK) return cudaErrorInvalidValue;
  GemmParams p{};
  p.w_scales = a.w_scales;
  p.x_scales = a.act_scales;
  p.y = a.y;
  p.N = a.N;
  p.K = a.K;
  p.G = a.G;
  p.rows_total = a.rows_total;
  p.a_tx_bytes = kWeightTileTxBytes;
  p.status = a.status;
  // small-M list
  p.items = a.small_items;
  p.item_count = a.item_counts;
  cudaError_t e = launch_one<kSmallBN, kSmallStages>(tmW, tmX, p, a.max_small, st);
  if (e != cudaSuccess) return e;
  p.items = a.large_items;
  p.item_count = a.item_counts + 1;
  return launch_one<kLargeBN, kLargeStages>(tmW, tmX, p, a.max_large, st);
}

}  // namespace moe
