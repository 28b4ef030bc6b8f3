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
//   * Warp-specialised, persistent CTAs: warp 0 issues TMA (the weight tiles; in the
//     large variant warp 3 issues the token tiles), warp 1 issues MMAs, warp 2 stages
//     scale factors (own barrier, so their TMEM copies issue before the tiles land),
//     warps 4-7 drain the double-buffered TMEM accumulator (fp32 -> bf16) while the
//     next tile's MMAs run.
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
  uint32_t* status;
  int early;  // the plan may be read, and weights loaded, before griddepcontrol.wait
  // f2 (W2 only; null out = off): the epilogue also performs a7.  After a tile's y2
  // rows are stored, each row bumps its (token, 128-column block) arrival counter; the
  // tile that completes a block (k + has_shared arrivals) sums that token's rows for
  // the block's 128 columns exactly as k_combine does and writes out.
  uint16_t* out;            // [T][N] bf16
  const int32_t* perm_src;  // [R] packed row -> routed row t*k+j
  const int32_t* inv;       // [R] routed row -> packed row
  const float* cw;          // [T][k] routing weights
  int32_t* cnt;             // [T][N/128] arrival counters, zero before the launch
  int T, k, has_shared;
  // f1 (W13 on SM pairs only; null hq = off): the epilogue performs a5 -- h = silu(gate)
  // * up from the bf16-rounded accumulators, quantised per row per 128 features -- and
  // writes W2's operand hq [rows_total][N/2] and scales hs [rows_total][N/256] instead
  // of y13.
  uint8_t* hq;
  uint8_t* hs;
};

// Quads (4 sub-tiles = 512 K elements) of scale bytes the scale-factor warp keeps in
// flight ahead of the stage it is staging.
constexpr int kSfQuads = 4;

// Shared-memory layout of one pipeline configuration.  A stage holds KO sub-tiles of
// 128 K elements: weights [KO][128 rows][128 B] (FP4 in its 16-byte-aligned form),
// tokens [KO][BN_MAX rows][128 B] (FP8), KO weight scale atoms and one token scale
// atoms (512 B each).  Each stage is one weight TMA (box 128 x 128 x KO) and one
// token TMA (box 128 x BN_MAX x KO; rows past the chunk are loaded and ignored).
template <int BN_MAX, int STAGES, int KO, int OCC>
struct GemmCfg {
  static constexpr int kASub = 128 * 128;
  static constexpr int kBSub = BN_MAX * 128;
  static constexpr int kABytes = KO * kASub;
  static constexpr int kBBytes = KO * kBSub;
  static constexpr int kSfBytes = 512;
  static constexpr int kSfbAtoms = (BN_MAX + 127) / 128;  // token scale atoms per stage
  // Wide scale staging (the 1-CTA-per-SM large variant): each 32-row atom is written
  // four times (rows r, r+32, r+64, r+96) so that one tcgen05.cp.128x{128,256}b per
  // operand moves every sub-tile's / token block's scales of a stage -- the same TMEM
  // contents as one 32x128b.warpx4 copy per atom, with fewer instructions to issue.
  static constexpr bool kWideSf = OCC == 1;
  static constexpr int kSfaStage = kWideSf ? KO * 2048 : KO * kSfBytes;
  static constexpr int kSfbStage = kWideSf ? kSfbAtoms * 2048 : kSfbAtoms * kSfBytes;
  // Wide staging goes first, so reads through its (larger-stride) copy descriptors can
  // only reach the tiles that follow, never past the CTA's shared memory; otherwise the
  // 1024-byte-aligned tiles go first and the scale atoms after them.
  static constexpr int kSfTotal = STAGES * (kSfaStage + kSfbStage);
  static constexpr int kOffSfa = kWideSf ? 0 : STAGES * (kABytes + kBBytes);
  static constexpr int kOffSfb = kOffSfa + STAGES * kSfaStage;
  static constexpr int kOffA = kWideSf ? (kSfTotal + 1023) / 1024 * 1024 : 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffBar = kWideSf ? kOffB + STAGES * kBBytes : kOffSfa + kSfTotal;
  // Large variant: token tiles (up to 56 KB a stage) get their own TMA thread, and the
  // scale factors their own barrier, so the MMA thread issues the scale copies while
  // the tiles are still landing (measured: -0.5 ms on the 32K-token layer; the
  // small and medium variants measured no better and keep one barrier per stage).
  static constexpr bool kTokenThread = BN_MAX > 64;
  static constexpr bool kSfFirst = BN_MAX > 64;
  // Small variant: two MMA-issuing threads (warps 1 and 3) take the even and odd K
  // stages of a tile into two accumulators that the epilogue adds, so a stage waits
  // for half as much MMA issue before its shared memory is released.  (The medium
  // variant's second accumulators would not fit two CTAs' TMEM.)
  static constexpr int kIssuers = BN_MAX <= 16 ? 2 : 1;
  static constexpr int kAccCols = kIssuers * BN_MAX;  // one accumulator buffer
  // full[issuer][stage] (each issuer waits only on its own, so it sees every phase of
  // every barrier it waits on), empty[stage], acc_full[2], acc_empty[2], sf_full[stage],
  // drain[issuer] (the abort path's wait for MMAs already issued)
  static constexpr int kNumBars = (kIssuers + 2) * STAGES + 4 + kIssuers;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // f2's list of the tokens a tile completed: [count, tokens...]
  static constexpr int kOffFc = kOffMisc + 16;
  static constexpr int kSmemBytes = kOffFc + 4 * (BN_MAX + 1);
  static constexpr int kSfCols = 4 * (KO + kSfbAtoms);      // TMEM columns per stage
  static constexpr int kTmemNeed = 2 * kAccCols + STAGES * kSfCols;
  static constexpr int kTmemCols =
      kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
  static_assert(BN_MAX % 16 == 0 && BN_MAX <= 256, "token tile");
  static_assert(KO == 1 || KO == 2 || KO == 4, "sub-tiles per stage");
  static_assert(!kWideSf || (KO <= 2 && kSfbAtoms <= 2), "wide scale copies move <= 256 bits");
  static_assert(kTmemNeed <= 512, "TMEM");
  static_assert(kTmemCols * OCC <= 512, "co-resident CTAs must fit TMEM together");
  static_assert(OCC == 1 || OCC * (kSmemBytes + 1024) <= 233472,
                "co-resident CTAs must fit shared memory together");
  static_assert(!(kTokenThread && kIssuers > 1), "warp 3 has one role");
  static_assert(kSmemBytes <= 232448, "dynamic shared memory of one CTA");
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

__device__ __forceinline__ void epilogue_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");  // warps 4-7 only
}

// f2: the combine for the tokens whose (token, block nt) this tile completed.  et: the
// epilogue thread (0..127); U: tokens per thread per pass.  Called by all 128 epilogue
// threads after their y2 stores of the tile.
template <int U>
__device__ __forceinline__ void fused_combine_tile(const GemmParams& p, int row0, int rows,
                                                   int nt, int et, int* fc) {
  const int R = p.T * p.k;
  const int Rs = R + (p.has_shared ? p.T : 0);
  const int need = p.k + (p.has_shared ? 1 : 0);
  const int nblk = p.N / 128;
  if (et == 0) fc[0] = 0;
  __threadfence();  // release: this thread's y2 stores of the tile, device-wide
  epilogue_bar_sync();
  for (int rl = et; rl < rows; rl += 128) {
    const int r = row0 + rl;
    const int t = r < R ? p.perm_src[r] / p.k : r - R;
    if (t < 0 || t >= p.T) {
      set_status(p.status, STATUS_BAD_INDEX);
      continue;
    }
    if (atomicAdd(&p.cnt[static_cast<size_t>(t) * nblk + nt], 1) == need - 1)
      fc[1 + atomicAdd(&fc[0], 1)] = t;
  }
  epilogue_bar_sync();
  const int nc = fc[0];
  if (nc > 0) __threadfence();  // acquire: the other tiles' rows of the completed tokens
  // 16 threads per token, each 8 columns (one 16-byte load per row); 8 token slots, U
  // tokens per thread per pass, so a pass has up to U x 9 row loads of each thread in
  // flight before any is summed
  const int slot = et >> 4;
  const int col = nt * 128 + (et & 15) * 8;
  for (int i0 = 0; i0 < nc; i0 += 8 * U) {
    int tk[U];
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * 8 + slot;
      tk[u] = i < nc ? fc[1 + i] : -1;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[u][c] = 0.f;
    }
    // k_combine's order: fp32 fma in j order, then the shared row
    for (int j0 = 0; j0 < p.k; j0 += 8) {
      uint4 v[U][8];
      float w[U][8];
      uint32_t okm[U];  // rows loaded (a bad index is skipped, as k_combine does)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        okm[u] = 0u;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          v[u][jj] = make_uint4(0, 0, 0, 0);
          w[u][jj] = 0.f;
          if (tk[u] >= 0 && j < p.k) {
            const size_t tj = static_cast<size_t>(tk[u]) * p.k + j;
            const int r = p.inv[tj];
            if (r >= 0 && r < Rs) {
              v[u][jj] = __ldcg(
                  reinterpret_cast<const uint4*>(p.y + static_cast<size_t>(r) * p.N + col));
              w[u][jj] = p.cw[tj];
              okm[u] |= 1u << jj;
            } else {
              set_status(p.status, STATUS_BAD_INDEX);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (!((okm[u] >> jj) & 1u)) continue;
          const uint32_t q[4] = {v[u][jj].x, v[u][jj].y, v[u][jj].z, v[u][jj].w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t bits = (c & 1) ? (q[c >> 1] & 0xFFFF0000u) : (q[c >> 1] << 16);
            acc[u][c] = fmaf(w[u][jj], __uint_as_float(bits), acc[u][c]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (tk[u] < 0) continue;
      if (p.has_shared) {
        const uint4 sv = __ldcg(reinterpret_cast<const uint4*>(
            p.y + static_cast<size_t>(R + tk[u]) * p.N + col));
        const uint32_t q[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t bits = (c & 1) ? (q[c >> 1] & 0xFFFF0000u) : (q[c >> 1] << 16);
          acc[u][c] += __uint_as_float(bits);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[u][2 * c], acc[u][2 * c + 1]);
        o[c] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(tk[u]) * p.N + col) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  epilogue_bar_sync();  // the list is reused by the next tile
}

__device__ __forceinline__ uint32_t u4_comp(const uint4& v, int t) {
  return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
}

// Tiles of a list of `count` items (n-tiles of 128 rows per item).
__device__ __forceinline__ long long tiles_of(const GemmParams& p, int count) {
  return static_cast<long long>(count < p.max_items ? count : p.max_items) * (p.N / 128);
}

// The walk's stride for `total` tiles: at most gridDim.x, and the fewest CTAs that
// still take ceil(total / gridDim.x) tiles each.
__device__ __forceinline__ int walk_stride(long long total) {
  if (total <= 0) return static_cast<int>(gridDim.x);
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  return static_cast<int>((total + per - 1) / per);
}

template <int BN_MAX, int STAGES, int KO, int OCC, bool F2>
__global__ void __launch_bounds__(256, OCC)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const GemmParams p) {
  using C = GemmCfg<BN_MAX, STAGES, KO, OCC>;
  // An empty work list (the plan found no group for this variant): with the plan
  // complete two launches back, the CTA leaves before setting anything up -- after
  // waiting for the preceding kernel, so that the launches after it stay ordered
  // behind that kernel.
  // Likewise a CTA that the balanced walk leaves without tiles (below).
  if (p.early &&
      (*p.item_count <= 0 ||
       static_cast<int>(blockIdx.x) >= walk_stride(tiles_of(p, *p.item_count)))) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  // The 128B-swizzled tiles need 1024-byte alignment; the dynamic shared memory of a
  // kernel without static shared memory starts at such a boundary.  Checked, not
  // assumed: a misaligned base reports STATUS_BAD_PLAN and the CTA returns.
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;  // [kIssuers][STAGES]: stage kb goes to issuer kb % kIssuers
  uint64_t* empty = full + C::kIssuers * STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* sf_full = acc_empty + 2;
  uint64_t* drain = sf_full + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kIssuers * STAGES; ++s)
      // TMA arrival(s) (+tx), and the scale-factor warp unless it has its own barrier
      mbar_init(&full[s], (C::kTokenThread ? 2 : 1) + (C::kSfFirst ? 0 : 1));
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&empty[s], 1);    // tcgen05.commit
      mbar_init(&sf_full[s], 1);  // the scale-factor warp (kSfFirst)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], C::kIssuers);  // one tcgen05.commit per issuer
      mbar_init(&acc_empty[b], 4);  // four epilogue warps
    }
    for (int i = 0; i < C::kIssuers; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Prologue done.  Wait for the preceding kernel (the producer of the activations,
  // and of the tile plan unless p.early).  With p.early the plan is already complete,
  // so only the roles that read the preceding kernel's output wait: the weight
  // producer after issuing its first stages' weight loads, the token thread and the
  // scale-factor warp; the MMA issuer and the epilogue consume only what those load.
  if (!p.early) pdl_wait();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles = p.N / 128;
  const int nk = p.K / (128 * KO);  // pipeline stages per tile
  int count = *p.item_count;
  if (count > p.max_items) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    count = p.max_items;
  }
  long long total = tiles_of(p, count);
  if (total > 0x7FFFFFFFll) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    total = 0;
  }
  // Balanced waves: the walk's stride is the number of CTAs that gives each the same
  // number of tiles give or take one; the CTAs past it walk nothing.  (With the full
  // grid, a last wave of a few CTAs streams its tiles at those CTAs' own rate, too few
  // loads in flight to keep HBM busy.)
  const int wstride = walk_stride(total);
  const int wstart = static_cast<int>(blockIdx.x);
  if (wstart >= wstride) total = 0;

  // Validates one work item; every role sees the same result.
  auto check_item = [&](const int4 it, int& g, int& row0, int& rows) -> bool {
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
  // Tile L directly (the scale stager's look-ahead): item L / n_tiles, n-tile L % n_tiles.
  auto load_item = [&](long long L, int& g, int& row0, int& rows, int& nt) -> bool {
    const int Li = static_cast<int>(L);  // total < 2^31 (checked above)
    nt = Li % n_tiles;
    return check_item(__ldg(p.items + Li / n_tiles), g, row0, rows);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      // Early start: the weights of the first item's first stages (free ring slots)
      // before the wait, their token tiles after it.
      long long L0 = -1;
      int pre = 0;
      if (p.early) {
        int g, row0, rows, nt;
        for (long long L = blockIdx.x; L < total; L += wstride)
          if (load_item(L, g, row0, rows, nt)) {
            L0 = L;
            break;
          }
        if (L0 >= 0) {
          pre = nk < STAGES ? nk : STAGES;
          for (int kb = 0; kb < pre; ++kb) {  // ring slot kb, first use: no empty wait
            uint64_t* fb = &full[(kb % C::kIssuers) * STAGES + kb];
            mbar_arrive_expect_tx(fb, C::kTokenThread ? KO * kWeightTileTxBytes
                                                      : KO * kWeightTileTxBytes + BN_MAX * KO * 128);
            tma_load_4d(smem + C::kOffA + kb * C::kABytes, &tmW, fb, 0, nt * 128, kb * KO, g);
          }
        }
        pdl_wait();
        if constexpr (!C::kTokenThread) {
          for (int kb = 0; kb < pre; ++kb)
            tma_load_3d(smem + C::kOffB + kb * C::kBBytes, &tmX,
                        &full[(kb % C::kIssuers) * STAGES + kb], 0, row0, kb * KO);
        }
      }
      uint32_t it = 0;
      for (TileWalk tw(p.items, total, n_tiles, wstart, wstride); tw.valid() && !*abort_flag;
           tw.next()) {
        int g, row0, rows;
        const int nt = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          if (tw.L == L0 && kb < pre) continue;  // issued above
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1u, p.status, abort_flag)) break;
          uint64_t* fb = &full[(kb % C::kIssuers) * STAGES + s];
          if constexpr (C::kTokenThread) {
            mbar_arrive_expect_tx(fb, KO * kWeightTileTxBytes);
            tma_load_4d(smem + C::kOffA + s * C::kABytes, &tmW, fb, 0, nt * 128, kb * KO, g);
          } else {
            mbar_arrive_expect_tx(fb, KO * kWeightTileTxBytes + BN_MAX * KO * 128);
            tma_load_4d(smem + C::kOffA + s * C::kABytes, &tmW, fb, 0, nt * 128, kb * KO, g);
            tma_load_3d(smem + C::kOffB + s * C::kBBytes, &tmX, fb, 0, row0, kb * KO);
          }
        }
      }
    }
  } else if (warp == 3 && C::kTokenThread) {
    // ---------------------------------------------------------------- token TMA
    // (its own thread, so the weight stream's issue slots carry weight loads only)
    if (lane == 0) {
      if (p.early) pdl_wait();
      uint32_t it = 0;
      for (TileWalk tw(p.items, total, n_tiles, wstart, wstride); tw.valid() && !*abort_flag;
           tw.next()) {
        int g, row0, rows;
        const int nt = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1u, p.status, abort_flag)) break;
          mbar_arrive_expect_tx(&full[s], BN_MAX * KO * 128);
          tma_load_3d(smem + C::kOffB + s * C::kBBytes, &tmX, &full[s], 0, row0, kb * KO);
        }
      }
    }
  } else if (warp == 1 || (C::kIssuers == 2 && warp == 3)) {
    // ---------------------------------------------------------------- MMA issuer(s)
    // Issuer `par` takes the stages kb with kb % kIssuers == par into its own
    // accumulator; every issuer walks every stage to keep the ring's phase.
    const int par = warp == 1 ? 0 : 1;
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      uint32_t phases = 0;  // bit s: parity of the next phase of full[par][s] to wait for
      for (TileWalk tw(p.items, total, n_tiles, wstart, wstride); tw.valid() && !*abort_flag;
           tw.next()) {
        int g, row0, rows;
        const int nt = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        const int bn = (rows + 15) & ~15;
        const uint32_t b = tc & 1u, use = tc >> 1;
        if (tc >= 2 && !mbar_wait(&acc_empty[b], (use - 1) & 1u, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * C::kAccCols + par * BN_MAX;
        const uint32_t idesc = idesc_mxf4_e4m3(bn);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          if (C::kIssuers == 2 && (kb & 1) != par) continue;
          const int s = it % STAGES;
          const uint32_t ph = (phases >> s) & 1u;
          phases ^= 1u << s;
          uint64_t* fb = &full[par * STAGES + s];
          if (!mbar_wait(C::kSfFirst ? &sf_full[s] : fb, ph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_t = tmem + 2 * C::kAccCols + s * C::kSfCols;
          const uint32_t sfb_t = sf_t + 4 * KO;
          if constexpr (C::kWideSf) {
            // [KO][128 rows][16 B] -> KO * 4 columns; [NA][128][16 B] -> NA * 4 columns
            const uint64_t da = smem_desc(smem_u32(smem + C::kOffSfa + s * C::kSfaStage), 2048,
                                          128, kLayoutNone);
            const uint64_t db = smem_desc(smem_u32(smem + C::kOffSfb + s * C::kSfbStage), 2048,
                                          128, kLayoutNone);
            if (KO == 2) tc_cp_128x256b(sf_t, da);
            else tc_cp_128x128b(sf_t, da);
            if (C::kSfbAtoms == 2) tc_cp_128x256b(sfb_t, db);
            else tc_cp_128x128b(sfb_t, db);
          } else {
#pragma unroll
            for (int ko = 0; ko < KO; ++ko)
              tc_cp_32x128b_x4(sf_t + 4 * ko,
                               smem_desc(smem_u32(smem + C::kOffSfa + s * C::kSfaStage +
                                                  ko * C::kSfBytes),
                                         0, 128, kLayoutNone));
#pragma unroll
            for (int a = 0; a < C::kSfbAtoms; ++a)  // tokens 128a .. 128a+127 at columns +4a
              tc_cp_32x128b_x4(sfb_t + 4 * a,
                               smem_desc(smem_u32(smem + C::kOffSfb + s * C::kSfbStage +
                                                  a * C::kSfBytes),
                                         0, 128, kLayoutNone));
          }
          if (C::kSfFirst) {
            if (!mbar_wait(fb, ph, p.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t a0 = smem_u32(smem + C::kOffA + s * C::kABytes);
          const uint32_t b0 = smem_u32(smem + C::kOffB + s * C::kBBytes);
#pragma unroll
          for (int ko = 0; ko < KO; ++ko) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(a0 + ko * C::kASub + kk * 32, 0, 1024, kLayoutSw128);
              const uint64_t bd = smem_desc(b0 + ko * C::kBSub + kk * 32, 0, 1024, kLayoutSw128);
              // A scale: byte kk (32-K block) of the sub-tile's atom; B scale: byte ko.
              const uint32_t id = idesc | (static_cast<uint32_t>(kk) << 29) |
                                  (static_cast<uint32_t>(ko) << 4);
              mma_mxf8f6f4(d_tmem, ad, bd, id, sf_t + 4 * ko, sfb_t,
                           kb > par || ko != 0 || kk != 0);
            }
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
    // Per stage: KO weight atoms (row r at byte (r % 32) * 16 + (r / 32) * 4 + kblock)
    // and one token atom per 128 tokens whose byte ko holds the token's scale for
    // sub-tile ko (token r of atom a at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + ko).
    constexpr int NA = C::kSfbAtoms;
    const int kw = p.K / 32, kx = p.K / 128;
    constexpr int REP = C::kWideSf ? 4 : 1;  // copies of each atom row (see GemmCfg)
    constexpr int ATOM = C::kWideSf ? 2048 : C::kSfBytes;
    auto put_stage = [&](int s, int kb, const uint32_t (&wa)[KO][4],
                         const uint32_t (&xb)[4 * NA]) {
#pragma unroll
      for (int ko = 0; ko < KO; ++ko) {
        const uint4 v = make_uint4(wa[ko][0], wa[ko][1], wa[ko][2], wa[ko][3]);
#pragma unroll
        for (int rep = 0; rep < REP; ++rep)
          *reinterpret_cast<uint4*>(smem + C::kOffSfa + s * C::kSfaStage + ko * ATOM +
                                    (rep * 32 + lane) * 16) = v;
      }
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        const uint4 v = make_uint4(xb[4 * a], xb[4 * a + 1], xb[4 * a + 2], xb[4 * a + 3]);
#pragma unroll
        for (int rep = 0; rep < REP; ++rep)
          *reinterpret_cast<uint4*>(smem + C::kOffSfb + s * C::kSfbStage + a * ATOM +
                                    (rep * 32 + lane) * 16) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        mbar_arrive(C::kSfFirst ? &sf_full[s] : &full[(kb % C::kIssuers) * STAGES + s]);
    };
    auto wait_slot = [&](uint32_t it) -> bool {
      if (it < STAGES) return true;
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait(&empty[it % STAGES], ((it / STAGES) & 1u) ^ 1u, p.status, abort_flag);
      return __shfl_sync(0xFFFFFFFFu, w_ok, 0) != 0;
    };
    if ((p.K & 511) == 0) {
      // Pipelined path.  Scale bytes are fetched a quad (4 sub-tiles) at a time -- one
      // 16-byte load per weight row, one 4-byte load per token -- kSfQuads quads ahead
      // of the stage being staged, so their latency overlaps the MMAs.
      constexpr int Q = kSfQuads;
      constexpr int J = (BN_MAX + 31) / 32;
      constexpr int SPQ = 4 / KO;  // stages per quad
      const int nq = p.K / 512;
      struct Pos {
        long long L;
        int kq, g, row0, rows, nt;
      };
      auto seek = [&](long long L, Pos& P) -> bool {
        for (; L < total; L += wstride) {
          if (load_item(L, P.g, P.row0, P.rows, P.nt)) {
            P.L = L;
            P.kq = 0;
            return true;
          }
        }
        return false;
      };
      auto step = [&](Pos& P) -> bool {
        if (++P.kq < nq) return true;
        return seek(P.L + wstride, P);
      };
      uint4 wv[Q][4];
      uint32_t av[Q][J];
      Pos ld{}, cs{};
      bool ld_ok = seek(blockIdx.x, ld);
      bool cs_ok = seek(blockIdx.x, cs);
      auto fetch_w = [&](const Pos& P, uint4 (&w4)[4]) {
        const uint8_t* wsp =
            p.w_scales + (static_cast<size_t>(P.g) * p.N + P.nt * 128) * kw + P.kq * 16;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w4[j] = __ldg(reinterpret_cast<const uint4*>(wsp + static_cast<size_t>(j * 32 + lane) * kw));
      };
      auto fetch_x = [&](const Pos& P, uint32_t (&a)[J]) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int r = j * 32 + lane;
          a[j] = r < P.rows ? __ldg(reinterpret_cast<const uint32_t*>(
                                  p.x_scales + static_cast<size_t>(P.row0 + r) * kx + P.kq * 4))
                            : 0x7F7F7F7Fu;
        }
      };
      auto fetch = [&](uint4 (&w4)[4], uint32_t (&a)[J]) {
        fetch_w(ld, w4);
        fetch_x(ld, a);
        ld_ok = step(ld);
      };
      // The first Q quads: weight scales before the wait for the preceding kernel
      // (with p.early), token scales (its output) after it.
      Pos first[Q];
      bool first_ok[Q];
#pragma unroll
      for (int i = 0; i < Q; ++i) {
        first_ok[i] = ld_ok;
        if (ld_ok) {
          first[i] = ld;
          fetch_w(ld, wv[i]);
          ld_ok = step(ld);
        }
      }
      if (p.early) pdl_wait();
#pragma unroll
      for (int i = 0; i < Q; ++i)
        if (first_ok[i]) fetch_x(first[i], av[i]);
      uint32_t it = 0;
      bool ok = true;
      while (cs_ok && ok) {
#pragma unroll
        for (int i = 0; i < Q; ++i) {
          if (!cs_ok || !ok) break;
#pragma unroll
          for (int b = 0; b < SPQ; ++b) {
            if (!wait_slot(it)) {
              ok = false;
              break;
            }
            uint32_t wa[KO][4], xb[4 * NA];
#pragma unroll
            for (int ko = 0; ko < KO; ++ko)
#pragma unroll
              for (int j = 0; j < 4; ++j) wa[ko][j] = u4_comp(wv[i][j], b * KO + ko);
#pragma unroll
            for (int j = 0; j < 4 * NA; ++j) {
              if (j < J) {
                const uint32_t a = av[i][j < J ? j : 0] >> (8 * b * KO);
                xb[j] = KO == 4 ? a : (KO == 2 ? (a & 0xFFFFu) : (a & 0xFFu));
              } else {
                xb[j] = 0x7F7F7F7Fu;
              }
            }
            put_stage(it % STAGES, cs.kq * SPQ + b, wa, xb);
            ++it;
          }
          if (!ok) break;
          cs_ok = step(cs);
          if (ld_ok) fetch(wv[i], av[i]);  // refill slot i with the quad Q ahead
        }
      }
    } else {
      // General path (K not a multiple of 512): one stage at a time.
      if (p.early) pdl_wait();  // token scales come from the preceding kernel
      uint32_t it = 0;
      for (TileWalk tw(p.items, total, n_tiles, wstart, wstride); tw.valid() && !*abort_flag;
           tw.next()) {
        int g, row0, rows;
        const int nt = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        const uint8_t* wsp = p.w_scales + (static_cast<size_t>(g) * p.N + nt * 128) * kw;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          if (!wait_slot(it)) {
            ok = false;
            break;
          }
          uint32_t wa[KO][4], xb[4 * NA];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = j * 32 + lane;
#pragma unroll
            for (int ko = 0; ko < KO; ++ko)
              wa[ko][j] = __ldg(reinterpret_cast<const uint32_t*>(
                  wsp + static_cast<size_t>(r) * kw + (kb * KO + ko) * 4));
          }
#pragma unroll
          for (int j = 0; j < 4 * NA; ++j) {
            const int r = j * 32 + lane;
            uint32_t packed = 0;
#pragma unroll
            for (int ko = 0; ko < KO; ++ko) {
              uint32_t sb = 127u;
              if (r < rows)
                sb = __ldg(p.x_scales + static_cast<size_t>(row0 + r) * kx + kb * KO + ko);
              packed |= sb << (8 * ko);
            }
            xb[j] = packed;
          }
          put_stage(it % STAGES, kb, wa, xb);
        }
        if (!ok) break;
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp - 4;
    uint32_t tc = 0;
    // with the fused combine the four warps meet at named barriers: they leave the loop
    // together on the collective wait's verdict (an abort makes it fail), never one by
    // one on the abort flag
    for (TileWalk tw(p.items, total, n_tiles, wstart, wstride); tw.valid() && (F2 || !*abort_flag);
         tw.next()) {
      int g, row0, rows;
      const int nt = tw.nt;
      if (!check_item(tw.cur, g, row0, rows)) continue;
      const uint32_t b = tc & 1u, use = tc >> 1;
      if constexpr (F2) {
        // the fused combine meets at named barriers: one thread waits for the four warps,
        // so that none leaves the loop alone
        volatile int* go = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
        if (q == 0 && lane == 0) *go = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
        epilogue_bar_sync();
        const int ok_all = *go;
        epilogue_bar_sync();
        if (!ok_all) break;
      } else {
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, w_ok, 0)) break;
      }
      tc_fence_after();
      const int n = nt * 128 + q * 32 + lane;
      uint16_t* ycol = p.y + static_cast<size_t>(row0) * p.N + n;
      const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * C::kAccCols;
      for (int c0 = 0; c0 < rows; c0 += 16) {
        uint32_t r[16];
        float v[16];
        tmem_ld_32x32b_x16(acc + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
        if (C::kIssuers == 2 && nk > 1) {  // even-stage + odd-stage sums, in that order
          tmem_ld_32x32b_x16(acc + BN_MAX + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] += __uint_as_float(r[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (c0 + i < rows) {
            __nv_bfloat16 h = __float2bfloat16_rn(v[i]);
            ycol[static_cast<size_t>(c0 + i) * p.N] = *reinterpret_cast<uint16_t*>(&h);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++tc;
      // four tokens per thread per pass where one CTA holds the SM's registers
      if constexpr (F2)
        fused_combine_tile<(OCC == 1 ? 4 : 2)>(p, row0, rows, nt, q * 32 + lane,
                                                reinterpret_cast<int*>(smem + C::kOffFc));
    }
  }

  // After an abort, each MMA issuer waits (briefly, bounded) until the MMAs it already
  // issued have completed, so that TMEM is not released under them.  TMA loads still in
  // flight at an abort are not waited for: that unwind is best effort.
  if ((warp == 1 || (C::kIssuers == 2 && warp == 3)) && lane == 0 && *abort_flag) {
    uint64_t* db = &drain[warp == 1 ? 0 : 1];
    tc_commit(db);
    mbar_wait_drain(db, 0);
  }
  // Let the next kernel's CTAs in only now, so that none of them sits on an SM waiting
  // for this grid for the whole GEMM; the overlap left is this grid's drain.
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- SM pairs ---------
// The mid and large tiles on SM pairs (a cluster of two CTAs, cta_group::2 MMAs): one
// MMA covers 256 weight rows, CTA r of the pair holding rows 128 r .. 128 r + 127 of
// the pair's weight tile, the accumulator of those rows in its TMEM, and half of the
// token tile (tokens r * bn/2 .. of the item's bn); the even-ranked CTA issues the
// MMAs.  Against one CTA per tile this halves the MMA instructions per flop and the
// token bytes each SM stages per stage, which leaves shared memory for a third stage.
//   * both CTAs load their weight and token halves by TMA, completing on the leader's
//     full barrier (the leader expects the bytes of all four loads);
//   * both stage their scale factors (own weight rows; the item's whole token range --
//     each SM's MMA scales every token column from its own TMEM) and arrive on the
//     leader's scale barrier; the leader copies both CTAs' scales to their TMEM (tcgen05.cp for
//     the pair), then issues the MMAs;
//   * MMA completion is multicast to both CTAs' empty / accumulator-full barriers; both
//     epilogues arrive on the leader's accumulator-empty barrier.
template <int BN2, int STAGES, int SFS, bool F1>
struct GemmCfg2 {
  static constexpr int KO = 2;
  static constexpr int BH = BN2 / 2;              // token rows per CTA
  static constexpr int kASub = 128 * 128;
  static constexpr int kBSub = BH * 128;
  static constexpr int kABytes = KO * kASub;
  static constexpr int kBBytes = KO * kBSub;
  static constexpr int kSfbAtoms = (BN2 + 127) / 128;  // the item's whole token range
  // wide scale staging (every 32-row atom written four times, one tcgen05.cp.128xNb per
  // operand and stage; see GemmCfg)
  static constexpr int kSfaStage = KO * 2048;
  static constexpr int kSfbStage = kSfbAtoms * 2048;
  // The scale factors have a ring of their own (SFS slots, deeper than the data ring),
  // so that their staging runs ahead of the stage the MMAs wait for instead of starting
  // only when the data stage's slot frees up.
  static constexpr int kSfTotal = SFS * (kSfaStage + kSfbStage);
  static constexpr int kOffSfa = 0;
  static constexpr int kOffSfb = SFS * kSfaStage;
  static constexpr int kOffA = (kSfTotal + 1023) / 1024 * 1024;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffBar = kOffB + STAGES * kBBytes;
  // full[S] (leader: 1 + tx), empty[S] (1: multicast commit), sf_full[SFS] (leader: 2),
  // sf_empty[SFS] (1: multicast commit after the copies), sf_ready[SFS] (peer: its
  // scale warp, relayed to the leader's sf_full by the peer's warp 1), acc_full[2] (1:
  // multicast commit), acc_empty[2] (leader: 8 epilogue warps), drain
  // (+ xchg_full[2] with F1: the peer's per-token amax arrived)
  static constexpr int kNumBars = 2 * STAGES + 3 * SFS + 5 + (F1 ? 2 : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // F1 epilogue scratch: up values of a 16-token chunk [64 features][16] fp32, the two
  // gate warps' per-token amax [2][16], this CTA's amax per token [BN2], the peer's
  // [2 slots][BN2], a chunk's codes [16 tokens][64 B], its scale bytes [16]
  static constexpr int kOffUp = (kOffMisc + 16 + 15) / 16 * 16;
  static constexpr int kOffAm32 = kOffUp + 64 * 16 * 4;
  static constexpr int kOffAmMine = kOffAm32 + 2 * 16 * 4;
  static constexpr int kOffAmPeer = kOffAmMine + BN2 * 4;
  static constexpr int kOffCodes = kOffAmPeer + 2 * BN2 * 4;
  static constexpr int kOffEs = kOffCodes + 16 * 64;
  static constexpr int kSmemBytes = F1 ? kOffEs + 16 * 4 + 16 : kOffMisc + 16;
  static constexpr int kSfCols = 4 * (KO + kSfbAtoms);
  static constexpr int kTmemNeed = 2 * BN2 + STAGES * kSfCols;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static constexpr uint32_t kTxBytes = 2u * (KO * kWeightTileTxBytes + kBBytes);
  static_assert(BN2 % 32 == 0 && BN2 <= 256, "token tile: two halves of multiples of 16");
  static_assert(kSfbAtoms <= 2, "wide scale copies move <= 256 bits");
  static_assert(kTmemNeed <= 512, "TMEM");
  static_assert(kSmemBytes <= 232448, "dynamic shared memory of one CTA");
};

// F1 epilogue of the W13 pair kernel (warps 4-7 of each CTA).  TMEM lanes 0-63 hold
// this CTA's 64 gate features, lanes 64-127 the same 64 up features; columns are the
// item's tokens.  Per tile: pass 1 computes h = silu(g) * u (g, u the accumulators
// rounded to bf16, as y13 would be) per 16-token chunk, the up warps handing their
// values to the gate warps through shared memory, and each token's amax over the 64
// features; the two CTAs swap those amaxes (distributed shared memory, one remote
// arrive); pass 2 recomputes h, takes the scale exponent of the 128-feature block from
// the larger of the two amaxes and writes the FP8 codes (rows of 64 bytes) and, in the
// leader, the scale bytes.  The arithmetic is k_swiglu_quant's, value for value.
template <int BN2, typename LoadItem, typename LeaderAddr>
__device__ __forceinline__ void f1_epilogue(const GemmParams& p, uint32_t tmem, uint8_t* smem,
                                            int off_up, int off_am32, int off_am_mine,
                                            int off_am_peer, int off_codes, int off_es,
                                            uint64_t* acc_full, uint64_t* acc_empty,
                                            uint64_t* xchg_full, volatile int* abort_flag,
                                            uint32_t rank, bool leader, long long cl,
                                            long long ncl, long long total, LoadItem load_item,
                                            LeaderAddr leader_addr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp - 4;  // 0, 1: gate warps; 2, 3: up warps
  const int et = q * 32 + lane;
  float* upbuf = reinterpret_cast<float*>(smem + off_up);           // [64][16]
  float* am32 = reinterpret_cast<float*>(smem + off_am32);          // [2][16]
  float* am_mine = reinterpret_cast<float*>(smem + off_am_mine);    // [BN2]
  float* am_peer = reinterpret_cast<float*>(smem + off_am_peer);    // [2][BN2]
  uint8_t* codes = smem + off_codes;                                // [16][64]
  int* es = reinterpret_cast<int*>(smem + off_es);                  // [16]
  volatile int* go = reinterpret_cast<volatile int*>(smem + off_es + 16 * 4);  // shared answer
  const int I = p.N / 2;
  const int nblk = I / 128;
  const uint32_t peer = rank ^ 1u;
  uint32_t tc = 0;
  // (no abort-flag test in the loop condition: the warps leave together, on the
  // collective wait's verdict, which an abort makes fail)
  for (long long L = cl; L < total; L += ncl) {
    int g, row0, rows, nt2;
    if (!load_item(L, g, row0, rows, nt2)) continue;
    const uint32_t b = tc & 1u, use = tc >> 1;
    // one thread waits and the four warps take its answer together: they meet at named
    // barriers below, which a warp that left the loop alone would never reach
    int w_ok = 1;
    if (q == 0 && lane == 0) *go = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
    epilogue_bar_sync();
    if (!*go) break;
    tc_fence_after();
    const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN2;
    // h of this thread's feature for tokens c0 .. c0 + 15 (gate warps only)
    auto chunk_h = [&](int c0, float (&h)[16]) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(acc + c0, r);
      tmem_ld_wait();
      if (q >= 2) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          upbuf[(et - 64) * 16 + i] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i])));
      }
      epilogue_bar_sync();
      if (q < 2) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float gv = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i])));
          const float uv = upbuf[et * 16 + i];
          h[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
        }
      }
    };
    // pass 1: this CTA's per-token amax over its 64 features
    for (int c0 = 0; c0 < rows; c0 += 16) {
      float h[16];
      chunk_h(c0, h);
      if (q < 2) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float m = fabsf(h[i]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
          if (lane == 0) am32[q * 16 + i] = m;
        }
      }
      epilogue_bar_sync();
      if (q == 0 && lane < 16 && c0 + lane < BN2) am_mine[c0 + lane] = fmaxf(am32[lane], am32[16 + lane]);
    }
    epilogue_bar_sync();
    // swap with the peer: my amaxes into its am_peer[b], then its arrival on mine
    if (q == 0 && lane == 0) {
      const uint32_t dst = mapa_shared(smem_u32(am_peer + b * BN2), peer);
      for (int c = 0; c < rows; ++c)
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + 4u * c), "f"(am_mine[c])
                     : "memory");
      mbar_arrive_cluster(mapa_shared(smem_u32(&xchg_full[b]), peer));
      w_ok = mbar_wait(&xchg_full[b], use & 1u, p.status, abort_flag);
      *go = w_ok;
    }
    epilogue_bar_sync();
    if (!*go) break;
    // pass 2: codes and scales
    for (int c0 = 0; c0 < rows; c0 += 16) {
      float h[16];
      chunk_h(c0, h);
      if (q < 2) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c0 + i < BN2 ? c0 + i : BN2 - 1;
          const int e = fp8_scale_exponent(fmaxf(am_mine[c], am_peer[b * BN2 + c]));
          codes[i * 64 + et] = static_cast<uint8_t>(
              __nv_cvt_float_to_fp8(h[i] * pow2_neg(e), __NV_SATFINITE, __NV_E4M3));
          if (q == 0 && lane == 0) es[i] = e;
        }
      }
      epilogue_bar_sync();
      if (et < 64) {
        const int i = et >> 2, part = et & 3;
        if (c0 + i < rows) {
          const size_t row = static_cast<size_t>(row0 + c0 + i);
          *reinterpret_cast<uint4*>(p.hq + row * I + nt2 * 128 + rank * 64 + part * 16) =
              *reinterpret_cast<const uint4*>(codes + i * 64 + part * 16);
          if (leader && part == 0) p.hs[row * nblk + nt2] = static_cast<uint8_t>(es[i] + 127);
        }
      }
      epilogue_bar_sync();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (leader) mbar_arrive(&acc_empty[b]);
      else mbar_arrive_cluster(leader_addr(&acc_empty[b]));
    }
    ++tc;
  }
}

// Instruction descriptor of the pair MMA: as idesc_mxf4_e4m3 with M = 256.
__device__ __forceinline__ uint32_t idesc_mxf4_e4m3_m256(int n) {
  uint32_t d = 0;
  d |= 5u << 7;
  d |= 0u << 10;
  d |= static_cast<uint32_t>(n >> 3) << 17;
  d |= 1u << 23;
  d |= static_cast<uint32_t>(256 >> 4) << 24;
  return d;
}

template <int BN2, int STAGES, int SFS, bool F1>
__global__ void __launch_bounds__(256, 1)
    k_gemm_mx2(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               const GemmParams p) {
  using C = GemmCfg2<BN2, STAGES, SFS, F1>;
  constexpr int KO = C::KO;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* sf_full = empty + STAGES;
  uint64_t* sf_empty = sf_full + SFS;
  uint64_t* sf_ready = sf_empty + SFS;
  uint64_t* acc_full = sf_ready + SFS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* xchg_full = drain + 1;  // F1 only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < SFS; ++j) {
      mbar_init(&sf_full[j], 2);
      mbar_init(&sf_empty[j], 1);
      mbar_init(&sf_ready[j], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);
    }
    mbar_init(drain, 1);
    if constexpr (F1) {
      mbar_init(&xchg_full[0], 1);
      mbar_init(&xchg_full[1], 1);
    }
    // the 128B-swizzled tiles need 1024-byte alignment: checked, and a misaligned base
    // turns every role into a no-op (the CTA still takes part in the pair's set-up and
    // teardown, which its peer waits for)
    const bool bad = (smem_u32(smem) & 1023u) != 0;
    *abort_flag = bad ? 1 : 0;
    if (bad) set_status(p.status, STATUS_BAD_PLAN);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote arrive or multicast
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles2 = p.N / 256;
  const int nk = p.K / (128 * KO);
  int count = *p.item_count;
  if (count > p.max_items) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    count = p.max_items;
  }
  long long total = static_cast<long long>(count) * n_tiles2;
  if (total > 0x7FFFFFFFll) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    total = 0;
  }
  const long long cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  // validates one work item; every role sees the same result
  auto check_item = [&](const int4 it, int& g, int& row0, int& rows) -> bool {
    g = it.x;
    row0 = it.y;
    rows = it.z;
    if (rows <= 0) return false;
    if (g < 0 || g >= p.G || row0 < 0 || rows > BN2 || row0 + rows > p.rows_total) {
      if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
      return false;
    }
    return true;
  };
  // tile L directly (the scale stager's look-ahead, the fused epilogue)
  auto load_item = [&](long long L, int& g, int& row0, int& rows, int& nt2) -> bool {
    const int Li = static_cast<int>(L);  // total < 2^31 (checked above)
    nt2 = Li % n_tiles2;
    return check_item(__ldg(p.items + Li / n_tiles2), g, row0, rows);
  };
  // the leader's copies of the barriers the peer completes
  auto leader_addr = [&](const uint64_t* b) -> uint32_t { return mapa_shared(smem_u32(b), 0); };

  if (warp == 0) {
    // ---------------------------------------------------------------- weight TMA
    if (lane == 0) {
      uint32_t it = 0;
      for (TileWalk tw(p.items, total, n_tiles2, static_cast<int>(cl), static_cast<int>(ncl));
           tw.valid() && !*abort_flag; tw.next()) {
        int g, row0, rows;
        const int nt2 = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          if (it >= STAGES &&
              !mbar_wait(&empty[s], ((it / STAGES) & 1u) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[s], C::kTxBytes);
          if constexpr (F1) {
            // rows 0-63: gate rows 128 nt2 + 64 r ..; rows 64-127: the same up rows
            const int gate0 = nt2 * 128 + static_cast<int>(rank) * 64;
            const uint32_t fb = leader_addr(&full[s]);
#pragma unroll
            for (int ko = 0; ko < KO; ++ko) {
              uint8_t* dst = smem + C::kOffA + s * C::kABytes + ko * C::kASub;
              tma_load_4d_pair(dst, &tmW, fb, 0, gate0, kb * KO + ko, g);
              tma_load_4d_pair(dst + 64 * 128, &tmW, fb, 0, p.N / 2 + gate0, kb * KO + ko, g);
            }
          } else {
            tma_load_4d_pair(smem + C::kOffA + s * C::kABytes, &tmW, leader_addr(&full[s]), 0,
                             (nt2 * 2 + static_cast<int>(rank)) * 128, kb * KO, g);
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------------- token TMA
    if (lane == 0) {
      uint32_t it = 0;
      for (TileWalk tw(p.items, total, n_tiles2, static_cast<int>(cl), static_cast<int>(ncl));
           tw.valid() && !*abort_flag; tw.next()) {
        int g, row0, rows;
        const int nt2 = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        const int half = ((rows + 15) & ~15) >> 1;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          if (it >= STAGES &&
              !mbar_wait(&empty[s], ((it / STAGES) & 1u) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tma_load_3d_pair(smem + C::kOffB + s * C::kBBytes, &tmX, leader_addr(&full[s]), 0,
                           row0 + static_cast<int>(rank) * half, kb * KO);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1 && !leader) {
    // ---------------------------------------------------------------- scale relay
    // The peer's scale warp arrives on its own sf_ready; this thread, which has no
    // memory operations in flight, forwards each arrival to the leader's sf_full.  (A
    // cluster-scope release by the scale warp itself would wait for the scale loads
    // it keeps in flight several stages ahead.)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (TileWalk tw(p.items, total, n_tiles2, static_cast<int>(cl), static_cast<int>(ncl));
           tw.valid() && ok && !*abort_flag; tw.next()) {
        int g, row0, rows;
        const int nt2 = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int j = it % SFS;
          if (!mbar_wait(&sf_ready[j], (it / SFS) & 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(leader_addr(&sf_full[j]));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      for (TileWalk tw(p.items, total, n_tiles2, static_cast<int>(cl), static_cast<int>(ncl));
           tw.valid() && !*abort_flag; tw.next()) {
        int g, row0, rows;
        const int nt2 = tw.nt;
        if (!check_item(tw.cur, g, row0, rows)) continue;
        const int bn = (rows + 15) & ~15;
        const uint32_t b = tc & 1u, use = tc >> 1;
        if (tc >= 2 && !mbar_wait(&acc_empty[b], (use - 1) & 1u, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * BN2;
        const uint32_t idesc = idesc_mxf4_e4m3_m256(bn);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          const int j = it % SFS;
          if (!mbar_wait(&sf_full[j], (it / SFS) & 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          // TMEM scale slot s is free once the MMAs of stage it - STAGES completed
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_t = tmem + 2 * BN2 + s * C::kSfCols;
          const uint32_t sfb_t = sf_t + 4 * KO;
          const uint64_t da = smem_desc(smem_u32(smem + C::kOffSfa + j * C::kSfaStage), 2048, 128,
                                        kLayoutNone);
          const uint64_t db = smem_desc(smem_u32(smem + C::kOffSfb + j * C::kSfbStage), 2048, 128,
                                        kLayoutNone);
          tc_cp_128x256b_pair(sf_t, da);
          if (C::kSfbAtoms == 2) tc_cp_128x256b_pair(sfb_t, db);
          else tc_cp_128x128b_pair(sfb_t, db);
          tc_commit_pair_mc(&sf_empty[j], 3);  // both CTAs' scale slot j, once copied
          if (!mbar_wait(&full[s], ph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + C::kOffA + s * C::kABytes);
          const uint32_t b0 = smem_u32(smem + C::kOffB + s * C::kBBytes);
#pragma unroll
          for (int ko = 0; ko < KO; ++ko) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(a0 + ko * C::kASub + kk * 32, 0, 1024, kLayoutSw128);
              const uint64_t bd = smem_desc(b0 + ko * C::kBSub + kk * 32, 0, 1024, kLayoutSw128);
              const uint32_t id = idesc | (static_cast<uint32_t>(kk) << 29) |
                                  (static_cast<uint32_t>(ko) << 4);
              mma_mxf8f6f4_pair(d_tmem, ad, bd, id, sf_t + 4 * ko, sfb_t,
                                kb > 0 || ko != 0 || kk != 0);
            }
          }
          tc_commit_pair_mc(&empty[s], 3);
        }
        if (!ok) break;
        tc_commit_pair_mc(&acc_full[b], 3);
        ++tc;
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- scale factors
    // Weight atoms: this CTA's 128 rows (row r at byte (r % 32) * 16 + (r / 32) * 4 +
    // kblock); token atoms: the item's whole token range in both CTAs (the MMA scales
    // every token column on both SMs from their own TMEM), token c of atom a at byte
    // (c % 32) * 16 + ((c / 32) % 4) * 4 + ko.  Each 32-row atom is written four times
    // (the wide layout: one 128-lane copy per operand).  Scale bytes are fetched a quad
    // of 128-K sub-tiles (two stages) at a time, kSfQuads quads ahead of the stage
    // being staged, so their latency overlaps the MMAs.
    constexpr int NA = C::kSfbAtoms;
    constexpr int J = (BN2 + 31) / 32;
    constexpr int Q = kSfQuads;
    constexpr int SPQ = 4 / KO;  // stages per quad
    const int kw = p.K / 32, kx = p.K / 128;
    const int nq = p.K / 512;
    struct Pos {
      long long L;
      int kq, g, row0, rows, nt2;
    };
    auto seek = [&](long long L, Pos& P) -> bool {
      for (; L < total; L += ncl) {
        if (load_item(L, P.g, P.row0, P.rows, P.nt2)) {
          P.L = L;
          P.kq = 0;
          return true;
        }
      }
      return false;
    };
    auto step = [&](Pos& P) -> bool {
      if (++P.kq < nq) return true;
      return seek(P.L + ncl, P);
    };
    auto fetch = [&](const Pos& P, uint4 (&w4)[4], uint32_t (&a)[J]) {
      const uint8_t* wsp = p.w_scales + static_cast<size_t>(P.g) * p.N * kw + P.kq * 16;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // this CTA's weight row j * 32 + lane (F1: gate rows, then the same up rows)
        const int row = F1 ? (j < 2 ? 0 : p.N / 2) + P.nt2 * 128 + static_cast<int>(rank) * 64 +
                                 (j & 1) * 32 + lane
                           : (P.nt2 * 2 + static_cast<int>(rank)) * 128 + j * 32 + lane;
        w4[j] = __ldg(reinterpret_cast<const uint4*>(wsp + static_cast<size_t>(row) * kw));
      }
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = j * 32 + lane;
        a[j] = c < P.rows ? __ldg(reinterpret_cast<const uint32_t*>(
                                p.x_scales + static_cast<size_t>(P.row0 + c) * kx + P.kq * 4))
                          : 0x7F7F7F7Fu;
      }
    };
    uint4 wv[Q][4];
    uint32_t av[Q][J];
    Pos ld{}, cs{};
    bool ld_ok = seek(cl, ld);
    bool cs_ok = seek(cl, cs);
#pragma unroll
    for (int i = 0; i < Q; ++i)
      if (ld_ok) {
        fetch(ld, wv[i], av[i]);
        ld_ok = step(ld);
      }
    uint32_t it = 0;
    bool ok = nq > 0;
    while (cs_ok && ok && !*abort_flag) {
#pragma unroll
      for (int i = 0; i < Q; ++i) {
        if (!cs_ok || !ok) break;
#pragma unroll
        for (int b = 0; b < SPQ; ++b) {
          const int s = it % SFS;  // scale ring slot
          if (it >= SFS) {
            int w_ok = 1;
            if (lane == 0)
              w_ok = mbar_wait(&sf_empty[s], ((it / SFS) & 1u) ^ 1u, p.status, abort_flag);
            if (!__shfl_sync(0xFFFFFFFFu, w_ok, 0)) {
              ok = false;
              break;
            }
          }
#pragma unroll
          for (int ko = 0; ko < KO; ++ko) {
            const uint4 v = make_uint4(u4_comp(wv[i][0], b * KO + ko), u4_comp(wv[i][1], b * KO + ko),
                                       u4_comp(wv[i][2], b * KO + ko), u4_comp(wv[i][3], b * KO + ko));
#pragma unroll
            for (int rep = 0; rep < 4; ++rep)
              *reinterpret_cast<uint4*>(smem + C::kOffSfa + s * C::kSfaStage + ko * 2048 +
                                        (rep * 32 + lane) * 16) = v;
          }
#pragma unroll
          for (int a = 0; a < NA; ++a) {
            uint32_t xb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int jj = a * 4 + j;
              xb[j] = jj < J ? (av[i][jj < J ? jj : 0] >> (8 * b * KO)) & 0xFFFFu : 0x7F7Fu;
            }
            const uint4 v = make_uint4(xb[0], xb[1], xb[2], xb[3]);
#pragma unroll
            for (int rep = 0; rep < 4; ++rep)
              *reinterpret_cast<uint4*>(smem + C::kOffSfb + s * C::kSfbStage + a * 2048 +
                                        (rep * 32 + lane) * 16) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(leader ? &sf_full[s] : &sf_ready[s]);
          ++it;
        }
        if (!ok) break;
        cs_ok = step(cs);
        if (ld_ok) {  // refill slot i with the quad Q ahead
          fetch(ld, wv[i], av[i]);
          ld_ok = step(ld);
        }
      }
    }
  } else if (warp >= 4 && F1) {
    // ---------------------------------------------------------------- F1 epilogue
    f1_epilogue<BN2>(p, tmem, smem, C::kOffUp, C::kOffAm32, C::kOffAmMine, C::kOffAmPeer,
                     C::kOffCodes, C::kOffEs, acc_full, acc_empty, xchg_full, abort_flag, rank,
                     leader, cl, ncl, total, load_item, leader_addr);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp - 4;
    uint32_t tc = 0;
    for (TileWalk tw(p.items, total, n_tiles2, static_cast<int>(cl), static_cast<int>(ncl));
         tw.valid() && !*abort_flag; tw.next()) {
      int g, row0, rows;
      const int nt2 = tw.nt;
      if (!check_item(tw.cur, g, row0, rows)) continue;
      const uint32_t b = tc & 1u, use = tc >> 1;
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, w_ok, 0)) break;
      tc_fence_after();
      const int n = (nt2 * 2 + static_cast<int>(rank)) * 128 + q * 32 + lane;
      uint16_t* ycol = p.y + static_cast<size_t>(row0) * p.N + n;
      const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN2;
      for (int c0 = 0; c0 < rows; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(acc + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (c0 + i < rows) {
            const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(r[i]));
            ycol[static_cast<size_t>(c0 + i) * p.N] = *reinterpret_cast<const uint16_t*>(&h);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&acc_empty[b]);
        else mbar_arrive_cluster(leader_addr(&acc_empty[b]));
      }
      ++tc;
    }
  }

  // After an abort the leader's MMA thread waits (bounded) for the MMAs it issued.
  if (warp == 1 && lane == 0 && leader && *abort_flag) {
    tc_commit_pair_mc(drain, 1);
    mbar_wait_drain(drain, 0);
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA releases TMEM or shared memory the pair still uses
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side -------

EncodeTiledFn get_encode_tiled_fn() {
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

namespace {

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

template <int BN_MAX, int STAGES, int KO, int OCC, bool F2>
cudaError_t launch_one_f(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p,
                         int max_items, cudaStream_t st) {
  using C = GemmCfg<BN_MAX, STAGES, KO, OCC>;
  auto kern = k_gemm_mx<BN_MAX, STAGES, KO, OCC, F2>;
  // the shared-memory attribute is set once per context (again after a reset)
  static unsigned long long attr_ctx[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long ctx = current_context_id();
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (ctx == 0 || attr_ctx[dev] != ctx) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_ctx[dev] = current_context_id();
  }
  const long long tiles = static_cast<long long>(max_items) * (p.N / 128);
  if (tiles == 0) return cudaSuccess;
  const int slots = dev_info().sms * OCC;
  const int grid = static_cast<int>(tiles < slots ? tiles : slots);
  GemmParams q = p;
  q.max_items = max_items;
  // The large variant (one CTA per SM) runs slower at 32K tokens when launched as a
  // programmatic dependent (measured: 17.4 vs 17.05 ms per layer, ~8% before the tile
  // walk; cause not identified), so the one-CTA-per-SM variants wait for their
  // predecessor the plain way.  The two-CTA-per-SM small and medium variants keep the
  // overlap.
  return launch_k_pdl(OCC > 1, kern, grid, 256, C::kSmemBytes, st, tmW, tmX, q);
}

// The combine-fused W2 epilogue (f2) is its own instantiation, so that its gather's
// registers do not weigh on the plain epilogue's allocation.
template <int BN_MAX, int STAGES, int KO, int OCC>
cudaError_t launch_one(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p,
                       int max_items, cudaStream_t st) {
  if (p.out) return launch_one_f<BN_MAX, STAGES, KO, OCC, true>(tmW, tmX, p, max_items, st);
  return launch_one_f<BN_MAX, STAGES, KO, OCC, false>(tmW, tmX, p, max_items, st);
}

// The pair kernel for one list: clusters of two CTAs, as many clusters as fit at once.
template <int BN2, int STAGES, int SFS, bool F1>
cudaError_t launch_pair(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p,
                        int max_items, cudaStream_t st) {
  using C = GemmCfg2<BN2, STAGES, SFS, F1>;
  auto kern = k_gemm_mx2<BN2, STAGES, SFS, F1>;
  static unsigned long long attr_ctx[64] = {};
  static int max_clusters[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const long long pairs = static_cast<long long>(max_items) * (p.N / 256);
  if (pairs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || attr_ctx[dev] != ctx) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (dev_info().sms / 2));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters[dev] = n;
    attr_ctx[dev] = current_context_id();
  }
  const long long clusters = pairs < max_clusters[dev] ? pairs : max_clusters[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  GemmParams q = p;
  q.max_items = max_items;
  return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, q);
}

}  // namespace

// Tensor maps for one launch: weights as a 4D view {128 K elements, N rows, K/128
// sub-tiles, G} (box {128, 128, ko, 1}, FP4 unpacked to the 16-byte-aligned form),
// packed activation rows as a 3D view {128 bytes, rows, K/128} (box {128, xr, ko}).
int gemm_encode_maps(const uint8_t* w_codes, int G, int N, int K, const uint8_t* act,
                     int rows_total, int ko, int xr, CUtensorMap* tmW, CUtensorMap* tmX,
                     int wr = 128) {
  EncodeTiledFn enc = get_encode_tiled_fn();
  if (!enc) return MOE_ERR_CUDA;
  {
    cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / 128),
                          static_cast<cuuint64_t>(G)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(K / 2), 64,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[4] = {128, static_cast<cuuint32_t>(wr), static_cast<cuuint32_t>(ko), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<uint8_t*>(w_codes), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows_total > 0 ? rows_total : 1),
                          static_cast<cuuint64_t>(K / 128)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), 128};
    cuuint32_t box[3] = {128, static_cast<cuuint32_t>(xr), static_cast<cuuint32_t>(ko)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(act), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

namespace {

// One variant: KO = 2 sub-tiles per stage when K allows it, else the KO = 1 layout.
template <int BN, int ST2, int ST1, int OCC>
cudaError_t launch_variant(const GemmLaunch& a, GemmParams p, const int4* items,
                           const int32_t* count, int max_items, cudaStream_t st) {
  // ST2 == 0: this variant always stages one sub-tile at a time
  const bool two = ST2 > 0 && (a.K / 128) % 2 == 0;
  CUtensorMap tmW, tmX;
  if (gemm_encode_maps(a.w_codes, a.G, a.N, a.K, a.act, a.rows_total, two ? 2 : 1, BN, &tmW,
                       &tmX) != MOE_OK)
    return cudaErrorInvalidValue;
  p.items = items;
  p.item_count = count;
  if constexpr (ST2 > 0) {
    if (two) return launch_one<BN, ST2, 2, OCC>(tmW, tmX, p, max_items, st);
  }
  return launch_one<BN, ST1, 1, OCC>(tmW, tmX, p, max_items, st);
}

}  // namespace

// f1: W13 with SwiGLU + quantisation in the epilogue: every list on the SM-pair kernel
// (its tile of 2 x (64 gate + 64 up) weight rows is one 128-feature quantisation block).
static cudaError_t launch_w13_fused_swiglu(const GemmLaunch& a, GemmParams p, cudaStream_t st) {
  if (a.N % 256 != 0 || a.K % 512 != 0) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmX;
  if (gemm_encode_maps(a.w_codes, a.G, a.N, a.K, a.act, a.rows_total, 1, kPairBN / 2, &tmW,
                       &tmX, 64) != MOE_OK)
    return cudaErrorInvalidValue;
  // the token map moves two 128-K sub-tiles per load, the weight map one 64-row box
  CUtensorMap tmW2, tmX2;
  if (gemm_encode_maps(a.w_codes, a.G, a.N, a.K, a.act, a.rows_total, 2, kPairBN / 2, &tmW2,
                       &tmX2) != MOE_OK)
    return cudaErrorInvalidValue;
  const int bounds[kNumVariants] = {kSmallBN, kMediumBN, kMidBN, kLargeBN};
  for (int v = 0; v < kNumVariants; ++v) {
    GemmParams q = p;
    q.items = a.items[v];
    q.item_count = a.item_counts + v;
    const cudaError_t e =
        launch_pair<kPairBN, kPairStages, kPairSfSlotsF1, true>(tmW, tmX2, q, a.max_items[v], st);
    if (e != cudaSuccess || a.max_group_rows <= bounds[v]) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_grouped_gemm(const GemmLaunch& a, cudaStream_t st) {
  GemmParams p{};
  p.w_scales = a.w_scales;
  p.x_scales = a.act_scales;
  p.y = a.y;
  p.N = a.N;
  p.K = a.K;
  p.G = a.G;
  p.rows_total = a.rows_total;
  p.status = a.status;
  p.out = a.out;
  p.perm_src = a.perm_src;
  p.inv = a.inv;
  p.cw = a.cw;
  p.cnt = a.cnt;
  p.T = a.T;
  p.k = a.k;
  p.has_shared = a.has_shared;
  p.hq = a.hq;
  p.hs = a.hs;
  if (a.hq) return launch_w13_fused_swiglu(a, p, st);
  // A list whose groups cannot exist (no group has more than max_group_rows rows) is
  // provably empty and not launched.
  // The first launch inherits the caller's word on the plan; each later variant
  // follows a GEMM launch that waited for the plan's producer before it started.
  p.early = a.early_plan;
  cudaError_t e = launch_variant<kSmallBN, kSmallStages, kSmallStagesKO1, kSmallOcc>(
      a, p, a.items[0], a.item_counts, a.max_items[0], st);
  if (e != cudaSuccess || a.max_group_rows <= kSmallBN) return e;
  p.early = 1;
  e = launch_variant<kMediumBN, kMediumStages, kMediumStagesKO1, kMediumOcc>(
      a, p, a.items[1], a.item_counts + 1, a.max_items[1], st);
  if (e != cudaSuccess || a.max_group_rows <= kMediumBN) return e;
  if (a.pair_tiles && a.N % 256 == 0 && a.K % 512 == 0 && a.out == nullptr) {
    // mid and large tiles on SM pairs (same kernel for both lists; the combine-fused
    // W2 epilogue stays on the one-SM kernels)
    CUtensorMap tmW, tmX;
    if (gemm_encode_maps(a.w_codes, a.G, a.N, a.K, a.act, a.rows_total, 2, kPairBN / 2, &tmW,
                         &tmX) != MOE_OK)
      return cudaErrorInvalidValue;
    GemmParams q = p;
    q.items = a.items[2];
    q.item_count = a.item_counts + 2;
    e = launch_pair<kPairBN, kPairStages, kPairSfSlots, false>(tmW, tmX, q, a.max_items[2], st);
    if (e != cudaSuccess || a.max_group_rows <= kMidBN) return e;
    q.items = a.items[3];
    q.item_count = a.item_counts + 3;
    return launch_pair<kPairBN, kPairStages, kPairSfSlots, false>(tmW, tmX, q, a.max_items[3],
                                                                   st);
  }
  e = launch_variant<kMidBN, kMidStages, kMidStagesKO1, 1>(a, p, a.items[2],
                                                           a.item_counts + 2, a.max_items[2], st);
  if (e != cudaSuccess || a.max_group_rows <= kMidBN) return e;
  return launch_variant<kLargeBN, kLargeStages, kLargeStagesKO1, 1>(
      a, p, a.items[3], a.item_counts + 3, a.max_items[3], st);
}

}  // namespace moe
