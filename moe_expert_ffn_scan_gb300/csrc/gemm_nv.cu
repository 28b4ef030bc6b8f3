// f3: grouped GEMM with NVFP4 expert weights and FP8 activations on the tcgen05
// tensor cores.
//
// Pages: GB10 "Optimization progress report", Optimization 05 (native NVFP4 MoE: the
// expert weights stay NVFP4 in memory and the expert kernel reads them as such, with
// no up-front dequantisation of whole matrices); "Pushing the Limits of Serving
// DeepSeek-V4-Pro" (LMSYS, H20), §3.3 (W13 and W2 as grouped GEMMs shaped by the
// routing histogram).
//
// NVFP4 = E2M1 codes, one E4M3 scale per 16 K elements, one fp32 scale per weight
// tensor.  No block-scaled tensor-core kind pairs E4M3 block scales with FP8
// activations (kind::mxf8f6f4 takes UE8M0 scales per 32; kind::mxf4nvf4 wants FP4 on
// both sides), so this kernel multiplies in bf16, where both operands are exact:
//   * a weight e2m1 x e4m3 has at most 2 + 4 significant bits and lies in
//     [2^-10, 2688]: exact in bf16 (8 significant bits);
//   * an FP8 activation code x its power-of-two block scale 2^e has 4 significant
//     bits: exact in bf16 down to bf16's subnormal floor (a 128-block whose amax is
//     below about 2^-116 loses its smallest codes).  The activations arrive already
//     expanded to bf16 rows by the quantisation kernels.
// kind::f16 MMAs accumulate those exact products in fp32, as the MXFP4 path does; the
// tensor scale multiplies the fp32 sum in the epilogue before the bf16 rounding.
//
// Design (per CTA, one per SM, 8 + 4 NG warps):
//   * warp 0: TMA of the packed codes (0.5 B / weight, 128B- or 64B-swizzled so the
//     converters read them without bank conflicts) and the E4M3 scales of a K stage
//     -- the weights cross HBM in their 0.5625 B / weight NVFP4 form;
//   * warp 2: TMA of the bf16 token rows of the stage (their own ring);
//   * warps 4 .. 4 + 4 NG - 1: NG converter groups of four warps.  Group g converts the
//     K stages it with it % NG == g, so NG stages are decoded at once; warp w of a group
//     owns TMEM lanes 32 (w % 4) .. +31 (one weight row per thread).  A thread decodes
//     its row's KS codes to bf16 -- two codes (one byte) per lookup in a 256-entry
//     shared-memory table of bf16 pairs, replicated per lane so the lookups never
//     conflict; with 256-byte entries (whose second half is the E4M3 scale table) one
//     byte permute forms a lookup's whole offset and the table address rides in the
//     load's immediate, so a lookup costs a permute and a load (where shared memory is
//     short: 128-byte entries, or byte-permute lookups of two 8-entry byte tables) --
//     multiplies them by the block scale (exact) and writes them into TMEM with
//     tcgen05.st: the MMA's A operand lives in tensor memory, so the dequantised
//     weights never pass through shared memory;
//   * warp 1 (and warp 3 in the small variant): MMA issue, tcgen05.mma kind::f16 with
//     A from TMEM and B (tokens) from shared memory, fp32 accumulators in TMEM;
//   * the last four warps: epilogue (TMEM -> registers, x tensor scale, -> bf16 rows).
// Persistent CTAs walk the tiles round robin; in the small tiles the last partial wave is
// cut along K (SegWalk) so that no CTA decodes a whole tile alone while the others idle,
// the part that completes a split tile adding the fp32 partials in part order.
// Every wait is bounded; an expired wait sets a status bit and the CTA unwinds.
#include "kernels.cuh"

namespace moe {

namespace {

// Shared-window address at which a kernel's dynamic shared memory starts when it has no
// static shared memory: right after the per-block reserved shared memory (1 KB on
// sm_100-class GPUs; the launcher checks the device attribute, the kernel its own
// base).  The LUT-2 decode addresses its table as an immediate from it.
constexpr uint32_t kDynSmemBase = 1024;

struct NvParams {
  const int4* items;          // {group, row0, rows, 0}
  const int32_t* item_count;  // device
  int max_items;
  uint16_t* y;                // [rows_total][N]
  const float* gs;            // [G][S] tensor scales, or null (1.0)
  int gs_segments;            // S: equal row segments of N with their own tensor scale
  int N, K, G, rows_total;
  uint32_t* status;
  int early;  // 1: the tile plan was written two or more launches back
  int32_t* share_cnt;   // [kShareSlots], zero between launches
  float* share_part;    // [kShareSlots][2][BN][128]
};

// A CTA's sequence of segments: stage ranges [kb0, kb1) of tiles (tile L = n-tile
// L % n_tiles of work item L / n_tiles).  The full waves -- W = total / P tiles per CTA,
// P = gridDim.x -- go round robin (tiles c, c + P, ..., whole; TileWalk).  Without a
// split tail the R = total - W P tiles left go one per CTA as well.  A CTA's rate is
// bound by its own decoding, so a CTA left alone in that last partial wave does not
// speed up; with the split tail each of those R tiles is cut into S = min(4, P / R, nk)
// K parts, one per CTA (CTA c < R S takes part c % S of tile W P + c / S), and the
// part that completes last adds the S fp32 partials in part order (the result does
// not depend on the order the parts finish in).
struct SegWalk {
  TileWalk tw;
  const int4* items;
  long long main_total, total;
  int nk, n_tiles, kb0, kb1, nt;
  int parts, part, tail_tile;  // tail unit: S, its part, r (tile W P + r)
  int phase;                   // 0 full waves, 1 the tail unit, 2 done
  int4 cur;
  __device__ __forceinline__ SegWalk(const int4* it, long long tot, int ntiles, int nk_,
                                     bool split_tail)
      : tw(it, split_tail ? tot / gridDim.x * gridDim.x : tot, ntiles), items(it),
        main_total(split_tail ? tot / gridDim.x * gridDim.x : tot), total(tot), nk(nk_),
        n_tiles(ntiles), kb0(0), kb1(nk_), nt(0), parts(1), part(0), tail_tile(0), phase(0),
        cur(make_int4(0, 0, 0, 0)) {
    if (tw.valid()) {
      nt = tw.nt;
      cur = tw.cur;
    } else {
      enter_tail();
    }
  }
  __device__ __forceinline__ void enter_tail() {
    phase = 2;
    const long long R = total - main_total;
    if (R <= 0) return;  // no split tail (or none left)
    long long S = static_cast<long long>(gridDim.x) / R;
    if (S > 4) S = 4;
    if (S > nk) S = nk;
    const long long c = blockIdx.x;
    if (c >= R * S) return;
    parts = static_cast<int>(S);
    tail_tile = static_cast<int>(c / S);
    part = static_cast<int>(c % S);
    kb0 = part * nk / parts;
    kb1 = (part + 1) * nk / parts;
    const long long L = main_total + tail_tile;
    cur = __ldg(items + L / n_tiles);
    nt = static_cast<int>(L % n_tiles);
    phase = 1;
  }
  __device__ __forceinline__ bool valid() const { return phase < 2; }
  __device__ __forceinline__ void next() {
    if (phase == 0) {
      tw.next();
      if (tw.valid()) {
        nt = tw.nt;
        cur = tw.cur;
      } else {
        enter_tail();
      }
    } else {
      phase = 2;
    }
  }
  // a part of a split tile (its partial goes through the slots)
  __device__ __forceinline__ bool split() const { return phase == 1 && parts > 1; }
};

__device__ __forceinline__ void nv_epi_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
}

// BN: token tile; KS: K elements per stage; CS: code/scale ring slots; NA: token ring
// slots = TMEM A buffers; ACC: accumulator buffers; ISS: MMA-issuing threads (each
// takes every ISS-th stage of a tile into its own accumulator); NG: converter groups;
// LUT: how codes are decoded: 0 = byte permutes, 1 = a shared-memory table of 128-byte
// entries, 2 = a table of 256-byte entries whose free half holds the E4M3 scale table.
template <int BN, int KS, int CS, int NA, int ACC, int ISS, int NG, int LUT>
struct NvCfg {
  static constexpr int kCodeBytes = 128 * (KS / 2);  // [128 rows][KS/2 B], swizzled
  static constexpr int kScaleBytes = 128 * 16;       // [128 rows][16 B] (256 K of scales)
  static constexpr int kCodeStage = kCodeBytes + kScaleBytes;
  static constexpr int kTokBytes = BN * KS * 2;      // [KS/64][BN rows][128 B], SW128
  static constexpr int kOffTok = 0;
  static constexpr int kOffCode = kOffTok + NA * kTokBytes;
  static constexpr int kOffBar = kOffCode + CS * kCodeStage;
  // code_full[CS], code_empty[CS], tok_full[NA], conv_full[ISS][NA], mma_done[NA],
  // acc_full[ACC], acc_empty[ACC], drain[ISS]
  static constexpr int kNumBars = 2 * CS + NA + ISS * NA + NA + 2 * ACC + ISS;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // decode table: 256 code bytes x 32 lanes x one bf16 pair, entry b of lane l at byte
  // b * 128 + 4 l (LUT 1) or b * 256 + 4 l (LUT 2, whose bytes b * 256 + 128 + 4 l hold
  // the bf16 pair of E4M3 scale byte b): every lane reads its own bank
  static constexpr int kOffLut = (kOffMisc + 16 + 255) / 256 * 256;
  static constexpr int kLutBytes = LUT == 2 ? 256 * 256 : LUT == 1 ? 256 * 128 : 0;
  static constexpr int kSmemBytes = kOffLut + kLutBytes;
  static constexpr int kAccCols = ISS * BN;          // one accumulator buffer
  static constexpr int kACols = KS / 2;              // bf16 pairs per A buffer row
  static constexpr int kTmemNeed = ACC * kAccCols + NA * kACols;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kWarps = 8 + 4 * NG;          // 4 control, 4 NG converters, 4 epilogue
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kEpiWarp0 = 4 + 4 * NG;
  static constexpr int kBlocks = KS / 16;            // E4M3 scale blocks per thread per stage
  static_assert(BN % 16 == 0 && BN <= 256, "token tile");
  static_assert(KS == 128 || KS == 256, "stage K");
  static_assert(kTmemNeed <= 512, "TMEM");
  static_assert(kSmemBytes + 1024 <= 232448, "shared memory");
  static_assert(kCodeBytes % 1024 == 0 && kTokBytes % 1024 == 0, "tile alignment");
  static_assert(ISS == 1 || ISS == 2, "issuers");
  static_assert(NG <= NA && NG <= CS && ISS <= NA, "ring slots advance by at most one lap a step");
  static_assert(KS == 128 || LUT == 0, "the table-decoding converter takes 128-K stages");
  static_assert(LUT >= 0 && LUT <= 2, "decode form");
  static_assert(kThreads <= 1024, "threads");
};

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
  uint32_t d = 0;
  d |= 1u << 4;                                 // D format: F32
  d |= 1u << 7;                                 // A format: BF16
  d |= 1u << 10;                                // B format: BF16
  d |= static_cast<uint32_t>(n >> 3) << 17;     // N >> 3
  d |= static_cast<uint32_t>(128 >> 4) << 24;   // M >> 4
  return d;
}

// Eight E2M1 codes (one 32-bit word, element j in nibble j) -> eight bf16 values, two
// per word (element 2w in the low half of word w).  Magnitudes come from two 8-entry
// byte tables (high and low byte of the bf16 pattern of 0, 0.5, 1, 1.5, 2, 3, 4, 6),
// looked up four at a time with byte permutes; the sign bits are moved into place the
// same way.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t c, uint32_t (&o)[4]) {
  const uint32_t mag = c & 0x77777777u;
  uint32_t hb0 = __byte_perm(0x3F3F3F00u, 0x40404040u, mag);
  uint32_t hb1 = __byte_perm(0x3F3F3F00u, 0x40404040u, mag >> 16);
  const uint32_t lb0 = __byte_perm(0xC0800000u, 0xC0804000u, mag);
  const uint32_t lb1 = __byte_perm(0xC0800000u, 0xC0804000u, mag >> 16);
  const uint32_t even_s = (c << 4) & 0x80808080u;  // bit 7 of byte w: sign of element 2w
  const uint32_t odd_s = c & 0x80808080u;          // bit 7 of byte w: sign of element 2w+1
  hb0 |= __byte_perm(even_s, odd_s, 0x5140);
  hb1 |= __byte_perm(even_s, odd_s, 0x7362);
  o[0] = __byte_perm(lb0, hb0, 0x5140);
  o[1] = __byte_perm(lb0, hb0, 0x7362);
  o[2] = __byte_perm(lb1, hb1, 0x5140);
  o[3] = __byte_perm(lb1, hb1, 0x7362);
}

// E4M3 byte -> the same value as a pair of bf16 (exact: 4 significant bits).
__device__ __forceinline__ __nv_bfloat162 e4m3_to_bf16x2(uint32_t b) {
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  const float f = __half2float(__half(hr));
  return __float2bfloat162_rn(f);
}

// Two E4M3 scale bytes (the low byte is the first block's) -> each as a pair of equal
// bf16 values (exact: 4 significant bits), for the table-decoding converter.
__device__ __forceinline__ void e4m3x2_to_bf16x2_dup(uint32_t two, uint32_t& s0, uint32_t& s1) {
  const __half2_raw h2 =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  const __half2 h(h2);
  const __nv_bfloat162 b0 = __float2bfloat162_rn(__low2float(h));
  const __nv_bfloat162 b1 = __float2bfloat162_rn(__high2float(h));
  s0 = *reinterpret_cast<const uint32_t*>(&b0);
  s1 = *reinterpret_cast<const uint32_t*>(&b1);
}

// Eight E2M1 codes (one 32-bit word) -> four bf16 pairs times the block scale `sc`
// (a bf16 pair): byte i of the word indexes the decode table (shared-memory address
// `lut_lane` + 128 * byte: this lane's copy of the entry), the pair is multiplied by
// the scale (exact).
__device__ __forceinline__ void decode8_lut(uint32_t w, uint32_t lut_lane, uint32_t sc,
                                            uint32_t* o) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t addr = lut_lane + (__byte_perm(w, 0u, 0x4440u | i) << 7);
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(v), "r"(sc));
  }
}

// LUT 2: eight codes -> four bf16 pairs times the scale pair.  One byte permute forms
// the table offset of code byte i (byte i of the word as the offset's second byte, this
// lane's 4 l as its first), so the lookup needs no address arithmetic beyond the add
// of the table base.
// The table's shared-window address TAB is a compile-time constant (the dynamic shared
// memory starts right after the per-block reserved shared memory, kDynSmemBase; the
// kernel checks that on entry), so it rides in the load's immediate offset and a lookup
// is one byte permute + one load.
template <uint32_t TAB>
__device__ __forceinline__ void decode8_lut2(uint32_t w, uint32_t lane4, uint32_t sc,
                                             uint32_t* o) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1+%2];"
        : "=r"(v)
        : "r"(__byte_perm(w, lane4, 0x5504u | (i << 4))), "n"(TAB));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(v), "r"(sc));
  }
}

// LUT 2: the bf16 pair of E4M3 scale byte j of `word` (the table's second half).
template <uint32_t TAB>
__device__ __forceinline__ uint32_t scale_lut2(uint32_t word, int j, uint32_t lane4) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1+%2];"
      : "=r"(v)
      : "r"(__byte_perm(word, lane4, 0x5504u | (j << 4))), "n"(TAB + 128));
  return v;
}

// tcgen05.st of 16 columns; no "memory" clobber: it reads only registers, and its
// order against the other tcgen05 / mbarrier instructions (all volatile asm) is kept.
__device__ __forceinline__ void tmem_st_x16_regs(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]));
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, __nv_bfloat162 s) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&a);
  v = __hmul2(v, s);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int BN, int KS, int CS, int NA, int ACC, int ISS, int NG, int LUT>
__global__ void __launch_bounds__(NvCfg<BN, KS, CS, NA, ACC, ISS, NG, LUT>::kThreads, 1)
    k_gemm_nv(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS,
              const __grid_constant__ CUtensorMap tmX, const NvParams p) {
  using C = NvCfg<BN, KS, CS, NA, ACC, ISS, NG, LUT>;
  // An empty work list: leave before any setup (after the wait that keeps the launch
  // chain ordered), when the plan is known to be complete.
  if (p.early && *p.item_count <= 0) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0 || (LUT == 2 && smem_u32(smem) != kDynSmemBase)) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* code_full = bars;
  uint64_t* code_empty = code_full + CS;
  uint64_t* tok_full = code_empty + CS;
  uint64_t* conv_full = tok_full + NA;   // [ISS][NA]
  uint64_t* mma_done = conv_full + ISS * NA;
  uint64_t* acc_full = mma_done + NA;
  uint64_t* acc_empty = acc_full + ACC;
  uint64_t* drain = acc_empty + ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < CS; ++s) {
      mbar_init(&code_full[s], 1);                 // TMA (+tx)
      mbar_init(&code_empty[s], 4);                // the converting group's four warps
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&tok_full[s], 1);                  // TMA (+tx)
      mbar_init(&mma_done[s], 1);                  // tcgen05.commit
      for (int i = 0; i < ISS; ++i) mbar_init(&conv_full[i * NA + s], 4);
    }
    for (int b = 0; b < ACC; ++b) {
      mbar_init(&acc_full[b], ISS);
      mbar_init(&acc_empty[b], 4);
    }
    for (int i = 0; i < ISS; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmS);
    tma_prefetch_desc(&tmX);
  }
  if constexpr (LUT == 1) {
    // the decode table: entry b = the bf16 pair of code byte b (low nibble first)
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + C::kOffLut);
    for (int i = threadIdx.x; i < 256 * 32; i += C::kThreads) {
      uint32_t o[4];
      e2m1x8_to_bf16(static_cast<uint32_t>(i >> 5), o);
      lut[i] = o[0];
    }
  } else if constexpr (LUT == 2) {
    // 256-byte entries: words 0-31 the bf16 pair of code byte b, words 32-63 the
    // value of E4M3 byte b as a pair of equal bf16 (one copy per lane each)
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + C::kOffLut);
    for (int i = threadIdx.x; i < 256 * 64; i += C::kThreads) {
      const uint32_t b = static_cast<uint32_t>(i >> 6);
      if ((i & 63) < 32) {
        uint32_t o[4];
        e2m1x8_to_bf16(b, o);
        lut[i] = o[0];
      } else {
        const __nv_bfloat162 sc = e4m3_to_bf16x2(b);
        lut[i] = *reinterpret_cast<const uint32_t*>(&sc);
      }
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles = p.N / 128;
  const int nk = (p.K + KS - 1) / KS;
  int count = *p.item_count;
  if (count > p.max_items) {
    if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
    count = p.max_items;
  }
  const long long total = static_cast<long long>(count) * n_tiles;
  // The small tiles split their last partial wave (the slots hold up to kShareSlots
  // parts of at most kShareSlots tiles).
  const bool split_tail = BN == kSmallBN && p.share_cnt != nullptr &&
                          p.share_part != nullptr && gridDim.x <= kShareSlots;
  // the current tile of a walk: its group, first packed row and rows; false for an
  // empty item (skipped by every role alike) or an inconsistent one (flagged)
  auto load_item = [&](const SegWalk& w, int& g, int& row0, int& rows, int& nt) -> bool {
    const int4 it = w.cur;
    nt = w.nt;
    g = it.x;
    row0 = it.y;
    rows = it.z;
    if (rows <= 0) return false;
    if (g < 0 || g >= p.G || row0 < 0 || rows > BN || row0 + rows > p.rows_total) {
      if (threadIdx.x == 0) set_status(p.status, STATUS_BAD_PLAN);
      return false;
    }
    return true;
  };
  const uint32_t a_base = tmem + ACC * C::kAccCols;  // NA buffers of kACols columns

  if (warp == 0) {
    // ------------------------------------------------------------ codes + scales TMA
    if (lane == 0) {
      uint32_t s = 0, ph = 0;  // code ring slot and lap parity of the next stage
      for (SegWalk tw(p.items, total, n_tiles, nk, split_tail); tw.valid() && !*abort_flag; tw.next()) {
        int g, row0, rows, nt;
        if (!load_item(tw, g, row0, rows, nt)) continue;
        bool ok = true;
        for (int kb = tw.kb0; kb < tw.kb1; ++kb) {
          // the slot is free once its converters released it (a fresh barrier's
          // parity-1 phase counts as complete on the first lap)
          if (!mbar_wait(&code_empty[s], ph ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::kOffCode + s * C::kCodeStage;
          mbar_arrive_expect_tx(&code_full[s], C::kCodeStage);
          tma_load_3d(dst, &tmC, &code_full[s], kb * (KS / 2), nt * 128, g);
          tma_load_3d(dst + C::kCodeBytes, &tmS, &code_full[s], ((kb * KS) / 256) * 16,
                      nt * 128, g);
          if (++s == CS) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ token TMA
    if (lane == 0) {
      uint32_t s = 0, ph = 0;  // token ring slot and lap parity of the next stage
      for (SegWalk tw(p.items, total, n_tiles, nk, split_tail); tw.valid() && !*abort_flag; tw.next()) {
        int g, row0, rows, nt;
        if (!load_item(tw, g, row0, rows, nt)) continue;
        bool ok = true;
        for (int kb = tw.kb0; kb < tw.kb1; ++kb) {
          if (!mbar_wait(&mma_done[s], ph ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&tok_full[s], C::kTokBytes);
          tma_load_3d(smem + C::kOffTok + s * C::kTokBytes, &tmX, &tok_full[s], 0, row0,
                      kb * (KS / 64));
          if (++s == NA) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1 || (ISS == 2 && warp == 3)) {
    // ------------------------------------------------------------ MMA issuer(s)
    const int par = warp == 1 ? 0 : 1;
    if (lane == 0) {
      uint32_t it0 = 0, tc = 0;  // it0: this CTA's index of the segment's first stage
      uint32_t phases = 0;  // bit s: parity of the next phase of conv_full[par][s]
      for (SegWalk tw(p.items, total, n_tiles, nk, split_tail); tw.valid() && !*abort_flag; tw.next()) {
        int g, row0, rows, nt;
        if (!load_item(tw, g, row0, rows, nt)) continue;
        const int bn = (rows + 15) & ~15;
        const uint32_t b = tc % ACC, use = tc / ACC;
        if (tc >= ACC && !mbar_wait(&acc_empty[b], (use - 1) & 1u, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * C::kAccCols + par * BN;
        const uint32_t idesc = idesc_bf16(bn);
        bool ok = true;
        // this issuer's first stage of the segment (parity par of the tile's stage index)
        const int kb_first = ISS == 2 ? tw.kb0 + ((par - tw.kb0) & 1) : tw.kb0;
        // ring slot of the stage (index it0 + kb - kb0) and the parity of its token
        // phase, advanced by ISS stages per step (one division per segment)
        const uint32_t i0 = it0 + static_cast<uint32_t>(kb_first - tw.kb0);
        uint32_t s = i0 % NA, tph = (i0 / NA) & 1u;
        for (int kb = kb_first; kb < tw.kb1; kb += ISS) {  // this issuer's stages
          const uint32_t ph = (phases >> s) & 1u;
          phases ^= 1u << s;
          // the stage's weights are in TMEM (its converters) and its tokens have landed
          if (!mbar_wait(&conv_full[par * NA + s], ph, p.status, abort_flag) ||
              !mbar_wait(&tok_full[s], tph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_t = a_base + s * C::kACols;
          // the 16-K steps of the token tile are fixed offsets from its descriptor (the
          // start-address field holds address / 16; the tile lies below 256 KB, so
          // adding to the low word never carries out of the field)
          const uint64_t bd0 =
              smem_desc(smem_u32(smem + C::kOffTok + s * C::kTokBytes), 0, 1024, kLayoutSw128);
          const uint32_t bd_lo = static_cast<uint32_t>(bd0);
          const uint64_t bd_hi = bd0 & 0xFFFFFFFF00000000ull;
#pragma unroll
          for (int kk = 0; kk < KS / 16; ++kk) {
            const uint32_t off =
                static_cast<uint32_t>(((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4);
            mma_bf16_ts(d_tmem, a_t + kk * 8, bd_hi | (bd_lo + off), idesc,
                        kb != kb_first || kk != 0);
          }
          tc_commit(&mma_done[s]);
          s += ISS;
          if (s >= NA) {
            s -= NA;
            tph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[b]);
        ++tc;
        it0 += static_cast<uint32_t>(tw.kb1 - tw.kb0);
      }
    }
  } else if (warp >= 4 && warp < C::kEpiWarp0) {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;            // TMEM lane quarter = weight rows 32q .. 32q+31
    const int cg = (warp - 4) >> 2;    // converter group: stages it with it % NG == cg
    const int r = q * 32 + lane;       // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t lut_lane = smem_u32(smem + C::kOffLut) + 4u * lane;
    const uint32_t lane4 = 4u * lane;
    constexpr uint32_t kTab = kDynSmemBase + C::kOffLut;  // the table's shared address
    // This group's stages have global indices cg, cg + NG, cg + 2 NG, ... across all
    // tiles, so their ring slots and phase parities advance by NG per stage.
    uint32_t s = cg, ps = 0;    // TMEM A buffer / token ring (NA slots)
    uint32_t cs = cg, pc = 0;   // code ring (CS slots)
    uint32_t it0 = 0;           // this CTA's index of the segment's first stage
    bool ok = true;
    // With two or more spare TMEM buffers (NA >= NG + 2) a group waits for a stage's
    // TMEM stores, and releases the stage to the MMA, only after its next stage's codes
    // are in registers, so the store latency overlaps those loads.  (With NA == NG the
    // next stage reuses the deferred stage's own buffer -- a deadlock; with one spare
    // buffer the deferral serialises the groups behind the MMAs: measured slower.)
    constexpr bool kDefer = NA >= NG + 2;
    int pend = -1;  // conv_full barrier of the stage whose TMEM stores are in flight
    for (SegWalk tw(p.items, total, n_tiles, nk, split_tail); tw.valid() && ok && !*abort_flag;
         tw.next()) {
      int g, row0, rows, nt;
      if (!load_item(tw, g, row0, rows, nt)) {
        continue;
      }
      for (int kb = tw.kb0 + static_cast<int>((cg + NG - it0 % NG) % NG); kb < tw.kb1;
           kb += NG) {
        // the TMEM A buffer of this stage is free once the MMAs of stage it - NA are
        // done (their commit; the first pass finds the fresh barrier's parity-1 phase
        // complete); the code slot once its TMA has landed.  The whole warp waits.
        const bool w_ok = mbar_wait(&mma_done[s], ps ^ 1u, p.status, abort_flag) &&
                          mbar_wait(&code_full[cs], pc, p.status, abort_flag);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* cbase = smem + C::kOffCode + cs * C::kCodeStage;
        // this thread's codes: row r of KS/2 bytes, in 16-byte chunks stored at
        // chunk ^ swizzle(r)
        constexpr int kChunks = KS / 32;
        uint4 cw[kChunks];
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int phys = KS == 256 ? (j ^ (r & 7)) : (j ^ ((r >> 1) & 3));
          cw[j] = *reinterpret_cast<const uint4*>(cbase + r * (KS / 2) + phys * 16);
        }
        // this thread's scale bytes: row r of the 16-byte scale row; a 128-K stage uses
        // the half of the 256 K it covers
        const uint4 sv = *reinterpret_cast<const uint4*>(cbase + C::kCodeBytes + r * 16);
        const int sbyte0 = KS == 128 ? (kb & 1) * 8 : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&code_empty[cs]);
        if (kDefer && pend >= 0) {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&conv_full[pend]);
          pend = -1;
        }
        const uint32_t col0 = a_base + s * C::kACols;
        if constexpr (LUT == 2) {
          // a 128-K stage: scale bytes 0-7 (even 128-K step) or 8-15 (odd) of the row
          const uint32_t s_lo = (kb & 1) ? sv.z : sv.x;
          const uint32_t s_hi = (kb & 1) ? sv.w : sv.y;
#pragma unroll
          for (int bp = 0; bp < C::kBlocks / 2; ++bp) {  // two 16-element blocks = chunk bp
            const uint32_t sw = bp < 2 ? s_lo : s_hi;
            const uint32_t sc0 = scale_lut2<kTab>(sw, 2 * (bp & 1), lane4);
            const uint32_t sc1 = scale_lut2<kTab>(sw, 2 * (bp & 1) + 1, lane4);
            const uint4 cv = cw[bp];
            uint32_t o[16];
            decode8_lut2<kTab>(cv.x, lane4, sc0, o);
            decode8_lut2<kTab>(cv.y, lane4, sc0, o + 4);
            decode8_lut2<kTab>(cv.z, lane4, sc1, o + 8);
            decode8_lut2<kTab>(cv.w, lane4, sc1, o + 12);
            tmem_st_x16_regs(lane_base + col0 + bp * 16, o);
          }
        } else if constexpr (LUT == 1) {
          // a 128-K stage: scale bytes 0-7 (even 128-K step) or 8-15 (odd) of the row
          const uint32_t s_lo = (kb & 1) ? sv.z : sv.x;
          const uint32_t s_hi = (kb & 1) ? sv.w : sv.y;
#pragma unroll
          for (int bp = 0; bp < C::kBlocks / 2; ++bp) {  // two 16-element blocks = chunk bp
            uint32_t sc0, sc1;
            e4m3x2_to_bf16x2_dup((bp < 2 ? s_lo : s_hi) >> (16 * (bp & 1)), sc0, sc1);
            const uint4 cv = cw[bp];
            uint32_t o[16];
            decode8_lut(cv.x, lut_lane, sc0, o);
            decode8_lut(cv.y, lut_lane, sc0, o + 4);
            decode8_lut(cv.z, lut_lane, sc1, o + 8);
            decode8_lut(cv.w, lut_lane, sc1, o + 12);
            tmem_st_x16_regs(lane_base + col0 + bp * 16, o);
          }
        } else {
#pragma unroll
          for (int blk = 0; blk < C::kBlocks; ++blk) {
            const int sb = sbyte0 + blk;
            const uint32_t sw = sb < 4 ? sv.x : sb < 8 ? sv.y : sb < 12 ? sv.z : sv.w;
            const __nv_bfloat162 sc = e4m3_to_bf16x2((sw >> (8 * (sb & 3))) & 0xFFu);
            // 16 elements = 8 code bytes = two 32-bit words of chunk blk / 2
            const uint4 cv = cw[blk >> 1];
            const uint32_t w0 = (blk & 1) ? cv.z : cv.x;
            const uint32_t w1 = (blk & 1) ? cv.w : cv.y;
            uint32_t o[8];
            uint32_t t[4];
            e2m1x8_to_bf16(w0, t);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = bf16x2_mul(t[i], sc);
            e2m1x8_to_bf16(w1, t);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[4 + i] = bf16x2_mul(t[i], sc);
            tmem_st_32x32b_x8(lane_base + col0 + blk * 8, o);
          }
        }
        if constexpr (kDefer) {
          pend = (ISS == 2 ? (kb & 1) : 0) * NA + s;
        } else {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&conv_full[(ISS == 2 ? (kb & 1) : 0) * NA + s]);
        }
        s += NG;
        if (s >= NA) {
          s -= NA;
          ps ^= 1u;
        }
        cs += NG;
        if (cs >= CS) {
          cs -= CS;
          pc ^= 1u;
        }
      }
      it0 += static_cast<uint32_t>(tw.kb1 - tw.kb0);
    }
    tmem_st_wait();  // (also on the abort path: no TMEM store outlives the role)
    if (kDefer && pend >= 0 && ok && !*abort_flag) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv_full[pend]);
    }
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    // per-CTA scratch of the split tail: the accumulator wait's verdict and a split
    // tile's arrival count, each handed to all four epilogue warps at a named barrier
    volatile int* go = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile int* arrived = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 12);
    uint32_t tc = 0;
    // (with a split tail the warps leave the loop only together, on the collective
    // wait's verdict -- an abort makes that wait fail -- never one by one on the flag)
    for (SegWalk tw(p.items, total, n_tiles, nk, split_tail); tw.valid() && (split_tail || !*abort_flag);
         tw.next()) {
      int g, row0, rows, nt;
      if (!load_item(tw, g, row0, rows, nt)) continue;
      const uint32_t b = tc % ACC, use = tc / ACC;
      int w_ok = 1;
      if (split_tail) {  // the four warps meet at named barriers: they decide together
        if (q == 0 && lane == 0) *go = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
        nv_epi_bar();
        w_ok = *go;
        nv_epi_bar();
      } else {
        if (lane == 0) w_ok = mbar_wait(&acc_full[b], use & 1u, p.status, abort_flag);
        w_ok = __shfl_sync(0xFFFFFFFFu, w_ok, 0);
      }
      if (!w_ok) break;
      tc_fence_after();
      const int n = nt * 128 + q * 32 + lane;
      float gsc = 1.0f;
      if (p.gs) gsc = __ldg(p.gs + static_cast<size_t>(g) * p.gs_segments +
                            n / (p.N / p.gs_segments));
      uint16_t* ycol = p.y + static_cast<size_t>(row0) * p.N + n;
      const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * C::kAccCols;
      // with two issuers, which of the even-stage / odd-stage accumulators this
      // segment wrote (a one-stage segment writes one)
      const bool two = tw.kb1 - tw.kb0 > 1;
      const bool has_even = ISS == 1 || two || (tw.kb0 & 1) == 0;
      const bool has_odd = ISS == 2 && (two || (tw.kb0 & 1) == 1);
      const bool shared = split_tail && tw.split();
      // a split tile's part: slot r S + part of the partials, counter r
      float* mine = shared ? p.share_part +
                                 (static_cast<size_t>(tw.tail_tile * tw.parts + tw.part) * BN) *
                                     128 + q * 32 + lane
                           : nullptr;
      for (int c0 = 0; c0 < rows; c0 += 16) {
        uint32_t rr[16];
        float v[16];
        if (has_even) {
          tmem_ld_32x32b_x16(acc + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rr[i]);
        }
        if (has_odd) {  // even-stage + odd-stage sums, in that order
          tmem_ld_32x32b_x16(acc + BN + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = has_even ? v[i] + __uint_as_float(rr[i])
                                                       : __uint_as_float(rr[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (c0 + i < rows) {
            if (shared) {
              mine[static_cast<size_t>(c0 + i) * 128] = v[i];
            } else {
              const __nv_bfloat16 hv = __float2bfloat16_rn(v[i] * gsc);
              ycol[static_cast<size_t>(c0 + i) * p.N] = *reinterpret_cast<const uint16_t*>(&hv);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++tc;
      if (shared) {
        // publish this part, count the arrival; the part that completes the tile adds
        // all S partials, in part order
        __threadfence();
        nv_epi_bar();
        if (q == 0 && lane == 0) *arrived = atomicAdd(&p.share_cnt[tw.tail_tile], 1);
        nv_epi_bar();
        if (*arrived == tw.parts - 1) {
          __threadfence();
          const float* first = p.share_part +
                               (static_cast<size_t>(tw.tail_tile * tw.parts) * BN) * 128 +
                               q * 32 + lane;
          for (int r = 0; r < rows; ++r) {
            float sum = __ldcg(first + static_cast<size_t>(r) * 128);
            for (int j = 1; j < tw.parts; ++j)
              sum += __ldcg(first + (static_cast<size_t>(j) * BN + r) * 128);
            const __nv_bfloat16 hv = __float2bfloat16_rn(sum * gsc);
            ycol[static_cast<size_t>(r) * p.N] = *reinterpret_cast<const uint16_t*>(&hv);
          }
          if (q == 0 && lane == 0) p.share_cnt[tw.tail_tile] = 0;  // for the next launch
        }
        nv_epi_bar();  // *arrived is read by all before a later part writes it
      }
    }
  }

  // After an abort, each MMA issuer waits (briefly, bounded) until the MMAs it issued
  // have completed, so that TMEM is not released under them; TMA loads still in flight
  // are not waited for (best effort).
  if ((warp == 1 || (ISS == 2 && warp == 3)) && lane == 0 && *abort_flag) {
    uint64_t* db = &drain[warp == 1 ? 0 : 1];
    tc_commit(db);
    mbar_wait_drain(db, 0);
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side -------

template <int BN, int KS, int CS, int NA, int ACC, int ISS, int NG, int LUT>
cudaError_t launch_nv_one(const NvGemmLaunch& a, int v, cudaStream_t st) {
  using C = NvCfg<BN, KS, CS, NA, ACC, ISS, NG, LUT>;
  auto kern = k_gemm_nv<BN, KS, CS, NA, ACC, ISS, NG, LUT>;
  const int max_items = a.max_items[v];
  const long long tiles = static_cast<long long>(max_items) * (a.N / 128);
  if (tiles == 0) return cudaSuccess;
  static unsigned long long attr_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || attr_ctx[dev] != ctx) {
    if (LUT == 2) {  // the table-address immediate assumes this reserved size
      int reserved = -1;
      e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
      if (e != cudaSuccess) return e;
      if (reserved != static_cast<int>(kDynSmemBase)) return cudaErrorNotSupported;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_ctx[dev] = current_context_id();
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  CUtensorMap tmC, tmS, tmX;
  if (nv_encode_maps(a, KS, BN, &tmC, &tmS, &tmX) != MOE_OK) return cudaErrorInvalidValue;
  NvParams p{};
  p.items = a.items[v];
  p.item_count = a.item_counts + v;
  p.max_items = max_items;
  p.y = a.y;
  p.gs = a.gs;
  p.gs_segments = a.gs_segments;
  p.N = a.N;
  p.K = a.K;
  p.G = a.G;
  p.rows_total = a.rows_total;
  p.status = a.status;
  // every variant after the first follows the first's launch, which follows the plan
  p.early = v > 0 ? 1 : 0;
  p.share_cnt = a.share_cnt;
  p.share_part = a.share_part;
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  return launch_k(kern, grid, C::kThreads, C::kSmemBytes, st, tmC, tmS, tmX, p);
}

}  // namespace

// Tensor maps: codes as {K/2 bytes, N rows, G} (box {KS/2, 128, 1}, swizzled so that
// each converter thread's 16-byte chunks fall in distinct banks), scales as {K/16
// bytes, N rows, G} (box {16, 128, 1}: 256 K of scales), bf16 token rows as {64
// elements, rows, K/64} (box {64, BN, KS/64}, 128B-swizzled: the MMA's K-major layout).
int nv_encode_maps(const NvGemmLaunch& a, int ks, int bn, CUtensorMap* tmC, CUtensorMap* tmS,
                   CUtensorMap* tmX) {
  EncodeTiledFn enc = get_encode_tiled_fn();
  if (!enc) return MOE_ERR_CUDA;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.K / 2), static_cast<cuuint64_t>(a.N),
                          static_cast<cuuint64_t>(a.G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.K / 2),
                             static_cast<cuuint64_t>(a.N) * static_cast<cuuint64_t>(a.K / 2)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(ks / 2), 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.w_codes), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            ks == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.K / 16), static_cast<cuuint64_t>(a.N),
                          static_cast<cuuint64_t>(a.G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.K / 16),
                             static_cast<cuuint64_t>(a.N) * static_cast<cuuint64_t>(a.K / 16)};
    cuuint32_t box[3] = {16, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.w_scales), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(a.rows_total > 0 ? a.rows_total : 1),
                          static_cast<cuuint64_t>(a.K / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.K) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(bn), static_cast<cuuint32_t>(ks / 64)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.act), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Variants by the tile plan's lists (same row bounds as the MXFP4 GEMM's); 128-K
// stages, four converter groups (three in the large variant):
//   small  rows <= 16:  8 code slots, 7 token/TMEM slots, 2 issuers, table decoding;
//   medium rows <= 64:  6 code slots, 5 token/TMEM slots, table decoding;
//   mid    rows <= 128: 4 code slots, 4 token/TMEM slots, table decoding;
//   large  rows <= 224: 3 slots (a 224-row bf16 token tile is 56 KB per 128 K), one
//          accumulator (224 of TMEM's 512 columns), byte-permute decoding (no shared
//          memory left for the table).
cudaError_t launch_grouped_gemm_nv(const NvGemmLaunch& a, cudaStream_t st) {
  cudaError_t e = launch_nv_one<kSmallBN, 128, 8, 7, 2, 2, 4, 2>(a, 0, st);
  if (e != cudaSuccess || a.max_group_rows <= kSmallBN) return e;
  e = launch_nv_one<kMediumBN, 128, 6, 5, 2, 1, 4, 2>(a, 1, st);
  if (e != cudaSuccess || a.max_group_rows <= kMediumBN) return e;
  e = launch_nv_one<kMidBN, 128, 4, 4, 2, 1, 4, 1>(a, 2, st);
  if (e != cudaSuccess || a.max_group_rows <= kMidBN) return e;
  return launch_nv_one<kLargeBN, 128, 3, 3, 1, 1, 3, 0>(a, 3, st);
}

}  // namespace moe
