// a1 top-k routing, a2 histogram / exclusive scan / permutation, a8 tile plan.
//
// Routing follows the TopK step of "Pushing the Limits of Serving DeepSeek-V4-Pro"
// (LMSYS, H20), §3.2; the per-expert M that shapes the grouped GEMMs comes from the
// routing histogram (§3.3); packing tokens by expert ahead of the expert GEMMs is
// Optimization 14 ("direct route preplan") of the GB10 optimisation report.
//
// Everything here is integer-exact and deterministic: ranks inside an expert's
// segment come from per-warp bit masks and prefix sums, never from the order in
// which atomics happen to land.
#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------- a1: route -------
//
// One warp per token.  Lane l holds logits l, l+32, ... (coalesced loads) as
// order-preserving unsigned keys (key(a) > key(b) <=> a > b for finite floats, -0
// folded onto +0 so that equal values have equal keys; key 0 marks a taken or absent
// slot, which no finite logit maps to).  k rounds: each lane's best untaken key
// (lowest slot on ties), the warp's largest key (redux.sync max), then the lowest
// expert index among the lanes holding it (redux.sync min) -- ties to the lower
// index.  On return lane j < k holds the j-th selection (expert, renormalised weight).
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k,
                                            int lane, int& my_e, float& my_w) {
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(row[e]) : 0u;
  }
  float my_v = 0.f;
  my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (key[i] > bk) {  // ascending slot: strict > keeps the lower index
        bk = key[i];
        bi = i;
      }
    }
    const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t cand = bk == mk ? static_cast<uint32_t>(lane + 32 * bi) : 0xFFFFFFFFu;
    const uint32_t be = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (static_cast<int>(be & 31u) == lane) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == static_cast<int>(be >> 5)) key[i] = 0u;
    }
    if (lane == j) {
      my_v = key_logit(mk);
      my_e = static_cast<int>(be);
    }
  }
  // weights: exp(l_j - l_0) / sum over the selected
  float l0 = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  float ex = lane < k ? expf(my_v - l0) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  my_w = ex / s;
}

template <int EPL>
__global__ void __launch_bounds__(256) k_route(const float* __restrict__ logits, int T, int E,
                                               int k, int32_t* __restrict__ idx,
                                               float* __restrict__ w, uint32_t* clear_status) {
  pdl_wait();
  pdl_trigger();
  // the first kernel of a call clears the call's status word
  if (clear_status && blockIdx.x == 0 && threadIdx.x == 0) *clear_status = 0;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  int e;
  float wt;
  route_token<EPL>(logits + static_cast<size_t>(t) * E, E, k, lane, e, wt);
  if (lane < k) {
    idx[static_cast<size_t>(t) * k + lane] = e;
    w[static_cast<size_t>(t) * k + lane] = wt;
  }
}

// ---------------------------------------------------------------- a2: histogram ---
//
// Tokens are processed in blocks of kPermTokens (one per thread).  Pass 1 counts
// per (block, expert); pass 2 scans those counts per expert and over experts;
// pass 3 recomputes each warp's masks and writes every routed row's position.
constexpr int kPermTokens = 256;

__global__ void __launch_bounds__(kPermTokens) k_hist_block(const int32_t* __restrict__ idx,
                                                            int T, int E, int k,
                                                            int32_t* __restrict__ blockcnt,
                                                            uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t s_cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * kPermTokens + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      int e = idx[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) {
        set_status(status, STATUS_BAD_INDEX);
        continue;
      }
      atomicAdd(&s_cnt[e], 1);  // integer count: order-independent result
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blockcnt[static_cast<size_t>(blockIdx.x) * E + e] = s_cnt[e];
}

// One CTA.  blockbase[b][e] = sum of blockcnt[b'][e] for b' < b; counts; offsets
// over G = E + has_shared groups (the shared group holds T rows).
__global__ void __launch_bounds__(1024) k_scan(const int32_t* __restrict__ blockcnt, int nblk,
                                               int T, int E, int has_shared,
                                               int32_t* __restrict__ blockbase,
                                               int32_t* __restrict__ counts,
                                               int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t s_part[1024];
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x;
  const int G = E + has_shared;
  // per-expert totals over blocks (thread per expert, E <= 1024)
  int32_t total = 0;
  if (tid < E) {
    for (int b = 0; b < nblk; ++b) {
      int32_t c = blockcnt[static_cast<size_t>(b) * E + tid];
      blockbase[static_cast<size_t>(b) * E + tid] = total;
      total += c;
    }
    counts[tid] = total;
  }
  int32_t gsize = tid < E ? total : (tid == E && has_shared ? T : 0);
  // exclusive scan of gsize over threads 0..1023 (G <= 1025: group 1024 handled below)
  int32_t x = gsize;
  const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int32_t y = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int32_t z = __shfl_up_sync(0xFFFFFFFFu, y, off);
      if (lane >= off) y += z;
    }
    s_warp[lane] = y;  // inclusive over warps
  }
  __syncthreads();
  int32_t incl = x + (wid > 0 ? s_warp[wid - 1] : 0);
  s_part[tid] = incl;
  if (tid < G) offsets[tid] = incl - gsize;
  __syncthreads();
  if (tid == 0) {
    int32_t end = s_part[1023];
    if (G == 1025) {  // E == 1024 with a shared expert: group 1024 = the shared rows
      offsets[1024] = end;
      offsets[1025] = end + T;
    } else {
      offsets[G] = end;
    }
  }
}

__global__ void __launch_bounds__(kPermTokens) k_permute_block(
    const int32_t* __restrict__ idx, int T, int E, int k, const int32_t* __restrict__ blockbase,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ inv) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t s_bits[];  // [8 warps][E] masks, then [8][E] warp bases
  constexpr int kWarps = kPermTokens / 32;
  int32_t* s_wbase = reinterpret_cast<int32_t*>(s_bits + kWarps * E);
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) s_bits[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int t = blockIdx.x * kPermTokens + threadIdx.x;
  const bool live = t < T;
  if (live) {
    for (int j = 0; j < k; ++j) {
      int e = idx[static_cast<size_t>(t) * k + j];
      if (e >= 0 && e < E) atomicOr(&s_bits[wid * E + e], 1u << lane);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = 0;
    for (int w = 0; w < kWarps; ++w) {
      s_wbase[w * E + e] = run;
      run += __popc(s_bits[w * E + e]);
    }
  }
  __syncthreads();
  if (live) {
    const uint32_t lt = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      int e = idx[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) continue;
      int32_t pos = offsets[e] + blockbase[static_cast<size_t>(blockIdx.x) * E + e] +
                    s_wbase[wid * E + e] + __popc(s_bits[wid * E + e] & lt);
      int32_t src = t * k + j;
      perm_src[pos] = src;
      inv[src] = pos;
    }
  }
}

// ---------------------------------------------------------------- a8: tile plan ---
//
// Per group g with M = offsets[g+1] - offsets[g] rows (the effective M the pages tune
// for): M <= kSmallBN -> one small-M item (padded only to 16 tokens, never to a large
// tile); M <= kMediumBN -> one medium item; larger groups are split into
// ceil(M / C) near-equal chunks (multiples of 16 rows except the last; C = the plan's
// chunk_rows, kLargeBN by default, a tunable of the exact-shape tuning of LMSYS-H20
// §3.3), which go to the mid kernel when they are at most kMidBN rows and to the large
// kernel otherwise.  Items are {group, row0, rows, 0}.  One CTA of 1024 threads; each
// thread owns a contiguous run of groups; positions come from block-wide scans, so
// the lists are in group order (or with the last group first, below) and
// deterministic.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* s_warp,
                                                        int32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int32_t y = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int32_t z = __shfl_up_sync(0xFFFFFFFFu, y, off);
      if (lane >= off) y += z;
    }
    s_warp[lane] = y;
  }
  __syncthreads();
  const int32_t excl = x - v + (wid > 0 ? s_warp[wid - 1] : 0);
  *total = s_warp[31];
  __syncthreads();
  return excl;
}

// Variant of a group with m > 0 rows and the chunking of the two chunked variants
// (chunks of at most `chunk` rows).
__device__ __forceinline__ int plan_variant(int32_t m, int32_t chunk, int32_t& nch,
                                            int32_t& base) {
  nch = 1;
  base = m;
  if (m <= kSmallBN) return 0;
  if (m <= kMediumBN) return 1;
  nch = (m + chunk - 1) / chunk;
  base = ((m + nch - 1) / nch + 15) / 16 * 16;
  return base <= kMidBN ? 2 : 3;
}

// Builds the per-variant item lists from group offsets (global or shared memory).
// Called by all 1024 threads of one CTA.  last_first: the last group's items lead
// their list, the others following in group order (the decode path puts its shared
// expert first: measured 1% faster with NVFP4 weights at 7 tokens, W2 0.148 vs 0.152
// ms; no change with MXFP4); otherwise the lists follow the group order.
__device__ void plan_groups(const int32_t* offsets, int G, const PlanOut& plan,
                            uint32_t* status, int32_t* s_warp, bool last_first) {
  const int tid = threadIdx.x;
  if (plan.share_cnt)
    for (int i = tid; i < kShareSlots; i += blockDim.x) plan.share_cnt[i] = 0;
  int32_t chunk = plan.chunk_rows == 0 ? kLargeBN : plan.chunk_rows;
  if (chunk < kMinChunkRows || chunk > kLargeBN || chunk % 16 != 0) {  // host-checked
    if (tid == 0) set_status(status, STATUS_BAD_PLAN);
    chunk = kLargeBN;
  }
  const int per = (G + 1023) / 1024;
  const int g0 = tid * per, g1 = min(G, g0 + per);
  int32_t n[kNumVariants] = {0, 0, 0, 0};
  // list position j holds group gj(j): the identity, or the last group first
  auto gj = [&](int j) { return last_first ? (j == 0 ? G - 1 : j - 1) : j; };
  for (int j = g0; j < g1; ++j) {
    const int g = gj(j);
    int32_t m = offsets[g + 1] - offsets[g];
    if (m < 0) set_status(status, STATUS_BAD_PLAN);
    if (m <= 0) continue;
    int32_t nch, base;
    const int v = plan_variant(m, chunk, nch, base);  // (not folded into n[...] += nch: the
    n[v] += nch;                               // right operand would be read first)
  }
  int32_t pos[kNumVariants], tot[kNumVariants];
#pragma unroll
  for (int v = 0; v < kNumVariants; ++v) pos[v] = block_exclusive_scan(n[v], s_warp, &tot[v]);
  for (int j = g0; j < g1; ++j) {
    const int g = gj(j);
    int32_t r0 = offsets[g], m = offsets[g + 1] - r0;
    if (m <= 0) continue;
    int32_t nch, base;
    const int v = plan_variant(m, chunk, nch, base);
    for (int c = 0; c < nch; ++c) {
      int32_t a = c * base, b = min(m, a + base);
      const int32_t p = pos[v]++;
      if (p >= plan.capacity[v]) {  // cannot happen with consistent offsets; never write past
        set_status(status, STATUS_BAD_PLAN);
        continue;
      }
      plan.items[v][p] = make_int4(g, r0 + a, a < m ? b - a : 0, 0);
    }
  }
  if (tid == 0) {
#pragma unroll
    for (int v = 0; v < kNumVariants; ++v) plan.counts[v] = min(tot[v], plan.capacity[v]);
  }
}

__global__ void __launch_bounds__(1024) k_plan(const int32_t* __restrict__ offsets, int G,
                                               const PlanOut plan, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t s_warp[32];
  plan_groups(offsets, G, plan, status, s_warp, false);
}

// ------------------------------------------------ a1 + a2 + a8 in one CTA (small T) ---
//
// The decode path ("route preplan", GB10 report Optimization 14): for T <= kPrepMaxT
// one CTA routes every token, builds per-expert token bit masks, the counts, the
// offsets (block scan), each routed row's position (its token's rank among the
// expert's tokens = popcount of the mask below it) and the tile plan.  One launch
// instead of five; same results as the multi-kernel path.
template <int EPL>
__global__ void __launch_bounds__(1024) k_prep_small(
    const float* __restrict__ logits, int T, int E, int k, int has_shared,
    int32_t* __restrict__ idx, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src, int32_t* __restrict__ inv,
    const PlanOut plan, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  // the first kernel of a call clears the call's status word; every later set of a
  // status bit in this kernel comes after the barriers below
  if (threadIdx.x == 0) *status = 0;
  constexpr int kWords = kPrepMaxT / 32;
  __shared__ uint32_t s_mask[1024 * kWords];  // [expert][token word]
  __shared__ int32_t s_idx[kPrepMaxT * 16];
  __shared__ int32_t s_off[1026];
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int G = E + has_shared;
  for (int i = tid; i < E * kWords; i += 1024) s_mask[i] = 0;
  __syncthreads();
  for (int t = wid; t < T; t += 32) {
    int e;
    float wt;
    route_token<EPL>(logits + static_cast<size_t>(t) * E, E, k, lane, e, wt);
    if (lane < k) {
      idx[t * k + lane] = e;
      w[t * k + lane] = wt;
      s_idx[t * k + lane] = e;
      atomicOr(&s_mask[e * kWords + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();
  // counts and offsets (thread-contiguous runs of groups, block scan)
  const int per = (G + 1023) / 1024;
  const int g0 = tid * per, g1 = min(G, g0 + per);
  int32_t run = 0;
  for (int g = g0; g < g1; ++g) {
    int32_t c = 0;
    if (g < E) {
#pragma unroll
      for (int i = 0; i < kWords; ++i) c += __popc(s_mask[g * kWords + i]);
      counts[g] = c;
    } else {
      c = T;  // the shared expert: one row per token
    }
    run += c;
  }
  int32_t total;
  int32_t pos = block_exclusive_scan(run, s_warp, &total);
  for (int g = g0; g < g1; ++g) {
    s_off[g] = pos;
    offsets[g] = pos;
    pos += g < E ? counts[g] : T;
  }
  if (tid == 0) {
    s_off[G] = total;
    offsets[G] = total;
  }
  __syncthreads();
  // positions: rank of token t among expert e's tokens
  for (int i = tid; i < T * k; i += 1024) {
    const int t = i / k, e = s_idx[i];
    int32_t rank = 0;
#pragma unroll
    for (int wd = 0; wd < kWords; ++wd) {
      const uint32_t m = s_mask[e * kWords + wd];
      if (wd < (t >> 5)) rank += __popc(m);
      else if (wd == (t >> 5)) rank += __popc(m & ((1u << (t & 31)) - 1u));
    }
    const int32_t p = s_off[e] + rank;
    perm_src[p] = i;
    inv[i] = p;
  }
  plan_groups(s_off, G, plan, status, s_warp, has_shared != 0);
}

// ---------------------------------------------------------------- launchers -------

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         uint32_t* clear_status, cudaStream_t st) {
  const int warps = 8;
  dim3 grid((T + warps - 1) / warps), block(32 * warps);
  const int epl = (E + 31) / 32;
#define MOE_ROUTE_CASE(N) \
  if (epl <= N) {         \
    return launch_k(k_route<N>, grid, block, 0, st, logits, T, E, k, idx, w, clear_status); \
  }
  MOE_ROUTE_CASE(1)
  MOE_ROUTE_CASE(2)
  MOE_ROUTE_CASE(4)
  MOE_ROUTE_CASE(8)
  MOE_ROUTE_CASE(12)
  MOE_ROUTE_CASE(16)
  MOE_ROUTE_CASE(32)
#undef MOE_ROUTE_CASE
  return cudaErrorInvalidValue;
}

int perm_blocks(int T) { return (T + kPermTokens - 1) / kPermTokens; }

cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int has_shared,
                           int32_t* blockcnt, int32_t* blockbase, int32_t* counts,
                           int32_t* offsets, int32_t* perm_src, int32_t* inv, uint32_t* status,
                           cudaStream_t st) {
  const int nblk = perm_blocks(T);
  cudaError_t e = launch_k(k_hist_block, nblk, kPermTokens, E * sizeof(int32_t), st, idx, T, E,
                           k, blockcnt, status);
  if (e != cudaSuccess) return e;
  e = launch_k(k_scan, 1, 1024, 0, st, blockcnt, nblk, T, E, has_shared, blockbase, counts,
               offsets);
  if (e != cudaSuccess) return e;
  size_t smem = 2 * (kPermTokens / 32) * E * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(k_permute_block,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_k(k_permute_block, nblk, kPermTokens, smem, st, idx, T, E, k, blockbase, offsets,
                  perm_src, inv);
}

cudaError_t launch_plan(const int32_t* offsets, int G, PlanOut plan, uint32_t* status,
                        cudaStream_t st) {
  return launch_k(k_plan, 1, 1024, 0, st, offsets, G, plan, status);
}

cudaError_t launch_prep_small(const float* logits, int T, int E, int k, int has_shared,
                              int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                              int32_t* perm_src, int32_t* inv, PlanOut plan, uint32_t* status,
                              cudaStream_t st) {
  if (T > kPrepMaxT) return cudaErrorInvalidValue;
  const int epl = (E + 31) / 32;
#define MOE_PREP_CASE(N)                                                                    \
  if (epl <= N) {                                                                           \
    return launch_k(k_prep_small<N>, 1, 1024, 0, st, logits, T, E, k, has_shared, idx, w,   \
                    counts, offsets, perm_src, inv, plan, status);                          \
  }
  MOE_PREP_CASE(1)
  MOE_PREP_CASE(2)
  MOE_PREP_CASE(4)
  MOE_PREP_CASE(8)
  MOE_PREP_CASE(12)
  MOE_PREP_CASE(16)
  MOE_PREP_CASE(32)
#undef MOE_PREP_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
