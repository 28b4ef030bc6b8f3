// moe_route_static: the routing + permutation call of moe_route, with its scratch
// held in a fixed device array inside this library instead of a caller workspace.
//
// Who needs it: callers that may not allocate device memory themselves -- code
// embedded in a host framework whose memory pool owns every device byte and
// forbids side allocations, or latency-critical loops that cannot afford
// cudaMalloc / cudaFree (both can synchronise the device).  Such a caller passes
// only its inputs and outputs; this file provides the scratch.
//
// The scratch is one file-scope __device__ array of kStaticScratchBytes.  Every GPU
// that loads the library holds it until the process exits.  Every call shares it and
// it keeps the last call's contents, so calls that overlap on the GPU (two streams,
// or two host threads) race on it and must be serialised by the caller.
#include <mutex>

#include "kernels.cuh"

namespace {

// A 256-byte status block plus two [token blocks][E] int32 tables of up to 128 KiB
// each: ceil(T/256) * E <= 32768.
constexpr size_t kStaticScratchBytes = 256 + 256 * 1024;
constexpr size_t kStatusBytes = 256;

__device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

// Device address of g_route_scratch per device, looked up once per device with that
// device current (in host code the array's name is only a host-side stand-in).
struct SymbolCache {
  std::mutex mu;
  void* addr[64] = {};
};

SymbolCache& cache() {
  static SymbolCache c;
  return c;
}

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SymbolCache& c = cache();
  std::lock_guard<std::mutex> lock(c.mu);
  if (!c.addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    c.addr[dev] = p;
  }
  *out = c.addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int moe_route_static(const moe_dims* d, const float* logits, int32_t* idx, float* w,
                                int32_t* counts, int32_t* offsets, int32_t* perm_src,
                                int32_t* inv, void* stream) {
  if (!d || d->T < 1 || d->E < 1 || d->E > 1024 || d->k < 1 || d->k > 16 || d->k > d->E ||
      (d->has_shared != 0 && d->has_shared != 1))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(d->T) * d->k + d->T >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!logits || !idx || !w || !counts || !offsets || !perm_src || !inv)
    return MOE_ERR_INVALID_ARG;
  // the two per-(token block, expert) tables must fit the fixed scratch
  const size_t table = static_cast<size_t>(moe::perm_blocks(d->T)) * d->E * sizeof(int32_t);
  const size_t table_al = (table + 255) / 256 * 256;
  if (kStatusBytes + 2 * table_al > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  uint8_t* b = static_cast<uint8_t*>(base);
  uint32_t* status = reinterpret_cast<uint32_t*>(b);
  int32_t* blockcnt = reinterpret_cast<int32_t*>(b + kStatusBytes);
  int32_t* blockbase = reinterpret_cast<int32_t*>(b + kStatusBytes + table_al);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // blockcnt and blockbase are fully rewritten by every call; only the status word
  // must start at zero (the routing kernel clears it).
  if (moe::launch_route(logits, d->T, d->E, d->k, idx, w, status, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_permute(idx, d->T, d->E, d->k, d->has_shared, blockcnt, blockbase, counts,
                          offsets, perm_src, inv, status, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
