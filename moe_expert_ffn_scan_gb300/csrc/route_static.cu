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

// Device address of g_route_scratch, looked up with cudaGetSymbolAddress (in host code
// the array's name is only a host-side stand-in) once per CUDA context and cached
// under that context's unique id.  A context that replaces the one the address was
// taken in (after cudaDeviceReset, or a different context made current on the same
// device) has another id, so the address is looked up again there: the module, and
// with it the array, may have moved.
struct SymbolCache {
  std::mutex mu;
  unsigned long long ctx_id[64] = {};
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
  // id 0: no current context yet, or a destroyed one (cudaDeviceReset) still reads as
  // current; the lookup below makes the runtime's context current, and the id is read
  // again after it.
  const unsigned long long id = moe::current_context_id();
  if (id == 0 || c.ctx_id[dev] != id || !c.addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    c.ctx_id[dev] = moe::current_context_id();
    c.addr[dev] = p;
  }
  *out = c.addr[dev];
  return cudaSuccess;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

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
  if (!aligned4(logits) || !aligned4(idx) || !aligned4(w) || !aligned4(counts) ||
      !aligned4(offsets) || !aligned4(perm_src) || !aligned4(inv))
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

extern "C" int moe_route_static_status(void* stream, uint32_t* bits_out) {
  if (bits_out) *bits_out = 0;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  // the status word is the first word of the fixed array (see moe_route_static)
  return moe_check_status(base, stream, bits_out);
}
