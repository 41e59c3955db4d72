// moe_route_dispatch_noalloc: the dispatch entry point for callers that cannot allocate
// device memory.
//
// moe_route_dispatch needs a caller-provided workspace for its per-CTA histograms and
// bases.  Some callers have no way to provide one: code embedded in a host framework that
// owns every device allocation and forbids raw cudaMalloc, latency-critical serving loops
// where an allocation (and the synchronisation a later cudaFree implies) is not allowed, or
// runtimes whose device memory budget is fixed at start-up.  This variant keeps that scratch
// in a fixed-size array that is part of the library image instead, so the caller passes only
// inputs and outputs.
//
// The array (kScratchBytes, 2 MiB) lives in device memory of every GPU that loads the
// library, for the life of the process.  All calls share it and it keeps whatever the last
// call left: the error record is cleared at the start of each call; the histograms and
// bases are fully rewritten by every call.  Two calls that overlap on the GPU (different
// streams without ordering, or different host threads) race on the array.  The array's
// device address is cached per device at the first call, so a device reset after that call
// (cudaDeviceReset, or a new primary context) is not supported.
// moe_route_dispatch_noalloc_get_error reads the error record the last call left.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kScratchBytes = size_t{2} << 20;
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Device address of g_route_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached; the first call on a device does this.
void* scratch_on_current_device(cudaError_t* st) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  *st = cudaGetDevice(&dev);
  if (*st != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *st = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *st = cudaGetSymbolAddress(&p, g_route_scratch);
    if (*st != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_dispatch_noalloc(
    const moe_bf16_t* x, const float* logits, int64_t T, int d, int E, int k,
    int32_t* topk_idx, float* gate, int32_t* counts, int32_t* offsets, int32_t* perm,
    int32_t* pos, moe_bf16_t* x_perm, cudaStream_t stream) {
  // the argument rules of moe_route_dispatch, from the same function
  const moe_status_t chk = check_route_args(x, logits, T, d, E, k, topk_idx, gate, counts,
                                            offsets, perm, pos, x_perm);
  if (chk != MOE_OK) return chk;
  // the fixed scratch holds an error record and two [ceil(T/128), E] int32 tables
  const int64_t nblk = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  const size_t table = round256(static_cast<size_t>(nblk) * E * 4);
  if (256 + 2 * table > kScratchBytes) return MOE_ERR_UNSUPPORTED;

  cudaError_t st = cudaSuccess;
  char* scratch = static_cast<char*>(scratch_on_current_device(&st));
  if (!scratch) return MOE_ERR_CUDA;
  DevErr* err = reinterpret_cast<DevErr*>(scratch);
  int32_t* hist = reinterpret_cast<int32_t*>(scratch + 256);
  int32_t* bbase = reinterpret_cast<int32_t*>(scratch + 256 + table);
  if (cudaMemsetAsync(err, 0, sizeof(DevErr), stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (launch_route_topk(logits, T, E, k, topk_idx, gate, pos, hist, err, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_scan_cols(hist, nblk, E, bbase, counts, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_offsets(counts, E, 1, nullptr, offsets, nullptr, err, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_scatter(x, T, d, E, k, topk_idx, bbase, offsets, pos, perm, x_perm, T * k, err,
                     stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status_t moe_route_dispatch_noalloc_get_error(cudaStream_t stream) {
  cudaError_t st = cudaSuccess;
  const char* scratch = static_cast<const char*>(scratch_on_current_device(&st));
  if (!scratch) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  DevErr e{};
  if (cudaMemcpy(&e, scratch, sizeof e, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(e.status);
}
