// fa_noalloc.cu -- fa_bwd_noalloc: the attention backward for callers that
// cannot allocate device memory.
//
// fa_bwd needs a scratch workspace (the fp32 dQ accumulator, the per-row LSE/D
// terms and, in deterministic mode, ordering counters) that the caller must
// allocate.  Some callers have no way to do that at the point of the call: a
// plugin or operator run by a host framework that owns all device memory and
// hands out no scratch buffers, or code on a latency-critical path where
// cudaMalloc is not allowed because it can synchronise the whole device.  For
// them this entry point takes its scratch from a fixed array in device memory
// that belongs to the library, and calls no allocating routine at all (no
// cudaMalloc, cudaFree, or any library call that allocates).
//
// Limits and sharing:
//  * the array holds FA_NOALLOC_SCRATCH_BYTES (32 MiB); a problem whose
//    fa_bwd_workspace_bytes() is larger is rejected with FA_ERR_WORKSPACE;
//  * every GPU that loads the library holds one such array until the process
//    exits;
//  * all calls share the array and it keeps whatever the last call left in it;
//    the preprocess kernel clears everything that must start at zero (the dQ
//    accumulator and the counters), so stale contents are harmless;
//  * calls that can overlap on the GPU (different streams, or different host
//    threads on one device) race on the array: order them on one stream.
//  * the first call on each device looks up the array's device address (with
//    that device current) and caches it; make that first call before any
//    stream capture.  The cached address belongs to the device's primary
//    context: calling cudaDeviceReset while the library is loaded is not
//    supported (the same holds for the library's status word).
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// The library-owned scratch.  In host code this name is only a host-side
// stand-in for the symbol, not a device address: host code must use the
// address from cudaGetSymbolAddress (see scratch_on_current_device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device.  Returns nullptr (and sets *err) if the lookup fails.
void* scratch_on_current_device(cudaError_t* err) {
  static void* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                              int causal, float scale, int deterministic, void* stream) {
  // fa_bwd's own checks, in its order, with the scratch standing in for the workspace (any
  // non-null 256-byte aligned address of the scratch's size: only its size and alignment are
  // checked), so that every status matches fa_bwd's and a rejected call touches no GPU state.
  bool launch = false;
  int st = fa::bwd_validate(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, N, d, causal, scale, deterministic,
                            reinterpret_cast<const void*>(uintptr_t{256}), (size_t)FA_NOALLOC_SCRATCH_BYTES, &launch);
  if (st || !launch) return st;
  cudaError_t e = cudaSuccess;
  void* ws = scratch_on_current_device(&e);
  if (!ws) {
    cudaGetLastError();  // leave no sticky error behind for the caller's CUDA calls
    return fa::report_cuda_error("cudaGetSymbolAddress(fa_bwd_noalloc scratch)", e);
  }
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, scale, deterministic, ws,
                (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
