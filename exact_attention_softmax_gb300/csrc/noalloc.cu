// noalloc.cu -- sdpa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory at the point where they
// run the backward: code running under an allocator that must not grow (a
// fixed memory pool sized ahead of time), plugins and embedded runtimes that
// are handed only their input and output buffers, and hosts that forbid
// cudaMalloc after start-up. sdpa_bwd needs a workspace for the row statistic
// D = rowsum(dO * O) and the fp32 dQ accumulator; this entry point supplies
// it from a fixed array compiled into the library instead of asking the
// caller for one.
//
// The scratch is a file-scope device array of kNoAllocScratchBytes, held on
// every GPU where it has been loaded until the process exits. Host code only
// sees a host-side stand-in under the array's name, so the device address is
// looked up with cudaGetSymbolAddress once per device, on the first call made
// while that device is current. Under CUDA's lazy module loading that lookup
// is also what loads this file's device module, and with it the 16 MiB, onto
// the device: callers on a fixed memory budget make that first call at
// start-up, and before any stream capture. All calls share the one array and
// it keeps whatever the last call left in it: the backward's prep kernel
// rewrites D and zeroes the dQ accumulator at the start of every call, so
// nothing carries over between calls, but two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on the array and
// give wrong gradients.
#include "common.cuh"
#include "sdpa.h"

namespace sdpa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_dev_ptr[kMaxDev] = {nullptr};

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" int sdpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dO, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
                                float scale, int is_causal, int dtype, void* stream) {
  const size_t need = sdpa_bwd_workspace_size(B, H, Lq, d, dtype);
  if (need > kNoAllocScratchBytes) {
    // reported before anything touches the GPU
    return set_last_error(SDPA_ERR_WORKSPACE,
                          "sdpa_bwd_noalloc: this problem needs %zu bytes of scratch but the built-in scratch holds "
                          "%zu bytes; use sdpa_bwd with a caller-provided workspace",
                          need, kNoAllocScratchBytes);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_last_error(SDPA_ERR_CUDA, "sdpa_bwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return set_last_error(SDPA_ERR_UNSUPPORTED, "sdpa_bwd_noalloc: device %d", dev);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    // set-up, once per device, with that device current
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess)
      return set_last_error(SDPA_ERR_CUDA, "sdpa_bwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    if (ptr == nullptr)
      return set_last_error(SDPA_ERR_CUDA, "sdpa_bwd_noalloc: cudaGetSymbolAddress returned no address for the scratch array");
    g_scratch_dev_ptr[dev] = ptr;
  }
  return sdpa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Lq, Lk, d, scale, is_causal, nullptr, dtype,
                  g_scratch_dev_ptr[dev], kNoAllocScratchBytes, stream);
}
