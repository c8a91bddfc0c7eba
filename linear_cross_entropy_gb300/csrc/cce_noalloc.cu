// cce_forward_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they need the loss: code running inside a CUDA-graph capture
// that must not allocate, a runtime whose memory is fully pre-partitioned by
// its own pool, or a host framework that forbids allocation on its hot path.
// cce_forward needs a caller-provided workspace; this entry point instead uses
// a scratch array the library owns, declared below as a file-scope
// __device__ array of fixed size.  Every GPU that loads the library holds that
// array until the process exits.
//
// The array's name in host code is only a host-side stand-in, not a device
// address, so the device address is looked up with cudaGetSymbolAddress once
// per device, with that device current, on the first call made on it.  Make
// that first call before any stream capture begins.
//
// All calls share the one array and it keeps the contents of the last call.
// The forward writes every scratch word it later reads, so nothing needs
// clearing between calls, but calls whose work overlaps on the GPU (for
// example on two streams at once) race on the array and must be serialised
// by the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/cce.h"

static constexpr size_t kScratchBytes = CCE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};  // device address of the array, per device

}  // namespace

extern "C" cce_status cce_forward_noalloc(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D,
                                          int64_t V, int64_t ignore_index, int reduction, float* loss, float* lse,
                                          int32_t* dev_err, void* stream) {
  const size_t need = cce_forward_workspace_bytes(N, D, V);
  if (need == 0) return CCE_ERR_SHAPE;
  if (need > kScratchBytes) return CCE_ERR_WORKSPACE;  // problem too large for the fixed scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return CCE_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return CCE_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return cce_forward(E, C, x, N, D, V, ignore_index, reduction, loss, lse, scratch, kScratchBytes, dev_err,
                     stream);
}
