// Instantiations and launcher of the three tcgen05 GEMM kernels.
#include "gemm.cuh"
#include "internal.h"

namespace cce {

template <int MODE>
static cudaError_t set_smem() {
  return cudaFuncSetAttribute(cce_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t prepare_gemm_kernels() {
  cudaError_t e;
  if ((e = set_smem<MODE_FWD>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G>()) != cudaSuccess) return e;
  return set_smem<MODE_GRAD>();
}

cudaError_t launch_gemm(int mode, const GemmArgs& args, int grid, cudaStream_t stream) {
  const dim3 g(static_cast<unsigned>(grid)), b(NUM_THREADS);
  switch (mode) {
    case MODE_FWD: cce_gemm_kernel<MODE_FWD><<<g, b, SMEM_BYTES, stream>>>(args); break;
    case MODE_BWD_G: cce_gemm_kernel<MODE_BWD_G><<<g, b, SMEM_BYTES, stream>>>(args); break;
    case MODE_GRAD: cce_gemm_kernel<MODE_GRAD><<<g, b, SMEM_BYTES, stream>>>(args); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace cce
