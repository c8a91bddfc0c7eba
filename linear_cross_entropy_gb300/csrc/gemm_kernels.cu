// Instantiations and launcher of the tcgen05 GEMM kernels.
#include "gemm.cuh"
#include "internal.h"

namespace cce {

template <int MODE, bool CAP>
static cudaError_t set_smem() {
  return cudaFuncSetAttribute(cce_gemm_kernel<MODE, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t prepare_gemm_kernels() {
  cudaError_t e;
  if ((e = set_smem<MODE_FWD, false>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G, false>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD_STAGE, false>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD_STAGE, true>()) != cudaSuccess) return e;
  return set_smem<MODE_GRAD, false>();
}

// One thread waits on an mbarrier that nothing ever arrives on, through the
// same bounded wait the GEMM pipelines use; the wait must run out and report
// CCE_DEVERR_TIMEOUT instead of hanging.
__global__ void selftest_wait_timeout_kernel(int32_t* dev_err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  wait_bounded_ns(&bar, 0, &abort_flag, dev_err, timeout_ns);
}

cudaError_t launch_selftest_wait_timeout(int32_t* dev_err, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_wait_timeout_kernel<<<1, 1, 0, stream>>>(dev_err, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_gemm(int mode, const GemmArgs& args, int grid, cudaStream_t stream) {
  const dim3 g(static_cast<unsigned>(grid)), b(NUM_THREADS);
  const bool cap = args.softcap > 0.0f;
  switch (mode) {
    case MODE_FWD:
      if (cap) {
        cce_gemm_kernel<MODE_FWD, true><<<g, b, SMEM_BYTES, stream>>>(args);
      } else {
        cce_gemm_kernel<MODE_FWD, false><<<g, b, SMEM_BYTES, stream>>>(args);
      }
      break;
    case MODE_BWD_G:
      if (cap) {
        cce_gemm_kernel<MODE_BWD_G, true><<<g, b, SMEM_BYTES, stream>>>(args);
      } else {
        cce_gemm_kernel<MODE_BWD_G, false><<<g, b, SMEM_BYTES, stream>>>(args);
      }
      break;
    case MODE_FWD_STAGE:
      if (cap) {
        cce_gemm_kernel<MODE_FWD_STAGE, true><<<g, b, SMEM_BYTES, stream>>>(args);
      } else {
        cce_gemm_kernel<MODE_FWD_STAGE, false><<<g, b, SMEM_BYTES, stream>>>(args);
      }
      break;
    case MODE_GRAD: cce_gemm_kernel<MODE_GRAD, false><<<g, b, SMEM_BYTES, stream>>>(args); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace cce
