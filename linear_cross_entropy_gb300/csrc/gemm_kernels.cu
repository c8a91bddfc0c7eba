// Instantiations and launcher of the tcgen05 GEMM kernels.
#include "gemm.cuh"
#include "internal.h"

namespace cce {

template <int MODE, bool CAP, bool PAIR = false>
static cudaError_t set_smem() {
  return cudaFuncSetAttribute(cce_gemm_kernel<MODE, CAP, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SMEM_BYTES);
}

cudaError_t prepare_gemm_kernels() {
  cudaError_t e;
  if ((e = set_smem<MODE_FWD, false>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G, false>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD_STAGE, false>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD_STAGE, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD, false, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD, true, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G, false, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_BWD_G, true, true>()) != cudaSuccess) return e;
  return set_smem<MODE_GRAD, false>();
}

static cudaLaunchConfig_t pair_config(int clusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = 2;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int gemm_pair_clusters(int sms) {
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pair_config(sms / 2, nullptr, &attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, cce_gemm_kernel<MODE_FWD, false, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gemm_pairs(int mode, const GemmArgs& args, int clusters, cudaStream_t stream) {
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pair_config(clusters, stream, &attr);
  const bool cap = args.softcap > 0.0f;
  switch (mode) {
    case MODE_FWD:
      return cap ? cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_FWD, true, true>, args)
                 : cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_FWD, false, true>, args);
    case MODE_BWD_G:
      return cap ? cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_BWD_G, true, true>, args)
                 : cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_BWD_G, false, true>, args);
    default: return cudaErrorInvalidValue;
  }
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
