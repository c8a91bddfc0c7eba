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
  if ((e = set_smem<MODE_GRAD, false, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD_STAGE, false, true>()) != cudaSuccess) return e;
  if ((e = set_smem<MODE_FWD_STAGE, true, true>()) != cudaSuccess) return e;
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
    case MODE_GRAD: return cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_GRAD, false, true>, args);
    case MODE_FWD_STAGE:
      return cap ? cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_FWD_STAGE, true, true>, args)
                 : cudaLaunchKernelEx(&cfg, cce_gemm_kernel<MODE_FWD_STAGE, false, true>, args);
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

// The CTA-pair handshake of the pair GEMM, reduced to its waits: the odd
// CTA arrives on the even CTA's barrier (as its copies complete on the even
// CTA's full barriers) and the even CTA then arrives on the odd CTA's barrier
// (as the accumulator hand-back does).  With hold != 0 the odd CTA holds its
// arrive back: the even CTA's bounded wait runs out and raises its abort
// flag, the odd CTA's next wait runs out too, the odd CTA gives its copies
// the same bounded grace as the GEMM, and both meet at the final cluster
// barrier -- the kernel ends with CCE_DEVERR_TIMEOUT instead of hanging.
// Every wait is bounded by timeout_ns; no CTA leaves before the final
// barrier, so no arrive reaches a CTA that has exited.
__global__ void selftest_pair_timeout_kernel(int32_t* dev_err, uint64_t timeout_ns, int hold) {
  __shared__ uint64_t bar_in;    // even CTA: the odd CTA's arrive
  __shared__ uint64_t bar_back;  // odd CTA: the even CTA's answer
  __shared__ int abort_flag;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    mbar_init(&bar_in, 1);
    mbar_init(&bar_back, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  if (threadIdx.x == 0) {
    if (rank == 0) {
      if (wait_bounded_ns(&bar_in, 0, &abort_flag, dev_err, timeout_ns))
        mbar_arrive_cluster(mapa_shared(smem_u32(&bar_back), 1));
    } else {
      if (!hold) mbar_arrive_cluster(mapa_shared(smem_u32(&bar_in), 0));
      wait_bounded_ns(&bar_back, 0, &abort_flag, dev_err, timeout_ns);
      if (abort_flag) {  // the pair GEMM's grace for copies in flight
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 10000000ull) {
        }
      }
    }
  }
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
}

cudaError_t launch_selftest_pair_timeout(int32_t* dev_err, uint64_t timeout_ns, int hold, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, selftest_pair_timeout_kernel, dev_err, timeout_ns, hold);
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
