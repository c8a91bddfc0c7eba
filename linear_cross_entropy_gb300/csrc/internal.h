// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gemm_args.h"

namespace cce {

// Launches cce_gemm_kernel<mode> with `grid` persistent CTAs on `stream`.
cudaError_t launch_gemm(int mode, const GemmArgs& args, int grid, cudaStream_t stream);

// Launches the bounded-wait self-test kernel (see cce_selftest_wait_timeout).
cudaError_t launch_selftest_wait_timeout(int32_t* dev_err, uint64_t timeout_ns, cudaStream_t stream);

// Opt the GEMM kernels into their dynamic shared-memory size (once per device).
cudaError_t prepare_gemm_kernels();

}  // namespace cce
