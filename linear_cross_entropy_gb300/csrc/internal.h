// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gemm_args.h"

namespace cce {

// Launches cce_gemm_kernel<mode> with `grid` persistent CTAs on `stream`.
cudaError_t launch_gemm(int mode, const GemmArgs& args, int grid, cudaStream_t stream);

// cce_gemm_kernel<mode> (FWD, BWD_G, GRAD) as `clusters` persistent
// clusters of two CTAs sharing each MMA (M = 256) over pairs of row blocks.
// FWD / BWD_G: args.tmB2 holds C in 128-row boxes and args.group_n is even.
// GRAD: the MN-major B maps come in 128-column (two-group) boxes, args.bn is
// 256, and args.tmZ is a 16 KiB box of zeros.
cudaError_t launch_gemm_pairs(int mode, const GemmArgs& args, int clusters, cudaStream_t stream);

// How many CTA pairs of the GEMM kernel fit on the device at once (0: none).
int gemm_pair_clusters(int sms);

// Launches the bounded-wait self-test kernel (see cce_selftest_wait_timeout).
cudaError_t launch_selftest_wait_timeout(int32_t* dev_err, uint64_t timeout_ns, cudaStream_t stream);
// Launches the CTA-pair handshake self-test (see cce_selftest_pair_timeout).
cudaError_t launch_selftest_pair_timeout(int32_t* dev_err, uint64_t timeout_ns, int hold, cudaStream_t stream);

// Opt the GEMM kernels into their dynamic shared-memory size (once per device).
cudaError_t prepare_gemm_kernels();

// Vocabulary sorting (cce_sort.cu).  Every launcher adds the number of
// kernels it launched to *launches.
size_t vocab_keys_scratch_bytes(int64_t N, int64_t D);
size_t vocab_order_scratch_bytes(int64_t V);
// keys[v] = C_v . (sum of the rows of E [N, D] that take part): rows below
// *n_dev (all N when null) whose target, when x is given, is in [0, V) and
// not ignore_index.
cudaError_t launch_vocab_keys(const void* E, int64_t N, const int* n_dev, const int64_t* x, long long ignore_index,
                              int64_t D, const void* C, int64_t V, float* keys, void* scratch, cudaStream_t s,
                              int sms, int* launches);
// perm = the stable ascending order of keys (perm[j] = token at position j);
// inv (optional) = perm^-1.  Five launches.
cudaError_t launch_vocab_order(const float* keys, int64_t V, int* perm, void* scratch, cudaStream_t s,
                               int* launches, int* inv);
// Compact targets xc[k < *n_dev] become sorted positions inv[xc[k]], the
// zero rows padding the last 128-row block get -1.
cudaError_t launch_remap_targets(const int* inv, int64_t* xc, const int* n_dev, int64_t N, cudaStream_t s, int sms,
                                 int* launches);
// dst[j] = src[rows[j]] (bf16 rows of D) for j < count, zero rows up to total.
cudaError_t launch_gather_vocab_rows(const void* src, const int* rows, int64_t count, int64_t total, int64_t D,
                                     void* dst, cudaStream_t s, int sms, int* launches);

// Single call (cce_flce.cu).
// Staged fp16 logits (minus the 32-column chunk maxima in mtile) of the
// chunk's rows -> bf16 G-hat in place, and
// the chunk's survival map (bitmap [ceil(rows/128)][bm_ld], bitmapT
// [bm_ld][ceil(rows/128)]).
cudaError_t launch_gpass(uint16_t* stage, int64_t pitch, const float* mtile, int64_t rows, int64_t V,
                         const int64_t* x, long long ignore_index, const float* lse, const int* count, int reduction,
                         float softcap, float eps, bool store_skipped, uint8_t* bitmap, uint8_t* bitmapT,
                         int64_t bm_ld, const int* n_dev, int64_t n_row0, int* kept, cudaStream_t s,
                         int* launches);
// the chunk has clamp(*n_dev - n_row0, 0, rows) rows (rows when n_dev is null);
// rows is also the pitch of mtile.  kept (may be null): counts the kept tiles.
cudaError_t launch_finalize_de_slabs(const float* acc, int S, int64_t slab, int64_t N, int64_t D, const int* pos,
                                     void* dE, cudaStream_t s, int sms, int* launches);
cudaError_t launch_stats_add(const uint8_t* bitmap, const int* n_dev, int64_t n_row0, int64_t max_rows,
                             int64_t ncols, int64_t bm_ld, int64_t* stats, cudaStream_t s, int* launches);
cudaError_t launch_scale_bf16(void* a, int64_t na, void* b, int64_t nb, const float* g, cudaStream_t s, int sms,
                              int* launches);

}  // namespace cce
