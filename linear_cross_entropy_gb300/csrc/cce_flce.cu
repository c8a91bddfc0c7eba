// Bandwidth-bound kernels of the single call (loss and both gradients in one
// pass, "fused-linear-cross-entropy" page, section "2. Fused Linear
// Cross-Entropy (FLCE)"): the forward GEMM of a token chunk has staged its
// logits (fp16, minus each row's max over each 32-column chunk); here they
// become the weighted logit gradient G-hat in bf16, in place, with the
// 128 x 128 filter votes ("Cut Your Losses in Large-Vocabulary Language
// Models", "Gradient Filtering").  Also: the dE / dC finalisation, the filter
// statistics and the scaling by the upstream gradient.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "../../include/cce.h"
#include "internal.h"

namespace cce {
namespace {

constexpr float LOG2E_F = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// One 128-row x 128-column tile per block (256 threads).  First the block
// loads, coalesced, each row's target, LSE and the four 32-column chunk
// maxima of the tile into shared memory (c_row = (max - LSE) * log2e, -inf
// for rows that take no part, so their G is 0); then every thread issues its
// eight independent 16-byte loads of staged values (16 threads of eight
// columns per row, 16 rows per pass, 8 passes) and computes
// G = exp2(h * log2e + c_row) - onehot.  The vote is any |G| >= eps
// (unscaled G, before the softcap slope); the stored value is w * G * slope
// in bf16.  A tile that both outputs skip is not written back (nothing reads
// it).
template <bool CAP>
__global__ void __launch_bounds__(256, CAP ? 3 : 4) gpass_kernel(uint16_t* __restrict__ stage, int pitch,
                                                    const float* __restrict__ mtile, int rows, int V,
                                                    const int64_t* __restrict__ x, long long ignore_index,
                                                    const float* __restrict__ lse, const int* __restrict__ count,
                                                    int reduction, float softcap, float eps, int store_skipped,
                                                    uint8_t* __restrict__ bitmap, uint8_t* __restrict__ bitmapT,
                                                    int bm_ld, int n_blocks, const int* __restrict__ n_dev,
                                                    int n_row0, int* __restrict__ kept) {
  __shared__ float s_c[4][128];  // c_row per 32-column chunk of the tile
  __shared__ float s_m[4][128];  // the chunk maxima (softcap slope)
  __shared__ int s_rel[128];     // target column within the tile, or -1
  const int vt = blockIdx.x, tb = blockIdx.y;
  // Compact rows that exist (their count is in device memory): row blocks
  // past them are never read and get no survival byte.  Inside the last
  // block the rows past the count are zero rows with an ignored target, so
  // they get G = 0 below (the gradient GEMM reads them as part of its K).
  const int nrows = n_dev ? max(0, min(rows, *n_dev - n_row0)) : rows;
  if (tb * 128 >= nrows) return;
  const int t = threadIdx.x;
  {
    const int r = t & 127, row = tb * 128 + r;
    const bool ok = row < rows;
    const long long xr = ok ? static_cast<long long>(x[row]) : ignore_index;
    const bool part = xr != ignore_index && xr >= 0 && xr < V;
    const float l = part ? lse[row] : 0.0f;
    const int c_lo = (t >> 7) * 2;  // threads 0..127: chunks 0, 1; 128..255: chunks 2, 3
#pragma unroll
    for (int c = c_lo; c < c_lo + 2; ++c) {
      const float m = ok ? mtile[static_cast<size_t>(vt * 4 + c) * rows + row] : 0.0f;
      s_m[c][r] = m;
      s_c[c][r] = part ? (m - l) * LOG2E_F : -INFINITY;
    }
    if (t < 128) {
      const long long rel = xr - static_cast<long long>(vt) * 128;
      s_rel[r] = (part && rel >= 0 && rel < 128) ? static_cast<int>(rel) : -1;
    }
  }
  const int c8 = t & 15;
  const int r_in = t >> 4;
  const int col0 = vt * 128 + c8 * 8;
  const int ch = c8 >> 2;  // 32-column chunk of these eight columns
  uint4 h[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int row = tb * 128 + r_in + 16 * k;
    h[k] = row < rows ? *reinterpret_cast<const uint4*>(stage + static_cast<size_t>(row) * pitch + col0)
                      : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  const bool ragged = col0 + 8 > V;  // only in the last column tile
  const float w = reduction == CCE_RED_SUM ? 1.0f : 1.0f / static_cast<float>(max(*count, 1));
  const float inv_cap = CAP ? 1.0f / softcap : 0.0f;
  float amax = 0.0f;  // largest unscaled |G| this thread saw
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = r_in + 16 * k;
    const float cr = s_c[ch][r];
    const uint32_t hw[4] = {h[k].x, h[k].y, h[k].z, h[k].w};
    float g[8];
    float sl[8];  // softcap slope 1 - tanh^2 (the staged value + max is the capped logit)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[j]));
      g[2 * j] = ex2f(fmaf(f.x, LOG2E_F, cr));
      g[2 * j + 1] = ex2f(fmaf(f.y, LOG2E_F, cr));
      if constexpr (CAP) {
        const float m = s_m[ch][r];
        const float t0 = (f.x + m) * inv_cap, t1 = (f.y + m) * inv_cap;
        sl[2 * j] = 1.0f - t0 * t0;
        sl[2 * j + 1] = 1.0f - t1 * t1;
      }
    }
    const int rel = s_rel[r] - c8 * 8;
    if (rel >= 0 && rel < 8) {  // the target column is one of these eight (one thread per row)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == rel) g[j] -= 1.0f;
    }
    if (ragged) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col0 + j >= V) g[j] = 0.0f;
    }
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fmaxf(fabsf(g[2 * j]), fabsf(g[2 * j + 1])));
      float a0 = w * g[2 * j], a1 = w * g[2 * j + 1];
      if constexpr (CAP) {  // only where G != 0: columns past V stage +inf, whose slope is not a number
        a0 = g[2 * j] != 0.0f ? a0 * sl[2 * j] : 0.0f;
        a1 = g[2 * j + 1] != 0.0f ? a1 * sl[2 * j + 1] : 0.0f;
      }
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
      std::memcpy(&out[j], &b2, 4);
    }
    h[k] = make_uint4(out[0], out[1], out[2], out[3]);
  }
  const bool keep = __syncthreads_or(!(eps > 0.0f) || amax >= eps) != 0;  // eps = 0: nothing is skipped
  if (keep || store_skipped) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = tb * 128 + r_in + 16 * k;
      if (row < rows) *reinterpret_cast<uint4*>(stage + static_cast<size_t>(row) * pitch + col0) = h[k];
    }
  }
  if (t == 0) {
    bitmap[static_cast<size_t>(tb) * bm_ld + vt] = keep ? 1 : 0;
    bitmapT[static_cast<size_t>(vt) * n_blocks + tb] = keep ? 1 : 0;
    if (keep && kept) atomicAdd(kept + (blockIdx.x + blockIdx.y) % KEPT_SLOTS, 1);
  }
}

// dE[r] = bf16(sum over the S slabs of acc[s * slab + p]), slabs in order,
// where p = pos[r] is row r's compact row (rows with p < 0 took no part: +0).
__global__ void finalize_de_slabs_kernel(const float4* __restrict__ acc, int S, int slab, int N, int D,
                                         const int* __restrict__ pos, uint2* __restrict__ dE) {
  const size_t per_row = static_cast<size_t>(D) / 4;
  const size_t total = static_cast<size_t>(N) * per_row;
  const size_t slab4 = static_cast<size_t>(slab) * per_row;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = i / per_row;
    const int p = pos[row];
    if (p < 0) {
      dE[i] = make_uint2(0u, 0u);
      continue;
    }
    const size_t at = static_cast<size_t>(p) * per_row + (i - row * per_row);
    float4 v = acc[at];
    for (int s = 1; s < S; ++s) {
      const float4 u = acc[s * slab4 + at];
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 out;
    std::memcpy(&out.x, &lo, 4);
    std::memcpy(&out.y, &hi, 4);
    dE[i] = out;
  }
}

// stats[0] += tiles, stats[1] += skipped tiles of one chunk's survival map
// (ceil(rows / 128) rows of ncols bytes, pitch bm_ld; rows = clamp(*n_dev -
// n_row0, 0, max_rows)).  One block; launches run in stream order, so the
// sums are deterministic.
__global__ void stats_add_kernel(const uint8_t* __restrict__ bitmap, const int* __restrict__ n_dev, int n_row0,
                                 int max_rows, int ncols, int bm_ld, int64_t* __restrict__ stats) {
  __shared__ long long sz[1024];
  const int nb = (max(0, min(max_rows, *n_dev - n_row0)) + 127) / 128;
  const long long n = static_cast<long long>(nb) * ncols;
  long long z = 0;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) z += bitmap[(i / ncols) * bm_ld + (i % ncols)] == 0 ? 1 : 0;
  sz[threadIdx.x] = z;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) sz[threadIdx.x] += sz[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    stats[0] += n;
    stats[1] += sz[0];
  }
}

// x *= *g for bf16 arrays (eight values per thread); nothing when *g == 1.
__global__ void scale_bf16_kernel(uint4* __restrict__ a, size_t n8a, uint4* __restrict__ b, size_t n8b,
                                  const float* __restrict__ g) {
  const float s = *g;
  if (s == 1.0f) return;
  const size_t total = n8a + n8b;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    uint4* p = i < n8a ? a + i : b + (i - n8a);
    uint4 v = *p;
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h;
      std::memcpy(&h, &w[j], 4);
      const float2 f = __bfloat1622float2(h);
      h = __floats2bfloat162_rn(f.x * s, f.y * s);
      std::memcpy(&w[j], &h, 4);
    }
    *p = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

int grid_cap(size_t work, int per_block, int cap) {
  return static_cast<int>(std::max<size_t>(1, std::min<size_t>(static_cast<size_t>(cap), (work + per_block - 1) / per_block)));
}

}  // namespace

cudaError_t launch_gpass(uint16_t* stage, int64_t pitch, const float* mtile, int64_t rows, int64_t V,
                         const int64_t* x, long long ignore_index, const float* lse, const int* count, int reduction,
                         float softcap, float eps, bool store_skipped, uint8_t* bitmap, uint8_t* bitmapT,
                         int64_t bm_ld, const int* n_dev, int64_t n_row0, int* kept, cudaStream_t s,
                         int* launches) {
  const int nb = static_cast<int>((rows + 127) / 128);
  const dim3 grid(static_cast<unsigned>((V + 127) / 128), static_cast<unsigned>(nb));
  if (softcap > 0.0f) {
    gpass_kernel<true><<<grid, 256, 0, s>>>(stage, static_cast<int>(pitch), mtile, static_cast<int>(rows),
                                            static_cast<int>(V), x, ignore_index, lse, count, reduction, softcap, eps,
                                            store_skipped ? 1 : 0, bitmap, bitmapT, static_cast<int>(bm_ld), nb, n_dev,
                                            static_cast<int>(n_row0), kept);
  } else {
    gpass_kernel<false><<<grid, 256, 0, s>>>(stage, static_cast<int>(pitch), mtile, static_cast<int>(rows),
                                             static_cast<int>(V), x, ignore_index, lse, count, reduction, softcap,
                                             eps, store_skipped ? 1 : 0, bitmap, bitmapT, static_cast<int>(bm_ld), nb,
                                             n_dev, static_cast<int>(n_row0), kept);
  }
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_finalize_de_slabs(const float* acc, int S, int64_t slab, int64_t N, int64_t D, const int* pos,
                                     void* dE, cudaStream_t s, int sms, int* launches) {
  const size_t n4 = static_cast<size_t>(N) * D / 4;
  finalize_de_slabs_kernel<<<grid_cap(n4, 256, sms * 8), 256, 0, s>>>(
      reinterpret_cast<const float4*>(acc), S, static_cast<int>(slab), static_cast<int>(N), static_cast<int>(D), pos,
      static_cast<uint2*>(dE));
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_stats_add(const uint8_t* bitmap, const int* n_dev, int64_t n_row0, int64_t max_rows,
                             int64_t ncols, int64_t bm_ld, int64_t* stats, cudaStream_t s, int* launches) {
  stats_add_kernel<<<1, 1024, 0, s>>>(bitmap, n_dev, static_cast<int>(n_row0), static_cast<int>(max_rows),
                                      static_cast<int>(ncols), static_cast<int>(bm_ld), stats);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_scale_bf16(void* a, int64_t na, void* b, int64_t nb, const float* g, cudaStream_t s, int sms,
                              int* launches) {
  const size_t n8a = static_cast<size_t>(na) / 8, n8b = static_cast<size_t>(nb) / 8;
  scale_bf16_kernel<<<grid_cap(n8a + n8b, 256, sms * 8), 256, 0, s>>>(static_cast<uint4*>(a), n8a,
                                                                      static_cast<uint4*>(b), n8b, g);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace cce
