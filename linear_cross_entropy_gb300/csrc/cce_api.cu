// Host side of the C ABI (include/cce.h): argument checks, workspace layout,
// tensor maps, launches, phase timing; plus the small bandwidth-bound kernels
// of the path (forward combine and loss reduction, backward target count,
// dE finalisation, filter statistics).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "../../include/cce.h"
#include "internal.h"

namespace cce {
namespace {

constexpr int REF_SMS = 152;          // split count heuristic assumes this many SMs
constexpr size_t ALIGN = 256;         // sub-buffer alignment inside a workspace
#ifndef CCE_G_CHUNK_BUDGET_MIB
#define CCE_G_CHUNK_BUDGET_MIB 512
#endif
constexpr size_t G_CHUNK_BUDGET = size_t(CCE_G_CHUNK_BUDGET_MIB) << 20;  // bytes of the backward G chunk buffer
constexpr int64_t MIN_CHUNK = 2048, MAX_CHUNK = 65536;
constexpr int COMBINE_THREADS = 256;
// per vocabulary or token chunk: the recompute's and the gradient GEMM's
// scheduler counters, then KEPT_SLOTS counters of kept filter tiles
constexpr int CHUNK_COUNTERS = 2 + KEPT_SLOTS;
constexpr size_t ZERO_BOX_BYTES = PAIR_A_BYTES;  // one A operand box of the pair gradient GEMM

std::atomic<uint64_t> g_launches{0};
// survival words a gradient-GEMM pair's work item carries (a test hook lowers it)
std::atomic<int> g_pair_words{PAIR_MAP_WORDS};
// gradient GEMM with the filter on: 0 picks the layout by the kept tiles, 1
// always runs CTA pairs where they apply, 2 one CTA per tile (a test hook)
std::atomic<int> g_grad_layout{0};

// ------------------------------------------------------------ small kernels
// Per row: LSE from the per-split partials (fixed split order), loss, and a
// deterministic per-block partial sum for the reduction.  With n_dev the rows
// are compact and only the first clamp(*n_dev - n_row0, 0, N) exist.
__global__ void combine_kernel(const float* __restrict__ part_m, const float* __restrict__ part_s,
                               const float* __restrict__ tgt, const int64_t* __restrict__ x, int N, int S, int V,
                               long long ignore_index, int reduction, float* __restrict__ lse,
                               float* __restrict__ loss_rows, double* __restrict__ blk_sum,
                               int* __restrict__ blk_cnt, int32_t* dev_err, const int* __restrict__ n_dev,
                               int n_row0) {
  __shared__ double ssum[COMBINE_THREADS];
  __shared__ int scnt[COMBINE_THREADS];
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  const int nrow = n_dev ? max(0, min(N, *n_dev - n_row0)) : N;
  double my = 0.0;
  int mycnt = 0;
  if (row < nrow) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, part_m[static_cast<size_t>(s) * N + row]);
    float sum = 0.0f;
    for (int s = 0; s < S; ++s) {
      const size_t i = static_cast<size_t>(s) * N + row;
      sum += part_s[i] * exp2f(part_m[i] - M);
    }
    const float L = (M + log2f(sum)) * 0.6931471805599453f;
    lse[row] = L;
    const long long xi = static_cast<long long>(x[row]);
    bool valid = xi != ignore_index;
    if (valid && (xi < 0 || xi >= V)) {
      if (dev_err) atomicOr(reinterpret_cast<int*>(dev_err), CCE_DEVERR_TARGET_RANGE);
      valid = false;
    }
    const float lr = valid ? (L - tgt[row]) : 0.0f;
    if (reduction == CCE_RED_NONE) loss_rows[row] = lr;
    my = static_cast<double>(lr);
    mycnt = valid ? 1 : 0;
  }
  ssum[threadIdx.x] = my;
  scnt[threadIdx.x] = mycnt;
  __syncthreads();
  for (int w = COMBINE_THREADS / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) {
      ssum[threadIdx.x] += ssum[threadIdx.x + w];
      scnt[threadIdx.x] += scnt[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk_sum[blockIdx.x] = ssum[0];
    blk_cnt[blockIdx.x] = scnt[0];
  }
}

// One block: fixed-order sum of the per-block partials -> the reduced loss.
__global__ void finish_loss_kernel(const double* __restrict__ blk_sum, const int* __restrict__ blk_cnt, int nblk,
                                   int reduction, float* __restrict__ loss) {
  __shared__ double ssum[COMBINE_THREADS];
  __shared__ long long scnt[COMBINE_THREADS];
  double s = 0.0;
  long long c = 0;
  for (int i = threadIdx.x; i < nblk; i += COMBINE_THREADS) {
    s += blk_sum[i];
    c += blk_cnt[i];
  }
  ssum[threadIdx.x] = s;
  scnt[threadIdx.x] = c;
  __syncthreads();
  for (int w = COMBINE_THREADS / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) {
      ssum[threadIdx.x] += ssum[threadIdx.x + w];
      scnt[threadIdx.x] += scnt[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double total = ssum[0];
    const long long cnt = scnt[0];
    loss[0] = static_cast<float>(reduction == CCE_RED_SUM ? total : total / static_cast<double>(cnt > 0 ? cnt : 1));
  }
}

// Order-preserving compaction of the rows that take part in the backward
// (non-ignored, in-range target): pos[r] = compact index or -1; ridx[k] =
// original row; *count = number of such rows (the mean's divisor).
// Out-of-range targets are flagged and dropped like ignored rows.  Three
// launches over tiles of COMPACT_THREADS consecutive rows, one row per thread:
// per-tile counts, one block's exclusive scan of them, then each tile ranks
// its rows by warp ballots and a scan of the warp counts from its tile offset.
constexpr int COMPACT_THREADS = 1024;

__device__ __forceinline__ bool takes_part(const int64_t* __restrict__ x, int r, int N, int V,
                                           long long ignore_index, bool* bad) {
  if (r >= N) return false;
  const long long xi = static_cast<long long>(x[r]);
  if (xi == ignore_index) return false;
  if (xi < 0 || xi >= V) {
    *bad = true;
    return false;
  }
  return true;
}

__global__ void compact_count_kernel(const int64_t* __restrict__ x, int N, int V, long long ignore_index,
                                     int* __restrict__ tile_cnt, int32_t* dev_err) {
  bool bad = false;
  const int r = blockIdx.x * COMPACT_THREADS + static_cast<int>(threadIdx.x);
  const int c = __syncthreads_count(takes_part(x, r, N, V, ignore_index, &bad));
  if (threadIdx.x == 0) tile_cnt[blockIdx.x] = c;
  if (bad && dev_err) atomicOr(reinterpret_cast<int*>(dev_err), CCE_DEVERR_TARGET_RANGE);
}

__global__ void compact_scan_kernel(const int* __restrict__ tile_cnt, int ntiles, int* __restrict__ tile_off,
                                    int* count) {
  static_assert(COMPACT_THREADS == 32 * 32, "one scan lane per warp");
  __shared__ int warp_off[32];
  __shared__ int chunk_total;
  const int t = static_cast<int>(threadIdx.x), lane = t & 31, w = t >> 5;
  int carry = 0;
  for (int b0 = 0; b0 < ntiles; b0 += COMPACT_THREADS) {
    const int b = b0 + t;
    const int v = b < ntiles ? tile_cnt[b] : 0;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += u;
    }
    if (lane == 31) warp_off[w] = inc;
    __syncthreads();
    if (w == 0) {
      const int ws = warp_off[lane];
      int winc = ws;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, winc, off);
        if (lane >= off) winc += u;
      }
      warp_off[lane] = winc - ws;
      if (lane == 31) chunk_total = winc;
    }
    __syncthreads();
    if (b < ntiles) tile_off[b] = carry + warp_off[w] + inc - v;
    carry += chunk_total;
    __syncthreads();  // warp_off and chunk_total are rewritten by the next chunk
  }
  if (t == 0) *count = carry;
}

__global__ void compact_scatter_kernel(const int64_t* __restrict__ x, int N, int V, long long ignore_index,
                                       const int* __restrict__ tile_off, int* __restrict__ pos,
                                       int* __restrict__ ridx) {
  __shared__ int warp_off[32];
  const int t = static_cast<int>(threadIdx.x), lane = t & 31, w = t >> 5;
  const int r = blockIdx.x * COMPACT_THREADS + t;
  bool bad = false;
  const bool take = takes_part(x, r, N, V, ignore_index, &bad);
  const unsigned m = __ballot_sync(0xffffffffu, take);
  if (lane == 0) warp_off[w] = __popc(m);
  __syncthreads();
  if (w == 0) {  // exclusive scan of the warp counts
    const int v = warp_off[lane];
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += u;
    }
    warp_off[lane] = inc - v;
  }
  __syncthreads();
  if (r < N) {
    const int k = tile_off[blockIdx.x] + warp_off[w] + __popc(m & ((1u << lane) - 1u));
    pos[r] = take ? k : -1;
    if (take) ridx[k] = r;
  }
}

int compact_tiles(int64_t N) { return static_cast<int>((N + COMPACT_THREADS - 1) / COMPACT_THREADS); }

// Scratch of the compaction: per-tile counts and offsets.
size_t compact_scratch_bytes(int64_t N) { return sizeof(int) * 2 * static_cast<size_t>(compact_tiles(N)); }

cudaError_t launch_compact(const int64_t* x, int64_t N, int64_t V, long long ignore_index, int* pos, int* ridx,
                           int* count, int* scratch, int32_t* dev_err, cudaStream_t s) {
  const int nt = compact_tiles(N);
  int* cnt = scratch;
  int* off = scratch + nt;
  compact_count_kernel<<<nt, COMPACT_THREADS, 0, s>>>(x, static_cast<int>(N), static_cast<int>(V), ignore_index,
                                                       cnt, dev_err);
  compact_scan_kernel<<<1, COMPACT_THREADS, 0, s>>>(cnt, nt, off, count);
  compact_scatter_kernel<<<nt, COMPACT_THREADS, 0, s>>>(x, static_cast<int>(N), static_cast<int>(V),
                                                         ignore_index, off, pos, ridx);
  return cudaGetLastError();
}

// Compact copies of the rows that take part: E_c [k] = E[ridx[k]] and the
// per-row x, LSE and (reduction none) grad_out.  Rows from the count up to the
// next multiple of 128 are zero rows with an ignored target, so the last
// token block of every GEMM sees zeros.  One warp per row, 16-byte copies.
__global__ void gather_rows_kernel(const uint4* __restrict__ E, const int64_t* __restrict__ x,
                                   const float* __restrict__ lse, const float* __restrict__ g,
                                   const int* __restrict__ ridx, const int* __restrict__ count, int N, int D,
                                   long long ignore_index, uint4* __restrict__ Ec, int64_t* __restrict__ xc,
                                   float* __restrict__ lsec, float* __restrict__ gc) {
  const int n = *count;
  const int nz = min(N, (n + 127) / 128 * 128);
  const int lane = threadIdx.x & 31;
  const int per_row = D / 8;  // 16-byte chunks
  for (int k = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); k < nz; k += gridDim.x * (blockDim.x / 32)) {
    uint4* dst = Ec + static_cast<size_t>(k) * per_row;
    if (k < n) {
      const int r = ridx[k];
      const uint4* src = E + static_cast<size_t>(r) * per_row;
#pragma unroll 4
      for (int j = lane; j < per_row; j += 32) dst[j] = src[j];  // several 16-byte loads in flight per lane
      if (lane == 0) {
        xc[k] = x[r];
        if (lsec) lsec[k] = lse[r];
        if (gc) gc[k] = g[r];
      }
    } else {
      for (int j = lane; j < per_row; j += 32) dst[j] = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0) {
        xc[k] = ignore_index;
        if (lsec) lsec[k] = 0.0f;
        if (gc) gc[k] = 0.0f;
      }
    }
  }
}

// Compact per-row results back to the original rows: lse[r] (and, when
// given, loss_rows[r]) from compact row pos[r], 0 for rows that took no part.
__global__ void scatter_rows_kernel(const float* __restrict__ lsec, const float* __restrict__ lossc,
                                    const int* __restrict__ pos, int N, float* __restrict__ lse,
                                    float* __restrict__ loss_rows) {
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < N; r += gridDim.x * blockDim.x) {
    const int p = pos[r];
    if (lse) lse[r] = p >= 0 ? lsec[p] : 0.0f;
    if (loss_rows) loss_rows[r] = p >= 0 ? lossc[p] : 0.0f;
  }
}

// dE (bf16) from the compact fp32 accumulator, scattered back to the original
// rows; rows that took no part are exactly +0.
__global__ void finalize_de_kernel(const float4* __restrict__ acc, const int* __restrict__ pos, int N, int D,
                                   uint2* __restrict__ dE) {
  const size_t per_row = static_cast<size_t>(D) / 4;
  const size_t total = static_cast<size_t>(N) * per_row;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = i / per_row;
    const int p = pos[row];  // compact row, or -1 for a row that took no part
    uint2 out = make_uint2(0u, 0u);
    if (p >= 0) {
      const float4 v = acc[static_cast<size_t>(p) * per_row + (i - row * per_row)];
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
      std::memcpy(&out.x, &lo, 4);
      std::memcpy(&out.y, &hi, 4);
    }
    dE[i] = out;
  }
}

// Filter statistics over the token blocks of the compact rows.
__global__ void stats_kernel(const uint8_t* __restrict__ bitmap, const int* __restrict__ count, int bm_ld,
                             int64_t* stats) {
  __shared__ long long sz[1024];
  const long long n = static_cast<long long>((*count + 127) / 128) * bm_ld;
  long long z = 0;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) z += bitmap[i] == 0 ? 1 : 0;
  sz[threadIdx.x] = z;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) sz[threadIdx.x] += sz[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    stats[0] = n;
    stats[1] = sz[0];
  }
}

// ------------------------------------------------------------ host helpers
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int fwd_splits(int64_t N, int64_t V) {
  const int64_t n_blocks = cdiv(N, BM), v_tiles = cdiv(V, BN);
  const int64_t s_max = std::max<int64_t>(1, v_tiles / 4);
  const int64_t base = REF_SMS / std::gcd<int64_t>(n_blocks, REF_SMS);
  int64_t S;
  if (base <= s_max) {
    S = base;
    while (n_blocks * S < 2 * REF_SMS && S + base <= s_max) S += base;
  } else {
    S = std::min<int64_t>(s_max, std::max<int64_t>(1, cdiv(2 * REF_SMS, n_blocks)));
  }
  return static_cast<int>(std::min(S, v_tiles));
}

// Columns of the backward's G-hat chunk [N][vc] bf16 within `budget` bytes
// (0: the default budget, and at least MIN_CHUNK columns; an explicit budget
// goes down to one 256-column tile).
int64_t bwd_chunk_cols(int64_t N, int64_t V, size_t budget = 0) {
  const int64_t vpad = cdiv(V, BN) * BN;
  const bool dflt = budget == 0;
  int64_t vc = static_cast<int64_t>((dflt ? G_CHUNK_BUDGET : budget) / (2 * static_cast<size_t>(N))) / BN * BN;
  vc = std::max<int64_t>(dflt ? MIN_CHUNK : BN, std::min<int64_t>(MAX_CHUNK, vc));
  // At least two chunks whenever V spans more than one tile, so the staging
  // buffer is never an N x V matrix.
  if (V > BN) vc = std::min(vc, cdiv(cdiv(V, 2), BN) * BN);
  return std::min(vc, vpad);
}

// Token blocks per raster group of the logit GEMMs: the group's E rows
// (group_n * 128 * D * 2 bytes) stay around 32 MiB, a quarter of L2.
int raster_group(int64_t n_blocks, int64_t D) {
  return static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>(n_blocks, std::max<int64_t>(8, (int64_t(32) << 20) / (BM * 2 * D)))));
}

// Width of the D tiles of the gradient GEMMs.  Measured on GB300: MMAs with
// N = 256 run fastest (N = 224 about 10% slower per column, N = 192 and 128
// far slower), so tiles are 256 wide even when that pads D (D = 896: 1024),
// and only narrower when D itself is smaller (rounded up to `step`).  Cutting
// D = 896 into 4 x 224 measured 16% slower in the gradient GEMM with the B
// operand in four 64-column 2-D boxes per stage, and still 2% slower with B
// in one 3-D box of seven 64-byte-swizzled 32-column groups, although both
// issue 1/8 fewer MMAs.
int grad_tile_width(int64_t D, int step) {
  if (D >= BN) return BN;
  return static_cast<int>(cdiv(D, step) * step);
}

struct FwdLayout {
  size_t counter, part_m, part_s, tgt, blk_sum, blk_cnt, total;
  // CCE_FWD_SKIP_IGNORED only: compaction map and scratch, compact rows and results
  size_t pos, ridx, count, cscr, xc, ec, lsec, lossc;
  int S, nblk;
};

FwdLayout fwd_layout(int64_t N, int64_t V, int64_t D = 0, bool compact = false) {
  FwdLayout L{};
  L.S = fwd_splits(N, V);
  L.nblk = static_cast<int>(cdiv(N, COMBINE_THREADS));
  size_t o = 0;
  L.counter = o;
  o = align_up(o + sizeof(int), ALIGN);
  L.part_m = o;
  o = align_up(o + sizeof(float) * L.S * N, ALIGN);
  L.part_s = o;
  o = align_up(o + sizeof(float) * L.S * N, ALIGN);
  L.tgt = o;
  o = align_up(o + sizeof(float) * N, ALIGN);
  L.blk_sum = o;
  o = align_up(o + sizeof(double) * L.nblk, ALIGN);
  L.blk_cnt = o;
  o = align_up(o + sizeof(int) * L.nblk, ALIGN);
  if (compact) {
    L.pos = o;
    o = align_up(o + sizeof(int) * static_cast<size_t>(N), ALIGN);
    L.ridx = o;
    o = align_up(o + sizeof(int) * static_cast<size_t>(N), ALIGN);
    L.count = o;
    o = align_up(o + sizeof(int), ALIGN);
    L.cscr = o;
    o = align_up(o + compact_scratch_bytes(N), ALIGN);
    L.xc = o;
    o = align_up(o + sizeof(int64_t) * static_cast<size_t>(N), ALIGN);
    L.ec = o;
    o = align_up(o + static_cast<size_t>(N) * D * 2, ALIGN);
    L.lsec = o;
    o = align_up(o + sizeof(float) * static_cast<size_t>(N), ALIGN);
    L.lossc = o;
    o = align_up(o + sizeof(float) * static_cast<size_t>(N), ALIGN);
  }
  L.total = o;
  return L;
}

struct BwdLayout {
  size_t count, counters, zero, cscr, pos, ridx, xc, lsec, gc, ec, bitmap, bitmapT, gbuf, deacc, total;
  // vocabulary sorting only: sort keys, order and its inverse, scratch, and
  // the chunk of C in sorted order
  size_t keys, perm, inv, sortscr, cs;
  int64_t vc, bm_ld, n128, nchunks;
};

BwdLayout bwd_layout(int64_t N, int64_t D, int64_t V, bool sort = false, size_t budget = 0) {
  BwdLayout L{};
  L.vc = bwd_chunk_cols(N, V, budget);
  L.bm_ld = cdiv(V, 128);
  L.n128 = cdiv(N, 128);
  L.nchunks = cdiv(V, L.vc);
  size_t o = 0;
  L.count = o;
  o = align_up(o + sizeof(int), ALIGN);
  L.counters = o;  // per chunk: the two launches' scheduler counters and the kept filter tiles
  o = align_up(o + sizeof(int) * CHUNK_COUNTERS * static_cast<size_t>(L.nchunks), ALIGN);
  L.zero = o;  // 16 KiB of zeros: the A box of a CTA pair's skipped K-block
  o = align_up(o + ZERO_BOX_BYTES, ALIGN);
  L.cscr = o;  // compaction scratch
  o = align_up(o + compact_scratch_bytes(N), ALIGN);
  L.pos = o;  // compaction map and compact copies of the rows that take part
  o = align_up(o + sizeof(int) * static_cast<size_t>(N), ALIGN);
  L.ridx = o;
  o = align_up(o + sizeof(int) * static_cast<size_t>(N), ALIGN);
  L.xc = o;
  o = align_up(o + sizeof(int64_t) * static_cast<size_t>(N), ALIGN);
  L.lsec = o;
  o = align_up(o + sizeof(float) * static_cast<size_t>(N), ALIGN);
  L.gc = o;
  o = align_up(o + sizeof(float) * static_cast<size_t>(N), ALIGN);
  L.ec = o;
  o = align_up(o + static_cast<size_t>(N) * D * 2, ALIGN);
  L.bitmap = o;
  o = align_up(o + static_cast<size_t>(L.n128 * L.bm_ld), ALIGN);
  L.bitmapT = o;
  o = align_up(o + static_cast<size_t>(L.n128 * L.bm_ld), ALIGN);
  L.gbuf = o;
  o = align_up(o + static_cast<size_t>(N) * L.vc * 2, ALIGN);
  L.deacc = o;
  o = align_up(o + static_cast<size_t>(N) * D * 4, ALIGN);
  if (sort) {
    L.keys = o;
    o = align_up(o + sizeof(float) * static_cast<size_t>(V), ALIGN);
    L.perm = o;
    o = align_up(o + sizeof(int) * static_cast<size_t>(V), ALIGN);
    L.inv = o;
    o = align_up(o + sizeof(int) * static_cast<size_t>(V), ALIGN);
    L.sortscr = o;
    o = align_up(o + std::max(vocab_keys_scratch_bytes(N, D), vocab_order_scratch_bytes(V)), ALIGN);
    L.cs = o;
    o = align_up(o + static_cast<size_t>(L.vc) * D * 2, ALIGN);
  }
  L.total = o;
  return L;
}

// Single call: the rows that take part are compacted first (pos, ridx, the
// compact E and x), then token chunks of Nc compact rows (a multiple of 256) whose staged
// logits, fp16 [Nc][Vp] with Vp = V rounded up to 256, fit in max_staging
// bytes (at least one 256-row chunk); per chunk the forward partials, the
// 32-column chunk maxima and the survival maps; dE in de_splits fp32 slabs of
// roundup(N, 128) rows; with more than one chunk an fp32 dC accumulator.
constexpr size_t FLCE_STAGING_DEFAULT = size_t(2) << 30;

struct FlceLayout {
  size_t counters, count, zero, cscr, pos, ridx, xc, ec, part_m, part_s, tgt, lse, blk_sum, blk_cnt, stage, mtile,
      bitmap, bitmapT, deacc, dcacc, total;
  int64_t Nc, nchunks, Vp, bm_ld, slab, n_tiles, bn, kps;
  int S, Sde, nblk;
};

FlceLayout flce_layout(int64_t N, int64_t D, int64_t V, size_t max_staging) {
  FlceLayout L{};
  if (max_staging == 0) max_staging = FLCE_STAGING_DEFAULT;
  L.Vp = cdiv(V, 256) * 256;
  const int64_t fit = static_cast<int64_t>(max_staging / (static_cast<size_t>(L.Vp) * 2)) / 256 * 256;
  L.Nc = std::min(std::max<int64_t>(256, fit), cdiv(N, 256) * 256);
  L.nchunks = cdiv(N, L.Nc);
  L.bm_ld = cdiv(V, 128);
  L.slab = cdiv(N, 128) * 128;
  L.S = fwd_splits(L.Nc, V);
  L.nblk = static_cast<int>(cdiv(N, COMBINE_THREADS));
  // dE: split the vocabulary (K) so that no dE tile is much longer than the
  // average work per SM of a chunk's gradient launch
  L.bn = grad_tile_width(D, D % 64 == 0 ? 64 : 32);
  L.n_tiles = cdiv(D, L.bn);
  const int64_t nb = L.Nc / BM, kde = cdiv(V, BK);
  const double units = static_cast<double>(nb * L.n_tiles) * kde + static_cast<double>(cdiv(V, BM) * L.n_tiles) * 2 * nb;
  const double avg = std::max(1.0, units / REF_SMS);
  L.Sde = static_cast<int>(std::min<double>(8.0, std::max(1.0, std::ceil(kde / avg))));
  L.kps = cdiv(cdiv(kde, L.Sde), 2) * 2;
  L.Sde = static_cast<int>(cdiv(kde, L.kps));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, ALIGN);
    return at;
  };
  L.counters = take(sizeof(int) * CHUNK_COUNTERS * static_cast<size_t>(L.nchunks));
  L.count = take(sizeof(int));
  L.zero = take(ZERO_BOX_BYTES);  // the A box of a CTA pair's skipped K-block
  L.cscr = take(compact_scratch_bytes(N));
  L.pos = take(sizeof(int) * static_cast<size_t>(N));
  L.ridx = take(sizeof(int) * static_cast<size_t>(N));
  L.xc = take(sizeof(int64_t) * static_cast<size_t>(N));
  L.ec = take(static_cast<size_t>(N) * D * 2);
  L.part_m = take(sizeof(float) * L.S * static_cast<size_t>(L.Nc));
  L.part_s = take(sizeof(float) * L.S * static_cast<size_t>(L.Nc));
  L.tgt = take(sizeof(float) * static_cast<size_t>(L.Nc));
  L.lse = take(sizeof(float) * static_cast<size_t>(N));
  L.blk_sum = take(sizeof(double) * L.nblk);
  L.blk_cnt = take(sizeof(int) * L.nblk);
  L.stage = take(static_cast<size_t>(L.Nc) * L.Vp * 2);
  L.mtile = take(sizeof(float) * static_cast<size_t>(L.Vp / 32) * L.Nc);
  L.bitmap = take(static_cast<size_t>(L.Nc / BM) * L.bm_ld);
  L.bitmapT = take(static_cast<size_t>(L.Nc / BM) * L.bm_ld);
  L.deacc = take(sizeof(float) * static_cast<size_t>(L.Sde) * L.slab * D);
  L.dcacc = take(L.nchunks > 1 ? sizeof(float) * static_cast<size_t>(V) * D : 0);
  L.total = o;
  return L;
}

bool sizes_ok(int64_t N, int64_t D, int64_t V) {
  const int64_t lim = int64_t(1) << 31;
  return N >= 1 && N < lim && V >= 1 && V < lim && D >= 8 && D < lim && D % 8 == 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------- device state
struct DeviceInfo {
  bool init = false;
  bool ok = false;
  int sms = 0;
  int pair_clusters = 0;  // CTA pairs of the forward GEMM resident at once
};
std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cce_status device_check(int* sms, int* pair_clusters = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return CCE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return CCE_ERR_CUDA;
    }
    d.ok = (major == 10 && minor == 3);
    d.sms = sms;
    if (d.ok) {
      if (prepare_gemm_kernels() != cudaSuccess) {
        cudaGetLastError();
        return CCE_ERR_CUDA;
      }
      d.pair_clusters = gemm_pair_clusters(sms);
      if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          cudaGetLastError();
          return CCE_ERR_CUDA;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    d.init = true;
  }
  if (!d.ok) return CCE_ERR_DEVICE;
  *sms = d.sms;
  if (pair_clusters) *pair_clusters = d.pair_clusters;
  return CCE_OK;
}

// 2-D row-major tensor map; the box's inner extent is the swizzle span (128 B
// by default, 64 B for the dC store box).
bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* ptr, uint64_t inner,
               uint64_t outer, uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_elems * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 [rows][D] viewed as {64 d, rows, D / 64 groups} with box {64,
// box_rows, groups}: one TMA instruction brings all 64-column groups of an
// MN-major operand stage (D % 64 == 0, so the view never reaches past a row).
// The same view of a K-major operand (D = K) brings box_rows rows of `groups`
// consecutive 64-column K-blocks, one after the other.
bool make_tmap_mn3(CUtensorMap* m, const void* ptr, uint64_t D, uint64_t rows, uint32_t groups = 4,
                   uint32_t box_rows = 64) {
  cuuint64_t dims[3] = {64, rows, D / 64};
  cuuint64_t strides[2] = {D * 2, 128};
  cuuint32_t box[3] = {64, box_rows, groups};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// CTA pairs (FWD, BWD_G), whose stages are 128 deep in K: A = E (n rows)
// in boxes of 128 rows and B = C (or a chunk of sorted C rows, `rows` of
// them) in 128-row boxes, each CTA's half of a 256-row tile, both as two
// 64-column K groups in one 3-D box (D % 64 == 0); raster groups hold whole
// pairs.
bool pair_operands(GemmArgs* a, const void* E, int64_t n, const void* C, int64_t D, int64_t rows) {
  a->group_n = std::max(2, a->group_n & ~1);
  return make_tmap_mn3(&a->tmA, E, D, n, 2, BM) && make_tmap_mn3(&a->tmB2, C, D, rows, 2, BN / 2);
}

// ---------------------------------------------------------- phase timing
struct PhaseRec {
  int phase;
  cudaEvent_t a, b;
};
bool g_prof = false;
std::vector<PhaseRec> g_recs;
std::vector<cudaEvent_t> g_pool;
double g_ms[CCE_NUM_PHASES];
int64_t g_cnt[CCE_NUM_PHASES];

cudaEvent_t pool_get() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct PhaseScope {
  bool on;
  PhaseRec rec;
  cudaStream_t s;
  PhaseScope(int phase, cudaStream_t st) : on(false), s(st) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_prof) return;
    rec.phase = phase;
    rec.a = pool_get();
    rec.b = pool_get();
    on = rec.a && rec.b;
    if (on) cudaEventRecord(rec.a, s);
  }
  ~PhaseScope() {
    if (!on) return;
    cudaEventRecord(rec.b, s);
    std::lock_guard<std::mutex> lk(g_mu);
    g_recs.push_back(rec);
  }
};

cce_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CCE_OK;
  return CCE_ERR_CUDA;
}

}  // namespace
}  // namespace cce

using namespace cce;

extern "C" {

int cce_abi_version(void) { return 101; }

uint64_t cce_kernel_launch_count(void) { return g_launches.load(); }

const char* cce_status_string(cce_status s) {
  switch (s) {
    case CCE_OK: return "ok";
    case CCE_ERR_NULL: return "null pointer";
    case CCE_ERR_SHAPE: return "bad shape (need 1 <= N, V < 2^31; 8 <= D < 2^31, D % 8 == 0)";
    case CCE_ERR_ALIGN: return "buffer not 16-byte aligned";
    case CCE_ERR_ARG: return "bad argument (reduction or filter_eps)";
    case CCE_ERR_WORKSPACE: return "workspace too small";
    case CCE_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
    case CCE_ERR_CUDA: return "CUDA error";
    case CCE_ERR_TARGET_RANGE: return "target index outside [0, V) and not ignore_index";
    case CCE_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
  }
  return "unknown status";
}

size_t cce_forward_workspace_bytes(int64_t N, int64_t D, int64_t V) {
  if (!sizes_ok(N, D, V)) return 0;
  return fwd_layout(N, V).total;
}

size_t cce_backward_workspace_bytes(int64_t N, int64_t D, int64_t V) {
  if (!sizes_ok(N, D, V)) return 0;
  return bwd_layout(N, D, V).total;
}

size_t cce_backward_workspace_bytes_ex(int64_t N, int64_t D, int64_t V, int flags) {
  return cce_backward_workspace_bytes_ex2(N, D, V, flags, 0);
}

size_t cce_backward_workspace_bytes_ex2(int64_t N, int64_t D, int64_t V, int flags, size_t max_staging_bytes) {
  if (!sizes_ok(N, D, V) || (flags & ~(CCE_FILTER_BOTH | CCE_SORT_VOCAB))) return 0;
  return bwd_layout(N, D, V, (flags & CCE_SORT_VOCAB) != 0, max_staging_bytes).total;
}

uint64_t cce_backward_chunk_cols(int64_t N, int64_t V, size_t max_staging_bytes) {
  if (!sizes_ok(N, 8, V)) return 0;
  return static_cast<uint64_t>(bwd_chunk_cols(N, V, max_staging_bytes));
}

size_t cce_vocab_sort_workspace_bytes(int64_t N, int64_t D, int64_t V) {
  if (!sizes_ok(N, D, V)) return 0;
  return std::max(vocab_keys_scratch_bytes(N, D), vocab_order_scratch_bytes(V));
}

cce_status cce_vocab_logit_sums(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                                int64_t ignore_index, float* sums, void* workspace, size_t ws_bytes, void* stream) {
  if (!E || !C || !x || !sums || !workspace) return CCE_ERR_NULL;
  if (!sizes_ok(N, D, V)) return CCE_ERR_SHAPE;
  if (!aligned16(E) || !aligned16(C) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(x) & 7u) ||
      (reinterpret_cast<uintptr_t>(sums) & 3u))
    return CCE_ERR_ALIGN;
  if (ws_bytes < cce_vocab_sort_workspace_bytes(N, D, V)) return CCE_ERR_WORKSPACE;
  int sms = 0;
  cce_status st = device_check(&sms);
  if (st != CCE_OK) return st;
  int launched = 0;
  cudaError_t e = launch_vocab_keys(E, N, nullptr, x, static_cast<long long>(ignore_index), D, C, V, sums,
                                    workspace, static_cast<cudaStream_t>(stream), sms, &launched);
  g_launches += static_cast<uint64_t>(launched);
  return cuda_status(e);
}

cce_status cce_vocab_order(const float* keys, int64_t V, int32_t* perm, void* workspace, size_t ws_bytes,
                           void* stream) {
  if (!keys || !perm || !workspace) return CCE_ERR_NULL;
  if (!sizes_ok(1, 8, V)) return CCE_ERR_SHAPE;
  if (!aligned16(workspace) || (reinterpret_cast<uintptr_t>(keys) & 3u) || (reinterpret_cast<uintptr_t>(perm) & 3u))
    return CCE_ERR_ALIGN;
  if (ws_bytes < vocab_order_scratch_bytes(V)) return CCE_ERR_WORKSPACE;
  int sms = 0;
  cce_status st = device_check(&sms);
  if (st != CCE_OK) return st;
  int launched = 0;
  cudaError_t e = launch_vocab_order(keys, V, perm, workspace, static_cast<cudaStream_t>(stream), &launched, nullptr);
  g_launches += static_cast<uint64_t>(launched);
  return cuda_status(e);
}

cce_status cce_memory_accounting(int64_t N, int64_t D, int64_t V, cce_memory_report* out) {
  if (!out) return CCE_ERR_NULL;
  if (!sizes_ok(N, D, V)) return CCE_ERR_SHAPE;
  out->logits_fp32_bytes = static_cast<uint64_t>(N) * V * 4;
  out->dE_bytes = static_cast<uint64_t>(N) * D * 2;
  out->dC_bytes = static_cast<uint64_t>(V) * D * 2;
  out->lse_bytes = static_cast<uint64_t>(N) * 4;
  out->fwd_workspace_bytes = fwd_layout(N, V).total;
  const BwdLayout b = bwd_layout(N, D, V);
  out->bwd_workspace_bytes = b.total;
  out->bwd_chunk_cols = static_cast<uint64_t>(b.vc);
  out->fwd_vocab_splits = static_cast<uint64_t>(fwd_layout(N, V).S);
  return CCE_OK;
}

cce_status cce_forward(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                       int64_t ignore_index, int reduction, float* loss, float* lse, void* workspace,
                       size_t ws_bytes, int32_t* dev_err, void* stream) {
  return cce_forward_ex(E, C, x, N, D, V, ignore_index, reduction, 0.0f, loss, lse, workspace, ws_bytes, dev_err,
                        stream);
}

static cce_status forward_impl(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                               int64_t ignore_index, int reduction, float softcap, int flags, float* loss, float* lse,
                               void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!E || !C || !x || !loss || !lse || !workspace) return CCE_ERR_NULL;
  if (!sizes_ok(N, D, V)) return CCE_ERR_SHAPE;
  if (!aligned16(E) || !aligned16(C) || !aligned16(loss) || !aligned16(lse) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(x) & 7u))
    return CCE_ERR_ALIGN;
  if (reduction != CCE_RED_NONE && reduction != CCE_RED_SUM && reduction != CCE_RED_MEAN) return CCE_ERR_ARG;
  if (!(softcap >= 0.0f) || !std::isfinite(softcap)) return CCE_ERR_ARG;
  if (flags & ~CCE_FWD_SKIP_IGNORED) return CCE_ERR_ARG;
  const bool compact = (flags & CCE_FWD_SKIP_IGNORED) != 0;
  const FwdLayout W = fwd_layout(N, V, D, compact);
  if (ws_bytes < W.total) return CCE_ERR_WORKSPACE;
  int sms = 0, pair_clusters = 0;
  cce_status st = device_check(&sms, &pair_clusters);
  if (st != CCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  // Skipping ignored rows ("Cut Your Losses ...", Table A1: removing ignored
  // tokens): the rows that take part are compacted first and the GEMM runs
  // over them only, with their count read from device memory.
  const void* Eg = E;
  const int64_t* xg = x;
  int* count = nullptr;
  int* pos = nullptr;
  if (compact) {
    PhaseScope ps(2, s);
    count = reinterpret_cast<int*>(ws + W.count);
    pos = reinterpret_cast<int*>(ws + W.pos);
    int* ridx = reinterpret_cast<int*>(ws + W.ridx);
    int64_t* xc = reinterpret_cast<int64_t*>(ws + W.xc);
    void* Ec = ws + W.ec;
    {
      cudaError_t ce = launch_compact(x, N, V, static_cast<long long>(ignore_index), pos, ridx, count,
                                      reinterpret_cast<int*>(ws + W.cscr), dev_err, s);
      g_launches += 3;
      if (ce != cudaSuccess) return cuda_status(ce);
    }
    const int rows_per_block = 8;
    const int blocks = static_cast<int>(std::min<int64_t>(int64_t(sms) * 16, cdiv(N, rows_per_block)));
    gather_rows_kernel<<<std::max(blocks, 1), 32 * rows_per_block, 0, s>>>(
        static_cast<const uint4*>(E), x, nullptr, nullptr, ridx, count, static_cast<int>(N), static_cast<int>(D),
        static_cast<long long>(ignore_index), static_cast<uint4*>(Ec), xc, nullptr, nullptr);
    g_launches++;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    Eg = Ec;
    xg = xc;
  }

  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  // A = E [N, D]: box 64 (D) x 128 rows.  B = C [V, D]: box 64 (D) x 256 rows.
  if (!make_tmap(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Eg, D, N, D, BK, BM) ||
      !make_tmap(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, D, V, D, BK, BN))
    return CCE_ERR_CUDA;
  a.tmOut = a.tmA;  // unused
  a.N = static_cast<int>(N);
  a.D = static_cast<int>(D);
  a.V = static_cast<int>(V);
  a.n_blocks = static_cast<int>(cdiv(N, BM));
  a.k_blocks = static_cast<int>(cdiv(D, BK));
  a.splits = W.S;
  a.v_tiles = static_cast<int>(cdiv(V, BN));
  a.group_n = raster_group(a.n_blocks, D);
  a.x = xg;
  a.ignore_index = ignore_index;
  a.part_m = reinterpret_cast<float*>(ws + W.part_m);
  a.part_s = reinterpret_cast<float*>(ws + W.part_s);
  a.tgt = reinterpret_cast<float*>(ws + W.tgt);
  a.softcap = softcap;
  a.inv_softcap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
  a.dev_err = dev_err;
  a.counter = reinterpret_cast<int*>(ws + W.counter);
  a.n_dev = count;  // null without compaction: all N rows
  // Clusters of two CTAs share each MMA (M = 256), each CTA loading its 128
  // rows of E and half of the C tile, so a CTA moves two thirds of the
  // operand bytes per MMA.
  const bool pairs = pair_clusters > 0 && D % 64 == 0;
  if (pairs && !pair_operands(&a, Eg, N, C, D, V)) return CCE_ERR_CUDA;
  const int units = pairs ? ((a.n_blocks + 1) / 2) * a.splits : a.n_blocks * a.splits;
  a.items = units;
  {
    PhaseScope ps(0, s);
    cudaError_t e = cudaMemsetAsync(a.counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_status(e);
    e = pairs ? launch_gemm_pairs(MODE_FWD, a, std::min(units, pair_clusters), s)
              : launch_gemm(MODE_FWD, a, std::min(units, sms), s);
    g_launches++;
    if (e != cudaSuccess) return cuda_status(e);
  }
  {
    PhaseScope ps(1, s);
    float* lse_out = compact ? reinterpret_cast<float*>(ws + W.lsec) : lse;
    float* loss_rows = (reduction == CCE_RED_NONE) ? (compact ? reinterpret_cast<float*>(ws + W.lossc) : loss)
                                                   : nullptr;
    combine_kernel<<<W.nblk, COMBINE_THREADS, 0, s>>>(
        a.part_m, a.part_s, a.tgt, xg, a.N, W.S, a.V, static_cast<long long>(ignore_index), reduction, lse_out,
        loss_rows, reinterpret_cast<double*>(ws + W.blk_sum), reinterpret_cast<int*>(ws + W.blk_cnt), dev_err,
        count, 0);
    g_launches++;
    if (reduction != CCE_RED_NONE) {
      finish_loss_kernel<<<1, COMBINE_THREADS, 0, s>>>(reinterpret_cast<double*>(ws + W.blk_sum),
                                                       reinterpret_cast<int*>(ws + W.blk_cnt), W.nblk, reduction,
                                                       loss);
      g_launches++;
    }
    if (compact) {  // back to the original rows; rows that took no part get 0
      scatter_rows_kernel<<<static_cast<unsigned>(std::min<int64_t>(int64_t(sms) * 8, cdiv(N, 256))), 256, 0, s>>>(
          lse_out, loss_rows, pos, static_cast<int>(N), lse, reduction == CCE_RED_NONE ? loss : nullptr);
      g_launches++;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }
  return CCE_OK;
}

cce_status cce_forward_ex(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                          int64_t ignore_index, int reduction, float softcap, float* loss, float* lse,
                          void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  return forward_impl(E, C, x, N, D, V, ignore_index, reduction, softcap, 0, loss, lse, workspace, ws_bytes, dev_err,
                      stream);
}

cce_status cce_forward_ex2(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                           int64_t ignore_index, int reduction, float softcap, int flags, float* loss, float* lse,
                           void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  return forward_impl(E, C, x, N, D, V, ignore_index, reduction, softcap, flags, loss, lse, workspace, ws_bytes,
                      dev_err, stream);
}

size_t cce_forward_workspace_bytes_ex(int64_t N, int64_t D, int64_t V, int flags) {
  if (!sizes_ok(N, D, V) || (flags & ~CCE_FWD_SKIP_IGNORED)) return 0;
  return fwd_layout(N, V, D, (flags & CCE_FWD_SKIP_IGNORED) != 0).total;
}

cce_status cce_backward(const void* E, const void* C, const int64_t* x, const float* lse, const float* grad_out,
                        int64_t N, int64_t D, int64_t V, int64_t ignore_index, int reduction, float filter_eps,
                        void* dE, void* dC, void* workspace, size_t ws_bytes, int32_t* dev_err,
                        int64_t* dev_stats, void* stream) {
  return cce_backward_ex(E, C, x, lse, grad_out, N, D, V, ignore_index, reduction, 0.0f, filter_eps,
                         CCE_FILTER_BOTH, dE, dC, workspace, ws_bytes, dev_err, dev_stats, stream);
}

cce_status cce_backward_ex(const void* E, const void* C, const int64_t* x, const float* lse, const float* grad_out,
                           int64_t N, int64_t D, int64_t V, int64_t ignore_index, int reduction, float softcap,
                           float filter_eps, int filter_flags, void* dE, void* dC, void* workspace, size_t ws_bytes,
                           int32_t* dev_err, int64_t* dev_stats, void* stream) {
  return cce_backward_ex2(E, C, x, lse, grad_out, N, D, V, ignore_index, reduction, softcap, filter_eps, filter_flags,
                          0, dE, dC, workspace, ws_bytes, dev_err, dev_stats, stream);
}

cce_status cce_backward_ex2(const void* E, const void* C, const int64_t* x, const float* lse, const float* grad_out,
                            int64_t N, int64_t D, int64_t V, int64_t ignore_index, int reduction, float softcap,
                            float filter_eps, int filter_flags, size_t max_staging_bytes, void* dE, void* dC,
                            void* workspace, size_t ws_bytes, int32_t* dev_err, int64_t* dev_stats, void* stream) {
  if (!E || !C || !x || !lse || !grad_out || !dE || !dC || !workspace) return CCE_ERR_NULL;
  if (!sizes_ok(N, D, V)) return CCE_ERR_SHAPE;
  if (!aligned16(E) || !aligned16(C) || !aligned16(lse) || !aligned16(dE) || !aligned16(dC) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(x) & 7u) || (reinterpret_cast<uintptr_t>(grad_out) & 3u) ||
      (reinterpret_cast<uintptr_t>(dev_stats) & 7u))
    return CCE_ERR_ALIGN;
  if (reduction != CCE_RED_NONE && reduction != CCE_RED_SUM && reduction != CCE_RED_MEAN) return CCE_ERR_ARG;
  if (!(filter_eps >= 0.0f) || !std::isfinite(filter_eps)) return CCE_ERR_ARG;
  if (filter_flags & ~(CCE_FILTER_BOTH | CCE_SORT_VOCAB)) return CCE_ERR_ARG;
  if (!(softcap >= 0.0f) || !std::isfinite(softcap)) return CCE_ERR_ARG;
  const bool sort = (filter_flags & CCE_SORT_VOCAB) != 0;
  const BwdLayout W = bwd_layout(N, D, V, sort, max_staging_bytes);
  if (ws_bytes < W.total) return CCE_ERR_WORKSPACE;
  int sms = 0, pair_clusters = 0;
  cce_status st = device_check(&sms, &pair_clusters);
  if (st != CCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* count = reinterpret_cast<int*>(ws + W.count);
  uint8_t* bitmap = ws + W.bitmap;
  void* gbuf = ws + W.gbuf;
  float* deacc = reinterpret_cast<float*>(ws + W.deacc);

  // Compact away the rows that take no part ("Cut Your Losses ...", Table A1:
  // removing ignored tokens); the GEMMs below read the count from the device.
  int* pos = reinterpret_cast<int*>(ws + W.pos);
  int* ridx = reinterpret_cast<int*>(ws + W.ridx);
  int64_t* xc = reinterpret_cast<int64_t*>(ws + W.xc);
  float* lsec = reinterpret_cast<float*>(ws + W.lsec);
  float* gc = reinterpret_cast<float*>(ws + W.gc);
  void* Ec = ws + W.ec;
  {
    PhaseScope ps(2, s);
    {
      cudaError_t ce = launch_compact(x, N, V, static_cast<long long>(ignore_index), pos, ridx, count,
                                      reinterpret_cast<int*>(ws + W.cscr), dev_err, s);
      g_launches += 3;
      if (ce != cudaSuccess) return cuda_status(ce);
    }
    const int rows_per_block = 8;
    const int blocks = static_cast<int>(std::min<int64_t>(int64_t(sms) * 16, cdiv(N, rows_per_block)));
    gather_rows_kernel<<<std::max(blocks, 1), 32 * rows_per_block, 0, s>>>(
        static_cast<const uint4*>(E), x, lse, grad_out, ridx, count, static_cast<int>(N), static_cast<int>(D),
        static_cast<long long>(ignore_index), static_cast<uint4*>(Ec), xc, lsec,
        reduction == CCE_RED_NONE ? gc : nullptr);
    g_launches++;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }
  // Vocabulary sorting ("Cut Your Losses ...", section "Vocabulary
  // Sorting"): order the vocabulary by the logit sum over the compact rows,
  // and move every compact target to its sorted position.  The chunks below
  // then cover consecutive sorted positions.
  int* perm = sort ? reinterpret_cast<int*>(ws + W.perm) : nullptr;
  void* Cs = sort ? static_cast<void*>(ws + W.cs) : nullptr;
  if (sort) {
    PhaseScope ps(6, s);
    int launched = 0;
    float* keys = reinterpret_cast<float*>(ws + W.keys);
    void* scr = ws + W.sortscr;
    cudaError_t e = launch_vocab_keys(Ec, N, count, nullptr, 0, D, C, V, keys, scr, s, sms, &launched);
    int* inv = reinterpret_cast<int*>(ws + W.inv);
    if (e == cudaSuccess) e = launch_vocab_order(keys, V, perm, scr, s, &launched, inv);
    if (e == cudaSuccess) e = launch_remap_targets(inv, xc, count, N, s, sms, &launched);
    g_launches += static_cast<uint64_t>(launched);
    if (e != cudaSuccess) return cuda_status(e);
  }

  GemmArgs g;  // recompute + G
  std::memset(&g, 0, sizeof(g));
  GemmArgs r;  // dC and dE of the chunk
  std::memset(&r, 0, sizeof(r));
  const uint64_t vc = static_cast<uint64_t>(W.vc);
  bool ok = true;
  // C as the GEMMs see it: the whole tensor, or (sorted) one chunk's rows
  // gathered into sorted order; sorted dC tiles write their token rows of dC
  // directly (dc_rows), unsorted ones through the dC tensor map
  const void* Cg = sort ? Cs : C;
  const uint64_t c_rows = sort ? vc : static_cast<uint64_t>(V);
  ok &= make_tmap(&g.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ec, D, N, D, BK, BM);
  ok &= make_tmap(&g.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Cg, D, c_rows, D, BK, BN);
  ok &= make_tmap(&g.tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, gbuf, vc, N, vc, 64, 32);
  r.b3d = (D % 64 == 0) ? 1 : 0;
  ok &= make_tmap_mn3(&r.tmA, gbuf, vc, N, BM / 64);  // G chunk, MN-major A of dC (vc % 256 == 0)
  if (r.b3d) {
    ok &= make_tmap_mn3(&r.tmB, Ec, D, N);
    ok &= make_tmap_mn3(&r.tmB2, Cg, D, c_rows);
  } else {
    ok &= make_tmap(&r.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ec, D, N, D, 64, 64);
    ok &= make_tmap(&r.tmB2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Cg, D, c_rows, D, 64, 64);
  }
  ok &= make_tmap(&r.tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dC, D, V, D, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  ok &= make_tmap(&r.tmA2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, gbuf, vc, N, vc, 64, BM);
  ok &= make_tmap(&r.tmOut2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, deacc, D, N, D, 32, 32);
  if (!ok) return CCE_ERR_CUDA;

  for (GemmArgs* p : {&g, &r}) {
    p->N = static_cast<int>(N);
    p->D = static_cast<int>(D);
    p->V = static_cast<int>(V);
    p->n_blocks = static_cast<int>(cdiv(N, BM));
    p->x = xc;  // every per-row input in compact order
    // sorted: targets are sorted positions in [0, V) and the padding rows
    // hold -1, so no compact target can collide with the ignore index
    p->ignore_index = sort ? -1 : ignore_index;
    p->lse = lsec;
    p->grad_out = reduction == CCE_RED_NONE ? gc : grad_out;
    p->count = count;
    p->n_dev = count;
    p->reduction = reduction;
    p->eps = filter_eps;
    p->softcap = softcap;
    p->inv_softcap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
    p->filter_de = (filter_flags & CCE_FILTER_DE) ? 1 : 0;
    p->filter_dc = (filter_flags & CCE_FILTER_DC) ? 1 : 0;
    p->bitmap = bitmap;
    p->bitmapT = ws + W.bitmapT;
    p->bm_ld = static_cast<int>(W.bm_ld);
    p->dev_err = dev_err;
  }
  g.k_blocks = static_cast<int>(cdiv(D, BK));
  g.group_n = raster_group(cdiv(N, BM), D);
  // The recompute as CTA pairs (see forward_impl) when there are many token
  // blocks.  Its items are single tiles taken in a fixed order, and with an
  // odd number of compacted blocks the last pair runs half empty; at 32
  // blocks (the Qwen shape) that cost more than the pairs saved (0.737 ->
  // 0.777 ms), at 64 and 128 blocks the pairs won (Llama: 9.85 -> 9.48 ms).
  const bool pairs = pair_clusters > 0 && cdiv(N, BM) >= PAIR_MIN_BLOCKS && D % 64 == 0;
  if (pairs && !pair_operands(&g, Ec, N, Cg, D, c_rows)) return CCE_ERR_CUDA;
  r.bn = grad_tile_width(D, r.b3d ? 64 : 32);
  r.n_tiles = static_cast<int>(cdiv(D, r.bn));
  // The gradient GEMM as CTA pairs (M = 256, each CTA loading its own 128 A
  // rows and half of the MN-major B tile, K = 128 per stage) when the D tiles
  // are 256 wide and B comes in 3-D boxes: every operand is one 3-D box of
  // two 64-column groups and 128 rows.
  const int layout = g_grad_layout.load();
  const bool grad_pairs = pair_clusters > 0 && r.b3d && r.bn == BN && layout != 2;
  // With the filter on, one CTA per tile is launched beside the pairs and the
  // chunk's kept-tile count picks the one that runs (pairs run the union of
  // two tiles' K-blocks, which costs more than it saves when many are skipped)
  const bool dual = grad_pairs && (r.filter_de || r.filter_dc) && layout == 0;
  GemmArgs rs = r;  // the one-CTA-per-tile layout
  if (grad_pairs) {
    ok &= make_tmap_mn3(&r.tmA, gbuf, vc, N, 2, PAIR_BK);  // dC: 128 vocabulary columns x 128 tokens (K)
    ok &= make_tmap_mn3(&r.tmA2, gbuf, vc, N, 2, BM);      // dE: 128 tokens x two 64-column K-blocks
    ok &= make_tmap_mn3(&r.tmB, Ec, D, N, 2, PAIR_BK);
    ok &= make_tmap_mn3(&r.tmB2, Cg, D, c_rows, 2, PAIR_BK);
    ok &= make_tmap(&r.tmZ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws + W.zero, 64, 2 * BM, 64, 64, 2 * BM);
    if (!ok) return CCE_ERR_CUDA;
    r.pair_words = g_pair_words.load();
    cudaError_t e = cudaMemsetAsync(ws + W.zero, 0, ZERO_BOX_BYTES, s);
    if (e != cudaSuccess) return cuda_status(e);
  }

  int* counters = reinterpret_cast<int*>(ws + W.counters);
  {
    cudaError_t e = cudaMemsetAsync(counters, 0, sizeof(int) * CHUNK_COUNTERS * static_cast<size_t>(W.nchunks), s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  for (int64_t ch = 0; ch < W.nchunks; ++ch) {
    const int v0 = static_cast<int>(ch * W.vc);
    const int w = static_cast<int>(std::min<int64_t>(W.vc, V - v0));
    for (GemmArgs* p : {&g, &r}) {
      p->chunk_v0 = v0;
      p->chunk_w = w;
      p->c_row0 = sort ? 0 : v0;
    }
    r.dc_rows = sort ? perm + v0 : nullptr;
    r.dC_out = static_cast<uint16_t*>(dC);
    g.v_tiles = static_cast<int>(cdiv(w, BN));
    g.counter = counters + CHUNK_COUNTERS * ch;
    r.dc_m_tiles = static_cast<int>(cdiv(w, BM));
    r.de_k_blocks = static_cast<int>(cdiv(w, BK));
    r.dc_first = cdiv(N, BK) >= r.de_k_blocks ? 1 : 0;  // longest tiles first
    r.first_chunk = (ch == 0) ? 1 : 0;
    r.counter = counters + CHUNK_COUNTERS * ch + 1;
    // filter on: both gradient-GEMM layouts are launched, the kept-tile count
    // of the chunk's recompute picks the one that runs
    g.kept_tiles = dual ? counters + CHUNK_COUNTERS * ch + 2 : nullptr;
    r.kept_tiles = g.kept_tiles;
    cudaError_t e;
    if (sort) {  // the chunk's C rows in sorted order, zero rows up to the last 256-row tile
      PhaseScope ps(6, s);
      int launched = 0;
      e = launch_gather_vocab_rows(C, perm + v0, w, std::min<int64_t>(W.vc, cdiv(w, BN) * BN), D, Cs, s, sms,
                                   &launched);
      g_launches += static_cast<uint64_t>(launched);
      if (e != cudaSuccess) return cuda_status(e);
    }
    {
      PhaseScope ps(3, s);
      e = pairs ? launch_gemm_pairs(MODE_BWD_G, g, std::min(pair_clusters, ((g.n_blocks + 1) / 2) * g.v_tiles), s)
                : launch_gemm(MODE_BWD_G, g, std::min(sms, g.n_blocks * g.v_tiles), s);
      g_launches++;
      if (e != cudaSuccess) return cuda_status(e);
    }
    {
      PhaseScope ps(4, s);
      if (grad_pairs) {
        const int items = ((r.dc_m_tiles + 1) / 2 + (r.n_blocks + 1) / 2) * r.n_tiles;
        r.grad_path = dual ? 1 : -1;
        e = launch_gemm_pairs(MODE_GRAD, r, std::min(pair_clusters, items), s);
        g_launches++;
        if (e == cudaSuccess && dual) {
          GemmArgs one = r;  // the same chunk, one CTA per tile
          one.tmA = rs.tmA;
          one.tmA2 = rs.tmA2;
          one.tmB = rs.tmB;
          one.tmB2 = rs.tmB2;
          one.grad_path = 0;
          e = launch_gemm(MODE_GRAD, one, std::min(sms, (one.dc_m_tiles + one.n_blocks) * one.n_tiles), s);
          g_launches++;
        }
      } else {
        r.grad_path = -1;
        e = launch_gemm(MODE_GRAD, r, std::min(sms, (r.dc_m_tiles + r.n_blocks) * r.n_tiles), s);
        g_launches++;
      }
      if (e != cudaSuccess) return cuda_status(e);
    }
  }
  {
    PhaseScope ps(5, s);
    const size_t n4 = static_cast<size_t>(N) * D / 4;
    const int blocks = static_cast<int>(std::min<size_t>(static_cast<size_t>(sms) * 8, (n4 + 255) / 256));
    finalize_de_kernel<<<std::max(blocks, 1), 256, 0, s>>>(reinterpret_cast<const float4*>(deacc), pos,
                                                           static_cast<int>(N), static_cast<int>(D),
                                                           static_cast<uint2*>(dE));
    g_launches++;
    if (dev_stats) {
      stats_kernel<<<1, 1024, 0, s>>>(bitmap, count, static_cast<int>(W.bm_ld), dev_stats);
      g_launches++;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }
  return CCE_OK;
}

size_t cce_loss_and_grad_workspace_bytes(int64_t N, int64_t D, int64_t V, size_t max_staging_bytes) {
  if (!sizes_ok(N, D, V)) return 0;
  return flce_layout(N, D, V, max_staging_bytes).total;
}

cce_status cce_loss_and_grad(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                             int64_t ignore_index, int reduction, float softcap, float filter_eps, int filter_flags,
                             size_t max_staging_bytes, float* loss, float* lse, void* dE, void* dC, void* workspace,
                             size_t ws_bytes, int32_t* dev_err, int64_t* dev_stats, void* stream) {
  if (!E || !C || !x || !loss || !dE || !dC || !workspace) return CCE_ERR_NULL;
  if (!sizes_ok(N, D, V)) return CCE_ERR_SHAPE;
  if (!aligned16(E) || !aligned16(C) || !aligned16(dE) || !aligned16(dC) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(x) & 7u) || (reinterpret_cast<uintptr_t>(loss) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(dev_stats) & 7u))
    return CCE_ERR_ALIGN;
  if (reduction != CCE_RED_SUM && reduction != CCE_RED_MEAN) return CCE_ERR_ARG;
  if (!(filter_eps >= 0.0f) || !std::isfinite(filter_eps)) return CCE_ERR_ARG;
  if (filter_flags & ~CCE_FILTER_BOTH) return CCE_ERR_ARG;
  if (!(softcap >= 0.0f) || !std::isfinite(softcap)) return CCE_ERR_ARG;
  const FlceLayout W = flce_layout(N, D, V, max_staging_bytes);
  if (ws_bytes < W.total) return CCE_ERR_WORKSPACE;
  int sms = 0, pair_clusters = 0;
  cce_status st = device_check(&sms, &pair_clusters);
  if (st != CCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* counters = reinterpret_cast<int*>(ws + W.counters);
  int* count = reinterpret_cast<int*>(ws + W.count);
  int* pos = reinterpret_cast<int*>(ws + W.pos);
  int* ridx = reinterpret_cast<int*>(ws + W.ridx);
  int64_t* xc = reinterpret_cast<int64_t*>(ws + W.xc);
  uint16_t* Ecmp = reinterpret_cast<uint16_t*>(ws + W.ec);
  float* lsec = reinterpret_cast<float*>(ws + W.lse);  // LSE of the compact rows
  double* blk_sum = reinterpret_cast<double*>(ws + W.blk_sum);
  int* blk_cnt = reinterpret_cast<int*>(ws + W.blk_cnt);
  uint16_t* stage = reinterpret_cast<uint16_t*>(ws + W.stage);
  float* mtile = reinterpret_cast<float*>(ws + W.mtile);
  uint8_t* bitmap = ws + W.bitmap;
  uint8_t* bitmapT = ws + W.bitmapT;
  float* deacc = reinterpret_cast<float*>(ws + W.deacc);
  float* dcacc = reinterpret_cast<float*>(ws + W.dcacc);
  const bool filter_de = (filter_flags & CCE_FILTER_DE) != 0, filter_dc = (filter_flags & CCE_FILTER_DC) != 0;
  const bool multi = W.nchunks > 1;
  {  // the rows that take part, compacted ("Cut Your Losses ...", Table A1: removing ignored tokens)
    PhaseScope ps(2, s);
    cudaError_t e = cudaMemsetAsync(counters, 0, sizeof(int) * CHUNK_COUNTERS * static_cast<size_t>(W.nchunks), s);
    if (e == cudaSuccess && dev_stats) e = cudaMemsetAsync(dev_stats, 0, 2 * sizeof(int64_t), s);
    if (e != cudaSuccess) return cuda_status(e);
    {
      cudaError_t ce = launch_compact(x, N, V, static_cast<long long>(ignore_index), pos, ridx, count,
                                      reinterpret_cast<int*>(ws + W.cscr), dev_err, s);
      g_launches += 3;
      if (ce != cudaSuccess) return cuda_status(ce);
    }
    const int rows_per_block = 8;
    const int blocks = static_cast<int>(std::min<int64_t>(int64_t(sms) * 16, cdiv(N, rows_per_block)));
    gather_rows_kernel<<<std::max(blocks, 1), 32 * rows_per_block, 0, s>>>(
        static_cast<const uint4*>(E), x, nullptr, nullptr, ridx, count, static_cast<int>(N), static_cast<int>(D),
        static_cast<long long>(ignore_index), reinterpret_cast<uint4*>(Ecmp), xc, nullptr, nullptr);
    g_launches++;
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }
  const bool b3d = D % 64 == 0;
  // The gradient GEMM as CTA pairs, as in the two-call backward (D tiles 256
  // wide, 3-D boxes; the dE K ranges start at multiples of 128).
  const int layout = g_grad_layout.load();
  const bool grad_pairs = pair_clusters > 0 && b3d && W.bn == BN && W.kps % 2 == 0 && layout != 2;
  if (grad_pairs) {
    cudaError_t e = cudaMemsetAsync(ws + W.zero, 0, ZERO_BOX_BYTES, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  // Chunks cover compact rows r0 .. r0 + Nc - 1; how many compact rows exist
  // is only known on the device, so every launch reads the count and a chunk
  // past it does nothing (its dC contribution is zero).
  for (int64_t c = 0; c < W.nchunks; ++c) {
    const int64_t r0 = c * W.Nc, rows = std::min(W.Nc, N - r0);
    const int64_t nb = cdiv(rows, BM);
    const uint16_t* Ec = Ecmp + r0 * D;
    // (1) logits of the chunk: fold + target capture + staging
    GemmArgs f;
    std::memset(&f, 0, sizeof(f));
    bool ok = make_tmap(&f.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ec, D, rows, D, BK, BM) &&
              make_tmap(&f.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, D, V, D, BK, BN) &&
              make_tmap(&f.tmOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, stage, W.Vp, rows, W.Vp, 64, 32);
    if (!ok) return CCE_ERR_CUDA;
    f.N = static_cast<int>(rows);
    f.D = static_cast<int>(D);
    f.V = static_cast<int>(V);
    f.n_blocks = static_cast<int>(nb);
    f.k_blocks = static_cast<int>(cdiv(D, BK));
    f.splits = W.S;
    f.v_tiles = static_cast<int>(cdiv(V, BN));
    f.group_n = raster_group(nb, D);
    f.items = f.n_blocks * f.splits;  // upper bound; the kernel uses the device count
    // As CTA pairs with 128-deep stages (with 64-deep ones the pairs had
    // measured slower here: Qwen 0.702 -> 0.738 ms, Llama 10.42 -> 10.47 ms)
    const bool fpairs = pair_clusters > 0 && D % 64 == 0;
    if (fpairs && !pair_operands(&f, Ec, rows, C, D, V)) return CCE_ERR_CUDA;
    f.n_dev = count;
    f.n_row0 = static_cast<int>(r0);
    f.x = xc + r0;
    f.ignore_index = ignore_index;
    f.part_m = reinterpret_cast<float*>(ws + W.part_m);
    f.part_s = reinterpret_cast<float*>(ws + W.part_s);
    f.tgt = reinterpret_cast<float*>(ws + W.tgt);
    f.mtile = mtile;
    f.softcap = softcap;
    f.inv_softcap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
    f.dev_err = dev_err;
    f.counter = counters + CHUNK_COUNTERS * c;
    cudaError_t e;
    {
      PhaseScope ps(0, s);
      e = fpairs ? launch_gemm_pairs(MODE_FWD_STAGE, f, std::min((f.n_blocks + 1) / 2 * f.splits, pair_clusters), s)
                 : launch_gemm(MODE_FWD_STAGE, f, std::min(f.items, sms), s);
      g_launches++;
      if (e != cudaSuccess) return cuda_status(e);
    }
    {  // (2) LSE of the chunk's rows and their block sums of the loss
      PhaseScope ps(1, s);
      combine_kernel<<<static_cast<unsigned>(cdiv(rows, COMBINE_THREADS)), COMBINE_THREADS, 0, s>>>(
          f.part_m, f.part_s, f.tgt, xc + r0, f.N, W.S, f.V, static_cast<long long>(ignore_index), reduction,
          lsec + r0, nullptr, blk_sum + r0 / COMBINE_THREADS, blk_cnt + r0 / COMBINE_THREADS, dev_err, count,
          static_cast<int>(r0));
      g_launches++;
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_status(e);
    }
    {  // (3) staged logits -> G-hat (bf16, in place) and the filter votes
      PhaseScope ps(7, s);
      int launched = 0;
      // the kept-tile count that picks the gradient GEMM's layout (filter on)
      int* kept = grad_pairs && (filter_de || filter_dc) && layout == 0 ? counters + CHUNK_COUNTERS * c + 2 : nullptr;
      e = launch_gpass(stage, W.Vp, mtile, rows, V, xc + r0, static_cast<long long>(ignore_index), lsec + r0, count,
                       reduction, softcap, filter_eps, !(filter_de && filter_dc), bitmap, bitmapT, W.bm_ld, count, r0,
                       kept, s, &launched);
      g_launches += static_cast<uint64_t>(launched);
      if (e != cudaSuccess) return cuda_status(e);
    }
    // (4) dE rows of the chunk (K = the whole vocabulary, in W.Sde ranges)
    //     and its contribution to dC (K = the chunk's rows)
    GemmArgs r;
    std::memset(&r, 0, sizeof(r));
    ok = make_tmap_mn3(&r.tmA, stage, W.Vp, rows, BM / 64) &&
         make_tmap(&r.tmA2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, stage, W.Vp, rows, W.Vp, 64, BM);
    if (b3d) {
      ok = ok && make_tmap_mn3(&r.tmB, Ec, D, rows) && make_tmap_mn3(&r.tmB2, C, D, V);
    } else {
      ok = ok && make_tmap(&r.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ec, D, rows, D, 64, 64) &&
           make_tmap(&r.tmB2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, D, V, D, 64, 64);
    }
    // dC: fp32 accumulator for all chunks but the last, which adds the
    // accumulator and writes bf16 (a single chunk writes bf16 directly)
    const bool last = c == W.nchunks - 1;
    if (!last) {
      ok = ok && make_tmap(&r.tmOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dcacc, D, V, D, 32, 32);
    } else {
      ok = ok && make_tmap(&r.tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dC, D, V, D, 32, 32,
                           CU_TENSOR_MAP_SWIZZLE_64B);
    }
    ok = ok && make_tmap(&r.tmOut2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, deacc, D,
                         static_cast<uint64_t>(W.Sde) * W.slab, D, 32, 32);
    GemmArgs one = r;  // the one-CTA-per-tile layout (see the two-call backward)
    if (grad_pairs) {  // every operand one 3-D box of two 64-column groups and 128 rows
      ok = ok && make_tmap_mn3(&r.tmA, stage, W.Vp, rows, 2, PAIR_BK) && make_tmap_mn3(&r.tmA2, stage, W.Vp, rows, 2, BM) &&
           make_tmap_mn3(&r.tmB, Ec, D, rows, 2, PAIR_BK) && make_tmap_mn3(&r.tmB2, C, D, V, 2, PAIR_BK) &&
           make_tmap(&r.tmZ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws + W.zero, 64, 2 * BM, 64, 64, 2 * BM);
      r.pair_words = g_pair_words.load();
    }
    if (!ok) return CCE_ERR_CUDA;
    r.N = static_cast<int>(rows);
    r.D = static_cast<int>(D);
    r.V = static_cast<int>(V);
    r.n_blocks = static_cast<int>(nb);
    r.n_dev = count;
    r.n_row0 = static_cast<int>(r0);
    r.x = xc + r0;
    r.ignore_index = ignore_index;
    r.filter_de = filter_de ? 1 : 0;
    r.filter_dc = filter_dc ? 1 : 0;
    r.bitmap = bitmap;
    r.bitmapT = bitmapT;
    r.bm_ld = static_cast<int>(W.bm_ld);
    r.dev_err = dev_err;
    r.chunk_v0 = 0;
    r.chunk_w = static_cast<int>(V);
    r.c_row0 = 0;
    r.b3d = b3d ? 1 : 0;
    r.bn = static_cast<int>(W.bn);
    r.n_tiles = static_cast<int>(W.n_tiles);
    r.dc_m_tiles = static_cast<int>(cdiv(V, BM));
    r.de_k_blocks = static_cast<int>(cdiv(V, BK));
    r.de_splits = W.Sde;
    r.de_kps = static_cast<int>(W.kps);
    r.de_slab = static_cast<int>(W.slab);
    r.de_row0 = static_cast<int>(r0);
    r.first_chunk = 1;  // every dE slab row is written once
    r.dc_f32 = last ? 0 : 1;
    r.dc_reduce = (!last && c > 0) ? 1 : 0;
    r.dc_acc = (last && multi) ? dcacc : nullptr;
    r.dc_first = 2 * nb >= W.kps ? 1 : 0;  // longest tiles first
    r.counter = counters + CHUNK_COUNTERS * c + 1;
    {
      PhaseScope ps(4, s);
      if (grad_pairs) {
        const bool dual = (filter_de || filter_dc) && layout == 0;
        const int64_t items = ((r.dc_m_tiles + 1) / 2 + (nb + 1) / 2 * W.Sde) * r.n_tiles;
        r.kept_tiles = dual ? counters + CHUNK_COUNTERS * c + 2 : nullptr;
        r.grad_path = dual ? 1 : -1;
        e = launch_gemm_pairs(MODE_GRAD, r, static_cast<int>(std::min<int64_t>(pair_clusters, items)), s);
        if (e == cudaSuccess && dual) {
          g_launches++;
          const GemmArgs pr = r;
          r.tmA = one.tmA;
          r.tmA2 = one.tmA2;
          r.tmB = one.tmB;
          r.tmB2 = one.tmB2;
          r.grad_path = 0;
          const int64_t tiles = (r.dc_m_tiles + nb * W.Sde) * r.n_tiles;
          e = launch_gemm(MODE_GRAD, r, static_cast<int>(std::min<int64_t>(sms, tiles)), s);
          r = pr;
        }
      } else {
        r.grad_path = -1;
        const int64_t items = (r.dc_m_tiles + nb * W.Sde) * r.n_tiles;
        e = launch_gemm(MODE_GRAD, r, static_cast<int>(std::min<int64_t>(sms, items)), s);
      }
      g_launches++;
      if (e != cudaSuccess) return cuda_status(e);
    }
    if (dev_stats) {
      int launched = 0;
      e = launch_stats_add(bitmap, count, r0, rows, cdiv(V, 128), W.bm_ld, dev_stats, s, &launched);
      g_launches += static_cast<uint64_t>(launched);
      if (e != cudaSuccess) return cuda_status(e);
    }
  }
  {
    PhaseScope ps(5, s);
    finish_loss_kernel<<<1, COMBINE_THREADS, 0, s>>>(blk_sum, blk_cnt, W.nblk, reduction, loss);
    g_launches++;
    if (lse) {  // back to the original rows; rows that took no part get 0
      scatter_rows_kernel<<<static_cast<unsigned>(std::min<int64_t>(int64_t(sms) * 8, cdiv(N, 256))), 256, 0, s>>>(
          lsec, nullptr, pos, static_cast<int>(N), lse, nullptr);
      g_launches++;
    }
    int launched = 0;
    cudaError_t e = launch_finalize_de_slabs(deacc, W.Sde, W.slab, N, D, pos, dE, s, sms, &launched);
    g_launches += static_cast<uint64_t>(launched);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }
  return CCE_OK;
}

cce_status cce_scale_grads(void* dE, int64_t nE, void* dC, int64_t nC, const float* grad_out, void* stream) {
  if (!dE || !dC || !grad_out) return CCE_ERR_NULL;
  if (nE < 0 || nC < 0 || nE % 8 || nC % 8) return CCE_ERR_SHAPE;
  if (!aligned16(dE) || !aligned16(dC) || (reinterpret_cast<uintptr_t>(grad_out) & 3u)) return CCE_ERR_ALIGN;
  int sms = 0;
  cce_status st = device_check(&sms);
  if (st != CCE_OK) return st;
  int launched = 0;
  cudaError_t e = launch_scale_bf16(dE, nE, dC, nC, grad_out, static_cast<cudaStream_t>(stream), sms, &launched);
  g_launches += static_cast<uint64_t>(launched);
  return cuda_status(e);
}

cce_status cce_selftest_wait_timeout(int32_t* dev_err, uint32_t timeout_us, void* stream) {
  if (!dev_err) return CCE_ERR_NULL;
  if (timeout_us == 0 || timeout_us > 10000000u) return CCE_ERR_ARG;
  int sms = 0;
  cce_status st = device_check(&sms);
  if (st != CCE_OK) return st;
  cudaError_t e = launch_selftest_wait_timeout(dev_err, static_cast<uint64_t>(timeout_us) * 1000u,
                                               static_cast<cudaStream_t>(stream));
  g_launches++;
  return cuda_status(e);
}

cce_status cce_selftest_pair_timeout(int32_t* dev_err, uint32_t timeout_us, int hold, void* stream) {
  if (!dev_err) return CCE_ERR_NULL;
  if (timeout_us == 0 || timeout_us > 10000000u || (hold != 0 && hold != 1)) return CCE_ERR_ARG;
  int sms = 0;
  cce_status st = device_check(&sms);
  if (st != CCE_OK) return st;
  cudaError_t e = launch_selftest_pair_timeout(dev_err, static_cast<uint64_t>(timeout_us) * 1000u, hold,
                                               static_cast<cudaStream_t>(stream));
  g_launches++;
  return cuda_status(e);
}

int cce_selftest_pair_map_words(int words) {
  if (words <= 0 || words > PAIR_MAP_WORDS) words = PAIR_MAP_WORDS;
  return g_pair_words.exchange(words);
}

int cce_selftest_grad_layout(int layout) {
  if (layout < 0 || layout > 2) layout = 0;
  return g_grad_layout.exchange(layout);
}

cce_status cce_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof = enable != 0;
  return CCE_OK;
}

cce_status cce_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& r : g_recs) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  for (int i = 0; i < CCE_NUM_PHASES; ++i) {
    g_ms[i] = 0.0;
    g_cnt[i] = 0;
  }
  return CCE_OK;
}

cce_status cce_profile_read(double* ms, int64_t* launches) {
  if (!ms || !launches) return CCE_ERR_NULL;
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return CCE_ERR_CUDA;
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return CCE_ERR_CUDA;
    g_ms[r.phase] += t;
    g_cnt[r.phase] += 1;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  for (int i = 0; i < CCE_NUM_PHASES; ++i) {
    ms[i] = g_ms[i];
    launches[i] = g_cnt[i];
  }
  return CCE_OK;
}

const char* cce_profile_phase_name(int phase) {
  static const char* names[CCE_NUM_PHASES] = {"fwd_lse_gemm",  "fwd_combine",  "bwd_prep",       "bwd_recompute_g",
                                               "bwd_grad_gemm", "bwd_finalize", "bwd_vocab_sort", "single_g_pass"};
  if (phase < 0 || phase >= CCE_NUM_PHASES) return "";
  return names[phase];
}

}  // extern "C"
