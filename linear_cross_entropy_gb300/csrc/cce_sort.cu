// Vocabulary sorting by average logit ("Cut Your Losses in Large-Vocabulary
// Language Models", section "Vocabulary Sorting"): the backward can walk the
// vocabulary in order of average logit, so the tokens that carry softmax
// mass share few tiles and the filter skips the rest.
//
// The pages accumulate each token's logit sum in the forward pass.  Here the
// sum follows from linearity: sum_n C_v . E_n = C_v . (sum_n E_n), so the key
// of token v is C_v . e_sum, where e_sum is the column sum of the rows taking
// part -- one reduction over E and one matrix-vector product over C, both in
// a fixed order, so the keys are deterministic.  The order is a stable LSD
// radix sort of the keys (ascending; equal keys keep token order).
//
// Also here: the row gather the backward uses to bring a chunk of C into
// sorted order (the dC tiles write their token rows directly).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"

namespace cce {
namespace {

constexpr int SORT_THREADS = 256;                      // threads per block of a radix pass
constexpr int SORT_ROUNDS = 4;                         // keys per thread (one per round)
constexpr int SORT_TILE = SORT_THREADS * SORT_ROUNDS;  // keys per block
constexpr int SORT_WARPS = SORT_THREADS / 32;
static_assert(SORT_THREADS == 256, "one thread per 8-bit digit in the scatter set-up");
constexpr int COLSUM_THREADS = 256;                    // each thread sums two columns
constexpr int MAX_COLSUM_PARTS = 256;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rows per partial column sum: at least 32, at most MAX_COLSUM_PARTS parts.
int64_t colsum_rows(int64_t N) { return std::max<int64_t>(32, cdiv64(N, MAX_COLSUM_PARTS)); }

// Partial column sums over the rows that take part.  Block (bx, by) sums rows
// [by * rows, (by + 1) * rows) of columns 2 * (bx * 256 + threadIdx.x) + {0, 1}.
// A row takes part when it lies below *n_dev (all N rows when n_dev is null)
// and, when x is given, its target is in [0, V) and is not ignore_index.
__global__ void colsum_partial_kernel(const uint32_t* __restrict__ E, int N, const int* __restrict__ n_dev,
                                      const int64_t* __restrict__ x, int V, long long ignore_index, int D,
                                      int rows, float2* __restrict__ part) {
  const int c2 = blockIdx.x * blockDim.x + threadIdx.x;  // column pair
  if (2 * c2 >= D) return;
  const int n = n_dev ? min(N, *n_dev) : N;
  const int r0 = blockIdx.y * rows, r1 = min(n, r0 + rows);
  const int pitch = D / 2;
  float s0 = 0.0f, s1 = 0.0f;
  for (int r = r0; r < r1; ++r) {
    if (x) {
      const long long t = static_cast<long long>(x[r]);
      if (t == ignore_index || t < 0 || t >= V) continue;
    }
    const uint32_t v = E[static_cast<size_t>(r) * pitch + c2];
    s0 += __uint_as_float(v << 16);
    s1 += __uint_as_float(v & 0xFFFF0000u);
  }
  part[static_cast<size_t>(blockIdx.y) * pitch + c2] = make_float2(s0, s1);
}

// e_sum from the partials: block b covers column pairs 32b .. 32b + 31 (one
// per lane); warp w sums parts w, w + 8, w + 16, ... in that order, then warp
// 0 adds the eight warp sums in warp order.
__global__ void colsum_final_kernel(const float2* __restrict__ part, int nparts, int D, float2* __restrict__ esum) {
  __shared__ float2 ws[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pitch = D / 2;
  const int c2 = blockIdx.x * 32 + lane;
  float s0 = 0.0f, s1 = 0.0f;
  if (c2 < pitch) {
    for (int p = warp; p < nparts; p += 8) {
      const float2 v = part[static_cast<size_t>(p) * pitch + c2];
      s0 += v.x;
      s1 += v.y;
    }
  }
  ws[warp][lane] = make_float2(s0, s1);
  __syncthreads();
  if (warp == 0 && c2 < pitch) {
    float t0 = 0.0f, t1 = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      t0 += ws[w][lane].x;
      t1 += ws[w][lane].y;
    }
    esum[c2] = make_float2(t0, t1);
  }
}

// keys[v] = C_v . e_sum: one warp per vocabulary row, 16-byte loads, four in
// flight per lane; each lane sums its 8-column chunks c = lane, lane + 32, ...
// in increasing c, then a fixed butterfly adds the lanes.
__global__ void vocab_key_kernel(const uint4* __restrict__ C, const float* __restrict__ esum, int V, int D,
                                 float* __restrict__ keys) {
  const int warps = blockDim.x / 32;
  const int lane = threadIdx.x & 31;
  const int per_row = D / 8;
  for (int v = blockIdx.x * warps + (threadIdx.x >> 5); v < V; v += gridDim.x * warps) {
    const uint4* row = C + static_cast<size_t>(v) * per_row;
    float s = 0.0f;
    for (int c0 = lane; c0 < per_row; c0 += 128) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = (c0 + 32 * u < per_row) ? row[c0 + 32 * u] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
        if (c >= per_row) break;
        const float4 e0 = *reinterpret_cast<const float4*>(esum + 8 * c);
        const float4 e1 = *reinterpret_cast<const float4*>(esum + 8 * c + 4);
        s = fmaf(__uint_as_float(q[u].x << 16), e0.x, s);
        s = fmaf(__uint_as_float(q[u].x & 0xFFFF0000u), e0.y, s);
        s = fmaf(__uint_as_float(q[u].y << 16), e0.z, s);
        s = fmaf(__uint_as_float(q[u].y & 0xFFFF0000u), e0.w, s);
        s = fmaf(__uint_as_float(q[u].z << 16), e1.x, s);
        s = fmaf(__uint_as_float(q[u].z & 0xFFFF0000u), e1.y, s);
        s = fmaf(__uint_as_float(q[u].w << 16), e1.z, s);
        s = fmaf(__uint_as_float(q[u].w & 0xFFFF0000u), e1.w, s);
      }
    }
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) keys[v] = s;
  }
}

// Order-preserving map of a float to an unsigned integer: an ascending
// unsigned sort of the result is an ascending sort of the floats, with -0.0
// and +0.0 mapped alike (they compare equal).
__device__ __forceinline__ uint32_t ascending_bits(float k) {
  uint32_t u = __float_as_uint(k);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void order_init_kernel(const float* __restrict__ keys, int V, uint32_t* __restrict__ bits,
                                  int* __restrict__ vals) {
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
    bits[v] = ascending_bits(keys[v]);
    vals[v] = v;
  }
}

// Radix pass, step 1: per-block digit counts, stored digit-major
// (hist[digit * nblocks + block]) so that scanning a row gives every block's
// offset within that digit.
__global__ void radix_hist_kernel(const uint32_t* __restrict__ keys, int n, int shift, int nblocks,
                                  int* __restrict__ hist) {
  __shared__ int h[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * SORT_TILE;
  for (int i = threadIdx.x; i < SORT_TILE; i += blockDim.x) {
    const int k = base + i;
    if (k < n) atomicAdd(&h[(keys[k] >> shift) & 0xFF], 1);  // a count: order does not matter
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i * nblocks + blockIdx.x] = h[i];
}

// Exclusive scan of one value per thread over a block of SORT_THREADS
// threads (warp shuffles, then the warp totals); *total gets the sum.
// `warp_sums` holds SORT_WARPS ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += u;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < SORT_WARPS; ++w) {
    const int ws = warp_sums[w];
    before += w < warp ? ws : 0;
    all += ws;
  }
  __syncthreads();  // warp_sums may be reused by the caller's next scan
  *total = all;
  return before + inc - v;
}

// Radix pass, step 2: block d turns row d of the counts (one count per
// sort block) into exclusive offsets within digit d, and writes the row's
// total to totals[d].
__global__ void radix_scan_kernel(int* __restrict__ hist, int nblocks, int* __restrict__ totals) {
  __shared__ int warp_sums[SORT_WARPS];
  int* row = hist + static_cast<size_t>(blockIdx.x) * nblocks;
  int carry = 0;
  for (int base = 0; base < nblocks; base += SORT_THREADS) {
    const int i = base + static_cast<int>(threadIdx.x);
    const int v = i < nblocks ? row[i] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_sums, &tot);
    if (i < nblocks) row[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) totals[blockIdx.x] = carry;
}

// Radix pass, step 3: stable scatter.  A block walks its keys in order, 256
// per round; a key's output position is the first position of its digit
// (keys of smaller digits) + its block's offset within the digit + keys with
// that digit in earlier rounds + in earlier warps of this round + in earlier
// lanes of its warp.
__global__ void radix_scatter_kernel(const uint32_t* __restrict__ keys, const int* __restrict__ vals, int n,
                                     int shift, int nblocks, const int* __restrict__ offsets,
                                     const int* __restrict__ totals, uint32_t* __restrict__ keys_out,
                                     int* __restrict__ vals_out) {
  __shared__ int running[256];
  __shared__ int wcount[SORT_WARPS][256];
  __shared__ int warp_sums[SORT_WARPS];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  {
    int tot;
    const int digit_base = block_exclusive_scan(totals[t], warp_sums, &tot);  // SORT_THREADS == 256 digits
    running[t] = digit_base + offsets[static_cast<size_t>(t) * nblocks + blockIdx.x];
  }
  const int base = blockIdx.x * SORT_TILE;
  for (int round = 0; round < SORT_ROUNDS; ++round) {
    for (int i = t; i < SORT_WARPS * 256; i += blockDim.x) (&wcount[0][0])[i] = 0;
    __syncthreads();
    const int k = base + round * SORT_THREADS + t;
    const bool live = k < n;
    const uint32_t key = live ? keys[k] : 0u;
    const int digit = live ? static_cast<int>((key >> shift) & 0xFF) : 256 + lane;  // dead lanes match nothing
    const unsigned peers = __match_any_sync(0xffffffffu, digit);
    const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
    if (live && rank_in_warp == 0) wcount[warp][digit] = __popc(peers);
    __syncthreads();
    if (live) {
      int pos = running[digit] + rank_in_warp;
      for (int w = 0; w < warp; ++w) pos += wcount[w][digit];
      keys_out[pos] = key;
      vals_out[pos] = vals[k];
    }
    __syncthreads();
    for (int d = t; d < 256; d += blockDim.x) {
      int c = 0;
      for (int w = 0; w < SORT_WARPS; ++w) c += wcount[w][d];
      running[d] += c;
    }
    __syncthreads();
  }
}

// inv[perm[j]] = j
__global__ void invert_kernel(const int* __restrict__ perm, int V, int* __restrict__ inv) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < V; j += gridDim.x * blockDim.x) inv[perm[j]] = j;
}

// Compact targets -> sorted positions for the n rows that take part; the
// zero rows that pad the last 128-row block get -1 (outside [0, V)).
__global__ void remap_targets_kernel(int64_t* __restrict__ xc, const int* __restrict__ n_dev, int N,
                                     const int* __restrict__ inv) {
  const int n = min(N, *n_dev);
  const int nz = min(N, (n + 127) / 128 * 128);
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < nz; k += gridDim.x * blockDim.x)
    xc[k] = k < n ? static_cast<int64_t>(inv[static_cast<int>(xc[k])]) : int64_t(-1);
}

// dst[j] = src[rows[j]] for j < count; dst[j] = 0 for count <= j < total.
// One warp per row, 16-byte copies.
__global__ void gather_vocab_rows_kernel(const uint4* __restrict__ src, const int* __restrict__ rows, int count,
                                         int total, int D, uint4* __restrict__ dst) {
  const int per_row = D / 8;
  const int lane = threadIdx.x & 31;
  for (int j = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); j < total; j += gridDim.x * (blockDim.x / 32)) {
    uint4* d = dst + static_cast<size_t>(j) * per_row;
    if (j < count) {
      const uint4* s = src + static_cast<size_t>(rows[j]) * per_row;
#pragma unroll 4
      for (int c = lane; c < per_row; c += 32) d[c] = s[c];  // several 16-byte loads in flight per lane
    } else {
      for (int c = lane; c < per_row; c += 32) d[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

int grid_for(int64_t work, int per_block, int cap) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cap, cdiv64(work, per_block))));
}

}  // namespace

size_t vocab_keys_scratch_bytes(int64_t N, int64_t D) {
  const int64_t nparts = cdiv64(N, colsum_rows(N));
  return align256(static_cast<size_t>(nparts) * D * 4) + align256(static_cast<size_t>(D) * 4);
}

size_t vocab_order_scratch_bytes(int64_t V) {
  const int64_t nblocks = cdiv64(V, SORT_TILE);
  return 3 * align256(static_cast<size_t>(V) * 4) + align256(static_cast<size_t>(256) * nblocks * 4) +
         align256(256 * 4);
}

cudaError_t launch_vocab_keys(const void* E, int64_t N, const int* n_dev, const int64_t* x, long long ignore_index,
                              int64_t D, const void* C, int64_t V, float* keys, void* scratch, cudaStream_t s,
                              int sms, int* launches) {
  const int64_t rows = colsum_rows(N);
  const int nparts = static_cast<int>(cdiv64(N, rows));
  uint8_t* p = static_cast<uint8_t*>(scratch);
  float2* part = reinterpret_cast<float2*>(p);
  float* esum = reinterpret_cast<float*>(p + align256(static_cast<size_t>(nparts) * D * 4));
  const int pairs = static_cast<int>(D / 2);
  const dim3 grid(static_cast<unsigned>(cdiv64(pairs, COLSUM_THREADS)), static_cast<unsigned>(nparts));
  colsum_partial_kernel<<<grid, COLSUM_THREADS, 0, s>>>(static_cast<const uint32_t*>(E), static_cast<int>(N), n_dev,
                                                        x, static_cast<int>(V), ignore_index, static_cast<int>(D),
                                                        static_cast<int>(rows), part);
  colsum_final_kernel<<<static_cast<unsigned>(cdiv64(pairs, 32)), 256, 0, s>>>(
      part, nparts, static_cast<int>(D), reinterpret_cast<float2*>(esum));
  vocab_key_kernel<<<grid_for(V, 8, sms * 16), 256, 0, s>>>(static_cast<const uint4*>(C), esum, static_cast<int>(V),
                                                            static_cast<int>(D), keys);
  *launches += 3;
  return cudaGetLastError();
}

cudaError_t launch_vocab_order(const float* keys, int64_t V, int* perm, void* scratch, cudaStream_t s, int sms,
                               int* launches) {
  const int n = static_cast<int>(V);
  const int nblocks = static_cast<int>(cdiv64(V, SORT_TILE));
  uint8_t* p = static_cast<uint8_t*>(scratch);
  const size_t vb = align256(static_cast<size_t>(V) * 4);
  uint32_t* keys_a = reinterpret_cast<uint32_t*>(p);
  uint32_t* keys_b = reinterpret_cast<uint32_t*>(p + vb);
  int* vals_b = reinterpret_cast<int*>(p + 2 * vb);
  int* hist = reinterpret_cast<int*>(p + 3 * vb);
  int* totals = reinterpret_cast<int*>(p + 3 * vb + align256(static_cast<size_t>(256) * nblocks * 4));
  order_init_kernel<<<grid_for(V, 256, sms * 4), 256, 0, s>>>(keys, n, keys_a, perm);
  ++*launches;
  // four stable 8-bit passes, ping-ponging between (keys_a, perm) and
  // (keys_b, vals_b); after the fourth the result is back in (keys_a, perm)
  uint32_t* kin = keys_a;
  int* vin = perm;
  uint32_t* kout = keys_b;
  int* vout = vals_b;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    radix_hist_kernel<<<nblocks, SORT_THREADS, 0, s>>>(kin, n, shift, nblocks, hist);
    radix_scan_kernel<<<256, SORT_THREADS, 0, s>>>(hist, nblocks, totals);
    radix_scatter_kernel<<<nblocks, SORT_THREADS, 0, s>>>(kin, vin, n, shift, nblocks, hist, totals, kout, vout);
    *launches += 3;
    std::swap(kin, kout);
    std::swap(vin, vout);
  }
  return cudaGetLastError();
}

cudaError_t launch_remap_targets(const int* perm, int64_t V, int* inv, int64_t* xc, const int* n_dev, int64_t N,
                                 cudaStream_t s, int sms, int* launches) {
  invert_kernel<<<grid_for(V, 256, sms * 4), 256, 0, s>>>(perm, static_cast<int>(V), inv);
  remap_targets_kernel<<<grid_for(N, 256, sms * 4), 256, 0, s>>>(xc, n_dev, static_cast<int>(N), inv);
  *launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_gather_vocab_rows(const void* src, const int* rows, int64_t count, int64_t total, int64_t D,
                                     void* dst, cudaStream_t s, int sms, int* launches) {
  gather_vocab_rows_kernel<<<grid_for(total, 8, sms * 8), 256, 0, s>>>(
      static_cast<const uint4*>(src), rows, static_cast<int>(count), static_cast<int>(total), static_cast<int>(D),
      static_cast<uint4*>(dst));
  ++*launches;
  return cudaGetLastError();
}

}  // namespace cce
