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

// Per-block digit counts: a block holds at most SORT_TILE = 1024 keys, so a
// count fits 16 bits; a row of 256 counts is 128 words, word w holding digit
// 2w in its low half and 2w + 1 in its high half (block-major: row b of a
// pass at hist + 128 b).  One 16-byte load brings a lane eight counts.
constexpr int HIST_WORDS = 128;

// Radix sort, launch 1: each block takes SORT_TILE keys, writes their
// ascending bits and the identity order, and counts the keys' lowest digits
// into its row of the first pass's counts.  It also zeroes its rows of the
// later passes' counts, which the passes before them fill with atomics.
__global__ void radix_init_kernel(const float* __restrict__ keys, int n, uint32_t* __restrict__ hist, int nblocks,
                                  uint32_t* __restrict__ bits, int* __restrict__ vals) {
  __shared__ int h[256];
  const int t = threadIdx.x;
  h[t] = 0;  // SORT_THREADS == 256 digits
  __syncthreads();
  const int base = blockIdx.x * SORT_TILE;
  for (int i = t; i < SORT_TILE; i += SORT_THREADS) {
    const int k = base + i;
    if (k < n) {
      const uint32_t u = ascending_bits(keys[k]);
      bits[k] = u;
      vals[k] = k;
      atomicAdd(&h[u & 0xFF], 1);  // a count: order does not matter
    }
  }
  __syncthreads();
  if (t < HIST_WORDS) {
    const size_t w = static_cast<size_t>(blockIdx.x) * HIST_WORDS + t;
    const size_t pass_stride = static_cast<size_t>(nblocks) * HIST_WORDS;
    hist[w] = static_cast<uint32_t>(h[2 * t]) | (static_cast<uint32_t>(h[2 * t + 1]) << 16);
    for (int p = 1; p < 4; ++p) hist[p * pass_stride + w] = 0u;
  }
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

// One stable radix pass on digit (key >> shift) & 0xFF, in one launch.
//  1. Offsets: from the pass's per-block digit counts, every block sums each
//     digit over all blocks (its total) and over the blocks before it; digit
//     d starts at the totals of the smaller digits.  Warp w reads the count
//     rows w, w + 8, ..., each row 512 coalesced bytes, eight digits a lane.
//     The block's keys and values are loaded first, so their latency
//     overlaps these reads.  A pass thus reads nblocks^2 x 512 bytes, about
//     V^2 / 2048, of counts from L2 (11 MB at V = 151,936, 32 MB at
//     256,000): quadratic in V, and less than one pass over C (2 V D bytes)
//     while V < 4096 D (3.7 M at D = 896).
//  2. Scatter: the block walks its keys in order, 256 per round; a key's
//     output position is its digit's start + the keys with that digit in
//     earlier blocks, earlier rounds, earlier warps of this round and earlier
//     lanes of its warp.
//  3. The next pass's counts (hist_next, unless this is the last pass): each
//     key adds one to the count of its next digit in the block that its
//     output position falls in; lanes with the same target add once,
//     together.  The counts are integers, so the order of the atomics does
//     not matter.
// The last pass may also write inv[value] = position (the inverse order).
__global__ void radix_pass_kernel(const uint32_t* __restrict__ keys, const int* __restrict__ vals, int n, int shift,
                                  int nblocks, const uint32_t* __restrict__ hist, uint32_t* __restrict__ hist_next,
                                  uint32_t* __restrict__ keys_out, int* __restrict__ vals_out, int* __restrict__ inv) {
  __shared__ int part_tot[SORT_WARPS][256];
  __shared__ int part_bef[SORT_WARPS][256];
  __shared__ int running[256];
  __shared__ int wcount[SORT_WARPS][256];
  __shared__ int warp_sums[SORT_WARPS];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int blk = static_cast<int>(blockIdx.x);
  const int base = blk * SORT_TILE;
  uint32_t kr[SORT_ROUNDS];
  int vr[SORT_ROUNDS];
#pragma unroll
  for (int r = 0; r < SORT_ROUNDS; ++r) {
    const int k = base + r * SORT_THREADS + t;
    kr[r] = k < n ? keys[k] : 0u;
    vr[r] = k < n ? vals[k] : 0;
  }
  {
    int tot[8], bef[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) tot[j] = bef[j] = 0;
#pragma unroll 8
    for (int b = warp; b < nblocks; b += SORT_WARPS) {
      // written by atomics in the previous launch: read from L2
      const uint4 q = __ldcg(reinterpret_cast<const uint4*>(hist + static_cast<size_t>(b) * HIST_WORDS) + lane);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
      const bool earlier = b < blk;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int lo = static_cast<int>(w[i] & 0xFFFFu), hi = static_cast<int>(w[i] >> 16);
        tot[2 * i] += lo;
        tot[2 * i + 1] += hi;
        bef[2 * i] += earlier ? lo : 0;
        bef[2 * i + 1] += earlier ? hi : 0;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // lane's digits: 8 lane .. 8 lane + 7
      part_tot[warp][8 * lane + j] = tot[j];
      part_bef[warp][8 * lane + j] = bef[j];
    }
  }
  __syncthreads();
  {
    int total = 0, before = 0;
#pragma unroll
    for (int w = 0; w < SORT_WARPS; ++w) {
      total += part_tot[w][t];
      before += part_bef[w][t];
    }
    int all;
    const int digit_base = block_exclusive_scan(total, warp_sums, &all);  // SORT_THREADS == 256 digits
    running[t] = digit_base + before;
  }
  const int shift_next = shift + 8;
#pragma unroll
  for (int round = 0; round < SORT_ROUNDS; ++round) {
    for (int i = t; i < SORT_WARPS * 256; i += SORT_THREADS) (&wcount[0][0])[i] = 0;
    __syncthreads();
    const int k = base + round * SORT_THREADS + t;
    const bool live = k < n;
    const uint32_t key = kr[round];
    const int digit = live ? static_cast<int>((key >> shift) & 0xFF) : 256 + lane;  // dead lanes match nothing
    const unsigned peers = __match_any_sync(0xffffffffu, digit);
    const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
    if (live && rank_in_warp == 0) wcount[warp][digit] = __popc(peers);
    __syncthreads();
    int pos = 0;
    if (live) {
      pos = running[digit] + rank_in_warp;
      for (int w = 0; w < warp; ++w) pos += wcount[w][digit];
      const int v = vr[round];
      keys_out[pos] = key;
      vals_out[pos] = v;
      if (inv) inv[v] = pos;
    }
    if (hist_next) {
      const int slot = live ? (pos / SORT_TILE) * 256 + static_cast<int>((key >> shift_next) & 0xFF) : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, slot);
      if (live && (same & ((1u << lane) - 1u)) == 0u)  // digit 2w + h: half h of word w
        atomicAdd(hist_next + (slot >> 1), static_cast<uint32_t>(__popc(same)) << (16 * (slot & 1)));
    }
    __syncthreads();
    for (int d = t; d < 256; d += SORT_THREADS) {
      int c = 0;
      for (int w = 0; w < SORT_WARPS; ++w) c += wcount[w][d];
      running[d] += c;
    }
    __syncthreads();
  }
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
  return 3 * align256(static_cast<size_t>(V) * 4) + align256(static_cast<size_t>(4) * HIST_WORDS * nblocks * 4);
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

cudaError_t launch_vocab_order(const float* keys, int64_t V, int* perm, void* scratch, cudaStream_t s,
                               int* launches, int* inv) {
  const int n = static_cast<int>(V);
  const int nblocks = static_cast<int>(cdiv64(V, SORT_TILE));
  uint8_t* p = static_cast<uint8_t*>(scratch);
  const size_t vb = align256(static_cast<size_t>(V) * 4);
  uint32_t* keys_a = reinterpret_cast<uint32_t*>(p);
  uint32_t* keys_b = reinterpret_cast<uint32_t*>(p + vb);
  int* vals_b = reinterpret_cast<int*>(p + 2 * vb);
  uint32_t* hist = reinterpret_cast<uint32_t*>(p + 3 * vb);  // [4 passes][nblocks][HIST_WORDS]
  const size_t pass_stride = static_cast<size_t>(nblocks) * HIST_WORDS;
  radix_init_kernel<<<nblocks, SORT_THREADS, 0, s>>>(keys, n, hist, nblocks, keys_a, perm);
  ++*launches;
  // four stable 8-bit passes, ping-ponging between (keys_a, perm) and
  // (keys_b, vals_b); after the fourth the result is back in (keys_a, perm)
  uint32_t* kin = keys_a;
  int* vin = perm;
  uint32_t* kout = keys_b;
  int* vout = vals_b;
  for (int pass = 0; pass < 4; ++pass) {
    uint32_t* next = pass < 3 ? hist + (pass + 1) * pass_stride : nullptr;
    radix_pass_kernel<<<nblocks, SORT_THREADS, 0, s>>>(kin, vin, n, 8 * pass, nblocks, hist + pass * pass_stride, next,
                                                        kout, vout, pass == 3 ? inv : nullptr);
    ++*launches;
    std::swap(kin, kout);
    std::swap(vin, vout);
  }
  return cudaGetLastError();
}

cudaError_t launch_remap_targets(const int* inv, int64_t* xc, const int* n_dev, int64_t N, cudaStream_t s, int sms,
                                 int* launches) {
  remap_targets_kernel<<<grid_for(N, 256, sms * 4), 256, 0, s>>>(xc, n_dev, static_cast<int>(N), inv);
  *launches += 1;
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
