// Tile geometry and kernel arguments of the tcgen05 GEMM (shared by host and device code).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace cce {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;                  // 16 KiB
constexpr int B_STAGE_BYTES = BN * BK * 2;                  // 32 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;  // 48 KiB
constexpr int NUM_EPI_WARPS = 4;
constexpr int EPI_WARP_BYTES = 8192;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_EPI_WARPS * EPI_WARP_BYTES + BAR_BYTES;
constexpr int FILTER_TILE = 128;  // filter decisions are per 128 tokens x 128 vocab

constexpr float LOG2E = 1.4426950408889634f;
constexpr float NEG_BIG = -3.0e38f;  // finite "minus infinity" for the running max

enum Mode { MODE_FWD = 0, MODE_BWD_G = 1, MODE_DC = 2, MODE_DE = 3 };

struct GemmArgs {
  CUtensorMap tmA;    // loads of operand A
  CUtensorMap tmB;    // loads of operand B
  CUtensorMap tmOut;  // BWD_G: G chunk; DC: dC; DE: dE accumulator
  int N, D, V;
  int n_blocks;  // ceil(N / 128)
  int k_blocks;  // BK steps along the contraction
  int splits;    // FWD: vocabulary splits
  int v_tiles;   // FWD: ceil(V / 256); BWD_G: 256-wide tiles in the chunk
  int chunk_v0;  // BWD: first vocabulary row of the chunk (multiple of 256)
  int chunk_w;   // BWD: vocabulary rows in the chunk
  int m_tiles, n_tiles;  // DC / DE output tile grid
  int first_chunk;       // DE: store (1) or reduce-add (0)
  const int64_t* x;
  long long ignore_index;
  float* part_m;  // FWD: [splits][N] running max (log2 units)
  float* part_s;  // FWD: [splits][N] running sum of 2^(y - max)
  float* tgt;     // FWD: [N] target logit
  const float* lse;
  const float* grad_out;
  const int* count;
  int reduction;
  float eps;
  uint8_t* bitmap;   // [ceil(N/128)][bm_ld] tile survival, token-block major
  uint8_t* bitmapT;  // [bm_ld][ceil(N/128)] the same, vocabulary-block major (read along K by dC)
  int bm_ld;         // ceil(V / 128)
  int group_n;       // BWD_G: token blocks per raster group
  int32_t* dev_err;
};

}  // namespace cce
