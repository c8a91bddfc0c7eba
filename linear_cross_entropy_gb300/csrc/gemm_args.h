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
// warps: 0 producer, 1 MMA, 2-5 epilogue, 6 scheduler (gradient-GEMM pairs;
// idle otherwise)
constexpr int NUM_THREADS = 96 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
// CTA pairs: TMEM columns allocated (together, by both CTAs) and accumulators
constexpr uint32_t PAIR_TMEM_COLS = 512;
constexpr int PAIR_ACCS = 2;
constexpr int PAIR_MIN_BLOCKS = 64;  // recompute as CTA pairs from this many 128-row token blocks
constexpr int RING = 4;  // depth of the work-item ring between the scheduler and the consumers
// gradient-GEMM pairs: survival words of an item (64 filter columns, one
// 128-deep K-block each) in WORD_SLOTS slots: K ranges up to 2560 K-blocks
// (327,680 tokens or vocabulary entries) take the scheduler's words
constexpr int PAIR_MAP_WORDS = 40;
constexpr int WORD_SLOTS = 2;
// barriers, flags, ring ids, stage tags and the pairs' survival words
constexpr int BAR_BYTES = 1792;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_EPI_WARPS * EPI_WARP_BYTES + BAR_BYTES;
constexpr int FILTER_TILE = 128;  // filter decisions are per 128 tokens x 128 vocab
constexpr int KEPT_SLOTS = 32;    // kept-tile counters per chunk (spread to keep the atomics apart)

constexpr float LOG2E = 1.4426950408889634f;
constexpr float NEG_BIG = -3.0e38f;  // finite "minus infinity" for the running max

// MODE_GRAD runs the two gradient contractions of one vocabulary chunk in
// one launch; each of its tiles is of kind KIND_DC or KIND_DE.  MODE_FWD_STAGE
// is MODE_FWD that also stages its logits for the single call (see mtile).
enum Mode { MODE_FWD = 0, MODE_BWD_G = 1, MODE_GRAD = 2, MODE_FWD_STAGE = 3 };
enum Kind { KIND_MAIN = 0, KIND_DC = 1, KIND_DE = 2 };

// Pipeline depth and stage size of one CTA.  CTA pairs run stages two
// K-blocks deep (K = 128): a CTA's stage is its 128 A rows and half (128
// rows or columns) of B, 64 KiB, three of them in the stage memory.  The
// producer then issues one stage per 128 of K, half as often as with 64-deep
// stages; in the gradient GEMM the producer's work per stage is what paces
// the pair.
constexpr int PAIR_BK = 128;
constexpr int PAIR_A_BYTES = BM * PAIR_BK * 2;                        // 32 KiB
constexpr int PAIR_STAGE_BYTES = 2 * PAIR_A_BYTES;                    // + half of B: 64 KiB
constexpr int PAIR_STAGES = STAGES * STAGE_BYTES / PAIR_STAGE_BYTES;  // 3
constexpr int MAX_STAGES = PAIR_STAGES > STAGES ? PAIR_STAGES : STAGES;
template <int MODE, bool PAIR>
struct Pipe {
  static constexpr int kStages = PAIR ? PAIR_STAGES : STAGES;
  static constexpr int kStageBytes = PAIR ? PAIR_STAGE_BYTES : STAGE_BYTES;
  static constexpr int kABytes = PAIR ? PAIR_A_BYTES : A_STAGE_BYTES;
  static constexpr int kBK = PAIR ? PAIR_BK : BK;
};

struct GemmArgs {
  // FWD / BWD_G: A = E, B = C, Out = G chunk (BWD_G).  GRAD: the dC kind's
  // A = G chunk (MN-major boxes), B = E (MN-major boxes), Out = dC.
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmOut;
  // GRAD: the dE kind's A = G chunk (K-major boxes), B = C (MN-major: 3-D view
  // {64 d, V, D/64} or 64x64 boxes), Out = dE accumulator (fp32).  FWD run as
  // CTA pairs: tmB2 = C in boxes of 64 x 128 rows (each CTA's half of a B tile).
  CUtensorMap tmA2;
  CUtensorMap tmB2;
  CUtensorMap tmOut2;
  // GRAD as CTA pairs: one A-sized box (32 KiB) of zeros, loaded in place of
  // a CTA's A operand for a K-block its own tile skips but the other CTA's
  // tile keeps (the pair's MMA walks the union of the two tiles' K-blocks)
  CUtensorMap tmZ;
  int N, D, V;
  int n_blocks;  // ceil(N / 128)
  int k_blocks;  // FWD / BWD_G: ceil(D / 64)
  int splits;    // FWD: vocabulary splits
  int v_tiles;   // FWD: ceil(V / 256); BWD_G: 256-wide tiles in the chunk
  int chunk_v0;  // BWD: first vocabulary row of the chunk (multiple of 256)
  int chunk_w;   // BWD: vocabulary rows in the chunk
  int c_row0;    // BWD: row of the chunk's first vocabulary entry in the C / dC tensor maps
                 // (chunk_v0, or 0 when the chunk was gathered into sorted order)
  // GRAD, sorted vocabulary: dc_rows[j] = the token of the chunk's row j; the
  // dC tiles then write dC_out [V, D] bf16 rows directly (null: TMA stores)
  const int* dc_rows;
  uint16_t* dC_out;
  int group_n;   // FWD, FWD_STAGE, BWD_G: token blocks per raster group (>= 1)
  // GRAD
  int bn;           // width of a D tile (multiple of 32, <= 256; of 64 when b3d)
  int b3d;          // 1: the MN-major B operands come in one 3-D box per stage (D % 64 == 0)
  int n_tiles;      // ceil(D / bn)
  int dc_m_tiles;   // ceil(chunk_w / 128)
  int dc_k_blocks;  // ceil(N / 64)
  int de_k_blocks;  // ceil(chunk_w / 64)
  int dc_first;     // 1: dC tiles are handed out first (they have the longer K)
  int pair_words;   // GRAD pairs: survival words a work item may carry (1 .. PAIR_MAP_WORDS)
  // BWD_G: counts the chunk's kept 128 x 128 filter tiles into
  // kept_tiles[0 .. KEPT_SLOTS) (any slot; the sum is the count).  GRAD with
  // the filter on is launched twice, as CTA pairs (grad_path = 1) and one CTA
  // per tile (grad_path = 0); from the count each launch sees whether it is
  // the one that runs (grad_path = -1: always runs).
  int* kept_tiles;
  int grad_path;
  int first_chunk;  // dE: store (1) or reduce-add (0)
  // dynamic scheduling: work items are handed out by atomicAdd on *counter
  int* counter;     // zeroed before the launch
  int items;        // FWD: work items (BWD_G / GRAD derive theirs from the row count)
  // Device-side number of token rows taking part (rows that take no part are
  // compacted away on the device); the launch covers rows n_row0 .. of that
  // compact list, at most N of them: n = clamp(*n_dev - n_row0, 0, N).  N and
  // n_blocks above are the upper bounds.  Null: all N rows.
  const int* n_dev;
  int n_row0;
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
  float softcap;      // > 0: logits are softcap * tanh(logit / softcap)
  float inv_softcap;  // 1 / softcap
  int filter_de;  // 1: dE skips the K-blocks of skipped filter tiles
  int filter_dc;  // 1: dC skips them (0: dC uses every tile, as CCE-Kahan-FullC)
  uint8_t* bitmap;   // [ceil(N/128)][bm_ld] tile survival, token-block major
  uint8_t* bitmapT;  // [bm_ld][ceil(N/128)] the same, vocabulary-block major (read along K by dC)
  int bm_ld;         // ceil(V / 128)
  // FWD_STAGE: each row's max over each 32-column chunk, [v_tiles * 8][N]
  // fp32; the logits minus that max go to tmOut as fp16 [N][v_tiles * 256]
  float* mtile;
  // GRAD, single call: the dE tiles split the vocabulary (K) into de_splits
  // ranges of de_kps K-blocks (even); split s stores its fp32 tile to rows
  // s * de_slab + de_row0 + ... of the tmOut2 tensor (de_splits = 0 or 1:
  // one range, rows de_row0 + ...)
  int de_splits;
  int de_kps;
  int de_slab;
  int de_row0;
  // GRAD: the dC tiles write fp32 through tmOut (SW128 32-column boxes),
  // stored (dc_reduce = 0) or reduce-added (1), instead of bf16
  int dc_f32;
  int dc_reduce;
  // GRAD, bf16 dC tiles: when set, the fp32 [V][D] sum of earlier chunks that
  // each tile adds to its result before rounding (single call, last chunk)
  const float* dc_acc;
  int32_t* dev_err;
};

}  // namespace cce
