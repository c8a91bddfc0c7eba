// Persistent, warp-specialised tcgen05 GEMM with three epilogue modes -- the
// dense contractions of Cut Cross-Entropy on one template:
//
//   MODE_FWD   A = E [N,D] (K-major), B = C [V,D] (K-major).  Epilogue: each
//              row folds its logit tile into a running (max, sumexp) over the
//              work item's vocabulary split and captures the target logit when
//              its column passes ("Cut Your Losses in Large-Vocabulary
//              Language Models", "Memory-Efficient Linear-Log-Sum-Exp, Forward
//              Pass (Algorithm 2)" and "Memory-Efficient Indexed Matrix
//              Multiplication (Algorithm 1)"; the online fold of the
//              "cut-cross-entropy" card's "Method").  Writes per-(row, split)
//              partials; a separate kernel combines them in a fixed order.
//   MODE_BWD_G Same operands over one vocabulary chunk.  Epilogue: G =
//              exp(A - LSE) - onehot(x), the tile filter (skip when every
//              unscaled |G| < eps, decided by warp votes and a shared-memory
//              flag), then G * w rounded to bf16 and stored to the chunk
//              buffer for surviving 128x128 tiles only ("The Combined Backward
//              Pass (Algorithm 4)", "Gradient Filtering").
//   MODE_GRAD  Both gradient contractions of the chunk in one launch:
//              KIND_DC tiles: dC[chunk rows] = G_chunk^T E (A = G MN-major,
//              B = E MN-major, K = tokens; each MN-major operand arrives in one
//              3-D TMA box per stage -- B when D % 64 == 0, else in four 2-D
//              boxes, which cost about 15% of the MMA rate), each tile owns its dC rows and
//              writes them once in bf16, no atomics.  KIND_DE tiles: dE_acc
//              (+)= G_chunk C_chunk (A = G K-major, B = C MN-major, K = chunk
//              columns), fp32 tiles stored (first chunk) or reduce-added by
//              TMA (later chunks): one writer per tile per chunk, chunks in
//              stream order, so the result is deterministic.  K-blocks of
//              skipped filter tiles are not loaded and issue no MMA; CTA pairs
//              run the union of their two tiles' kept K-blocks, loading zeros
//              as A where a CTA's own tile skips one.
//
//   MODE_FWD_STAGE  MODE_FWD whose epilogue also writes each 32-column logit
//              chunk, minus its per-row max, as fp16 to a staging buffer (and
//              the max to mtile) for the single call ("fused-linear-cross-
//              entropy" page, "2. Fused Linear Cross-Entropy (FLCE)": the
//              chunk's logits are kept for the gradient instead of being
//              recomputed).  There MODE_GRAD also covers a token chunk over
//              the whole vocabulary: dE tiles split K into ranges written to
//              separate fp32 slabs, dC tiles may write fp32 (store or add).
//
// Roles (224 threads): warp 0 lane 0 is the scheduler and TMA producer (a
// 4-stage ring of 48 KiB stages); warp 1 owns TMEM (512 columns = two 128x256
// fp32 accumulators) and lane 0 issues tcgen05.mma; warps 2..5 are the
// epilogue (warp w reads TMEM lanes 32*(w%4) .. +31, i.e. tile rows); warp 6
// is the gradient-GEMM pairs' scheduler and idle otherwise.  Work items are
// handed out dynamically (atomicAdd on a counter) and passed to the MMA and
// epilogue warps through a small ring in shared memory, so every CTA stays
// busy until the work runs out; the longest tiles are handed out first.
//
// CTA pairs (template flag PAIR; MODE_FWD and MODE_FWD_STAGE when D % 64 ==
// 0, MODE_BWD_G from 64 token blocks, MODE_GRAD when the D tiles are 256 wide
// and, with the filter on, at least 80% of the chunk's filter tiles are kept):
// clusters of two CTAs on neighbouring SMs work on a pair of neighbouring row
// blocks.  Each CTA loads its 128 rows of A and half of the 256-row B tile;
// the even CTA issues one MMA of M = 256 for both (tcgen05 cta_group::2) and
// commits to both CTAs' barriers, and each CTA's epilogue reads its own 128
// accumulator rows.  FWD and BWD_G pairs take their items in a fixed order;
// GRAD pairs take them from the even CTA's scheduler warp, which also reads
// the two tiles' survival maps for the producers (their K-blocks differ).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_args.h"
#include "ptx.cuh"

namespace cce {

struct Tile {
  int kind;   // KIND_MAIN (FWD, BWD_G), KIND_DC or KIND_DE (GRAD)
  int m;      // A-row block (128)
  int n;      // B-row block (256) or output column block
  int split;  // FWD: vocabulary split; GRAD dE: K range
  bool first, last;  // FWD: first / last tile of a (row block, split) unit
  // false: the odd CTA's half of a pair whose second token block does not
  // exist (an odd number of blocks): the MMA runs on whatever rows are there
  // and the epilogue writes nothing
  bool live = true;
};

// Work sizes that depend on the device-side row count (BWD_G / GRAD run over
// the compacted rows).  Every role computes them from the same value.
struct Dims {
  int nb;     // token blocks of 128 taking part
  int dc_kb;  // K-blocks of the dC contraction (tokens / 64)
  int items;  // work items of the launch
};

template <int MODE, bool PAIR = false>
__device__ __forceinline__ Dims dims_of(const GemmArgs& a) {
  const int n = a.n_dev ? max(0, min(a.N, *a.n_dev - a.n_row0)) : a.N;
  Dims d;
  d.nb = (n + BM - 1) / BM;
  d.dc_kb = (n + BK - 1) / BK;
  if constexpr (PAIR && MODE == MODE_GRAD) {  // items are pairs of vocabulary blocks (dC) or token blocks (dE)
    d.items = (((a.dc_m_tiles + 1) >> 1) + ((d.nb + 1) >> 1) * max(a.de_splits, 1)) * a.n_tiles;
  } else if constexpr (PAIR) {  // items are pairs of token blocks
    const int nbx = (MODE == MODE_BWD_G || a.n_dev) ? d.nb : a.n_blocks;
    d.items = ((nbx + 1) >> 1) * (MODE == MODE_BWD_G ? a.v_tiles : a.splits);
  } else if constexpr (MODE == MODE_FWD || MODE == MODE_FWD_STAGE) {
    d.items = a.n_dev ? d.nb * a.splits : a.items;
  } else if constexpr (MODE == MODE_BWD_G) {
    d.items = d.nb * a.v_tiles;
  } else {
    d.items = (a.dc_m_tiles + d.nb * max(a.de_splits, 1)) * a.n_tiles;
  }
  return d;
}

// Calls f(tile) for every tile of work item `item`; false if f asked to stop.
template <int MODE, bool PAIR = false, typename F>
__device__ __forceinline__ bool for_each_tile_of_item(const GemmArgs& a, const Dims& dm, int item, F&& f) {
  if constexpr (PAIR && MODE == MODE_GRAD) {
    // Gradient GEMM as CTA pairs: an item is a pair of neighbouring row
    // blocks of one kind -- vocabulary blocks 2p, 2p + 1 of the chunk (dC)
    // or token blocks 2p, 2p + 1 (dE, with its K range) -- and a D tile; the
    // CTA of rank r owns block 2p + r, which does not exist for the last pair
    // of an odd count.  Same order as one CTA per tile: the longer kind first,
    // the D tile fastest.
    const int r = static_cast<int>(cluster_ctarank());
    const int nsplit = max(a.de_splits, 1);
    const int dc_items = ((a.dc_m_tiles + 1) >> 1) * a.n_tiles;
    const int de_items = ((dm.nb + 1) >> 1) * nsplit * a.n_tiles;
    int i = item, kind;
    if (a.dc_first) {
      kind = i < dc_items ? KIND_DC : KIND_DE;
      if (kind == KIND_DE) i -= dc_items;
    } else {
      kind = i < de_items ? KIND_DE : KIND_DC;
      if (kind == KIND_DC) i -= de_items;
    }
    if (kind == KIND_DC) {
      const int m = 2 * (i / a.n_tiles) + r;
      return f(Tile{kind, m, i % a.n_tiles, 0, true, true, m < a.dc_m_tiles});
    }
    const int ms = i / a.n_tiles;
    const int m = 2 * (ms / nsplit) + r;
    return f(Tile{kind, m, i % a.n_tiles, ms % nsplit, true, true, m < dm.nb});
  } else if constexpr (PAIR) {
    // CTA pairs (FWD, BWD_G): an item is a pair of neighbouring
    // token blocks with a vocabulary split (FWD) or tile (BWD_G), in the same
    // grouped raster (group_n even, so groups hold whole pairs); the CTA of
    // rank r takes block 2p + r, which does not exist for the last pair of an
    // odd number of blocks.
    constexpr bool kFwd = MODE != MODE_BWD_G;
    const int nbx = (!kFwd || a.n_dev) ? dm.nb : a.n_blocks;
    const int nbp = (nbx + 1) >> 1, gp = a.group_n >> 1;
    const int width = kFwd ? a.splits : a.v_tiles;
    const int per_group = gp * width;
    const int g = item / per_group, j = item - g * per_group;
    const int gpn = min(gp, nbp - g * gp);
    const int m = 2 * (g * gp + j % gpn) + static_cast<int>(cluster_ctarank());
    const bool live = m < nbx;
    if constexpr (!kFwd) {
      return f(Tile{KIND_MAIN, m, j / gpn, 0, true, true, live});
    } else {
      const int s = j / gpn;
      const int t0 = static_cast<int>(static_cast<long long>(s) * a.v_tiles / a.splits);
      const int t1 = static_cast<int>(static_cast<long long>(s + 1) * a.v_tiles / a.splits);
      for (int t = t0; t < t1; ++t) {
        if (!f(Tile{KIND_MAIN, m, t, s, t == t0, t == t1 - 1, live})) return false;
      }
      return true;
    }
  } else if constexpr (MODE == MODE_FWD || MODE == MODE_FWD_STAGE) {
    // Grouped raster as in BWD_G: groups of group_n token blocks, the token
    // block fastest inside a group, then the vocabulary split.  The CTAs of
    // a split share its C tiles, and a group's E rows stay in L2 while the
    // group's items run.
    const int nbx = a.n_dev ? dm.nb : a.n_blocks;  // items only exist when nbx > 0
    const int per_group = a.group_n * a.splits;
    const int g = item / per_group, j = item - g * per_group;
    const int gn = min(a.group_n, nbx - g * a.group_n);
    const int m = g * a.group_n + j % gn, s = j / gn;
    const int t0 = static_cast<int>(static_cast<long long>(s) * a.v_tiles / a.splits);
    const int t1 = static_cast<int>(static_cast<long long>(s + 1) * a.v_tiles / a.splits);
    for (int t = t0; t < t1; ++t) {
      if (!f(Tile{KIND_MAIN, m, t, s, t == t0, t == t1 - 1})) return false;
    }
    return true;
  } else if constexpr (MODE == MODE_BWD_G) {
    // Grouped raster: groups of group_n token blocks; inside a group the
    // token block varies fastest, then the vocabulary tile.  CTAs running at
    // the same time share a few C tiles and a group's E rows stay in L2.
    const int per_group = a.group_n * a.v_tiles;
    const int g = item / per_group, j = item - g * per_group;
    const int gn = min(a.group_n, dm.nb - g * a.group_n);
    return f(Tile{KIND_MAIN, g * a.group_n + j % gn, j / gn, 0, true, true});
  } else {
    const int dc_tiles = a.dc_m_tiles * a.n_tiles;
    const int nsplit = max(a.de_splits, 1);
    const int de_tiles = dm.nb * nsplit * a.n_tiles;
    int i = item, kind;
    if (a.dc_first) {
      kind = i < dc_tiles ? KIND_DC : KIND_DE;
      if (kind == KIND_DE) i -= dc_tiles;
    } else {
      kind = i < de_tiles ? KIND_DE : KIND_DC;
      if (kind == KIND_DC) i -= de_tiles;
    }
    // the column (D) tile varies fastest: neighbouring CTAs share the A operand
    if (kind == KIND_DC) return f(Tile{kind, i / a.n_tiles, i % a.n_tiles, 0, true, true});
    const int ms = i / a.n_tiles;  // (token block, K range)
    return f(Tile{kind, ms / nsplit, i % a.n_tiles, ms % nsplit, true, true});
  }
}

// K-blocks [kblock_begin, kblocks_of) of tile t.
template <int MODE>
__device__ __forceinline__ int kblocks_of(const GemmArgs& a, const Dims& dm, const Tile& t) {
  if constexpr (MODE == MODE_GRAD) {
    if (t.kind == KIND_DC) return dm.dc_kb;
    return a.de_splits > 1 ? min(a.de_k_blocks, (t.split + 1) * a.de_kps) : a.de_k_blocks;
  }
  return a.k_blocks;
}

template <int MODE>
__device__ __forceinline__ int kblock_begin(const GemmArgs& a, const Tile& t) {
  if constexpr (MODE == MODE_GRAD) {
    if (t.kind == KIND_DE && a.de_splits > 1) return t.split * a.de_kps;
  }
  return 0;
}

// The first K-block >= kb of tile t that the filter keeps (nk when none).
// dC: K = tokens, read from the vocabulary-major map; dE: K = chunk columns;
// FWD and BWD_G never skip.  Filter tile j covers K-blocks 2j and 2j + 1;
// the survival bytes are read 8
// at a time with independent loads, so a long run of skipped tiles costs one
// load latency per 16 K-blocks instead of one per K-block.
template <int MODE>
__device__ __forceinline__ int next_kblock(const GemmArgs& a, const Tile& t, int kb, int nk) {
  if constexpr (MODE != MODE_GRAD) {
    return kb;
  } else {
    const uint8_t* row;
    if (t.kind == KIND_DC) {
      if (!a.filter_dc) return kb;
      row = a.bitmapT + static_cast<size_t>((a.chunk_v0 >> 7) + t.m) * a.n_blocks;
    } else {
      if (!a.filter_de) return kb;
      row = a.bitmap + static_cast<size_t>(t.m) * a.bm_ld + (a.chunk_v0 >> 7);
    }
    const int jn = (nk + 1) >> 1;
    int j = kb >> 1;
    if (j >= jn) return nk;
    if (__ldg(row + j)) return kb;  // kept: the common case of a dense tile costs one load
    ++j;
    while (j < jn) {
      if (j + 8 <= jn) {
        uint8_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldg(row + j + u);
        int f = 8;
#pragma unroll
        for (int u = 7; u >= 0; --u) f = v[u] ? u : f;
        if (f < 8) return max(kb, 2 * (j + f));
        j += 8;
      } else {
        if (__ldg(row + j)) return max(kb, 2 * j);
        ++j;
      }
    }
    return nk;
  }
}

// Reader of one tile's survival map along its K range (gradient GEMM as CTA
// pairs): dC tiles (K = tokens) read the vocabulary-major map, dE tiles
// (K = chunk columns) the token-major one; filter column j covers K-blocks 2j
// and 2j + 1.  The map is read 64 columns (128 K-blocks) at a time, with 64
// independent byte loads, into a bit mask.
struct KeepCursor {
  const uint8_t* row;  // survival bytes of the tile's filter row (column j at row[j])
  int jn;              // filter columns up to the end of the tile's K range
  int w;               // window of columns held in bits (-1: none)
  uint64_t bits;       // bit i: column 64 w + i is kept
  bool all;            // the tile's output is not filtered: every K-block is kept
};

__device__ __forceinline__ KeepCursor keep_cursor(const GemmArgs& a, const Tile& t, int nk) {
  KeepCursor c;
  c.jn = (nk + 1) >> 1;
  c.w = -1;
  c.bits = 0;
  if (t.kind == KIND_DC) {
    c.all = !a.filter_dc;
    c.row = a.bitmapT + static_cast<size_t>((a.chunk_v0 >> 7) + t.m) * a.n_blocks;
  } else {
    c.all = !a.filter_de;
    c.row = a.bitmap + static_cast<size_t>(t.m) * a.bm_ld + (a.chunk_v0 >> 7);
  }
  return c;
}

__device__ __forceinline__ void keep_window(KeepCursor& c, int w) {
  const int j0 = 64 * w;
  uint8_t v[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = (j0 + i < c.jn) ? __ldg(c.row + j0 + i) : uint8_t(0);
  uint64_t b = 0;
#pragma unroll
  for (int i = 0; i < 64; ++i) b |= static_cast<uint64_t>(v[i] != 0) << i;
  c.bits = b;
  c.w = w;
}

// The first filter column >= j that the cursor's tile keeps (jn when none).
__device__ __forceinline__ int keep_next(KeepCursor& c, int j) {
  if (c.all) return min(j, c.jn);
  while (j < c.jn) {
    const int w = j >> 6;
    if (w != c.w) keep_window(c, w);
    const uint64_t m = c.bits >> (j & 63);
    if (m) return j + __ffsll(static_cast<long long>(m)) - 1;
    j = 64 * (w + 1);
  }
  return c.jn;
}

// Warp-wide: does the output tile have no surviving K-block at all?
__device__ __forceinline__ bool tile_empty(const GemmArgs& a, const Dims& dm, const Tile& t) {
  // no K-block at all (no row of a dC tile's chunk takes part): the MMA thread
  // never wrote the accumulator
  if (kblocks_of<MODE_GRAD>(a, dm, t) <= kblock_begin<MODE_GRAD>(a, t)) return true;
  if (!(t.kind == KIND_DC ? a.filter_dc : a.filter_de)) return false;  // this output is not filtered
  int any = 0;
  if (t.kind == KIND_DC) {
    const uint8_t* row = a.bitmapT + static_cast<size_t>((a.chunk_v0 >> 7) + t.m) * a.n_blocks;
    for (int r = lane_id(); r < dm.nb; r += 32) any |= __ldg(row + r);
  } else {
    // the filter columns of the tile's K range (two K-blocks per column)
    const int j0 = kblock_begin<MODE_GRAD>(a, t) >> 1;
    const int j1 = (kblocks_of<MODE_GRAD>(a, dm, t) + 1) >> 1;
    const uint8_t* row = a.bitmap + static_cast<size_t>(t.m) * a.bm_ld + (a.chunk_v0 >> 7);
    for (int j = j0 + lane_id(); j < j1; j += 32) any |= __ldg(row + j);
  }
  return __any_sync(0xffffffffu, any) == 0;
}

// GRAD as CTA pairs: the pair's MMAs run over the union of the K-blocks its
// two tiles keep, and a CTA whose own tile skips a K-block of it loads zeros
// as its A operand there.  Its K-blocks are 128 deep, one filter column each.
// PairKeep walks that union on the two tiles' maps (both CTAs the same
// union); a tile whose block does not exist (the last pair of an odd count)
// keeps nothing.  The producer walks it only for a K range longer than the
// scheduler's survival words (see RING_WIDE).
struct PairKeep {
  KeepCursor own, peer;
  bool own_live, peer_live;
  int jn;      // end of the K range in columns
  int on, pn;  // the next column each tile keeps (jn: none left)
};

__device__ __forceinline__ PairKeep pair_keep(const GemmArgs& a, const Dims& dm, const Tile& t, int nk) {
  PairKeep p;
  Tile peer = t;
  peer.m = t.m ^ 1;
  p.own_live = t.live;
  p.peer_live = peer.m < (t.kind == KIND_DC ? a.dc_m_tiles : dm.nb);
  p.own = keep_cursor(a, t, nk);
  p.peer = keep_cursor(a, peer, nk);
  p.jn = p.own.jn;
  const int j0 = kblock_begin<MODE_GRAD>(a, t) >> 1;
  p.on = p.own_live ? keep_next(p.own, j0) : p.jn;
  p.pn = p.peer_live ? keep_next(p.peer, j0) : p.jn;
  return p;
}

// The pair's current column (jn when the union is exhausted).
__device__ __forceinline__ int pair_kb(const PairKeep& p) { return min(p.on, p.pn); }

// Moves past column j (the current one).
__device__ __forceinline__ void pair_advance(PairKeep& p, int j) {
  if (p.on == j) p.on = p.own_live ? keep_next(p.own, j + 1) : p.jn;
  if (p.pn == j) p.pn = p.peer_live ? keep_next(p.peer, j + 1) : p.jn;
}

__device__ __forceinline__ float ex2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled box
// (128-byte rows, box 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// The same for a 64-byte-swizzled box (64-byte rows, box 512-byte aligned).
__device__ __forceinline__ uint32_t swz64(uint32_t r, uint32_t c) {
  return r * 64u + ((c ^ ((r >> 1) & 3u)) << 4);
}

struct SmemLayout {
  uint8_t* stages;
  uint8_t* epi;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tmem_full;
  uint64_t* tmem_empty;
  uint64_t* vote;
  uint64_t* drain;
  uint64_t* ring_full;
  uint64_t* ring_empty;
  uint32_t* tmem_base;
  int* abort_flag;
  int* flags;       // [2 parity][2 half][4 warps]
  int* ring_ids;    // [RING]
  int* stage_meta;  // [MAX_STAGES] what the producer put in the stage (META_*)
  // gradient-GEMM pairs: per word slot, this CTA's own survival words, the
  // union's, and the union's last (128-deep) K-block; the even CTA's
  // words_free[s] counts both producers' releases of slot s
  uint64_t* ring_own;  // [WORD_SLOTS][PAIR_MAP_WORDS]
  uint64_t* ring_uni;  // [WORD_SLOTS][PAIR_MAP_WORDS]
  int* ring_last;      // [WORD_SLOTS]
  uint64_t* words_free;  // [WORD_SLOTS]
  // CTA pairs: cluster address of the even CTA's tmem_empty[0] (0: no pair)
  uint32_t tmem_empty_lead;
};

// Stage tags written by the producer before it arms the stage's full
// barrier: the MMA thread learns where a tile's K loop ends (or that the
// tile has no K-block left after filtering) without reading the filter map.
constexpr int META_LAST = 1;   // the tile's last K-block
constexpr int META_EMPTY = 2;  // no data: the tile has no K-block at all

__device__ __forceinline__ SmemLayout carve_smem(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.stages = base;
  L.epi = base + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(L.epi + NUM_EPI_WARPS * EPI_WARP_BYTES);
  L.full = bars;                          // MAX_STAGES
  L.empty = L.full + MAX_STAGES;          // MAX_STAGES
  L.tmem_full = L.empty + MAX_STAGES;     // 2
  L.tmem_empty = L.tmem_full + 2;         // 2
  L.vote = L.tmem_empty + 2;              // 2
  L.drain = L.vote + 2;                   // 1
  L.ring_full = L.drain + 1;              // RING
  L.ring_empty = L.ring_full + RING;      // RING
  L.words_free = L.ring_empty + RING;     // WORD_SLOTS
  uint8_t* tail = reinterpret_cast<uint8_t*>(L.words_free + WORD_SLOTS);
  L.tmem_base = reinterpret_cast<uint32_t*>(tail);
  L.abort_flag = reinterpret_cast<int*>(tail + 4);
  L.flags = reinterpret_cast<int*>(tail + 8);      // 16 ints
  L.ring_ids = reinterpret_cast<int*>(tail + 72);  // RING ints
  L.stage_meta = reinterpret_cast<int*>(tail + 72 + 4 * RING);  // MAX_STAGES ints
  constexpr int kWords = 72 + 4 * RING + 4 * MAX_STAGES;
  L.ring_own = reinterpret_cast<uint64_t*>(tail + ((kWords + 7) & ~7));
  L.ring_uni = L.ring_own + WORD_SLOTS * PAIR_MAP_WORDS;
  L.ring_last = reinterpret_cast<int*>(L.ring_uni + WORD_SLOTS * PAIR_MAP_WORDS);
  static_assert(8 * (2 * MAX_STAGES + 7 + 2 * RING + WORD_SLOTS) + ((kWords + 7) & ~7) +
                        16 * WORD_SLOTS * PAIR_MAP_WORDS + 4 * WORD_SLOTS <=
                    BAR_BYTES,
                "barriers and ring data fit their region");
  L.tmem_empty_lead = 0;
  return L;
}

// ------------------------------------------------------- work-item ring
// Consumer side: the k-th work item, or -1 when the work has run out (or the
// CTA aborted).  Single thread.
__device__ __forceinline__ int ring_take(const SmemLayout& L, int k, const GemmArgs& a) {
  const int slot = k % RING;
  const uint32_t par = static_cast<uint32_t>((k / RING) & 1);
  if (!wait_bounded(&L.ring_full[slot], par, L.abort_flag, a.dev_err)) return -1;
  const int item = *reinterpret_cast<volatile int*>(&L.ring_ids[slot]);
  mbar_arrive(&L.ring_empty[slot]);
  return item;
}

// GRAD as CTA pairs: the even CTA's scheduler warp hands out the items and
// writes each into both CTAs' rings.  The odd CTA's consumers (its producer
// and its epilogue warps) take theirs with a cluster-scope wait and free the
// slot on the even CTA's ring_empty barrier, which counts both CTAs'
// consumers.
__device__ __forceinline__ int ring_take_odd(const SmemLayout& L, int k, const GemmArgs& a) {
  const int slot = k % RING;
  const uint32_t par = static_cast<uint32_t>((k / RING) & 1);
  if (!wait_bounded<true>(&L.ring_full[slot], par, L.abort_flag, a.dev_err)) return -1;
  const int item = *reinterpret_cast<volatile int*>(&L.ring_ids[slot]);
  mbar_arrive_cluster(mapa_shared(smem_u32(&L.ring_empty[slot]), 0));
  return item;
}

// The k-th work item for a consumer of this CTA (pairs of the gradient GEMM:
// the odd CTA's consumers read what the even CTA's scheduler wrote).
template <int MODE, bool PAIR>
__device__ __forceinline__ int ring_take_any(const SmemLayout& L, int k, const GemmArgs& a) {
  if constexpr (PAIR && MODE == MODE_GRAD) {
    if (cluster_ctarank() != 0) return ring_take_odd(L, k, a);
  }
  return ring_take(L, k, a);
}

// ------------------------------------------------------------ L2 prefetch
// FWD_STAGE only: the CTAs of one raster group and vocabulary split walk the
// split's C tiles together, and this kernel's epilogue also streams the
// staged logits to DRAM; at the start of tile n the CTA at place r of the
// group asks the copy engine to bring K-blocks r, r + gn, ... of tile n + 1
// into L2, so each box is requested once, a tile ahead of need.  (Measured:
// 5.6% off this kernel at the Qwen shape, 2% at Gemma; the same prefetch
// made the two-call forward and the recompute up to 2.6% slower, and an A
// prefetch 12 K-blocks ahead made the gradient GEMM 25% slower.)
__device__ __forceinline__ void prefetch_next_b(const GemmArgs& a, const Dims& dm, const Tile& t) {
  if (t.last) return;
  const int nbx = a.n_dev ? dm.nb : a.n_blocks;
  const int g0 = t.m - t.m % a.group_n, gn = min(a.group_n, nbx - g0);
  for (int kb = t.m - g0; kb < a.k_blocks; kb += gn) tma_prefetch_l2_2d(&a.tmB, kb * BK, a.c_row0 + (t.n + 1) * BN);
}

// ---------------------------------------------------------------- producer
template <int MODE, bool PAIR = false>
__device__ __forceinline__ void producer_loop(const GemmArgs& a, const SmemLayout& L) {
  using P = Pipe<MODE, PAIR>;
  volatile int* abort_flag = L.abort_flag;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued_mask = 0, issued_par = 0;  // per stage: ever issued, parity of last issue
  const Dims dm = dims_of<MODE, PAIR>(a);
  // BWD_G: the next work item is fetched while the current one's loads are
  // issued; the atomic's latency (about a microsecond) would otherwise stall
  // the pipeline at every boundary of its short one-tile items.  The other
  // modes fetch when they need one: their items are long, and holding a
  // reserved item while busy would unbalance the end of a launch.
  constexpr bool kAhead = MODE == MODE_BWD_G && !PAIR;
  int next = kAhead ? atomicAdd(a.counter, 1) : 0;
  // CTA pairs take items in a fixed order (cluster c: c, c + clusters, ...),
  // the same in both CTAs, so neither needs the other's schedule; forward
  // items are all of one size.  The even CTA's full barriers count both
  // CTAs' copies.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int pair_first = PAIR ? static_cast<int>(cluster_id_x()) : 0;
  const int pair_step = PAIR ? static_cast<int>(cluster_count_x()) : 0;
  for (int k = 0;; ++k) {
    const int slot = k % RING;
    if (!wait_bounded(&L.ring_empty[slot], static_cast<uint32_t>(((k / RING) & 1) ^ 1), abort_flag, a.dev_err))
      break;
    int item = PAIR ? pair_first + k * pair_step : (kAhead ? next : atomicAdd(a.counter, 1));
    if (item >= dm.items) item = -1;
    L.ring_ids[slot] = item;
    mbar_arrive(&L.ring_full[slot]);  // release: the id is visible to the waiting consumers
    if (item < 0) break;
    if (kAhead) next = atomicAdd(a.counter, 1);
    const bool ok = for_each_tile_of_item<MODE, PAIR>(a, dm, item, [&](const Tile& t) -> bool {
      // pairs: K-blocks 128 deep
      const int nk = PAIR ? (kblocks_of<MODE>(a, dm, t) + 1) >> 1 : kblocks_of<MODE>(a, dm, t);
      if (MODE == MODE_FWD_STAGE) prefetch_next_b(a, dm, t);
      int kb = next_kblock<MODE>(a, t, kblock_begin<MODE>(a, t), nk);
      if (MODE == MODE_GRAD && kb >= nk) {  // nothing survives the filter: an empty tagged stage
        if (!wait_bounded(&L.empty[stage], phase ^ 1u, abort_flag, a.dev_err)) return false;
        L.stage_meta[stage] = META_EMPTY;
        mbar_arrive(&L.full[stage]);
        // tracked like a copy, so the abort drain below waits on this stage's latest phase
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == P::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        return true;
      }
      while (kb < nk) {
        const int next = next_kblock<MODE>(a, t, kb + 1, nk);
        if (!wait_bounded(&L.empty[stage], phase ^ 1u, abort_flag, a.dev_err)) return false;
        if (MODE == MODE_GRAD) L.stage_meta[stage] = next >= nk ? META_LAST : 0;
        uint8_t* sA = L.stages + stage * P::kStageBytes;
        uint8_t* sB = sA + P::kABytes;
        uint64_t* fb = &L.full[stage];
        const int k0 = kb * P::kBK;
        if constexpr (PAIR) {
          // this CTA's 128 rows of A and its half (128 rows) of the B tile,
          // each one 3-D box of two 64-column K groups
          const uint32_t fb_lead = mapa_shared(smem_u32(fb), 0);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * P::kStageBytes);
          tma_load_3d_pair(&a.tmA, fb_lead, sA, 0, t.m * BM, k0 >> 6);
          tma_load_3d_pair(&a.tmB2, fb_lead, sB, 0, a.c_row0 + t.n * BN + static_cast<int>(rank) * (BN / 2), k0 >> 6);
        } else if (MODE != MODE_GRAD) {
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_2d(&a.tmA, fb, sA, k0, t.m * BM);
          tma_load_2d(&a.tmB, fb, sB, k0, a.c_row0 + t.n * BN);
        } else if (t.kind == KIND_DC) {
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_3d(&a.tmA, fb, sA, 0, k0, (t.m * BM) >> 6);  // both 64-column groups of A
          if (a.b3d) {  // the four 64-column groups of B in one instruction
            tma_load_3d(&a.tmB, fb, sB, 0, k0, (t.n * a.bn) >> 6);
          } else {
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(&a.tmB, fb, sB + j * 8192, t.n * a.bn + j * 64, k0);
          }
        } else {
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_2d(&a.tmA2, fb, sA, k0, t.m * BM);
          if (a.b3d) {
            tma_load_3d(&a.tmB2, fb, sB, 0, a.c_row0 + k0, (t.n * a.bn) >> 6);
          } else {
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(&a.tmB2, fb, sB + j * 8192, t.n * a.bn + j * 64, a.c_row0 + k0);
          }
        }
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == P::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        kb = next;
      }
      return true;
    });
    if (!ok) break;
  }
  if (PAIR && rank != 0 && *abort_flag) {
    // This CTA's copies complete on the even CTA's barriers; give any still
    // in flight a bounded 10 ms to land before the CTA exits.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 10000000ull) {
    }
  } else if (*abort_flag) {
    // Let every copy this thread issued land before the CTA exits.
    for (int s = 0; s < P::kStages; ++s) {
      if (issued_mask & (1u << s)) {
        volatile int dummy = 0;
        wait_bounded(&L.full[s], (issued_par >> s) & 1u, &dummy, nullptr);
      }
    }
  }
}

// The tile that work item `item` gives this CTA (gradient GEMM as CTA pairs).
__device__ __forceinline__ Tile grad_pair_tile(const GemmArgs& a, const Dims& dm, int item) {
  Tile t{};
  for_each_tile_of_item<MODE_GRAD, true>(a, dm, item, [&](const Tile& u) -> bool {
    t = u;
    return true;
  });
  return t;
}

// Width of a gradient-GEMM pair's tile: BN, or 128 for a last D tile of 128
// columns (D = 896: 3 x 256 + 128), which then runs MMAs of N = 128 instead
// of multiplying 128 columns of padding.  Each CTA of a pair holds half of N
// in whole 64-column groups, so narrower remainders keep N = 256.
__device__ __forceinline__ int pair_tile_n(const GemmArgs& a, const Tile& t) {
  return a.D - t.n * a.bn == BN / 2 ? BN / 2 : BN;
}

// Ring entries of the gradient GEMM as CTA pairs: 4 item + kind, -1 when no
// work is left.  Kinds: RING_NONE, neither tile keeps a K-block; RING_DENSE,
// both keep every K-block of the range; RING_BITS, the slot's survival words
// say which K-blocks (one per filter column) the pair runs (their union) and
// which of them this CTA's own tile keeps; RING_WIDE, a K range of more than
// a.pair_words words, which the producer walks on the maps itself.
constexpr int RING_BITS = 0, RING_NONE = 1, RING_DENSE = 2, RING_WIDE = 3;

// One word of a tile's survival map: bit i for filter column 64 w + i, kept
// and inside [j0, jn).
__device__ __forceinline__ uint64_t keep_word(KeepCursor& c, bool live, int w, int j0) {
  if (!live) return 0;
  uint64_t b;
  if (c.all) {
    b = ~0ull;
  } else {
    keep_window(c, w);
    b = c.bits;
  }
  const int lo = j0 - 64 * w, hi = c.jn - 64 * w;  // the range in this word's bits
  if (lo > 0) b &= ~0ull << lo;
  if (hi < 64) b &= (1ull << hi) - 1;
  return b;
}

// Scheduler of the gradient GEMM as CTA pairs (the even CTA's warp 6): takes
// the work items from the counter, reads both tiles' survival maps and
// writes each entry, with its survival words, into both CTAs' rings, up to
// RING items ahead of the consumers.  The map reads and the counter's atomic
// latency are thus off the producers' critical path: the producer's work per
// K-block sets the pace of the pair (the M = 256 MMAs of one K-block take
// about 500 cycles), and measured, every instruction added to it showed.
__device__ __forceinline__ void scheduler_loop_grad_pair(const GemmArgs& a, const SmemLayout& L) {
  volatile int* abort_flag = L.abort_flag;
  const Dims dm = dims_of<MODE_GRAD, true>(a);
  for (int k = 0;; ++k) {
    const int slot = k % RING;
    // both CTAs' consumers have released the slot's previous item (cluster
    // scope: the odd CTA's reads of its copy come before the slot is rewritten)
    if (!wait_bounded<true>(&L.ring_empty[slot], static_cast<uint32_t>(((k / RING) & 1) ^ 1), abort_flag,
                            a.dev_err))
      break;
    // both producers are done with the word slot's previous item
    const int ws = k % WORD_SLOTS;
    if (!wait_bounded<true>(&L.words_free[ws], static_cast<uint32_t>(((k / WORD_SLOTS) & 1) ^ 1), abort_flag,
                            a.dev_err))
      break;
    const int item = atomicAdd(a.counter, 1);
    int v = -1;
    if (item < dm.items) {
      const Tile t = grad_pair_tile(a, dm, item);  // the even CTA's tile (always live)
      Tile peer = t;
      peer.m = t.m + 1;
      const bool peer_live = peer.m < (t.kind == KIND_DC ? a.dc_m_tiles : dm.nb);
      const int nk = kblocks_of<MODE_GRAD>(a, dm, t);
      const int j0 = kblock_begin<MODE_GRAD>(a, t) >> 1;
      KeepCursor oc = keep_cursor(a, t, nk), pc = keep_cursor(a, peer, nk);
      const int jn = oc.jn;
      const int w0 = j0 >> 6, wn = jn > j0 ? ((jn - 1) >> 6) + 1 : w0;
      int kind = RING_WIDE;
      if (wn - w0 <= a.pair_words) {
        bool any = false, dense = peer_live;
        int last = -1;
        uint64_t* own = L.ring_own + ws * PAIR_MAP_WORDS;
        uint64_t* uni = L.ring_uni + ws * PAIR_MAP_WORDS;
        const uint32_t own_odd = mapa_shared(smem_u32(own), 1), uni_odd = mapa_shared(smem_u32(uni), 1);
        for (int w = w0; w < wn; ++w) {
          const uint64_t ob = keep_word(oc, true, w, j0);
          const uint64_t pb = keep_word(pc, peer_live, w, j0);
          const uint64_t ub = ob | pb;
          uint64_t full = ~0ull;  // the range's bits in this word
          if (j0 - 64 * w > 0) full &= ~0ull << (j0 - 64 * w);
          if (jn - 64 * w < 64) full &= (1ull << (jn - 64 * w)) - 1;
          dense = dense && ob == full && pb == full;
          if (ub) {
            any = true;
            last = 64 * w + 63 - __clzll(static_cast<long long>(ub));
          }
          own[w - w0] = ob;
          uni[w - w0] = ub;
          st_shared_cluster_u64(own_odd + 8u * static_cast<uint32_t>(w - w0), pb);  // the odd CTA's own tile
          st_shared_cluster_u64(uni_odd + 8u * static_cast<uint32_t>(w - w0), ub);
        }
        kind = !any ? RING_NONE : (dense ? RING_DENSE : RING_BITS);
        L.ring_last[ws] = last;
        st_shared_cluster_u32(mapa_shared(smem_u32(&L.ring_last[ws]), 1), static_cast<uint32_t>(last));
      }
      v = 4 * item + kind;
    }
    L.ring_ids[slot] = v;
    st_shared_cluster_u32(mapa_shared(smem_u32(&L.ring_ids[slot]), 1), static_cast<uint32_t>(v));
    mbar_arrive(&L.ring_full[slot]);
    mbar_arrive_cluster(mapa_shared(smem_u32(&L.ring_full[slot]), 1));  // release: the slot is visible first
    if (v < 0) break;
  }
}

// Producer of the gradient GEMM as CTA pairs (both CTAs).  Each CTA loads its
// 128 rows of A (or 32 KiB of zeros where its own tile skips a K-block the
// other tile keeps) and its half (128 columns) of the MN-major B tile, all
// completing on the even CTA's full barrier, whose MMA thread issues one
// M = 256 MMA for both.  The producer holds the item's word slot (and reads
// its survival words) until the tile's loads are issued.
__device__ __forceinline__ void producer_loop_grad_pair(const GemmArgs& a, const SmemLayout& L) {
  using P = Pipe<MODE_GRAD, true>;
  volatile int* abort_flag = L.abort_flag;
  const uint32_t rank = cluster_ctarank();
  const Dims dm = dims_of<MODE_GRAD, true>(a);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued_mask = 0, issued_par = 0;
  const uint32_t full_lead = mapa_shared(smem_u32(&L.full[0]), 0);  // the even CTA's full barriers
  // Loads K-block kb (128 deep) of tile t into the next stage: this CTA's A
  // rows (zeros where `mine` is false) and its half of B, each one 3-D box.
  auto issue = [&](const Tile& t, int kb, bool mine, bool last) -> bool {
    if (!wait_bounded(&L.empty[stage], phase ^ 1u, abort_flag, a.dev_err)) return false;
    uint8_t* sA = L.stages + stage * P::kStageBytes;
    uint8_t* sB = sA + P::kABytes;
    const uint32_t fb_lead = full_lead + 8u * static_cast<uint32_t>(stage);
    if (rank == 0) {
      L.stage_meta[stage] = last ? META_LAST : 0;
      mbar_arrive_expect_tx(&L.full[stage], 2 * P::kStageBytes);
    }
    const int k0 = kb * P::kBK;
    // first 64-column group of this CTA's half of the B tile (of N columns)
    const int bz = (t.n * a.bn + static_cast<int>(rank) * (pair_tile_n(a, t) / 2)) >> 6;
    if (!mine) {
      tma_load_2d_pair(&a.tmZ, fb_lead, sA, 0, 0);
    } else if (t.kind == KIND_DC) {
      tma_load_3d_pair(&a.tmA, fb_lead, sA, 0, k0, (t.m * BM) >> 6);
    } else {
      tma_load_3d_pair(&a.tmA2, fb_lead, sA, 0, t.m * BM, k0 >> 6);  // two 64-column groups of K
    }
    if (t.kind == KIND_DC) {
      tma_load_3d_pair(&a.tmB, fb_lead, sB, 0, k0, bz);
    } else {
      tma_load_3d_pair(&a.tmB2, fb_lead, sB, 0, a.c_row0 + k0, bz);
    }
    issued_mask |= 1u << stage;
    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
    if (++stage == P::kStages) {
      stage = 0;
      phase ^= 1u;
    }
    return true;
  };
  for (int k = 0;; ++k) {
    const int slot = k % RING;
    if (!wait_bounded<true>(&L.ring_full[slot], static_cast<uint32_t>((k / RING) & 1), abort_flag, a.dev_err))
      break;
    const int v = *reinterpret_cast<volatile int*>(&L.ring_ids[slot]);
    if (rank == 0) {
      mbar_arrive(&L.ring_empty[slot]);
    } else {
      mbar_arrive_cluster(mapa_shared(smem_u32(&L.ring_empty[slot]), 0));
    }
    if (v < 0) break;
    const int ws = k % WORD_SLOTS;
    auto free_words = [&] {  // this producer is done with the item's survival words
      if (rank == 0) {
        mbar_arrive(&L.words_free[ws]);
      } else {
        mbar_arrive_cluster(mapa_shared(smem_u32(&L.words_free[ws]), 0));
      }
    };
    const int kind = v & 3;
    // RING_NONE: no stage at all; the MMA thread reads the same from the ring
    // entry and signals the epilogues without an MMA.  (A stage without
    // copies would let the even CTA's MMA thread release this CTA's stage
    // twice before this CTA waits on it: only the odd CTA's copies, which
    // complete on the even CTA's full barrier, keep the two CTAs' stage
    // phases in step.)
    if (kind == RING_NONE) {
      free_words();
      continue;
    }
    const Tile t = grad_pair_tile(a, dm, v >> 2);
    const int nk = kblocks_of<MODE_GRAD>(a, dm, t);  // 64-deep K-blocks
    const int j0 = kblock_begin<MODE_GRAD>(a, t) >> 1, jn = (nk + 1) >> 1;  // 128-deep ones
    bool ok = true;
    if (kind == RING_DENSE) {
      free_words();
      for (int j = j0; ok && j < jn; ++j) ok = issue(t, j, true, j + 1 == jn);
    } else if (kind == RING_BITS) {
      const uint64_t* own = L.ring_own + ws * PAIR_MAP_WORDS;
      const uint64_t* uni = L.ring_uni + ws * PAIR_MAP_WORDS;
      const int last = L.ring_last[ws];
      const int w0 = j0 >> 6, wn = jn > j0 ? ((jn - 1) >> 6) + 1 : w0;
      for (int w = w0; ok && w < wn; ++w) {
        uint64_t u = uni[w - w0];
        const uint64_t o = own[w - w0];
        while (ok && u) {
          const int i = __ffsll(static_cast<long long>(u)) - 1;
          u &= u - 1;
          const int j = 64 * w + i;
          ok = issue(t, j, (o >> i) & 1u, j == last);
        }
      }
      free_words();
    } else {  // RING_WIDE
      free_words();
      PairKeep pk = pair_keep(a, dm, t, nk);
      for (int j = pair_kb(pk); ok && j < jn;) {
        const bool mine = pk.on == j;
        pair_advance(pk, j);
        const int next = pair_kb(pk);
        ok = issue(t, j, mine, next >= jn);
        j = next;
      }
    }
    if (!ok) break;
  }
  if (rank != 0 && *abort_flag) {
    // This CTA's copies complete on the even CTA's barriers; give any still
    // in flight a bounded 10 ms to land before the CTA exits.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 10000000ull) {
    }
  } else if (*abort_flag) {
    for (int s = 0; s < P::kStages; ++s) {
      if (issued_mask & (1u << s)) {
        volatile int dummy = 0;
        wait_bounded(&L.full[s], (issued_par >> s) & 1u, &dummy, nullptr);
      }
    }
  }
}

// --------------------------------------------------------------------- MMA
template <int MODE, bool PAIR = false>
__device__ __forceinline__ void mma_loop(const GemmArgs& a, const SmemLayout& L, uint32_t tmem_base) {
  // CTA pairs: the even CTA issues every MMA (M = 256) for both; the odd
  // CTA's MMA thread has nothing to do.
  if (PAIR && cluster_ctarank() != 0) return;
  constexpr int kStages = Pipe<MODE, PAIR>::kStages, kStageBytes = Pipe<MODE, PAIR>::kStageBytes;
  constexpr int kABytes = Pipe<MODE, PAIR>::kABytes, kBK = Pipe<MODE, PAIR>::kBK;
  volatile int* abort_flag = L.abort_flag;
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool issued_any = false;
  const Dims dm = dims_of<MODE, PAIR>(a);
  for (int k = 0;; ++k) {
    int item = ring_take(L, k, a);
    if (item < 0) break;
    bool none_kept = false;  // gradient-GEMM pairs: neither tile keeps a K-block
    if constexpr (PAIR && MODE == MODE_GRAD) {
      none_kept = (item & 3) == RING_NONE;
      item >>= 2;
    }
    const bool ok = for_each_tile_of_item<MODE, PAIR>(a, dm, item, [&](const Tile& t) -> bool {
      // Operand majorness and tile width of this tile.
      const bool a_mn = (MODE == MODE_GRAD) && t.kind == KIND_DC;
      const bool b_mn = (MODE == MODE_GRAD);
      const int n = (MODE == MODE_GRAD) ? (PAIR ? pair_tile_n(a, t) : a.bn) : BN;
      const uint32_t idesc = idesc_bf16(PAIR ? 2 * BM : BM, n, a_mn, b_mn);
      // MN-major: 64-element groups kBK rows apart, a K=16 step is 16 rows;
      // K-major: a K=16 step is 32 bytes of a 128-byte row, and each 64 of K
      // is a box of its own (BM rows of A further on)
      const uint32_t a_lbo = a_mn ? kBK * 128u : 16u, b_lbo = b_mn ? kBK * 128u : 16u;
      auto a_off = [&](int kk) -> uint64_t {
        return a_mn ? (2048u >> 4) * kk : ((kk >> 2) * (BM * 128u >> 4) + (kk & 3) * (32u >> 4));
      };
      // K-major B: BN rows per 64 of K (a pair's CTA holds 128 of them)
      auto b_off = [&](int kk) -> uint64_t {
        return b_mn ? (2048u >> 4) * kk : ((kk >> 2) * ((PAIR ? BN / 2 : BN) * 128u >> 4) + (kk & 3) * (32u >> 4));
      };
      if (!wait_bounded(&L.tmem_empty[acc], acc_phase ^ 1u, abort_flag, a.dev_err)) return false;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      bool any = false;
      if constexpr (PAIR && MODE == MODE_GRAD) {
        // a pair whose two tiles keep no K-block has no stage (see the producer)
        if (none_kept) {
          mbar_arrive(&L.tmem_full[acc]);
          mbar_arrive_cluster(mapa_shared(smem_u32(&L.tmem_full[acc]), 1));
          if (++acc == PAIR_ACCS) {
            acc = 0;
            acc_phase ^= 1u;
          }
          return true;
        }
      }
      // FWD / BWD_G: every K-block; GRAD: the producer's stage tags end the loop
      const int nk = MODE == MODE_GRAD ? 0 : (PAIR ? (kblocks_of<MODE>(a, dm, t) + 1) >> 1 : kblocks_of<MODE>(a, dm, t));
      for (int kb = 0;; ++kb) {
        if (MODE != MODE_GRAD && kb >= nk) break;
        if (!wait_bounded(&L.full[stage], phase, abort_flag, a.dev_err)) return false;
        tc_fence_after();
        int meta = 0;
        if constexpr (MODE == MODE_GRAD) {
          meta = *reinterpret_cast<volatile int*>(&L.stage_meta[stage]);
          if (meta & META_EMPTY) {
            mbar_arrive(&L.empty[stage]);  // hand the stage straight back (one CTA per tile only)
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
            break;
          }
        }
        const uint32_t sA = smem_u32(L.stages + stage * kStageBytes);
        const uint32_t sB = sA + kABytes;
        const uint64_t adesc = smem_desc_sw128(sA, a_lbo, 1024u);
        const uint64_t bdesc = smem_desc_sw128(sB, b_lbo, 1024u);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          if constexpr (PAIR) {
            mma_bf16_pair(d_tmem, adesc + a_off(kk), bdesc + b_off(kk), idesc, (any || kk > 0) ? 1u : 0u);
          } else {
            mma_bf16(d_tmem, adesc + a_off(kk), bdesc + b_off(kk), idesc, (any || kk > 0) ? 1u : 0u);
          }
        }
        any = true;
        issued_any = true;
        if constexpr (PAIR) {
          mma_commit_pair_both(&L.empty[stage]);  // frees the stage in both CTAs
        } else {
          mma_commit(&L.empty[stage]);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (MODE == MODE_GRAD && (meta & META_LAST)) break;
      }
      if (PAIR) {
        mma_commit_pair_both(&L.tmem_full[acc]);  // both CTAs' epilogues (pairs: every tile here has MMAs)
      } else if (any) {
        mma_commit(&L.tmem_full[acc]);
      } else {
        mbar_arrive(&L.tmem_full[acc]);  // nothing to wait for: the epilogue writes zeros
      }
      if (++acc == (PAIR ? PAIR_ACCS : 2)) {
        acc = 0;
        acc_phase ^= 1u;
      }
      return true;
    });
    if (!ok) break;
  }
  if (*abort_flag && issued_any) {
    if constexpr (PAIR) {
      mma_commit_pair_local(L.drain);
    } else {
      mma_commit(L.drain);  // fires once every MMA issued so far has finished
    }
    volatile int dummy = 0;
    wait_bounded(L.drain, 0, &dummy, nullptr);
  }
}

// ---------------------------------------------------------------- epilogues
struct EpiCtx {
  uint32_t taddr;  // TMEM address of this warp's lane quadrant, accumulator column 0
  int q;           // lane quadrant = tile rows 32q .. 32q + 31
  uint8_t* buf;    // this warp's 8 KiB staging area (two 4 KiB halves)
  int iter;        // tiles processed so far by this warp
  int last_buf;    // staging half read by the most recent bulk group (-1: none)
  int kept;        // BWD_G: filter tiles this thread found kept
};

// Before overwriting staging half b: if the most recent bulk group reads b,
// wait for every group; otherwise all but that most recent one (older groups
// may have used b).  Correct however many stores were skipped.
__device__ __forceinline__ void staging_acquire(EpiCtx& e, int b) {
  if (lane_id() == 0) {
    if (e.last_buf == b) {
      bulk_wait_read<0>();
    } else {
      bulk_wait_read<1>();
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void release_tmem(const SmemLayout& L, int acc) {
  tc_fence_before();
  __syncwarp();
  if (lane_id() == 0) {
    if (L.tmem_empty_lead) {  // CTA pairs: the even CTA's MMA thread waits for both CTAs
      mbar_arrive_cluster(L.tmem_empty_lead + 8u * static_cast<uint32_t>(acc));
    } else {
      mbar_arrive(&L.tmem_empty[acc]);
    }
  }
}

// FWD: fold a 128 x 256 logit tile into the running (max, sumexp) of each row.
struct FwdState {
  float run_m, run_s;
};

// Softcapped logits: a' = cap * tanh(a / cap), in place (tanhf: accurate to a
// few ulp, which the 1e-5 LSE bar needs).
__device__ __forceinline__ void softcap_chunk(uint32_t (&r)[32], float cap, float inv_cap) {
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(cap * tanhf(__uint_as_float(r[j]) * inv_cap));
}

__device__ __forceinline__ void fold_chunk(const uint32_t (&r)[32], int col0, int V, long long xr, float& run_m,
                                           float& run_s, float& tval, bool& tfound, float& chunk_max) {
  const int nvalid = min(32, V - col0);  // < 32 only in the last tile of a ragged vocabulary
  const long long rel = xr - col0;
  if (rel >= 0 && rel < nvalid) {  // the target column passes: capture its logit (rare)
    const int ri = static_cast<int>(rel);
    float tv = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) tv = (j == ri) ? __uint_as_float(r[j]) : tv;
    tval = tv;
    tfound = true;
  }
  // max of the raw logits; scaling by log2(e) afterwards gives the same value
  // (rounding is monotonic), so each element costs one max, one FMA, one exp2
  // and one add.
  float cmax = NEG_BIG;
  if (nvalid == 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) cmax = fmaxf(cmax, __uint_as_float(r[j]));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nvalid) cmax = fmaxf(cmax, __uint_as_float(r[j]));
  }
  chunk_max = fmaxf(chunk_max, cmax);
  const float nm = fmaxf(run_m, cmax * LOG2E);
  float s = run_s * ex2(run_m - nm);
  if (nvalid == 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) s += ex2(fmaf(__uint_as_float(r[j]), LOG2E, -nm));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nvalid) s += ex2(fmaf(__uint_as_float(r[j]), LOG2E, -nm));
  }
  run_s = s;
  run_m = nm;
}

template <bool CAP>
__device__ __forceinline__ void epi_fwd(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc,
                                        EpiCtx& e, FwdState& st) {
  const int row = t.m * BM + e.q * 32 + static_cast<int>(lane_id());
  const bool in_range = t.live && row < a.N;
  const long long xr = in_range ? static_cast<long long>(__ldg(a.x + row)) : -1ll;
  if (t.first) {
    st.run_m = NEG_BIG;
    st.run_s = 0.0f;
  }
  float tval = 0.0f;
  bool tfound = false;
  float tmax = NEG_BIG;  // unused here (the staging epilogue needs it)
  const int vt0 = t.n * BN;
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
  for (int c = 0; c < BN / 32; c += 2) {
    const int col0 = vt0 + 32 * c;
    if (col0 >= a.V) break;  // uniform across the warp
    uint32_t r0[32], r1[32];
    tmem_ld32(tbase + 32 * c, r0);
    tmem_ld32(tbase + 32 * (c + 1), r1);
    tmem_ld_wait();
    if constexpr (CAP) {
      softcap_chunk(r0, a.softcap, a.inv_softcap);
      softcap_chunk(r1, a.softcap, a.inv_softcap);
    }
    fold_chunk(r0, col0, a.V, xr, st.run_m, st.run_s, tval, tfound, tmax);
    if (col0 + 32 < a.V) fold_chunk(r1, col0 + 32, a.V, xr, st.run_m, st.run_s, tval, tfound, tmax);
  }
  release_tmem(L, acc);
  if (in_range && tfound) a.tgt[row] = tval;
  if (t.last && in_range) {
    a.part_m[static_cast<size_t>(t.split) * a.N + row] = st.run_m;
    a.part_s[static_cast<size_t>(t.split) * a.N + row] = st.run_s;
  }
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// FWD_STAGE: the fold of epi_fwd; each 32-column chunk is also staged as
// fp16 (logit minus the row's max over the chunk: <= 0, and fp16 keeps about
// 11 bits of it, so the entries within a few units of the max -- the ones
// that carry softmax mass -- keep an absolute error near 2^-12 per unit) in
// 64-column boxes (128-byte swizzle), and the chunk max goes to mtile.  One
// pass over TMEM.
template <bool CAP>
__device__ __forceinline__ void epi_fwd_stage(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc,
                                              EpiCtx& e, FwdState& st) {
  const uint32_t lane = lane_id();
  const int row0 = t.m * BM + e.q * 32;  // first row of this warp's quadrant
  const int row = row0 + static_cast<int>(lane);
  const bool in_range = t.live && row < a.N;
  const bool store = t.live && row0 < a.N;  // uniform: the box starts inside the staging rows
  const long long xr = in_range ? static_cast<long long>(__ldg(a.x + row)) : -1ll;
  if (t.first) {
    st.run_m = NEG_BIG;
    st.run_s = 0.0f;
  }
  float tval = 0.0f;
  bool tfound = false;
  const int vt0 = t.n * BN;
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
  for (int c = 0; c < BN / 32; c += 2) {
    const int col0 = vt0 + 32 * c;
    if (col0 >= a.V) break;  // uniform across the warp
    uint32_t r0[32], r1[32];
    tmem_ld32(tbase + 32 * c, r0);
    tmem_ld32(tbase + 32 * (c + 1), r1);
    tmem_ld_wait();
    if constexpr (CAP) {
      softcap_chunk(r0, a.softcap, a.inv_softcap);
      softcap_chunk(r1, a.softcap, a.inv_softcap);
    }
    float m0 = NEG_BIG, m1 = NEG_BIG;
    fold_chunk(r0, col0, a.V, xr, st.run_m, st.run_s, tval, tfound, m0);
    const bool has1 = col0 + 32 < a.V;
    if (has1) fold_chunk(r1, col0 + 32, a.V, xr, st.run_m, st.run_s, tval, tfound, m1);
    if (store) {
      const int b = (c >> 1) & 1;
      uint8_t* buf = e.buf + b * 4096;
      staging_acquire(e, b);
      const uint32_t sb = smem_u32(buf);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        st_shared_v4(sb + swz(lane, u),
                     pack_f16x2(__uint_as_float(r0[8 * u + 0]) - m0, __uint_as_float(r0[8 * u + 1]) - m0),
                     pack_f16x2(__uint_as_float(r0[8 * u + 2]) - m0, __uint_as_float(r0[8 * u + 3]) - m0),
                     pack_f16x2(__uint_as_float(r0[8 * u + 4]) - m0, __uint_as_float(r0[8 * u + 5]) - m0),
                     pack_f16x2(__uint_as_float(r0[8 * u + 6]) - m0, __uint_as_float(r0[8 * u + 7]) - m0));
        st_shared_v4(sb + swz(lane, 4 + u),
                     pack_f16x2(__uint_as_float(r1[8 * u + 0]) - m1, __uint_as_float(r1[8 * u + 1]) - m1),
                     pack_f16x2(__uint_as_float(r1[8 * u + 2]) - m1, __uint_as_float(r1[8 * u + 3]) - m1),
                     pack_f16x2(__uint_as_float(r1[8 * u + 4]) - m1, __uint_as_float(r1[8 * u + 5]) - m1),
                     pack_f16x2(__uint_as_float(r1[8 * u + 6]) - m1, __uint_as_float(r1[8 * u + 7]) - m1));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&a.tmOut, buf, col0, row0);
        bulk_commit();
      }
      e.last_buf = b;
    }
    if (in_range) {
      a.mtile[static_cast<size_t>(col0 >> 5) * a.N + row] = m0;
      if (has1) a.mtile[static_cast<size_t>((col0 >> 5) + 1) * a.N + row] = m1;
    }
  }
  release_tmem(L, acc);
  if (in_range) {
    if (tfound) a.tgt[row] = tval;
    if (t.last) {
      a.part_m[static_cast<size_t>(t.split) * a.N + row] = st.run_m;
      a.part_s[static_cast<size_t>(t.split) * a.N + row] = st.run_s;
    }
  }
}

// BWD_G: G = exp(A - LSE) - onehot, filter vote per 128-column half, bf16 store.
template <bool CAP>
__device__ __forceinline__ bool epi_bwd_g(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc,
                                          EpiCtx& e) {
  const uint32_t lane = lane_id();
  const int row = t.m * BM + e.q * 32 + static_cast<int>(lane);
  // Rows that take no part (ignored, out-of-range target, beyond N) get
  // LSE = +inf: every exp2 is then exactly 0 and no one-hot is subtracted, so
  // their G is 0 without a per-element test.
  long long xr = -1;
  float lse2 = INFINITY, w = 0.0f;
  if (t.live && row < a.N) {
    const long long xi = static_cast<long long>(__ldg(a.x + row));
    if ((xi != a.ignore_index) && xi >= 0 && xi < a.V) {
      xr = xi;
      lse2 = __ldg(a.lse + row) * LOG2E;
      if (a.reduction == CCE_RED_NONE) {
        w = __ldg(a.grad_out + row);
      } else if (a.reduction == CCE_RED_SUM) {
        w = __ldg(a.grad_out);
      } else {
        w = __ldg(a.grad_out) / static_cast<float>(max(__ldg(a.count), 1));
      }
    }
  }
  const int vt0 = a.chunk_v0 + t.n * BN;  // global vocabulary column of the tile
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
  const uint32_t sbuf = smem_u32(e.buf);
  const int par = e.iter & 1;
  bool ok = true;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    if (lane == 0) bulk_wait_read<0>();  // staging buffer free again
    __syncwarp();
    e.last_buf = -1;
    float amax = 0.0f;  // largest unscaled |G| this thread saw in the half
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c = 4 * h + cc;
      const int col0 = vt0 + 32 * c;
      uint32_t r[32];
      tmem_ld32(tbase + 32 * c, r);
      tmem_ld_wait();
      float g[32];
      float slope[32];  // d(capped logit) / d(logit); 1 without a cap
      if constexpr (CAP) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float th = tanhf(__uint_as_float(r[j]) * a.inv_softcap);
          slope[j] = 1.0f - th * th;
          g[j] = ex2(fmaf(a.softcap * th, LOG2E, -lse2));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          slope[j] = 1.0f;
          g[j] = ex2(fmaf(__uint_as_float(r[j]), LOG2E, -lse2));
        }
      }
      if (col0 + 32 > a.V) {  // ragged last tile: columns past V are zero (uniform branch)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j >= a.V) g[j] = 0.0f;
      }
      const long long rel = xr - col0;
      if (rel >= 0 && rel < 32) {  // the target column: subtract the one-hot (rare)
        const int ri = static_cast<int>(rel);
#pragma unroll
        for (int j = 0; j < 32; ++j) g[j] = (j == ri) ? g[j] - 1.0f : g[j];
      }
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        amax = fmaxf(amax, fmaxf(fabsf(g[j]), fabsf(g[j + 1])));  // the filter tests |G| before the slope
        pk[j / 2] = pack_bf16x2(g[j] * slope[j] * w, g[j + 1] * slope[j + 1] * w);
      }
      const uint32_t box = sbuf + static_cast<uint32_t>((cc >> 1) * 4096);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        st_shared_v4(box + swz(lane, (cc & 1) * 4 + u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
    }
    const bool surv = amax >= a.eps;
    if (h == 1) release_tmem(L, acc);
    // Tile-wide vote: every epilogue warp contributes, one mbarrier phase per tile.
    const int any = __any_sync(0xffffffffu, surv) ? 1 : 0;
    int* fl = L.flags + (par * 2 + h) * 4;
    if (lane == 0) {
      fl[e.q] = any;
      mbar_arrive(&L.vote[h]);
    }
    if (!warp_wait_bounded(&L.vote[h], static_cast<uint32_t>(par), L.abort_flag, a.dev_err)) {
      ok = false;
      break;
    }
    int kv = 0;
    if (lane == 0) kv = fl[0] | fl[1] | fl[2] | fl[3];  // lane 0 performed the acquiring wait
    const bool keep = __shfl_sync(0xffffffffu, kv, 0) != 0;
    // A skipped tile's G is still needed when one of the outputs is unfiltered.
    if (keep || !(a.filter_de && a.filter_dc)) {
      fence_proxy_async_smem();
      __syncwarp();
      const int gx = t.n * BN + 128 * h;  // column inside the chunk buffer
      const int gy = t.m * BM + e.q * 32;
      if (lane == 0 && t.live && gy < a.N) {  // no store starts outside the buffer
        tma_store_2d(&a.tmOut, e.buf, gx, gy);
        tma_store_2d(&a.tmOut, e.buf + 4096, gx + 64, gy);
        bulk_commit();
      }
    }
    if (e.q == 0 && lane == 0 && t.live) {
      const int vt128 = (vt0 >> 7) + h;
      if (vt128 < a.bm_ld) {
        a.bitmap[static_cast<size_t>(t.m) * a.bm_ld + vt128] = keep ? 1 : 0;
        a.bitmapT[static_cast<size_t>(vt128) * a.n_blocks + t.m] = keep ? 1 : 0;
        e.kept += keep ? 1 : 0;
      }
    }
  }
  return ok;
}

// An empty output tile's boxes: staging half 0 is zeroed once (`bytes` of
// it: one 32-row box) and lane 0 stores all nbox boxes of 32 columns from
// it, x0 + 32 j, one bulk group, instead of staging and waiting box by box.
// Sparse survival leaves most tiles of a chunk empty, and their zeros are
// most of what such a launch writes.
__device__ __forceinline__ void zero_boxes(const CUtensorMap* tm, EpiCtx& e, int x0, int gy, int nbox, int bytes,
                                           bool reduce) {
  const uint32_t lane = lane_id();
  staging_acquire(e, 0);
  const uint32_t sb = smem_u32(e.buf);
  for (int o = static_cast<int>(lane) * 16; o < bytes; o += 32 * 16) st_shared_v4(sb + o, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    for (int j = 0; j < nbox; ++j) {
      if (reduce) {
        tma_reduce_add_2d(tm, e.buf, x0 + 32 * j, gy);
      } else {
        tma_store_2d(tm, e.buf, x0 + 32 * j, gy);
      }
    }
    bulk_commit();
  }
  e.last_buf = 0;
}

// fp32 output rows gy .. gy + 31 of tensor map tm, columns x0 .. x0 + 32 * nbox - 1:
// 32-column boxes (128-byte swizzle) from TMEM, or zeros when the tile is
// empty; stored, or reduce-added by TMA.
__device__ __forceinline__ void store_f32_boxes(const CUtensorMap* tm, EpiCtx& e, uint32_t tbase, int x0, int gy,
                                                int nbox, bool empty, bool reduce) {
  const uint32_t lane = lane_id();
  if (empty) {  // every box from one zeroed staging half, in one bulk group
    if (nbox > 0) zero_boxes(tm, e, x0, gy, nbox, 4096, reduce);
    return;
  }
#pragma unroll 1
  for (int j = 0; j < nbox; ++j) {
    const int b = j & 1;
    uint8_t* buf = e.buf + b * 4096;
    staging_acquire(e, b);
    const uint32_t sb = smem_u32(buf);
    if (!empty) {
      uint32_t r[32];
      tmem_ld32(tbase + 32 * j, r);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 8; ++u) st_shared_v4(sb + swz(lane, u), r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) st_shared_v4(sb + swz(lane, u), 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (reduce) {
        tma_reduce_add_2d(tm, buf, x0 + 32 * j, gy);
      } else {
        tma_store_2d(tm, buf, x0 + 32 * j, gy);
      }
      bulk_commit();
    }
    e.last_buf = b;
  }
}

// GRAD, KIND_DC: bf16 output tile, rows = vocabulary (c_row0 + 128m ...),
// cols = D tile of width bn, stored in 32-column boxes (64-byte swizzle).
__device__ __forceinline__ void epi_dc(const GemmArgs& a, const Dims& dm, const SmemLayout& L, const Tile& t,
                                       int acc, EpiCtx& e) {
  const uint32_t lane = lane_id();
  const bool empty = tile_empty(a, dm, t);
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
  const int ly = t.m * BM + e.q * 32;  // first row of the box within the chunk
  const int gy = a.c_row0 + ly;        // ... in the dC tensor map
  const int x0 = t.n * a.bn;
  if (a.dc_f32) {  // fp32 rows through tmOut (the single call accumulates dC over token chunks)
    if (empty && a.dc_reduce) {
      release_tmem(L, acc);
      return;
    }
    const int nb = (ly < a.chunk_w) ? min(a.bn / 32, (a.D - x0 + 31) / 32) : 0;
    store_f32_boxes(&a.tmOut, e, tbase, x0, gy, nb, empty, a.dc_reduce != 0);
    release_tmem(L, acc);
    return;
  }
  if (a.dc_rows) {
    // Sorted vocabulary: row ly + lane of the chunk is token dc_rows[ly + lane];
    // each lane writes its own row of dC directly, 16 bytes at a time.
    const int lr = ly + static_cast<int>(lane);
    const bool row_ok = lr < a.chunk_w;
    const size_t grow = row_ok ? static_cast<size_t>(__ldg(a.dc_rows + lr)) : 0;
    if (empty) {
      // zeros need no TMEM lane of their own: the warp writes one row at a
      // time, 16 bytes a lane, each store a contiguous run of the row
      release_tmem(L, acc);
      const int rows = min(32, a.chunk_w - ly);
      const bool col_ok = x0 + 8 * static_cast<int>(lane) < min(a.D, x0 + a.bn);
#pragma unroll 4
      for (int i = 0; i < rows; ++i) {
        const size_t gi = __shfl_sync(0xffffffffu, grow, i);
        if (col_ok) reinterpret_cast<uint4*>(a.dC_out + gi * a.D + x0)[lane] = make_uint4(0u, 0u, 0u, 0u);
      }
      return;
    }
    uint4* dst = reinterpret_cast<uint4*>(a.dC_out + grow * a.D + x0);
    const int nb = (ly < a.chunk_w) ? min(a.bn / 32, (a.D - x0 + 31) / 32) : 0;
#pragma unroll 1
    for (int j = 0; j < nb; ++j) {
      uint32_t r[32];
      if (!empty) {
        tmem_ld32(tbase + 32 * j, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = 0u;
      }
      if (row_ok) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (x0 + 32 * j + 8 * u < a.D)
            dst[4 * j + u] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * u + 0]), __uint_as_float(r[8 * u + 1])),
                                        pack_bf16x2(__uint_as_float(r[8 * u + 2]), __uint_as_float(r[8 * u + 3])),
                                        pack_bf16x2(__uint_as_float(r[8 * u + 4]), __uint_as_float(r[8 * u + 5])),
                                        pack_bf16x2(__uint_as_float(r[8 * u + 6]), __uint_as_float(r[8 * u + 7])));
        }
      }
    }
    release_tmem(L, acc);
    return;
  }
  // boxes that start inside the chunk and dC (no store may start outside the tensor)
  const int nbox = (ly < a.chunk_w) ? min(a.bn / 32, (a.D - x0 + 31) / 32) : 0;
  // dc_acc (single call, last token chunk): add the fp32 sum of the earlier
  // chunks, read by each lane for its own row, before rounding to bf16
  const int arow = ly + static_cast<int>(lane);
  const float* accrow = (a.dc_acc && arow < a.chunk_w) ? a.dc_acc + static_cast<size_t>(a.c_row0 + arow) * a.D : nullptr;
  if (empty && !a.dc_acc) {
    if (nbox > 0) zero_boxes(&a.tmOut, e, x0, gy, nbox, 2048, false);
    release_tmem(L, acc);
    return;
  }
#pragma unroll 1
  for (int j = 0; j < nbox; ++j) {
    const int b = j & 1;
    uint8_t* buf = e.buf + b * 4096;
    staging_acquire(e, b);
    const uint32_t sb = smem_u32(buf);
    if (!empty || a.dc_acc) {
      uint32_t r[32];
      if (!empty) {
        tmem_ld32(tbase + 32 * j, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = 0u;
      }
      if (accrow) {
        const int c0 = x0 + 32 * j;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (c0 + 4 * u < a.D) {  // D % 8 == 0: groups of four lie wholly inside or outside
            const float4 v = *reinterpret_cast<const float4*>(accrow + c0 + 4 * u);
            r[4 * u + 0] = __float_as_uint(__uint_as_float(r[4 * u + 0]) + v.x);
            r[4 * u + 1] = __float_as_uint(__uint_as_float(r[4 * u + 1]) + v.y);
            r[4 * u + 2] = __float_as_uint(__uint_as_float(r[4 * u + 2]) + v.z);
            r[4 * u + 3] = __float_as_uint(__uint_as_float(r[4 * u + 3]) + v.w);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        st_shared_v4(sb + swz64(lane, u), pack_bf16x2(__uint_as_float(r[8 * u + 0]), __uint_as_float(r[8 * u + 1])),
                     pack_bf16x2(__uint_as_float(r[8 * u + 2]), __uint_as_float(r[8 * u + 3])),
                     pack_bf16x2(__uint_as_float(r[8 * u + 4]), __uint_as_float(r[8 * u + 5])),
                     pack_bf16x2(__uint_as_float(r[8 * u + 6]), __uint_as_float(r[8 * u + 7])));
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) st_shared_v4(sb + swz64(lane, u), 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&a.tmOut, buf, x0 + 32 * j, gy);
      bulk_commit();
    }
    e.last_buf = b;
  }
  release_tmem(L, acc);
}

// GRAD, KIND_DE: fp32 output tile, rows = tokens, cols = D tile; store (first
// chunk) or reduce-add, in 32-column boxes (128-byte swizzle).  With K ranges
// (single call) range s stores to its own slab of rows.
__device__ __forceinline__ void epi_de(const GemmArgs& a, const Dims& dm, const SmemLayout& L, const Tile& t,
                                       int acc, EpiCtx& e) {
  const bool empty = tile_empty(a, dm, t);
  if (empty && !a.first_chunk) {  // adding zero: nothing to do
    release_tmem(L, acc);
    return;
  }
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
  const int ly = t.m * BM + e.q * 32;  // row within the launch's rows
  const int gy = (a.de_splits > 1 ? t.split * a.de_slab : 0) + a.de_row0 + ly;
  const int x0 = t.n * a.bn;
  // boxes that start inside dE (no store or reduce may start outside the tensor)
  const int nbox = (ly < a.N) ? min(a.bn / 32, (a.D - x0 + 31) / 32) : 0;
  store_f32_boxes(&a.tmOut2, e, tbase, x0, gy, nbox, empty, !a.first_chunk);
  release_tmem(L, acc);
}

template <int MODE, bool CAP, bool PAIR = false>
__device__ __forceinline__ void epilogue_loop(const GemmArgs& a, const SmemLayout& L, uint32_t tmem_base,
                                              int warp) {
  EpiCtx e;
  e.q = warp & 3;
  e.taddr = tmem_base + (static_cast<uint32_t>(e.q * 32) << 16);
  e.buf = L.epi + (warp - 2) * EPI_WARP_BYTES;
  e.iter = 0;
  e.last_buf = -1;
  e.kept = 0;
  FwdState st{NEG_BIG, 0.0f};
  int acc = 0;
  uint32_t acc_phase = 0;
  const Dims dm = dims_of<MODE, PAIR>(a);
  for (int k = 0;; ++k) {
    int item = 0;
    if (lane_id() == 0) item = ring_take_any<MODE, PAIR>(L, k, a);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item < 0) break;
    if (PAIR && MODE == MODE_GRAD) item >>= 2;  // the entry's low bits are for the MMA and producers
    const bool ok = for_each_tile_of_item<MODE, PAIR>(a, dm, item, [&](const Tile& t) -> bool {
      if (!warp_wait_bounded(&L.tmem_full[acc], acc_phase, L.abort_flag, a.dev_err)) return false;
      tc_fence_after();
      bool r = true;
      if (MODE == MODE_GRAD && !t.live) {
        release_tmem(L, acc);  // the missing block of the last pair: nothing to write
      } else if constexpr (MODE == MODE_FWD) {
        epi_fwd<CAP>(a, L, t, acc, e, st);
      } else if constexpr (MODE == MODE_FWD_STAGE) {
        epi_fwd_stage<CAP>(a, L, t, acc, e, st);
      } else if constexpr (MODE == MODE_BWD_G) {
        r = epi_bwd_g<CAP>(a, L, t, acc, e);
      } else {
        if (t.kind == KIND_DC) {
          epi_dc(a, dm, L, t, acc, e);
        } else {
          epi_de(a, dm, L, t, acc, e);
        }
      }
      ++e.iter;
      if (++acc == (PAIR ? PAIR_ACCS : 2)) {
        acc = 0;
        acc_phase ^= 1u;
      }
      return r;
    });
    if (!ok) break;
  }
  // BWD_G: one add per thread that wrote survival bytes, in a slot of its own
  if (MODE == MODE_BWD_G && a.kept_tiles && e.kept) atomicAdd(a.kept_tiles + blockIdx.x % KEPT_SLOTS, e.kept);
  if (lane_id() == 0) bulk_wait_all();
  __syncwarp();
}

// GRAD with the filter on: CTA pairs run the union of two tiles' K-blocks, so
// they pay off when nearly every filter tile is kept; when many are skipped,
// one CTA per tile does less work.  Both are launched; this says whether the
// launch with this kernel's layout is the one that runs (at least 80% of the
// chunk's filter tiles kept: pairs).
template <int MODE, bool PAIR>
__device__ __forceinline__ bool grad_launch_runs(const GemmArgs& a) {
  if (MODE != MODE_GRAD || a.grad_path < 0) return true;
  const Dims dm = dims_of<MODE, PAIR>(a);
  const long long total = static_cast<long long>(dm.nb) * ((a.chunk_w + FILTER_TILE - 1) / FILTER_TILE);
  // written by the previous launch: plain loads, all in flight at once
  int v[KEPT_SLOTS];
#pragma unroll
  for (int i = 0; i < KEPT_SLOTS; ++i) v[i] = __ldcg(a.kept_tiles + i);
  long long kept = 0;
#pragma unroll
  for (int i = 0; i < KEPT_SLOTS; ++i) kept += v[i];
  const bool pairs = 5 * kept >= 4 * total;
  return pairs == (a.grad_path == 1);
}

// CAP: logit softcapping in the FWD / BWD_G epilogues (a separate
// instantiation, so the common path carries none of its registers).
// PAIR: launched as clusters of two CTAs sharing each MMA (M = 256).
template <int MODE, bool CAP = false, bool PAIR = false>
__global__ void __launch_bounds__(NUM_THREADS, 1) cce_gemm_kernel(const __grid_constant__ GemmArgs a) {
  if (MODE == MODE_GRAD && a.grad_path >= 0) {  // one thread reads the counts; every CTA decides alike
    __shared__ int runs;
    if (threadIdx.x == 0) runs = grad_launch_runs<MODE, PAIR>(a) ? 1 : 0;
    __syncthreads();
    if (!runs) return;  // the other launch does the work
  }
  extern __shared__ uint8_t smem_raw[];
  SmemLayout L = carve_smem(smem_raw);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const bool lead = !PAIR || cluster_ctarank() == 0;
  if (PAIR) L.tmem_empty_lead = mapa_shared(smem_u32(&L.tmem_empty[0]), 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < Pipe<MODE, PAIR>::kStages; ++s) {
      mbar_init(&L.full[s], 1);
      mbar_init(&L.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&L.tmem_full[i], 1);
      // pairs: the even CTA's accumulators are released by both CTAs' epilogues
      mbar_init(&L.tmem_empty[i], PAIR ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS);
      mbar_init(&L.vote[i], NUM_EPI_WARPS);
    }
    for (int i = 0; i < RING; ++i) {
      mbar_init(&L.ring_full[i], 1);
      // the MMA thread (the odd CTA of a pair has none at work) and every
      // epilogue warp; gradient-GEMM pairs: the even CTA's barrier counts the
      // consumers of both CTAs (its producer, MMA thread and epilogue warps,
      // the odd CTA's producer and epilogue warps)
      mbar_init(&L.ring_empty[i],
                (PAIR && MODE == MODE_GRAD) ? 2 * (1 + NUM_EPI_WARPS) + 1 : (lead ? 1 : 0) + NUM_EPI_WARPS);
    }
    for (int i = 0; i < WORD_SLOTS; ++i) mbar_init(&L.words_free[i], 2);  // both producers of a pair
    mbar_init(L.drain, 1);
    *L.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&a.tmA);
    tma_prefetch_desc(&a.tmB);
    if (MODE != MODE_FWD) tma_prefetch_desc(&a.tmOut);
    if (MODE == MODE_GRAD) {
      tma_prefetch_desc(&a.tmA2);
      tma_prefetch_desc(&a.tmB2);
      tma_prefetch_desc(&a.tmOut2);
      if (PAIR) tma_prefetch_desc(&a.tmZ);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // one warp of each CTA of the pair, together
      tmem_alloc_pair(L.tmem_base, PAIR_TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(L.tmem_base, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before any copy or arrive reaches them
  tc_fence_after();
  const uint32_t tmem_base = *L.tmem_base;

  if (warp == 0) {
    if (lane_id() == 0) {
      if constexpr (PAIR && MODE == MODE_GRAD) {
        producer_loop_grad_pair(a, L);
      } else {
        producer_loop<MODE, PAIR>(a, L);
      }
    }
  } else if (warp == 1) {
    if (lane_id() == 0) mma_loop<MODE, PAIR>(a, L, tmem_base);
  } else if (warp < 2 + NUM_EPI_WARPS) {
    epilogue_loop<MODE, CAP, PAIR>(a, L, tmem_base, warp);
  } else if constexpr (PAIR && MODE == MODE_GRAD) {
    if (lane_id() == 0 && cluster_ctarank() == 0) scheduler_loop_grad_pair(a, L);
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) {
      tmem_dealloc_pair(tmem_base, PAIR_TMEM_COLS);
    } else {
      tmem_dealloc(tmem_base, TMEM_COLS);
    }
  }
}

}  // namespace cce
