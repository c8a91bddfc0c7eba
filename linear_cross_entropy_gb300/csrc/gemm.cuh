// Persistent, warp-specialised tcgen05 GEMM with four epilogues -- the four
// dense contractions of Cut Cross-Entropy on one template:
//
//   MODE_FWD   A = E [N,D] (K-major), B = C [V,D] (K-major).  Epilogue: each
//              row folds its logit tile into a running (max, sumexp) over the
//              CTA's vocabulary split and captures the target logit when its
//              column passes ("Cut Your Losses in Large-Vocabulary Language
//              Models", "Memory-Efficient Linear-Log-Sum-Exp, Forward Pass
//              (Algorithm 2)" and "Memory-Efficient Indexed Matrix
//              Multiplication (Algorithm 1)"; the online fold of the
//              "cut-cross-entropy" card's "Method").  Writes per-(row, split)
//              partials; a separate kernel combines them in a fixed order.
//   MODE_BWD_G Same operands over one vocabulary chunk.  Epilogue: G =
//              exp(A - LSE) - onehot(x), the tile filter (skip when every
//              unscaled |G| < eps, decided by warp votes and a shared-memory
//              flag), then G * w rounded to bf16 and stored to the chunk
//              buffer for surviving 128x128 tiles only ("The Combined Backward
//              Pass (Algorithm 4)", "Gradient Filtering").
//   MODE_DC    dC[chunk rows] = G_chunk^T E: A = G_chunk (MN-major), B = E
//              (MN-major), K = tokens; K-blocks of skipped tiles are not
//              loaded and issue no MMA.  Each CTA owns its dC rows: written
//              once in bf16, no atomics.
//   MODE_DE    dE_acc (+)= G_chunk C_chunk: A = G_chunk (K-major), B = C
//              (MN-major), K = chunk columns; fp32 tiles stored (first chunk)
//              or reduce-added by TMA (later chunks) -- one writer per tile
//              per chunk, chunks in stream order, so the result is
//              deterministic.
//
// Roles (192 threads): warp 0 lane 0 issues TMA loads into a 4-stage ring;
// warp 1 owns TMEM (512 columns = two 128x256 fp32 accumulators) and lane 0
// issues tcgen05.mma; warps 2..5 are the epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31, i.e. tile rows).  The accumulator is double-buffered so the
// epilogue of one tile overlaps the MMAs of the next.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_args.h"
#include "ptx.cuh"

namespace cce {

struct Tile {
  int m;      // A-row block (128)
  int n;      // B-row block (256) or output column block
  int split;  // FWD
  bool first, last;  // FWD: first / last tile of a (row block, split) unit
};

// The tile sequence of this CTA; every role walks the same sequence.
template <int MODE, typename F>
__device__ __forceinline__ void for_each_tile(const GemmArgs& a, F&& f) {
  if constexpr (MODE == MODE_FWD) {
    const int units = a.n_blocks * a.splits;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int m = u % a.n_blocks, s = u / a.n_blocks;
      const int t0 = static_cast<int>(static_cast<long long>(s) * a.v_tiles / a.splits);
      const int t1 = static_cast<int>(static_cast<long long>(s + 1) * a.v_tiles / a.splits);
      for (int t = t0; t < t1; ++t) {
        if (!f(Tile{m, t, s, t == t0, t == t1 - 1})) return;
      }
    }
  } else if constexpr (MODE == MODE_BWD_G) {
    // Grouped raster: groups of group_n token blocks; inside a group the
    // token block varies fastest, then the vocabulary tile.  CTAs running at
    // the same time share a few C tiles and a group's E rows stay in L2.
    const int total = a.n_blocks * a.v_tiles;
    const int per_group = a.group_n * a.v_tiles;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      const int g = i / per_group, j = i - g * per_group;
      const int gn = min(a.group_n, a.n_blocks - g * a.group_n);
      if (!f(Tile{g * a.group_n + j % gn, j / gn, 0, true, true})) return;
    }
  } else {
    const int total = a.m_tiles * a.n_tiles;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      if (!f(Tile{i / a.n_tiles, i % a.n_tiles, 0, true, true})) return;
    }
  }
}

// Is K-block kb of tile t skipped by the filter?  (DC: K = tokens; DE: K =
// chunk columns.)  FWD and BWD_G never skip.
template <int MODE>
__device__ __forceinline__ bool kblock_skipped(const GemmArgs& a, const Tile& t, int kb) {
  if constexpr (MODE == MODE_DC) {  // contiguous along K: L1 hits
    return __ldg(a.bitmapT + static_cast<size_t>((a.chunk_v0 >> 7) + t.m) * a.n_blocks + (kb >> 1)) == 0;
  } else if constexpr (MODE == MODE_DE) {
    return __ldg(a.bitmap + static_cast<size_t>(t.m) * a.bm_ld + (a.chunk_v0 >> 7) + (kb >> 1)) == 0;
  } else {
    return false;
  }
}

// Warp-wide: does the output tile have no surviving K-block at all?
template <int MODE>
__device__ __forceinline__ bool tile_empty(const GemmArgs& a, const Tile& t) {
  int any = 0;
  if constexpr (MODE == MODE_DC) {
    const uint8_t* row = a.bitmapT + static_cast<size_t>((a.chunk_v0 >> 7) + t.m) * a.n_blocks;
    for (int r = lane_id(); r < a.n_blocks; r += 32) any |= __ldg(row + r);
  } else if constexpr (MODE == MODE_DE) {
    const int ncols = (a.chunk_w + FILTER_TILE - 1) / FILTER_TILE;
    const uint8_t* row = a.bitmap + static_cast<size_t>(t.m) * a.bm_ld + (a.chunk_v0 >> 7);
    for (int j = lane_id(); j < ncols; j += 32) any |= __ldg(row + j);
  } else {
    any = 1;
  }
  return __any_sync(0xffffffffu, any) == 0;
}

__device__ __forceinline__ float ex2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

struct SmemLayout {
  uint8_t* stages;
  uint8_t* epi;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tmem_full;
  uint64_t* tmem_empty;
  uint64_t* vote;
  uint64_t* drain;
  uint32_t* tmem_base;
  int* abort_flag;
  int* flags;  // [2 parity][2 half][4 warps]
};

__device__ __forceinline__ SmemLayout carve_smem(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.stages = base;
  L.epi = base + STAGES * STAGE_BYTES;
  uint8_t* b = L.epi + NUM_EPI_WARPS * EPI_WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(b);
  L.full = bars;                  // STAGES
  L.empty = bars + STAGES;        // STAGES
  L.tmem_full = bars + 2 * STAGES;      // 2
  L.tmem_empty = bars + 2 * STAGES + 2;  // 2
  L.vote = bars + 2 * STAGES + 4;        // 2
  L.drain = bars + 2 * STAGES + 6;       // 1
  uint8_t* tail = reinterpret_cast<uint8_t*>(bars + 2 * STAGES + 7);
  L.tmem_base = reinterpret_cast<uint32_t*>(tail);
  L.abort_flag = reinterpret_cast<int*>(tail + 4);
  L.flags = reinterpret_cast<int*>(tail + 8);  // 16 ints
  return L;
}

// ---------------------------------------------------------------- producer
template <int MODE>
__device__ __forceinline__ void producer_loop(const GemmArgs& a, const SmemLayout& L) {
  volatile int* abort_flag = L.abort_flag;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued_mask = 0, issued_par = 0;  // per stage: ever issued, parity of last issue
  for_each_tile<MODE>(a, [&](const Tile& t) -> bool {
    for (int kb = 0; kb < a.k_blocks; ++kb) {
      if (kblock_skipped<MODE>(a, t, kb)) continue;
      if (!wait_bounded(&L.empty[stage], phase ^ 1u, abort_flag, a.dev_err)) return false;
      uint8_t* sA = L.stages + stage * STAGE_BYTES;
      uint8_t* sB = sA + A_STAGE_BYTES;
      mbar_arrive_expect_tx(&L.full[stage], STAGE_BYTES);
      const int k0 = kb * BK;
      if constexpr (MODE == MODE_FWD || MODE == MODE_BWD_G) {
        tma_load_2d(&a.tmA, &L.full[stage], sA, k0, t.m * BM);
        tma_load_2d(&a.tmB, &L.full[stage], sB, k0, a.chunk_v0 + t.n * BN);
      } else if constexpr (MODE == MODE_DC) {
        for (int j = 0; j < BM / 64; ++j) tma_load_2d(&a.tmA, &L.full[stage], sA + j * 8192, t.m * BM + j * 64, k0);
        for (int j = 0; j < BN / 64; ++j) tma_load_2d(&a.tmB, &L.full[stage], sB + j * 8192, t.n * BN + j * 64, k0);
      } else {  // MODE_DE
        tma_load_2d(&a.tmA, &L.full[stage], sA, k0, t.m * BM);
        for (int j = 0; j < BN / 64; ++j)
          tma_load_2d(&a.tmB, &L.full[stage], sB + j * 8192, t.n * BN + j * 64, a.chunk_v0 + k0);
      }
      issued_mask |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    return true;
  });
  if (*abort_flag) {
    // Let every copy this thread issued land before the CTA exits.
    for (int s = 0; s < STAGES; ++s) {
      if (issued_mask & (1u << s)) {
        volatile int dummy = 0;
        wait_bounded(&L.full[s], (issued_par >> s) & 1u, &dummy, nullptr);
      }
    }
  }
}

// --------------------------------------------------------------------- MMA
template <int MODE>
__device__ __forceinline__ void mma_loop(const GemmArgs& a, const SmemLayout& L, uint32_t tmem_base) {
  constexpr bool A_MN = (MODE == MODE_DC);
  constexpr bool B_MN = (MODE == MODE_DC || MODE == MODE_DE);
  constexpr uint32_t IDESC = idesc_bf16(BM, BN, A_MN, B_MN);
  constexpr uint32_t A_LBO = A_MN ? 8192u : 16u;
  constexpr uint32_t B_LBO = B_MN ? 8192u : 16u;
  constexpr uint64_t A_KSTEP = A_MN ? (2048u >> 4) : (32u >> 4);  // one K=16 step, encoded
  constexpr uint64_t B_KSTEP = B_MN ? (2048u >> 4) : (32u >> 4);
  volatile int* abort_flag = L.abort_flag;
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool issued_any = false;
  for_each_tile<MODE>(a, [&](const Tile& t) -> bool {
    if (!wait_bounded(&L.tmem_empty[acc], acc_phase ^ 1u, abort_flag, a.dev_err)) return false;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
    bool any = false;
    for (int kb = 0; kb < a.k_blocks; ++kb) {
      if (kblock_skipped<MODE>(a, t, kb)) continue;
      if (!wait_bounded(&L.full[stage], phase, abort_flag, a.dev_err)) return false;
      tc_fence_after();
      const uint32_t sA = smem_u32(L.stages + stage * STAGE_BYTES);
      const uint32_t sB = sA + A_STAGE_BYTES;
      const uint64_t adesc = smem_desc_sw128(sA, A_LBO, 1024u);
      const uint64_t bdesc = smem_desc_sw128(sB, B_LBO, 1024u);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        mma_bf16(d_tmem, adesc + A_KSTEP * k, bdesc + B_KSTEP * k, IDESC, (any || k > 0) ? 1u : 0u);
      }
      any = true;
      issued_any = true;
      mma_commit(&L.empty[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (any) {
      mma_commit(&L.tmem_full[acc]);
    } else {
      mbar_arrive(&L.tmem_full[acc]);  // nothing to wait for: the epilogue writes zeros
    }
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
    return true;
  });
  if (*abort_flag && issued_any) {
    mma_commit(L.drain);  // fires once every MMA issued so far has finished
    volatile int dummy = 0;
    wait_bounded(L.drain, 0, &dummy, nullptr);
  }
}

// ---------------------------------------------------------------- epilogues
struct EpiCtx {
  uint32_t taddr;  // TMEM address of this warp's lane quadrant, accumulator column 0
  int q;           // lane quadrant = tile rows 32q .. 32q + 31
  uint8_t* buf;    // this warp's 8 KiB staging area
  int iter;        // tiles processed so far by this warp
  int last_buf;    // staging half read by the most recent bulk group (-1: none)
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
  if (lane_id() == 0) mbar_arrive(&L.tmem_empty[acc]);
}

// FWD: fold a 128 x 256 logit tile into the running (max, sumexp) of each row.
struct FwdState {
  float run_m, run_s;
};

__device__ __forceinline__ void fold_chunk(const uint32_t (&r)[32], int col0, int V, long long xr, float& run_m,
                                           float& run_s, float& tval, bool& tfound) {
  const int nvalid = min(32, V - col0);
  const long long rel = xr - col0;
  if (rel >= 0 && rel < nvalid) {  // the target column passes: capture its logit
    const int ri = static_cast<int>(rel);
    float tv = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) tv = (j == ri) ? __uint_as_float(r[j]) : tv;
    tval = tv;
    tfound = true;
  }
  float y[32];
  float cmax = NEG_BIG;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    y[j] = (j < nvalid) ? __uint_as_float(r[j]) * LOG2E : -INFINITY;
    cmax = fmaxf(cmax, y[j]);
  }
  const float nm = fmaxf(run_m, cmax);
  float s = run_s * ex2(run_m - nm);
#pragma unroll
  for (int j = 0; j < 32; ++j) s += ex2(y[j] - nm);
  run_s = s;
  run_m = nm;
}

__device__ __forceinline__ void epi_fwd(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc,
                                        EpiCtx& e, FwdState& st) {
  const int row = t.m * BM + e.q * 32 + static_cast<int>(lane_id());
  const bool in_range = row < a.N;
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
    fold_chunk(r0, col0, a.V, xr, st.run_m, st.run_s, tval, tfound);
    if (col0 + 32 < a.V) fold_chunk(r1, col0 + 32, a.V, xr, st.run_m, st.run_s, tval, tfound);
  }
  release_tmem(L, acc);
  if (in_range && tfound) a.tgt[row] = tval;
  if (t.last && in_range) {
    a.part_m[static_cast<size_t>(t.split) * a.N + row] = st.run_m;
    a.part_s[static_cast<size_t>(t.split) * a.N + row] = st.run_s;
  }
}

// BWD_G: G = exp(A - LSE) - onehot, filter vote per 128-column half, bf16 store.
__device__ __forceinline__ bool epi_bwd_g(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc,
                                          EpiCtx& e) {
  const uint32_t lane = lane_id();
  const int row = t.m * BM + e.q * 32 + static_cast<int>(lane);
  long long xr = -1;
  bool valid = false;
  float lse2 = 0.0f, w = 0.0f;
  if (row < a.N) {
    xr = static_cast<long long>(__ldg(a.x + row));
    valid = (xr != a.ignore_index) && xr >= 0 && xr < a.V;
    if (valid) {
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
    bool surv = false;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c = 4 * h + cc;
      const int col0 = vt0 + 32 * c;
      uint32_t r[32];
      tmem_ld32(tbase + 32 * c, r);
      tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float g2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = col0 + j + u;
          float g = ex2(fmaf(__uint_as_float(r[j + u]), LOG2E, -lse2));
          if (static_cast<long long>(col) == xr) g -= 1.0f;
          if (!valid || col >= a.V) g = 0.0f;
          surv |= fabsf(g) >= a.eps;
          g2[u] = g * w;
        }
        pk[j / 2] = pack_bf16x2(g2[0], g2[1]);
      }
      const uint32_t box = sbuf + static_cast<uint32_t>((cc >> 1) * 4096);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        st_shared_v4(box + swz(lane, (cc & 1) * 4 + u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
    }
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
    if (keep) {
      fence_proxy_async_smem();
      __syncwarp();
      const int gx = t.n * BN + 128 * h;  // column inside the chunk buffer
      const int gy = t.m * BM + e.q * 32;
      if (lane == 0 && gy < a.N) {  // no store starts outside the buffer
        tma_store_2d(&a.tmOut, e.buf, gx, gy);
        tma_store_2d(&a.tmOut, e.buf + 4096, gx + 64, gy);
        bulk_commit();
      }
    }
    if (e.q == 0 && lane == 0) {
      const int vt128 = (vt0 >> 7) + h;
      if (vt128 < a.bm_ld) {
        a.bitmap[static_cast<size_t>(t.m) * a.bm_ld + vt128] = keep ? 1 : 0;
        a.bitmapT[static_cast<size_t>(vt128) * a.n_blocks + t.m] = keep ? 1 : 0;
      }
    }
  }
  return ok;
}

// DC: bf16 output tile, rows = vocabulary (chunk_v0 + 128m ...), cols = D.
__device__ __forceinline__ void epi_dc(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc, EpiCtx& e) {
  const uint32_t lane = lane_id();
  const bool empty = tile_empty<MODE_DC>(a, t);
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
  const int gy = a.chunk_v0 + t.m * BM + e.q * 32;
  // boxes that start inside dC (no store may start outside the tensor)
  const int nbox = (gy < a.V) ? min(BN / 64, (a.D - t.n * BN + 63) / 64) : 0;
#pragma unroll 1
  for (int j = 0; j < nbox; ++j) {
    const int b = j & 1;
    uint8_t* buf = e.buf + b * 4096;
    staging_acquire(e, b);
    const uint32_t sb = smem_u32(buf);
    if (!empty) {
      uint32_t r0[32], r1[32];
      tmem_ld32(tbase + 64 * j, r0);
      tmem_ld32(tbase + 64 * j + 32, r1);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        st_shared_v4(sb + swz(lane, u), pack_bf16x2(__uint_as_float(r0[8 * u + 0]), __uint_as_float(r0[8 * u + 1])),
                     pack_bf16x2(__uint_as_float(r0[8 * u + 2]), __uint_as_float(r0[8 * u + 3])),
                     pack_bf16x2(__uint_as_float(r0[8 * u + 4]), __uint_as_float(r0[8 * u + 5])),
                     pack_bf16x2(__uint_as_float(r0[8 * u + 6]), __uint_as_float(r0[8 * u + 7])));
        st_shared_v4(sb + swz(lane, 4 + u),
                     pack_bf16x2(__uint_as_float(r1[8 * u + 0]), __uint_as_float(r1[8 * u + 1])),
                     pack_bf16x2(__uint_as_float(r1[8 * u + 2]), __uint_as_float(r1[8 * u + 3])),
                     pack_bf16x2(__uint_as_float(r1[8 * u + 4]), __uint_as_float(r1[8 * u + 5])),
                     pack_bf16x2(__uint_as_float(r1[8 * u + 6]), __uint_as_float(r1[8 * u + 7])));
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) st_shared_v4(sb + swz(lane, u), 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&a.tmOut, buf, t.n * BN + 64 * j, gy);
      bulk_commit();
    }
    e.last_buf = b;
  }
  release_tmem(L, acc);
}

// DE: fp32 output tile, rows = tokens, cols = D; store (first chunk) or reduce-add.
__device__ __forceinline__ void epi_de(const GemmArgs& a, const SmemLayout& L, const Tile& t, int acc, EpiCtx& e) {
  const uint32_t lane = lane_id();
  const bool empty = tile_empty<MODE_DE>(a, t);
  if (empty && !a.first_chunk) {  // adding zero: nothing to do
    release_tmem(L, acc);
    return;
  }
  const uint32_t tbase = e.taddr + static_cast<uint32_t>(acc * BN);
  const int gy = t.m * BM + e.q * 32;
  // boxes that start inside dE (no store or reduce may start outside the tensor)
  const int nbox = (gy < a.N) ? min(BN / 32, (a.D - t.n * BN + 31) / 32) : 0;
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
      if (a.first_chunk) {
        tma_store_2d(&a.tmOut, buf, t.n * BN + 32 * j, gy);
      } else {
        tma_reduce_add_2d(&a.tmOut, buf, t.n * BN + 32 * j, gy);
      }
      bulk_commit();
    }
    e.last_buf = b;
  }
  release_tmem(L, acc);
}

template <int MODE>
__device__ __forceinline__ void epilogue_loop(const GemmArgs& a, const SmemLayout& L, uint32_t tmem_base,
                                              int warp) {
  EpiCtx e;
  e.q = warp & 3;
  e.taddr = tmem_base + (static_cast<uint32_t>(e.q * 32) << 16);
  e.buf = L.epi + (warp - 2) * EPI_WARP_BYTES;
  e.iter = 0;
  e.last_buf = -1;
  FwdState st{NEG_BIG, 0.0f};
  int acc = 0;
  uint32_t acc_phase = 0;
  for_each_tile<MODE>(a, [&](const Tile& t) -> bool {
    if (!warp_wait_bounded(&L.tmem_full[acc], acc_phase, L.abort_flag, a.dev_err)) return false;
    tc_fence_after();
    bool ok = true;
    if constexpr (MODE == MODE_FWD) {
      epi_fwd(a, L, t, acc, e, st);
    } else if constexpr (MODE == MODE_BWD_G) {
      ok = epi_bwd_g(a, L, t, acc, e);
    } else if constexpr (MODE == MODE_DC) {
      epi_dc(a, L, t, acc, e);
    } else {
      epi_de(a, L, t, acc, e);
    }
    ++e.iter;
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
    return ok;
  });
  if (lane_id() == 0) bulk_wait_all();
  __syncwarp();
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) cce_gemm_kernel(const __grid_constant__ GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout L = carve_smem(smem_raw);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&L.full[s], 1);
      mbar_init(&L.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&L.tmem_full[i], 1);
      mbar_init(&L.tmem_empty[i], NUM_EPI_WARPS);
      mbar_init(&L.vote[i], NUM_EPI_WARPS);
    }
    mbar_init(L.drain, 1);
    *L.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&a.tmA);
    tma_prefetch_desc(&a.tmB);
    if (MODE != MODE_FWD) tma_prefetch_desc(&a.tmOut);
  }
  if (warp == 1) {
    tmem_alloc(L.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *L.tmem_base;

  if (warp == 0) {
    if (lane_id() == 0) producer_loop<MODE>(a, L);
  } else if (warp == 1) {
    if (lane_id() == 0) mma_loop<MODE>(a, L, tmem_base);
  } else {
    epilogue_loop<MODE>(a, L, tmem_base, warp);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace cce
