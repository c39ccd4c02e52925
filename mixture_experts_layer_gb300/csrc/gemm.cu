// Padding-free grouped GEMMs of the layer on the 5th-generation tensor cores.
//
// "UniEP: Unified Expert-Parallel MoE MegaKernel for LLM Training":
//   - background, Forward Propagation: GroupGEMM -> SwiGLU -> GroupGEMM per expert;
//   - section 3 (Scoreboard-based Synchronization, Comp Worker Logic): a
//     padding-free GroupGEMM that follows each expert's irregular row count with
//     pointer arithmetic instead of padding;
//   - background, Backward Propagation and Numerical Stability: dgrad
//     GroupGEMMs and the weight-gradient Transposed GroupGEMM, which reduces
//     over the token dimension.  Each output tile here has exactly one owner
//     and reduces its expert's rows in ascending order, so the bits do not
//     depend on the grid size or on scheduling.
//   - section 3 (Persistent Worker Architecture): one resident CTA per SM
//     loops over the tile list.
//
// Kernel structure (one CTA per SM, 320 threads):
//   warp 0     TMA producer: fills a ring of shared-memory stages
//   warp 1     allocates tensor memory, issues tcgen05.mma (one elected lane)
//   warps 2-9  epilogue, two warps per TMEM lane quarter (32 rows), each taking
//              half of the tile's columns: tcgen05.ld of the fp32 accumulator
//              (the next chunk's load in flight while this one is stored),
//              fused elementwise work (SwiGLU forward or backward), stores.  The
//              fp32 weight gradients go out through a swizzled shared-memory
//              box per warp, re-read row-wise for coalesced 16-byte stores.
// The accumulator is double-buffered in tensor memory (2 x 256 columns), so the
// epilogue of one tile overlaps the main loop of the next.
//
// Tiles are 128 rows x 256 columns (the last tile of an N extent that is an odd
// multiple of 128 is 128 wide).  Operand layouts in shared memory are the
// 128-byte-swizzled canonical forms:
//   K-major  (rows of 64 K-elements, 128 B each, 8-row atoms of 1 KB):
//            SBO = 1024 B between 8-row groups; +32 B per K step of 16.
//   MN-major (panels of 64 MN-elements x 64 K-rows, 8 KB each):
//            LBO = 8192 B between panels, SBO = 1024 B between 8-row K groups;
//            +2048 B per K step of 16.
#include <string.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each taking half of the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;   // TMEM columns per accumulator buffer
constexpr int kPanelBytes = 64 * 128;  // one MN-major panel: 64 K-rows x 128 B
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytesMax = BN * BK * 2;
constexpr int kStageBytes = kABytes + kBBytesMax;
constexpr int kStageOutBytes = 32 * 128;  // one warp's 32x32 fp32 staging box
constexpr int kEpiRing = 2;                // dgrad2 epilogue: G/U chunk boxes in flight per warp
constexpr int kEpiRingBytes = kEpiRing * 2048;

// Per-warp epilogue staging of a mode: fp32 store boxes (weight gradients) or
// the G/U chunk ring (dgrad2).
template <int MODE>
__host__ __device__ constexpr int epi_stage_bytes() {
  return MODE == kDgrad2 ? kEpiRingBytes : (MODE == kWgrad13 || MODE == kWgrad2) ? kStageOutBytes : 0;
}

template <int MODE>
struct ModeTraits {
  static constexpr bool wgrad = (MODE == kWgrad13 || MODE == kWgrad2);
  static constexpr bool router = (MODE == kRfwd || MODE == kRwgrad);
  static constexpr bool a_mn = wgrad || MODE == kRwgrad;
  static constexpr bool b_mn = (MODE == kFwd1 || MODE == kFwd2 || wgrad || router);
  // Output columns per tile are 2 x 128 (two weights side by side) or up to 256.
  static constexpr bool paired = (MODE == kFwd1 || MODE == kWgrad13);
  static constexpr int kStages = 4;
  static constexpr int kStagingBytes = kEpiWarps * epi_stage_bytes<MODE>();
  static constexpr int kSmemBytes = kStages * kStageBytes + kStagingBytes + 1024 /*align*/ + 512 /*barriers*/;
};

struct Maps {
  CUtensorMap a;   // A operand
  CUtensorMap b0;  // B operand (full-width box)
  CUtensorMap b1;  // second B tensor (W3), full-width box
  CUtensorMap b2;  // B, 128-row box for a 128-wide tail tile (K-major B only)
  CUtensorMap b3;  // W3, 128-row box
  CUtensorMap a64; // A operand, 64-row box: the 64 rows of an M = 128 pair tile's CTA
  CUtensorMap gu;  // dgrad2 epilogue: GU [R, 2F], 16-column x 32-row boxes, 32-byte swizzle
  // Pair tiles, MN-major operands: 3-D views {64 columns, rows, 64-column panels}
  // whose box holds two neighbouring panels (one TMA instruction instead of two).
  CUtensorMap a_p2;   // A (weight gradients)
  CUtensorMap b0_p2;  // B (W1, W2, dGU or dY)
  CUtensorMap b1_p2;  // second B tensor (W3)
};

// The gated combine fused into GEMM2's epilogue (null cnt: not fused).
struct CombineParams {
  int32_t* cnt;            // [T][N tiles][2] arrivals of (token, 256-column tile, column half); zero at launch
  const int32_t* row_src;  // [R] token of each grouped row
  const int32_t* dest;     // [T,k]
  const float* w;          // [T,k]
  __nv_bfloat16* out;      // [T,H]
  int k;
};

struct GemmParams {
  int H, F, E, R;
  int T, splits, ks;  // router modes: tokens, token splits of the weight gradient, tokens per split
  CombineParams cmb;
  const int32_t* tiles;
  const int32_t* pairs;  // first 256-row pair tile of each expert (E + 1)
  const int32_t* offsets;
  const int32_t* counts;
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  const __nv_bfloat16* aux;
  float* f0;
  float* f1;
  // Weight gradients reduced as two token sub-batches: 0 one chain over all of
  // an expert's rows; 1 the first sb_rows[e] rows (stored); 2 the rest, added
  // onto the stored values.
  int sb;
  const int32_t* sb_rows;
  // GEMM1 with the dispatch in its A-operand load: A rows are gathered from x by
  // row_src (16-byte cp.async copies into the swizzled stage) and the first N tile
  // of each row block stores them to Xp.
  int gather;
  const __nv_bfloat16* x;  // [T, H] (gather)
  const int32_t* row_src;
  // Pair tiles (forward and dgrad modes): an expert's last 256-row block with at
  // most 128 rows runs as an M = 128 pair tile, 64 rows per CTA.
  int halfm_ok;
  // Pair tiles: the two-panel 3-D maps (a_p2, b0_p2, b1_p2) were encoded, so each
  // pair of 64-column MN-major panels is one TMA instruction.
  int panels2;
  WsHeader* ws;
};

// Restricts a weight-gradient tile's K range (the expert's rows) to one token
// sub-batch.  Rows of an expert are in token order, so sub-batch 0 is a prefix.
__device__ __forceinline__ void subbatch_range(const GemmParams& p, int e, int& row0, int& nrows) {
  if (p.sb == 0) return;
  const int m = __ldg(p.sb_rows + e);
  if (p.sb == 1) {
    nrows = m;
  } else {
    row0 += m;
    nrows -= m;
  }
}

struct Tile {
  int e;      // expert
  int row0;   // first grouped row of the tile (forward/dgrad) or of the expert (wgrad)
  int nrows;  // valid rows of the tile (forward/dgrad) or rows of the expert (wgrad)
  int m0;     // wgrad: first output row inside the expert's weight
  int n0;     // first output column
  int nw;     // MMA N of the tile: 256, or 128 for a tail tile
  int kblocks;
  int mt;     // forward/dgrad: index of the 128-row tile in the plan's tile table
  int halfm = 0;  // pair tiles: 1 when the pair's MMA is M = 128 (this CTA holds 64 rows)
};

template <int MODE>
__device__ __forceinline__ int n_extent(const GemmParams& p) {
  if (ModeTraits<MODE>::router) return p.E;
  return (MODE == kFwd2 || MODE == kDgrad1 || MODE == kWgrad2) ? p.H : p.F;
}

// MMA N of a router tile: the remaining expert columns rounded up to 16 (the
// B columns past E are zero-filled by TMA), at most 256.
__device__ __forceinline__ int router_nw(int E, int n0) { return min(BN, (E - n0 + 15) & ~15); }

// Bytes one k-block's TMA loads bring into a stage (the A box plus B).
template <int MODE>
__device__ __forceinline__ uint32_t stage_tx_bytes(int nw) {
  if (ModeTraits<MODE>::router) return kABytes + ((nw + 63) / 64) * kPanelBytes;
  return kABytes + nw * 128;
}

template <int MODE>
__device__ __forceinline__ int n_ntiles(const GemmParams& p) {
  if (ModeTraits<MODE>::paired) return p.F / 128;
  return (n_extent<MODE>(p) + BN - 1) / BN;
}

template <int MODE>
__device__ __forceinline__ int n_tiles(const GemmParams& p) {
  const int nn = n_ntiles<MODE>(p);
  if (MODE == kRfwd) return ((p.T + BM - 1) / BM) * nn;
  if (MODE == kRwgrad) return p.splits * (p.H / BM) * nn;
  if (MODE == kWgrad13) return p.E * (p.H / BM) * nn;
  if (MODE == kWgrad2) return p.E * (p.F / BM) * nn;
  return __ldg(p.tiles) * nn;
}

template <int MODE>
__device__ __forceinline__ Tile decode(const GemmParams& p, int tile) {
  Tile t;
  const int nn = n_ntiles<MODE>(p);
  int nt;
  if (MODE == kRfwd) {  // 128 token rows x up to 256 experts; K = H
    const int mt = tile / nn;
    nt = tile - mt * nn;
    t.e = 0;
    t.row0 = mt * BM;
    t.nrows = min(BM, p.T - t.row0);
    t.m0 = 0;
    t.mt = -1;
    t.kblocks = p.H / BK;
    t.n0 = nt * BN;
    t.nw = router_nw(p.E, t.n0);
    return t;
  }
  if (MODE == kRwgrad) {  // 128 rows of H x up to 256 experts; K = the tokens of split s
    const int MT = p.H / BM;
    const int sp = tile / (MT * nn);
    const int rem = tile - sp * MT * nn;
    const int mt = rem / nn;
    nt = rem - mt * nn;
    t.e = sp;  // the split (partial buffer index)
    t.row0 = sp * p.ks;
    t.nrows = min(p.ks, p.T - t.row0);
    t.m0 = mt * BM;
    t.mt = -1;
    t.kblocks = (t.nrows + BK - 1) / BK;
    t.n0 = nt * BN;
    t.nw = router_nw(p.E, t.n0);
    return t;
  }
  if (ModeTraits<MODE>::wgrad) {
    const int MT = (MODE == kWgrad13) ? p.H / BM : p.F / BM;
    t.e = tile / (MT * nn);
    const int rem = tile - t.e * MT * nn;
    nt = rem / MT;
    t.m0 = (rem - nt * MT) * BM;
    t.row0 = __ldg(p.offsets + t.e);
    t.nrows = __ldg(p.counts + t.e);
    subbatch_range(p, t.e, t.row0, t.nrows);
    t.kblocks = (t.nrows + BK - 1) / BK;
    t.mt = -1;
  } else {
    const int entries = tiles_entry_base(p.E);
    const int4* ent = reinterpret_cast<const int4*>(p.tiles + entries);
    // Tiles of one expert are ordered (n tile, m tile) with m fastest, so the CTAs
    // working side by side share the same weight columns (L2 reuse).
    const int q = tile / nn;
    const int e = __ldg(&ent[q].x);
    const int first = __ldg(p.tiles + 1 + e);
    const int cnt = __ldg(p.tiles + 2 + e) - first;
    const int local = tile - nn * first;
    nt = local / cnt;
    const int mt = first + (local - nt * cnt);
    const int4 en = ent[mt];
    t.e = e;
    t.row0 = en.y;
    t.nrows = en.z;
    t.m0 = 0;
    t.mt = mt;
    const int K = (MODE == kFwd1 || MODE == kDgrad2) ? p.H : (MODE == kFwd2) ? p.F : 2 * p.F;
    t.kblocks = K / BK;
  }
  if (ModeTraits<MODE>::paired) {
    t.n0 = nt * 128;
    t.nw = 256;
  } else {
    t.n0 = nt * BN;
    t.nw = min(BN, n_extent<MODE>(p) - t.n0);
  }
  return t;
}

// Issues the TMA loads of one k-block into stage buffers sA / sB.
template <int MODE>
__device__ __forceinline__ void load_kblock(const GemmParams& p, const Maps& m, const Tile& t, int kb, uint8_t* sA,
                                            uint8_t* sB, uint64_t* bar) {
  const int k0 = kb * BK;
  const bool tail = t.nw < BN;
  if (MODE == kFwd1) {
    tma_load_2d(sA, &m.a, bar, k0, t.row0);
    const int y = t.e * p.H + k0;
    tma_load_2d(sB + 0 * kPanelBytes, &m.b0, bar, t.n0, y);
    tma_load_2d(sB + 1 * kPanelBytes, &m.b0, bar, t.n0 + 64, y);
    tma_load_2d(sB + 2 * kPanelBytes, &m.b1, bar, t.n0, y);
    tma_load_2d(sB + 3 * kPanelBytes, &m.b1, bar, t.n0 + 64, y);
  } else if (MODE == kFwd2) {
    tma_load_2d(sA, &m.a, bar, k0, t.row0);
    const int y = t.e * p.F + k0;
    for (int q = 0; q < t.nw / 64; ++q) tma_load_2d(sB + q * kPanelBytes, &m.b0, bar, t.n0 + 64 * q, y);
  } else if (MODE == kDgrad2) {
    tma_load_2d(sA, &m.a, bar, k0, t.row0);
    tma_load_2d(sB, tail ? &m.b2 : &m.b0, bar, k0, t.e * p.F + t.n0);
  } else if (MODE == kDgrad1) {
    tma_load_2d(sA, &m.a, bar, k0, t.row0);
    if (k0 < p.F)
      tma_load_2d(sB, tail ? &m.b2 : &m.b0, bar, k0, t.e * p.H + t.n0);
    else
      tma_load_2d(sB, tail ? &m.b3 : &m.b1, bar, k0 - p.F, t.e * p.H + t.n0);
  } else if (MODE == kWgrad13) {
    const int y = t.row0 + k0;
    tma_load_2d(sA, &m.a, bar, t.m0, y);
    tma_load_2d(sA + kPanelBytes, &m.a, bar, t.m0 + 64, y);
    tma_load_2d(sB + 0 * kPanelBytes, &m.b0, bar, t.n0, y);
    tma_load_2d(sB + 1 * kPanelBytes, &m.b0, bar, t.n0 + 64, y);
    tma_load_2d(sB + 2 * kPanelBytes, &m.b0, bar, p.F + t.n0, y);
    tma_load_2d(sB + 3 * kPanelBytes, &m.b0, bar, p.F + t.n0 + 64, y);
  } else if (MODE == kWgrad2) {
    const int y = t.row0 + k0;
    tma_load_2d(sA, &m.a, bar, t.m0, y);
    tma_load_2d(sA + kPanelBytes, &m.a, bar, t.m0 + 64, y);
    for (int q = 0; q < t.nw / 64; ++q) tma_load_2d(sB + q * kPanelBytes, &m.b0, bar, t.n0 + 64 * q, y);
  } else if (MODE == kRfwd) {  // A = x rows (K-major), B = Wr [H, E] panels (MN-major)
    tma_load_2d(sA, &m.a, bar, k0, t.row0);
    for (int q = 0; q < (t.nw + 63) / 64; ++q) tma_load_2d(sB + q * kPanelBytes, &m.b0, bar, t.n0 + 64 * q, k0);
  } else {  // kRwgrad: A = x^T (MN-major panels of H), B = dl [T, E] panels; rows past T read as zeros
    const int y = t.row0 + k0;
    tma_load_2d(sA, &m.a, bar, t.m0, y);
    tma_load_2d(sA + kPanelBytes, &m.a, bar, t.m0 + 64, y);
    for (int q = 0; q < (t.nw + 63) / 64; ++q) tma_load_2d(sB + q * kPanelBytes, &m.b0, bar, t.n0 + 64 * q, y);
  }
}

__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void store_zero_f32(float* dst) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) st_v4(dst + i, 0u, 0u, 0u, 0u);
}

// One warp's fp32 output path (weight gradients): its 32 rows x 32 columns go
// to a 128B-swizzled 4 KB box in shared memory, are read back row-wise (8 lanes
// per 128-byte row, conflict-free) and written with plain 16-byte stores, each
// store instruction covering 4 whole rows.  (TMA bulk stores of the same boxes
// measured slower: one 4 KB bulk store at a time kept each SM near 16 B/clk.)
struct OutStager {
  uint8_t* buf;  // one 4 KB box, 1024-byte aligned
  // dgrad2: buf holds a ring of kEpiRing 2 KB slots, each a (G, U) pair of
  // 16-column x 32-row boxes filled by TMA; ebar[kEpiRing] their barriers (null:
  // G and U are read directly from global memory); eph the parity each barrier
  // waits for next.
  uint64_t* ebar = nullptr;
  uint32_t eph = 0;
  uint32_t pending = 0;  // slots whose load was issued and not yet consumed
  // Before the CTA exits (also after an abort): wait (bounded) for loads still in flight.
  __device__ __forceinline__ void drain(WsHeader* ws) {
    for (int s = 0; s < kEpiRing && ebar != nullptr; ++s)
      if ((pending >> s) & 1u) {
        mbar_wait(&ebar[s], (eph >> s) & 1u, ws, 271, nullptr);
        eph ^= 1u << s;
      }
    pending = 0;
  }
  // dst points at the block's first element; ld is the row stride in floats.
  // ACC: add the values already stored there (the second sub-batch's partial).
  template <bool ACC = false>
  __device__ __forceinline__ void put(float* dst, size_t ld, const uint32_t (&r)[32], int lane) {
    const uint32_t base = smem_u32(buf);
    const uint32_t row = base + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(row + ((j ^ (lane & 7)) << 4), r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    __syncwarp();
    const int j = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3);
      uint32_t a, b, c, d;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                   : "r"(base + rr * 128 + ((j ^ (rr & 7)) << 4)));
      float* q = dst + static_cast<size_t>(rr) * ld + 4 * j;
      if (ACC)  // the L2 adds (one add per element onto the stored value: no ordering question)
        asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(q), "f"(__uint_as_float(a)),
                     "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d))
                     : "memory");
      else
        asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(q), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
    }
    __syncwarp();
  }
};

// Weight-gradient K tail: the last k-block of an expert holds `valid` < 64 of
// its rows.  The MMAs cover ceil(valid/16)*16 rows; the rows in between that
// belong to the next expert are cleared in both operands (A: 2 panels, B: nw/64
// panels), so neither stale values nor the next expert's rows contribute.
__device__ __forceinline__ int clear_k_tail(uint8_t* sA, uint8_t* sB, int valid, int nw, int lane) {
  const int nkk = (valid + 15) >> 4;
  const int nz = nkk * 16 - valid;  // < 16 rows
  const int panels = 2 + nw / 64;
  // Lane -> (row offset lane / 8, 16-byte chunk lane % 8); 4 rows per pass.
  for (int r = valid + (lane >> 3); r < valid + nz; r += 4) {
    const int off = r * 128 + (lane & 7) * 16;
    for (int pnl = 0; pnl < panels; ++pnl) {
      uint8_t* base = pnl < 2 ? sA + pnl * kPanelBytes : sB + (pnl - 2) * kPanelBytes;
      *reinterpret_cast<uint4*>(base + off) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  fence_proxy_async_smem();
  return nkk;
}

// The gated combine in GEMM2's epilogue ("UniEP", section 3, Top-k
// accumulation constraint, and section 5, Reduce Workers: a token's output is
// summed only when all k of its expert rows are ready, in a fixed order).  Each
// thread has just stored columns [c_lo, c_hi) of the 256-column tile for its
// row; it counts that half-row done for its token (release: a fence before the
// atomic).  The thread whose count completes the token's k rows flags it, and
// the warp then writes out[t] for those columns for every flagged token:
// out = bf16(sum_j w[t,j] Y[dest[t,j]]) in slot order, the arithmetic of the
// separate combine kernel, so both give the same bits.
__device__ __forceinline__ void combine_in_epilogue(const GemmParams& p, const Tile& t, size_t grow, bool valid,
                                                    int half, int c_lo, int c_hi, int lane) {
  const CombineParams& c = p.cmb;
  const int nn = (p.H + BN - 1) / BN;
  __threadfence();
  int tok = -1, done = 0;
  if (valid) {
    tok = __ldg(c.row_src + grow);
    if (tok == -1) {
      // a padding row: no token to combine
    } else if (tok < 0 || tok >= p.T) {
      report(p.ws, MOE_ERR_BOUNDS, 30, static_cast<int>(grow));
    } else {
      const int old = atomicAdd(c.cnt + (static_cast<size_t>(tok) * nn + t.n0 / BN) * 2 + half, 1);
      done = (old == c.k - 1);
    }
  }
  uint32_t m = __ballot_sync(0xffffffffu, done);
  if (m == 0) return;
  __threadfence();  // acquire: the other rows' Y stores are visible to this warp
  // Lane groups of nvec lanes (one 16-byte vector each) take one completed token
  // apiece; every slot's row is loaded before any is summed.
  const int nvec = (c_hi - c_lo) / 8;  // 8 or 16
  const int per = 32 / nvec;
  const int grp = lane / nvec, l = lane % nvec;
  const int hv = p.H / 8;
  const int v = (t.n0 + c_lo) / 8 + l;
  while (m) {
    int src = -1;
    for (int i = 0; i < per; ++i) {
      const int f = m ? __ffs(m) - 1 : -1;
      if (i == grp) src = f;
      if (m) m &= m - 1;
    }
    const int tt = __shfl_sync(0xffffffffu, tok, src < 0 ? 0 : src);
    if (src < 0) continue;
    constexpr int K = 8;
    if (c.k <= K) {
      int r[K];
      float wj[K];
      uint4 y[K];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        r[j] = j < c.k ? __ldg(c.dest + static_cast<size_t>(tt) * c.k + j) : 0;
        wj[j] = j < c.k ? __ldg(c.w + static_cast<size_t>(tt) * c.k + j) : 0.f;
      }
      bool bad = false;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j < c.k) {
          if (r[j] < 0 || r[j] >= p.R) {
            bad = true;
            r[j] = 0;
          }
          asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(y[j].x), "=r"(y[j].y), "=r"(y[j].z), "=r"(y[j].w)
                       : "l"(reinterpret_cast<const uint4*>(p.out0) + static_cast<size_t>(r[j]) * hv + v));
        }
      }
      if (bad) {
        report(p.ws, MOE_ERR_BOUNDS, 31, tt);
        continue;
      }
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j < c.k) {
          const uint32_t yw[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(wj[j], bf16lo(yw[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(wj[j], bf16hi(yw[i]), acc[2 * i + 1]);
          }
        }
      }
      st_v4(reinterpret_cast<uint4*>(c.out) + static_cast<size_t>(tt) * hv + v, pack_bf16x2(acc[0], acc[1]),
            pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    } else {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      bool bad = false;
      for (int j = 0; j < c.k; ++j) {
        const int rj = __ldg(c.dest + static_cast<size_t>(tt) * c.k + j);
        const float wjj = __ldg(c.w + static_cast<size_t>(tt) * c.k + j);
        if (rj < 0 || rj >= p.R) {
          bad = true;
          break;
        }
        uint4 y;
        asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(y.x), "=r"(y.y), "=r"(y.z), "=r"(y.w)
                     : "l"(reinterpret_cast<const uint4*>(p.out0) + static_cast<size_t>(rj) * hv + v));
        const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wjj, bf16lo(yw[i]), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wjj, bf16hi(yw[i]), acc[2 * i + 1]);
        }
      }
      if (bad) {
        report(p.ws, MOE_ERR_BOUNDS, 31, tt);
        continue;
      }
      st_v4(reinterpret_cast<uint4*>(c.out) + static_cast<size_t>(tt) * hv + v, pack_bf16x2(acc[0], acc[1]),
            pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// SwiGLU backward of one element, with every rounding step spelled out so that
// each epilogue that uses it gives the same bits: s = sigmoid(G),
// dG = dH U s (1 + G (1 - s)), dU = dH G s.
__device__ __forceinline__ void swiglu_bwd(float G, float U, float dh, float& dg, float& du) {
  const float sg = __frcp_rn(__fadd_rn(1.0f, expf(-G)));
  const float tt = __fmaf_rn(G, __fsub_rn(1.0f, sg), 1.0f);
  dg = __fmul_rn(__fmul_rn(__fmul_rn(dh, U), sg), tt);
  du = __fmul_rn(__fmul_rn(dh, G), sg);
}

// dgrad2 epilogue with staged operands: this warp's 32 rows x [c_lo, c_hi)
// columns in 16-column chunks.  The G and U blocks of a chunk (32 rows x 16
// columns, 32-byte swizzle) arrive by TMA into a ring of kEpiRing slots: the
// first kEpiRing are requested before the accumulator is ready
// (dgrad2_prefetch), each later one as soon as its slot is free.  Each lane
// reads its row, writes dG and dU back in place, and the warp then stores the
// two blocks with row-contiguous 32-byte segments (16 rows per instruction),
// skipping the rows past the tile's valid rows.
__device__ __forceinline__ void dgrad2_cols(const Tile& t, int half, int& c_lo, int& c_hi) {
  c_lo = half * (t.nw / 2);
  c_hi = c_lo + t.nw / 2;
}

__device__ __forceinline__ void dgrad2_issue(const GemmParams& p, const Maps& m, const Tile& t, int q, int c_lo, int k,
                                             int lane, OutStager& st) {
  const int slot = k % kEpiRing;
  __syncwarp();
  if (lane == 0) {
    fence_proxy_async_smem();  // this warp's earlier reads and writes of the slot come first
    mbar_arrive_expect_tx(&st.ebar[slot], 2048);
    const int col = t.n0 + c_lo + 16 * k;
    tma_load_2d(st.buf + slot * 2048, &m.gu, &st.ebar[slot], col, t.row0 + 32 * q);
    tma_load_2d(st.buf + slot * 2048 + 1024, &m.gu, &st.ebar[slot], p.F + col, t.row0 + 32 * q);
  }
  st.pending |= 1u << slot;
}

__device__ __forceinline__ void dgrad2_prefetch(const GemmParams& p, const Maps& m, const Tile& t, int q, int half,
                                                int lane, OutStager& st) {
  int c_lo, c_hi;
  dgrad2_cols(t, half, c_lo, c_hi);
  const int nch = (c_hi - c_lo) / 16;
  for (int k = 0; k < nch && k < kEpiRing; ++k) dgrad2_issue(p, m, t, q, c_lo, k, lane, st);
}

__device__ __forceinline__ void dgrad2_epilogue_staged(const GemmParams& p, const Maps& m, const Tile& t, uint32_t tacc,
                                                       int q, int c_lo, int c_hi, int lane, OutStager& st) {
  const int y0 = t.row0 + 32 * q;
  const int nch = (c_hi - c_lo) / 16;
  const uint32_t base = smem_u32(st.buf);
  // Byte offset of 16-byte chunk j of row r in a 32-byte-swizzled box.
  auto sw = [](int r, int j) { return static_cast<uint32_t>(r * 32 + ((j ^ ((r >> 2) & 1)) << 4)); };
#pragma unroll 1
  for (int k = 0; k < nch; ++k) {
    const int slot = k % kEpiRing;
    uint32_t d[16];
    tc_ld_32x32b_x16(tacc + c_lo + 16 * k, d);
    mbar_wait(&st.ebar[slot], (st.eph >> slot) & 1u, p.ws, 270, nullptr);
    st.eph ^= 1u << slot;
    st.pending &= ~(1u << slot);
    tc_wait_ld();
    const uint32_t gbox = base + slot * 2048, ubox = gbox + 1024;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t g0, g1, g2, g3, u0, u1, u2, u3;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(g0), "=r"(g1), "=r"(g2), "=r"(g3)
                   : "r"(gbox + sw(lane, j)));
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(u0), "=r"(u1), "=r"(u2), "=r"(u3)
                   : "r"(ubox + sw(lane, j)));
      const uint32_t gw[4] = {g0, g1, g2, g3}, uw[4] = {u0, u1, u2, u3};
      uint32_t dgw[4], duw[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float dg0, du0, dg1, du1;
        swiglu_bwd(bf16lo(gw[qq]), bf16lo(uw[qq]), __uint_as_float(d[8 * j + 2 * qq]), dg0, du0);
        swiglu_bwd(bf16hi(gw[qq]), bf16hi(uw[qq]), __uint_as_float(d[8 * j + 2 * qq + 1]), dg1, du1);
        dgw[qq] = pack_bf16x2(dg0, dg1);
        duw[qq] = pack_bf16x2(du0, du1);
      }
      st_shared_v4(gbox + sw(lane, j), dgw[0], dgw[1], dgw[2], dgw[3]);
      st_shared_v4(ubox + sw(lane, j), duw[0], duw[1], duw[2], duw[3]);
    }
    __syncwarp();
    // Row-contiguous stores: lane l covers row 16 i + l / 2, 16-byte chunk l % 2.
    const int j = lane & 1;
    const int col = t.n0 + c_lo + 16 * k + 8 * j;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int rr = 16 * i + (lane >> 1);
      if (32 * q + rr < t.nrows) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                     : "r"(gbox + sw(rr, j)));
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                     : "r"(ubox + sw(rr, j)));
        __nv_bfloat16* dst = p.out0 + static_cast<size_t>(y0 + rr) * (2 * p.F) + col;
        st_v4(dst, a0, a1, a2, a3);
        st_v4(dst + p.F, b0, b1, b2, b3);
      }
    }
    if (k + kEpiRing < nch) dgrad2_issue(p, m, t, q, c_lo, k + kEpiRing, lane, st);  // the slot is free again
  }
  __syncwarp();
}

template <int MODE>
__device__ __forceinline__ void epilogue(const GemmParams& p, const Maps& m, const Tile& t, uint32_t tacc, int q,
                                         int half, int lane, OutStager& st) {
  const int row = q * 32 + lane;
  if (ModeTraits<MODE>::router) {
    // fp32 rows of the output (logits [T, E], or the split's dWr partial
    // [H, E]); this warp takes every other 32-column chunk, columns >= E skipped.
    float* orow;
    bool ok;
    if (MODE == kRfwd) {
      ok = row < t.nrows;
      orow = p.f0 + static_cast<size_t>(t.row0 + row) * p.E + t.n0;
    } else {
      ok = true;
      orow = p.f0 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.E + t.n0;
    }
    const int ncol = min(t.nw, p.E - t.n0);
#pragma unroll 1
    for (int c = 32 * half; c < t.nw; c += 64) {
      uint32_t d[32];
      tc_ld_32x32b_x32(tacc + c, d);
      tc_wait_ld();
      if (!ok) continue;
      if (c + 32 <= ncol) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) st_v4(orow + c + i, d[i], d[i + 1], d[i + 2], d[i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c + i < ncol) orow[c + i] = __uint_as_float(d[i]);
      }
    }
    return;
  }
  // This warp's columns: [c_lo, c_hi) of each output (NC / 2 is a multiple of 16).
  // An M = 128 pair tile (halfm) holds half of the tile's columns per lane half.
  const int NCall = ModeTraits<MODE>::paired ? (t.halfm ? 64 : 128) : t.nw;
  const int c_lo = half * (NCall / 2), c_hi = c_lo + NCall / 2;
  if (ModeTraits<MODE>::wgrad) {
    const int y = (MODE == kWgrad13) ? t.e * p.H + t.m0 + q * 32 : t.e * p.F + t.m0 + q * 32;
    const size_t ld = (MODE == kWgrad13) ? p.F : p.H;
#pragma unroll 1
    for (int out = 0; out < ((MODE == kWgrad13) ? 2 : 1); ++out) {
      float* obase = (out ? p.f1 : p.f0) + static_cast<size_t>(y) * ld;
      const uint32_t tbase = tacc + (out ? 128 : 0);
      uint32_t a[32];
      tc_ld_32x32b_x32(tbase + c_lo, a);
      tc_wait_ld();
#pragma unroll 1
      for (int c = c_lo; c < c_hi; c += 32) {
        const bool more = c + 32 < c_hi;
        uint32_t b[32];
        if (more) tc_ld_32x32b_x32(tbase + c + 32, b);  // next chunk in flight during this chunk's stores
        if (p.sb == 2)
          st.put<true>(obase + t.n0 + c, ld, a, lane);
        else
          st.put(obase + t.n0 + c, ld, a, lane);
        if (more) {
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = b[i];
        }
      }
    }
    return;
  }
  if (MODE == kDgrad2 && st.ebar != nullptr) {
    dgrad2_epilogue_staged(p, m, t, tacc, q, c_lo, c_hi, lane, st);
    return;
  }
  const bool valid = row < t.nrows;
  const size_t grow = static_cast<size_t>(t.row0) + row;
  uint4 gcur[4], ucur[4];
  if (MODE == kDgrad2 && valid) {
    const __nv_bfloat16* gsrc = p.aux + grow * (2 * p.F) + t.n0 + c_lo;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      gcur[i] = ld_v4(gsrc + 8 * i);
      ucur[i] = ld_v4(gsrc + p.F + 8 * i);
    }
  }
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 32) {
    if (MODE == kFwd1) {
      uint32_t g[32], u[32];
      tc_ld_32x32b_x32(tacc + c, g);
      tc_ld_32x32b_x32(tacc + (t.halfm ? 64 : 128) + c, u);
      tc_wait_ld();
      if (valid) {
        uint32_t hw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = __uint_as_float(g[2 * i]), a1 = __uint_as_float(g[2 * i + 1]);
          const float b0 = __uint_as_float(u[2 * i]), b1 = __uint_as_float(u[2 * i + 1]);
          hw[i] = pack_bf16x2(a0 * __frcp_rn(1.0f + expf(-a0)) * b0, a1 * __frcp_rn(1.0f + expf(-a1)) * b1);
          g[i] = pack_bf16x2(a0, a1);  // G, U packed in place (entries i < 16 are no longer needed)
          u[i] = pack_bf16x2(b0, b1);
        }
        __nv_bfloat16* hdst = p.out0 + grow * p.F + t.n0 + c;
        __nv_bfloat16* gdst = p.out1 + grow * (2 * p.F) + t.n0 + c;
#pragma unroll
        for (int i = 0; i < 16; i += 4) st_v4(hdst + 2 * i, hw[i], hw[i + 1], hw[i + 2], hw[i + 3]);
#pragma unroll
        for (int i = 0; i < 16; i += 4) st_v4(gdst + 2 * i, g[i], g[i + 1], g[i + 2], g[i + 3]);
#pragma unroll
        for (int i = 0; i < 16; i += 4) st_v4(gdst + p.F + 2 * i, u[i], u[i + 1], u[i + 2], u[i + 3]);
      }
    } else if (MODE == kDgrad2) {
      // Without staging boxes (the fused backward): G and U of this row are read
      // from global memory; the loads of the next 32 columns are issued before
      // this chunk's arithmetic.
      uint32_t d[32];
      tc_ld_32x32b_x32(tacc + c, d);
      uint4 gn[4], un[4];
      if (valid && c + 32 < c_hi) {
        const __nv_bfloat16* gsrc = p.aux + grow * (2 * p.F) + t.n0 + c + 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          gn[i] = ld_v4(gsrc + 8 * i);
          un[i] = ld_v4(gsrc + p.F + 8 * i);
        }
      }
      tc_wait_ld();
      if (valid) {
        __nv_bfloat16* ddst = p.out0 + grow * (2 * p.F) + t.n0 + c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t gw[4] = {gcur[i].x, gcur[i].y, gcur[i].z, gcur[i].w};
          const uint32_t uw[4] = {ucur[i].x, ucur[i].y, ucur[i].z, ucur[i].w};
          uint32_t dgw[4], duw[4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float dg2[2], du2[2];
#pragma unroll
            for (int hbit = 0; hbit < 2; ++hbit) {
              const float G = hbit ? bf16hi(gw[qq]) : bf16lo(gw[qq]);
              const float U = hbit ? bf16hi(uw[qq]) : bf16lo(uw[qq]);
              swiglu_bwd(G, U, __uint_as_float(d[8 * i + 2 * qq + hbit]), dg2[hbit], du2[hbit]);
            }
            dgw[qq] = pack_bf16x2(dg2[0], dg2[1]);
            duw[qq] = pack_bf16x2(du2[0], du2[1]);
          }
          st_v4(ddst + 8 * i, dgw[0], dgw[1], dgw[2], dgw[3]);
          st_v4(ddst + p.F + 8 * i, duw[0], duw[1], duw[2], duw[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          gcur[i] = gn[i];
          ucur[i] = un[i];
        }
      }
    } else {  // kFwd2 (Y) or kDgrad1 (dXp): plain bf16 store, row stride H
      uint32_t d[32];
      tc_ld_32x32b_x32(tacc + c, d);
      tc_wait_ld();
      if (valid) {
        __nv_bfloat16* dst = p.out0 + grow * p.H + t.n0 + c;
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          st_v4(dst + i, pack_bf16x2(__uint_as_float(d[i]), __uint_as_float(d[i + 1])),
                pack_bf16x2(__uint_as_float(d[i + 2]), __uint_as_float(d[i + 3])),
                pack_bf16x2(__uint_as_float(d[i + 4]), __uint_as_float(d[i + 5])),
                pack_bf16x2(__uint_as_float(d[i + 6]), __uint_as_float(d[i + 7])));
      }
    }
  }
  if (MODE == kFwd2 && p.cmb.cnt != nullptr) combine_in_epilogue(p, t, grow, valid, half, c_lo, c_hi, lane);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ Maps maps,
                                                                   const GemmParams p) {
  using TR = ModeTraits<MODE>;
  constexpr int S = TR::kStages;
  constexpr uint32_t kAStep = TR::a_mn ? 2048u : 32u;
  constexpr uint32_t kBStep = TR::b_mn ? 2048u : 32u;
  constexpr uint32_t kIdesc256 = idesc_bf16_f32(BM, 256, TR::a_mn, TR::b_mn);
  constexpr uint32_t kIdesc128 = idesc_bf16_f32(BM, 128, TR::a_mn, TR::b_mn);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + S * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + TR::kStagingBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* ebar = tempty + 3;  // dgrad2: kEpiRing G/U chunk barriers per epilogue warp

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    for (int i = 0; i < kEpiRing * kEpiWarps && MODE == kDgrad2; ++i) mbar_init(&ebar[i], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = n_tiles<MODE>(p);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    uint32_t issued = 0;       // bit i: stage i was ever filled
    uint32_t last_parity = 0;  // bit i: parity of stage i's last fill
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const Tile t = decode<MODE>(p, tile);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1u, p.ws, 100 + MODE, abort_flag)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], stage_tx_bytes<MODE>(t.nw));
          uint8_t* sA = smem + s * kStageBytes;
          load_kblock<MODE>(p, maps, t, kb, sA, sA + kABytes, &full[s]);
        }
        __syncwarp();
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // Never leave with copies in flight: wait (bounded) for every stage's last fill.
    for (int i = 0; i < S; ++i)
      if ((issued >> i) & 1u) mbar_wait(&full[i], (last_parity >> i) & 1u, p.ws, 110 + MODE, nullptr);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const Tile t = decode<MODE>(p, tile);
      if (t.kblocks == 0) continue;  // empty expert (wgrad): the epilogue writes zeros
      if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, p.ws, 120 + MODE, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kAccStride;
      const uint32_t idesc = TR::router ? idesc_bf16_f32(BM, t.nw, TR::a_mn, TR::b_mn)
                                       : (t.nw == 256) ? kIdesc256 : kIdesc128;
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait(&full[s], ph, p.ws, 130 + MODE, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* sA = smem + s * kStageBytes;
        uint8_t* sB = sA + kABytes;
        // The expert's last k-block (weight gradients) may run past its rows:
        // only the K steps of 16 that hold valid rows are issued (clear_k_tail).
        int nkk = BK / 16;
        if (TR::wgrad) {
          const int valid = t.nrows - kb * BK;
          if (valid < BK) nkk = clear_k_tail(sA, sB, valid, t.nw, lane);
          __syncwarp();
        }
        if (elect_one()) {
          const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk < nkk) {
              const uint64_t ad = smem_desc_sw128(a0 + kk * kAStep, TR::a_mn ? kPanelBytes : 16, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + kk * kBStep, TR::b_mn ? kPanelBytes : 16, 1024);
              tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
            }
          }
          tc_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;    // which half of the columns
    const int row = q * 32 + lane;
    OutStager st;
    st.buf = staging + (warp - 2) * epi_stage_bytes<MODE>();
    if (MODE == kDgrad2) st.ebar = ebar + kEpiRing * (warp - 2);
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = decode<MODE>(p, tile);
      if (t.kblocks == 0) {
        if (TR::wgrad && p.sb != 2) {  // an empty second sub-batch leaves the first one's values
          const int NCall = (MODE == kWgrad13) ? 128 : t.nw;
          const int c_lo = half * (NCall / 2), c_hi = c_lo + NCall / 2;
          float* d0 = (MODE == kWgrad13) ? p.f0 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0
                                         : p.f0 + (static_cast<size_t>(t.e) * p.F + t.m0 + row) * p.H + t.n0;
          for (int c = c_lo; c < c_hi; c += 32) store_zero_f32(d0 + c);
          if (MODE == kWgrad13) {
            float* d1 = p.f1 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0;
            for (int c = c_lo; c < c_hi; c += 32) store_zero_f32(d1 + c);
          }
        }
        continue;
      }
      if (MODE == kDgrad2) dgrad2_prefetch(p, maps, t, q, half, lane, st);  // G/U need no accumulator
      if (!mbar_wait(&tfull[acc], acc_ph, p.ws, 140 + MODE, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      epilogue<MODE>(p, maps, t, tacc, q, half, lane, st);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
    // Bulk stores must finish reading shared memory (and land) before the CTA exits.
    if (TR::wgrad && lane == 0) bulk_wait_all();
    if (MODE == kDgrad2) st.drain(p.ws);  // no G/U load may land after the CTA is gone
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Two-SM pair tiles (tcgen05 cta_group::2).
//
// A cluster of two CTAs owns one 256 x N output tile: CTA r of the pair holds
// its 128 rows of A (the 128-row tile 2 pi + r of the expert, or rows
// m0 + 128 r of a weight gradient) and half of B (columns r N/2 .. of the
// tile; for the paired W1|W3 and dG|dU tiles, CTA 0 holds the W1 / dG half and
// CTA 1 the W3 / dU half).  One thread of the even CTA issues the MMAs, which
// read both CTAs' shared memory and write both CTAs' tensor memory (each CTA
// holds its own 128 rows x N of the accumulator), so each SM moves half of B
// into shared memory and reads a third less shared memory per MMA than a
// 128 x 256 single-CTA tile.
//
// Synchronisation per stage: each CTA's TMA loads complete on its own `full`
// barrier; the odd CTA's warp 1 waits for it (and clears a weight-gradient
// K tail in its own shared memory) and arrives on the even CTA's `pfull`; the
// even CTA's warp 1 waits for its own `full`, clears its own tail, waits on
// `pfull` and issues the MMAs.  MMA completion arrives on `empty` (stage free)
// and, after a tile's last k-block, on `tfull` in both CTAs (multicast commit).
// Both CTAs' epilogue warps arrive on the even CTA's `tempty` when they have
// read their accumulator.  Tile order and arithmetic are those of the
// single-CTA kernels, so results do not depend on the grid size either.
// ---------------------------------------------------------------------------
// Pipeline timeline of the pair kernels, for diagnosis only: compiled in with
// -DMOE_TIMELINE (never in a normal build).  With moe_debug_timeline() set,
// the pair kernel of the selected mode stamps its SM's cycle counter (clock64,
// cheap enough not to disturb the pipeline much) for every k-block
// n < cap of every CTA into buf[(cta * cap + n) * 5 + event]: 0 the producer
// found the stage free, 1 the MMA warp saw it land, 2 the leader saw the
// partner's stage (the relay: the odd CTA's arrive), 3 the MMAs and the commit
// were issued, 4 (first k-block of a tile) the leader got the accumulator.
#ifdef MOE_TIMELINE
__device__ unsigned long long* g_tl_buf = nullptr;
__device__ int g_tl_cap = 0;
__device__ int g_tl_mode = -1;
template <int MODE>
__device__ __forceinline__ void tl_mark(int n, int ev) {
  if (g_tl_mode == MODE && g_tl_buf != nullptr && n < g_tl_cap)
    g_tl_buf[(static_cast<size_t>(blockIdx.x) * g_tl_cap + n) * 5 + ev] = static_cast<unsigned long long>(clock64());
}
#define MOE_TL(n, ev) tl_mark<MODE>((n), (ev))
#else
#define MOE_TL(n, ev) ((void)0)
#endif

constexpr int kPairBHalfBytes = 128 * BK * 2;  // half of a 256-wide B tile
constexpr int kPairStageBytes = kABytes + kPairBHalfBytes;

template <int MODE>
struct PairTraits {
  static constexpr int kStages = MODE == kDgrad2 ? 5 : 6;  // dgrad2 gives a stage to its G/U chunk ring
  static constexpr int kStagingBytes = kEpiWarps * epi_stage_bytes<MODE>();
  static constexpr int kSmemBytes = kStages * kPairStageBytes + kStagingBytes + 1024 /*align*/ + 512 /*barriers*/;
};
// Shared memory of the staged per-expert tables (4 arrays of E + 1 ints).
inline size_t pair_table_bytes(int E) { return 4 * (static_cast<size_t>(E) + 1) * 4; }

template <int MODE>
__device__ __forceinline__ int pair_n_tiles(const GemmParams& p, const int* pairs) {
  const int nn = n_ntiles<MODE>(p);
  if (MODE == kWgrad13) return p.E * ((p.H + 255) / 256) * nn;
  if (MODE == kWgrad2) return p.E * ((p.F + 255) / 256) * nn;
  return pairs[p.E] * nn;
}

// This CTA's part of pair tile `tile`: row0 / nrows of its 128-row tile
// (forward, dgrad; nrows = 0 for the missing half of an expert's last pair) or
// its 128-row slice m0 of the weight gradient (m0 >= the extent: no rows).
// Per-expert tables of the pair kernels, staged in shared memory at launch.
struct ExpertTables {
  const int* pairs;   // [E + 1] first pair tile
  const int* counts;  // [E]
  const int* offsets; // [E]
  const int* tstart;  // [E]     first 128-row tile
};

template <int MODE>
__device__ __forceinline__ Tile pair_decode(const GemmParams& p, const ExpertTables& x, int tile, uint32_t rank) {
  Tile t;
  const int nn = n_ntiles<MODE>(p);
  int nt;
  if (ModeTraits<MODE>::wgrad) {
    // Order (expert, M pair, N tile), N fastest: the pairs running side by side
    // write whole rows of dW (long contiguous DRAM runs) and share A.
    const int MT2 = ((MODE == kWgrad13 ? p.H : p.F) + 255) / 256;
    t.e = tile / (MT2 * nn);
    const int rem = tile - t.e * MT2 * nn;
    const int mp = rem / nn;
    nt = rem - mp * nn;
    t.m0 = mp * 256 + 128 * static_cast<int>(rank);
    t.row0 = __ldg(p.offsets + t.e);  // weight gradients: no staged tables (their shared memory holds store boxes)
    t.nrows = __ldg(p.counts + t.e);
    subbatch_range(p, t.e, t.row0, t.nrows);
    t.kblocks = (t.nrows + BK - 1) / BK;
    t.mt = -1;
  } else {
    // Expert: the last e with pairs[e] * nn <= tile (empty experts own no pairs).
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (x.pairs[mid] * nn <= tile)
        lo = mid;
      else
        hi = mid;
    }
    const int e = lo;
    const int first = x.pairs[e];
    const int cnt = x.pairs[e + 1] - first;
    const int local = tile - nn * first;
    // (M pair, N tile) with N fastest: the clusters running side by side share
    // one expert's weights and a few 256-row blocks of A, so both stay in the L2
    // (with M fastest, a wave swept every row block of an expert once per N tile
    // and re-read A from DRAM two to three times).
    (void)cnt;
    const int mp = local / nn;
    nt = local - mp * nn;
    const int j = 2 * mp + static_cast<int>(rank);  // this CTA's 128-row tile of the expert
    const int n_e = x.counts[e];
    t.e = e;
    t.row0 = x.offsets[e] + kTileRows * j;
    t.nrows = max(0, min(kTileRows, n_e - kTileRows * j));
    t.m0 = 0;
    t.mt = x.tstart[e] + j;
    t.halfm = 0;
    const int rem = n_e - kTileRows * (j & ~1);  // rows left in this pair's 256-row block
    if (p.halfm_ok && rem <= kTileRows) {
      // M = 128 pair tile: CTA r takes rows [64 r, 64 r + 64) of the block.
      t.halfm = 1;
      t.row0 = x.offsets[e] + kTileRows * (j & ~1) + 64 * static_cast<int>(rank);
      t.nrows = max(0, min(64, rem - 64 * static_cast<int>(rank)));
    }
    const int K = (MODE == kFwd1 || MODE == kDgrad2) ? p.H : (MODE == kFwd2) ? p.F : 2 * p.F;
    t.kblocks = K / BK;
  }
  if (ModeTraits<MODE>::paired) {
    t.n0 = nt * 128;
    t.nw = 256;
  } else {
    t.n0 = nt * BN;
    t.nw = min(BN, n_extent<MODE>(p) - t.n0);
  }
  return t;
}

// TMA loads of one k-block of this CTA's half: A (its 128 rows) into sA, its
// half of B into sB.
template <int MODE>
__device__ __forceinline__ void load_kblock_pair(const GemmParams& p, const Maps& m, const Tile& t, int kb,
                                                 uint8_t* sA, uint8_t* sB, uint64_t* bar, uint32_t rank) {
  const int k0 = kb * BK;
  const int hb = t.nw / 2;  // B columns of this CTA
  const int r = static_cast<int>(rank);
  if (MODE == kFwd1) {
    if (sA != nullptr) tma_load_2d(sA, &m.a, bar, k0, t.row0);  // null: A is gathered from x
    const int y = t.e * p.H + k0;
    if (t.halfm) {
      // M = 128 tiles: CTA r holds W1 and W3 columns [n0 + 64 r, +64), so each lane
      // half of the accumulator has G and U of the same 64 features.
      tma_load_2d(sB, &m.b0, bar, t.n0 + 64 * r, y);
      tma_load_2d(sB + kPanelBytes, &m.b1, bar, t.n0 + 64 * r, y);
    } else if (p.panels2) {
      tma_load_3d(sB, r ? &m.b1_p2 : &m.b0_p2, bar, 0, y, t.n0 / 64);
    } else {
      const CUtensorMap* w = r ? &m.b1 : &m.b0;  // W1 (G columns) on CTA 0, W3 (U columns) on CTA 1
      tma_load_2d(sB, w, bar, t.n0, y);
      tma_load_2d(sB + kPanelBytes, w, bar, t.n0 + 64, y);
    }
  } else if (MODE == kFwd2) {
    if (sA != nullptr) tma_load_2d(sA, &m.a, bar, k0, t.row0);
    const int y = t.e * p.F + k0;
    if (p.panels2 && hb == 128)
      tma_load_3d(sB, &m.b0_p2, bar, 0, y, (t.n0 + r * hb) / 64);
    else
      for (int q = 0; q < hb / 64; ++q) tma_load_2d(sB + q * kPanelBytes, &m.b0, bar, t.n0 + r * hb + 64 * q, y);
  } else if (MODE == kDgrad2) {
    if (sA != nullptr) tma_load_2d(sA, &m.a, bar, k0, t.row0);
    tma_load_2d(sB, hb == 128 ? &m.b0 : &m.b2, bar, k0, t.e * p.F + t.n0 + r * hb);
  } else if (MODE == kDgrad1) {
    if (sA != nullptr) tma_load_2d(sA, &m.a, bar, k0, t.row0);
    const int yb = t.e * p.H + t.n0 + r * hb;
    if (k0 < p.F)
      tma_load_2d(sB, hb == 128 ? &m.b0 : &m.b2, bar, k0, yb);
    else
      tma_load_2d(sB, hb == 128 ? &m.b1 : &m.b3, bar, k0 - p.F, yb);
  } else if (MODE == kWgrad13) {
    const int y = t.row0 + k0;
    const int c = r ? p.F + t.n0 : t.n0;  // dG half on CTA 0, dU half on CTA 1
    if (p.panels2) {
      tma_load_3d(sA, &m.a_p2, bar, 0, y, t.m0 / 64);
      tma_load_3d(sB, &m.b0_p2, bar, 0, y, c / 64);
    } else {
      tma_load_2d(sA, &m.a, bar, t.m0, y);
      tma_load_2d(sA + kPanelBytes, &m.a, bar, t.m0 + 64, y);
      tma_load_2d(sB, &m.b0, bar, c, y);
      tma_load_2d(sB + kPanelBytes, &m.b0, bar, c + 64, y);
    }
  } else {  // kWgrad2
    const int y = t.row0 + k0;
    if (p.panels2) {
      tma_load_3d(sA, &m.a_p2, bar, 0, y, t.m0 / 64);
    } else {
      tma_load_2d(sA, &m.a, bar, t.m0, y);
      tma_load_2d(sA + kPanelBytes, &m.a, bar, t.m0 + 64, y);
    }
    if (p.panels2 && hb == 128)
      tma_load_3d(sB, &m.b0_p2, bar, 0, y, (t.n0 + r * hb) / 64);
    else
      for (int q = 0; q < hb / 64; ++q) tma_load_2d(sB + q * kPanelBytes, &m.b0, bar, t.n0 + r * hb + 64 * q, y);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) pair_gemm_kernel(const __grid_constant__ Maps maps,
                                                                const GemmParams p) {
  using TR = ModeTraits<MODE>;
  constexpr int S = PairTraits<MODE>::kStages;
  constexpr uint32_t kAStep = TR::a_mn ? 2048u : 32u;
  constexpr uint32_t kBStep = TR::b_mn ? 2048u : 32u;
  constexpr uint32_t kIdesc256 = idesc_bf16_f32(256, 256, TR::a_mn, TR::b_mn);
  constexpr uint32_t kIdesc128 = idesc_bf16_f32(256, 128, TR::a_mn, TR::b_mn);
  // M = 128 pair tiles: 64 rows per CTA; the accumulator's lanes 0-63 hold the
  // first half of the N columns of those rows, lanes 64-127 the second half.
  constexpr uint32_t kIdescH256 = idesc_bf16_f32(128, 256, TR::a_mn, TR::b_mn);
  constexpr uint32_t kIdescH128 = idesc_bf16_f32(128, 128, TR::a_mn, TR::b_mn);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + S * kPairStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + PairTraits<MODE>::kStagingBytes);
  uint64_t* empty = full + S;
  uint64_t* pfull = empty + S;
  uint64_t* tfull = pfull + S;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* ebar = tempty + 3;  // dgrad2: kEpiRing G/U chunk barriers per epilogue warp
  int* tab = reinterpret_cast<int*>(smem + S * kPairStageBytes + PairTraits<MODE>::kStagingBytes + 512);
  ExpertTables xt;
  xt.pairs = tab;
  xt.counts = tab + (p.E + 1);
  xt.offsets = tab + 2 * (p.E + 1);
  xt.tstart = tab + 3 * (p.E + 1);
  for (int e = threadIdx.x; e <= p.E && !TR::wgrad; e += blockDim.x) {
    tab[e] = __ldg(p.pairs + e);
    tab[(p.E + 1) + e] = e < p.E ? __ldg(p.counts + e) : 0;
    tab[2 * (p.E + 1) + e] = __ldg(p.offsets + e);
    tab[3 * (p.E + 1) + e] = __ldg(p.tiles + 1 + e);
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // rank in the pair
  const bool leader = (rank == 0);
  constexpr uint32_t pair_leader = 0;
  constexpr uint16_t kEmptyMask = 0x3;  // commits arrive in both CTAs of the pair
  constexpr uint16_t tfull_mask = 0x3;
  // Gathered A (GEMM1 with the dispatch fused): a stage is full after the B
  // bytes and the 32 producer lanes' cp.async arrivals.
  const bool gather_a = (MODE == kFwd1) && p.gather;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], gather_a ? 1 + 32 : 1);
      mbar_init(&empty[i], 1);
      mbar_init(&pfull[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * kEpiWarps);
    }
    for (int i = 0; i < kEpiRing * kEpiWarps && MODE == kDgrad2; ++i) mbar_init(&ebar[i], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = pair_n_tiles<MODE>(p, xt.pairs);
  const int npairs = gridDim.x / 2;  // clusters
  const int pid = blockIdx.x / 2;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (every CTA)
    int s = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, last_parity = 0;
    bool ok = true;
    int tl_n = 0;  // k-blocks so far (timeline index)
    (void)tl_n;
    for (int tile = pid; tile < ntiles && ok; tile += npairs) {
      const Tile t = pair_decode<MODE>(p, xt, tile, rank);
      const bool gather = gather_a;
      // gather: lane l copies 16-byte chunk (l & 7) of rows 4 i + (l >> 3), i < 32, of the
      // tile; src[i] is the token of that row (rows past R read token 0 and are never stored).
      int src[32];
      if (gather) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int r = t.row0 + 4 * i + (lane >> 3);
          const int tok = r < p.R ? __ldg(p.row_src + r) : 0;
          src[i] = (tok >= 0 && tok < p.T) ? tok : 0;
        }
      }
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait_cluster(&empty[s], ph ^ 1u, p.ws, 200 + MODE, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) MOE_TL(tl_n, 0);
        ++tl_n;
        uint8_t* sA = smem + s * kPairStageBytes;
        if (gather) {
          if (elect_one()) {
            mbar_arrive_expect_tx(&full[s], t.nw * 64);  // B only: A arrives by cp.async
            load_kblock_pair<MODE>(p, maps, t, kb, nullptr, sA + kABytes, &full[s], rank);
          }
          __syncwarp();
          // A: 128 rows x 128 bytes of x into the 128-byte-swizzled stage (chunk c of
          // row r at chunk c ^ (r & 7)); a warp-wide copy covers four whole rows.
          const int c = lane & 7;
          const uint32_t a_base = smem_u32(sA);
          const __nv_bfloat16* xk = p.x + kb * BK + 8 * c;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int r = 4 * i + (lane >> 3);
            cp_async_16(a_base + r * 128 + ((c ^ (r & 7)) << 4), xk + static_cast<size_t>(src[i]) * p.H);
          }
          cp_async_mbar_arrive_noinc(&full[s]);
        } else if (elect_one()) {
          if (t.halfm) {  // M = 128 pair tile: 64 A rows per CTA
            mbar_arrive_expect_tx(&full[s], kABytes / 2 + t.nw * 64);
            tma_load_2d(sA, &maps.a64, &full[s], kb * BK, t.row0);
            load_kblock_pair<MODE>(p, maps, t, kb, nullptr, sA + kABytes, &full[s], rank);
          } else {
            mbar_arrive_expect_tx(&full[s], kABytes + t.nw * 64);
            load_kblock_pair<MODE>(p, maps, t, kb, sA, sA + kABytes, &full[s], rank);
          }
        }
        __syncwarp();
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    for (int i = 0; i < S; ++i)
      if ((issued >> i) & 1u) mbar_wait(&full[i], (last_parity >> i) & 1u, p.ws, 210 + MODE, nullptr);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA) / relay (odd CTA)
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    bool ok = true;
    int tl_n = 0;  // k-blocks so far (timeline index)
    (void)tl_n;
    const uint32_t pfull_leader = mapa_shared(smem_u32(pfull), pair_leader);
    for (int tile = pid; tile < ntiles && ok; tile += npairs) {
      const Tile t = pair_decode<MODE>(p, xt, tile, rank);
      if (t.kblocks == 0) continue;  // empty expert (weight gradients): the epilogue writes zeros
      if (leader) {
        if (!mbar_wait_cluster(&tempty[acc], acc_ph ^ 1u, p.ws, 220 + MODE, abort_flag)) break;
        tc_fence_after();
        if (lane == 0) MOE_TL(tl_n, 4);
      }
      const uint32_t d_tmem = tmem_base + acc * kAccStride;
      const uint32_t idesc = t.halfm ? ((t.nw == 256) ? kIdescH256 : kIdescH128) : (t.nw == 256) ? kIdesc256 : kIdesc128;
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait(&full[s], ph, p.ws, 230 + MODE, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) MOE_TL(tl_n, 1);
        uint8_t* sA = smem + s * kPairStageBytes;
        uint8_t* sB = sA + kABytes;
        int nkk = BK / 16;
        if (TR::wgrad) {
          const int valid = t.nrows - kb * BK;
          if (valid < BK) nkk = clear_k_tail(sA, sB, valid, t.nw / 2, lane);
        }
        // Gathered A rows of a row block's first N tile go out to Xp (the backward
        // reads them); the store reads the stage before the stage is released.
        const bool store_xp = (MODE == kFwd1) && p.gather && t.n0 == 0 && t.nrows > 0;
        __syncwarp();
        if (!leader) {
          if (lane == 0) {
            if (gather_a) fence_proxy_async_smem();  // the cp.async rows, for the MMA and the Xp store
            if (store_xp) {
              tma_store_2d(&maps.a, sA, kb * BK, t.row0);
              bulk_commit();
              bulk_wait_read<0>();
            }
            mbar_arrive_cluster(pfull_leader + s * 8);
            MOE_TL(tl_n, 2);
          }
          __syncwarp();
        } else {
          if (!mbar_wait_cluster(&pfull[s], ph, p.ws, 240 + MODE, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) MOE_TL(tl_n, 2);
          tc_fence_after();
          // One elected thread issues the Xp store, the MMAs and the commits, so each
          // commit tracks that thread's MMAs and the store's bulk group.
          if (elect_one()) {
            if (gather_a) fence_proxy_async_smem();  // the cp.async rows, for the MMA and the Xp store
            if (store_xp) {
              tma_store_2d(&maps.a, sA, kb * BK, t.row0);
              bulk_commit();
            }
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if (kk < nkk) {
                const uint64_t ad = smem_desc_sw128(a0 + kk * kAStep, TR::a_mn ? kPanelBytes : 16, 1024);
                const uint64_t bd = smem_desc_sw128(b0 + kk * kBStep, TR::b_mn ? kPanelBytes : 16, 1024);
                tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
              }
            }
            if (store_xp) bulk_wait_read<0>();
            tc_commit_pair(&empty[s], kEmptyMask);
            MOE_TL(tl_n, 3);
          }
          __syncwarp();
        }
        ++tl_n;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (leader) {
        if (elect_one()) tc_commit_pair(&tfull[acc], tfull_mask);
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
    if ((MODE == kFwd1) && p.gather) bulk_wait_all();  // Xp stores complete before exit (any lane)
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs, own rows)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int mext = (MODE == kWgrad13) ? p.H : p.F;
    OutStager st;
    st.buf = staging + (warp - 2) * epi_stage_bytes<MODE>();
    if (MODE == kDgrad2) st.ebar = ebar + kEpiRing * (warp - 2);
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), pair_leader);
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int tile = pid; tile < ntiles; tile += npairs) {
      const Tile t = pair_decode<MODE>(p, xt, tile, rank);
      const bool mine = TR::wgrad ? (t.m0 < mext) : (t.nrows > 0);
      if (t.kblocks == 0) {
        if (TR::wgrad && mine && p.sb != 2) {  // an empty second sub-batch leaves the first one's values
          const int NCall = (MODE == kWgrad13) ? 128 : t.nw;
          const int c_lo = half * (NCall / 2), c_hi = c_lo + NCall / 2;
          float* d0 = (MODE == kWgrad13) ? p.f0 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0
                                         : p.f0 + (static_cast<size_t>(t.e) * p.F + t.m0 + row) * p.H + t.n0;
          for (int c = c_lo; c < c_hi; c += 32) store_zero_f32(d0 + c);
          if (MODE == kWgrad13) {
            float* d1 = p.f1 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0;
            for (int c = c_lo; c < c_hi; c += 32) store_zero_f32(d1 + c);
          }
        }
        continue;
      }
      // M = 128 pair tile: lane quarter q holds rows 32 (q & 1) + lane and the
      // (q >> 1)-th half of the tile's columns, at accumulator columns [0, N/2).
      Tile te = t;
      int qe = q;
      if (t.halfm) {
        const int hw = ModeTraits<MODE>::paired ? 64 : t.nw / 2;
        te.n0 = t.n0 + (q >> 1) * hw;
        if (!ModeTraits<MODE>::paired) te.nw = hw;
        qe = q & 1;
      }
      const bool mine_e = mine && (!t.halfm || 32 * qe < t.nrows);
      if (MODE == kDgrad2 && mine_e) dgrad2_prefetch(p, maps, te, qe, half, lane, st);  // G/U need no accumulator
      if (!mbar_wait_cluster(&tfull[acc], acc_ph, p.ws, 250 + MODE, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      if (mine_e) epilogue<MODE>(p, maps, te, tacc, qe, half, lane, st);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_cluster(tempty_leader + acc * 8);
      }
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
    if (TR::wgrad && lane == 0) bulk_wait_all();
    if (MODE == kDgrad2) st.drain(p.ws);  // no G/U load may land after the CTA is gone
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its pair may still use its shared or tensor memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Fused persistent forward: dispatch row gathers, GEMM1 (+SwiGLU) tiles and
// GEMM2 tiles in one launch.
//
// "UniEP: Unified Expert-Parallel MoE MegaKernel for LLM Training", section 3:
// persistent workers (one CTA per SM) take tasks from a global atomic cursor
// over a linearised task space -- dispatch tasks first, then computation tasks
// (here: row gathers, then GEMM1 tiles, then GEMM2 tiles, each in ascending
// expert order, the priority order of section 4) -- and a scoreboard in global
// memory says when a computation may start: a GEMM1 tile once its 128 rows are
// gathered, a GEMM2 tile once every GEMM1 tile of its rows has stored h.  A task
// waits only on tasks with smaller indices, which running CTAs have already
// taken, so progress never needs every CTA to be resident.
//
// Inside a CTA the producer warp takes the tasks and hands them to the MMA warp
// and the epilogue warps through a small ring in shared memory.  The epilogue
// warps also execute the gather tasks (one warp per row, 16-byte vectors).
// ---------------------------------------------------------------------------
constexpr int kTaskRing = 4;
constexpr int kTaskEnd = -1;
constexpr int kTaskGather = -2;

struct FusedFwdParams {
  GemmParams p1;  // GEMM1: out0 = h, out1 = GU
  GemmParams p2;  // GEMM2: out0 = Y
  const uint4* x;
  uint4* Xp;
  const int32_t* row_src;
  int T;
  int32_t* cursor;
  int32_t* cnt_gather;  // per 128-row tile: epilogue warps done gathering its rows
  int32_t* cnt_g1;      // per 128-row tile: GEMM1 epilogue warps done storing h
  int drop_task;        // failure injection: task + 1 whose gather signal is withheld (0: none)
};

struct FusedFwdMaps {
  Maps g1;
  Maps g2;
};

struct FwdTask {
  int kind;  // kTaskGather, kFwd1 or kFwd2
  Tile t;
};

__device__ __forceinline__ FwdTask fwd_decode(const FusedFwdParams& f, int task) {
  const int nmt = __ldg(f.p1.tiles);
  const int nn1 = f.p1.F / 128;
  FwdTask k;
  if (task < nmt) {
    const int4 en = __ldg(reinterpret_cast<const int4*>(f.p1.tiles + tiles_entry_base(f.p1.E)) + task);
    k.kind = kTaskGather;
    k.t.e = en.x;
    k.t.row0 = en.y;
    k.t.nrows = en.z;
    k.t.mt = task;
    k.t.m0 = k.t.n0 = k.t.nw = k.t.kblocks = 0;
  } else if (task < nmt * (1 + nn1)) {
    k.kind = kFwd1;
    k.t = decode<kFwd1>(f.p1, task - nmt);
  } else {
    k.kind = kFwd2;
    k.t = decode<kFwd2>(f.p2, task - nmt * (1 + nn1));
  }
  return k;
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Dispatch of one 128-row tile by one epilogue warp (rows ew, ew+8, ...):
// Xp[r] = x[row_src[r]] ("MoonEP": zero-copy dispatch into the expert-grouped
// layout); a padding row (row_src = -1) is written as zeros.
__device__ __forceinline__ void gather_rows_task(const FusedFwdParams& f, const Tile& t, int ew, int lane) {
  const int hv = f.p1.H / 8;
  for (int i = ew; i < t.nrows; i += kEpiWarps) {
    const int r = t.row0 + i;
    const int tok = __ldg(f.row_src + r);
    if (tok == -1) {
      uint4* dst = f.Xp + static_cast<size_t>(r) * hv;
      for (int v = lane; v < hv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    if (tok < 0 || tok >= f.T) {
      if (lane == 0) report(f.p1.ws, MOE_ERR_BOUNDS, 20, r);
      continue;
    }
    const uint4* src = f.x + static_cast<size_t>(tok) * hv;
    uint4* dst = f.Xp + static_cast<size_t>(r) * hv;
    // 8 x 16 B in flight per lane (a 4 KB row per pass over the warp).
    int v = lane;
    for (; v + 224 < hv; v += 256) {
      uint4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ld_nc_v4(src + v + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[v + 32 * u] = a[u];
    }
    for (; v < hv; v += 32) dst[v] = ld_nc_v4(src + v);
  }
}

__global__ void __launch_bounds__(kThreads, 1) fused_forward_kernel(const __grid_constant__ FusedFwdMaps maps,
                                                                    const FusedFwdParams f) {
  constexpr int S = 4;
  constexpr uint32_t kIdesc256 = idesc_bf16_f32(BM, 256, false, true);
  constexpr uint32_t kIdesc128 = idesc_bf16_f32(BM, 128, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* rfull = tempty + 2;
  uint64_t* rempty = rfull + kTaskRing;
  volatile int* ring = reinterpret_cast<volatile int*>(rempty + kTaskRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kTaskRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* ws = f.p1.ws;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    for (int i = 0; i < kTaskRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 1 + kEpiWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nmt = __ldg(f.p1.tiles);
  const int nn1 = f.p1.F / 128;
  const int nn2 = (f.p1.H + BN - 1) / BN;
  const int total = nmt * (1 + nn1 + nn2);

  if (warp == 0) {
    // ------------------------------------------------------------ producer + task fetch
    int s = 0, slot = 0;
    uint32_t ph = 0, rph = 0;
    uint32_t issued = 0, last_parity = 0;
    // The next task id is fetched one task ahead, so the atomic's round trip
    // overlaps the current task's work.
    int next = (lane == 0) ? atomicAdd(f.cursor, 1) : 0;
    while (true) {
      if (!mbar_wait(&rempty[slot], rph ^ 1u, ws, 150, abort_flag)) break;
      int task = 0;
      if (lane == 0) {
        task = next;
        if (task >= total || *abort_flag) task = kTaskEnd;
        if (task != kTaskEnd) next = atomicAdd(f.cursor, 1);
        ring[slot] = task;
      }
      task = __shfl_sync(0xffffffffu, task, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[slot]);
      if (++slot == kTaskRing) {
        slot = 0;
        rph ^= 1u;
      }
      if (task == kTaskEnd) break;
      const FwdTask k = fwd_decode(f, task);
      if (k.kind == kTaskGather) continue;
      // Scoreboard: the tile's input rows must be complete.
      const bool g1 = (k.kind == kFwd1);
      if (!wait_counter(g1 ? f.cnt_gather + k.t.mt : f.cnt_g1 + k.t.mt, g1 ? kEpiWarps : nn1 * kEpiWarps, ws,
                        g1 ? 151 : 152, abort_flag))
        continue;  // abort: the consumers see the flag and stop
      fence_proxy_async_global();
      for (int kb = 0; kb < k.t.kblocks; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1u, ws, 153, abort_flag)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], kABytes + k.t.nw * 128);
          uint8_t* sA = smem + s * kStageBytes;
          if (g1)
            load_kblock<kFwd1>(f.p1, maps.g1, k.t, kb, sA, sA + kABytes, &full[s]);
          else
            load_kblock<kFwd2>(f.p2, maps.g2, k.t, kb, sA, sA + kABytes, &full[s]);
        }
        __syncwarp();
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    for (int i = 0; i < S; ++i)
      if ((issued >> i) & 1u) mbar_wait(&full[i], (last_parity >> i) & 1u, ws, 154, nullptr);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0, slot = 0, acc = 0;
    uint32_t ph = 0, rph = 0, acc_ph = 0;
    bool ok = true;
    while (ok) {
      if (!mbar_wait(&rfull[slot], rph, ws, 155, abort_flag)) break;
      const int task = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[slot]);
      if (++slot == kTaskRing) {
        slot = 0;
        rph ^= 1u;
      }
      if (task == kTaskEnd) break;
      const FwdTask k = fwd_decode(f, task);
      if (k.kind == kTaskGather) continue;
      if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, ws, 156, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kAccStride;
      const uint32_t idesc = (k.t.nw == 256) ? kIdesc256 : kIdesc128;
      for (int kb = 0; kb < k.t.kblocks; ++kb) {
        if (!mbar_wait(&full[s], ph, ws, 157, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t a0 = smem_u32(smem + s * kStageBytes), b0 = a0 + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a0 + kk * 32u, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b0 + kk * 2048u, kPanelBytes, 1024);
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
          }
          tc_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ epilogue + gathers
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    OutStager st;  // unused by the forward modes
    st.buf = nullptr;
    int slot = 0, acc = 0;
    uint32_t rph = 0, acc_ph = 0;
    while (true) {
      if (!mbar_wait(&rfull[slot], rph, ws, 158, abort_flag)) break;
      const int task = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[slot]);
      if (++slot == kTaskRing) {
        slot = 0;
        rph ^= 1u;
      }
      if (task == kTaskEnd) break;
      const FwdTask k = fwd_decode(f, task);
      if (k.kind == kTaskGather) {
        gather_rows_task(f, k.t, ew, lane);
        if (task + 1 != f.drop_task) signal_counter(f.cnt_gather + k.t.mt, lane);
        continue;
      }
      if (!mbar_wait(&tfull[acc], acc_ph, ws, 159, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      if (k.kind == kFwd1)
        epilogue<kFwd1>(f.p1, maps.g1, k.t, tacc, q, half, lane, st);
      else
        epilogue<kFwd2>(f.p2, maps.g2, k.t, tacc, q, half, lane, st);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
      if (k.kind == kFwd1) signal_counter(f.cnt_g1 + k.t.mt, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Fused persistent forward on two-SM pair tiles: the same task space as
// fused_forward_kernel -- dispatch gathers, then GEMM1 (+SwiGLU) tiles, then
// GEMM2 tiles, expert-ascending -- with a task of each kind covering one
// 256-row pair of 128-row tiles, and the pair-tile pipeline of
// pair_gemm_kernel for the GEMM tasks.
//
// The even CTA's producer warp takes the task ids from the global cursor and
// writes each into the task rings of both CTAs (a shared::cluster store into
// the odd CTA's ring, released with the arrive on its `rfull`).  Every other
// role warp of both CTAs reads its own ring and releases the slot on the even
// CTA's `rempty` (count 9 + 10).  A gather task has each CTA gather the rows
// of its own 128-row tile; a GEMM task has each CTA's producer wait on the
// scoreboard counters of its own rows ("UniEP", section 3, Scoreboard-based
// Synchronization: a GEMM1 tile once its rows are gathered, a GEMM2 tile once
// every GEMM1 tile of its rows has stored h).  Tasks wait only on smaller task
// indices, so progress needs no more pairs than the ones resident.
// ---------------------------------------------------------------------------
constexpr int kFusedPairStages = 6;

struct PairFwdTask {
  int kind;  // kTaskGather, kFwd1, kFwd2 or kTaskEnd
  Tile t;    // this CTA's part
};

// Task order: the gathers of every pair first, then the GEMM1 tiles, then the
// GEMM2 tiles, each in ascending expert order ("UniEP", section 4: dispatch
// before computation).  (Interleaving an expert's gathers with the previous
// experts' GEMM tiles measured slower: the GEMM tiles then wait on gathers
// still in flight.)
__device__ __forceinline__ PairFwdTask fwd_pair_decode(const FusedFwdParams& f, const ExpertTables& x, int task,
                                                       uint32_t rank) {
  const int P = x.pairs[f.p1.E];
  const int nn1 = f.p1.F / 128;
  PairFwdTask k;
  if (task < P) {  // gather of pair `task`: this CTA's 128-row tile of it
    int lo = 0, hi = f.p1.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (x.pairs[mid] <= task)
        lo = mid;
      else
        hi = mid;
    }
    const int e = lo;
    const int j = 2 * (task - x.pairs[e]) + static_cast<int>(rank);
    k.kind = kTaskGather;
    k.t.e = e;
    k.t.row0 = x.offsets[e] + kTileRows * j;
    k.t.nrows = max(0, min(kTileRows, x.counts[e] - kTileRows * j));
    k.t.mt = x.tstart[e] + j;
    k.t.m0 = k.t.n0 = k.t.nw = k.t.kblocks = 0;
  } else if (task < P * (1 + nn1)) {
    k.kind = kFwd1;
    k.t = pair_decode<kFwd1>(f.p1, x, task - P, rank);
  } else {
    k.kind = kFwd2;
    k.t = pair_decode<kFwd2>(f.p2, x, task - P * (1 + nn1), rank);
  }
  return k;
}

__global__ void __launch_bounds__(kThreads, 1) fused_forward_pair_kernel(const __grid_constant__ FusedFwdMaps maps,
                                                                         const FusedFwdParams f) {
  constexpr int S = kFusedPairStages;
  constexpr uint32_t kIdesc256 = idesc_bf16_f32(256, 256, false, true);
  constexpr uint32_t kIdesc128 = idesc_bf16_f32(256, 128, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kPairStageBytes);
  uint64_t* empty = full + S;
  uint64_t* pfull = empty + S;
  uint64_t* tfull = pfull + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* rfull = tempty + 2;
  uint64_t* rempty = rfull + kTaskRing;
  volatile int* ring = reinterpret_cast<volatile int*>(rempty + kTaskRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kTaskRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tab = reinterpret_cast<int*>(smem + S * kPairStageBytes + 512);
  const int E = f.p1.E;
  ExpertTables xt;
  xt.pairs = tab;
  xt.counts = tab + (E + 1);
  xt.offsets = tab + 2 * (E + 1);
  xt.tstart = tab + 3 * (E + 1);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    tab[e] = __ldg(f.p1.pairs + e);
    tab[(E + 1) + e] = e < E ? __ldg(f.p1.counts + e) : 0;
    tab[2 * (E + 1) + e] = __ldg(f.p1.offsets + e);
    tab[3 * (E + 1) + e] = __ldg(f.p1.tiles + 1 + e);
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  WsHeader* ws = f.p1.ws;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&pfull[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * kEpiWarps);
    }
    for (int i = 0; i < kTaskRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], (1 + kEpiWarps) + (2 + kEpiWarps));  // even CTA: MMA + epilogue; odd: all role warps
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int P = xt.pairs[E];
  const int nn1 = f.p1.F / 128;
  const int nn2 = (f.p1.H + BN - 1) / BN;
  const int total = P * (1 + nn1 + nn2);
  const uint32_t rempty_leader = mapa_shared(smem_u32(rempty), 0);

  // Next task of the ring: the even CTA's producer fills slots, every other role
  // warp of both CTAs consumes them.  Returns kTaskEnd when done or aborted.
  auto consume = [&](int& slot, uint32_t& rph, int where) -> int {
    const bool ok = leader ? mbar_wait(&rfull[slot], rph, ws, where, abort_flag)
                           : mbar_wait_acq_cluster(&rfull[slot], rph, ws, where, abort_flag);
    int task = kTaskEnd;
    if (ok) task = ring[slot];
    __syncwarp();
    if (ok && lane == 0) {
      if (leader)
        mbar_arrive(&rempty[slot]);
      else
        mbar_arrive_cluster(rempty_leader + slot * 8);
    }
    if (++slot == kTaskRing) {
      slot = 0;
      rph ^= 1u;
    }
    return task;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ task fetch (even CTA) + producer (both)
    int s = 0, slot = 0;
    uint32_t ph = 0, rph = 0;
    uint32_t issued = 0, last_parity = 0;
    const uint32_t ring_peer = mapa_shared(smem_u32(const_cast<int*>(ring)), 1);
    const uint32_t rfull_peer = mapa_shared(smem_u32(rfull), 1);
    int next = (leader && lane == 0) ? atomicAdd(f.cursor, 1) : 0;
    while (true) {
      int task;
      if (leader) {
        if (!mbar_wait(&rempty[slot], rph ^ 1u, ws, 180, abort_flag)) break;
        task = 0;
        if (lane == 0) {
          task = next;
          if (task >= total || *abort_flag) task = kTaskEnd;
          if (task != kTaskEnd) next = atomicAdd(f.cursor, 1);
          ring[slot] = task;
          st_shared_cluster_u32(ring_peer + slot * 4, static_cast<uint32_t>(task));
        }
        task = __shfl_sync(0xffffffffu, task, 0);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&rfull[slot]);
          mbar_arrive_release_cluster(rfull_peer + slot * 8);
        }
        if (++slot == kTaskRing) {
          slot = 0;
          rph ^= 1u;
        }
      } else {
        task = consume(slot, rph, 181);
      }
      if (task == kTaskEnd) break;
      const PairFwdTask k = fwd_pair_decode(f, xt, task, rank);
      if (k.kind == kTaskGather) continue;
      const bool g1 = (k.kind == kFwd1);
      // Scoreboard: this CTA's input rows must be complete.
      if (k.t.nrows > 0) {
        if (!wait_counter(g1 ? f.cnt_gather + k.t.mt : f.cnt_g1 + k.t.mt, g1 ? kEpiWarps : nn1 * kEpiWarps, ws,
                          g1 ? 182 : 183, abort_flag))
          continue;
        fence_proxy_async_global();
      }
      for (int kb = 0; kb < k.t.kblocks; ++kb) {
        if (!mbar_wait_cluster(&empty[s], ph ^ 1u, ws, 184, abort_flag)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], kABytes + k.t.nw * 64);
          uint8_t* sA = smem + s * kPairStageBytes;
          if (g1)
            load_kblock_pair<kFwd1>(f.p1, maps.g1, k.t, kb, sA, sA + kABytes, &full[s], rank);
          else
            load_kblock_pair<kFwd2>(f.p2, maps.g2, k.t, kb, sA, sA + kABytes, &full[s], rank);
        }
        __syncwarp();
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    for (int i = 0; i < S; ++i)
      if ((issued >> i) & 1u) mbar_wait(&full[i], (last_parity >> i) & 1u, ws, 185, nullptr);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA) / relay (odd CTA)
    int s = 0, slot = 0, acc = 0;
    uint32_t ph = 0, rph = 0, acc_ph = 0;
    bool ok = true;
    const uint32_t pfull_leader = mapa_shared(smem_u32(pfull), 0);
    while (ok) {
      const int task = consume(slot, rph, 186);
      if (task == kTaskEnd) break;
      const PairFwdTask k = fwd_pair_decode(f, xt, task, rank);
      if (k.kind == kTaskGather) continue;
      if (leader) {
        if (!mbar_wait_cluster(&tempty[acc], acc_ph ^ 1u, ws, 187, abort_flag)) break;
        tc_fence_after();
      }
      const uint32_t d_tmem = tmem_base + acc * kAccStride;
      const uint32_t idesc = (k.t.nw == 256) ? kIdesc256 : kIdesc128;
      for (int kb = 0; kb < k.t.kblocks; ++kb) {
        if (!mbar_wait(&full[s], ph, ws, 188, abort_flag)) {
          ok = false;
          break;
        }
        if (!leader) {
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(pfull_leader + s * 8);
          __syncwarp();
        } else {
          if (!mbar_wait_cluster(&pfull[s], ph, ws, 189, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t a0 = smem_u32(smem + s * kPairStageBytes), b0 = a0 + kABytes;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(a0 + kk * 32u, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + kk * 2048u, kPanelBytes, 1024);
              tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
            }
            tc_commit_pair(&empty[s]);
          }
          __syncwarp();
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (leader) {
        if (elect_one()) tc_commit_pair(&tfull[acc]);
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ epilogue + gathers (both CTAs)
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    OutStager st;  // unused by the forward modes
    st.buf = nullptr;
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
    int slot = 0, acc = 0;
    uint32_t rph = 0, acc_ph = 0;
    while (true) {
      const int task = consume(slot, rph, 190);
      if (task == kTaskEnd) break;
      const PairFwdTask k = fwd_pair_decode(f, xt, task, rank);
      if (k.kind == kTaskGather) {
        if (k.t.nrows > 0) {
          gather_rows_task(f, k.t, ew, lane);
          if (task + 1 != f.drop_task) signal_counter(f.cnt_gather + k.t.mt, lane);
        }
        continue;
      }
      if (!mbar_wait_cluster(&tfull[acc], acc_ph, ws, 191, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      if (k.t.nrows > 0) {
        if (k.kind == kFwd1)
          epilogue<kFwd1>(f.p1, maps.g1, k.t, tacc, q, half, lane, st);
        else
          epilogue<kFwd2>(f.p2, maps.g2, k.t, tacc, q, half, lane, st);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_cluster(tempty_leader + acc * 8);
      }
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
      if (k.kind == kFwd1 && k.t.nrows > 0) signal_counter(f.cnt_g1 + k.t.mt, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Fused persistent backward: dgrad GEMM2 (+SwiGLU backward), dgrad GEMM1 and
// both weight-gradient Transposed GroupGEMMs in one launch.
//
// The weight-gradient tiles are bound by their fp32 stores to HBM, the dgrad
// tiles by the tensor cores and the operand feed, so the task list interleaves
// them, expert by expert, with a skew of kBwdSkew experts: stage s holds the
// dgrad2 tiles of expert s and then the dgrad1, wgrad13 and wgrad2 tiles of
// expert s - kBwdSkew.  Scoreboard ("UniEP: Unified Expert-Parallel MoE
// MegaKernel for LLM Training", section 3): a dgrad1 tile needs every dgrad2
// tile of its 128 rows, a wgrad13 tile needs every dgrad2 tile of its expert;
// the dgrad2 epilogue warps count themselves done per 128-row tile and per
// expert.  As in the forward, a task waits only on smaller task indices, and a
// producer fetches its next task id one task ahead (still in increasing order).
// ---------------------------------------------------------------------------
constexpr int kBwdSkew = 2;
constexpr int kBwdStages = 4;

struct FusedBwdParams {
  GemmParams d2;   // out0 = dGU, aux = GU
  GemmParams d1;   // out0 = dXp
  GemmParams w13;  // f0 = dW1, f1 = dW3
  GemmParams w2;   // f0 = dW2
  int32_t* cursor;
  int32_t* cnt_d2;  // per 128-row tile: dgrad2 epilogue warps done storing dG, dU
  int32_t* cnt_e;   // per expert: the same count over all of the expert's tiles
};

struct FusedBwdMaps {
  Maps d2, d1, w13, w2;
};

struct BwdTask {
  int kind;  // kDgrad2, kDgrad1, kWgrad13, kWgrad2
  Tile t;
};

__device__ __forceinline__ int bwd_stage_start(const int32_t* tiles, int E, int s, int nnF2, int nnH2, int per_w) {
  const int a = min(s, E);
  const int b = max(0, min(s - kBwdSkew, E));
  return nnF2 * __ldg(tiles + 1 + a) + nnH2 * __ldg(tiles + 1 + b) + per_w * b;
}

__device__ __forceinline__ BwdTask bwd_decode(const FusedBwdParams& f, int task) {
  const GemmParams& p = f.d2;
  const int E = p.E;
  const int nnF2 = (p.F + BN - 1) / BN;   // dgrad2 N tiles
  const int nnH2 = (p.H + BN - 1) / BN;   // dgrad1 / wgrad2 N tiles
  const int n_w13 = (p.H / BM) * (p.F / 128);
  const int n_w2 = (p.F / BM) * nnH2;
  const int per_w = n_w13 + n_w2;
  // Binary search of the stage s with start(s) <= task < start(s + 1).
  int lo = 0, hi = E + kBwdSkew;  // stages 0 .. E + kBwdSkew - 1
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (bwd_stage_start(p.tiles, E, mid, nnF2, nnH2, per_w) <= task)
      lo = mid;
    else
      hi = mid;
  }
  const int s = lo;
  int o = task - bwd_stage_start(p.tiles, E, s, nnF2, nnH2, per_w);
  BwdTask k;
  if (s < E) {
    const int first = __ldg(p.tiles + 1 + s);
    const int n_d2 = nnF2 * (__ldg(p.tiles + 2 + s) - first);
    if (o < n_d2) {
      k.kind = kDgrad2;
      k.t = decode<kDgrad2>(f.d2, nnF2 * first + o);
      return k;
    }
    o -= n_d2;
  }
  const int e = s - kBwdSkew;  // 0 <= e < E here
  const int first = __ldg(p.tiles + 1 + e);
  const int n_d1 = nnH2 * (__ldg(p.tiles + 2 + e) - first);
  if (o < n_d1) {
    k.kind = kDgrad1;
    k.t = decode<kDgrad1>(f.d1, nnH2 * first + o);
  } else if (o < n_d1 + n_w13) {
    k.kind = kWgrad13;
    k.t = decode<kWgrad13>(f.w13, e * n_w13 + (o - n_d1));
  } else {
    k.kind = kWgrad2;
    k.t = decode<kWgrad2>(f.w2, e * n_w2 + (o - n_d1 - n_w13));
  }
  return k;
}

__device__ __forceinline__ uint32_t bwd_idesc(int kind, int nw) {
  const bool mn = (kind == kWgrad13 || kind == kWgrad2);
  return nw == 256 ? (mn ? idesc_bf16_f32(BM, 256, true, true) : idesc_bf16_f32(BM, 256, false, false))
                   : (mn ? idesc_bf16_f32(BM, 128, true, true) : idesc_bf16_f32(BM, 128, false, false));
}

__global__ void __launch_bounds__(kThreads, 1) fused_backward_kernel(const __grid_constant__ FusedBwdMaps maps,
                                                                     const FusedBwdParams f) {
  constexpr int S = kBwdStages;
  constexpr int kStaging = kEpiWarps * kStageOutBytes;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + S * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kStaging);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* rfull = tempty + 2;
  uint64_t* rempty = rfull + kTaskRing;
  volatile int* ring = reinterpret_cast<volatile int*>(rempty + kTaskRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kTaskRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* ws = f.d2.ws;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    for (int i = 0; i < kTaskRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 1 + kEpiWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const GemmParams& P = f.d2;
  const int nnF2 = (P.F + BN - 1) / BN;
  const int nnH2 = (P.H + BN - 1) / BN;
  const int total = bwd_stage_start(P.tiles, P.E, P.E + kBwdSkew, nnF2, nnH2,
                                    (P.H / BM) * (P.F / 128) + (P.F / BM) * nnH2);

  if (warp == 0) {
    // ------------------------------------------------------------ producer + task fetch
    int s = 0, slot = 0;
    uint32_t ph = 0, rph = 0;
    uint32_t issued = 0, last_parity = 0;
    int next = (lane == 0) ? atomicAdd(f.cursor, 1) : 0;  // one task ahead
    while (true) {
      if (!mbar_wait(&rempty[slot], rph ^ 1u, ws, 160, abort_flag)) break;
      int task = 0;
      if (lane == 0) {
        task = next;
        if (task >= total || *abort_flag) task = kTaskEnd;
        if (task != kTaskEnd) next = atomicAdd(f.cursor, 1);
        ring[slot] = task;
      }
      task = __shfl_sync(0xffffffffu, task, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[slot]);
      if (++slot == kTaskRing) {
        slot = 0;
        rph ^= 1u;
      }
      if (task == kTaskEnd) break;
      const BwdTask k = bwd_decode(f, task);
      // Scoreboard: dG, dU of the rows this tile reads must be complete.
      bool ready = true;
      if (k.kind == kDgrad1) {
        ready = wait_counter(f.cnt_d2 + k.t.mt, nnF2 * kEpiWarps, ws, 161, abort_flag);
      } else if (k.kind == kWgrad13) {
        const int n_mt = __ldg(P.tiles + 2 + k.t.e) - __ldg(P.tiles + 1 + k.t.e);
        ready = wait_counter(f.cnt_e + k.t.e, n_mt * nnF2 * kEpiWarps, ws, 162, abort_flag);
      }
      if (!ready) continue;  // abort: the consumers see the flag and stop
      if (k.kind == kDgrad1 || k.kind == kWgrad13) fence_proxy_async_global();
      for (int kb = 0; kb < k.t.kblocks; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1u, ws, 163, abort_flag)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], kABytes + k.t.nw * 128);
          uint8_t* sA = smem + s * kStageBytes;
          switch (k.kind) {
            case kDgrad2: load_kblock<kDgrad2>(f.d2, maps.d2, k.t, kb, sA, sA + kABytes, &full[s]); break;
            case kDgrad1: load_kblock<kDgrad1>(f.d1, maps.d1, k.t, kb, sA, sA + kABytes, &full[s]); break;
            case kWgrad13: load_kblock<kWgrad13>(f.w13, maps.w13, k.t, kb, sA, sA + kABytes, &full[s]); break;
            default: load_kblock<kWgrad2>(f.w2, maps.w2, k.t, kb, sA, sA + kABytes, &full[s]); break;
          }
        }
        __syncwarp();
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    for (int i = 0; i < S; ++i)
      if ((issued >> i) & 1u) mbar_wait(&full[i], (last_parity >> i) & 1u, ws, 164, nullptr);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0, slot = 0, acc = 0;
    uint32_t ph = 0, rph = 0, acc_ph = 0;
    bool ok = true;
    while (ok) {
      if (!mbar_wait(&rfull[slot], rph, ws, 165, abort_flag)) break;
      const int task = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[slot]);
      if (++slot == kTaskRing) {
        slot = 0;
        rph ^= 1u;
      }
      if (task == kTaskEnd) break;
      const BwdTask k = bwd_decode(f, task);
      if (k.t.kblocks == 0) continue;  // empty expert (wgrad): the epilogue writes zeros
      const bool mn = (k.kind == kWgrad13 || k.kind == kWgrad2);
      if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, ws, 166, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kAccStride;
      const uint32_t idesc = bwd_idesc(k.kind, k.t.nw);
      const uint32_t a_step = mn ? 2048u : 32u;
      const uint32_t a_lbo = mn ? kPanelBytes : 16u;
      const uint32_t b_step = mn ? 2048u : 32u;
      const uint32_t b_lbo = mn ? kPanelBytes : 16u;
      for (int kb = 0; kb < k.t.kblocks; ++kb) {
        if (!mbar_wait(&full[s], ph, ws, 167, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* sA = smem + s * kStageBytes;
        int nkk = BK / 16;
        if (mn) {
          // Last k-block of the expert: only the K steps holding valid rows.
          const int valid = k.t.nrows - kb * BK;
          if (valid < BK) nkk = clear_k_tail(sA, sA + kABytes, valid, k.t.nw, lane);
          __syncwarp();
        }
        if (elect_one()) {
          const uint32_t a0 = smem_u32(sA), b0 = a0 + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk < nkk) {
              const uint64_t ad = smem_desc_sw128(a0 + kk * a_step, a_lbo, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + kk * b_step, b_lbo, 1024);
              tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
            }
          }
          tc_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    const int row = q * 32 + lane;
    OutStager st;
    st.buf = staging + ew * kStageOutBytes;
    int slot = 0, acc = 0;
    uint32_t rph = 0, acc_ph = 0;
    while (true) {
      if (!mbar_wait(&rfull[slot], rph, ws, 168, abort_flag)) break;
      const int task = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[slot]);
      if (++slot == kTaskRing) {
        slot = 0;
        rph ^= 1u;
      }
      if (task == kTaskEnd) break;
      const BwdTask k = bwd_decode(f, task);
      if (k.t.kblocks == 0) {  // empty expert: zero weight gradients
        const bool w13 = (k.kind == kWgrad13);
        const GemmParams& gp = w13 ? f.w13 : f.w2;
        const int NCall = w13 ? 128 : k.t.nw;
        const int c_lo = half * (NCall / 2), c_hi = c_lo + NCall / 2;
        float* d0 = w13 ? gp.f0 + (static_cast<size_t>(k.t.e) * gp.H + k.t.m0 + row) * gp.F + k.t.n0
                        : gp.f0 + (static_cast<size_t>(k.t.e) * gp.F + k.t.m0 + row) * gp.H + k.t.n0;
        for (int c = c_lo; c < c_hi; c += 32) store_zero_f32(d0 + c);
        if (w13) {
          float* d1 = gp.f1 + (static_cast<size_t>(k.t.e) * gp.H + k.t.m0 + row) * gp.F + k.t.n0;
          for (int c = c_lo; c < c_hi; c += 32) store_zero_f32(d1 + c);
        }
        continue;
      }
      if (!mbar_wait(&tfull[acc], acc_ph, ws, 169, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      switch (k.kind) {
        case kDgrad2: epilogue<kDgrad2>(f.d2, maps.d2, k.t, tacc, q, half, lane, st); break;
        case kDgrad1: epilogue<kDgrad1>(f.d1, maps.d1, k.t, tacc, q, half, lane, st); break;
        case kWgrad13: epilogue<kWgrad13>(f.w13, maps.w13, k.t, tacc, q, half, lane, st); break;
        default: epilogue<kWgrad2>(f.w2, maps.w2, k.t, tacc, q, half, lane, st); break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
      if (k.kind == kDgrad2) {
        signal_counter(f.cnt_d2 + k.t.mt, lane);
        if (lane == 0) atomicAdd(f.cnt_e + k.t.e, 1);  // ordered by the fence in signal_counter
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = []() -> EncodeFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeFn>(f);
  }();
  return fn;
}

// 2-D bf16 tensor [outer, inner] (inner contiguous), box {box_inner, box_outer}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a row-major bf16 matrix [outer, inner] as {64 columns, outer rows,
// inner / 64 panels} (strides: the row pitch, then 128 bytes per panel), box
// {64, box_rows, 2}: two neighbouring 64-column panels per instruction, each
// landing as its own 128-byte-swizzled block of box_rows rows.
bool make_map_panels2(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  EncodeFn enc = encoder();
  if (!enc || inner % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, outer, inner / 64};
  const cuuint64_t strides[2] = {inner * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_mode(const GemmLaunch& L, const Maps& maps, const GemmParams& p, cudaStream_t s,
                        LaunchHook& hook) {
  constexpr int kSmem = ModeTraits<MODE>::kSmemBytes;
  auto kern = grouped_gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  hook.before(s);
  kern<<<L.grid, kThreads, kSmem, s>>>(maps, p);
  hook.after(s);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_pair_mode(const GemmLaunch& L, const Maps& maps, const GemmParams& p, cudaStream_t s,
                             LaunchHook& hook) {
  const int kSmem = PairTraits<MODE>::kSmemBytes + (ModeTraits<MODE>::wgrad ? 0 : static_cast<int>(pair_table_bytes(L.E)));
  auto kern = pair_gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // At most as many clusters as can be resident at once (a persistent grid).
  static int max_pairs = -1, max_pairs_smem = -1;
  if (max_pairs < 0 || max_pairs_smem != kSmem) {
    max_pairs_smem = kSmem;
    cfg.gridDim = dim3(2, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    max_pairs = n;
  }
  int pairs = L.grid / 2;
  if (pairs < 1) pairs = 1;
  if (max_pairs > 0 && pairs > max_pairs) pairs = max_pairs;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  hook.before(s);
  e = cudaLaunchKernelEx(&cfg, kern, maps, p);
  hook.after(s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Tensor maps of the pair kernels: as the single-CTA ones, except that K-major
// B boxes are half a tile high (128 rows, or 64 for a 128-wide tail tile).
cudaError_t launch_gemm_pair(GemmMode mode, const GemmLaunch& L, Maps& m, const GemmParams& p, cudaStream_t s,
                             LaunchHook& hook) {
  const uint64_t H = L.H, F = L.F, E = L.E;
  bool ok = true;
  if (mode == kDgrad2)
    ok = make_map(&m.b0, L.W2, H, E * F, 64, 128) && make_map(&m.b2, L.W2, H, E * F, 64, 64);
  else if (mode == kDgrad1)
    ok = make_map(&m.b0, L.W1, F, E * H, 64, 128) && make_map(&m.b1, L.W3, F, E * H, 64, 128) &&
         make_map(&m.b2, L.W1, F, E * H, 64, 64) && make_map(&m.b3, L.W3, F, E * H, 64, 64);
  if (!ok) return cudaErrorInvalidValue;
  // Expert tails of at most 128 rows as M = 128 pair tiles (not with the
  // gather-fused A, which loads 128 rows, nor with the combine in GEMM2's
  // epilogue, which counts column halves of whole rows).
  GemmParams ph = p;
  if ((mode == kFwd1 && !L.gather) || (mode == kFwd2 && L.cmb.cnt == nullptr) || mode == kDgrad1 || mode == kDgrad2) {
    const void* a = mode == kFwd1 ? L.Xp : mode == kFwd2 ? L.h : mode == kDgrad2 ? L.dY : L.dGU;
    const uint64_t K = mode == kFwd1 || mode == kDgrad2 ? H : mode == kFwd2 ? F : 2 * F;
    if (!make_map(&m.a64, a, K, static_cast<uint64_t>(L.R), 64, 64)) return cudaErrorInvalidValue;
    ph.halfm_ok = 1;
  }
  // MN-major operands: two 64-column panels per TMA instruction where the 3-D
  // views encode (otherwise one instruction per panel, the same bytes).
  const uint64_t R = static_cast<uint64_t>(L.R);
  bool p2 = false;
  switch (mode) {
    case kFwd1:
      p2 = make_map_panels2(&m.b0_p2, L.W1, F, E * H, 64) && make_map_panels2(&m.b1_p2, L.W3, F, E * H, 64);
      break;
    case kFwd2: p2 = make_map_panels2(&m.b0_p2, L.W2, H, E * F, 64); break;
    case kWgrad13:
      p2 = make_map_panels2(&m.a_p2, L.Xp, H, R, 64) && make_map_panels2(&m.b0_p2, L.dGU, 2 * F, R, 64);
      break;
    case kWgrad2: p2 = make_map_panels2(&m.a_p2, L.h, F, R, 64) && make_map_panels2(&m.b0_p2, L.dY, H, R, 64); break;
    default: break;
  }
  ph.panels2 = p2 ? 1 : 0;
  switch (mode) {
    case kFwd1: return launch_pair_mode<kFwd1>(L, m, ph, s, hook);
    case kFwd2: return launch_pair_mode<kFwd2>(L, m, ph, s, hook);
    case kDgrad2: return launch_pair_mode<kDgrad2>(L, m, ph, s, hook);
    case kDgrad1: return launch_pair_mode<kDgrad1>(L, m, ph, s, hook);
    case kWgrad13: return launch_pair_mode<kWgrad13>(L, m, ph, s, hook);
    case kWgrad2: return launch_pair_mode<kWgrad2>(L, m, ph, s, hook);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool tensor_map_encoder_ready() { return encoder() != nullptr; }

#ifdef MOE_TIMELINE
// Diagnosis builds only (-DMOE_TIMELINE; no declaration in the public header):
// points the pair kernels' timeline at a device buffer of cap * 5 stamps per
// CTA, for the GEMM mode `mode` (0 fwd1 ... 5 wgrad2); buf = null switches it off.
extern "C" MOE_API int moe_debug_timeline(void* buf, int cap, int mode) {
  unsigned long long* b = static_cast<unsigned long long*>(buf);
  if (cudaMemcpyToSymbol(g_tl_buf, &b, sizeof(b)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_tl_cap, &cap, sizeof(cap)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_tl_mode, &mode, sizeof(mode)) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  return MOE_OK;
}
#endif

cudaError_t launch_fused_backward(const GemmLaunch& L, int32_t* cursor, int32_t* cnt_d2, int32_t* cnt_e,
                                  cudaStream_t s, LaunchHook& hook) {
  const uint64_t R = L.R, H = L.H, F = L.F, E = L.E;
  FusedBwdMaps m;
  memset(&m, 0, sizeof(m));
  bool ok = make_map(&m.d2.a, L.dY, H, R, 64, BM) && make_map(&m.d2.b0, L.W2, H, E * F, 64, BN) &&
            make_map(&m.d2.b2, L.W2, H, E * F, 64, 128);
  ok = ok && make_map(&m.d1.a, L.dGU, 2 * F, R, 64, BM) && make_map(&m.d1.b0, L.W1, F, E * H, 64, BN) &&
       make_map(&m.d1.b1, L.W3, F, E * H, 64, BN) && make_map(&m.d1.b2, L.W1, F, E * H, 64, 128) &&
       make_map(&m.d1.b3, L.W3, F, E * H, 64, 128);
  ok = ok && make_map(&m.w13.a, L.Xp, H, R, 64, 64) && make_map(&m.w13.b0, L.dGU, 2 * F, R, 64, 64);
  ok = ok && make_map(&m.w2.a, L.h, F, R, 64, 64) && make_map(&m.w2.b0, L.dY, H, R, 64, 64);
  if (!ok) return cudaErrorInvalidValue;
  GemmParams p{};
  p.H = L.H;
  p.F = L.F;
  p.E = L.E;
  p.R = L.R;
  p.tiles = L.tiles;
  p.pairs = L.pairs;
  p.offsets = L.offsets;
  p.counts = L.counts;
  p.ws = L.ws;
  FusedBwdParams f{};
  f.d2 = p;
  f.d2.out0 = static_cast<__nv_bfloat16*>(L.out_dGU);
  f.d2.aux = static_cast<const __nv_bfloat16*>(L.GU);
  f.d1 = p;
  f.d1.out0 = static_cast<__nv_bfloat16*>(L.out_dXp);
  f.w13 = p;
  f.w13.f0 = L.dW1;
  f.w13.f1 = L.dW3;
  f.w2 = p;
  f.w2.f0 = L.dW2;
  f.cursor = cursor;
  f.cnt_d2 = cnt_d2;
  f.cnt_e = cnt_e;
  constexpr int kSmem = kBwdStages * kStageBytes + kEpiWarps * kStageOutBytes + 1024 + 512;
  cudaError_t e = cudaFuncSetAttribute(fused_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  hook.before(s);
  fused_backward_kernel<<<L.grid, kThreads, kSmem, s>>>(m, f);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_fused_forward(const GemmLaunch& L, const void* x, const int32_t* row_src, int32_t* cursor,
                                 int32_t* cnt_gather, int32_t* cnt_g1, cudaStream_t s, LaunchHook& hook) {
  const uint64_t R = L.R, H = L.H, F = L.F, E = L.E;
  FusedFwdMaps m;
  memset(&m, 0, sizeof(m));
  if (!(make_map(&m.g1.a, L.Xp, H, R, 64, BM) && make_map(&m.g1.b0, L.W1, F, E * H, 64, 64) &&
        make_map(&m.g1.b1, L.W3, F, E * H, 64, 64) && make_map(&m.g2.a, L.out_h, F, R, 64, BM) &&
        make_map(&m.g2.b0, L.W2, H, E * F, 64, 64)))
    return cudaErrorInvalidValue;
  FusedFwdParams f{};
  GemmParams p{};
  p.H = L.H;
  p.F = L.F;
  p.E = L.E;
  p.R = L.R;
  p.tiles = L.tiles;
  p.pairs = L.pairs;
  p.offsets = L.offsets;
  p.counts = L.counts;
  p.ws = L.ws;
  f.p1 = p;
  f.p1.out0 = static_cast<__nv_bfloat16*>(L.out_h);
  f.p1.out1 = static_cast<__nv_bfloat16*>(L.out_GU);
  f.p2 = p;
  f.p2.out0 = static_cast<__nv_bfloat16*>(L.out_Y);
  f.x = static_cast<const uint4*>(x);
  f.Xp = static_cast<uint4*>(const_cast<void*>(L.Xp));
  f.row_src = row_src;
  f.T = L.T;
  f.cursor = cursor;
  f.cnt_gather = cnt_gather;
  f.cnt_g1 = cnt_g1;
  f.drop_task = L.drop_task;
  constexpr int kSmem = 4 * kStageBytes + 1024 + 512;
  cudaError_t e = cudaFuncSetAttribute(fused_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  hook.before(s);
  fused_forward_kernel<<<L.grid, kThreads, kSmem, s>>>(m, f);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_fused_forward_pair(const GemmLaunch& L, const void* x, const int32_t* row_src, int32_t* cursor,
                                      int32_t* cnt_gather, int32_t* cnt_g1, cudaStream_t s, LaunchHook& hook) {
  const uint64_t R = L.R, H = L.H, F = L.F, E = L.E;
  FusedFwdMaps m;
  memset(&m, 0, sizeof(m));
  if (!(make_map(&m.g1.a, L.Xp, H, R, 64, BM) && make_map(&m.g1.b0, L.W1, F, E * H, 64, 64) &&
        make_map(&m.g1.b1, L.W3, F, E * H, 64, 64) && make_map(&m.g2.a, L.out_h, F, R, 64, BM) &&
        make_map(&m.g2.b0, L.W2, H, E * F, 64, 64)))
    return cudaErrorInvalidValue;
  FusedFwdParams f{};
  GemmParams p{};
  p.H = L.H;
  p.F = L.F;
  p.E = L.E;
  p.R = L.R;
  p.tiles = L.tiles;
  p.pairs = L.pairs;
  p.offsets = L.offsets;
  p.counts = L.counts;
  p.ws = L.ws;
  f.p1 = p;
  f.p1.out0 = static_cast<__nv_bfloat16*>(L.out_h);
  f.p1.out1 = static_cast<__nv_bfloat16*>(L.out_GU);
  f.p2 = p;
  f.p2.out0 = static_cast<__nv_bfloat16*>(L.out_Y);
  f.x = static_cast<const uint4*>(x);
  f.Xp = static_cast<uint4*>(const_cast<void*>(L.Xp));
  f.row_src = row_src;
  f.T = L.T;
  f.cursor = cursor;
  f.cnt_gather = cnt_gather;
  f.cnt_g1 = cnt_g1;
  f.drop_task = L.drop_task;
  const int kSmem = kFusedPairStages * kPairStageBytes + 1024 + 512 + static_cast<int>(pair_table_bytes(L.E));
  auto kern = fused_forward_pair_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_pairs = -1, max_pairs_smem = -1;
  if (max_pairs < 0 || max_pairs_smem != kSmem) {
    max_pairs_smem = kSmem;
    cfg.gridDim = dim3(2, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    max_pairs = n;
  }
  int pairs = L.grid / 2;
  if (pairs < 1) pairs = 1;
  if (max_pairs > 0 && pairs > max_pairs) pairs = max_pairs;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  hook.before(s);
  e = cudaLaunchKernelEx(&cfg, kern, m, f);
  hook.after(s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm(GemmMode mode, const GemmLaunch& L, cudaStream_t s, LaunchHook& hook) {
  const uint64_t R = L.R, H = L.H, F = L.F, E = L.E;
  Maps m;
  memset(&m, 0, sizeof(m));
  GemmParams p{};
  p.H = L.H;
  p.F = L.F;
  p.E = L.E;
  p.R = L.R;
  p.tiles = L.tiles;
  p.pairs = L.pairs;
  p.offsets = L.offsets;
  p.counts = L.counts;
  p.ws = L.ws;
  bool ok = true;
  switch (mode) {
    case kFwd1:
      ok = make_map(&m.a, L.Xp, H, R, 64, BM) && make_map(&m.b0, L.W1, F, E * H, 64, 64) &&
           make_map(&m.b1, L.W3, F, E * H, 64, 64);
      p.out0 = static_cast<__nv_bfloat16*>(L.out_h);
      p.out1 = static_cast<__nv_bfloat16*>(L.out_GU);
      if (L.gather) {  // pair tiles only: the A rows come from x by cp.async
        if (!L.pair) return cudaErrorInvalidValue;
        p.x = static_cast<const __nv_bfloat16*>(L.x);
        p.gather = 1;
        p.row_src = L.row_src;
      }
      break;
    case kFwd2:
      ok = make_map(&m.a, L.h, F, R, 64, BM) && make_map(&m.b0, L.W2, H, E * F, 64, 64);
      p.out0 = static_cast<__nv_bfloat16*>(L.out_Y);
      p.cmb = CombineParams{L.cmb.cnt, L.cmb.row_src, L.cmb.dest, L.cmb.w,
                            static_cast<__nv_bfloat16*>(L.cmb.out), L.cmb.k};
      break;
    case kDgrad2:
      ok = make_map(&m.a, L.dY, H, R, 64, BM) && make_map(&m.b0, L.W2, H, E * F, 64, BN) &&
           make_map(&m.b2, L.W2, H, E * F, 64, 128);
      p.out0 = static_cast<__nv_bfloat16*>(L.out_dGU);
      p.aux = static_cast<const __nv_bfloat16*>(L.GU);
      ok = ok && make_map(&m.gu, L.GU, 2 * F, R, 16, 32, CU_TENSOR_MAP_SWIZZLE_32B);  // epilogue G/U boxes
      break;
    case kDgrad1:
      ok = make_map(&m.a, L.dGU, 2 * F, R, 64, BM) && make_map(&m.b0, L.W1, F, E * H, 64, BN) &&
           make_map(&m.b1, L.W3, F, E * H, 64, BN) && make_map(&m.b2, L.W1, F, E * H, 64, 128) &&
           make_map(&m.b3, L.W3, F, E * H, 64, 128);
      p.out0 = static_cast<__nv_bfloat16*>(L.out_dXp);
      break;
    case kWgrad13:
      ok = make_map(&m.a, L.Xp, H, R, 64, 64) && make_map(&m.b0, L.dGU, 2 * F, R, 64, 64);
      p.f0 = L.dW1;
      p.f1 = L.dW3;
      break;
    case kWgrad2:
      ok = make_map(&m.a, L.h, F, R, 64, 64) && make_map(&m.b0, L.dY, H, R, 64, 64);
      p.f0 = L.dW2;
      break;
    case kRfwd:
      ok = make_map(&m.a, L.x, H, static_cast<uint64_t>(L.T), 64, BM) && make_map(&m.b0, L.Wr, E, H, 64, 64);
      p.f0 = L.logits;
      break;
    case kRwgrad:
      ok = make_map(&m.a, L.x, H, static_cast<uint64_t>(L.T), 64, 64) &&
           make_map(&m.b0, L.dl, E, static_cast<uint64_t>(L.T), 64, 64);
      p.f0 = L.dwr_part;
      break;
  }
  p.T = L.T;
  p.splits = L.splits;
  p.ks = L.ks;
  if (mode == kWgrad13 || mode == kWgrad2) {
    p.sb = L.sb;
    p.sb_rows = L.sb_rows;
  }
  if (mode != kFwd2) p.cmb = CombineParams{};
  if (!ok) return cudaErrorInvalidValue;
  if (L.pair && mode != kRfwd && mode != kRwgrad) return launch_gemm_pair(mode, L, m, p, s, hook);
  switch (mode) {
    case kRfwd: return launch_mode<kRfwd>(L, m, p, s, hook);
    case kRwgrad: return launch_mode<kRwgrad>(L, m, p, s, hook);
    case kFwd1: return launch_mode<kFwd1>(L, m, p, s, hook);
    case kFwd2: return launch_mode<kFwd2>(L, m, p, s, hook);
    case kDgrad2: return launch_mode<kDgrad2>(L, m, p, s, hook);
    case kDgrad1: return launch_mode<kDgrad1>(L, m, p, s, hook);
    case kWgrad13: return launch_mode<kWgrad13>(L, m, p, s, hook);
    case kWgrad2: return launch_mode<kWgrad2>(L, m, p, s, hook);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
