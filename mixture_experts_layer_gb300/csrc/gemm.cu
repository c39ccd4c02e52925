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
// Kernel structure (one CTA per SM, 192 threads):
//   warp 0     TMA producer: fills a ring of shared-memory stages
//   warp 1     allocates tensor memory, issues tcgen05.mma (one elected lane)
//   warps 2-5  epilogue: tcgen05.ld of the fp32 accumulator, fused
//              elementwise work (SwiGLU forward or backward), global stores.
// The accumulator is double-buffered in tensor memory (2 x 256 columns), so the
// epilogue of one tile overlaps the main loop of the next.
//
// Operand layouts in shared memory are the 128-byte-swizzled canonical forms:
//   K-major  (rows of 64 K-elements, 128 B each, 8-row atoms of 1 KB):
//            SBO = 1024 B between 8-row groups; +32 B per K step of 16.
//   MN-major (panels of 64 MN-elements x 64 K-rows, 8 KB each):
//            LBO = 8192 B between panels, SBO = 1024 B between 8-row K groups;
//            +2048 B per K step of 16.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr int kEpiWarp0 = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;  // TMEM columns per accumulator buffer
constexpr int kPanelBytes = 64 * 128;  // one MN-major panel: 64 K-rows x 128 B

template <int MODE>
struct ModeTraits;
template <>
struct ModeTraits<kFwd1> {
  static constexpr bool a_mn = false, b_mn = true, wgrad = false;
};
template <>
struct ModeTraits<kFwd2> {
  static constexpr bool a_mn = false, b_mn = true, wgrad = false;
};
template <>
struct ModeTraits<kDgrad2> {
  static constexpr bool a_mn = false, b_mn = false, wgrad = false;
};
template <>
struct ModeTraits<kDgrad1> {
  static constexpr bool a_mn = false, b_mn = false, wgrad = false;
};
template <>
struct ModeTraits<kWgrad13> {
  static constexpr bool a_mn = true, b_mn = true, wgrad = true;
};
template <>
struct ModeTraits<kWgrad2> {
  static constexpr bool a_mn = true, b_mn = true, wgrad = true;
};

template <int BN>
struct Cfg {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
};

struct GemmParams {
  int H, F, E, R;
  int bn;
  const int32_t* tiles;
  const int32_t* offsets;
  const int32_t* counts;
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  const __nv_bfloat16* aux;
  float* f0;
  float* f1;
  WsHeader* ws;
};

struct Tile {
  int e;      // expert
  int row0;   // first grouped row of the tile (forward/dgrad) or of the expert (wgrad)
  int nrows;  // valid rows of the tile (forward/dgrad) or rows of the expert (wgrad)
  int m0;     // wgrad: first output row inside the expert's weight
  int n0;     // first output column
  int kblocks;
};

template <int MODE, int BN>
__device__ __forceinline__ int n_tiles(const GemmParams& p) {
  if (MODE == kWgrad13) return p.E * (p.H / BM) * (p.F / 128);
  if (MODE == kWgrad2) return p.E * (p.F / BM) * (p.H / BN);
  const int nn = (MODE == kFwd1) ? p.F / 128 : (MODE == kFwd2 || MODE == kDgrad1) ? p.H / BN : p.F / BN;
  return __ldg(p.tiles) * nn;
}

template <int MODE, int BN>
__device__ __forceinline__ Tile decode(const GemmParams& p, int tile) {
  Tile t;
  if (MODE == kWgrad13 || MODE == kWgrad2) {
    const int MT = (MODE == kWgrad13) ? p.H / BM : p.F / BM;
    const int NT = (MODE == kWgrad13) ? p.F / 128 : p.H / BN;
    t.e = tile / (MT * NT);
    const int rem = tile - t.e * MT * NT;
    const int nt = rem / MT;
    t.m0 = (rem - nt * MT) * BM;
    t.n0 = nt * ((MODE == kWgrad13) ? 128 : BN);
    t.row0 = __ldg(p.offsets + t.e);
    t.nrows = __ldg(p.counts + t.e);
    t.kblocks = (t.nrows + BK - 1) / BK;
    return t;
  }
  const int nn = (MODE == kFwd1) ? p.F / 128 : (MODE == kFwd2 || MODE == kDgrad1) ? p.H / BN : p.F / BN;
  const int entries = tiles_entry_base(p.E);
  const int4* ent = reinterpret_cast<const int4*>(p.tiles + entries);
  // Tiles of one expert are ordered (n tile, m tile) with m fastest, so the CTAs
  // working side by side share the same weight columns (L2 reuse).
  const int q = tile / nn;
  const int e = __ldg(&ent[q].x);
  const int first = __ldg(p.tiles + 1 + e);
  const int cnt = __ldg(p.tiles + 2 + e) - first;
  const int local = tile - nn * first;
  const int nt = local / cnt;
  const int mt = first + (local - nt * cnt);
  const int4 en = ent[mt];
  t.e = e;
  t.row0 = en.y;
  t.nrows = en.z;
  t.m0 = 0;
  t.n0 = nt * ((MODE == kFwd1) ? 128 : BN);
  const int K = (MODE == kFwd1 || MODE == kDgrad2) ? p.H : (MODE == kFwd2) ? p.F : 2 * p.F;
  t.kblocks = K / BK;
  return t;
}

// Issues the TMA loads of one k-block into stage buffers sA / sB.
template <int MODE, int BN>
__device__ __forceinline__ void load_kblock(const GemmParams& p, const Tile& t, int kb, uint8_t* sA, uint8_t* sB,
                                            uint64_t* bar, const CUtensorMap* mA, const CUtensorMap* mB0,
                                            const CUtensorMap* mB1) {
  const int k0 = kb * BK;
  if (MODE == kFwd1) {
    tma_load_2d(sA, mA, bar, k0, t.row0);
    const int y = t.e * p.H + k0;
    tma_load_2d(sB + 0 * kPanelBytes, mB0, bar, t.n0, y);
    tma_load_2d(sB + 1 * kPanelBytes, mB0, bar, t.n0 + 64, y);
    tma_load_2d(sB + 2 * kPanelBytes, mB1, bar, t.n0, y);
    tma_load_2d(sB + 3 * kPanelBytes, mB1, bar, t.n0 + 64, y);
  } else if (MODE == kFwd2) {
    tma_load_2d(sA, mA, bar, k0, t.row0);
    const int y = t.e * p.F + k0;
#pragma unroll
    for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * kPanelBytes, mB0, bar, t.n0 + 64 * q, y);
  } else if (MODE == kDgrad2) {
    tma_load_2d(sA, mA, bar, k0, t.row0);
    tma_load_2d(sB, mB0, bar, k0, t.e * p.F + t.n0);
  } else if (MODE == kDgrad1) {
    tma_load_2d(sA, mA, bar, k0, t.row0);
    if (k0 < p.F)
      tma_load_2d(sB, mB0, bar, k0, t.e * p.H + t.n0);
    else
      tma_load_2d(sB, mB1, bar, k0 - p.F, t.e * p.H + t.n0);
  } else if (MODE == kWgrad13) {
    const int y = t.row0 + k0;
    tma_load_2d(sA, mA, bar, t.m0, y);
    tma_load_2d(sA + kPanelBytes, mA, bar, t.m0 + 64, y);
    tma_load_2d(sB + 0 * kPanelBytes, mB0, bar, t.n0, y);
    tma_load_2d(sB + 1 * kPanelBytes, mB0, bar, t.n0 + 64, y);
    tma_load_2d(sB + 2 * kPanelBytes, mB0, bar, p.F + t.n0, y);
    tma_load_2d(sB + 3 * kPanelBytes, mB0, bar, p.F + t.n0 + 64, y);
  } else {  // kWgrad2
    const int y = t.row0 + k0;
    tma_load_2d(sA, mA, bar, t.m0, y);
    tma_load_2d(sA + kPanelBytes, mA, bar, t.m0 + 64, y);
#pragma unroll
    for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * kPanelBytes, mB0, bar, t.n0 + 64 * q, y);
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

// Stores 32 fp32 accumulator values of one row as bf16 (64 bytes).
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    st_v4(dst + i, pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]), pack_bf16x2(v[i + 4], v[i + 5]),
          pack_bf16x2(v[i + 6], v[i + 7]));
}

__device__ __forceinline__ void store_row_f32(float* dst, const uint32_t* r) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) st_v4(dst + i, r[i], r[i + 1], r[i + 2], r[i + 3]);
}

__device__ __forceinline__ void store_zero_f32(float* dst) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) st_v4(dst + i, 0u, 0u, 0u, 0u);
}

template <int MODE, int BN>
__device__ __forceinline__ void epilogue(const GemmParams& p, const Tile& t, uint32_t tacc, int row) {
  constexpr int NCOLS = (MODE == kFwd1 || MODE == kWgrad13) ? 128 : BN;
  if (MODE == kWgrad13 || MODE == kWgrad2) {
    float* d0 = (MODE == kWgrad13) ? p.f0 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0
                                   : p.f0 + (static_cast<size_t>(t.e) * p.F + t.m0 + row) * p.H + t.n0;
    float* d1 = (MODE == kWgrad13) ? p.f1 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0 : nullptr;
#pragma unroll 1
    for (int c = 0; c < NCOLS; c += 32) {
      uint32_t r[32];
      tc_ld_32x32b_x32(tacc + c, r);
      tc_wait_ld();
      store_row_f32(d0 + c, r);
      if (MODE == kWgrad13) {
        tc_ld_32x32b_x32(tacc + 128 + c, r);
        tc_wait_ld();
        store_row_f32(d1 + c, r);
      }
    }
    return;
  }
  const bool valid = row < t.nrows;
  const size_t grow = static_cast<size_t>(t.row0) + row;
#pragma unroll 1
  for (int c = 0; c < NCOLS; c += 32) {
    if (MODE == kFwd1) {
      uint32_t g[32], u[32];
      tc_ld_32x32b_x32(tacc + c, g);
      tc_ld_32x32b_x32(tacc + 128 + c, u);
      tc_wait_ld();
      if (valid) {
        float hv[32], gv[32], uv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a = __uint_as_float(g[i]);
          const float b = __uint_as_float(u[i]);
          hv[i] = a / (1.0f + expf(-a)) * b;
          gv[i] = a;
          uv[i] = b;
        }
        store_row_bf16(p.out0 + grow * p.F + t.n0 + c, hv);
        store_row_bf16(p.out1 + grow * (2 * p.F) + t.n0 + c, gv);
        store_row_bf16(p.out1 + grow * (2 * p.F) + p.F + t.n0 + c, uv);
      }
    } else if (MODE == kDgrad2) {
      uint32_t d[32];
      tc_ld_32x32b_x32(tacc + c, d);
      tc_wait_ld();
      if (valid) {
        const __nv_bfloat16* gsrc = p.aux + grow * (2 * p.F) + t.n0 + c;
        const __nv_bfloat16* usrc = gsrc + p.F;
        float dg[32], du[32];
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          const uint4 gq = ld_v4(gsrc + i), uq = ld_v4(usrc + i);
          const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w}, uw[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int hbit = 0; hbit < 2; ++hbit) {
              const int ii = i + 2 * q + hbit;
              const float G = hbit ? bf16hi(gw[q]) : bf16lo(gw[q]);
              const float U = hbit ? bf16hi(uw[q]) : bf16lo(uw[q]);
              const float dh = __uint_as_float(d[ii]);
              const float s = 1.0f / (1.0f + expf(-G));
              dg[ii] = dh * U * s * (1.0f + G * (1.0f - s));
              du[ii] = dh * G * s;
            }
          }
        }
        store_row_bf16(p.out0 + grow * (2 * p.F) + t.n0 + c, dg);
        store_row_bf16(p.out0 + grow * (2 * p.F) + p.F + t.n0 + c, du);
      }
    } else {  // kFwd2 (Y) or kDgrad1 (dXp): plain bf16 store, row stride H
      uint32_t d[32];
      tc_ld_32x32b_x32(tacc + c, d);
      tc_wait_ld();
      if (valid) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(d[i]);
        store_row_bf16(p.out0 + grow * p.H + t.n0 + c, v);
      }
    }
  }
}

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                        const __grid_constant__ CUtensorMap mB1, const GemmParams p) {
  using C = Cfg<BN>;
  using TR = ModeTraits<MODE>;
  constexpr int S = C::kStages;
  constexpr int NMMA = (MODE == kFwd1 || MODE == kWgrad13) ? 256 : BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(BM, NMMA, TR::a_mn, TR::b_mn);
  constexpr uint32_t kAStep = TR::a_mn ? 2048u : 32u;
  constexpr uint32_t kBStep = TR::b_mn ? 2048u : 32u;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB0);
    tma_prefetch_desc(&mB1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = n_tiles<MODE, BN>(p);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    uint32_t issued = 0;        // bit i: stage i was ever filled
    uint32_t last_parity = 0;   // bit i: parity of stage i's last fill
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const Tile t = decode<MODE, BN>(p, tile);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1u, p.ws, 100 + MODE, abort_flag)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          uint8_t* sA = smem + s * C::kStageBytes;
          load_kblock<MODE, BN>(p, t, kb, sA, sA + C::kABytes, &full[s], &mA, &mB0, &mB1);
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
      const Tile t = decode<MODE, BN>(p, tile);
      if (t.kblocks == 0) continue;  // empty expert (wgrad): the epilogue writes zeros
      if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, p.ws, 120 + MODE, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kAccStride;
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait(&full[s], ph, p.ws, 130 + MODE, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* sA = smem + s * C::kStageBytes;
        uint8_t* sB = sA + C::kABytes;
        if (TR::wgrad) {
          // The expert's last k-block may run past its rows: zero those K rows
          // of both operands so rows of the next expert add nothing.
          const int valid = t.nrows - kb * BK;
          if (valid < BK) {
            constexpr int kPanels = 2 + NMMA / 64;
            const int nchunks = (BK - valid) * 8 * kPanels;
            for (int i = lane; i < nchunks; i += 32) {
              const int panel = i / ((BK - valid) * 8);
              const int rem = i - panel * (BK - valid) * 8;
              const int rr = valid + (rem >> 3);
              uint8_t* base = (panel < 2) ? sA + panel * kPanelBytes : sB + (panel - 2) * kPanelBytes;
              *reinterpret_cast<uint4*>(base + rr * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (elect_one()) {
          const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a0 + kk * kAStep, TR::a_mn ? kPanelBytes : 16, 1024);
            const uint64_t bd = smem_desc_sw128(b0 + kk * kBStep, TR::b_mn ? kPanelBytes : 16, 1024);
            tc_mma_bf16(d_tmem, ad, bd, kIdesc, (kb | kk) != 0);
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
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = decode<MODE, BN>(p, tile);
      if (t.kblocks == 0) {
        if (TR::wgrad) {
          constexpr int NC = (MODE == kWgrad13) ? 128 : BN;
          float* d0 = (MODE == kWgrad13) ? p.f0 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0
                                         : p.f0 + (static_cast<size_t>(t.e) * p.F + t.m0 + row) * p.H + t.n0;
          for (int c = 0; c < NC; c += 32) store_zero_f32(d0 + c);
          if (MODE == kWgrad13) {
            float* d1 = p.f1 + (static_cast<size_t>(t.e) * p.H + t.m0 + row) * p.F + t.n0;
            for (int c = 0; c < NC; c += 32) store_zero_f32(d1 + c);
          }
        }
        continue;
      }
      if (!mbar_wait(&tfull[acc], acc_ph, p.ws, 140 + MODE, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      epilogue<MODE, BN>(p, t, tacc, row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
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
              uint32_t box_outer) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BN>
cudaError_t launch_mode(const GemmLaunch& L, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const GemmParams& p, cudaStream_t s, LaunchHook& hook) {
  using C = Cfg<BN>;
  auto kern = grouped_gemm_kernel<MODE, BN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  hook.before(s);
  kern<<<L.grid, kThreads, C::kSmemBytes, s>>>(a, b0, b1, p);
  hook.after(s);
  return cudaGetLastError();
}

}  // namespace

bool tensor_map_encoder_ready() { return encoder() != nullptr; }

cudaError_t launch_gemm(GemmMode mode, const GemmLaunch& L, cudaStream_t s, LaunchHook& hook) {
  const uint64_t R = L.R, H = L.H, F = L.F, E = L.E;
  const uint32_t bn = L.bn;
  CUtensorMap a, b0, b1;
  GemmParams p{};
  p.H = L.H;
  p.F = L.F;
  p.E = L.E;
  p.R = L.R;
  p.bn = L.bn;
  p.tiles = L.tiles;
  p.offsets = L.offsets;
  p.counts = L.counts;
  p.ws = L.ws;
  bool ok = true;
  switch (mode) {
    case kFwd1:
      ok = make_map(&a, L.Xp, H, R, 64, BM) && make_map(&b0, L.W1, F, E * H, 64, 64) &&
           make_map(&b1, L.W3, F, E * H, 64, 64);
      p.out0 = static_cast<__nv_bfloat16*>(L.out_h);
      p.out1 = static_cast<__nv_bfloat16*>(L.out_GU);
      break;
    case kFwd2:
      ok = make_map(&a, L.h, F, R, 64, BM) && make_map(&b0, L.W2, H, E * F, 64, 64);
      b1 = b0;
      p.out0 = static_cast<__nv_bfloat16*>(L.out_Y);
      break;
    case kDgrad2:
      ok = make_map(&a, L.dY, H, R, 64, BM) && make_map(&b0, L.W2, H, E * F, 64, bn);
      b1 = b0;
      p.out0 = static_cast<__nv_bfloat16*>(L.out_dGU);
      p.aux = static_cast<const __nv_bfloat16*>(L.GU);
      break;
    case kDgrad1:
      ok = make_map(&a, L.dGU, 2 * F, R, 64, BM) && make_map(&b0, L.W1, F, E * H, 64, bn) &&
           make_map(&b1, L.W3, F, E * H, 64, bn);
      p.out0 = static_cast<__nv_bfloat16*>(L.out_dXp);
      break;
    case kWgrad13:
      ok = make_map(&a, L.Xp, H, R, 64, 64) && make_map(&b0, L.dGU, 2 * F, R, 64, 64);
      b1 = b0;
      p.f0 = L.dW1;
      p.f1 = L.dW3;
      break;
    case kWgrad2:
      ok = make_map(&a, L.h, F, R, 64, 64) && make_map(&b0, L.dY, H, R, 64, 64);
      b1 = b0;
      p.f0 = L.dW2;
      break;
  }
  if (!ok) return cudaErrorInvalidValue;
  switch (mode) {
    case kFwd1:
      return launch_mode<kFwd1, 256>(L, a, b0, b1, p, s, hook);
    case kFwd2:
      return bn == 256 ? launch_mode<kFwd2, 256>(L, a, b0, b1, p, s, hook)
                       : launch_mode<kFwd2, 128>(L, a, b0, b1, p, s, hook);
    case kDgrad2:
      return bn == 256 ? launch_mode<kDgrad2, 256>(L, a, b0, b1, p, s, hook)
                       : launch_mode<kDgrad2, 128>(L, a, b0, b1, p, s, hook);
    case kDgrad1:
      return bn == 256 ? launch_mode<kDgrad1, 256>(L, a, b0, b1, p, s, hook)
                       : launch_mode<kDgrad1, 128>(L, a, b0, b1, p, s, hook);
    case kWgrad13:
      return launch_mode<kWgrad13, 256>(L, a, b0, b1, p, s, hook);
    case kWgrad2:
      return bn == 256 ? launch_mode<kWgrad2, 256>(L, a, b0, b1, p, s, hook)
                       : launch_mode<kWgrad2, 128>(L, a, b0, b1, p, s, hook);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
