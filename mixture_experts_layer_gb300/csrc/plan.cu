// Routing: router logits -> top-k experts and gate weights -> the stable
// token -> grouped-row table.
//
// The table follows section 3.1 (Deterministic Token Mapping, Algorithm 1) of
// "UniEP: Unified Expert-Parallel MoE MegaKernel for LLM Training": every
// source counts its tokens per expert, an exclusive prefix over the sources
// gives each source its base inside an expert's segment, and a source places
// its tokens at base + their stable index among its own tokens.  The sources
// here are 256-token chunks of one GPU instead of ranks, so no atomics decide
// any position and the order inside each expert is the original token order.
//
//   route_topk  one CTA per 64 tokens: top-k per token (four threads per
//               token with a min/max selection network where E % 4 == 0,
//               E <= 256 and k <= 8; a warp-wide argmax per pick otherwise),
//               renormalised weights, and its part of the chunk bitmap bm[e][w]
//               whose bit b says "token 32w+b of the chunk chose expert e";
//               per-chunk and per-super-chunk (32 chunks) counts by integer
//               atomics.
//   route_rank  one CTA per chunk: the rows of each expert before the chunk
//               (super-chunks before it, then chunks before it in its own
//               super-chunk) and the prefix over experts; stable index =
//               popcount of the chunk's bitmap below the token; dest, row_src,
//               row_slot; a share of the GEMM tile entries; CTA 0 writes the
//               counts, offsets and expert-level tile tables.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kTopkTokens = 64;    // tokens per top-k / rank CTA: two bitmap words per expert
constexpr int kTopkThreads = 256;  // 8 warps x 8 tokens

// A top-k CTA's count of expert e goes to its chunk's count and to its
// super-chunk's (integer atomics: the sums do not depend on their order).
// Counts are expert-major: ccount[e][chunk], then sc[e][chunk / kSuperChunks].
__device__ __forceinline__ void add_counts(int32_t* ccount, int T, int E, int e, int chunk, int c) {
  const int nchunks = (T + kChunk - 1) / kChunk;
  const int nsuper = (nchunks + kSuperChunks - 1) / kSuperChunks;
  atomicAdd(&ccount[static_cast<size_t>(e) * nchunks + chunk], c);
  atomicAdd(&ccount[static_cast<size_t>(E) * nchunks + static_cast<size_t>(e) * nsuper + chunk / kSuperChunks], c);
}

// NV = logits per lane (E <= 32 * NV); TPW = tokens whose logits a warp loads
// at once, so several rows' loads are in flight before the selection starts.
// One CTA covers 64 consecutive tokens: it owns two words of its chunk's bitmap
// per expert (written plainly) and adds its per-expert counts to the chunk's
// counts with integer atomics (the sum does not depend on their order).
template <int NV, int TPW>
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                  int k, int32_t* __restrict__ ids,
                                                                  float* __restrict__ wts, uint32_t* __restrict__ gbm,
                                                                  int32_t* __restrict__ ccount, WsHeader* ws) {
  extern __shared__ uint32_t sm[];
  uint32_t* bm = sm;            // [E][2] bitmap words of this CTA's 64 tokens
  int* cnt = reinterpret_cast<int*>(sm + 2 * E);  // [E]
  for (int i = threadIdx.x; i < 3 * E; i += blockDim.x) sm[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTopkTokens;
  for (int tb = warp * (kTopkTokens / 8); tb < (warp + 1) * (kTopkTokens / 8); tb += TPW) {
    float v[TPW][NV];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int t = t0 + tb + u;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        v[u][i] = (t < T && e < E) ? logits[static_cast<size_t>(t) * E + e] : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int tl = tb + u;
      const int t = t0 + tl;
      if (t >= T) break;
      uint32_t taken = 0;
      bool bad = false;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e >= E) {
          taken |= 1u << i;  // padding lanes are never chosen
        } else if (!isfinite(v[u][i])) {
          bad = true;
          v[u][i] = -INFINITY;
        }
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) report(ws, MOE_ERR_NONFINITE, 0, t);
      int my_id = 0;
      float my_v = 0.f;
      for (int j = 0; j < k; ++j) {
        // Largest untaken logit, ties to the lower expert id: a total order, so
        // every lane ends the butterfly with the same winner.
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int e = lane + 32 * i;
          if (!((taken >> i) & 1u) && (v[u][i] > bv || (v[u][i] == bv && e < bi))) {
            bv = v[u][i];
            bi = e;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
          my_id = bi;
          my_v = bv;
        }
      }
      // w_j = exp(l_j - l_max) / sum_{i<k} exp(l_i - l_max); the sum runs in slot order.
      const float m = __shfl_sync(0xffffffffu, my_v, 0);
      const float ex = (lane < k) ? expf(my_v - m) : 0.f;
      float sum = 0.f;
      for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
      if (lane < k) {
        ids[static_cast<size_t>(t) * k + lane] = my_id;
        wts[static_cast<size_t>(t) * k + lane] = ex / sum;
        atomicOr(&bm[my_id * 2 + (tl >> 5)], 1u << (tl & 31));
        atomicAdd(&cnt[my_id], 1);
      }
    }
  }
  __syncthreads();
  const int chunk = t0 / kChunk;
  const int w0 = (t0 % kChunk) / 32;
  uint32_t* out = gbm + static_cast<size_t>(chunk) * E * kChunkWords;
  for (int i = threadIdx.x; i < 2 * E; i += blockDim.x) out[(i >> 1) * kChunkWords + w0 + (i & 1)] = bm[i];
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (cnt[e] != 0) add_counts(ccount, T, E, e, chunk, cnt[e]);
}

// Fast path of the same selection for E % 4 == 0, E <= 256 and k <= 8: four
// threads per token, each holding a quarter of its logits (16-byte vectors
// 4i + q of the row, so a warp's loads are whole sectors).
//   1. Each thread sorts its values in blocks of 8 (Batcher's 19-comparator
//      network) and merges the blocks keeping the 8 largest (bitonic split +
//      3-stage sort); two shuffle rounds merge the four threads' lists the same
//      way.  Only values move, so no id comparisons are needed: the four
//      threads end with the token's 8 largest values, sorted, s[0] >= ... >= s[7].
//   2. th = s[k-1]; `need` of the top k equal th.  Each thread lists its values
//      >= th (with their ids) in shared memory.  When the token has exactly k
//      such values -- no extra ties at the threshold, the usual case -- all of
//      them are chosen; otherwise one thread rescans the row in ascending id
//      order, taking every value > th and the first `need` equal to th.
//   3. Slot of a chosen (x, e): #{m < k : s[m] > x}, plus, when x occurs more
//      than once in the top k, the number of chosen equal values with a lower
//      id -- the total order (value desc, id asc) of the warp-per-token path.
// Weights: exp(s[m] - s[0]) summed over m < k in slot order, then
// exp(x - s[0]) / sum: the same arithmetic as the warp-per-token path.
// Non-finite logits are detected with one fused multiply-add per value
// (x * 0 is NaN exactly for NaN and +-inf); a warp that holds one maps them to
// -inf and reports MOE_ERR_NONFINITE, as the warp-per-token path does.
constexpr int kTopkFastK = 8;

// Compare-exchange, descending.
__device__ __forceinline__ void cx_desc(float& a, float& b) {
  const float hi = fmaxf(a, b), lo = fminf(a, b);
  a = hi;
  b = lo;
}

// Sorts 8 values descending (Batcher's odd-even merge sort, 19 comparators).
__device__ __forceinline__ void sort8_desc(float* a) {
  cx_desc(a[0], a[1]); cx_desc(a[2], a[3]); cx_desc(a[4], a[5]); cx_desc(a[6], a[7]);
  cx_desc(a[0], a[2]); cx_desc(a[1], a[3]); cx_desc(a[4], a[6]); cx_desc(a[5], a[7]);
  cx_desc(a[1], a[2]); cx_desc(a[5], a[6]);
  cx_desc(a[0], a[4]); cx_desc(a[1], a[5]); cx_desc(a[2], a[6]); cx_desc(a[3], a[7]);
  cx_desc(a[2], a[4]); cx_desc(a[3], a[5]);
  cx_desc(a[1], a[2]); cx_desc(a[3], a[4]); cx_desc(a[5], a[6]);
}

// a := the 8 largest of a and b (both sorted descending), sorted descending.
__device__ __forceinline__ void merge8_top(float* a, const float* b) {
#pragma unroll
  for (int m = 0; m < 8; ++m) a[m] = fmaxf(a[m], b[7 - m]);
#pragma unroll
  for (int d = 4; d > 0; d >>= 1)
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if ((m & d) == 0) cx_desc(a[m], a[m + d]);
}

// KC: k when it is known at compile time (8, the usual value: every `m < k` test
// of the unrolled 8-slot loops then folds away), 0 for a runtime k.
template <int NV4, bool FULL, int KC>
__global__ void __launch_bounds__(kTopkThreads) route_topk4_kernel(const float* __restrict__ logits, int T, int E,
                                                                   int k_arg, int32_t* __restrict__ ids,
                                                                   float* __restrict__ wts,
                                                                   uint32_t* __restrict__ gbm,
                                                                   int32_t* __restrict__ ccount, WsHeader* ws) {
  const int k = KC ? KC : k_arg;
  constexpr int NV = 4 * NV4;                    // values per thread
  constexpr int NB = (NV + 7) / 8;               // blocks of 8
  extern __shared__ uint32_t sm[];
  uint32_t* bm = sm;                             // [E][2]
  int* cnt = reinterpret_cast<int*>(sm + 2 * E); // [E]
  float* cand_x = reinterpret_cast<float*>(cnt + E);  // [64 tokens][8] chosen values (tie path)
  for (int i = threadIdx.x; i < 3 * E; i += blockDim.x) sm[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int tl = threadIdx.x >> 2, q = threadIdx.x & 3;
  const int t = blockIdx.x * kTopkTokens + tl;
  const bool live = t < T;
  const float* row = logits + static_cast<size_t>(live ? t : 0) * E;

  float v[NB * 8];
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    const int e0 = 16 * i + 4 * q;
    float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (live && (FULL || e0 < E)) {
      f = __ldg(reinterpret_cast<const float4*>(row + e0));
      acc = fmaf(f.x, 0.f, acc);
      acc = fmaf(f.y, 0.f, acc);
      acc = fmaf(f.z, 0.f, acc);
      acc = fmaf(f.w, 0.f, acc);
    }
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
#pragma unroll
  for (int j = NV; j < NB * 8; ++j) v[j] = -INFINITY;
  const bool bad = acc != acc;
  if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
    for (int j = 0; j < NV; ++j)
      if (!isfinite(v[j])) v[j] = -INFINITY;
    if (bad) report(ws, MOE_ERR_NONFINITE, 0, t);
  }

  // 1. the token's 8 largest values, sorted
  float s[8];
  {
    float b[NB][8];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
      for (int m = 0; m < 8; ++m) b[blk][m] = v[8 * blk + m];
      sort8_desc(b[blk]);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) s[m] = b[0][m];
#pragma unroll
    for (int blk = 1; blk < NB; ++blk) merge8_top(s, b[blk]);
  }
#pragma unroll
  for (int mask = 1; mask <= 2; mask <<= 1) {
    float o[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) o[m] = __shfl_xor_sync(0xffffffffu, s[m], mask);
    merge8_top(s, o);
  }
  float th = s[0];
#pragma unroll
  for (int m = 1; m < 8; ++m)
    if (m < k) th = s[m];
  int need = 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) need += (m < k && s[m] == th) ? 1 : 0;

  // 2. this thread's values >= th, as a bit mask over its value index j
  //    (value j of thread q is expert 16 (j / 4) + 4 q + j % 4)
  using Mask = typename std::conditional<(NV > 32), unsigned long long, uint32_t>::type;
  Mask msk = 0;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e = 16 * (j >> 2) + 4 * q + (j & 3);
    if ((FULL || e < E) && v[j] >= th) msk |= Mask(1) << j;
  }
  const int n = (NV > 32) ? __popcll(static_cast<unsigned long long>(msk)) : __popc(static_cast<uint32_t>(msk));
  int ntot = n;
  ntot += __shfl_xor_sync(0xffffffffu, ntot, 1);
  ntot += __shfl_xor_sync(0xffffffffu, ntot, 2);
  int nq[4];
  Mask mq[4];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    nq[qq] = __shfl_sync(0xffffffffu, n, (lane & ~3) + qq);
    if (NV > 32) {
      const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(msk), (lane & ~3) + qq);
      const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(static_cast<unsigned long long>(msk) >> 32),
                                      (lane & ~3) + qq);
      mq[qq] = static_cast<Mask>((static_cast<unsigned long long>(hi) << 32) | lo);
    } else {
      mq[qq] = static_cast<Mask>(__shfl_sync(0xffffffffu, static_cast<uint32_t>(msk), (lane & ~3) + qq));
    }
  }
  // Expert of the li-th set bit of thread qq's mask.
  auto expert_of = [&](int qq, int li) {
    const Mask m = qq == 0 ? mq[0] : qq == 1 ? mq[1] : qq == 2 ? mq[2] : mq[3];
    int j;
    if (NV > 32) {
      const uint32_t lo = static_cast<uint32_t>(static_cast<unsigned long long>(m));
      const int nlo = __popc(lo);
      j = li < nlo ? static_cast<int>(__fns(lo, 0, li + 1))
                   : 32 + static_cast<int>(__fns(static_cast<uint32_t>(static_cast<unsigned long long>(m) >> 32),
                                                 0, li - nlo + 1));
    } else {
      j = static_cast<int>(__fns(static_cast<uint32_t>(m), 0, li + 1));
    }
    return 16 * (j >> 2) + 4 * qq + (j & 3);
  };

  // Weights: exp(s[m] - s[0]) for m = q and q + 4 here, gathered over the
  // token's four threads and summed in slot order.
  const float m0 = s[0];
  const float sq = q == 0 ? s[0] : q == 1 ? s[1] : q == 2 ? s[2] : s[3];
  const float sq4 = q == 0 ? s[4] : q == 1 ? s[5] : q == 2 ? s[6] : s[7];
  const float exa = (live && q < k) ? expf(sq - m0) : 0.f;
  const float exb = (live && q + 4 < k) ? expf(sq4 - m0) : 0.f;
  float ex[8];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    ex[m] = __shfl_sync(0xffffffffu, exa, (lane & ~3) + m);
    ex[m + 4] = __shfl_sync(0xffffffffu, exb, (lane & ~3) + m);
  }
  float sum = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m)
    if (m < k) sum += ex[m];
  if (live) {
    // 3. slots of the chosen values; writes
    auto emit = [&](float x, int e, int ties_below) {
      int slot = ties_below;
#pragma unroll
      for (int m = 0; m < 8; ++m) slot += (m < k && s[m] > x) ? 1 : 0;
      if (e < 0 || e >= E || slot >= k) {
        report(ws, MOE_ERR_BOUNDS, 1, t);
        return;
      }
      float exs = ex[0];
#pragma unroll
      for (int m = 1; m < 8; ++m)
        if (slot == m) exs = ex[m];
      ids[static_cast<size_t>(t) * k + slot] = e;
      wts[static_cast<size_t>(t) * k + slot] = exs / sum;
      atomicOr(&bm[e * 2 + (tl >> 5)], 1u << (tl & 31));
      atomicAdd(&cnt[e], 1);
    };
    if (ntot == k) {
      // The token's k chosen values, spread evenly: this thread takes entries
      // q and q + 4 of the concatenation of the four threads' lists; the
      // values are read back from the row (an L1 hit).
      for (int c = q; c < k; c += 4) {
        const int qq = c < nq[0] ? 0 : c < nq[0] + nq[1] ? 1 : c < nq[0] + nq[1] + nq[2] ? 2 : 3;
        const int li = c - (qq > 0 ? nq[0] : 0) - (qq > 1 ? nq[1] : 0) - (qq > 2 ? nq[2] : 0);
        const int e = expert_of(qq, li);
        float x = __ldg(row + e);
        if (!isfinite(x)) x = -INFINITY;
        int dup = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) dup += (m < k && s[m] == x) ? 1 : 0;
        int ties_below = 0;
        if (dup > 1) {  // equal chosen values: the lower ids take the earlier slots
          for (int q2 = 0; q2 < 4; ++q2)
            for (int l2 = 0; l2 < nq[q2]; ++l2) {
              const int e2 = expert_of(q2, l2);
              float x2 = __ldg(row + e2);
              if (!isfinite(x2)) x2 = -INFINITY;
              ties_below += (x2 == x && e2 < e) ? 1 : 0;
            }
        }
        emit(x, e, ties_below);
      }
    } else if (q == 0) {
      // More values equal th than slots left: ascending id order, every value
      // > th and the first `need` equal to th; equal chosen values take slots
      // in id order.
      float* chosen = cand_x + tl * kTopkFastK;
      int left = need, nch = 0;
      for (int e = 0; e < E && nch < k; ++e) {
        float x = row[e];
        if (!isfinite(x)) x = -INFINITY;
        if (!(x > th || (x == th && left > 0))) continue;
        if (!(x > th)) --left;
        int below = 0;
        for (int c = 0; c < nch; ++c) below += (chosen[c] == x) ? 1 : 0;
        chosen[nch++] = x;
        emit(x, e, below);
      }
    }
  }
  __syncthreads();
  const int t0 = blockIdx.x * kTopkTokens;
  const int chunk = t0 / kChunk;
  const int w0 = (t0 % kChunk) / 32;
  uint32_t* out = gbm + static_cast<size_t>(chunk) * E * kChunkWords;
  for (int i = threadIdx.x; i < 2 * E; i += blockDim.x) out[(i >> 1) * kChunkWords + w0 + (i & 1)] = bm[i];
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (cnt[e] != 0) add_counts(ccount, T, E, e, chunk, cnt[e]);
}

// One CTA per 256-token chunk: stable index = popcount of the chunk's bitmap
// below the token; dest, row_src, row_slot.  The chunk's rows of expert e form
// one run [base_e, base_e + c_e) of the grouped buffer, so the inverse table is
// first assembled in shared memory in expert order and then written run by
// run (contiguous stores instead of one scattered store per row).  Each CTA
// also writes its share of the 128-row tile entries {expert, first row, rows}.
//
// The prefix of Algorithm 1 over the sources comes in two levels, with no
// kernel of its own: the top-k CTAs added every count to its chunk and to its
// super-chunk (32 chunks), so the rows of expert e in the chunks before this
// one are the super-chunks before it plus the chunks before it in its own
// super-chunk (at most 31), and e's total is the sum of its super-chunks.  Every
// CTA takes the exclusive prefix over experts of the totals itself (offsets,
// first 128-row tile, first 256-row pair); CTA 0 also writes them, the counts,
// the GEMM row counts and, with a padding granule, the padding rows' markers.
constexpr int kRankItems = 8;  // items per thread whose ids are loaded before the prologue

__global__ void __launch_bounds__(256) route_rank_kernel(const int32_t* __restrict__ ids,
                                                         const uint32_t* __restrict__ gbm,
                                                         const int32_t* __restrict__ ccount, int T, int E, int k,
                                                         int R, int pad, int32_t* __restrict__ dest,
                                                         int32_t* __restrict__ row_src,
                                                         uint8_t* __restrict__ row_slot,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ tiles, int32_t* __restrict__ pairs,
                                                         int32_t* __restrict__ gcounts, WsHeader* ws) {
  extern __shared__ uint32_t sm[];
  __shared__ int s_wsum[4][8];
  uint32_t* words = sm;                                      // [E][8] the chunk's bitmap words
  uint32_t* lpre = words + kChunkWords * E;                  // [E][8] rank within the chunk of each word's first token
  int* base = reinterpret_cast<int*>(lpre + kChunkWords * E);  // [E] first grouped row of the chunk's run of e
  int* loff = base + E;                                      // [E + 1] start of e's run in the staging arrays
  int* tstart = loff + E + 1;                                // [E + 1] first tile of each expert
  int* offs = tstart + E + 1;                                // [E + 1] first grouped row of each expert
  int* gcnt = offs + E + 1;                                  // [E] rows each expert's GEMMs run (padded)
  int* st_src = gcnt + E;                                    // [256 k] staging: token of each run position
  uint16_t* st_e = reinterpret_cast<uint16_t*>(st_src + kChunk * k);  // expert of each run position
  uint8_t* st_slot = reinterpret_cast<uint8_t*>(st_e + kChunk * k);   // slot of each run position
  const int chunk = blockIdx.x;
  const int t0 = chunk * kChunk;
  const int n_items = min(kChunk, T - t0) * k;
  const int32_t* my_ids = ids + static_cast<size_t>(t0) * k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool writer = blockIdx.x == 0;
  // Item i is slot i % k of token t0 + i / k.  The first kRankItems ids of
  // this thread are loaded before the prologue so their latency overlaps it.
  int ev[kRankItems];
#pragma unroll
  for (int u = 0; u < kRankItems; ++u) {
    const int i = threadIdx.x + 256 * u;
    ev[u] = (i < n_items) ? __ldg(my_ids + i) : 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(gbm + static_cast<size_t>(chunk) * E * kChunkWords);
  const int nchunks = static_cast<int>(gridDim.x);
  const int nsuper = (nchunks + kSuperChunks - 1) / kSuperChunks;
  const int32_t* sc = ccount + static_cast<size_t>(E) * nchunks;
  const int s0 = chunk / kSuperChunks;
  auto padded = [pad](int n) { return pad > 1 ? (n + pad - 1) / pad * pad : n; };
  // Thread tid owns experts [tid * per, tid * per + per): their words, local
  // prefixes, chunk counts, rows before this chunk and totals; block-wide scans
  // give loff (over the chunk's counts) and the expert-level prefixes.
  // Rows of each expert before this chunk and in all.  Expert e's items are its
  // super-chunk counts (nsuper) and the counts of the chunks before this one in
  // its own super-chunk (fewer than 32), both contiguous; a group of tpe
  // threads (a power of two, 256 / E rounded down, at most 32, at least 1)
  // shares them and sums them with shuffles.  Every warp runs the same number
  // of rounds, so the shuffles always have all 32 lanes.
  {
    const int c0 = s0 * kSuperChunks;
    const int n_sup = nsuper, n_items_e = nsuper + (chunk - c0);
    int tpe = 1;
    while (tpe < 32 && tpe * 2 * E <= 256) tpe *= 2;
    const int groups = 256 / tpe, g0 = threadIdx.x / tpe, li = threadIdx.x % tpe;
    for (int round = 0; round * groups < E; ++round) {
      const int e = round * groups + g0;
      int tot = 0, before = 0;
      if (e < E) {
        const int32_t* scr = sc + static_cast<size_t>(e) * nsuper;
        const int32_t* ccr = ccount + static_cast<size_t>(e) * nchunks + c0;
#pragma unroll 4
        for (int j = li; j < n_items_e; j += tpe) {
          if (j < n_sup) {
            const int v = __ldg(scr + j);
            tot += v;
            before += j < s0 ? v : 0;
          } else {
            before += __ldg(ccr + (j - n_sup));
          }
        }
      }
      for (int off = 1; off < tpe; off <<= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, off);
        before += __shfl_xor_sync(0xffffffffu, before, off);
      }
      if (li == 0 && e < E) {
        base[e] = before;  // the expert's first row is added below
        gcnt[e] = tot;     // the real total for now; padded below
      }
    }
  }
  __syncthreads();
  const int per = (E + 255) / 256;
  int my_cnt = 0, my_n = 0, my_m = 0, my_p = 0;
  for (int u = 0; u < per; ++u) {
    const int e = threadIdx.x * per + u;
    if (e >= E) break;
    const uint4 a = __ldg(src + 2 * e), b = __ldg(src + 2 * e + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const int tot = gcnt[e];
    uint32_t run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      words[e * 8 + j] = w[j];
      lpre[e * 8 + j] = run;
      run += __popc(w[j]);
    }
    loff[e] = my_cnt;  // thread-local prefixes, completed below
    my_cnt += static_cast<int>(run);
    const int n = padded(tot);
    my_n += n;
    my_m += (n + kTileRows - 1) / kTileRows;
    my_p += (n + 2 * kTileRows - 1) / (2 * kTileRows);
  }
  int in_c = my_cnt, in_n = my_n, in_m = my_m, in_p = my_p;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int yc = __shfl_up_sync(0xffffffffu, in_c, off);
    const int yn = __shfl_up_sync(0xffffffffu, in_n, off);
    const int ym = __shfl_up_sync(0xffffffffu, in_m, off);
    const int yp = __shfl_up_sync(0xffffffffu, in_p, off);
    if (lane >= off) {
      in_c += yc;
      in_n += yn;
      in_m += ym;
      in_p += yp;
    }
  }
  if (lane == 31) {
    s_wsum[0][warp] = in_c;
    s_wsum[1][warp] = in_n;
    s_wsum[2][warp] = in_m;
    s_wsum[3][warp] = in_p;
  }
  __syncthreads();
  int run_c = in_c - my_cnt, run_n = in_n - my_n, run_m = in_m - my_m, run_p = in_p - my_p;
  for (int w = 0; w < warp; ++w) {
    run_c += s_wsum[0][w];
    run_n += s_wsum[1][w];
    run_m += s_wsum[2][w];
    run_p += s_wsum[3][w];
  }
  for (int u = 0; u < per; ++u) {
    const int e = threadIdx.x * per + u;
    if (e >= E) break;
    const int real = gcnt[e];
    const int n = padded(real);
    loff[e] += run_c;
    offs[e] = run_n;
    tstart[e] = run_m;
    base[e] += run_n;
    gcnt[e] = n;
    if (writer) {
      counts[e] = real;
      gcounts[e] = n;
      offsets[e] = run_n;
      tiles[1 + e] = run_m;
      pairs[e] = run_p;
      for (int r = run_n + real; r < run_n + n; ++r) {  // the padding rows of expert e
        if (r < 0 || r >= R) {
          report(ws, MOE_ERR_BOUNDS, 1, r);
          break;
        }
        row_src[r] = -1;
        row_slot[r] = 255;
      }
    }
    run_n += n;
    run_m += (n + kTileRows - 1) / kTileRows;
    run_p += (n + 2 * kTileRows - 1) / (2 * kTileRows);
    if (e == E - 1) {
      loff[E] = run_c + my_cnt;  // the chunk's items (run_c: this thread's exclusive prefix)
      offs[E] = run_n;
      tstart[E] = run_m;
      if (writer) {
        offsets[E] = run_n;
        tiles[1 + E] = run_m;
        tiles[0] = run_m;
        pairs[E] = run_p;
      }
    }
  }
  __syncthreads();

  auto place = [&](int i, int e) {
    const int tl = i / k, j = i - tl * k;
    const int t = t0 + tl;
    if (e < 0 || e >= E) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      return;
    }
    const int w = tl >> 5, b = tl & 31;
    const int rho = static_cast<int>(lpre[e * 8 + w] + __popc(words[e * 8 + w] & ((1u << b) - 1u)));
    const int r = base[e] + rho;
    if (r < 0 || r >= R) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      return;
    }
    dest[static_cast<size_t>(t0) * k + i] = r;
    const int pos = loff[e] + rho;
    if (pos < 0 || pos >= kChunk * k) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      return;
    }
    st_src[pos] = t;
    st_e[pos] = static_cast<uint16_t>(e);
    st_slot[pos] = static_cast<uint8_t>(j);
  };
#pragma unroll
  for (int u = 0; u < kRankItems; ++u) {
    const int i = threadIdx.x + 256 * u;
    if (i < n_items) place(i, ev[u]);
  }
  for (int i = threadIdx.x + 256 * kRankItems; i < n_items; i += 256) place(i, __ldg(my_ids + i));
  __syncthreads();
  // Run positions in expert order -> consecutive grouped rows.
  const int n_pos = min(loff[E], kChunk * k);
  for (int pos = threadIdx.x; pos < n_pos; pos += 256) {
    const int e = st_e[pos];
    const int r = e < E ? base[e] + (pos - loff[e]) : -1;
    if (r < 0 || r >= R) {
      report(ws, MOE_ERR_BOUNDS, 2, t0);
      continue;
    }
    row_src[r] = st_src[pos];
    row_slot[r] = st_slot[pos];
  }

  // Tile entries [m0, m1) of this CTA: the expert of tile m is the last e
  // with tstart[e] <= m.
  const int ntiles = tstart[E];
  const int tper = (ntiles + gridDim.x - 1) / gridDim.x;
  const int m0 = blockIdx.x * tper, m1 = min(ntiles, m0 + tper);
  int4* ent = reinterpret_cast<int4*>(tiles + tiles_entry_base(E));
  for (int m = m0 + threadIdx.x; m < m1; m += blockDim.x) {
    int lo = 0, hi = E;  // tstart[lo] <= m < tstart[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tstart[mid] <= m)
        lo = mid;
      else
        hi = mid;
    }
    const int j = m - tstart[lo];
    const int n = gcnt[lo];  // rows the GEMMs run: n_e, padded
    ent[m] = make_int4(lo, offs[lo] + kTileRows * j, min(kTileRows, n - kTileRows * j), 0);
  }
}

cudaError_t launch_plan(const PlanLaunch& p, cudaStream_t s, LaunchHook& hook) {
  const int nchunks = (p.T + kChunk - 1) / kChunk;
  const int nblocks = (p.T + kTopkTokens - 1) / kTopkTokens;
  const int nv = (p.E + 31) / 32;
  // The chunk and super-chunk counts start at zero (the bitmap words are all
  // written by the top-k CTAs).
  cudaError_t err = cudaMemsetAsync(p.ticket, 0, static_cast<size_t>(plan_count_words(p.T, p.E)) * 4, s);
  if (err != cudaSuccess) return err;
  const size_t topk_smem = static_cast<size_t>(p.E) * 3 * 4;
  hook.before(s);
  const int nv4 = (p.E + 15) / 16;
  if (p.E % 4 == 0 && p.E <= 256 && p.k <= kTopkFastK) {
    const size_t smem4 = (static_cast<size_t>(p.E) * 3 + static_cast<size_t>(kTopkTokens) * kTopkFastK) * 4;
    const bool full = (p.E % 16) == 0;
    switch ((nv4 <= 1 ? 1 : nv4 <= 2 ? 2 : nv4 <= 4 ? 4 : nv4 <= 8 ? 8 : 16) * (full ? 1 : -1)) {
#define MOE_TOPK4_CASE(NV4, FULL)                                                                              \
  case (FULL ? NV4 : -NV4):                                                                                    \
    if (p.k == 8)                                                                                              \
      route_topk4_kernel<NV4, FULL, 8><<<nblocks, kTopkThreads, smem4, s>>>(p.logits, p.T, p.E, p.k, p.ids,    \
                                                                            p.w, p.gbm, p.ccount, p.ws);       \
    else                                                                                                       \
      route_topk4_kernel<NV4, FULL, 0><<<nblocks, kTopkThreads, smem4, s>>>(p.logits, p.T, p.E, p.k, p.ids,    \
                                                                            p.w, p.gbm, p.ccount, p.ws);       \
    break;
      MOE_TOPK4_CASE(1, true)
      MOE_TOPK4_CASE(2, true)
      MOE_TOPK4_CASE(4, true)
      MOE_TOPK4_CASE(8, true)
      MOE_TOPK4_CASE(16, true)
      MOE_TOPK4_CASE(1, false)
      MOE_TOPK4_CASE(2, false)
      MOE_TOPK4_CASE(4, false)
      MOE_TOPK4_CASE(8, false)
      MOE_TOPK4_CASE(16, false)
#undef MOE_TOPK4_CASE
    }
  } else {
  switch (nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 8 ? 8 : nv <= 16 ? 16 : 32) {
#define MOE_TOPK_CASE(NV, TPW)                                                                                 \
  case NV:                                                                                                     \
    route_topk_kernel<NV, TPW><<<nblocks, kTopkThreads, topk_smem, s>>>(p.logits, p.T, p.E, p.k, p.ids, p.w, \
                                                                        p.gbm, p.ccount, p.ws);              \
    break;
    MOE_TOPK_CASE(1, 8)
    MOE_TOPK_CASE(2, 8)
    MOE_TOPK_CASE(4, 4)
    MOE_TOPK_CASE(8, 2)
    MOE_TOPK_CASE(16, 1)
    MOE_TOPK_CASE(32, 1)
#undef MOE_TOPK_CASE
  }
  }
  hook.after(s);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  hook.before(s);
  const size_t rank_smem = (static_cast<size_t>(2 * kChunkWords) * p.E + 5 * static_cast<size_t>(p.E) + 3) * 4 +
                           static_cast<size_t>(kChunk) * p.k * 7;
  if (rank_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(route_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(rank_smem));
    if (err != cudaSuccess) return err;
  }
  route_rank_kernel<<<nchunks, 256, rank_smem, s>>>(p.ids, p.gbm, p.ccount, p.T, p.E, p.k, p.R, p.pad, p.dest,
                                                    p.row_src, p.row_slot, p.counts, p.offsets, p.tiles, p.pairs,
                                                    p.gcounts, p.ws);
  hook.after(s);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Routing without a caller-provided workspace (moe_plan_noalloc).
//
// For callers that may not allocate device memory while they run, the scratch
// of the three routing kernels (per-chunk counts, bases and bitmaps) lives in
// the file-scope array below.  Host code must not use the array's name as a
// device address: it only names a host-side stand-in.  The device address is
// looked up with cudaGetSymbolAddress (with the device current) and passed to
// the kernels like any workspace pointer.
//
// The address belongs to one CUDA context: another context on the same device
// (a driver-API context an engine creates, or the primary context recreated
// after cudaDeviceReset) holds its own copy of the array at another address.
// The lookup is therefore cached per context, keyed on the context's unique id
// (cuCtxGetId: ids are never reused within a process, unlike context handles),
// and redone for every context not seen before.
// ---------------------------------------------------------------------------
#include <mutex>

namespace moe {
namespace {

constexpr size_t kNoAllocBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocCache = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
struct NoAllocEntry {
  unsigned long long ctx_id;
  void* ptr;
};
NoAllocEntry g_noalloc_cache[kNoAllocCache];
int g_noalloc_used = 0, g_noalloc_next = 0;

size_t na_align(size_t v) { return (v + 255) & ~size_t(255); }

// Unique id of the calling thread's current context (0 if none or unknown).
unsigned long long current_ctx_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
    resolved = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current context (looked up once
// per context; the lookup itself makes the device's primary context current
// when the thread has none yet).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_LAUNCH;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  unsigned long long id = current_ctx_id();
  if (id != 0)
    for (int i = 0; i < g_noalloc_used; ++i)
      if (g_noalloc_cache[i].ctx_id == id) {
        *out = g_noalloc_cache[i].ptr;
        return MOE_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_LAUNCH;
  if (id == 0) id = current_ctx_id();  // the lookup may have made the primary context current
  if (id != 0) {
    const int slot = g_noalloc_used < kNoAllocCache ? g_noalloc_used++ : (g_noalloc_next++ % kNoAllocCache);
    g_noalloc_cache[slot] = NoAllocEntry{id, p};
  }
  *out = p;
  return MOE_OK;
}

bool na_ok_ptr(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_plan_noalloc(moe_dims d, const float* logits, const moe_plan_t* plan, int32_t* status,
                                void* stream) {
  using namespace moe;
  if (d.T < 0 || d.H <= 0 || d.F <= 0 || d.E <= 0 || d.k <= 0 || d.k > d.E || d.k > 32 || d.pad < 0 ||
      d.pad > kMaxPad || grouped_rows(d.T, d.k, d.E, d.pad) >= (1ll << 31))
    return MOE_ERR_ARG;
  if (d.H % 128 != 0 || d.F % 128 != 0 || d.E > 1024) return MOE_ERR_SHAPE;
  const size_t nchunks = (static_cast<size_t>(d.T) + kChunk - 1) / kChunk;
  const size_t ccount = 0;  // 16-word header, then the per-chunk and per-super-chunk counts
  const size_t gbm = na_align(ccount + static_cast<size_t>(plan_count_words(d.T, d.E)) * 4);
  const size_t total = na_align(gbm + nchunks * d.E * kChunkWords * 4);
  if (total > kNoAllocBytes) return MOE_ERR_TOO_LARGE;
  if (d.T == 0) return MOE_OK;
  if (plan == nullptr || plan->row_slot == nullptr) return MOE_ERR_ARG;
  const void* ptrs[] = {logits, status, plan->topk_ids, plan->topk_w, plan->counts, plan->offsets, plan->dest,
                        plan->row_src, plan->tiles};
  for (const void* q : ptrs) {
    if (q == nullptr) return MOE_ERR_ARG;
    if (!na_ok_ptr(q)) return MOE_ERR_ALIGN;
  }
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != MOE_OK) return rc;
  uint8_t* w = static_cast<uint8_t*>(scratch);
  PlanLaunch p;
  p.logits = logits;
  p.T = d.T;
  p.E = d.E;
  p.k = d.k;
  p.pad = d.pad;
  const long long R = grouped_rows(d.T, d.k, d.E, d.pad);
  p.R = static_cast<int>(R);
  p.ids = plan->topk_ids;
  p.w = plan->topk_w;
  p.ticket = reinterpret_cast<int32_t*>(w + ccount);
  p.ccount = p.ticket + 16;
  p.gbm = reinterpret_cast<uint32_t*>(w + gbm);
  p.counts = plan->counts;
  p.offsets = plan->offsets;
  p.tiles = plan->tiles;
  p.pairs = plan->tiles + tiles_pair_base(R, d.E);
  p.gcounts = plan->tiles + tiles_gcount_base(R, d.E);
  p.dest = plan->dest;
  p.row_src = plan->row_src;
  p.row_slot = plan->row_slot;
  p.ws = reinterpret_cast<WsHeader*>(status);  // only status/where/detail are written
  LaunchHook hook;
  return launch_plan(p, static_cast<cudaStream_t>(stream), hook) == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
