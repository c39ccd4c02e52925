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
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kTopkTokens = 64;    // tokens per CTA of the warp-per-token top-k: two bitmap words per expert
constexpr int kTopkThreads = 256;  // 8 warps x 8 tokens
constexpr int kTopk4Tokens = 64;   // tokens per CTA of the four-threads-per-token top-k

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
//
// Every logit becomes one 32-bit key that carries its expert id:
//   key = (okey(x) with the low 8 bits cleared) | (255 - e),
// okey being an integer that orders like the float (-0 and +0 equal).  Keys
// compare like (x desc, e asc) except between two logits whose okeys agree in
// their top 24 bits (the key's "prefix"), where only the id decides.
//   1. Each thread sorts its keys in blocks of 8 (Batcher's 19-comparator
//      network, one integer min and max per comparator) and merges the blocks
//      keeping the 8 largest (bitonic split + 3-stage sort); two shuffle rounds
//      merge the four threads' lists the same way.  The ids ride along in the
//      keys, so the four threads end with the token's top 8 (value, id) pairs,
//      in slot order, with no search for the chosen ids.
//   2. The packed order is the exact order unless a prefix is shared where it
//      matters: two of the top k with one prefix, or a key outside the top k
//      with the prefix of the k-th.  The first shows in the sorted list; the
//      second in how many keys of each thread's own top 8 reach the k-th key's
//      prefix (a thread whose eight all do may hide more: counted as one more).
//      Such a token (a shared prefix among ~9 values: rare for real-valued
//      logits; always for exact ties, which the packed order gets right anyway)
//      is selected again with 64-bit keys okey << 32 | (255 - e), an exact
//      total order, through the same networks.
// Weights: exp(x_m - x_0) summed over m < k in slot order, then
// exp(x - x_0) / sum, with x_m the chosen logits read back from the row (an L1
// hit): the same arithmetic as the warp-per-token path.
// Non-finite logits are detected with one fused multiply-add per value
// (x * 0 is NaN exactly for NaN and +-inf); they take part as -inf and the
// warp reports MOE_ERR_NONFINITE, as the warp-per-token path does.
constexpr int kTopkFastK = 8;

// An integer that orders like the float (NaN excluded); -0 and +0 map to 0.
__device__ __forceinline__ int32_t okey(float x) {
  const int32_t i = __float_as_int(x);
  const int32_t sgn = i >> 31;
  return ((i & 0x7fffffff) ^ sgn) - sgn;
}

__device__ __forceinline__ int32_t kmax(int32_t a, int32_t b) { return max(a, b); }
__device__ __forceinline__ int32_t kmin(int32_t a, int32_t b) { return min(a, b); }
__device__ __forceinline__ long long kmax(long long a, long long b) { return a > b ? a : b; }
__device__ __forceinline__ long long kmin(long long a, long long b) { return a > b ? b : a; }

// Compare-exchange, descending.
template <class K>
__device__ __forceinline__ void cx_desc(K& a, K& b) {
  const K hi = kmax(a, b), lo = kmin(a, b);
  a = hi;
  b = lo;
}

// Sorts 8 keys descending (Batcher's odd-even merge sort, 19 comparators).
template <class K>
__device__ __forceinline__ void sort8_desc(K* a) {
  cx_desc(a[0], a[1]); cx_desc(a[2], a[3]); cx_desc(a[4], a[5]); cx_desc(a[6], a[7]);
  cx_desc(a[0], a[2]); cx_desc(a[1], a[3]); cx_desc(a[4], a[6]); cx_desc(a[5], a[7]);
  cx_desc(a[1], a[2]); cx_desc(a[5], a[6]);
  cx_desc(a[0], a[4]); cx_desc(a[1], a[5]); cx_desc(a[2], a[6]); cx_desc(a[3], a[7]);
  cx_desc(a[2], a[4]); cx_desc(a[3], a[5]);
  cx_desc(a[1], a[2]); cx_desc(a[3], a[4]); cx_desc(a[5], a[6]);
}

// a := the 8 largest of a and b (both sorted descending), sorted descending.
template <class K>
__device__ __forceinline__ void merge8_top(K* a, const K* b) {
#pragma unroll
  for (int m = 0; m < 8; ++m) a[m] = kmax(a[m], b[7 - m]);
#pragma unroll
  for (int d = 4; d > 0; d >>= 1)
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if ((m & d) == 0) cx_desc(a[m], a[m + d]);
}

// Value slot j of thread q is expert 16 (j / 4) + 4 q + j % 4.
__device__ __forceinline__ int topk4_expert(int j, int q) { return 16 * (j >> 2) + 4 * q + (j & 3); }

// Entry m of an 8-list with a runtime m in [0, 8), without local memory.
template <class K>
__device__ __forceinline__ K pick8(const K* a, int m) {
  K r = a[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if (m == i) r = a[i];
  return r;
}

__device__ __forceinline__ float finite_or_ninf(float x) { return isfinite(x) ? x : -INFINITY; }

// The low byte of value slot j's key before the thread's own id bits are
// added: 255 - (16 (j / 4) + j % 4), whose bits 2-3 (the thread's 4 q) are set.
// After the thread's own selection, XOR with 4 q turns it into 255 - e.
__device__ __forceinline__ int32_t slot_id_bits(int j) { return 0xff - (16 * (j >> 2) + (j & 3)); }

// Unit u's logits held by thread (tl, q): 16-byte vectors 4i + q of the row.
// Vectors past the row or past the last token are zeros: zeros pass the
// finiteness test, their keys are replaced, and nothing of a dead token is
// written.
template <int NV4, bool FULL, int TOK>
__device__ __forceinline__ void topk4_load(float4* f, const float* logits, int T, int E, int u, int tl, int q) {
  const int t = u * TOK + tl;
  const float* row = logits + static_cast<size_t>(t < T ? t : 0) * E;
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    const int e0 = 16 * i + 4 * q;
    f[i] = (t < T && (FULL || e0 < E)) ? __ldg(reinterpret_cast<const float4*>(row + e0))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// One CTA of 4 TOK threads per TOK-token unit (TOK = 64: a unit owns two
// bitmap words per expert; 32-token units measured slower).
// KC: k when it is known at compile time (8, the usual value: every `m < k` test
// of the unrolled 8-slot loops then folds away), 0 for a runtime k.
template <int NV4, bool FULL, int KC, int TOK>
__global__ void __launch_bounds__(4 * TOK) route_topk4_kernel(const float* __restrict__ logits, int T, int E,
                                                              int k_arg, int32_t* __restrict__ ids,
                                                              float* __restrict__ wts, uint32_t* __restrict__ gbm,
                                                              int32_t* __restrict__ ccount, WsHeader* ws) {
  const int k = KC ? KC : k_arg;
  constexpr int NV = 4 * NV4;                    // values per thread
  constexpr int NB = (NV + 7) / 8;               // blocks of 8
  constexpr int WPU = TOK / 32;                  // bitmap words per expert of the unit
  extern __shared__ uint32_t sm[];
  uint32_t* bm = sm;                             // [E][WPU]
  int* cnt = reinterpret_cast<int*>(sm + WPU * E);  // [E]
  const int lane = threadIdx.x & 31;
  const int tl = threadIdx.x >> 2, q = threadIdx.x & 3;
  const int u = blockIdx.x;
  // Value slot j of this thread holds a logit of the row: its vector j / 4
  // starts at 16 (j / 4) + 4 q < E (E % 4 == 0), i.e. j / 4 < nh.
  const int nh = FULL ? NV4 : (E - 4 * q + 15) / 16;
  auto held = [&](int j) { return j < NV && (FULL || (j >> 2) < nh); };
  float4 cur[NV4];
  topk4_load<NV4, FULL, TOK>(cur, logits, T, E, u, tl, q);
  for (int i = threadIdx.x; i < (WPU + 1) * E; i += blockDim.x) sm[i] = 0;
  __syncthreads();
  const int t = u * TOK + tl;
  const bool live = t < T;
  const float* row = logits + static_cast<size_t>(live ? t : 0) * E;

  float v[NB * 8];
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    v[4 * i] = cur[i].x;
    v[4 * i + 1] = cur[i].y;
    v[4 * i + 2] = cur[i].z;
    v[4 * i + 3] = cur[i].w;
  }
#pragma unroll
  for (int j = 0; j < NV; ++j) acc = fmaf(v[j], 0.f, acc);
#pragma unroll
  for (int j = NV; j < NB * 8; ++j) v[j] = -INFINITY;
  const bool bad = acc != acc;
  if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = finite_or_ninf(v[j]);
    if (bad) report(ws, MOE_ERR_NONFINITE, 0, t);
  }

  // 1. the token's 8 largest keys, sorted; loc = this thread's own 8 largest
  int32_t loc[8], s[8];
  {
    int32_t b[NB][8];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j = 8 * blk + m;
        b[blk][m] = held(j) ? ((okey(v[j]) & ~0xff) | slot_id_bits(j)) : INT_MIN;
      }
      sort8_desc(b[blk]);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) loc[m] = b[0][m];
#pragma unroll
    for (int blk = 1; blk < NB; ++blk) merge8_top(loc, b[blk]);
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    loc[m] ^= 4 * q;  // low byte: 255 - e (a padding key stays below every logit's key)
    s[m] = loc[m];
  }
#pragma unroll
  for (int mask = 1; mask <= 2; mask <<= 1) {
    int32_t o[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) o[m] = __shfl_xor_sync(0xffffffffu, s[m], mask);
    merge8_top(s, o);
  }

  // 2. exact unless a prefix is shared within the top k or across its edge
  int32_t sk = s[0];
#pragma unroll
  for (int m = 1; m < 8; ++m)
    if (m < k) sk = s[m];
  const int32_t edge = sk & ~0xff;  // the smallest key with the k-th key's prefix
  int c = 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) c += loc[m] >= edge ? 1 : 0;
  c += c == 8 ? 1 : 0;
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  bool amb = c > k;
#pragma unroll
  for (int m = 0; m + 1 < 8; ++m)
    if (m + 1 < k) amb = amb || (static_cast<uint32_t>(s[m] ^ s[m + 1]) >> 8) == 0;
  if (live && amb) {
    // The four threads of the token agree on amb: they alone take this branch.
    const unsigned grp = 0xfu << (lane & ~3);
    long long x8[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) x8[m] = LLONG_MIN;
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
      long long b[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j = 8 * blk + m;
        const int e = topk4_expert(j, q);
        b[m] = held(j) ? static_cast<long long>(
                             (static_cast<unsigned long long>(static_cast<uint32_t>(okey(finite_or_ninf(row[e]))))
                              << 32) |
                             static_cast<unsigned long long>(0xff - e))
                       : LLONG_MIN;
      }
      sort8_desc(b);
      merge8_top(x8, b);
    }
#pragma unroll
    for (int mask = 1; mask <= 2; mask <<= 1) {
      long long o[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) o[m] = __shfl_xor_sync(grp, x8[m], mask);
      merge8_top(x8, o);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) s[m] = static_cast<int32_t>(x8[m]);  // the low word: 255 - e
  }

  // 3. slots q and q + 4 of this token; weights in slot order
  const int ea = 0xff - (pick8(s, q) & 0xff);
  const int eb = 0xff - (pick8(s, q + 4) & 0xff);
  const bool has_a = live && q < k, has_b = live && q + 4 < k;
  const bool ok_a = has_a && ea < E, ok_b = has_b && eb < E;
  const float xa = ok_a ? finite_or_ninf(__ldg(row + ea)) : 0.f;
  const float xb = ok_b ? finite_or_ninf(__ldg(row + eb)) : 0.f;
  const float x0 = __shfl_sync(0xffffffffu, xa, lane & ~3);
  const float exa = has_a ? expf(xa - x0) : 0.f;
  const float exb = has_b ? expf(xb - x0) : 0.f;
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
  auto emit = [&](int e, int slot, float exs) {
    ids[static_cast<size_t>(t) * k + slot] = e;
    wts[static_cast<size_t>(t) * k + slot] = exs / sum;
    atomicOr(&bm[e * WPU + (tl >> 5)], 1u << (tl & 31));
    atomicAdd(&cnt[e], 1);
  };
  if ((has_a && !ok_a) || (has_b && !ok_b)) report(ws, MOE_ERR_BOUNDS, 1, t);
  if (ok_a) emit(ea, q, exa);
  if (ok_b) emit(eb, q + 4, exb);
  __syncthreads();
  const int t0 = u * TOK;
  const int chunk = t0 / kChunk;
  const int w0 = (t0 % kChunk) / 32;
  uint32_t* out = gbm + static_cast<size_t>(chunk) * E * kChunkWords;
  for (int i = threadIdx.x; i < WPU * E; i += blockDim.x) out[(i / WPU) * kChunkWords + w0 + (i % WPU)] = bm[i];
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

// Shared memory is laid out for the random expert of each item: a warp's 32
// items share their bitmap word w but not their expert, so the word table is
// [w][E] (consecutive experts in consecutive banks) and each lookup is one
// 8-byte load of {word, rank of the word's first token}; likewise one 8-byte
// load gives an expert's {first grouped row of the chunk's run, start of its
// run in the staging arrays}.
// KC: k when it is known at compile time (8), 0 for a runtime k.
template <int KC>
__global__ void __launch_bounds__(256) route_rank_kernel(const int32_t* __restrict__ ids,
                                                         const uint32_t* __restrict__ gbm,
                                                         const int32_t* __restrict__ ccount, int T, int E, int k_arg,
                                                         int R, int pad, int32_t* __restrict__ dest,
                                                         int32_t* __restrict__ row_src,
                                                         uint8_t* __restrict__ row_slot,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ tiles, int32_t* __restrict__ pairs,
                                                         int32_t* __restrict__ gcounts, WsHeader* ws) {
  const int k = KC ? KC : k_arg;
  extern __shared__ uint32_t sm[];
  __shared__ int s_wsum[4][8];
  uint2* wl = reinterpret_cast<uint2*>(sm);                  // [8][E] {bitmap word, rank of its first token}
  int2* bl = reinterpret_cast<int2*>(wl + kChunkWords * E);  // [E + 1] {first row of e's run, start of its staging run}
  int* tstart = reinterpret_cast<int*>(bl + E + 1);          // [E + 1] first tile of each expert
  int* offs = tstart + E + 1;                                // [E + 1] first grouped row of each expert
  int* gcnt = offs + E + 1;                                  // [E] rows each expert's GEMMs run (padded)
  // [256 k] staging, one word per run position: token in the chunk (bits 0-7),
  // slot (bits 8-12, k <= 32), expert (bits 13-22, E <= 1024).
  uint32_t* st = reinterpret_cast<uint32_t*>(gcnt + E);
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
  // The bitmap words of this thread's first expert, also before the prologue.
  const int per = (E + 255) / 256;
  uint4 wa0 = make_uint4(0, 0, 0, 0), wb0 = make_uint4(0, 0, 0, 0);
  if (threadIdx.x * per < E) {
    wa0 = __ldg(src + 2 * threadIdx.x * per);
    wb0 = __ldg(src + 2 * threadIdx.x * per + 1);
  }
  const int nchunks = static_cast<int>(gridDim.x);
  const int nsuper = (nchunks + kSuperChunks - 1) / kSuperChunks;
  const int32_t* sc = ccount + static_cast<size_t>(E) * nchunks;
  const int s0 = chunk / kSuperChunks;
  auto padded = [pad](int n) { return pad > 1 ? (n + pad - 1) / pad * pad : n; };
  // Thread tid owns experts [tid * per, tid * per + per): their words, local
  // prefixes, chunk counts, rows before this chunk and totals; block-wide scans
  // give the staging run starts (over the chunk's counts) and the expert-level prefixes.
  // Rows of each expert before this chunk and in all.  Expert e's items are its
  // super-chunk counts (nsuper) and the counts of the chunks before this one in
  // its own super-chunk (fewer than 32), both contiguous; a group of tpe
  // threads (a power of two, 256 / E rounded down, at most 32, at least 1)
  // shares them and sums them with shuffles.  Every warp runs the same number
  // of rounds, so the shuffles always have all 32 lanes.
  {
    const int c0 = s0 * kSuperChunks;
    const int n_sup = nsuper, n_items_e = nsuper + (chunk - c0);
    // Both count rows 16-byte aligned (ccount itself is: 16 words past a
    // 16-byte aligned place in the workspace).
    const bool vec = (nchunks & 3) == 0 && (nsuper & 3) == 0;
    int tpe = 1;
    while (tpe < 32 && tpe * 2 * E <= 256) tpe *= 2;
    const int groups = 256 / tpe, g0 = threadIdx.x / tpe, li = threadIdx.x % tpe;
    for (int round = 0; round * groups < E; ++round) {
      const int e = round * groups + g0;
      int tot = 0, before = 0;
      if (e < E) {
        const int32_t* scr = sc + static_cast<size_t>(e) * nsuper;
        const int32_t* ccr = ccount + static_cast<size_t>(e) * nchunks + c0;
        if (vec) {
          // 16-byte vectors, all in flight at once: nsuper / 4 of super-chunk
          // counts, then the chunk counts from c0 (a multiple of 32) up to this
          // chunk, the last vector masked (it ends inside the row: nchunks % 4 == 0).
          const int nvs = nsuper >> 2, lim = chunk - c0, nvc = (lim + 3) >> 2;
#pragma unroll 8
          for (int j = li; j < nvs + nvc; j += tpe) {
            if (j < nvs) {
              const int4 v = __ldg(reinterpret_cast<const int4*>(scr) + j);
              const int b = 4 * j;
              tot += v.x + v.y + v.z + v.w;
              before += (b < s0 ? v.x : 0) + (b + 1 < s0 ? v.y : 0) + (b + 2 < s0 ? v.z : 0) + (b + 3 < s0 ? v.w : 0);
            } else {
              const int4 v = __ldg(reinterpret_cast<const int4*>(ccr) + (j - nvs));
              const int b = 4 * (j - nvs);
              before += (b < lim ? v.x : 0) + (b + 1 < lim ? v.y : 0) + (b + 2 < lim ? v.z : 0) + (b + 3 < lim ? v.w : 0);
            }
          }
        } else {
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
      }
      for (int off = 1; off < tpe; off <<= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, off);
        before += __shfl_xor_sync(0xffffffffu, before, off);
      }
      if (li == 0 && e < E) {
        bl[e].x = before;  // the expert's first row is added below
        gcnt[e] = tot;     // the real total for now; padded below
      }
    }
  }
  __syncthreads();
  int my_cnt = 0, my_n = 0, my_m = 0, my_p = 0;
  for (int u = 0; u < per; ++u) {
    const int e = threadIdx.x * per + u;
    if (e >= E) break;
    const uint4 a = u == 0 ? wa0 : __ldg(src + 2 * e), b = u == 0 ? wb0 : __ldg(src + 2 * e + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const int tot = gcnt[e];
    uint32_t run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      wl[j * E + e] = make_uint2(w[j], run);
      run += __popc(w[j]);
    }
    bl[e].y = my_cnt;  // thread-local prefixes, completed below
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
    bl[e].y += run_c;
    offs[e] = run_n;
    tstart[e] = run_m;
    bl[e].x += run_n;
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
      bl[E].y = run_c + my_cnt;  // the chunk's items (run_c: this thread's exclusive prefix)
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
    const uint2 wr = wl[w * E + e];
    const int rho = static_cast<int>(wr.y + __popc(wr.x & ((1u << b) - 1u)));
    const int2 be = bl[e];
    const int r = be.x + rho;
    if (r < 0 || r >= R) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      return;
    }
    dest[static_cast<size_t>(t0) * k + i] = r;
    const int pos = be.y + rho;
    if (pos < 0 || pos >= kChunk * k) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      return;
    }
    st[pos] = static_cast<uint32_t>(tl) | (static_cast<uint32_t>(j) << 8) | (static_cast<uint32_t>(e) << 13);
  };
#pragma unroll
  for (int u = 0; u < kRankItems; ++u) {
    const int i = threadIdx.x + 256 * u;
    if (i < n_items) place(i, ev[u]);
  }
  for (int i = threadIdx.x + 256 * kRankItems; i < n_items; i += 256) place(i, __ldg(my_ids + i));
  __syncthreads();
  // Run positions in expert order -> consecutive grouped rows.
  const int n_pos = min(bl[E].y, kChunk * k);
  for (int pos = threadIdx.x; pos < n_pos; pos += 256) {
    const uint32_t word = st[pos];
    const int e = static_cast<int>(word >> 13);
    const int2 be = e < E ? bl[e] : make_int2(-1, 0);
    const int r = e < E ? be.x + (pos - be.y) : -1;
    if (r < 0 || r >= R) {
      report(ws, MOE_ERR_BOUNDS, 2, t0);
      continue;
    }
    row_src[r] = t0 + static_cast<int>(word & 0xffu);
    row_slot[r] = static_cast<uint8_t>((word >> 8) & 0x1fu);
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
    const int nv4p = nv4 <= 1 ? 1 : nv4 <= 2 ? 2 : nv4 <= 4 ? 4 : nv4 <= 8 ? 8 : 16;
    const bool full = p.E == 16 * nv4p;  // every one of the 16 * NV4 value slots is a logit of the row
    constexpr int tok = kTopk4Tokens;
    const size_t smem4 = static_cast<size_t>(p.E) * (tok / 32 + 1) * 4;
    const int nunits = (p.T + tok - 1) / tok;
    switch (nv4p * (full ? 1 : -1)) {
#define MOE_TOPK4_CASE(NV4, FULL)                                                                  \
  case (FULL ? NV4 : -NV4):                                                                        \
    if (p.k == 8)                                                                                  \
      route_topk4_kernel<NV4, FULL, 8, tok><<<nunits, 4 * tok, smem4, s>>>(                        \
          p.logits, p.T, p.E, p.k, p.ids, p.w, p.gbm, p.ccount, p.ws);                             \
    else                                                                                           \
      route_topk4_kernel<NV4, FULL, 0, tok><<<nunits, 4 * tok, smem4, s>>>(                        \
          p.logits, p.T, p.E, p.k, p.ids, p.w, p.gbm, p.ccount, p.ws);                             \
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
  const size_t rank_smem = (static_cast<size_t>(2 * kChunkWords) * p.E + 5 * static_cast<size_t>(p.E) + 4) * 4 +
                           static_cast<size_t>(kChunk) * p.k * 4;
  auto rank = p.k == 8 ? route_rank_kernel<8> : route_rank_kernel<0>;
  if (rank_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(rank, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(rank_smem));
    if (err != cudaSuccess) return err;
  }
  rank<<<nchunks, 256, rank_smem, s>>>(p.ids, p.gbm, p.ccount, p.T, p.E, p.k, p.R, p.pad, p.dest, p.row_src,
                                       p.row_slot, p.counts, p.offsets, p.tiles, p.pairs, p.gcounts, p.ws);
  hook.after(s);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Routing without a caller-provided workspace (moe_plan_noalloc).
//
// For callers that may not allocate device memory while they run, the scratch
// of the routing kernels (per-chunk and per-super-chunk counts, bitmaps) lives in
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
