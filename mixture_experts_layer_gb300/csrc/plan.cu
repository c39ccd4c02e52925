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
//   route_topk  one CTA per 64 tokens: warp-wide top-k per token, renormalised
//               weights, and its part of the chunk bitmap bm[e][w] whose bit b
//               says "token 32w+b of the chunk chose expert e" (a warp ballot in
//               shared memory); per-chunk counts by integer atomics.
//   route_scan  one warp per expert: exclusive prefix of the counts over
//               chunks; the last CTA takes the prefix over experts and writes
//               the 128-row GEMM tile table.
//   route_rank  one CTA per 64 tokens: stable index = popcount of the chunk's
//               bitmap below the token; dest, row_src, row_slot.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kTopkTokens = 64;    // tokens per top-k / rank CTA: two bitmap words per expert
constexpr int kTopkThreads = 256;  // 8 warps x 8 tokens
constexpr int kScanWarps = 8;      // experts per scan CTA

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
    if (cnt[e] != 0) atomicAdd(&ccount[static_cast<size_t>(chunk) * E + e], cnt[e]);
}

// Per expert (one warp each): exclusive prefix of the chunk counts over the
// chunks -- the O_all of Algorithm 1 -- and the expert's row count.  The last
// CTA to finish (ticket) then takes the prefix over experts and writes the
// 128-row tile table.
__global__ void __launch_bounds__(32 * kScanWarps) route_scan_kernel(const int32_t* __restrict__ ccount,
                                                                     int nchunks, int E, int32_t* __restrict__ cbase,
                                                                     int32_t* __restrict__ counts,
                                                                     int32_t* __restrict__ offsets,
                                                                     int32_t* __restrict__ tiles, int32_t* ticket) {
  __shared__ int s_last;
  __shared__ int s_wsum_n[32], s_wsum_m[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kScanWarps + warp;
  if (e < E) {
    int run = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
      const int c = c0 + lane;
      const int v = (c < nchunks) ? ccount[static_cast<size_t>(c) * E + e] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (c < nchunks) cbase[static_cast<size_t>(c) * E + e] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[e] = run;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Last CTA: exclusive prefix over experts of the row counts and of the
  // 128-row tile counts.  Thread i takes experts [i * per, (i + 1) * per).
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per;
  int my_n = 0, my_m = 0;
  for (int i = 0; i < per; ++i) {
    const int ee = e0 + i;
    if (ee < E) {
      const int n = __ldcg(counts + ee);
      my_n += n;
      my_m += (n + kTileRows - 1) / kTileRows;
    }
  }
  int in_n = my_n, in_m = my_m;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int yn = __shfl_up_sync(0xffffffffu, in_n, off);
    const int ym = __shfl_up_sync(0xffffffffu, in_m, off);
    if (lane >= off) {
      in_n += yn;
      in_m += ym;
    }
  }
  if (lane == 31) {
    s_wsum_n[warp] = in_n;
    s_wsum_m[warp] = in_m;
  }
  __syncthreads();
  int run_n = in_n - my_n, run_m = in_m - my_m;
  for (int w = 0; w < warp; ++w) {
    run_n += s_wsum_n[w];
    run_m += s_wsum_m[w];
  }
  const int entries = tiles_entry_base(E);
  for (int i = 0; i < per; ++i) {
    const int ee = e0 + i;
    if (ee >= E) break;
    const int n = __ldcg(counts + ee);
    const int mt = (n + kTileRows - 1) / kTileRows;
    offsets[ee] = run_n;
    tiles[1 + ee] = run_m;
    for (int j = 0; j < mt; ++j) {
      int4 ent;
      ent.x = ee;
      ent.y = run_n + kTileRows * j;
      ent.z = min(kTileRows, n - kTileRows * j);
      ent.w = 0;
      reinterpret_cast<int4*>(tiles + entries)[run_m + j] = ent;
    }
    run_n += n;
    run_m += mt;
    if (ee == E - 1) {
      offsets[E] = run_n;
      tiles[1 + E] = run_m;
      tiles[0] = run_m;
    }
  }
}

// One CTA per 64 tokens: stable index = popcount of the chunk's bitmap below
// the token; dest, row_src, row_slot.
__global__ void __launch_bounds__(256) route_rank_kernel(const int32_t* __restrict__ ids,
                                                         const uint32_t* __restrict__ gbm,
                                                         const int32_t* __restrict__ cbase,
                                                         const int32_t* __restrict__ offsets, int T, int E, int k,
                                                         int R, int32_t* __restrict__ dest,
                                                         int32_t* __restrict__ row_src,
                                                         uint8_t* __restrict__ row_slot, WsHeader* ws) {
  extern __shared__ uint32_t sm[];
  uint32_t* words = sm;     // [E][2]: this CTA's two words
  uint32_t* pre = sm + 2 * E;  // [E][2]: popcount of the chunk's words before each
  const int t0 = blockIdx.x * kTopkTokens;
  const int chunk = t0 / kChunk;
  const int w0 = (t0 % kChunk) / 32;
  const uint32_t* src = gbm + static_cast<size_t>(chunk) * E * kChunkWords;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t run = 0;
    for (int w = 0; w < w0; ++w) run += __popc(src[e * kChunkWords + w]);
    const uint32_t a = src[e * kChunkWords + w0], b = src[e * kChunkWords + w0 + 1];
    words[2 * e] = a;
    words[2 * e + 1] = b;
    pre[2 * e] = run;
    pre[2 * e + 1] = run + __popc(a);
  }
  __syncthreads();
  const int n_items = min(kTopkTokens, T - t0) * k;
  for (int i = threadIdx.x; i < n_items; i += blockDim.x) {
    const int tl = i / k, j = i - tl * k;
    const int t = t0 + tl;
    const size_t tk = static_cast<size_t>(t) * k + j;
    const int e = ids[tk];
    if (e < 0 || e >= E) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      continue;
    }
    const int w = tl >> 5, b = tl & 31;
    const int rank = pre[2 * e + w] + __popc(words[2 * e + w] & ((1u << b) - 1u));
    const int r = offsets[e] + cbase[static_cast<size_t>(chunk) * E + e] + rank;
    if (r < 0 || r >= R) {
      report(ws, MOE_ERR_BOUNDS, 2, t);
      continue;
    }
    dest[tk] = r;
    row_src[r] = t;
    row_slot[r] = static_cast<uint8_t>(j);
  }
}

cudaError_t launch_plan(const PlanLaunch& p, cudaStream_t s, LaunchHook& hook) {
  const int nchunks = (p.T + kChunk - 1) / kChunk;
  const int nblocks = (p.T + kTopkTokens - 1) / kTopkTokens;
  const int nv = (p.E + 31) / 32;
  // The chunk counts and the scan's ticket start at zero (the bitmap words are
  // all written by the top-k CTAs).
  cudaError_t err = cudaMemsetAsync(p.ticket, 0, (16 + static_cast<size_t>(nchunks) * p.E) * 4, s);
  if (err != cudaSuccess) return err;
  const size_t topk_smem = static_cast<size_t>(p.E) * 3 * 4;
  hook.before(s);
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
  hook.after(s);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  hook.before(s);
  route_scan_kernel<<<(p.E + kScanWarps - 1) / kScanWarps, 32 * kScanWarps, 0, s>>>(
      p.ccount, nchunks, p.E, p.cbase, p.counts, p.offsets, p.tiles, p.ticket);
  hook.after(s);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  hook.before(s);
  route_rank_kernel<<<nblocks, 256, static_cast<size_t>(p.E) * 4 * 4, s>>>(
      p.ids, p.gbm, p.cbase, p.offsets, p.T, p.E, p.k, p.T * p.k, p.dest, p.row_src, p.row_slot, p.ws);
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
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and passed to the kernels like any workspace pointer.
// ---------------------------------------------------------------------------
#include <mutex>

namespace moe {
namespace {

constexpr size_t kNoAllocBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

size_t na_align(size_t v) { return (v + 255) & ~size_t(255); }

// Device address of g_noalloc_scratch on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_LAUNCH;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_LAUNCH;
    if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_LAUNCH;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

bool na_ok_ptr(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_plan_noalloc(moe_dims d, const float* logits, const moe_plan_t* plan, int32_t* status,
                                void* stream) {
  using namespace moe;
  if (d.T < 0 || d.H <= 0 || d.F <= 0 || d.E <= 0 || d.k <= 0 || d.k > d.E || d.k > 32 ||
      static_cast<long long>(d.T) * d.k >= (1ll << 31))
    return MOE_ERR_ARG;
  if (d.H % 128 != 0 || d.F % 128 != 0 || d.E > 1024) return MOE_ERR_SHAPE;
  const size_t nchunks = (static_cast<size_t>(d.T) + kChunk - 1) / kChunk;
  const size_t ccount = 0;  // 16-word ticket, then the per-chunk counts
  const size_t cbase = na_align(ccount + (16 + nchunks * d.E) * 4);
  const size_t gbm = na_align(cbase + nchunks * d.E * 4);
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
  p.ids = plan->topk_ids;
  p.w = plan->topk_w;
  p.ticket = reinterpret_cast<int32_t*>(w + ccount);
  p.ccount = p.ticket + 16;
  p.cbase = reinterpret_cast<int32_t*>(w + cbase);
  p.gbm = reinterpret_cast<uint32_t*>(w + gbm);
  p.counts = plan->counts;
  p.offsets = plan->offsets;
  p.tiles = plan->tiles;
  p.dest = plan->dest;
  p.row_src = plan->row_src;
  p.row_slot = plan->row_slot;
  p.ws = reinterpret_cast<WsHeader*>(status);  // only status/where/detail are written
  LaunchHook hook;
  return launch_plan(p, static_cast<cudaStream_t>(stream), hook) == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
