// Row-wise, HBM-bound steps of the layer: dispatch (a gather by grouped row,
// or a scatter of each token's row to its k grouped rows when x is large),
// gated combine, combine backward, dispatch backward.  One warp per row or
// token (the combine and the dispatch backward split a token's row over several
// warps when a batch has fewer tokens than warps), 16-byte vector loads and
// stores, grid-stride.
//
// Sources: "UniEP: Unified Expert-Parallel MoE MegaKernel for LLM Training",
// section 3.1 (Comm-Worker: one warp per token, 128-bit vector loads) and
// section 5 (Relay & Reduce Workers: one warp aggregates one token's top-k
// replicas with vector loads and stores, no shared memory); the reduction
// waits for all k contributions and sums them in a fixed order (section 3,
// Top-k accumulation constraint).  "MoonEP: Balanced Expert Parallelism for
// MoE Training via Dynamic Redundant Experts": zero-copy dispatch, and the
// gradient of dispatch is a combine of each token's k row gradients.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxK = 32;

__device__ __forceinline__ uint4 ldg_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  return v;
}

// Grouped rows in use: the plan's offsets[E] (R itself without padding).
__device__ __forceinline__ int rows_in_use(const int32_t* rows_used, int R, WsHeader* ws, int where) {
  const int n = __ldg(rows_used);
  if (n < 0 || n > R) {
    if ((threadIdx.x & 31) == 0) report(ws, MOE_ERR_BOUNDS, where, n);
    return 0;
  }
  return n;
}

// The padding rows (row_src = -1) of a grouped buffer are written as zeros.  A
// warp tests 32 rows at a time and clears the padding rows among them.
__device__ __forceinline__ void zero_padding_rows(const int32_t* __restrict__ row_src, int n, uint4* __restrict__ buf,
                                                  int hv, int gwarp, int nwarps, int lane) {
  for (int r0 = gwarp * 32; r0 < n; r0 += nwarps * 32) {
    const int r = r0 + lane;
    unsigned m = __ballot_sync(0xffffffffu, r < n && row_src[r] == -1);
    while (m != 0u) {
      const int b = __ffs(m) - 1;
      m &= m - 1u;
      uint4* dst = buf + static_cast<size_t>(r0 + b) * hv;
      for (int v = lane; v < hv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// The gated combine, with fewer tokens than warps (short batches), gives each
// token to `parts` warps, each over a contiguous range of the row's 16-byte
// columns, so that more rows are in flight; every output element is still
// summed by one lane in slot order, so the bits do not change (fine-grained:
// 23.9 -> 19.9 us).
__device__ __forceinline__ int token_parts(int T, int nwarps) {
  return (T > 0 && nwarps >= 2 * T) ? min(4, nwarps / T) : 1;
}
__device__ __forceinline__ int part_span(int hv, int parts) { return ((hv + parts - 1) / parts + 31) / 32 * 32; }

// The dispatch backward launches one wave of CTAs (below); with fewer tokens
// than warps it splits each token over enough warps that every warp has rows in
// flight (fine-grained: 4096 tokens on 4864 warps, two parts per token).  Split
// on a grid of eight CTAs per SM, at 128 registers, it had measured slower.
__device__ __forceinline__ int unpermute_parts(int T, int nwarps) {
  return T > 0 ? max(1, min(8, (nwarps + T - 1) / T)) : 1;
}

// Dispatch as a gather, one warp per grouped row: Xp[r] = x[row_src[r]], zeros
// for a padding row.  Used while x fits comfortably in L2 (its re-reads are L2
// hits), where the R rows give more parallelism than the T tokens.
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const uint4* __restrict__ x,
                                                                 const int32_t* __restrict__ row_src,
                                                                 const int32_t* __restrict__ rows_used,
                                                                 uint4* __restrict__ Xp, int R, int T, int hv,
                                                                 WsHeader* ws) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (kThreads / 32);
  const int n = rows_in_use(rows_used, R, ws, 10);
  for (int r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < n; r += nwarps) {
    const int t = row_src[r];
    if (t == -1) {
      uint4* dst = Xp + static_cast<size_t>(r) * hv;
      for (int v = lane; v < hv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    if (t < 0 || t >= T) {
      if (lane == 0) report(ws, MOE_ERR_BOUNDS, 10, r);
      continue;
    }
    const uint4* src = x + static_cast<size_t>(t) * hv;
    uint4* dst = Xp + static_cast<size_t>(r) * hv;
    // Eight 16-byte vectors per lane in flight (a whole 4 KB row at H = 2048).
    int v = lane;
    for (; v + 224 < hv; v += 256) {
      uint4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ldg_nc(src + v + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[v + 32 * u] = a[u];
    }
    for (; v + 96 < hv; v += 128) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = ldg_nc(src + v + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[v + 32 * u] = a[u];
    }
    for (; v < hv; v += 32) dst[v] = ldg_nc(src + v);
  }
}

// Dispatch as a scatter, one warp per token: x[t] is read once and written to
// its k grouped rows Xp[dest[t, j]] (the Comm-Worker of "UniEP", section 3.1:
// one warp per token, 128-bit vector loads; "MoonEP": zero-copy dispatch into
// the expert-grouped layout).  Reading each token once keeps the HBM traffic at
// 2TH + 2RH even when x does not fit in L2, which a gather over the grouped
// rows (x re-read once per slot) would not.
template <int K>
__global__ void __launch_bounds__(kThreads) scatter_rows_kernel(const uint4* __restrict__ x,
                                                                  const int32_t* __restrict__ dest,
                                                                  uint4* __restrict__ Xp, int T, int k, int R,
                                                                  int hv, WsHeader* ws, const int32_t* row_src,
                                                                  const int32_t* rows_used);

// The k (row, weight) pairs of token t, held in registers by every lane
// (K = compile-time bound on k).  Returns false (and reports) if a row index is
// out of range.
template <int K>
__device__ __forceinline__ bool token_rows(const int32_t* dest, const float* w, int t, int k, int R, int lane,
                                           int (&rows)[K], float (&ws_)[K], WsHeader* ws, int where) {
  int my_r = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_r = dest[static_cast<size_t>(t) * k + lane];
    if (w != nullptr) my_w = w[static_cast<size_t>(t) * k + lane];
  }
  const bool bad = lane < k && (my_r < 0 || my_r >= R);
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) report(ws, MOE_ERR_BOUNDS, where, t);
    return false;
  }
#pragma unroll
  for (int j = 0; j < K; ++j) {
    rows[j] = __shfl_sync(0xffffffffu, my_r, j);
    ws_[j] = __shfl_sync(0xffffffffu, my_w, j);
  }
  return true;
}

// With padding (rows_used != nullptr) the padding rows are cleared after the tokens.
template <int K>
__global__ void __launch_bounds__(kThreads) scatter_rows_kernel(const uint4* __restrict__ x,
                                                                  const int32_t* __restrict__ dest,
                                                                  uint4* __restrict__ Xp, int T, int k, int R,
                                                                  int hv, WsHeader* ws, const int32_t* row_src,
                                                                  const int32_t* rows_used) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (kThreads / 32);
  for (int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < T; t += nwarps) {
    int rows[K];
    float unused[K];
    if (!token_rows<K>(dest, nullptr, t, k, R, lane, rows, unused, ws, 10)) continue;
    const uint4* src = x + static_cast<size_t>(t) * hv;
    int v = lane;
    for (; v + 96 < hv; v += 128) {
      const uint4 a = ldg_nc(src + v), b = ldg_nc(src + v + 32), c = ldg_nc(src + v + 64),
                  d = ldg_nc(src + v + 96);
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j < k) {
          uint4* dst = Xp + static_cast<size_t>(rows[j]) * hv;
          dst[v] = a;
          dst[v + 32] = b;
          dst[v + 64] = c;
          dst[v + 96] = d;
        }
      }
    }
    for (; v < hv; v += 32) {
      const uint4 a = ldg_nc(src + v);
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (j < k) Xp[static_cast<size_t>(rows[j]) * hv + v] = a;
    }
  }
  if (rows_used != nullptr)
    zero_padding_rows(row_src, rows_in_use(rows_used, R, ws, 10), Xp, hv,
                      blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5), nwarps, lane);
}

// out[t] = bf16(sum_j w[t,j] Y[dest[t,j]]), slots in ascending order.
template <int K>
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint4* __restrict__ Y,
                                                             const int32_t* __restrict__ dest,
                                                             const float* __restrict__ w, uint4* __restrict__ out,
                                                             int T, int k, int R, int hv, WsHeader* ws) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (kThreads / 32);
  const int parts = token_parts(T, nwarps), span = part_span(hv, parts);
  for (int tw = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); tw < T * parts; tw += nwarps) {
    const int t = tw / parts, v0 = (tw - t * parts) * span, v1 = min(hv, v0 + span);
    int rows[K];
    float wj[K];
    if (!token_rows<K>(dest, w, t, k, R, lane, rows, wj, ws, 11)) continue;
    for (int v = v0 + lane; v < v1; v += 32) {
      uint4 y[K];
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (j < k) y[j] = ldg_nc(Y + static_cast<size_t>(rows[j]) * hv + v);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j < k) {
          float f[8];
          unpack8(y[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[j], f[i], acc[i]);
        }
      }
      out[static_cast<size_t>(t) * hv + v] = pack8(acc);
    }
  }
}

// dY[dest[t,j]] = bf16(w[t,j] dout[t]); dgate[t,j] = <dout[t], Y[dest[t,j]]>.
// Each lane accumulates its columns in order; the lanes' partial sums are then
// combined by a fixed butterfly, so the result does not depend on the grid.
template <int K>
__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(const uint4* __restrict__ dout,
                                                                 const uint4* __restrict__ Y,
                                                                 const int32_t* __restrict__ dest,
                                                                 const float* __restrict__ w,
                                                                 uint4* __restrict__ dY, float* __restrict__ dgate,
                                                                 int T, int k, int R, int hv, WsHeader* ws,
                                                                 RouterRows rt, const int32_t* row_src,
                                                                 const int32_t* rows_used) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (kThreads / 32);
  for (int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < T; t += nwarps) {
    int rows[K];
    float wj[K];
    if (!token_rows<K>(dest, w, t, k, R, lane, rows, wj, ws, 12)) continue;
    float part[K];
#pragma unroll
    for (int j = 0; j < K; ++j) part[j] = 0.f;
    for (int v = lane; v < hv; v += 32) {
      float d[8];
      unpack8(ldg_nc(dout + static_cast<size_t>(t) * hv + v), d);
      uint4 y[K];
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (j < k) y[j] = ldg_nc(Y + static_cast<size_t>(rows[j]) * hv + v);
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j < k) {
          float f[8], g[8];
          unpack8(y[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            part[j] = fmaf(d[i], f[i], part[j]);
            g[i] = wj[j] * d[i];
          }
          dY[static_cast<size_t>(rows[j]) * hv + v] = pack8(g);
        }
      }
    }
    float dg[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      float s = part[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      dg[j] = s;
      if (j < k && lane == 0) dgate[static_cast<size_t>(t) * k + j] = s;
    }
    if (rt.dlogits != nullptr) {
      // Gradient through the renormalised top-k softmax (routing fixed):
      // dl_j = w_j (dgate_j - sum_i w_i dgate_i), slots in ascending order;
      // the logits of the other experts get 0.
      float sw = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (j < k) sw = fmaf(wj[j], dg[j], sw);
      int ej[K];
      float dl[K];
      const int my_e = (lane < k) ? rt.ids[static_cast<size_t>(t) * k + lane] : -1;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        ej[j] = __shfl_sync(0xffffffffu, my_e, j);
        dl[j] = wj[j] * (dg[j] - sw);
        if (j < k && lane == 0) rt.dl_slot[static_cast<size_t>(t) * k + j] = dl[j];
      }
      float* drow = rt.dlogits + static_cast<size_t>(t) * rt.E;
      __nv_bfloat16* brow = rt.dl_bf16 + static_cast<size_t>(t) * rt.E;
      for (int e = lane; e < rt.E; e += 32) {
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (j < k && ej[j] == e) v = dl[j];
        drow[e] = v;
        brow[e] = __float2bfloat16_rn(v);
      }
    }
  }
  if (rows_used != nullptr)  // padding rows of dY: zero, so the GEMMs that read them add nothing
    zero_padding_rows(row_src, rows_in_use(rows_used, R, ws, 12), dY, hv,
                      blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5), nwarps, lane);
}

// dx[t] = bf16(sum_j dXp[dest[t,j]]), slots in ascending order.
// With the router on the path, dx[t] also gains the router's share
// sum_j dl[t,j] Wr[:, ids[t,j]] (only the k chosen logits have a gradient), read
// from rows of Wr^T; both shares are summed in fp32 and rounded once.
// The plain kernel (no router share, k <= 8) is held to 64 registers: four
// CTAs per SM instead of two, which measured 18% faster on a 4096-token batch.
template <int K, bool ROUTER>
__global__ void __launch_bounds__(kThreads, (K <= 8 && !ROUTER) ? 4 : 1) unpermute_kernel(
    const uint4* __restrict__ dXp, const int32_t* __restrict__ dest, uint4* __restrict__ dx, int T, int k, int R,
    int hv, WsHeader* ws, RouterRows rt) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (kThreads / 32);
  constexpr bool router = ROUTER;
  const int parts = unpermute_parts(T, nwarps), span = part_span(hv, parts);
  for (int tw = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); tw < T * parts; tw += nwarps) {
    const int t = tw / parts, v0 = (tw - t * parts) * span, v1 = min(hv, v0 + span);
    int rows[K];
    float wj[K];
    if (!token_rows<K>(dest, nullptr, t, k, R, lane, rows, wj, ws, 13)) continue;
    int ej[K];
    float dl[K];
    if (router) {
      const int my_e = (lane < k) ? rt.ids[static_cast<size_t>(t) * k + lane] : 0;
      const float my_d = (lane < k) ? rt.dl_slot[static_cast<size_t>(t) * k + lane] : 0.f;
      const bool bad = lane < k && (my_e < 0 || my_e >= rt.E);
      if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) report(ws, MOE_ERR_BOUNDS, 14, t);
        continue;
      }
#pragma unroll
      for (int j = 0; j < K; ++j) {
        ej[j] = __shfl_sync(0xffffffffu, my_e, j);
        dl[j] = __shfl_sync(0xffffffffu, my_d, j);
      }
    }
    for (int v = v0 + lane; v < v1; v += 32) {
      uint4 y[K];
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (j < k) y[j] = ldg_nc(dXp + static_cast<size_t>(rows[j]) * hv + v);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j < k) {
          float f[8];
          unpack8(y[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
      }
      if (router) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (j < k) {
            float f[8];
            unpack8(ldg_nc(rt.WrT + static_cast<size_t>(ej[j]) * hv + v), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(dl[j], f[i], acc[i]);
          }
        }
      }
      dx[static_cast<size_t>(t) * hv + v] = pack8(acc);
    }
  }
}

// WrT[e, h] = Wr[h, e] (bf16), through 32 x 32 tiles in shared memory.
__global__ void __launch_bounds__(256) transpose_wr_kernel(const __nv_bfloat16* __restrict__ Wr,
                                                             __nv_bfloat16* __restrict__ WrT, int H, int E) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int h = h0 + r, e = e0 + tx;
    if (h < H && e < E) tile[r][tx] = Wr[static_cast<size_t>(h) * E + e];
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, h = h0 + tx;
    if (h < H && e < E) WrT[static_cast<size_t>(e) * H + h] = tile[tx][r];
  }
}

// dWr[i] = sum_s part[s][i], s ascending (a fixed order: the same bits for any grid).
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float4* __restrict__ part, float4* __restrict__ out,
                                                              size_t n4, int splits) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int sp = 1; sp < splits; ++sp) {
      const float4 b = part[static_cast<size_t>(sp) * n4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    out[i] = a;
  }
}

// Rows of each expert that belong to token sub-batch 0 (tokens below t_split):
// an expert's rows are in token order, so this is the length of the prefix of
// its segment with row_src < t_split.  One warp per expert, 32-way search: the
// lanes probe 32 evenly spaced rows of the remaining interval [lo, hi] and the
// ballot narrows it to one gap between probes.
__global__ void __launch_bounds__(256) subbatch_rows_kernel(const int32_t* __restrict__ offsets,
                                                              const int32_t* __restrict__ counts,
                                                              const int32_t* __restrict__ row_src, int E, int t_split,
                                                              int32_t* __restrict__ sb_rows) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (e >= E) return;
  const int32_t* seg = row_src + offsets[e];
  int lo = 0, hi = counts[e];  // the answer m lies in [lo, hi]: rows below m are in sub-batch 0
  while (lo < hi) {
    const long long span = hi - lo;
    const int i = lo + static_cast<int>(((lane + 1) * span - 1) / 32);  // in [lo, hi - 1], ascending in lane
    const unsigned below = __ballot_sync(0xffffffffu, seg[i] < t_split);
    const int c = __popc(below);  // probes 0 .. c-1 are in sub-batch 0
    const int i0 = __shfl_sync(0xffffffffu, i, 0);
    const int ilast = __shfl_sync(0xffffffffu, i, c > 0 ? c - 1 : 0);
    const int inext = __shfl_sync(0xffffffffu, i, c < 32 ? c : 31);
    if (c == 0) {
      hi = i0;
    } else {
      lo = ilast + 1;
      if (c < 32) hi = inext;
    }
  }
  if (lane == 0) sb_rows[e] = lo;
}

// CTAs of a launch that all fit on the GPU at once: `per_sm` resident CTAs of
// the kernel (its occupancy, queried once) for each SM slot of the grid
// (p.grid counts eight CTAs per SM).  The kernel's token loop strides over its
// work, so no CTA waits for a slot while the first ones drain.
template <auto Kernel>
int one_wave(int grid) {
  static const int per_sm = [] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, kThreads, 0) == cudaSuccess && n > 0 ? n : 8;
  }();
  return max(1, min(grid, per_sm * max(1, grid / 8)));
}

}  // namespace

cudaError_t launch_subbatch_rows(const int32_t* offsets, const int32_t* counts, const int32_t* row_src, int E,
                                 int t_split, int32_t* sb_rows, cudaStream_t s, LaunchHook& hook) {
  hook.before(s);
  subbatch_rows_kernel<<<(E + 7) / 8, 256, 0, s>>>(offsets, counts, row_src, E, t_split, sb_rows);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_gather(const RowsLaunch& p, const void* x, void* Xp, cudaStream_t s, LaunchHook& hook) {
  hook.before(s);
  // x up to 32 MB: gather by grouped row (re-reads hit L2); larger: scatter by token.
  if (static_cast<size_t>(p.T) * p.H * 2 <= (size_t(32) << 20))
    gather_rows_kernel<<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(x), p.row_src, p.rows_used,
                                                    static_cast<uint4*>(Xp), p.R, p.T, p.H / 8, p.ws);
  else if (p.k <= 8)
    scatter_rows_kernel<8><<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(x), p.dest,
                                                        static_cast<uint4*>(Xp), p.T, p.k, p.R, p.H / 8, p.ws,
                                                        p.row_src, p.pad > 1 ? p.rows_used : nullptr);
  else
    scatter_rows_kernel<kMaxK><<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(x), p.dest,
                                                            static_cast<uint4*>(Xp), p.T, p.k, p.R, p.H / 8, p.ws,
                                                            p.row_src, p.pad > 1 ? p.rows_used : nullptr);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_combine(const RowsLaunch& p, const void* Y, void* out, cudaStream_t s, LaunchHook& hook) {
  hook.before(s);
  if (p.k <= 8)
    combine_kernel<8><<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(Y), p.dest, p.w,
                                                   static_cast<uint4*>(out), p.T, p.k, p.R, p.H / 8, p.ws);
  else
    combine_kernel<kMaxK><<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(Y), p.dest, p.w,
                                                       static_cast<uint4*>(out), p.T, p.k, p.R, p.H / 8, p.ws);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const RowsLaunch& p, const void* dout, const void* Y, void* dY, float* dgate,
                               cudaStream_t s, LaunchHook& hook) {
  hook.before(s);
  if (p.k <= 8)
    combine_bwd_kernel<8><<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(dout), static_cast<const uint4*>(Y),
                                                       p.dest, p.w, static_cast<uint4*>(dY), dgate, p.T, p.k, p.R,
                                                       p.H / 8, p.ws, p.rt, p.row_src, p.pad > 1 ? p.rows_used : nullptr);
  else
    combine_bwd_kernel<kMaxK><<<p.grid, kThreads, 0, s>>>(static_cast<const uint4*>(dout),
                                                           static_cast<const uint4*>(Y), p.dest, p.w,
                                                           static_cast<uint4*>(dY), dgate, p.T, p.k, p.R, p.H / 8,
                                                           p.ws, p.rt, p.row_src, p.pad > 1 ? p.rows_used : nullptr);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const RowsLaunch& p, const void* dXp, void* dx, cudaStream_t s, LaunchHook& hook) {
  hook.before(s);
  // The router's share of dx is a separate instantiation, so the plain kernel
  // holds fewer registers.
  const uint4* src = static_cast<const uint4*>(dXp);
  uint4* dst = static_cast<uint4*>(dx);
  const bool router = p.rt.WrT != nullptr;
#define MOE_UNPERMUTE(KK, RR)                                                                                 \
  unpermute_kernel<KK, RR><<<one_wave<unpermute_kernel<KK, RR>>(p.grid), kThreads, 0, s>>>(src, p.dest, dst, \
                                                                                          p.T, p.k, p.R, p.H / 8, \
                                                                                          p.ws, p.rt)
  if (p.k <= 8 && router)
    MOE_UNPERMUTE(8, true);
  else if (p.k <= 8)
    MOE_UNPERMUTE(8, false);
  else if (router)
    MOE_UNPERMUTE(kMaxK, true);
  else
    MOE_UNPERMUTE(kMaxK, false);
#undef MOE_UNPERMUTE
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_transpose_wr(const void* Wr, void* WrT, int H, int E, cudaStream_t s, LaunchHook& hook) {
  hook.before(s);
  transpose_wr_kernel<<<dim3((H + 31) / 32, (E + 31) / 32), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(Wr), static_cast<__nv_bfloat16*>(WrT), H, E);
  hook.after(s);
  return cudaGetLastError();
}

cudaError_t launch_reduce_splits(const float* part, float* out, size_t n, int splits, int grid, cudaStream_t s,
                                 LaunchHook& hook) {
  hook.before(s);
  reduce_splits_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(part), reinterpret_cast<float4*>(out),
                                            n / 4, splits);
  hook.after(s);
  return cudaGetLastError();
}

}  // namespace moe
