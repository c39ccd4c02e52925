// Declarations shared between the kernel files and the C ABI (host side).
#pragma once

#include <atomic>

#include "common.cuh"

namespace moe {

constexpr int kChunk = 256;               // tokens per routing chunk (one "source" of the mapping)
constexpr int kChunkWords = kChunk / 32;  // bitmap words per expert and chunk
constexpr int kSuperChunks = 32;          // chunks per super-chunk (8192 tokens): the coarse level of the chunk prefix

// Words of the routing's count area: a 16-word header, the per-chunk counts
// [E][nchunks] and the per-super-chunk counts [E][nsuper], both expert-major.
__host__ __device__ inline long long plan_count_words(long long T, int E) {
  const long long nchunks = (T + kChunk - 1) / kChunk;
  const long long nsuper = (nchunks + kSuperChunks - 1) / kSuperChunks;
  return 16 + (nchunks + nsuper) * E;
}
constexpr int kTileRows = 128;            // rows of a GEMM tile (the tcgen05 M)
constexpr int kMaxPad = 4096;             // largest padding granule of an expert's rows

// Grouped rows the [R, ...] buffers hold.  Padding-free (pad 0 or 1): T*k.
// With a padding granule pad >= 2 every expert's rows are rounded up to a
// multiple of pad, which adds at most pad - 1 rows to each non-empty expert: a
// bound that does not depend on the routing (static shapes).
__host__ __device__ inline long long grouped_rows(long long T, int k, int E, int pad) {
  const long long R = T * k;
  return pad > 1 ? R + (R < E ? R : static_cast<long long>(E)) * (pad - 1) : R;
}

// Layout of moe_plan_t.tiles (int32): [0] number of 128-row tiles; [1 + e]
// first tile of expert e (E + 1 entries); then, from tiles_entry_base(E),
// one int4 {expert, first row, rows, 0} per tile in expert order; then, from
// tiles_pair_base(R, E), the first 256-row pair of each expert (E + 1 entries);
// then, from tiles_gcount_base(R, E), the rows the GEMMs run for each expert
// (E entries: n_e rounded up to the padding granule).  R = grouped_rows.
__host__ __device__ inline int tiles_entry_base(int E) { return ((E + 2) + 3) & ~3; }

__host__ __device__ inline long long tiles_capacity(long long R, int E) { return R / kTileRows + E + 1; }

// After the entries: E + 1 ints, the first 256-row pair tile of each expert
// (exclusive prefix of ceil(n_e / 256)), used by the two-SM GEMMs.
__host__ __device__ inline long long tiles_pair_base(long long R, int E) {
  return tiles_entry_base(E) + 4 * tiles_capacity(R, E);
}
__host__ __device__ inline long long tiles_gcount_base(long long R, int E) { return tiles_pair_base(R, E) + E + 1; }
__host__ __device__ inline long long tiles_elems(long long R, int E) { return tiles_gcount_base(R, E) + E; }

extern std::atomic<unsigned long long> g_launches;

// Records the caller's timing events around each kernel and counts launches.
struct LaunchHook {
  void** events = nullptr;
  int n_events = 0;
  int idx = 0;
  // Timing is optional: a null or unusable event is skipped, and a failed
  // record is cleared so it cannot be mistaken for a failed kernel launch.
  static void record(void* ev, cudaStream_t s) {
    if (ev != nullptr && cudaEventRecord(static_cast<cudaEvent_t>(ev), s) != cudaSuccess) (void)cudaGetLastError();
  }
  void before(cudaStream_t s) {
    if (events && idx < n_events) record(events[2 * idx], s);
  }
  void after(cudaStream_t s) {
    if (events && idx < n_events) record(events[2 * idx + 1], s);
    ++idx;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
};

struct PlanLaunch {
  const float* logits;
  int T, E, k;
  int pad;          // padding granule of each expert's rows (0 or 1: none)
  int R;            // grouped_rows(T, k, E, pad)
  int32_t* ids;
  float* w;
  uint32_t* gbm;
  int32_t* ticket;  // 16-word header, then ccount and the super-chunk counts; all cleared by launch_plan
  int32_t* ccount;  // [E][nchunks] (expert-major) = ticket + 16, then [E][nsuper] super-chunk counts
  int32_t* counts;
  int32_t* offsets;
  int32_t* tiles;
  int32_t* pairs;  // tiles + tiles_pair_base(R, E)
  int32_t* gcounts;  // tiles + tiles_gcount_base(R, E)
  int32_t* dest;
  int32_t* row_src;
  uint8_t* row_slot;
  WsHeader* ws;
};
cudaError_t launch_plan(const PlanLaunch& p, cudaStream_t s, LaunchHook& hook);

// Router buffers of the row kernels (all null when the router is not on the path).
struct RouterRows {
  const int32_t* ids;         // [T,k] chosen experts
  float* dl_slot;             // [T,k] dl of each chosen logit (combine_bwd writes, unpermute reads)
  float* dlogits;             // [T,E] fp32 out (combine_bwd)
  __nv_bfloat16* dl_bf16;     // [T,E] bf16 copy for the dWr GEMM (combine_bwd)
  const uint4* WrT;           // [E,H] bf16 rows of Wr^T (unpermute)
  int E;
};

struct RowsLaunch {
  int T, H, k, R;
  int grid;  // CTAs (256 threads each)
  const int32_t* dest;
  const int32_t* row_src;
  const float* w;
  WsHeader* ws;
  RouterRows rt;
  const int32_t* rows_used;  // device count of the grouped rows in use (the plan's offsets[E])
  int pad;                   // padding granule (>= 2: the padding rows of Xp and dY are written as zeros)
};
// Xp[r] = x[row_src[r]]
cudaError_t launch_gather(const RowsLaunch& p, const void* x, void* Xp, cudaStream_t s, LaunchHook& hook);
// out[t] = bf16(sum_j w[t,j] Y[dest[t,j]])
cudaError_t launch_combine(const RowsLaunch& p, const void* Y, void* out, cudaStream_t s, LaunchHook& hook);
// dY[dest[t,j]] = bf16(w[t,j] dout[t]); dgate[t,j] = <dout[t], Y[dest[t,j]]>
cudaError_t launch_combine_bwd(const RowsLaunch& p, const void* dout, const void* Y, void* dY, float* dgate,
                               cudaStream_t s, LaunchHook& hook);
// dx[t] = bf16(sum_j dXp[dest[t,j]] (+ sum_j dl[t,j] WrT[ids[t,j]] with the router))
cudaError_t launch_unpermute(const RowsLaunch& p, const void* dXp, void* dx, cudaStream_t s, LaunchHook& hook);
// WrT = Wr^T (bf16 [H,E] -> [E,H])
cudaError_t launch_transpose_wr(const void* Wr, void* WrT, int H, int E, cudaStream_t s, LaunchHook& hook);
// sb_rows[e] = rows of expert e whose token is below t_split (a prefix of its segment)
cudaError_t launch_subbatch_rows(const int32_t* offsets, const int32_t* counts, const int32_t* row_src, int E,
                                 int t_split, int32_t* sb_rows, cudaStream_t s, LaunchHook& hook);
// out[i] = sum_s part[s][i] over `splits` partial buffers of n floats (n % 4 == 0)
cudaError_t launch_reduce_splits(const float* part, float* out, size_t n, int splits, int grid, cudaStream_t s,
                                 LaunchHook& hook);

enum GemmMode : int {
  kFwd1 = 0,    // [G|U] = Xp [W1|W3], h = silu(G) U           (A K-major, B MN-major)
  kFwd2 = 1,    // Y = h W2                                    (A K-major, B MN-major)
  kDgrad2 = 2,  // dH = dY W2^T, SwiGLU backward -> dG, dU      (A K-major, B K-major)
  kDgrad1 = 3,  // dXp = [dG dU] [W1 W3]^T                      (A K-major, B K-major)
  kWgrad13 = 4, // dW1 = Xp^T dG, dW3 = Xp^T dU per expert      (A MN-major, B MN-major)
  kWgrad2 = 5,  // dW2 = h^T dY per expert                      (A MN-major, B MN-major)
  kRfwd = 6,    // router logits = x Wr (fp32 out)              (A K-major, B MN-major)
  kRwgrad = 7,  // router dWr partial = x^T dl over a token split (A MN-major, B MN-major)
};

// The gated combine fused into GEMM2's epilogue (kFwd2; cnt = null: not fused).
struct CombineLaunch {
  int32_t* cnt;            // [T][ceil(H/256)][2], zeroed before the launch
  const int32_t* row_src;
  const int32_t* dest;
  const float* w;
  void* out;               // [T,H] bf16
  int k;
};

struct GemmLaunch {
  int T, H, F, E, k, R;
  int grid;
  int pair;  // 1: two-SM pair tiles (cta_group::2), 0: one CTA per 128-row tile
  const int32_t* tiles;
  const int32_t* pairs;  // first 256-row pair of each expert (tiles + tiles_pair_base)
  const int32_t* offsets;
  const int32_t* counts;
  // operands (bf16)
  const void* Xp;
  const void* W1;
  const void* W3;
  const void* W2;
  const void* h;
  const void* GU;
  const void* dY;
  const void* dGU;
  // outputs
  void* out_h;    // kFwd1
  void* out_GU;   // kFwd1
  void* out_Y;    // kFwd2
  void* out_dGU;  // kDgrad2
  void* out_dXp;  // kDgrad1
  float* dW1;     // kWgrad13
  float* dW3;     // kWgrad13
  float* dW2;     // kWgrad2
  // router
  const void* x;       // [T,H] bf16
  const void* Wr;      // [H,E] bf16
  const void* dl;      // [T,E] bf16 router logit gradient (kRwgrad B operand)
  float* logits;       // kRfwd out [T,E]
  float* dwr_part;     // kRwgrad out [splits][H][E] (or dWr itself when splits = 1)
  int splits, ks;      // token splits of kRwgrad and tokens per split (a multiple of 64)
  CombineLaunch cmb;   // kFwd2
  int drop_task;       // fused forward: failure injection (task + 1 whose gather signal is withheld; 0 none)
  int gather;              // kFwd1 on pair tiles: A rows gathered from x by row_src, Xp stored from the stages
  const int32_t* row_src;  // [R] (gather)
  int sb;                  // weight gradients: 0 one chain; 1 / 2 token sub-batch 0 (stored) / 1 (added)
  const int32_t* sb_rows;  // [E] rows of each expert that belong to token sub-batch 0
  WsHeader* ws;
};
cudaError_t launch_gemm(GemmMode mode, const GemmLaunch& p, cudaStream_t s, LaunchHook& hook);

// The forward's gather, GEMM1 and GEMM2 as one persistent kernel (task cursor
// and per-tile counters must be zero at launch).
cudaError_t launch_fused_forward(const GemmLaunch& L, const void* x, const int32_t* row_src, int32_t* cursor,
                                 int32_t* cnt_gather, int32_t* cnt_g1, cudaStream_t s, LaunchHook& hook);

// The same on two-SM pair tiles (clusters of two CTAs; counters per 128-row tile).
cudaError_t launch_fused_forward_pair(const GemmLaunch& L, const void* x, const int32_t* row_src, int32_t* cursor,
                                      int32_t* cnt_gather, int32_t* cnt_g1, cudaStream_t s, LaunchHook& hook);

// dgrad2, dgrad1 and both weight-gradient GEMMs as one persistent kernel
// (task cursor and per-tile counters must be zero at launch).
cudaError_t launch_fused_backward(const GemmLaunch& L, int32_t* cursor, int32_t* cnt_d2, int32_t* cnt_e,
                                  cudaStream_t s, LaunchHook& hook);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
bool tensor_map_encoder_ready();

}  // namespace moe
