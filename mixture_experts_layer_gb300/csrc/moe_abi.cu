// Host side of the C ABI declared in include/moe.h: argument checks, workspace
// layout, and the launch sequence of each call.  No memory is allocated here.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

std::atomic<unsigned long long> g_launches{0};

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  int ok = -1;  // -1 unknown, 0 not sm_103, 1 ok
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_LAUNCH;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.ok < 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_LAUNCH;
    d.sms = n;
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
  }
  if (!d.ok) return MOE_ERR_DEVICE;
  *sms = d.sms;
  return MOE_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Grouped rows of the [R, ...] buffers (padding rows included).
long long rows_of(const moe_dims& d) { return grouped_rows(d.T, d.k, d.E, d.pad); }

int check_dims(const moe_dims& d) {
  if (d.T < 0 || d.H <= 0 || d.F <= 0 || d.E <= 0 || d.k <= 0) return MOE_ERR_ARG;
  if (d.k > d.E || d.k > 32) return MOE_ERR_ARG;
  if (d.pad < 0 || d.pad > kMaxPad) return MOE_ERR_ARG;
  if (rows_of(d) >= (1ll << 31)) return MOE_ERR_ARG;
  if (d.H % 128 != 0 || d.F % 128 != 0 || d.E > 1024) return MOE_ERR_SHAPE;
  if (static_cast<long long>(d.E) * d.H >= (1ll << 31) || static_cast<long long>(d.E) * d.F >= (1ll << 31))
    return MOE_ERR_SHAPE;
  return MOE_OK;
}

struct WsLayout {
  size_t ccount, gbm, sched, sched_bytes, total;
  size_t cap;  // capacity of the 128-row tile table
  size_t wrT, dl_slot, dl_bf16, dwr_part;  // router backward
  size_t cmb_cnt, cmb_bytes;               // arrivals of the combine fused into GEMM2
  size_t sb_rows;                          // [E] rows of each expert in token sub-batch 0
  int splits, ks;                          // token splits of the dWr GEMM and tokens per split
};

// Token splits of the router's weight-gradient GEMM (K = the tokens): enough
// tiles for ~2 per SM, a function of the dims alone (so the reduction order,
// and the bits, do not depend on the GPU or the grid).
void router_splits(const moe_dims& d, int* splits, int* ks) {
  const long long tiles = static_cast<long long>(d.H / 128) * ((d.E + 255) / 256);
  const long long nkb = (static_cast<long long>(d.T) + 63) / 64;
  long long sp = (304 + tiles - 1) / tiles;
  if (sp > nkb) sp = nkb;
  if (sp < 1) sp = 1;
  const long long kb_per = (nkb + sp - 1) / sp;
  *ks = static_cast<int>(kb_per * 64);
  *splits = static_cast<int>(d.T > 0 ? (d.T + *ks - 1) / *ks : 1);
}

WsLayout ws_layout(const moe_dims& d) {
  const size_t nchunks = (static_cast<size_t>(d.T) + kChunk - 1) / kChunk;
  WsLayout L;
  size_t off = align256(sizeof(WsHeader));
  L.ccount = off;  // 16-word header, then the per-chunk and per-super-chunk counts
  off = align256(off + static_cast<size_t>(plan_count_words(d.T, d.E)) * 4);
  L.gbm = off;
  off = align256(off + nchunks * d.E * kChunkWords * 4);
  // Scheduling words of the persistent kernels: a task cursor (padded to 64 B)
  // and two counters per 128-row tile.
  L.cap = static_cast<size_t>(tiles_capacity(rows_of(d), d.E));
  L.sched = off;
  L.sched_bytes = 64 + 2 * L.cap * 4;
  off = align256(off + L.sched_bytes);
  router_splits(d, &L.splits, &L.ks);
  L.wrT = off;
  off = align256(off + static_cast<size_t>(d.E) * d.H * 2);
  L.dl_slot = off;
  off = align256(off + static_cast<size_t>(d.T) * d.k * 4);
  L.dl_bf16 = off;
  off = align256(off + static_cast<size_t>(d.T) * d.E * 2);
  L.dwr_part = off;
  off = align256(off + static_cast<size_t>(L.splits) * d.H * d.E * 4);
  L.cmb_cnt = off;
  L.cmb_bytes = static_cast<size_t>(d.T) * ((d.H + 255) / 256) * 2 * 4;
  off = align256(off + L.cmb_bytes);
  L.sb_rows = off;
  off = align256(off + static_cast<size_t>(d.E) * 4);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ws(const moe_dims& d, void* ws, size_t ws_bytes) {
  if (!aligned16(ws)) return ws == nullptr ? MOE_ERR_ARG : MOE_ERR_ALIGN;
  if (ws_bytes < ws_layout(d).total) return MOE_ERR_WS;
  return MOE_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (p == nullptr) return MOE_ERR_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  }
  return MOE_OK;
}

int check_plan(const moe_plan_t* plan) {
  if (plan == nullptr) return MOE_ERR_ARG;
  int rc = check_ptrs({plan->topk_ids, plan->topk_w, plan->counts, plan->offsets, plan->dest, plan->row_src,
                       plan->tiles});
  if (rc) return rc;
  return plan->row_slot == nullptr ? MOE_ERR_ARG : MOE_OK;
}

LaunchHook make_hook(const moe_opts* o) {
  LaunchHook h;
  if (o != nullptr && o->events != nullptr && o->n_events > 0) {
    h.events = o->events;
    h.n_events = o->n_events;
  }
  return h;
}

int grid_for(const moe_opts* o, int sms) {
  if (o != nullptr && o->grid > 0) return o->grid < sms ? o->grid : sms;
  return sms;
}

int finish(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

// Whether the phased forward runs the dispatch inside GEMM1's A-operand load
// (moe_opts.dispatch = 2; pair tiles, padding-free layout) instead of as its own
// kernel (1).  Default (0): its own kernel.
bool dispatch_in_gemm1(const moe_dims& d, const moe_opts* o, int pair) {
  const int mode = o != nullptr ? o->dispatch : 0;
  return mode == 2 && pair && d.pad <= 1;
}

// CTAs of the weight-gradient GEMMs.  When the experts are short (at most 256
// rows on average) each tile is a few k-blocks followed by 256 KB of fp32 dW
// stores, and the kernels are bound by DRAM writes; fewer concurrent writers
// measured faster on GB300 (large-expert workload: dW1/dW3 5.06 ms on 128 CTAs
// against 6.05 ms on 152, dW2 2.67 against 3.02; the fine-grained workload, 384
// rows per expert, is fastest on every SM).  Every tile has one owner, so the
// grid does not change the bits.  An explicit moe_opts.grid is kept.
int wgrad_grid(const moe_dims& d, const moe_opts* o, int sms) {
  const int grid = grid_for(o, sms);
  if (o != nullptr && o->grid > 0) return grid;
  if (static_cast<long long>(d.T) * d.k > 256ll * d.E) return grid;
  const int capped = (sms * 27 / 32) & ~1;
  return capped >= 2 && capped < grid ? capped : grid;
}

// Tile shape of a grouped GEMM launched on its own: the two-CTA pair tile
// wherever it measured faster, unless the caller asks for one shape everywhere.
int use_pair(const moe_opts* o, GemmMode m, const moe_dims& d) {
  const int c = (o != nullptr) ? o->cta_pair : 0;
  if (c == 1) return 0;
  if (c == 2) return 1;
  // dgrad2 (SwiGLU backward epilogue) measured faster on single-CTA tiles unless the
  // experts are long (long-seq, 8192 rows each: 9.8 against 10.9 ms), where the pair
  // tiles' 256-row granularity wastes nothing.
  if (m == kDgrad2) return static_cast<long long>(d.T) * d.k >= 2048ll * d.E;
  return 1;
}


const char* const kPlanKernels[] = {"route_topk", "route_rank", nullptr};
const char* const kFwdKernelsFused[] = {"fused_forward", "combine", nullptr};
const char* const kFwdKernels[] = {"gather_rows", "gemm_fwd1_swiglu", "gemm_fwd2", "combine", nullptr};
const char* const kFwdKernelsCombineFused[] = {"gather_rows", "gemm_fwd1_swiglu", "gemm_fwd2_combine", nullptr};
const char* const kFwdKernelsGather[] = {"gemm_fwd1_gather_swiglu", "gemm_fwd2", "combine", nullptr};
const char* const kFwdKernelsGatherCombine[] = {"gemm_fwd1_gather_swiglu", "gemm_fwd2_combine", nullptr};
const char* const kBwdKernels[] = {"combine_bwd", "gemm_dgrad2_swiglu_bwd", "gemm_dgrad1", "unpermute",
                                   "gemm_wgrad13", "gemm_wgrad2", nullptr};
const char* const kBwdKernelsFused[] = {"combine_bwd", "fused_backward", "unpermute", nullptr};
const char* const kBwdKernelsRouter[] = {"router_transpose", "combine_bwd", "gemm_dgrad2_swiglu_bwd", "gemm_dgrad1",
                                         "gemm_router_wgrad", "router_reduce", "unpermute", "gemm_wgrad13",
                                         "gemm_wgrad2", nullptr};
const char* const kRouterFwdKernels[] = {"gemm_router_fwd", nullptr};
const char* const kBwdKernelsNB[] = {"combine_bwd",      "gemm_dgrad2_swiglu_bwd", "gemm_dgrad1",
                                     "unpermute",        "subbatch_rows",          "gemm_wgrad13_sb0",
                                     "gemm_wgrad2_sb0",  "gemm_wgrad13_sb1",       "gemm_wgrad2_sb1",
                                     nullptr};
const char* const kBwdKernelsRouterNB[] = {"router_transpose", "combine_bwd",      "gemm_dgrad2_swiglu_bwd",
                                           "gemm_dgrad1",      "gemm_router_wgrad", "router_reduce",
                                           "unpermute",        "subbatch_rows",    "gemm_wgrad13_sb0",
                                           "gemm_wgrad2_sb0",  "gemm_wgrad13_sb1", "gemm_wgrad2_sb1",
                                           nullptr};

GemmLaunch gemm_common(const moe_dims& d, const moe_plan_t* plan, WsHeader* ws, int grid) {
  GemmLaunch g{};
  g.T = d.T;
  g.H = d.H;
  g.F = d.F;
  g.E = d.E;
  g.k = d.k;
  g.R = static_cast<int>(rows_of(d));
  g.grid = grid;
  g.tiles = plan->tiles;
  g.pairs = plan->tiles + tiles_pair_base(rows_of(d), d.E);
  g.offsets = plan->offsets;
  g.counts = plan->tiles + tiles_gcount_base(rows_of(d), d.E);  // rows the GEMMs run (padded counts)
  g.ws = ws;
  return g;
}

// The router's weight gradient (when the router is on the path) and the
// dispatch backward dx[t] = sum_j dXp[dest[t,j]] (+ the router's share).
int router_wgrad_and_unpermute(const moe_dims& d, const moe_plan_t* plan, WsHeader* wsh, int grid, const WsLayout& WL,
                               uint8_t* wsb, const moe_router_t* router, RowsLaunch& r, const void* dXp, void* dx,
                               cudaStream_t s, LaunchHook& hook) {
  if (router != nullptr) {
    // dWr = x^T dl over a fixed number of token splits, reduced in split order.
    GemmLaunch rg = gemm_common(d, plan, wsh, grid);
    rg.x = router->x;
    rg.dl = wsb + WL.dl_bf16;
    rg.dwr_part = reinterpret_cast<float*>(wsb + WL.dwr_part);
    rg.splits = WL.splits;
    rg.ks = WL.ks;
    if (launch_gemm(kRwgrad, rg, s, hook) != cudaSuccess) return MOE_ERR_LAUNCH;
    if (launch_reduce_splits(rg.dwr_part, router->dWr, static_cast<size_t>(d.H) * d.E, WL.splits, grid * 4, s,
                             hook) != cudaSuccess)
      return MOE_ERR_LAUNCH;
    r.rt.WrT = reinterpret_cast<const uint4*>(wsb + WL.wrT);
  }
  return finish(launch_unpermute(r, dXp, dx, s, hook));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return ws_layout(d).total;
}

size_t moe_plan_tiles_elems(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return static_cast<size_t>(tiles_elems(rows_of(d), d.E));
}

size_t moe_rows(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return static_cast<size_t>(rows_of(d));
}

int moe_plan(moe_dims d, const float* logits, const moe_plan_t* plan, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (d.T == 0) return MOE_OK;
  if ((rc = check_plan(plan))) return rc;
  if ((rc = check_ptrs({logits}))) return rc;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  const WsLayout L = ws_layout(d);
  uint8_t* w = static_cast<uint8_t*>(ws);
  PlanLaunch p;
  p.logits = logits;
  p.T = d.T;
  p.E = d.E;
  p.k = d.k;
  p.pad = d.pad;
  p.R = static_cast<int>(rows_of(d));
  p.ids = plan->topk_ids;
  p.w = plan->topk_w;
  p.gbm = reinterpret_cast<uint32_t*>(w + L.gbm);
  p.ticket = reinterpret_cast<int32_t*>(w + L.ccount);
  p.ccount = p.ticket + 16;
  p.counts = plan->counts;
  p.offsets = plan->offsets;
  p.tiles = plan->tiles;
  p.pairs = plan->tiles + tiles_pair_base(rows_of(d), d.E);
  p.gcounts = plan->tiles + tiles_gcount_base(rows_of(d), d.E);
  p.dest = plan->dest;
  p.row_src = plan->row_src;
  p.row_slot = plan->row_slot;
  p.ws = reinterpret_cast<WsHeader*>(w);
  LaunchHook hook;
  return finish(launch_plan(p, static_cast<cudaStream_t>(stream), hook));
}

int moe_forward(moe_dims d, const void* x, const void* W1, const void* W3, const void* W2, const moe_plan_t* plan,
                const moe_saved_t* saved, void* out, void* ws, size_t ws_bytes, const moe_opts* opts,
                void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (opts != nullptr && (opts->schedule < 0 || opts->schedule > 2 || opts->grid < 0 || opts->cta_pair < 0 ||
                          opts->cta_pair > 2 || opts->combine < 0 || opts->combine > 1 || opts->debug_drop_task < 0 ||
                          opts->dispatch < 0 || opts->dispatch > 2))
    return MOE_ERR_ARG;
  if (d.T == 0) return MOE_OK;
  if ((rc = check_plan(plan))) return rc;
  if (saved == nullptr) return MOE_ERR_ARG;
  if ((rc = check_ptrs({x, W1, W3, W2, out, saved->Xp, saved->GU, saved->h, saved->Y}))) return rc;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  if (!tensor_map_encoder_ready()) return MOE_ERR_LAUNCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader* wsh = static_cast<WsHeader*>(ws);
  const int grid = grid_for(opts, sms);
  LaunchHook hook = make_hook(opts);

  RowsLaunch r{d.T, d.H, d.k, static_cast<int>(rows_of(d)), grid * 8, plan->dest, plan->row_src, plan->topk_w, wsh};
  r.rows_used = plan->offsets + d.E;
  r.pad = d.pad;
  GemmLaunch g = gemm_common(d, plan, wsh, grid);
  g.Xp = saved->Xp;
  g.W1 = W1;
  g.W3 = W3;
  g.W2 = W2;
  g.out_h = saved->h;
  g.out_GU = saved->GU;
  g.h = saved->h;
  g.out_Y = saved->Y;
  cudaError_t e;
  if (opts != nullptr && opts->schedule != 0) {
    const WsLayout L = ws_layout(d);
    uint8_t* sched = static_cast<uint8_t*>(ws) + L.sched;
    if (cudaMemsetAsync(sched, 0, L.sched_bytes, s) != cudaSuccess) return MOE_ERR_LAUNCH;
    int32_t* cursor = reinterpret_cast<int32_t*>(sched);
    int32_t* cnt_gather = reinterpret_cast<int32_t*>(sched + 64);
    int32_t* cnt_g1 = cnt_gather + L.cap;
    g.drop_task = (opts != nullptr && opts->debug_drop_task > 0) ? opts->debug_drop_task : 0;
    e = use_pair(opts, kFwd1, d) ? launch_fused_forward_pair(g, x, plan->row_src, cursor, cnt_gather, cnt_g1, s, hook)
                              : launch_fused_forward(g, x, plan->row_src, cursor, cnt_gather, cnt_g1, s, hook);
    if (e != cudaSuccess) return MOE_ERR_LAUNCH;
  } else {
    g.pair = use_pair(opts, kFwd1, d);
    if (dispatch_in_gemm1(d, opts, g.pair)) {  // GEMM1 gathers its A rows from x and stores Xp
      g.gather = 1;
      g.x = x;
      g.row_src = plan->row_src;
    } else {
      e = launch_gather(r, x, saved->Xp, s, hook);
      if (e != cudaSuccess) return MOE_ERR_LAUNCH;
    }
    if ((e = launch_gemm(kFwd1, g, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
    g.gather = 0;
    g.pair = use_pair(opts, kFwd2, d);
    const bool fuse = (opts != nullptr && opts->combine == 1);
    if (fuse) {
      const WsLayout L = ws_layout(d);
      int32_t* cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.cmb_cnt);
      if (cudaMemsetAsync(cnt, 0, L.cmb_bytes, s) != cudaSuccess) return MOE_ERR_LAUNCH;
      g.cmb = CombineLaunch{cnt, plan->row_src, plan->dest, plan->topk_w, out, d.k};
    }
    if ((e = launch_gemm(kFwd2, g, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
    if (fuse) return MOE_OK;
  }
  return finish(launch_combine(r, saved->Y, out, s, hook));
}

int moe_backward(moe_dims d, const void* dout, const void* W1, const void* W3, const void* W2,
                 const moe_plan_t* plan, const moe_saved_t* saved, const moe_grads_t* grads, void* dx, float* dW1,
                 float* dW3, float* dW2, float* dgate, void* ws, size_t ws_bytes, const moe_opts* opts,
                 void* stream, const moe_router_t* router) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (opts != nullptr && (opts->schedule < 0 || opts->schedule > 2 || opts->grid < 0 || opts->cta_pair < 0 ||
                          opts->cta_pair > 2 || opts->combine < 0 || opts->combine > 1 || opts->debug_drop_task < 0 ||
                          opts->wgrad_subbatches < 0 || opts->wgrad_subbatches > 2 ||
                          (opts->wgrad_subbatches == 2 && opts->schedule == 2)))
    return MOE_ERR_ARG;
  if ((rc = check_ptrs({dW1, dW3, dW2}))) return rc;
  if (router != nullptr) {
    if (d.E % 8 != 0) return MOE_ERR_SHAPE;
    if ((rc = check_ptrs({router->x, router->Wr, router->dlogits, router->dWr}))) return rc;
  }
  if (d.T > 0) {
    if ((rc = check_plan(plan))) return rc;
    if (saved == nullptr || grads == nullptr) return MOE_ERR_ARG;
    if ((rc = check_ptrs({dout, W1, W3, W2, dx, dgate, saved->Xp, saved->GU, saved->h, saved->Y, grads->dY,
                          grads->dGU, grads->dXp})))
      return rc;
  }
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d.T == 0) {
    // No rows: every weight gradient is zero.
    const size_t n = static_cast<size_t>(d.E) * d.H * d.F * sizeof(float);
    if (cudaMemsetAsync(dW1, 0, n, s) != cudaSuccess || cudaMemsetAsync(dW3, 0, n, s) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, n, s) != cudaSuccess)
      return MOE_ERR_LAUNCH;
    if (router != nullptr &&
        cudaMemsetAsync(router->dWr, 0, static_cast<size_t>(d.H) * d.E * sizeof(float), s) != cudaSuccess)
      return MOE_ERR_LAUNCH;
    return MOE_OK;
  }
  if (!tensor_map_encoder_ready()) return MOE_ERR_LAUNCH;
  WsHeader* wsh = static_cast<WsHeader*>(ws);
  const int grid = grid_for(opts, sms);
  LaunchHook hook = make_hook(opts);

  RowsLaunch r{d.T, d.H, d.k, static_cast<int>(rows_of(d)), grid * 8, plan->dest, plan->row_src, plan->topk_w, wsh,
               RouterRows{}};
  r.rows_used = plan->offsets + d.E;
  r.pad = d.pad;
  const WsLayout WL = ws_layout(d);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  cudaError_t e;
  if (router != nullptr) {
    r.rt.ids = plan->topk_ids;
    r.rt.dl_slot = reinterpret_cast<float*>(wsb + WL.dl_slot);
    r.rt.dlogits = router->dlogits;
    r.rt.dl_bf16 = reinterpret_cast<__nv_bfloat16*>(wsb + WL.dl_bf16);
    r.rt.E = d.E;
    if ((e = launch_transpose_wr(router->Wr, wsb + WL.wrT, d.H, d.E, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
  }
  e = launch_combine_bwd(r, dout, saved->Y, grads->dY, dgate, s, hook);
  if (e != cudaSuccess) return MOE_ERR_LAUNCH;

  GemmLaunch g = gemm_common(d, plan, wsh, grid);
  g.W1 = W1;
  g.W3 = W3;
  g.W2 = W2;
  g.Xp = saved->Xp;
  g.h = saved->h;
  g.GU = saved->GU;
  g.dY = grads->dY;
  g.dGU = grads->dGU;
  g.out_dGU = grads->dGU;
  g.out_dXp = grads->dXp;
  g.dW1 = dW1;
  g.dW3 = dW3;
  g.dW2 = dW2;
  if (opts != nullptr && opts->schedule == 2) {
    const WsLayout L = ws_layout(d);
    uint8_t* sched = static_cast<uint8_t*>(ws) + L.sched;
    if (cudaMemsetAsync(sched, 0, L.sched_bytes, s) != cudaSuccess) return MOE_ERR_LAUNCH;
    int32_t* cursor = reinterpret_cast<int32_t*>(sched);
    int32_t* cnt_d2 = reinterpret_cast<int32_t*>(sched + 64);
    int32_t* cnt_e = cnt_d2 + L.cap;
    if ((e = launch_fused_backward(g, cursor, cnt_d2, cnt_e, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
  } else {
    g.pair = use_pair(opts, kDgrad2, d);
    if ((e = launch_gemm(kDgrad2, g, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
    g.pair = use_pair(opts, kDgrad1, d);
    if ((e = launch_gemm(kDgrad1, g, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
    // The dispatch backward right after dgrad1, while dXp is still in L2; the
    // weight gradients, which read Xp / h / dY / dGU, follow.
    if ((rc = router_wgrad_and_unpermute(d, plan, wsh, grid, WL, wsb, router, r, grads->dXp, dx, s, hook))) return rc;
    const bool nb = opts != nullptr && opts->wgrad_subbatches == 2;
    if (nb) {
      int32_t* sb_rows = reinterpret_cast<int32_t*>(wsb + WL.sb_rows);
      if (launch_subbatch_rows(plan->offsets, plan->counts, plan->row_src, d.E, (d.T + 1) / 2, sb_rows, s, hook) !=
          cudaSuccess)
        return MOE_ERR_LAUNCH;
      g.sb_rows = sb_rows;
    }
    // BW: one pass (sb 0).  NB: sub-batch 0 stored (sb 1), then sub-batch 1 added (sb 2).
    g.grid = wgrad_grid(d, opts, sms);
    for (int sb = nb ? 1 : 0; sb <= (nb ? 2 : 0); ++sb) {
      g.sb = sb;
      g.pair = use_pair(opts, kWgrad13, d);
      if ((e = launch_gemm(kWgrad13, g, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
      g.pair = use_pair(opts, kWgrad2, d);
      if ((e = launch_gemm(kWgrad2, g, s, hook)) != cudaSuccess) return MOE_ERR_LAUNCH;
    }
    return MOE_OK;
  }
  return router_wgrad_and_unpermute(d, plan, wsh, grid, WL, wsb, router, r, grads->dXp, dx, s, hook);
}

int moe_router_forward(moe_dims d, const void* x, const void* Wr, float* logits, void* ws, size_t ws_bytes,
                       const moe_opts* opts, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (d.E % 8 != 0) return MOE_ERR_SHAPE;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (opts != nullptr && opts->grid < 0) return MOE_ERR_ARG;
  if (d.T == 0) return MOE_OK;
  if ((rc = check_ptrs({x, Wr, logits}))) return rc;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  if (!tensor_map_encoder_ready()) return MOE_ERR_LAUNCH;
  GemmLaunch g{};
  g.T = d.T;
  g.H = d.H;
  g.F = d.F;
  g.E = d.E;
  g.k = d.k;
  g.R = static_cast<int>(rows_of(d));
  g.grid = grid_for(opts, sms);
  g.ws = static_cast<WsHeader*>(ws);
  g.x = x;
  g.Wr = Wr;
  g.logits = logits;
  LaunchHook hook = make_hook(opts);
  return finish(launch_gemm(kRfwd, g, static_cast<cudaStream_t>(stream), hook));
}

int moe_get_status(void* ws, void* stream, int32_t* device_status, int32_t* where, int32_t* detail) {
  if (ws == nullptr || device_status == nullptr) return MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_LAUNCH;
  int32_t h[3] = {0, 0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_LAUNCH;
  *device_status = h[0];
  if (where) *where = h[1];
  if (detail) *detail = h[2];
  if (h[0] != 0) {
    const int32_t z[3] = {0, 0, 0};
    if (cudaMemcpy(ws, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_LAUNCH;
  }
  return MOE_OK;
}

int moe_clear_status(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_ARG;
  // Only the three status words (status, where, detail): the call is also used
  // on moe_plan_noalloc's 16-byte status buffer.
  return cudaMemsetAsync(ws, 0, 3 * sizeof(int32_t), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_LAUNCH;
}

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument (null pointer, dimension, k > E or k > 32, R too large)";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_WS: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_LAUNCH: return "CUDA launch or API call failed";
    case MOE_ERR_SHAPE: return "unsupported shape (H, F must be multiples of 128; E <= 1024)";
    case MOE_ERR_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    case MOE_ERR_TIMEOUT: return "a bounded wait in a kernel expired";
    case MOE_ERR_NONFINITE: return "non-finite router logit";
    case MOE_ERR_BOUNDS: return "index out of bounds detected on the GPU";
    case MOE_ERR_TOO_LARGE: return "dims need more scratch than moe_plan_noalloc's fixed buffer (MOE_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown error";
  }
}

int32_t moe_version(void) { return 1; }

uint64_t moe_launch_count(void) { return g_launches.load(); }

const char* moe_kernel_name(int32_t call, int32_t i) {
  const char* const* t = call == 0   ? kPlanKernels
                         : call == 1 ? kFwdKernels
                         : call == 2 ? kBwdKernels
                         : call == 3 ? kFwdKernelsFused
                         : call == 4 ? kBwdKernelsFused
                         : call == 5 ? kBwdKernelsRouter
                         : call == 6 ? kRouterFwdKernels
                         : call == 7 ? kFwdKernelsCombineFused
                         : call == 8 ? kBwdKernelsNB
                         : call == 9 ? kBwdKernelsRouterNB
                         : call == 10 ? kFwdKernelsGather
                         : call == 11 ? kFwdKernelsGatherCombine
                                     : nullptr;
  if (t == nullptr || i < 0) return nullptr;
  for (int j = 0; j <= i; ++j)
    if (t[j] == nullptr) return nullptr;
  return t[i];
}

}  // extern "C"
