// C ABI of the MoE decode library: argument checks, workspace layout, kernel
// choice by batch size and the stream schedule of the MoE layer.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <utility>

#include "internal.h"

using namespace dec;

namespace {

constexpr int kMaxM = 64;
constexpr int kMaxTopK = 16;
constexpr int kMaxE = 1024;

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

#define DEC_CUDA(expr)                         \
  do {                                         \
    if ((expr) != cudaSuccess) return DEC_ERR_CUDA; \
  } while (0)

// Split a workspace into 256-byte-aligned pieces.
struct Carver {
  char* base;
  size_t used = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += al256(count * sizeof(T));
    return p;
  }
};

struct EngineRegion {
  float* partials = nullptr;
  int* counters = nullptr;
};

// Split-K tile counters must be zero when a call starts (each call leaves them
// zero). They are carved first in every layout, so that a workspace reused by
// a call of another shape finds its counters in bytes that were counters before.
void carve_counters(Carver& c, EngineRegion& r, long long max_tiles) {
  r.counters = c.take<int>((size_t)std::max<long long>(max_tiles, 1));
}
void carve_partials(Carver& c, EngineRegion& r, int grid, int nacc) {
  r.partials = c.take<float>((size_t)2 * grid * nacc * kTileN * kMaxCols);
}
EngineRegion carve_engine(Carver& c, int grid, int nacc, long long max_tiles) {
  EngineRegion r;
  carve_counters(c, r, max_tiles);
  carve_partials(c, r, grid, nacc);
  return r;
}

bool linear_shape_ok(int M, int N, int K, int ldx) {
  return M >= 1 && M <= kMaxM && N >= 1 && K >= 8 && K % 8 == 0 && ldx >= K && ldx % 8 == 0;
}

int choose_variant(const dec_handle* h, int M, int N, int K) {
  if (h->force_variant == DEC_VARIANT_SMALL_M || h->force_variant == DEC_VARIANT_SPLIT_K) return h->force_variant;
  // Measured on GB300 (CUDA-graph replay of back-to-back launches, weights rotated past L2): with
  // its L2 request-ahead the small-matrix kernel streams 115-174 MB weights at 6.9-7.0 TB/s with
  // one token and 6.1-6.3 TB/s with two, where the split-K kernel reaches 4.6-5.7; with three or
  // four tokens it drops to 1.8-3.8 TB/s (its FMA and unpacking work grows with the tokens)
  // against the split-K kernel's 4.6-5.5. But the split-K kernel costs about 15 us per launch
  // beyond its bytes, so small matrices (the tensor-parallel shard shapes) stay on the
  // small-matrix kernel up to four tokens.
  if (!gemv_supported(M, K)) return DEC_VARIANT_SPLIT_K;
  const double bytes = (double)N * K * 2.0;
  if (M <= 2 || bytes <= 48e6) return DEC_VARIANT_SMALL_M;
  return DEC_VARIANT_SPLIT_K;
}

// gamma (small-matrix kernel): the input rows are RMS-normalised inside the
// projection kernel.
dec_status linear_impl(dec_handle* h, const uint16_t* x, int ldx, const uint16_t* W, const uint16_t* r, uint16_t* y,
                       int M, int N, int K, EngineRegion eng, cudaStream_t s, const char* tag = "linear",
                       const uint16_t* gamma = nullptr, float eps = 0.f) {
  const int v = choose_variant(h, M, N, K);
  cudaError_t e;
  LaunchScope scope(h, tag, s);
  if (v == DEC_VARIANT_SMALL_M) {
    if (!gemv_supported(M, K)) return DEC_ERR_UNSUPPORTED;
    e = launch_gemv(h, x, ldx, W, r, N, y, N, M, N, K, s, gamma, eps);
  } else {
    EngineLaunch L;
    L.epi = EPI_LINEAR;
    L.A = W;
    L.a_rows = N;
    L.B = x;
    L.b_rows = M;
    L.ldb = ldx;
    L.K = K;
    L.N = N;
    L.count = M;
    L.out = y;
    L.ldo = N;
    L.res = r;
    L.ldr = N;
    L.partials = eng.partials;
    L.counters = eng.counters;
    e = launch_engine(h, L, s);
  }
  h->last_variant = v;
  return e == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

// ---------------------------------------------------------------- MoE workspace
struct MoeWs {
  int* table = nullptr;
  uint16_t* xs = nullptr;
  uint16_t* hbuf = nullptr;
  float* y = nullptr;
  uint16_t* hs = nullptr;
  float* ys = nullptr;
  EngineRegion r0, r1;
};

long long moe_tiles(int E, int H, int I) { return (long long)E * (std::max(H, I) / kTileN); }

void carve_moe_counters(Carver& c, int E, int H, int I, long long extra_tiles, MoeWs* w) {
  carve_counters(c, w->r0, std::max(moe_tiles(E, H, I), extra_tiles));
  carve_counters(c, w->r1, std::max(H, I) / kTileN);
}

void carve_moe_data(Carver& c, const dec_handle* h, int M, int k, int E, int H, int I, MoeWs* w) {
  const int n = M * k;
  w->table = c.take<int>(TableLayout(E, n).words());
  w->xs = c.take<uint16_t>((size_t)n * H);
  w->hbuf = c.take<uint16_t>((size_t)n * I);
  w->y = c.take<float>((size_t)n * H);
  w->hs = c.take<uint16_t>((size_t)M * I);
  w->ys = c.take<float>((size_t)M * H);
  carve_partials(c, w->r0, engine_grid(h), 2);
  carve_partials(c, w->r1, engine_grid(h), 2);
}

void carve_moe(Carver& c, const dec_handle* h, int M, int k, int E, int H, int I, long long extra_tiles,
               MoeWs* w) {
  carve_moe_counters(c, E, H, I, extra_tiles, w);
  carve_moe_data(c, h, M, k, E, H, I, w);
}

bool moe_shape_ok(int M, int k, int E, int H, int I) {
  return M >= 1 && M <= kMaxM && k >= 1 && k <= kMaxTopK && E >= k && E <= kMaxE && H >= kTileN &&
         H % kTileN == 0 && I >= kTileN && I % kTileN == 0;
}

// Expert kernel family: the small-matrix kernels for one token (unless the
// split-K family is forced), the split-K tcgen05 engine otherwise.
bool experts_small(const dec_handle* h, int M, int H, int I) {
  return M == 1 && h->force_variant != DEC_VARIANT_SPLIT_K && gemv_moe_supported(H) && gemv_moe_supported(I);
}

// A few tokens: the small-matrix kernels over one problem per (token, expert)
// entry (an expert chosen by several tokens is read once per entry), unless
// the split-K family is forced. Measured on GB300 (layer step, graph replay,
// this path against the split-K experts, one box):
//  - two tokens: 297 against 312 us (full shapes), 74 against 77 (TP8 shard
//    shapes), 54 against 67 (TP16);
//  - three tokens: slower at full shapes (409.7 against 402.6 us), faster at
//    TP8 (86.7 against 89.8) and TP16 (60.5 against 68.3): for small experts
//    the split-K chain's seven launches outweigh the extra reads (repeated
//    experts, the shared down projection once per token);
//  - four tokens: slower at full shapes (511.0 against 492.7) and TP8 (110.2
//    against 105.8), faster at TP16 (71.3 against 76.7).
// So: two tokens; three when one expert's gate/up is at most 8 MB; four when
// it is at most 4 MB; with the small-matrix family forced, two to four.
bool experts_few(const dec_handle* h, int M, int k, int E, int H, int I) {
  if (M < 2 || M > 4 || !gemv_moe_supported(H) || !gemv_moe_supported(I) || !route_shared_supported(h, M, H, E, k))
    return false;
  if (h->force_variant == DEC_VARIANT_SMALL_M) return true;
  if (h->force_variant != DEC_VARIANT_AUTO) return false;
  const double gate_up_bytes = 2.0 * I * H * 2;  // one expert's gate and up matrices, bf16
  return M == 2 || (M == 3 && gate_up_bytes <= 8e6) || (M == 4 && gate_up_bytes <= 4e6);
}

// SM shares of the shared and the routed experts ("the schedule controls how
// many GPU resources each op uses", Kimi K3 article, Part 1 §3).
//  - overlap (h->shared_ctas < 0): both use every SM; the hardware hands SMs
//    to the routed kernels as the shared expert's CTAs finish.
//  - byte share: the shared expert keeps its share of the expected weight
//    bytes, rounded up with a 25% margin (at least one SM, at most half).
//    Expected distinct experts for uniform routing: E (1 - (1 - k/E)^M).
//  - automatic (h->shared_ctas == 0, default): overlap from four tokens on
//    when the shared expert is large (at least 48 MB of weights), the byte
//    share otherwise.
//  - fixed (h->shared_ctas > 0): that many SMs for the shared expert.
// Measured on GB300 (layer step, CUDA-graph replay): with independent tokens
// overlap is within -0.7% / +0.3% of the byte share from four tokens on and
// 1.6% slower at three; with related tokens (speculative-verify groups of 8
// drafts) routing is far from uniform, U far below the expectation, and the
// byte share starves the shared expert: overlap is 8% faster at 8 tokens and
// 17% at 16. But a small shared expert (the tensor-parallel shard shapes:
// 11 MB) is mostly the split-K kernel's fixed per-launch cost, and on every
// SM it holds the whole GPU for it: there the byte share is 1.4-1.9x faster.
bool shared_overlap_auto(const dec_handle* h, int M, int H, int I) {
  return h->shared_ctas == 0 && M >= 4 && 3.0 * I * H * 2.0 >= 48e6;
}

int shared_grid(const dec_handle* h, int M, int k, int E, int H, int I) {
  if (h->shared_ctas > 0) return std::min(h->shared_ctas, h->sms - 1);
  if (h->shared_ctas < 0 || shared_overlap_auto(h, M, H, I)) return h->sms;
  const double eu = E * (1.0 - std::pow(1.0 - (double)k / E, (double)M));
  const int g = (int)std::ceil(1.25 * h->sms / (1.0 + eu));
  return std::max(1, std::min(g, h->sms / 2));
}

int routed_grid(const dec_handle* h, int M, int k, int E, int H, int I, bool has_shared) {
  if (!has_shared || h->shared_ctas < 0 || shared_overlap_auto(h, M, H, I)) return h->sms;
  return h->sms - shared_grid(h, M, k, E, H, I);
}

// The shared expert on the handle's side stream, forked from `s` now. It does
// not depend on routing, so it is launched before the router: its weight
// stream fills the bandwidth that the latency-bound router / top-k / routing
// table phase leaves idle (Kimi K3 article, Part 1 §3). Joined by moe_routed.
dec_status moe_shared_fork(dec_handle* h, const uint16_t* x, int M, int k, int E, int H, int I,
                           const uint16_t* Wg_s, const uint16_t* Wu_s, const uint16_t* Wd_s, const MoeWs& ws,
                           cudaStream_t s) {
  const bool has_shared = Wg_s != nullptr;
  const int g1 = has_shared ? shared_grid(h, M, k, E, H, I) : 0;
  // At one token the shared expert is problem 0 of the routed launches (see moe_routed).
  if (experts_small(h, M, H, I)) return DEC_OK;
  if (has_shared) {
    DEC_CUDA(cudaEventRecord(h->ev_fork, s));
    DEC_CUDA(cudaStreamWaitEvent(h->side, h->ev_fork, 0));
    EngineLaunch L;
    L.epi = EPI_SWIGLU;
    L.A = Wg_s;
    L.A2 = Wu_s;
    L.a_rows = I;
    L.B = x;
    L.b_rows = M;
    L.ldb = H;
    L.K = H;
    L.N = I;
    L.count = M;
    L.out = ws.hs;
    L.ldo = I;
    L.partials = ws.r1.partials;
    L.counters = ws.r1.counters;
    L.grid = g1;
    {
      LaunchScope scope(h, "shared_gate_up", h->side);
      DEC_CUDA(launch_engine(h, L, h->side));
    }
    EngineLaunch D;
    D.epi = EPI_F32;
    D.A = Wd_s;
    D.a_rows = H;
    D.B = ws.hs;
    D.b_rows = M;
    D.ldb = I;
    D.K = I;
    D.N = H;
    D.count = M;
    D.out = ws.ys;
    D.ldo = H;
    D.partials = ws.r1.partials;
    D.counters = ws.r1.counters;
    D.grid = g1;
    {
      LaunchScope scope(h, "shared_down", h->side);
      DEC_CUDA(launch_engine(h, D, h->side));
    }
    DEC_CUDA(cudaEventRecord(h->ev_join, h->side));
  }
  return DEC_OK;
}

// One token, small-matrix kernels: routed and shared experts in one balanced
// launch per matrix over every SM (the shared expert is problem 0), the down
// projection fused with the combine and the residual where supported. The
// routing table in ws.table is complete; slot j's activation row is at
// x + j * ldx (ldx 0: one row for all slots).
dec_status moe_small(dec_handle* h, const uint16_t* x, long long ldx, const float* w, int k, const uint16_t* Wg,
                     const uint16_t* Wu, const uint16_t* Wd, int E, int H, int I, const uint16_t* Wg_s,
                     const uint16_t* Wu_s, const uint16_t* Wd_s, const uint16_t* residual, uint16_t* out,
                     const MoeWs& ws, cudaStream_t s) {
  const bool has_shared = Wg_s != nullptr;
  h->last_expert_variant = DEC_VARIANT_SMALL_M;
  // the shared expert's activation: slot 0's row (every slot holds the token's row)
  const GemvMoeShared sgu{Wg_s, Wu_s, x, ws.hs}, sdn{Wd_s, nullptr, ws.hs, ws.ys};
  const bool fused_down = gemv_down_combine_supported(k, I);
  {
    LaunchScope scope(h, "gate_up", s);
    // Late trigger (dependents launch only after this launch's dependency
    // wait): lets the fused down kernel read the routing early, and keeps the
    // next routing launch from starting before this one's predecessor (the
    // routing launch, whose row queue it reuses) has completed.
    DEC_CUDA(launch_gemv_moe(h, true, Wg, Wu, I, I, H, x, ldx, ws.table, E, k, ws.hbuf, I, h->sms, s,
                             has_shared ? &sgu : nullptr, k, fused_down));
  }
  if (fused_down) {
    // down projection + weighted combine + residual in one kernel; the routing
    // is read before its dependency wait (the gate/up launch triggers its
    // dependents only after its own wait, when the routing is complete)
    LaunchScope scope(h, "down", s);
    DEC_CUDA(launch_gemv_down_combine(h, Wd, H, has_shared ? Wd_s : nullptr, H, I, ws.hbuf, ws.hs, ws.table, E, k, w,
                                      residual, out, h->sms, s, true));
    return DEC_OK;
  }
  {
    LaunchScope scope(h, "down", s);
    DEC_CUDA(launch_gemv_moe(h, false, Wd, nullptr, H, H, I, ws.hbuf, I, ws.table, E, k, ws.y, H, h->sms, s,
                             has_shared ? &sdn : nullptr, k, false));
  }
  {
    LaunchScope scope(h, "combine", s);
    DEC_CUDA(launch_combine(h, ws.y, ws.table, w, 1, k, E, has_shared ? ws.ys : nullptr, residual, out, H, s));
  }
  return DEC_OK;
}

// Two to four tokens after the routing launch (route_shared: entry table,
// normalised rows x [M][H], and the shared expert's h_s [M][I] when there is
// one): gate/up over the M k entries (each reads its token's row; skipped when
// the MoE front launch has written them, gate_up_done), down over the shared
// expert applied to the M rows of h_s plus the entries, then the weighted
// combine with the shared output and the residual.
dec_status moe_few(dec_handle* h, int M, const uint16_t* x, const float* w, int k, const uint16_t* Wg,
                   const uint16_t* Wu, const uint16_t* Wd, int E, int H, int I, const uint16_t* Wd_s,
                   const uint16_t* residual, uint16_t* out, const MoeWs& ws, cudaStream_t s,
                   bool gate_up_done = false) {
  const int n = M * k;
  h->last_expert_variant = DEC_VARIANT_SMALL_M;
  if (!gate_up_done) {
    // late trigger: the next routing launch reuses this launch's predecessor's row queue
    LaunchScope scope(h, "gate_up", s);
    DEC_CUDA(launch_gemv_moe(h, true, Wg, Wu, I, I, H, x, H, ws.table, E, n, ws.hbuf, I, h->sms, s, nullptr, n,
                             true, true));
  }
  if (M == 2 && gemv_down_combine2_supported(k, I)) {
    // two tokens: down, weighted combine and residual in one kernel (the shared
    // W_d read once for both rows); the routing is read before the dependency
    // wait, as the launch before triggers its dependents only once the routing
    // is written
    LaunchScope scope(h, "down", s);
    DEC_CUDA(launch_gemv_down_combine2(h, Wd, H, Wd_s, H, I, ws.hbuf, ws.hs, ws.table, E, k, w, residual, out, h->sms,
                                       s, true));
    return DEC_OK;
  }
  GemvMoeShared sdn{Wd_s, nullptr, ws.hs, ws.ys};
  sdn.n = M;
  sdn.ldx = I;
  sdn.ldo = H;
  {
    LaunchScope scope(h, "down", s);
    DEC_CUDA(launch_gemv_moe(h, false, Wd, nullptr, H, H, I, ws.hbuf, I, ws.table, E, n, ws.y, H, h->sms, s,
                             Wd_s != nullptr ? &sdn : nullptr, n, false, false));
  }
  {
    LaunchScope scope(h, "combine", s);
    DEC_CUDA(launch_combine(h, ws.y, ws.table, w, M, k, E, Wd_s != nullptr ? ws.ys : nullptr, residual, out, H, s));
  }
  return DEC_OK;
}

dec_status moe_routed(dec_handle* h, const uint16_t* x, const int32_t* idx, const float* w, int M, int k,
                      const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int E, int H, int I,
                      const uint16_t* Wg_s, const uint16_t* Wu_s, const uint16_t* Wd_s, const uint16_t* residual,
                      uint16_t* out, const MoeWs& ws, cudaStream_t s) {
  const bool has_shared = Wg_s != nullptr;
  const int n = M * k;
  const int g0 = routed_grid(h, M, k, E, H, I, has_shared);
  if (experts_small(h, M, H, I)) {
    {
      LaunchScope scope(h, "route_table", s);
      DEC_CUDA(launch_one_token_table(h, idx, E, k, ws.table, s));
    }
    return moe_small(h, x, 0, w, k, Wg, Wu, Wd, E, H, I, Wg_s, Wu_s, Wd_s, residual, out, ws, s);
  }
  {
    LaunchScope scope(h, "route_table", s);
    DEC_CUDA(launch_route_table(h, idx, M, k, E, x, H, ws.table, ws.xs, s));
  }
  h->last_expert_variant = DEC_VARIANT_SPLIT_K;
  EngineLaunch L;
  L.epi = EPI_SWIGLU;
  L.A = Wg;
  L.A2 = Wu;
  L.a_rows = (long long)E * I;
  L.a_rows_per_prob = I;
  L.B = ws.xs;
  L.b_rows = n;
  L.ldb = H;
  L.K = H;
  L.N = I;
  L.table = ws.table;
  L.E = E;
  L.n_entries = n;
  L.count = M;  // bound on the tokens of any one expert
  L.out = ws.hbuf;
  L.ldo = I;
  L.partials = ws.r0.partials;
  L.counters = ws.r0.counters;
  L.grid = g0;
  {
    LaunchScope scope(h, "gate_up", s);
    DEC_CUDA(launch_engine(h, L, s));
  }
  EngineLaunch D;
  D.epi = EPI_F32;
  D.A = Wd;
  D.a_rows = (long long)E * H;
  D.a_rows_per_prob = H;
  D.B = ws.hbuf;
  D.b_rows = n;
  D.ldb = I;
  D.K = I;
  D.N = H;
  D.table = ws.table;
  D.E = E;
  D.n_entries = n;
  D.count = M;
  D.out = ws.y;
  D.ldo = H;
  D.partials = ws.r0.partials;
  D.counters = ws.r0.counters;
  D.grid = g0;
  {
    LaunchScope scope(h, "down", s);
    DEC_CUDA(launch_engine(h, D, s));
  }
  if (has_shared) DEC_CUDA(cudaStreamWaitEvent(s, h->ev_join, 0));
  {
    LaunchScope scope(h, "combine", s);
    DEC_CUDA(launch_combine(h, ws.y, ws.table, w, M, k, E, has_shared ? ws.ys : nullptr, residual, out, H, s));
  }
  return DEC_OK;
}

dec_status moe_impl(dec_handle* h, const uint16_t* x, const int32_t* idx, const float* w, int M, int k,
                    const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int E, int H, int I,
                    const uint16_t* Wg_s, const uint16_t* Wu_s, const uint16_t* Wd_s, const uint16_t* residual,
                    uint16_t* out, const MoeWs& ws, cudaStream_t s) {
  dec_status st = moe_shared_fork(h, x, M, k, E, H, I, Wg_s, Wu_s, Wd_s, ws, s);
  if (st != DEC_OK) return st;
  return moe_routed(h, x, idx, w, M, k, Wg, Wu, Wd, E, H, I, Wg_s, Wu_s, Wd_s, residual, out, ws, s);
}

// ---------------------------------------------------------------- MoE layer / decode layer workspaces
struct MoeLayerWs {
  int* sel_counter = nullptr;  // the routing launches' counters (hand-off, row queue, done, routing flag, tail queue,
                               // tail owner, router-unit tickets)
  uint16_t* b = nullptr;       // the normalised rows (when a launch writes them out)
  float* parts = nullptr;
  int32_t* idx = nullptr;
  float* w = nullptr;
  MoeWs moe;
};

struct LayerWs {
  uint16_t* a = nullptr;
  uint16_t* yin = nullptr;
  uint16_t* h1 = nullptr;
  MoeLayerWs ml;
};

// Counters first: the routing counters, then the split-K tile counters
// (extra_tiles: room for the dense projections' tiles as well).
void carve_moe_layer_head(Carver& c, int E, int H, int I, long long extra_tiles, MoeLayerWs* w) {
  w->sel_counter = c.take<int>(8);
  carve_moe_counters(c, E, H, I, extra_tiles, &w->moe);
}

void carve_moe_layer_data(Carver& c, const dec_handle* h, int M, int k, int E, int H, int I, MoeLayerWs* w) {
  w->b = c.take<uint16_t>((size_t)M * H);
  w->parts = c.take<float>((size_t)router_ksplit(H) * M * E);
  w->idx = c.take<int32_t>((size_t)M * k);
  w->w = c.take<float>((size_t)M * k);
  carve_moe_data(c, h, M, k, E, H, I, &w->moe);
}

bool layer_ok(const dec_layer_weights* L, int M) {
  if (!L || M < 1 || M > kMaxM) return false;
  if (L->H < kTileN || L->H % kTileN != 0 || L->N_in < 8 || L->N_in % 8 != 0 || L->K_out < 8 ||
      L->K_out % 8 != 0 || L->K_out > L->N_in)
    return false;
  return moe_shape_ok(M, L->k, L->E, L->H, L->I);
}

void carve_layer(Carver& c, const dec_handle* h, const dec_layer_weights* L, int M, LayerWs* w) {
  const int H = L->H;
  const long long dense_tiles = std::max<long long>((L->N_in + kTileN - 1) / kTileN, H / kTileN);
  carve_moe_layer_head(c, L->E, H, L->I, dense_tiles, &w->ml);
  w->a = c.take<uint16_t>((size_t)M * H);
  w->yin = c.take<uint16_t>((size_t)M * L->N_in);
  w->h1 = c.take<uint16_t>((size_t)M * H);
  carve_moe_layer_data(c, h, M, L->k, L->E, H, L->I, &w->ml);
}

// ---------------------------------------------------------------- MoE layer
struct MoeLayerArgs {
  const uint16_t* x = nullptr;      // [M][H] the layer's input rows
  const uint16_t* gamma = nullptr;  // RMSNorm gains applied to x first, or null
  float eps = 0.f;
  const float* Wr = nullptr;
  int M = 0, k = 0, E = 0, H = 0, I = 0;
  const uint16_t *Wg = nullptr, *Wu = nullptr, *Wd = nullptr;
  const uint16_t *Wg_s = nullptr, *Wu_s = nullptr, *Wd_s = nullptr;
  const uint16_t* residual = nullptr;  // or null
  uint16_t* out = nullptr;
  int32_t* idx = nullptr;
  float* w = nullptr;
  float* scores = nullptr;             // or null
  const void* pf = nullptr;            // a region to pull into L2 during the routing (Part 1 §4), or null
  size_t pf_bytes = 0;
};

// The MoE layer: [RMSNorm,] router, top-k, routing table, routed and shared
// experts, combine [+ residual]; the kernel schedule by batch.
dec_status moe_layer_impl(dec_handle* h, const MoeLayerArgs& A, const MoeLayerWs& w, cudaStream_t s) {
  const int M = A.M, H = A.H;
  // One to a few tokens on the small-matrix experts: the RMSNorm, the router,
  // the top-k and the routing table are one launch (route_shared /
  // router_select / the MoE fronts), and the experts read the normalised rows
  // by token (no gather). Otherwise the split-K family's chain of launches.
  const bool one_token = experts_small(h, M, H, A.I);
  const bool few_tokens = !one_token && experts_few(h, M, A.k, A.E, H, A.I);
  // the rows the experts read: the routing launch writes them out when it normalises
  const uint16_t* b = A.gamma != nullptr ? w.b : A.x;
  if (!one_token && !few_tokens && A.gamma != nullptr) {
    LaunchScope scope(h, "rmsnorm2", s);
    if (launch_rmsnorm(h, A.x, A.gamma, w.b, M, H, A.eps, s) != cudaSuccess) return DEC_ERR_CUDA;
  }
  // Kimi K3 article, Part 1 §4: while the router / top-k phase leaves the
  // memory idle, a side-stream kernel pulls weights that come next into L2:
  // at one token the shared expert (it runs inside the routed launches), and
  // the caller's next-operator region if given.
  // The MoE front launches (one token; two to four on the small-matrix
  // family) pull the next-operator region themselves, from the CTAs that wait
  // for the routing, so the side stream then carries only the shared expert.
  const bool front1 = one_token && A.Wg_s != nullptr && h->moe_front && route_shared_supported(h, 1, H, A.E, A.k) &&
                      gemv_down_combine_supported(A.k, A.I);
  const bool front_few = few_tokens && A.Wg_s != nullptr && h->moe_front && M * A.k <= 32;
  const bool next_in_front = (front1 || front_few) && A.pf != nullptr && A.pf_bytes > 0;
  const bool pf = A.pf != nullptr && A.pf_bytes > 0 && !next_in_front;
  const void* pf_front = next_in_front ? A.pf : nullptr;
  const size_t pf_front_bytes = next_in_front ? A.pf_bytes : 0;
  if (pf) {
    DEC_CUDA(cudaEventRecord(h->ev_pf_fork, s));
    DEC_CUDA(cudaStreamWaitEvent(h->pf, h->ev_pf_fork, 0));
    {
      LaunchScope scope(h, "prefetch", h->pf);
      DEC_CUDA(launch_prefetch(h, A.pf, A.pf_bytes, 16, h->pf));
    }
    DEC_CUDA(cudaEventRecord(h->ev_pf_join, h->pf));
  }
  dec_status st = DEC_OK;
  // The router / top-k phase is latency-bound; the shared expert and the
  // prefetch stream use the idle bandwidth meanwhile.
  if (one_token) {
    if (front1) {
      // One MoE front launch (routing, shared gate/up, routed gate/up), then
      // the down projection with the combine and the residual.
      h->last_expert_variant = DEC_VARIANT_SMALL_M;
      {
        LaunchScope scope(h, "moe_front", s);
        DEC_CUDA(launch_moe_front(h, A.x, A.gamma, A.eps, A.Wr, H, A.E, A.k, w.parts, w.sel_counter, A.idx, A.w,
                                  A.scores, w.moe.table, A.Wg_s, A.Wu_s, A.I, w.moe.hs, A.Wg, A.Wu, w.moe.hbuf, s,
                                  pf_front, pf_front_bytes));
      }
      {
        LaunchScope scope(h, "down", s);
        DEC_CUDA(launch_gemv_down_combine(h, A.Wd, H, A.Wd_s, H, A.I, w.moe.hbuf, w.moe.hs, w.moe.table, A.E, A.k, A.w,
                                          A.residual, A.out, h->sms, s, true));
      }
      if (pf) DEC_CUDA(cudaStreamWaitEvent(s, h->ev_pf_join, 0));
      return DEC_OK;
    }
    // Without the front (no shared expert, or shapes outside its limits): the
    // routing launch, then the grouped kernels with the shared expert as
    // problem 0 of the gate/up launch and one more matrix of the down launch.
    {
      LaunchScope scope(h, "router", s);
      DEC_CUDA(launch_router_select(h, A.x, A.gamma, A.eps, A.Wr, H, A.E, A.k, w.b, w.parts, w.sel_counter, A.idx,
                                    A.w, A.scores, w.moe.table, s));
    }
    st = moe_small(h, b, 0, A.w, A.k, A.Wg, A.Wu, A.Wd, A.E, H, A.I, A.Wg_s, A.Wu_s, A.Wd_s, A.residual, A.out, w.moe,
                   s);
    if (st != DEC_OK) return st;
    if (pf) DEC_CUDA(cudaStreamWaitEvent(s, h->ev_pf_join, 0));
    return DEC_OK;
  }
  if (few_tokens) {
    // Two to four tokens: the RMSNorm, router, top-k, routing table (one
    // problem per entry) and the shared expert's gate/up in one launch; with
    // the MoE front schedule the entries' gate/up as well.
    if (front_few) {
      {
        LaunchScope scope(h, "moe_front", s);
        DEC_CUDA(launch_moe_front_multi(h, M, A.x, A.gamma, A.eps, A.Wr, H, A.E, A.k, w.parts, w.sel_counter, A.idx,
                                        A.w, A.scores, w.moe.table, A.Wg_s, A.Wu_s, A.I, w.moe.hs, A.Wg, A.Wu,
                                        w.moe.hbuf, s, pf_front, pf_front_bytes));
      }
      st = moe_few(h, M, w.b, A.w, A.k, A.Wg, A.Wu, A.Wd, A.E, H, A.I, A.Wd_s, A.residual, A.out, w.moe, s, true);
      if (st != DEC_OK) return st;
      if (pf) DEC_CUDA(cudaStreamWaitEvent(s, h->ev_pf_join, 0));
      return DEC_OK;
    }
    {
      LaunchScope scope(h, "router", s);
      DEC_CUDA(launch_route_shared(h, M, A.x, A.gamma, A.eps, A.Wr, H, A.E, A.k, w.b, w.parts, w.sel_counter, A.idx,
                                   A.w, A.scores, w.moe.table, A.Wg_s, A.Wu_s, A.Wg_s ? A.I : 0, w.moe.hs, s));
    }
    // (the routing launch writes its rows, normalised or as they are, to w.b)
    st = moe_few(h, M, w.b, A.w, A.k, A.Wg, A.Wu, A.Wd, A.E, H, A.I, A.Wd_s, A.residual, A.out, w.moe, s);
    if (st != DEC_OK) return st;
    if (pf) DEC_CUDA(cudaStreamWaitEvent(s, h->ev_pf_join, 0));
    return DEC_OK;
  }
  st = moe_shared_fork(h, b, M, A.k, A.E, H, A.I, A.Wg_s, A.Wu_s, A.Wd_s, w.moe, s);
  if (st != DEC_OK) return st;
  {
    LaunchScope scope(h, "router", s);
    if (launch_router(h, b, A.Wr, M, H, A.E, w.parts, s) != cudaSuccess) return DEC_ERR_CUDA;
  }
  {
    LaunchScope scope(h, "topk", s);
    if (launch_topk(h, w.parts, router_ksplit(H), M, A.E, A.k, A.idx, A.w, A.scores, s) != cudaSuccess)
      return DEC_ERR_CUDA;
  }
  st = moe_routed(h, b, A.idx, A.w, M, A.k, A.Wg, A.Wu, A.Wd, A.E, H, A.I, A.Wg_s, A.Wu_s, A.Wd_s, A.residual, A.out,
                  w.moe, s);
  if (st != DEC_OK) return st;
  if (pf) DEC_CUDA(cudaStreamWaitEvent(s, h->ev_pf_join, 0));
  return DEC_OK;
}

}  // namespace

extern "C" {

const char* dec_status_string(dec_status s) {
  switch (s) {
    case DEC_OK: return "ok";
    case DEC_ERR_INVALID_ARG: return "invalid argument";
    case DEC_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case DEC_ERR_CUDA: return "CUDA error";
    case DEC_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

dec_status dec_create(dec_handle** out, int device) {
  if (out == nullptr) return DEC_ERR_INVALID_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return DEC_ERR_CUDA;
  int prev = 0;
  DEC_CUDA(cudaGetDevice(&prev));
  DEC_CUDA(cudaSetDevice(device));
  dec_handle* h = new dec_handle();
  h->device = device;
  bool ok = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->pf, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->ev_pf_fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->ev_pf_join, cudaEventDisableTiming) == cudaSuccess &&
            cudaMalloc(&h->d_err, sizeof(int)) == cudaSuccess && cudaMemset(h->d_err, 0, sizeof(int)) == cudaSuccess;
  if (ok) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    ok = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
             cudaSuccess &&
         q == cudaDriverEntryPointSuccess && fn != nullptr;
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cudaSetDevice(prev);
  if (!ok) {
    dec_destroy(h);
    return DEC_ERR_CUDA;
  }
  *out = h;
  return DEC_OK;
}

dec_status dec_destroy(dec_handle* h) {
  if (h == nullptr) return DEC_OK;
  if (h->side) cudaStreamSynchronize(h->side);
  if (h->pf) cudaStreamSynchronize(h->pf);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->pf) cudaStreamDestroy(h->pf);
  for (cudaEvent_t e : {h->ev_fork, h->ev_join, h->ev_pf_fork, h->ev_pf_join})
    if (e) cudaEventDestroy(e);
  for (const auto& r : h->prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (cudaEvent_t e : h->event_pool) cudaEventDestroy(e);
  if (h->d_err) cudaFree(h->d_err);
  delete h;
  return DEC_OK;
}

dec_status dec_workspace_init(dec_handle* h, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (h == nullptr || (ws == nullptr && ws_bytes != 0)) return DEC_ERR_INVALID_ARG;
  if (ws_bytes == 0) return DEC_OK;
  return cudaMemsetAsync(ws, 0, ws_bytes, stream) == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_set_wait_limit_ns(dec_handle* h, uint64_t ns) {
  if (h == nullptr || ns == 0) return DEC_ERR_INVALID_ARG;
  h->wait_ns = ns;
  return DEC_OK;
}

dec_status dec_set_pdl(dec_handle* h, int enable) {
  if (h == nullptr) return DEC_ERR_INVALID_ARG;
  h->pdl = enable ? 1 : 0;
  return DEC_OK;
}

dec_status dec_test_set_moe_front(dec_handle* h, int enable) {
  if (h == nullptr) return DEC_ERR_INVALID_ARG;
  h->moe_front = enable ? 1 : 0;
  return DEC_OK;
}

dec_status dec_test_set_engine_finish(dec_handle* h, int mode) {
  if (h == nullptr || mode < 0 || mode > 2) return DEC_ERR_INVALID_ARG;
  h->engine_finish = mode;
  return DEC_OK;
}

dec_status dec_set_l2_ahead(dec_handle* h, int bytes) {
  if (h == nullptr || bytes < 0 || bytes > (16 << 20)) return DEC_ERR_INVALID_ARG;
  h->l2_ahead = bytes;
  return DEC_OK;
}

dec_status dec_set_shared_sms(dec_handle* h, int sms) {
  if (h == nullptr || sms < -1 || sms >= h->sms) return DEC_ERR_INVALID_ARG;
  h->shared_ctas = sms;
  return DEC_OK;
}

dec_status dec_set_force_variant(dec_handle* h, int variant) {
  if (h == nullptr || variant < DEC_VARIANT_AUTO || variant > DEC_VARIANT_SPLIT_K) return DEC_ERR_INVALID_ARG;
  h->force_variant = variant;
  return DEC_OK;
}

int dec_last_variant(const dec_handle* h) { return h ? h->last_variant : 0; }

int dec_last_expert_variant(const dec_handle* h) { return h ? h->last_expert_variant : 0; }

dec_status dec_check_device_error(dec_handle* h) {
  if (h == nullptr) return DEC_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return DEC_ERR_CUDA;
  int v = 0;
  DEC_CUDA(cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (v == 0) return DEC_OK;
  DEC_CUDA(cudaMemset(h->d_err, 0, sizeof(int)));
  return DEC_ERR_TIMEOUT;
}

// ---------------------------------------------------------------- projections
dec_status dec_linear_workspace_size(const dec_handle* h, int M, int N, int K, size_t* bytes) {
  if (h == nullptr || bytes == nullptr || !linear_shape_ok(M, N, K, K)) return DEC_ERR_INVALID_ARG;
  Carver c(nullptr);
  carve_engine(c, engine_grid(h), 1, (N + kTileN - 1) / kTileN);
  *bytes = c.used;
  return DEC_OK;
}

static dec_status linear_entry(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W, const dec_bf16* r,
                               dec_bf16* out, int M, int N, int K, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (h == nullptr || x == nullptr || W == nullptr || out == nullptr) return DEC_ERR_INVALID_ARG;
  if (!al16(x) || !al16(W) || !al16(out) || (r != nullptr && !al16(r))) return DEC_ERR_INVALID_ARG;
  if (!linear_shape_ok(M, N, K, ldx)) return DEC_ERR_INVALID_ARG;
  EngineRegion eng;
  if (choose_variant(h, M, N, K) == DEC_VARIANT_SPLIT_K) {
    size_t need = 0;
    dec_linear_workspace_size(h, M, N, K, &need);
    if (ws == nullptr || !al16(ws) || ws_bytes < need) return DEC_ERR_INVALID_ARG;
    Carver c(ws);
    eng = carve_engine(c, engine_grid(h), 1, (N + kTileN - 1) / kTileN);
  }
  return linear_impl(h, x, ldx, W, r, out, M, N, K, eng, s, r ? "linear_residual" : "linear");
}

dec_status dec_linear(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W, dec_bf16* y, int M, int N,
                      int K, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return linear_entry(h, x, ldx, W, nullptr, y, M, N, K, ws, ws_bytes, stream);
}

dec_status dec_linear_residual(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W, const dec_bf16* r,
                               dec_bf16* out, int M, int N, int K, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (r == nullptr) return DEC_ERR_INVALID_ARG;
  return linear_entry(h, x, ldx, W, r, out, M, N, K, ws, ws_bytes, stream);
}

dec_status dec_rmsnorm(dec_handle* h, const dec_bf16* x, const dec_bf16* gamma, dec_bf16* y, int M, int H, float eps,
                       cudaStream_t stream) {
  if (h == nullptr || x == nullptr || gamma == nullptr || y == nullptr) return DEC_ERR_INVALID_ARG;
  if (!al16(x) || !al16(gamma) || !al16(y) || M < 1 || M > kMaxM || H < 8 || H % 8 != 0 || H > 65536 ||
      !(eps >= 0.f))
    return DEC_ERR_INVALID_ARG;
  LaunchScope scope(h, "rmsnorm", stream);
  return launch_rmsnorm(h, x, gamma, y, M, H, eps, stream) == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

// ---------------------------------------------------------------- router
dec_status moe_route_topk_workspace_size(const dec_handle* h, int M, int H, int E, size_t* bytes) {
  if (h == nullptr || bytes == nullptr || M < 1 || M > kMaxM || H < 8 || H % 8 != 0 || E < 1 || E > kMaxE)
    return DEC_ERR_INVALID_ARG;
  *bytes = al256(sizeof(int)) + al256((size_t)router_ksplit(H) * M * E * sizeof(float));
  return DEC_OK;
}

dec_status moe_route_topk(dec_handle* h, const dec_bf16* x, const float* Wr, int M, int H, int E, int k,
                          int32_t* idx, float* w, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (h == nullptr || x == nullptr || Wr == nullptr || idx == nullptr || w == nullptr) return DEC_ERR_INVALID_ARG;
  if (!al16(x) || !al16(Wr) || !al16(ws)) return DEC_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxM || H < 8 || H % 8 != 0 || E < 1 || E > kMaxE || k < 1 || k > kMaxTopK || k > E)
    return DEC_ERR_INVALID_ARG;
  size_t need = 0;
  moe_route_topk_workspace_size(h, M, H, E, &need);
  if (ws == nullptr || ws_bytes < need) return DEC_ERR_INVALID_ARG;
  Carver c(ws);
  int* counter = c.take<int>(1);
  float* parts = c.take<float>((size_t)router_ksplit(H) * M * E);
  if (M == 1) {
    // one launch: logits, then the top-k by the last CTA
    LaunchScope scope(h, "router", stream);
    return launch_router_select(h, x, nullptr, 0.f, Wr, H, E, k, nullptr, parts, counter, idx, w, scores, nullptr,
                                stream) == cudaSuccess
               ? DEC_OK
               : DEC_ERR_CUDA;
  }
  {
    LaunchScope scope(h, "router", stream);
    if (launch_router(h, x, Wr, M, H, E, parts, stream) != cudaSuccess) return DEC_ERR_CUDA;
  }
  {
    LaunchScope scope(h, "topk", stream);
    if (launch_topk(h, parts, router_ksplit(H), M, E, k, idx, w, scores, stream) != cudaSuccess) return DEC_ERR_CUDA;
  }
  return DEC_OK;
}

// ---------------------------------------------------------------- experts
dec_status moe_experts_workspace_size(const dec_handle* h, int M, int k, int E, int H, int I, size_t* bytes) {
  if (h == nullptr || bytes == nullptr || !moe_shape_ok(M, k, E, H, I)) return DEC_ERR_INVALID_ARG;
  Carver c(nullptr);
  MoeWs w;
  carve_moe(c, h, M, k, E, H, I, 0, &w);
  *bytes = c.used;
  return DEC_OK;
}

dec_status moe_experts(dec_handle* h, const dec_bf16* x, const int32_t* idx, const float* w, int M, int k,
                       const dec_bf16* Wg, const dec_bf16* Wu, const dec_bf16* Wd, int E, int H, int I,
                       const dec_bf16* Wg_s, const dec_bf16* Wu_s, const dec_bf16* Wd_s, const dec_bf16* residual,
                       dec_bf16* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (h == nullptr || x == nullptr || idx == nullptr || w == nullptr || Wg == nullptr || Wu == nullptr ||
      Wd == nullptr || out == nullptr)
    return DEC_ERR_INVALID_ARG;
  const bool any_s = Wg_s || Wu_s || Wd_s, all_s = Wg_s && Wu_s && Wd_s;
  if (any_s && !all_s) return DEC_ERR_INVALID_ARG;
  for (const void* p : {(const void*)x, (const void*)idx, (const void*)w, (const void*)Wg, (const void*)Wu,
                        (const void*)Wd, (const void*)Wg_s, (const void*)Wu_s, (const void*)Wd_s,
                        (const void*)residual, (const void*)out, (const void*)ws})
    if (p != nullptr && !al16(p)) return DEC_ERR_INVALID_ARG;
  if (!moe_shape_ok(M, k, E, H, I)) return DEC_ERR_INVALID_ARG;
  if (out == x) return DEC_ERR_INVALID_ARG;
  size_t need = 0;
  moe_experts_workspace_size(h, M, k, E, H, I, &need);
  if (ws == nullptr || ws_bytes < need) return DEC_ERR_INVALID_ARG;
  Carver c(ws);
  MoeWs mw;
  carve_moe(c, h, M, k, E, H, I, 0, &mw);
  return moe_impl(h, x, idx, w, M, k, Wg, Wu, Wd, E, H, I, Wg_s, Wu_s, Wd_s, residual, out, mw, stream);
}

// ---------------------------------------------------------------- decode layer
dec_status decode_layer_workspace_size(const dec_handle* h, const dec_layer_weights* Wt, int M, size_t* bytes) {
  if (h == nullptr || bytes == nullptr || !layer_ok(Wt, M)) return DEC_ERR_INVALID_ARG;
  Carver c(nullptr);
  LayerWs w;
  carve_layer(c, h, Wt, M, &w);
  *bytes = c.used;
  return DEC_OK;
}

dec_status decode_layer(dec_handle* h, const dec_layer_weights* Wt, dec_bf16* hidden, int M,
                        const dec_layer_trace* trace, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (h == nullptr || Wt == nullptr || hidden == nullptr || !layer_ok(Wt, M)) return DEC_ERR_INVALID_ARG;
  const dec_layer_weights& L = *Wt;
  if (!L.gamma1 || !L.W_in || !L.W_o || !L.gamma2 || !L.W_r || !L.Wg || !L.Wu || !L.Wd) return DEC_ERR_INVALID_ARG;
  const bool any_s = L.Wg_s || L.Wu_s || L.Wd_s, all_s = L.Wg_s && L.Wu_s && L.Wd_s;
  if (any_s && !all_s) return DEC_ERR_INVALID_ARG;
  for (const void* p : {(const void*)hidden, (const void*)L.gamma1, (const void*)L.W_in, (const void*)L.W_o,
                        (const void*)L.gamma2, (const void*)L.W_r, (const void*)L.Wg, (const void*)L.Wu,
                        (const void*)L.Wd, (const void*)L.Wg_s, (const void*)L.Wu_s, (const void*)L.Wd_s,
                        (const void*)L.prefetch_next, (const void*)ws})
    if (p != nullptr && !al16(p)) return DEC_ERR_INVALID_ARG;
  if (L.prefetch_bytes % 16 != 0 || (L.prefetch_bytes && !L.prefetch_next) || !(L.eps >= 0.f))
    return DEC_ERR_INVALID_ARG;
  if (trace) {
    for (const void* p : {(const void*)trace->h1, (const void*)trace->idx, (const void*)trace->w,
                          (const void*)trace->scores})
      if (p != nullptr && !al16(p)) return DEC_ERR_INVALID_ARG;
  }
  size_t need = 0;
  decode_layer_workspace_size(h, Wt, M, &need);
  if (ws == nullptr || ws_bytes < need) return DEC_ERR_INVALID_ARG;
  Carver c(ws);
  LayerWs w;
  carve_layer(c, h, Wt, M, &w);
  uint16_t* h1 = (trace && trace->h1) ? trace->h1 : w.h1;
  const int H = L.H;

  // Small-matrix input projection (up to four tokens): the first RMSNorm runs
  // inside it (same arithmetic, one launch fewer).
  const bool fuse_norm1 = M <= 4 && choose_variant(h, M, L.N_in, H) == DEC_VARIANT_SMALL_M;
  if (!fuse_norm1) {
    LaunchScope scope(h, "rmsnorm1", s);
    if (launch_rmsnorm(h, hidden, L.gamma1, w.a, M, H, L.eps, s) != cudaSuccess) return DEC_ERR_CUDA;
  }
  EngineRegion dense = w.ml.moe.r0;
  dec_status st = fuse_norm1 ? linear_impl(h, hidden, H, L.W_in, nullptr, w.yin, M, L.N_in, H, dense, s, "in_proj",
                                           L.gamma1, L.eps)
                             : linear_impl(h, w.a, H, L.W_in, nullptr, w.yin, M, L.N_in, H, dense, s, "in_proj");
  if (st != DEC_OK) return st;
  st = linear_impl(h, w.yin, L.N_in, L.W_o, hidden, h1, M, H, L.K_out, dense, s, "out_proj");
  if (st != DEC_OK) return st;
  // The MoE block, pre-norm with its own residual: hidden = h1 + MoE(RMSNorm(h1)).
  MoeLayerArgs A;
  A.x = h1;
  A.gamma = L.gamma2;
  A.eps = L.eps;
  A.Wr = L.W_r;
  A.M = M;
  A.k = L.k;
  A.E = L.E;
  A.H = H;
  A.I = L.I;
  A.Wg = L.Wg;
  A.Wu = L.Wu;
  A.Wd = L.Wd;
  A.Wg_s = L.Wg_s;
  A.Wu_s = L.Wu_s;
  A.Wd_s = L.Wd_s;
  A.residual = h1;
  A.out = hidden;
  A.idx = (trace && trace->idx) ? trace->idx : w.ml.idx;
  A.w = (trace && trace->w) ? trace->w : w.ml.w;
  A.scores = trace ? trace->scores : nullptr;
  A.pf = L.prefetch_next;
  A.pf_bytes = L.prefetch_next != nullptr ? L.prefetch_bytes : 0;
  return moe_layer_impl(h, A, w.ml, s);
}

dec_status moe_layer_workspace_size(const dec_handle* h, const dec_moe_weights* Wt, int M, size_t* bytes) {
  if (h == nullptr || Wt == nullptr || bytes == nullptr || !moe_shape_ok(M, Wt->k, Wt->E, Wt->H, Wt->I))
    return DEC_ERR_INVALID_ARG;
  Carver c(nullptr);
  MoeLayerWs w;
  carve_moe_layer_head(c, Wt->E, Wt->H, Wt->I, 0, &w);
  carve_moe_layer_data(c, h, M, Wt->k, Wt->E, Wt->H, Wt->I, &w);
  *bytes = c.used;
  return DEC_OK;
}

dec_status moe_layer(dec_handle* h, const dec_moe_weights* Wt, const dec_bf16* x, const dec_bf16* residual,
                     dec_bf16* out, int M, int32_t* idx, float* w, float* scores, void* ws, size_t ws_bytes,
                     cudaStream_t s) {
  if (h == nullptr || Wt == nullptr || x == nullptr || out == nullptr) return DEC_ERR_INVALID_ARG;
  const dec_moe_weights& L = *Wt;
  if (!moe_shape_ok(M, L.k, L.E, L.H, L.I) || !L.W_r || !L.Wg || !L.Wu || !L.Wd || !(L.eps >= 0.f))
    return DEC_ERR_INVALID_ARG;
  const bool any_s = L.Wg_s || L.Wu_s || L.Wd_s, all_s = L.Wg_s && L.Wu_s && L.Wd_s;
  if (any_s && !all_s) return DEC_ERR_INVALID_ARG;
  for (const void* p : {(const void*)x, (const void*)residual, (const void*)out, (const void*)L.gamma,
                        (const void*)L.W_r, (const void*)L.Wg, (const void*)L.Wu, (const void*)L.Wd,
                        (const void*)L.Wg_s, (const void*)L.Wu_s, (const void*)L.Wd_s, (const void*)idx,
                        (const void*)w, (const void*)scores, (const void*)ws})
    if (p != nullptr && !al16(p)) return DEC_ERR_INVALID_ARG;
  if (out == x) return DEC_ERR_INVALID_ARG;
  size_t need = 0;
  moe_layer_workspace_size(h, Wt, M, &need);
  if (ws == nullptr || ws_bytes < need) return DEC_ERR_INVALID_ARG;
  Carver c(ws);
  MoeLayerWs mw;
  carve_moe_layer_head(c, L.E, L.H, L.I, 0, &mw);
  carve_moe_layer_data(c, h, M, L.k, L.E, L.H, L.I, &mw);
  MoeLayerArgs A;
  A.x = x;
  A.gamma = L.gamma;
  A.eps = L.eps;
  A.Wr = L.W_r;
  A.M = M;
  A.k = L.k;
  A.E = L.E;
  A.H = L.H;
  A.I = L.I;
  A.Wg = L.Wg;
  A.Wu = L.Wu;
  A.Wd = L.Wd;
  A.Wg_s = L.Wg_s;
  A.Wu_s = L.Wu_s;
  A.Wd_s = L.Wd_s;
  A.residual = residual;
  A.out = out;
  A.idx = idx != nullptr ? idx : mw.idx;
  A.w = w != nullptr ? w : mw.w;
  A.scores = scores;
  return moe_layer_impl(h, A, mw, s);
}

dec_status dec_prefetch_l2(dec_handle* h, const void* ptr, size_t bytes, cudaStream_t stream) {
  if (h == nullptr || (ptr == nullptr && bytes) || !al16(ptr) || bytes % 16 != 0) return DEC_ERR_INVALID_ARG;
  LaunchScope scope(h, "prefetch", stream);
  return launch_prefetch(h, ptr, bytes, 16, stream) == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_set_profiling(dec_handle* h, int enable) {
  if (h == nullptr) return DEC_ERR_INVALID_ARG;
  h->profiling = enable ? 1 : 0;
  return DEC_OK;
}

dec_status dec_profile_read(dec_handle* h, dec_kernel_time* out, int capacity, int* count) {
  if (h == nullptr || count == nullptr || capacity < 0 || (capacity > 0 && out == nullptr)) return DEC_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return DEC_ERR_CUDA;
  int n = 0;
  for (const auto& r : h->prof) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) ms = 0.f;
    int i = 0;
    while (i < n && std::strncmp(out[i].name, r.tag, sizeof(out[i].name)) != 0) ++i;
    if (i == n) {
      if (n >= capacity) continue;
      std::memset(&out[n], 0, sizeof(out[n]));
      std::strncpy(out[n].name, r.tag, sizeof(out[n].name) - 1);
      ++n;
    }
    out[i].launches += 1;
    out[i].total_ms += ms;
  }
  for (const auto& r : h->prof) {
    h->event_pool.push_back(r.a);
    h->event_pool.push_back(r.b);
  }
  h->prof.clear();
  *count = n;
  return DEC_OK;
}

uint64_t dec_launch_count(const dec_handle* h) { return h ? h->launches : 0; }

// ---------------------------------------------------------------- test hooks
dec_status dec_test_wait_timeout(dec_handle* h, cudaStream_t stream) {
  if (h == nullptr) return DEC_ERR_INVALID_ARG;
  LaunchScope scope(h, "test_wait_probe", stream);
  return launch_wait_timeout_probe(h, stream) == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_test_routing_wait_timeout(dec_handle* h, int tokens, cudaStream_t stream) {
  if (h == nullptr || (tokens != 1 && tokens != 2)) return DEC_ERR_INVALID_ARG;
  const int H = 256, E = 16, k = 4, I = 64, M = tokens;
  // one zeroed allocation carved into every buffer of the launch (16-byte aligned pieces)
  const size_t n_bank = (size_t)E * I * H, n_sh = (size_t)I * H;
  size_t off = 0;
  auto piece = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  const size_t o_h1 = piece((size_t)M * H * 2), o_g = piece((size_t)H * 2), o_wr = piece((size_t)E * H * 4),
               o_parts = piece((size_t)M * E * 4), o_ctr = piece(8 * 4), o_idx = piece((size_t)M * k * 4),
               o_w = piece((size_t)M * k * 4), o_sc = piece((size_t)M * E * 4),
               o_tab = piece((size_t)TableLayout(E, M * k).words() * 4), o_gs = piece(n_sh * 2),
               o_us = piece(n_sh * 2), o_hs = piece((size_t)M * I * 2), o_gb = piece(n_bank * 2),
               o_ub = piece(n_bank * 2), o_hb = piece((size_t)M * k * I * 2);
  char* base = nullptr;
  if (cudaMalloc(&base, off) != cudaSuccess) return DEC_ERR_CUDA;
  dec_status st = DEC_OK;
  const int past = 1 << 30;  // the hand-off count starts past any grid size
  if (cudaMemsetAsync(base, 0, off, stream) != cudaSuccess ||
      cudaMemcpyAsync(base + o_ctr, &past, sizeof(int), cudaMemcpyHostToDevice, stream) != cudaSuccess) {
    st = DEC_ERR_CUDA;
  } else {
    LaunchScope scope(h, "test_routing_wait", stream);
    const uint16_t* h1 = reinterpret_cast<const uint16_t*>(base + o_h1);
    const uint16_t* g = reinterpret_cast<const uint16_t*>(base + o_g);
    const float* wr = reinterpret_cast<const float*>(base + o_wr);
    float* parts = reinterpret_cast<float*>(base + o_parts);
    int* ctr = reinterpret_cast<int*>(base + o_ctr);
    int32_t* idx = reinterpret_cast<int32_t*>(base + o_idx);
    float* w = reinterpret_cast<float*>(base + o_w);
    float* sc = reinterpret_cast<float*>(base + o_sc);
    int* tab = reinterpret_cast<int*>(base + o_tab);
    const uint16_t* gs = reinterpret_cast<const uint16_t*>(base + o_gs);
    const uint16_t* us = reinterpret_cast<const uint16_t*>(base + o_us);
    uint16_t* hs = reinterpret_cast<uint16_t*>(base + o_hs);
    const uint16_t* gb = reinterpret_cast<const uint16_t*>(base + o_gb);
    const uint16_t* ub = reinterpret_cast<const uint16_t*>(base + o_ub);
    uint16_t* hb = reinterpret_cast<uint16_t*>(base + o_hb);
    const cudaError_t e =
        tokens == 1 ? launch_moe_front(h, h1, g, 1e-6f, wr, H, E, k, parts, ctr, idx, w, sc, tab, gs, us, I, hs, gb, ub,
                                       hb, stream)
                    : launch_moe_front_multi(h, M, h1, g, 1e-6f, wr, H, E, k, parts, ctr, idx, w, sc, tab, gs, us, I,
                                             hs, gb, ub, hb, stream);
    if (e != cudaSuccess) st = DEC_ERR_CUDA;
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) st = DEC_ERR_CUDA;
  cudaFree(base);
  return st;
}

dec_status dec_test_occupy_sms(dec_handle* h, int ctas, uint64_t hold_ns, cudaStream_t stream) {
  if (h == nullptr || ctas < 1 || ctas > h->sms || hold_ns > 2000000000ull) return DEC_ERR_INVALID_ARG;
  LaunchScope scope(h, "test_occupy", stream);
  return launch_occupy(h, ctas, hold_ns, stream) == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_test_delayed_copy(dec_handle* h, void* dst, const void* src, size_t bytes, uint64_t delay_ns,
                                 cudaStream_t stream) {
  if (h == nullptr || dst == nullptr || src == nullptr || !al16(dst) || !al16(src) || bytes % 16 != 0 ||
      delay_ns > 1000000000ull)
    return DEC_ERR_INVALID_ARG;
  LaunchScope scope(h, "test_delayed_copy", stream);
  return launch_delayed_copy(h, dst, src, bytes, delay_ns, stream) == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

}  // extern "C"
