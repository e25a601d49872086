// Internal interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <utility>
#include <vector>

#include "../../include/moe_decode.h"

struct dec_handle {
  int device = 0;
  int sms = 0;
  cudaStream_t side = nullptr;      // shared expert
  cudaStream_t pf = nullptr;        // L2 prefetch
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_pf_fork = nullptr, ev_pf_join = nullptr;
  int* d_err = nullptr;             // device error word
  uint64_t wait_ns = 500ull * 1000 * 1000;
  int pdl = 1;
  int force_variant = 0;
  int last_variant = 0;
  int last_expert_variant = 0;      // kernel family of the most recent expert launches
  int shared_ctas = 0;              // CTAs for the shared expert's kernels (0 = default)
  int moe_front = 1;                // one to a few tokens: the MoE front launches (0: test hook, the fallback path)
  int engine_finish = 0;            // split-K split-tile finish (test hook: 1, 2 force the fallback paths)
  int l2_ahead = 49152;             // small-matrix kernels: weight bytes per CTA requested into L2 ahead
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  // measurement
  uint64_t launches = 0;
  int profiling = 0;
  struct ProfRec {
    const char* tag;
    cudaEvent_t a, b;
  };
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> event_pool;
};

namespace dec {

enum EpiKind { EPI_LINEAR = 0, EPI_SWIGLU = 1, EPI_F32 = 2 };

constexpr int kTileN = 128;   // weight rows per tile (UMMA M)
constexpr int kBlockK = 64;   // reduction elements per k-block (one 128-byte swizzle row)
constexpr int kMaxCols = 64;  // tokens per problem (UMMA N up to 64)
constexpr int kEngineThreads = 192;

// Bytes of one engine workspace region (split-K partials + per-tile counters).
size_t engine_ws_bytes(int grid, int nacc, long long max_tiles);
int engine_grid(const dec_handle* h);

// Layout of the routing table written by the route-table kernel (int32 words).
struct TableLayout {
  int E, n;  // experts, entries (M * k)
  __host__ __device__ TableLayout(int E_, int n_) : E(E_), n(n_) {}
  __host__ __device__ int U() const { return 0; }
  __host__ __device__ int expert() const { return 1; }
  __host__ __device__ int offset() const { return 1 + E; }
  __host__ __device__ int count() const { return 1 + 2 * E; }
  __host__ __device__ int slot_token() const { return 1 + 3 * E; }
  __host__ __device__ int entry_slot() const { return 1 + 3 * E + n; }
  __host__ __device__ int words() const { return 1 + 3 * E + 2 * n; }
};

struct EngineLaunch {
  int epi = EPI_LINEAR;
  const uint16_t* A = nullptr;   // weights [a_rows][K]
  long long a_rows = 0;
  const uint16_t* A2 = nullptr;  // second weight bank for EPI_SWIGLU (up), same shape
  const uint16_t* B = nullptr;   // activations [b_rows][K], row stride ldb elements
  long long b_rows = 0, ldb = 0;
  int K = 0;
  int N = 0;                     // weight rows per problem
  long long a_rows_per_prob = 0; // row distance between problems in A (0 for one problem)
  int count = 0;                 // tokens (dense mode); the batch, bounding any expert's tokens (grouped)
  const int* table = nullptr;    // routing table (grouped mode) or null (dense mode, one problem)
  int E = 0;                     // table layout
  int n_entries = 0;
  void* out = nullptr;
  long long ldo = 0;
  const uint16_t* res = nullptr;
  long long ldr = 0;
  float* partials = nullptr;
  int* counters = nullptr;
  int grid = 0;                  // CTAs; 0 = all SMs
};

cudaError_t launch_engine(dec_handle* h, const EngineLaunch& L, cudaStream_t s);

// gamma: normalise the input rows first (RMSNorm with eps), fused.
cudaError_t launch_gemv(dec_handle* h, const uint16_t* x, long long ldx, const uint16_t* W, const uint16_t* res,
                        long long ldr, uint16_t* y, long long ldy, int M, int N, int K, cudaStream_t s,
                        const uint16_t* gamma = nullptr, float eps = 0.f);
bool gemv_supported(int M, int K);

// Small-matrix expert kernels for one token (gemv_moe.cu): gate/up with the
// SwiGLU epilogue (swiglu) or down with fp32 output; problems from the routing
// table, or one dense expert when table is null.
// A dense expert processed as problem 0 of the same launch (the shared
// expert at batch 1): its weights, its activation row and its output row.
// The shared expert as the leading dense problem(s) of a grouped launch: n
// activation rows x + t * ldx, outputs out + t * ldo.
struct GemvMoeShared {
  const uint16_t* A;
  const uint16_t* A2;
  const uint16_t* x;
  void* out;
  int n = 1;
  long long ldx = 0, ldo = 0;
};
cudaError_t launch_gemv_moe(dec_handle* h, bool swiglu, const uint16_t* A, const uint16_t* A2,
                            long long rows_per_prob_bank, int R, int K, const uint16_t* x, long long ldx,
                            const int* table, int E, int n_entries, void* out, long long ldo, int sms,
                            cudaStream_t s, const GemvMoeShared* shared = nullptr, int nprob_known = 0,
                            bool late_trigger = false, bool x_by_token = false);
bool gemv_moe_supported(int K);
// One token: down projection of the k routed (+ shared) experts fused with the
// weighted combine and the residual, written straight to out (bf16 [H]).
bool gemv_down_combine_supported(int k, int I);
// Two tokens, k = 8, I <= 2048: down of the 16 entries and the shared expert,
// weighted combine and residual in one kernel (out, res [2][H]).
bool gemv_down_combine2_supported(int k, int I);
cudaError_t launch_gemv_down_combine2(dec_handle* h, const uint16_t* Wd, long long rows_bank, const uint16_t* Wd_s,
                                      int H, int I, const uint16_t* hbuf, const uint16_t* hs, const int* table, int E,
                                      int k, const float* w, const uint16_t* res, uint16_t* out, int sms,
                                      cudaStream_t s, bool routing_ready = false);
cudaError_t launch_gemv_down_combine(dec_handle* h, const uint16_t* Wd, long long rows_bank, const uint16_t* Wd_s,
                                     int H, int I, const uint16_t* hbuf, const uint16_t* hs, const int* table, int E,
                                     int k, const float* w, const uint16_t* res, uint16_t* out, int sms,
                                     cudaStream_t s, bool routing_ready = false);

cudaError_t launch_rmsnorm(dec_handle* h, const uint16_t* x, const uint16_t* gamma, uint16_t* y, int M, int H,
                           float eps, cudaStream_t s);

int router_ksplit(int H);
cudaError_t launch_router(dec_handle* h, const uint16_t* x, const float* Wr, int M, int H, int E, float* parts,
                          cudaStream_t s);
cudaError_t launch_topk(dec_handle* h, const float* parts, int ks, int M, int E, int k, int32_t* idx, float* w,
                        float* scores, cudaStream_t s);
// One token: RMSNorm (if gamma) + router logits + top-k + routing table; counter zero on entry and on return.
cudaError_t launch_router_select(dec_handle* h, const uint16_t* x, const uint16_t* gamma, float eps, const float* Wr,
                                 int H, int E, int k, uint16_t* xn, float* parts, int* counter, int32_t* idx,
                                 float* w, float* scores, int* table, cudaStream_t s);
// One token: the routing table with entry j as problem j on slot j (expert idx[j]).
// One token: launch_router_select's work plus the shared expert's gate/up
// (h_s = bf16(silu(W_g,s b) * (W_u,s b))) streamed by the same CTAs; ctr: 3 ints, zero on entry and on return.
// M = 2..4 tokens: the same with one routing-table problem per (token, expert) entry (U = M k,
// slot p = t k + j), h_s [M][I] and xn [M][H]; without a shared expert (Wg_s null) routing only.
bool route_shared_supported(const dec_handle* h, int M, int H, int E, int k);
// One token: routing + shared gate/up + the k routed experts' gate/up in one
// launch (hbuf [k][I], slot j = entry j); counters ctr[5] zero between launches.
// pf / pf_bytes (16-byte aligned, multiple of 16): pulled into L2 by the CTAs
// while they wait for the routing.
cudaError_t launch_moe_front(dec_handle* h, const uint16_t* h1, const uint16_t* gamma, float eps, const float* Wr,
                             int H, int E, int k, float* parts, int* ctr, int32_t* idx, float* w, float* scores,
                             int* table, const uint16_t* Wg_s, const uint16_t* Wu_s, int I, uint16_t* hs,
                             const uint16_t* Wg, const uint16_t* Wu, uint16_t* hbuf, cudaStream_t s,
                             const void* pf = nullptr, size_t pf_bytes = 0);
// Two to four tokens: routing + shared gate/up + the M k entries' gate/up in
// one launch (hbuf [M k][I], slot p = entry p); counters ctr[5] zero between launches.
cudaError_t launch_moe_front_multi(dec_handle* h, int M, const uint16_t* h1, const uint16_t* gamma, float eps,
                                   const float* Wr, int H, int E, int k, float* parts, int* ctr, int32_t* idx, float* w,
                                   float* scores, int* table, const uint16_t* Wg_s, const uint16_t* Wu_s, int I,
                                   uint16_t* hs, const uint16_t* Wg, const uint16_t* Wu, uint16_t* hbuf,
                                   cudaStream_t s, const void* pf = nullptr, size_t pf_bytes = 0);
cudaError_t launch_route_shared(dec_handle* h, int M, const uint16_t* h1, const uint16_t* gamma, float eps,
                                const float* Wr, int H, int E, int k, uint16_t* xn, float* parts, int* ctr,
                                int32_t* idx, float* w, float* scores, int* table, const uint16_t* Wg_s,
                                const uint16_t* Wu_s, int I, uint16_t* hs, cudaStream_t s);
cudaError_t launch_one_token_table(dec_handle* h, const int32_t* idx, int E, int k, int* table, cudaStream_t s);
cudaError_t launch_route_table(dec_handle* h, const int32_t* idx, int M, int k, int E, const uint16_t* x, int H,
                               int* table, uint16_t* xs, cudaStream_t s);
cudaError_t launch_combine(dec_handle* h, const float* y, const int* table, const float* w, int M, int k, int E,
                           const float* ys, const uint16_t* res, uint16_t* out, int H, cudaStream_t s);
cudaError_t launch_prefetch(dec_handle* h, const void* p, size_t bytes, int ctas, cudaStream_t s);
cudaError_t launch_wait_timeout_probe(dec_handle* h, cudaStream_t s);
cudaError_t launch_occupy(dec_handle* h, int ctas, uint64_t hold_ns, cudaStream_t s);
cudaError_t launch_delayed_copy(dec_handle* h, void* dst, const void* src, size_t bytes, uint64_t delay_ns,
                                cudaStream_t s);

inline cudaEvent_t pool_event(dec_handle* h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Counts every kernel launch; when profiling, brackets it with events on its stream.
struct LaunchScope {
  dec_handle* h;
  cudaStream_t s;
  int rec = -1;
  LaunchScope(dec_handle* h_, const char* tag, cudaStream_t s_) : h(h_), s(s_) {
    h->launches++;
    if (h->profiling) {
      dec_handle::ProfRec r{tag, pool_event(h), pool_event(h)};
      if (r.a && r.b && cudaEventRecord(r.a, s) == cudaSuccess) {
        h->prof.push_back(r);
        rec = (int)h->prof.size() - 1;
      }
    }
  }
  ~LaunchScope() {
    if (rec >= 0) cudaEventRecord(h->prof[rec].b, s);
  }
};

// Launch with the handle's programmatic-dependent-launch setting.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const dec_handle* h, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = h->pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace dec
