// Small-matrix expert kernels for one token: the routed and shared SwiGLU
// experts at batch 1.
//
// Kimi K3 article, Part 1 §1 "Ajustar las formas" (small-matrix kernels at
// small batch) applied to Part 1 §3's experts. With one token every selected
// expert sees one activation row, so each expert matrix is a pure weight
// stream. The work unit is one output row of one expert: for the gate/up
// kernel the matching rows of W_g and W_u (the SwiGLU needs both), for the
// down kernel one row of W_d. All units of all selected experts form one
// sequence that is cut into one contiguous, equal range per CTA (two
// 256-thread CTAs per SM), so every SM streams the same bytes whatever the
// routing. Thread t owns the 16-byte column vectors t, t+256, ... of every row
// and keeps the expert's activation vectors in registers (reloaded when its
// range crosses into the next expert); weights stream with 128-bit,
// L1-bypassing, evict-first loads, the next step's issued before the current
// step's FMAs. Partial sums are reduced by warp shuffles, then across the
// eight warps in shared memory, in a fixed order.
//
// Problems come from the device routing table (routed experts) or are one
// dense expert (the shared expert, whose first rows are loaded before the
// dependency wait).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dec {

constexpr int kGmThreads = 256;

struct GemvMoeParams {
  // Optional extra problem 0: a dense expert (the shared expert) with its own
  // weights, activation row and output row; routed problems follow it.
  const uint16_t* sA;
  const uint16_t* sA2;
  const uint16_t* sx;
  void* sout;
  const uint16_t* A;   // first weight matrix (gate or down), row-major [rows][K]
  const uint16_t* A2;  // up matrix (SwiGLU) or unused
  long long rows_per_prob_bank;  // row distance between experts in the bank (0: one dense problem)
  int R;               // output rows per problem (I for gate/up, H for down)
  int K;
  const uint16_t* x;   // activation rows, [slots][K]
  long long ldx;
  const int* table;    // routing table, or null for one dense problem on slot 0
  int E, n_entries;
  void* out;           // SwiGLU: bf16 [slots][ldo]; down: fp32 [slots][ldo]
  long long ldo;
};

template <bool SWIGLU, int VPT>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_moe_kernel(const GemvMoeParams P) {
  constexpr int NR = SWIGLU ? 2 : 1;                            // weight rows per unit
  constexpr int RB = (8 / (VPT * NR)) > 0 ? (8 / (VPT * NR)) : 1;  // units per step
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K8 = P.K >> 3;
  __shared__ float red[2][kGmThreads / 32][RB * NR];
  const uint64_t pol = policy_evict_first();
  pdl_trigger();

  // Problem bookkeeping (the routed table is read only after the dependency wait).
  const TableLayout L(P.E, P.n_entries);
  const int ns = P.sA != nullptr ? 1 : 0;  // leading dense problem
  auto nprob = [&]() -> long long { return (P.table ? ld_act_s32(P.table + L.U()) : 1) + ns; };
  // Problem p: -1 marks the leading dense problem; otherwise the expert id.
  auto expert_of = [&](int p) -> long long {
    if (p < ns) return -1;
    return P.table ? ld_act_s32(P.table + L.expert() + (p - ns)) : 0;
  };
  auto slot_of = [&](int p) -> long long {
    if (p < ns) return 0;
    return P.table ? ld_act_s32(P.table + L.offset() + (p - ns)) : 0;
  };

  // Weight rows of one step: nu units starting at row r of the matrices at a0 / a1.
  uint4 wa[RB][NR][VPT];
  auto load_units = [&](uint4(&w)[RB][NR][VPT], const uint16_t* a0, const uint16_t* a1, int r, int nu) {
#pragma unroll
    for (int u = 0; u < RB; ++u)
#pragma unroll
      for (int a = 0; a < NR; ++a)
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = t + kGmThreads * i;
          if (u < nu && v < K8)
            w[u][a][i] = ld_stream((a == 0 ? a0 : a1) + (size_t)(r + u) * P.K + (size_t)v * 8, pol);
          else
            w[u][a][i] = make_uint4(0, 0, 0, 0);
        }
  };
  // Weight matrices of problem p (e < 0: the leading dense problem).
  auto mat0 = [&](long long e) { return e < 0 ? P.sA : P.A + e * P.rows_per_prob_bank * P.K; };
  auto mat1 = [&](long long e) { return e < 0 ? P.sA2 : P.A2 + e * P.rows_per_prob_bank * P.K; };

  const long long G = gridDim.x, c = blockIdx.x;
  long long q0 = 0, q1 = 0;
  int pre_nu = 0;
  if (P.table == nullptr) {  // dense: the range is known, start the weight stream now
    const long long T = (long long)(1 + ns) * P.R;
    q0 = c * T / G;
    q1 = (c + 1) * T / G;
    const long long e0 = (q0 / P.R < ns) ? -1 : 0;
    pre_nu = (int)min((long long)RB, min(q1, (q0 / P.R + 1) * (long long)P.R) - q0);
    if (pre_nu > 0) load_units(wa, mat0(e0), mat1(e0), (int)(q0 % P.R), pre_nu);
  }
  pdl_wait();
  if (P.table != nullptr) {
    const long long T = nprob() * P.R;
    q0 = c * T / G;
    q1 = (c + 1) * T / G;
  }
  if (q0 >= q1) return;  // no work (no barrier below is reached by any thread of this CTA)

  // Position as (problem, row), advanced incrementally: no division in the loop.
  int p = (int)(q0 / P.R), r = (int)(q0 % P.R);
  long long left = q1 - q0;
  long long e = expert_of(p);
  const uint16_t* A0 = mat0(e);
  const uint16_t* A1 = mat1(e);
  int nu = (int)min((long long)min(RB, P.R - r), left);
  if (pre_nu == 0) load_units(wa, A0, A1, r, nu);

  uint4 xr[VPT];
  long long slot = slot_of(p);
  auto load_x = [&]() {
    const uint16_t* xrow = e < 0 ? P.sx : P.x + slot * P.ldx;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = t + kGmThreads * i;
      xr[i] = (v < K8) ? ld_act16(xrow + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
    }
  };
  load_x();
  int buf = 0;
  while (left > 0) {
    // Next step's position (units never cross a problem boundary: their x differs).
    int pn = p, rn = r + nu;
    long long en = e;
    const uint16_t *N0 = A0, *N1 = A1;
    const long long leftn = left - nu;
    if (rn == P.R) {
      pn = p + 1;
      rn = 0;
      if (leftn > 0) {
        en = expert_of(pn);
        N0 = mat0(en);
        N1 = mat1(en);
      }
    }
    const int nun = (int)min((long long)min(RB, P.R - rn), leftn);
    uint4 wb[RB][NR][VPT];
    if (nun > 0) load_units(wb, N0, N1, rn, nun);  // issued before this step's FMAs

    float acc[RB][NR];
#pragma unroll
    for (int u = 0; u < RB; ++u)
#pragma unroll
      for (int a = 0; a < NR; ++a) {
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) sum = dot8(wa[u][a][i], xr[i], sum);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        acc[u][a] = sum;
      }
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < RB; ++u)
#pragma unroll
        for (int a = 0; a < NR; ++a) red[buf][warp][u * NR + a] = acc[u][a];
    }
    __syncthreads();
    if (t < nu) {
      float g = 0.f, up = 0.f;
#pragma unroll
      for (int w = 0; w < kGmThreads / 32; ++w) {
        g += red[buf][w][t * NR];
        if (SWIGLU) up += red[buf][w][t * NR + 1];
      }
      void* dst = e < 0 ? P.sout : P.out;
      const long long o = (e < 0 ? 0 : slot * P.ldo) + r + t;
      if (SWIGLU)
        reinterpret_cast<uint16_t*>(dst)[o] = f2bf(g / (1.0f + expf(-g)) * up);
      else
        reinterpret_cast<float*>(dst)[o] = g;
    }
    buf ^= 1;
    left = leftn;
    if (pn != p && left > 0) {
      p = pn;
      e = en;
      A0 = N0;
      A1 = N1;
      slot = slot_of(p);
      load_x();
    }
    r = rn;
    nu = nun;
#pragma unroll
    for (int u = 0; u < RB; ++u)
#pragma unroll
      for (int a = 0; a < NR; ++a)
#pragma unroll
        for (int i = 0; i < VPT; ++i) wa[u][a][i] = wb[u][a][i];
  }
}

bool gemv_moe_supported(int K) { return K >= 8 && K % 8 == 0 && K <= 8 * 4 * kGmThreads; }

template <bool SWIGLU>
static cudaError_t launch_mode(dec_handle* h, const GemvMoeParams& P, int grid, cudaStream_t s) {
  const int K8 = P.K / 8;
  const dim3 g(grid), b(kGmThreads);
  if (K8 <= kGmThreads) return launch_k(h, gemv_moe_kernel<SWIGLU, 1>, g, b, 0, s, P);
  if (K8 <= 2 * kGmThreads) return launch_k(h, gemv_moe_kernel<SWIGLU, 2>, g, b, 0, s, P);
  return launch_k(h, gemv_moe_kernel<SWIGLU, 4>, g, b, 0, s, P);
}

cudaError_t launch_gemv_moe(dec_handle* h, bool swiglu, const uint16_t* A, const uint16_t* A2,
                            long long rows_per_prob_bank, int R, int K, const uint16_t* x, long long ldx,
                            const int* table, int E, int n_entries, void* out, long long ldo, int sms,
                            cudaStream_t s, const GemvMoeShared* shared) {
  if (!gemv_moe_supported(K)) return cudaErrorInvalidValue;
  GemvMoeParams P;
  P.sA = shared ? shared->A : nullptr;
  P.sA2 = shared ? (shared->A2 ? shared->A2 : shared->A) : nullptr;
  P.sx = shared ? shared->x : nullptr;
  P.sout = shared ? shared->out : nullptr;
  P.A = A;
  P.A2 = A2 ? A2 : A;
  P.rows_per_prob_bank = rows_per_prob_bank;
  P.R = R;
  P.K = K;
  P.x = x;
  P.ldx = ldx;
  P.table = table;
  P.E = E;
  P.n_entries = n_entries;
  P.out = out;
  P.ldo = ldo;
  const int grid = std::max(1, 2 * sms);
  return swiglu ? launch_mode<true>(h, P, grid, s) : launch_mode<false>(h, P, grid, s);
}

}  // namespace dec
