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
  // Optional leading dense problems 0 .. ns-1: one dense expert (the shared
  // expert) applied to ns activation rows (sx + p * sldx -> sout + p * sldo);
  // the routed problems follow them.
  const uint16_t* sA;
  const uint16_t* sA2;
  const uint16_t* sx;
  void* sout;
  int ns;
  long long sldx, sldo;
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
  int x_by_token;      // routed activation row: the slot's token (x + token * ldx), else the slot's own row
  int nprob_known;     // routed problems if known at launch (one token: k), else 0
  int ahead;           // weight bytes per CTA requested into L2 ahead of the register loads (0: none)
  int late_trigger;    // trigger dependents after the dependency wait (they may then read the routing early)
};

template <bool SWIGLU, int VPT>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_moe_kernel(const GemvMoeParams P) {
  constexpr int NR = SWIGLU ? 2 : 1;                            // weight rows per unit
  constexpr int RB = (8 / (VPT * NR)) > 0 ? (8 / (VPT * NR)) : 1;  // units per step
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K8 = P.K >> 3;
  __shared__ float red[2][kGmThreads / 32][RB * NR];
  const uint64_t pol = policy_evict_first();
  if (!P.late_trigger) pdl_trigger();

  // Problem bookkeeping (the routed table is read only after the dependency wait).
  const TableLayout L(P.E, P.n_entries);
  const int ns = P.sA != nullptr ? P.ns : 0;  // leading dense problems
  auto nprob = [&]() -> long long { return (P.table ? ld_act_s32(P.table + L.U()) : 1) + ns; };
  // Problem p: -1 marks the leading dense problem; otherwise the expert id.
  auto expert_of = [&](int p) -> long long {
    if (p < ns) return -1;
    return P.table ? ld_act_s32(P.table + L.expert() + (p - ns)) : 0;
  };
  // Problem p's row: for a dense problem its index, for a routed one its slot.
  auto slot_of = [&](int p) -> long long {
    if (p < ns) return p;
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
  const int rowb = P.K * (int)sizeof(uint16_t);
  const int ahead_units = P.ahead > 0 ? max(1, P.ahead / (NR * rowb)) : 0;
  // With the problem count known at launch the range is too; a range that
  // starts in a dense problem starts its weight stream now.
  const bool range_known = P.table == nullptr || P.nprob_known > 0;
  if (range_known) {
    const long long T = (long long)((P.table ? P.nprob_known : 1) + ns) * P.R;
    q0 = c * T / G;
    q1 = (c + 1) * T / G;
    const long long p0 = q0 / P.R;
    if (p0 < ns || P.table == nullptr) {
      const long long e0 = p0 < ns ? -1 : 0;
      pre_nu = (int)max(0LL, min((long long)RB, min(q1, (p0 + 1) * (long long)P.R) - q0));
      if (pre_nu > 0) load_units(wa, mat0(e0), mat1(e0), (int)(q0 % P.R), pre_nu);
    }
  }
  pdl_wait();
  if (P.late_trigger) pdl_trigger();
  if (!range_known) {
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
  // the first units past this one, up to `ahead_units`, in the same problem
  if (t == 0 && ahead_units > 0) {
    const long long n = min(min((long long)ahead_units, (long long)(P.R - r - nu)), left - nu);
    if (n > 0) {
      request_l2(A0 + (size_t)(r + nu) * P.K, (size_t)n * rowb);
      if (NR == 2) request_l2(A1 + (size_t)(r + nu) * P.K, (size_t)n * rowb);
    }
  }

  uint4 xr[VPT];
  long long slot = slot_of(p);
  auto load_x = [&]() {
    const long long xr_row = (e >= 0 && P.x_by_token && P.table) ? ld_act_s32(P.table + L.slot_token() + slot) : slot;
    const uint16_t* xrow = e < 0 ? P.sx + slot * P.sldx : P.x + xr_row * P.ldx;
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
    // L2 request for the units `ahead_units` past the next step, when they lie
    // in the same problem and in this CTA's range (no lookup of later
    // problems: the few units after a problem boundary go without).
    if (t == 0 && ahead_units > 0 && nun > 0) {
      const int ra = rn + ahead_units;
      if (ra + nun <= P.R && (long long)ahead_units + nun <= leftn) {
        request_l2(N0 + (size_t)ra * P.K, (size_t)nun * rowb);
        if (NR == 2) request_l2(N1 + (size_t)ra * P.K, (size_t)nun * rowb);
      }
    }

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
      const long long o = slot * (e < 0 ? P.sldo : P.ldo) + r + t;
      if (SWIGLU)
        reinterpret_cast<uint16_t*>(dst)[o] = swiglu_bf16(g, up);
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

// One token, down projection fused with the weighted combine and residual:
//   out[n] = bf16( sum_j w_j (Wd_{e_j}[n] . h_j)  [+ Wd_s[n] . h_s]  [+ res[n]] )
// The unit is one output row n; it reads row n of every selected expert's W_d
// (and of the shared expert's), so no per-expert output is written and no
// combine kernel runs. Thread t owns the 16-byte column vectors t, t+256, ...
// of each row and holds the k (+1) activation rows' matching vectors in
// registers. The combine is linear, so each thread applies the weights to its
// own partial dot products first, a = sum_j w_j d_j (+ d_s), in entry order,
// and the unit needs one warp reduction instead of one per expert; the eight
// warp sums are added in order, then the residual. Weight vectors stream
// through a ring of NP x VPT registers: consuming row n's vector of entry j
// issues row n+1's, so NP x VPT loads stay in flight without a second buffer.
// NP = k (+1 with a shared expert) rows per unit.
template <int NP, int VPT, bool SHARED>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_down_combine_kernel(
    const uint16_t* __restrict__ Wd, long long rows_bank, const uint16_t* __restrict__ Wd_s, int H, int K,
    const uint16_t* hbuf, const uint16_t* hs, const int* table, int E, int k, const float* w, const uint16_t* res,
    uint16_t* out, int routing_ready, int ahead) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K8 = K >> 3;
  __shared__ __align__(16) float red[2][kGmThreads / 32];
  const uint64_t pol = policy_evict_first();
  pdl_trigger();
  const long long G = gridDim.x, c = blockIdx.x;
  const int n0 = (int)(c * H / G), n1 = (int)((c + 1) * H / G);
  if (n0 >= n1) return;  // (before any barrier)
  const TableLayout L(E, k);
  // Per selected row: the W_d row base, the activation row and the combine weight.
  __shared__ const uint16_t* s_rowbase[NP];
  __shared__ const uint16_t* s_xrow[NP];
  __shared__ float s_w[NP];
  auto routing = [&](bool cg) {
    if (t < NP) {
      if (SHARED && t == NP - 1) {
        s_rowbase[t] = Wd_s;
        s_xrow[t] = hs;
        s_w[t] = 1.f;
      } else {
        // token 0, entry t; one token: problem index == slot
        const int slot = cg ? ld_cg_s32(table + L.entry_slot() + t) : ld_act_s32(table + L.entry_slot() + t);
        const long long e = cg ? ld_cg_s32(table + L.expert() + slot) : ld_act_s32(table + L.expert() + slot);
        s_rowbase[t] = Wd + e * rows_bank * K;
        s_xrow[t] = hbuf + (size_t)slot * K;
        s_w[t] = cg ? ld_cg_f32(w + t) : ld_act_f32(w + t);
      }
    }
    __syncthreads();
  };
  uint4 ring[NP][VPT];
  auto load1 = [&](int j, int i, int n) {
    const int v = t + kGmThreads * i;
    return (v < K8) ? ld_stream(s_rowbase[j] + (size_t)n * K + (size_t)v * 8, pol) : make_uint4(0, 0, 0, 0);
  };
  auto load_row = [&](int n) {
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int i = 0; i < VPT; ++i) ring[j][i] = load1(j, i, n);
  };
  // L2 requests: rows [pf, ...) of every selected matrix are not yet
  // requested; thread j < NP requests matrix j's (contiguous) rows.
  const int rowb = K * (int)sizeof(uint16_t);
  const int ahead_rows = ahead > 0 ? max(1, ahead / (NP * rowb)) : 0;
  int pf = n0 + 1;
  auto request = [&](int upto) {
    upto = min(upto, n1);
    if (ahead_rows > 0 && upto > pf) {
      if (t < NP) request_l2(s_rowbase[t] + (size_t)pf * K, (size_t)(upto - pf) * rowb);
      pf = upto;
    }
  };
  // routing_ready: the launch before this one triggered its dependents only
  // after its own dependency wait, so the routing (written two launches back)
  // is complete now; read it at L2 and start the weight stream before the wait.
  if (routing_ready) {
    routing(true);
    load_row(n0);
    request(n0 + 1 + ahead_rows);
  }
  pdl_wait();
  if (!routing_ready) {
    routing(false);
    load_row(n0);
    request(n0 + 1 + ahead_rows);
  }
  uint4 xr[NP][VPT];
#pragma unroll
  for (int j = 0; j < NP; ++j)
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = t + kGmThreads * i;
      xr[j][i] = (v < K8) ? ld_act16(s_xrow[j] + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
    }
  // residual values of this CTA's rows, read once (kept off the per-row path)
  __shared__ float s_res[64];
  for (int q = t; q < n1 - n0 && q < 64; q += kGmThreads) s_res[q] = res ? bf2f(ld_act_u16(res + n0 + q)) : 0.f;
  __syncthreads();
  int buf = 0;
  for (int n = n0; n < n1; ++n) {
    const bool more = n + 1 < n1;
    request(n + 2 + ahead_rows);
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const uint4 wv = ring[j][i];
        if (more) ring[j][i] = load1(j, i, n + 1);
        d = dot8(wv, xr[j][i], d);
      }
      if (SHARED && j == NP - 1)
        a += d;
      else
        a = fmaf(s_w[j], d, a);  // (a broadcast shared-memory read: registers hold the weight ring)
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) red[buf][warp] = a;
    __syncthreads();
    if (t == 0) {
      const float4 p0 = *reinterpret_cast<const float4*>(&red[buf][0]);
      const float4 p1 = *reinterpret_cast<const float4*>(&red[buf][4]);
      float y = ((((((p0.x + p0.y) + p0.z) + p0.w) + p1.x) + p1.y) + p1.z) + p1.w;
      if (res != nullptr) y += (n - n0 < 64) ? s_res[n - n0] : bf2f(ld_act_u16(res + n));
      out[n] = f2bf(y);
    }
    buf ^= 1;
  }
}

// Narrow rows (K = I <= 256, K / 8 <= TPR in {16, 32}): as the kernel above,
// but a group of TPR threads owns a whole output row (one 16-byte vector of
// each of the NP matrices' row per thread), so a CTA works on 256 / TPR rows
// at a time and a row is reduced by shuffles alone, with no barrier in the
// loop. Groups take the CTA's rows interleaved (group g: n0 + g, n0 + g + NG,
// ...); the next row's NP vectors are loaded while this one's are consumed.
template <int NP, int TPR, bool SHARED>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_down_combine_narrow_kernel(
    const uint16_t* __restrict__ Wd, long long rows_bank, const uint16_t* __restrict__ Wd_s, int H, int K,
    const uint16_t* hbuf, const uint16_t* hs, const int* table, int E, int k, const float* w, const uint16_t* res,
    uint16_t* out, int routing_ready, int ahead) {
  constexpr int NG = kGmThreads / TPR;
  const int t = threadIdx.x, g = t / TPR, j = t % TPR;
  const int K8 = K >> 3;
  const uint64_t pol = policy_evict_first();
  pdl_trigger();
  const long long G = gridDim.x, c = blockIdx.x;
  const int n0 = (int)(c * H / G), n1 = (int)((c + 1) * H / G);
  if (n0 >= n1) return;  // (before any barrier)
  const TableLayout L(E, k);
  __shared__ const uint16_t* s_rowbase[NP];
  __shared__ const uint16_t* s_xrow[NP];
  __shared__ float s_w[NP];
  auto routing = [&](bool cg) {
    if (t < NP) {
      if (SHARED && t == NP - 1) {
        s_rowbase[t] = Wd_s;
        s_xrow[t] = hs;
        s_w[t] = 1.f;
      } else {
        const int slot = cg ? ld_cg_s32(table + L.entry_slot() + t) : ld_act_s32(table + L.entry_slot() + t);
        const long long e = cg ? ld_cg_s32(table + L.expert() + slot) : ld_act_s32(table + L.expert() + slot);
        s_rowbase[t] = Wd + e * rows_bank * K;
        s_xrow[t] = hbuf + (size_t)slot * K;
        s_w[t] = cg ? ld_cg_f32(w + t) : ld_act_f32(w + t);
      }
    }
    __syncthreads();
  };
  // Loads are unconditional at clamped, in-range addresses (a lane past the
  // row's vectors reads the row's last one and meets a zero activation; a
  // group past the CTA's rows reads its last row and writes nothing), so the
  // register ring holds no second copies.
  const int jj = min(j, K8 - 1);
  uint4 ring[NP];
  auto load_row = [&](int n) {
    const int nn = min(n, n1 - 1);
#pragma unroll
    for (int q = 0; q < NP; ++q) ring[q] = ld_stream(s_rowbase[q] + (size_t)nn * K + (size_t)jj * 8, pol);
  };
  const int rowb = K * (int)sizeof(uint16_t);
  const int ahead_rows = ahead > 0 ? max(1, ahead / (NP * rowb)) : 0;
  int pf = n0 + NG;
  auto request = [&](int upto) {
    upto = min(upto, n1);
    if (ahead_rows > 0 && upto > pf) {
      if (t < NP) request_l2(s_rowbase[t] + (size_t)pf * K, (size_t)(upto - pf) * rowb);
      pf = upto;
    }
  };
  if (routing_ready) {
    routing(true);
    load_row(n0 + g);
    request(n0 + NG + ahead_rows);
  }
  pdl_wait();
  if (!routing_ready) {
    routing(false);
    load_row(n0 + g);
    request(n0 + NG + ahead_rows);
  }
  uint4 xr[NP];
#pragma unroll
  for (int q = 0; q < NP; ++q) xr[q] = j < K8 ? ld_act16(s_xrow[q] + (size_t)j * 8) : make_uint4(0, 0, 0, 0);
  // The loop runs the same number of steps in every group (a group past the
  // CTA's rows computes on its clamped last row and writes nothing), so the
  // whole-warp shuffles below never meet diverged lanes.
  for (int nb = n0; nb < n1; nb += NG) {
    const int n = nb + g;
    if (g == 0) request(n + 2 * NG + ahead_rows);  // (only threads t < NP issue)
    float a = 0.f;
    const int nn = min(n + NG, n1 - 1);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const uint4 wv = ring[q];
      ring[q] = ld_stream(s_rowbase[q] + (size_t)nn * K + (size_t)jj * 8, pol);
      const float d = dot8(wv, xr[q], 0.f);
      if (SHARED && q == NP - 1)
        a += d;
      else
        a = fmaf(s_w[q], d, a);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (j == 0 && n < n1) {
      if (res != nullptr) a += bf2f(ld_act_u16(res + n));
      out[n] = f2bf(a);
    }
  }
}

// Rows of up to 2048 elements (one vector per thread per row, activations in registers).
// Two tokens: the down projection of the 2 k entries and of the shared
// expert, the weighted combine and the residual in one kernel (the one-token
// kernel above, extended). Output row n of token m:
//   out[m][n] = res[m][n] + sum_j w_j (W_d[e_j] h_j)[n] + (W_d_s h_s[m])[n]
// over token m's entries j (slots m k .. m k + k - 1). Unit: output row n of
// every selected matrix (row n of the shared W_d is read once and applied to
// both tokens' h_s rows). Thread t owns column vector t of every row; its
// activation vectors (one per entry, two for the shared expert) sit in
// shared memory (each thread reads only its own), which leaves the
// registers to the ring of weight vectors.
template <int NE, bool SHARED>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_down_combine2_kernel(
    const uint16_t* __restrict__ Wd, long long rows_bank, const uint16_t* __restrict__ Wd_s, int H, int K,
    const uint16_t* hbuf, const uint16_t* hs, const int* table, int E, int k, const float* w, const uint16_t* res,
    uint16_t* out, int routing_ready, int ahead) {
  constexpr int NP = SHARED ? NE + 1 : NE;  // matrices per unit
  constexpr int NX = SHARED ? NE + 2 : NE;  // activation vectors per thread
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K8 = K >> 3;
  __shared__ __align__(16) float red[2][kGmThreads / 32][2];
  extern __shared__ __align__(16) uint4 sxv[];  // [NX][kGmThreads]
  const uint64_t pol = policy_evict_first();
  pdl_trigger();
  const long long G = gridDim.x, c = blockIdx.x;
  const int n0 = (int)(c * H / G), n1 = (int)((c + 1) * H / G);
  if (n0 >= n1) return;  // (before any barrier)
  const TableLayout L(E, NE);
  __shared__ const uint16_t* s_rowbase[NP];
  __shared__ float s_w[NE];
  auto routing = [&](bool cg) {
    if (t < NP) {
      if (SHARED && t == NE) {
        s_rowbase[t] = Wd_s;
      } else {
        // entry t on slot t (one problem per entry)
        const long long e = cg ? ld_cg_s32(table + L.expert() + t) : ld_act_s32(table + L.expert() + t);
        s_rowbase[t] = Wd + e * rows_bank * K;
        s_w[t] = cg ? ld_cg_f32(w + t) : ld_act_f32(w + t);
      }
    }
    __syncthreads();
  };
  uint4 ring[NP];
  auto load1 = [&](int j, int n) {
    return t < K8 ? ld_stream(s_rowbase[j] + (size_t)n * K + (size_t)t * 8, pol) : make_uint4(0, 0, 0, 0);
  };
  const int rowb = K * (int)sizeof(uint16_t);
  const int ahead_rows = ahead > 0 ? max(1, ahead / (NP * rowb)) : 0;
  int pf = n0 + 1;
  auto request = [&](int upto) {
    upto = min(upto, n1);
    if (ahead_rows > 0 && upto > pf) {
      if (t < NP) request_l2(s_rowbase[t] + (size_t)pf * K, (size_t)(upto - pf) * rowb);
      pf = upto;
    }
  };
  if (routing_ready) {
    routing(true);
#pragma unroll
    for (int j = 0; j < NP; ++j) ring[j] = load1(j, n0);
    request(n0 + 1 + ahead_rows);
  }
  pdl_wait();
  if (!routing_ready) {
    routing(false);
#pragma unroll
    for (int j = 0; j < NP; ++j) ring[j] = load1(j, n0);
    request(n0 + 1 + ahead_rows);
  }
  // this thread's activation vectors: the entries' rows, then the two shared rows
#pragma unroll
  for (int j = 0; j < NX; ++j) {
    const uint16_t* row = j < NE ? hbuf + (size_t)j * K : hs + (size_t)(j - NE) * K;
    sxv[j * kGmThreads + t] = t < K8 ? ld_act16(row + (size_t)t * 8) : make_uint4(0, 0, 0, 0);
  }
  __shared__ float s_res[2][64];
  for (int q = t; q < 2 * 64; q += kGmThreads) {
    const int m = q / 64, r = q % 64;
    if (r < n1 - n0) s_res[m][r] = res ? bf2f(ld_act_u16(res + (size_t)m * H + n0 + r)) : 0.f;
  }
  __syncthreads();
  const int kk = NE / 2;  // entries per token
  int buf = 0;
  for (int n = n0; n < n1; ++n) {
    const bool more = n + 1 < n1;
    request(n + 2 + ahead_rows);
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int j = 0; j < NE; ++j) {
      const uint4 wv = ring[j];
      if (more) ring[j] = load1(j, n + 1);
      const float d = dot8(wv, sxv[j * kGmThreads + t], 0.f);
      if (j < kk)
        a0 = fmaf(s_w[j], d, a0);
      else
        a1 = fmaf(s_w[j], d, a1);
    }
    if constexpr (SHARED) {
      const uint4 wv = ring[NE];
      if (more) ring[NE] = load1(NE, n + 1);
      a0 += dot8(wv, sxv[NE * kGmThreads + t], 0.f);
      a1 += dot8(wv, sxv[(NE + 1) * kGmThreads + t], 0.f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a0 += __shfl_xor_sync(0xffffffffu, a0, o);
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    }
    if (lane == 0) {
      red[buf][warp][0] = a0;
      red[buf][warp][1] = a1;
    }
    __syncthreads();
    if (t < 2) {
      float y = 0.f;
#pragma unroll
      for (int q = 0; q < kGmThreads / 32; ++q) y += red[buf][q][t];
      if (res != nullptr) y += (n - n0 < 64) ? s_res[t][n - n0] : bf2f(ld_act_u16(res + (size_t)t * H + n));
      out[(size_t)t * H + n] = f2bf(y);
    }
    buf ^= 1;
  }
}

// Two tokens on narrow rows (K / 8 <= TPR <= 32 vectors): the kernel above in
// the layout of gemv_down_combine_narrow_kernel. A group of TPR threads owns
// an output row (256 / TPR rows at a time), thread j of a group column vector
// j of every selected matrix's row. The activation vectors (column j of the 16
// entries' rows and of both h_s rows) are the same for every group, so they
// sit once in shared memory. Loads are unconditional at clamped, in-range
// addresses (a lane past the row's vectors meets a zero activation; a group
// past the CTA's rows computes on its last row and writes nothing), and every
// group runs the same steps, so whole-warp shuffles never meet diverged lanes.
template <int NE, int TPR, bool SHARED>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_down_combine2_narrow_kernel(
    const uint16_t* __restrict__ Wd, long long rows_bank, const uint16_t* __restrict__ Wd_s, int H, int K,
    const uint16_t* hbuf, const uint16_t* hs, const int* table, int E, int k, const float* w, const uint16_t* res,
    uint16_t* out, int routing_ready, int ahead) {
  constexpr int NP = SHARED ? NE + 1 : NE;
  constexpr int NX = SHARED ? NE + 2 : NE;
  constexpr int NG = kGmThreads / TPR;
  const int t = threadIdx.x, g = t / TPR, j = t % TPR;
  const int K8 = K >> 3;
  const uint64_t pol = policy_evict_first();
  pdl_trigger();
  const long long G = gridDim.x, c = blockIdx.x;
  const int n0 = (int)(c * H / G), n1 = (int)((c + 1) * H / G);
  if (n0 >= n1) return;  // (before any barrier)
  const TableLayout L(E, NE);
  __shared__ const uint16_t* s_rowbase[NP];
  __shared__ float s_w[NE];
  __shared__ __align__(16) uint4 sx[NX][TPR];
  auto routing = [&](bool cg) {
    if (t < NP) {
      if (SHARED && t == NE) {
        s_rowbase[t] = Wd_s;
      } else {
        const long long e = cg ? ld_cg_s32(table + L.expert() + t) : ld_act_s32(table + L.expert() + t);
        s_rowbase[t] = Wd + e * rows_bank * K;
        s_w[t] = cg ? ld_cg_f32(w + t) : ld_act_f32(w + t);
      }
    }
    __syncthreads();
  };
  const int jj = min(j, K8 - 1);
  uint4 ring[NP];
  auto load_row = [&](int n) {
    const int nn = min(n, n1 - 1);
#pragma unroll
    for (int q = 0; q < NP; ++q) ring[q] = ld_stream(s_rowbase[q] + (size_t)nn * K + (size_t)jj * 8, pol);
  };
  const int rowb = K * (int)sizeof(uint16_t);
  const int ahead_rows = ahead > 0 ? max(1, ahead / (NP * rowb)) : 0;
  int pf = n0 + NG;
  auto request = [&](int upto) {
    upto = min(upto, n1);
    if (ahead_rows > 0 && upto > pf) {
      if (t < NP) request_l2(s_rowbase[t] + (size_t)pf * K, (size_t)(upto - pf) * rowb);
      pf = upto;
    }
  };
  if (routing_ready) {
    routing(true);
    load_row(n0 + g);
    request(n0 + NG + ahead_rows);
  }
  pdl_wait();
  if (!routing_ready) {
    routing(false);
    load_row(n0 + g);
    request(n0 + NG + ahead_rows);
  }
  for (int q = t; q < NX * TPR; q += kGmThreads) {
    const int r = q / TPR, jx = q % TPR;
    const uint16_t* row = r < NE ? hbuf + (size_t)r * K : hs + (size_t)(r - NE) * K;
    sx[r][jx] = jx < K8 ? ld_act16(row + (size_t)jx * 8) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  constexpr int KK = NE / 2;  // entries per token
  for (int nb = n0; nb < n1; nb += NG) {
    const int n = nb + g;
    if (g == 0) request(n + 2 * NG + ahead_rows);  // (only threads t < NP issue)
    float a0 = 0.f, a1 = 0.f;
    const int nn = min(n + NG, n1 - 1);
#pragma unroll
    for (int q = 0; q < NE; ++q) {
      const uint4 wv = ring[q];
      ring[q] = ld_stream(s_rowbase[q] + (size_t)nn * K + (size_t)jj * 8, pol);
      const float d = dot8(wv, sx[q][j], 0.f);
      if (q < KK)
        a0 = fmaf(s_w[q], d, a0);
      else
        a1 = fmaf(s_w[q], d, a1);
    }
    if constexpr (SHARED) {
      const uint4 wv = ring[NE];
      ring[NE] = ld_stream(s_rowbase[NE] + (size_t)nn * K + (size_t)jj * 8, pol);
      a0 += dot8(wv, sx[NE][j], 0.f);
      a1 += dot8(wv, sx[NE + 1][j], 0.f);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) {
      a0 += __shfl_xor_sync(0xffffffffu, a0, o);
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    }
    if (j == 0 && n < n1) {
      if (res != nullptr) {
        a0 += bf2f(ld_act_u16(res + n));
        a1 += bf2f(ld_act_u16(res + (size_t)H + n));
      }
      out[n] = f2bf(a0);
      out[(size_t)H + n] = f2bf(a1);
    }
  }
}

bool gemv_down_combine2_supported(int k, int I) {
  return k == 8 && I >= 8 && I % 8 == 0 && I <= 8 * kGmThreads;
}

cudaError_t launch_gemv_down_combine2(dec_handle* h, const uint16_t* Wd, long long rows_bank, const uint16_t* Wd_s,
                                      int H, int I, const uint16_t* hbuf, const uint16_t* hs, const int* table, int E,
                                      int k, const float* w, const uint16_t* res, uint16_t* out, int sms,
                                      cudaStream_t s, bool routing_ready) {
  if (!gemv_down_combine2_supported(k, I)) return cudaErrorInvalidValue;
  const dim3 g(std::max(1, 2 * sms)), b(kGmThreads);
  const int rr = (int)routing_ready, a = h->l2_ahead;
  auto go = [&](auto kern, int nx) -> cudaError_t {
    const size_t smem = (size_t)nx * kGmThreads * sizeof(uint4);
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    return launch_k(h, kern, g, b, smem, s, Wd, rows_bank, Wd_s, H, I, hbuf, hs, table, E, k, w, res, out, rr, a);
  };
  if (I / 8 <= 32) {  // narrow rows: a group of 16 or 32 threads per output row
    const bool n16 = I / 8 <= 16;
    if (Wd_s != nullptr)
      return n16 ? launch_k(h, gemv_down_combine2_narrow_kernel<16, 16, true>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I,
                            hbuf, hs, table, E, k, w, res, out, rr, a)
                 : launch_k(h, gemv_down_combine2_narrow_kernel<16, 32, true>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I,
                            hbuf, hs, table, E, k, w, res, out, rr, a);
    return n16 ? launch_k(h, gemv_down_combine2_narrow_kernel<16, 16, false>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I,
                          hbuf, hs, table, E, k, w, res, out, rr, a)
               : launch_k(h, gemv_down_combine2_narrow_kernel<16, 32, false>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I,
                          hbuf, hs, table, E, k, w, res, out, rr, a);
  }
  if (Wd_s != nullptr) return go(gemv_down_combine2_kernel<16, true>, 18);
  return go(gemv_down_combine2_kernel<16, false>, 16);
}

bool gemv_down_combine_supported(int k, int I) { return k == 8 && I >= 8 && I % 8 == 0 && I <= 8 * kGmThreads; }

cudaError_t launch_gemv_down_combine(dec_handle* h, const uint16_t* Wd, long long rows_bank, const uint16_t* Wd_s,
                                     int H, int I, const uint16_t* hbuf, const uint16_t* hs, const int* table, int E,
                                     int k, const float* w, const uint16_t* res, uint16_t* out, int sms,
                                     cudaStream_t s, bool routing_ready) {
  if (!gemv_down_combine_supported(k, I)) return cudaErrorInvalidValue;
  const dim3 g(std::max(1, 2 * sms)), b(kGmThreads);
  const int rr = (int)routing_ready, a = h->l2_ahead;
  const int K8 = I / 8;
  if (K8 <= 32) {
    // narrow rows: a group of 16 or 32 threads per output row
    if (Wd_s != nullptr)
      return K8 <= 16 ? launch_k(h, gemv_down_combine_narrow_kernel<9, 16, true>, g, b, 0, s, Wd, rows_bank, Wd_s, H,
                                 I, hbuf, hs, table, E, k, w, res, out, rr, a)
                      : launch_k(h, gemv_down_combine_narrow_kernel<9, 32, true>, g, b, 0, s, Wd, rows_bank, Wd_s, H,
                                 I, hbuf, hs, table, E, k, w, res, out, rr, a);
    return K8 <= 16 ? launch_k(h, gemv_down_combine_narrow_kernel<8, 16, false>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I,
                               hbuf, hs, table, E, k, w, res, out, rr, a)
                    : launch_k(h, gemv_down_combine_narrow_kernel<8, 32, false>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I,
                               hbuf, hs, table, E, k, w, res, out, rr, a);
  }
  if (Wd_s != nullptr)
    return launch_k(h, gemv_down_combine_kernel<9, 1, true>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I, hbuf, hs, table,
                    E, k, w, res, out, rr, a);
  return launch_k(h, gemv_down_combine_kernel<8, 1, false>, g, b, 0, s, Wd, rows_bank, Wd_s, H, I, hbuf, hs, table, E,
                  k, w, res, out, rr, a);
}

bool gemv_moe_supported(int K) { return K >= 8 && K % 8 == 0 && K <= 8 * 4 * kGmThreads; }

// Narrow rows (K <= 256: K / 8 <= TPR in {16, 32} vectors): the problems of
// gemv_moe_kernel with a group of TPR threads per unit, so that a CTA is
// 256 / TPR independent "virtual CTAs". Each group takes its own equal,
// contiguous range of the unit sequence, walks it RB units per step (one
// vector of each of the unit's rows per thread; the next step's loads are
// issued before this step's FMAs) and reduces by shuffles only: no barrier.
template <bool SWIGLU, int TPR>
__global__ void __launch_bounds__(kGmThreads, 2) gemv_moe_narrow_kernel(const GemvMoeParams P) {
  constexpr int NR = SWIGLU ? 2 : 1;
  constexpr int RB = 4;
  constexpr int NG = kGmThreads / TPR;
  const int t = threadIdx.x, g = t / TPR, j = t % TPR;
  // Groups walk ranges of their own, so two 16-thread groups of one warp may
  // diverge: every shuffle names only its own group's lanes.
  const unsigned gmask = TPR == 32 ? 0xffffffffu : (0xffffu << (t & 16));
  const int K8 = P.K >> 3;
  const int jj = min(j, K8 - 1);  // lanes past the row read its last vector and meet a zero activation
  const uint64_t pol = policy_evict_first();
  if (!P.late_trigger) pdl_trigger();
  const TableLayout L(P.E, P.n_entries);
  const int ns = P.sA != nullptr ? P.ns : 0;
  auto expert_of = [&](int p) -> long long {
    if (p < ns) return -1;
    return P.table ? ld_act_s32(P.table + L.expert() + (p - ns)) : 0;
  };
  auto slot_of = [&](int p) -> long long {
    if (p < ns) return p;
    return P.table ? ld_act_s32(P.table + L.offset() + (p - ns)) : 0;
  };
  auto mat0 = [&](long long e) { return e < 0 ? P.sA : P.A + e * P.rows_per_prob_bank * P.K; };
  auto mat1 = [&](long long e) { return e < 0 ? P.sA2 : P.A2 + e * P.rows_per_prob_bank * P.K; };
  const long long VG = (long long)gridDim.x * NG, vg = (long long)blockIdx.x * NG + g;
  pdl_wait();
  if (P.late_trigger) pdl_trigger();
  const long long T = ((P.table ? ld_act_s32(P.table + L.U()) : 1) + ns) * (long long)P.R;
  const long long q0 = vg * T / VG, q1 = (vg + 1) * T / VG;
  if (q0 >= q1) return;  // (no barrier in this kernel)
  int p = (int)(q0 / P.R), r = (int)(q0 % P.R);
  long long left = q1 - q0;
  long long e = expert_of(p);
  const uint16_t* A0 = mat0(e);
  const uint16_t* A1 = mat1(e);
  uint4 wa[RB][NR];
  auto load_units = [&](uint4(&w)[RB][NR], const uint16_t* a0, const uint16_t* a1, int rr, int nu) {
#pragma unroll
    for (int u = 0; u < RB; ++u)
#pragma unroll
      for (int a = 0; a < NR; ++a) {
        const int row = rr + min(u, nu - 1);  // past nu: re-read the last unit (in range), discarded
        w[u][a] = ld_stream((a == 0 ? a0 : a1) + (size_t)row * P.K + (size_t)jj * 8, pol);
      }
  };
  int nu = (int)min((long long)min(RB, P.R - r), left);
  load_units(wa, A0, A1, r, nu);
  uint4 xr;
  long long slot = slot_of(p);
  auto load_x = [&]() {
    const long long xr_row = (e >= 0 && P.x_by_token && P.table) ? ld_act_s32(P.table + L.slot_token() + slot) : slot;
    const uint16_t* xrow = e < 0 ? P.sx + slot * P.sldx : P.x + xr_row * P.ldx;
    xr = j < K8 ? ld_act16(xrow + (size_t)j * 8) : make_uint4(0, 0, 0, 0);
  };
  load_x();
  while (left > 0) {
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
    uint4 wb[RB][NR];
    if (nun > 0) load_units(wb, N0, N1, rn, nun);
    float acc[RB][NR];
#pragma unroll
    for (int u = 0; u < RB; ++u)
#pragma unroll
      for (int a = 0; a < NR; ++a) {
        float sum = dot8(wa[u][a], xr, 0.f);
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(gmask, sum, o);
        acc[u][a] = sum;
      }
    // lane u of the group writes unit u
#pragma unroll
    for (int u = 0; u < RB; ++u)
      if (j == u && u < nu) {
        void* dst = e < 0 ? P.sout : P.out;
        const long long o = slot * (e < 0 ? P.sldo : P.ldo) + r + u;
        if (SWIGLU) {
          const float gg = acc[u][0], up = acc[u][NR - 1];
          reinterpret_cast<uint16_t*>(dst)[o] = swiglu_bf16(gg, up);
        } else {
          reinterpret_cast<float*>(dst)[o] = acc[u][0];
        }
      }
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
      for (int a = 0; a < NR; ++a) wa[u][a] = wb[u][a];
  }
}

template <bool SWIGLU>
static cudaError_t launch_mode(dec_handle* h, const GemvMoeParams& P, int grid, cudaStream_t s) {
  const int K8 = P.K / 8;
  const dim3 g(grid), b(kGmThreads);
  if (K8 <= 16) return launch_k(h, gemv_moe_narrow_kernel<SWIGLU, 16>, g, b, 0, s, P);
  if (K8 <= 32) return launch_k(h, gemv_moe_narrow_kernel<SWIGLU, 32>, g, b, 0, s, P);
  if (K8 <= kGmThreads) return launch_k(h, gemv_moe_kernel<SWIGLU, 1>, g, b, 0, s, P);
  if (K8 <= 2 * kGmThreads) return launch_k(h, gemv_moe_kernel<SWIGLU, 2>, g, b, 0, s, P);
  return launch_k(h, gemv_moe_kernel<SWIGLU, 4>, g, b, 0, s, P);
}

cudaError_t launch_gemv_moe(dec_handle* h, bool swiglu, const uint16_t* A, const uint16_t* A2,
                            long long rows_per_prob_bank, int R, int K, const uint16_t* x, long long ldx,
                            const int* table, int E, int n_entries, void* out, long long ldo, int sms,
                            cudaStream_t s, const GemvMoeShared* shared, int nprob_known, bool late_trigger,
                            bool x_by_token) {
  if (!gemv_moe_supported(K)) return cudaErrorInvalidValue;
  GemvMoeParams P;
  P.sA = shared ? shared->A : nullptr;
  P.sA2 = shared ? (shared->A2 ? shared->A2 : shared->A) : nullptr;
  P.sx = shared ? shared->x : nullptr;
  P.sout = shared ? shared->out : nullptr;
  P.ns = shared ? std::max(1, shared->n) : 0;
  P.sldx = shared ? shared->ldx : 0;
  P.sldo = shared ? shared->ldo : 0;
  P.x_by_token = x_by_token ? 1 : 0;
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
  P.nprob_known = table ? nprob_known : 0;
  P.late_trigger = late_trigger ? 1 : 0;
  P.ahead = h->l2_ahead;
  const int grid = std::max(1, 2 * sms);
  return swiglu ? launch_mode<true>(h, P, grid, s) : launch_mode<false>(h, P, grid, s);
}

}  // namespace dec
