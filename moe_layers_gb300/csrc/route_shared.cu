// The MoE fronts: routing and expert gate/up in one launch at one to a few
// tokens, and the few-token routing launch.
//
// Kimi K3 article, Part 1 §3 "Mejorar la programación de MoE" (the shared
// expert runs beside the routing, on its own stream) and §4 (while the
// latency-bound router / top-k phase leaves the memory idle, weights that
// come next are streamed). At one token the routing chain (RMSNorm, router
// logits, hand-off, top-k, routing table) is a few microseconds of pure
// latency; the same CTAs stream the shared expert's 2 x I x H gate/up
// weights meanwhile, so the memory stays busy, and then the selected
// experts' gate/up rows once the routing is published.
//
// Grid: two 256-thread CTAs per SM. Every CTA of a front
//  1. takes a router unit (8 router rows x 1024 columns of fp32 W_r, one row
//     per warp) from a ticket counter and loads its rows, and its RMSNorm
//     gains, before the dependency wait;
//  2. normalises the token rows (the RMSNorm kernel's order, so the bits are
//     the same) into shared memory;
//  3. computes its units' logit pieces (taking further units while any
//     remain) and arrives on the hand-off once per unit; the arrival that
//     completes the last unit takes the top-k, writes idx, w, scores and the
//     routing table, and publishes the routing with a release flag;
//  4. streams shared-expert row pairs (row r of W_g and of W_u ->
//     h_s[r] = bf16(silu(g) * u)) taken from a row queue (an atomic counter),
//     so the CTA that ran the top-k simply takes fewer rows;
//  5. waits for the routing flag (bounded), then streams its static share of
//     the selected experts' gate/up rows and then rows from a tail queue.
// The queues, the flag and a "done" counter are reset by the last CTA to
// finish. Because the CTAs wait for a flag that one of them sets, the router
// units are not owned by block index: a CTA takes them from a ticket counter
// (take_unit) and the hand-off counts units, so the routing never waits for a
// CTA that the SMs cannot hold yet.
//
// Two to four tokens: moe_front_multi_kernel (the same for the (token,
// expert) entries), and route_shared_multi_kernel (the routing launch alone,
// with the shared expert's gate/up when there is one, for the shapes outside
// the front's limits).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace dec {

namespace {

constexpr int kThreads = 256;
constexpr int kUnitCols = 1024;  // router unit width (columns of W_r)

struct RouteSharedParams {
  const uint16_t* h1;     // the token's row, bf16 [H]
  const uint16_t* gamma;  // RMSNorm gains [H]
  float eps;
  const float* Wr;        // router weights fp32 [E][H]
  int H, E, k;
  int M;                  // tokens (the multi-token kernel)
  int nunits;             // ceil(E / 8) * ceil(H / 1024)
  uint16_t* xn;           // normalised row out [H]
  float* parts;           // logit pieces [ceil(H / 1024)][E]
  int* ctr;               // [0] hand-off, [1] row queue, [2] done; zero on entry and on return
  int32_t* idx;
  float* w;
  float* scores;          // [E] or null
  int* table;             // one-token routing table
  const uint16_t* Wg;     // shared gate [I][H]
  const uint16_t* Wu;     // shared up [I][H]
  int I;
  uint16_t* hs;           // shared SwiGLU output bf16 [I]
  // the MoE front kernel only: the routed gate/up
  const uint16_t* Wgb;    // routed gate bank [E][I][H]
  const uint16_t* Wub;    // routed up bank [E][I][H]
  uint16_t* hbuf;         // routed SwiGLU outputs bf16 [k][I] (slot j: entry j)
  int* err;               // device error word
  unsigned long long wait_ns;
  const char* pf = nullptr;  // the MoE fronts: a region pulled into L2 while the routing is awaited
  size_t pf_bytes = 0;       // (16-byte multiple; 0 for none)
  size_t pf_per = 0;         // bytes per CTA (16-byte multiple)
};

// The MoE fronts hand out their router units from a counter (ctr[6]) that
// cycles through nunits + G values: a CTA takes tickets until one is past the
// last unit, so every launch takes exactly nunits + G tickets and leaves the
// counter where it found it (a launch's CTAs take their tickets before they
// trigger the next launch, so launches never interleave on it). A unit is
// therefore computed by whichever running CTA took it, and the routing
// hand-off completes once the CTAs that are resident have computed all units,
// whether or not every CTA of the grid can be resident at once (another
// stream's kernels may hold SMs). The hand-off counts units, not CTAs.
__device__ __forceinline__ int take_unit(int* ctr, int nunits, int G) {
  return (int)atomicInc(reinterpret_cast<unsigned*>(ctr + 6), (unsigned)(nunits + G - 1));
}

// The token's row into xr (registers) and sx (shared memory), RMS-normalised
// with the gains that xr holds on entry, or as it is without gains (has_gamma
// false); also to xn when given. Normalising takes one barrier.
template <int VPT>
__device__ __forceinline__ void norm_row(const uint16_t* row, bool has_gamma, float eps, int H, uint4 (&xr)[VPT],
                                         uint16_t* sx, float* red, uint16_t* xn) {
  const int t = threadIdx.x, H8 = H >> 3;
  uint4 hv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = t + kThreads * i;
    hv[i] = v < H8 ? ld_act16(row + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
  }
  float r = 0.f;
  if (has_gamma) r = block_rms_scale<kThreads / 32>(thread_sumsq<VPT, kThreads>(hv, H8), H, eps, red);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = t + kThreads * i;
    xr[i] = has_gamma ? norm8(hv[i], xr[i], r) : hv[i];
    if (v < H8) {
      *reinterpret_cast<uint4*>(&sx[v * 8]) = xr[i];
      if (xn != nullptr) *reinterpret_cast<uint4*>(xn + (size_t)v * 8) = xr[i];
    }
  }
}

// M <= MT token rows [M][H] into sx [MT][H] (and xn when given), each
// RMS-normalised with the gains gv, or as they are without gains. One barrier
// per row when normalising (red: [MT][8] floats).
template <int VPT, int MT>
__device__ __forceinline__ void norm_rows(const uint16_t* rows, int M, bool has_gamma, const uint4 (&gv)[VPT],
                                          float eps, int H, uint16_t* sx, float (*red)[kThreads / 32], uint16_t* xn) {
  const int t = threadIdx.x, H8 = H >> 3;
#pragma unroll
  for (int q = 0; q < MT; ++q) {
    if (q < M) {
      uint4 hv[VPT];
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kThreads * i;
        hv[i] = v < H8 ? ld_act16(rows + (size_t)q * H + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
      }
      float r = 0.f;
      if (has_gamma) r = block_rms_scale<kThreads / 32>(thread_sumsq<VPT, kThreads>(hv, H8), H, eps, red[q]);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kThreads * i;
        if (v < H8) {
          const uint4 y = has_gamma ? norm8(hv[i], gv[i], r) : hv[i];
          *reinterpret_cast<uint4*>(&sx[(size_t)q * H + v * 8]) = y;
          if (xn != nullptr) *reinterpret_cast<uint4*>(xn + (size_t)q * H + (size_t)v * 8) = y;
        }
      }
    }
  }
}

// M = 2 .. MT tokens: the same launch for a few tokens. Every CTA
// normalises the M rows (two passes over them: sums of squares, then the
// normalised rows into shared memory; CTA 0 writes them out), adds its router
// units' logit pieces for every token, and arrives; the last CTA scores all
// tokens and warp t takes token t's top-k and writes its k entries of the
// routing table (block_topk_tokens; one problem per (token, expert) entry). The shared expert's gate/up
// rows stream from the queue meanwhile, each row pair applied to the M rows
// held in shared memory.
template <int J, int VPT, int MT>
__global__ void __launch_bounds__(kThreads, 2) route_shared_multi_kernel(const RouteSharedParams P) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = P.H, H8 = H >> 3, M = P.M;
  const int ngrp = (P.E + 7) / 8;
  const int ksplit = (H + kUnitCols - 1) / kUnitCols;
  extern __shared__ __align__(16) uint16_t sx[];  // the normalised rows [MT][H]
  __shared__ float s_norm[MT][kThreads / 32];
  __shared__ float red[2][kThreads / 32][2 * MT];
  __shared__ int s_row[2];
  __shared__ int s_next[2];
  __shared__ int s_last;
  const uint64_t pol = policy_evict_first();
  pdl_trigger();

  float4 wv[kUnitCols / 128];
  auto load_unit = [&](int u) {
    const int e = (u % ngrp) * 8 + warp, k0 = (u / ngrp) * kUnitCols;
    const int kn = min(kUnitCols, H - k0);
#pragma unroll
    for (int i = 0; i < kUnitCols / 128; ++i) {
      const int kk = 4 * (lane + 32 * i);
      wv[i] = (u < P.nunits && e < P.E && kk < kn)
                  ? __ldg(reinterpret_cast<const float4*>(P.Wr + (size_t)e * H + k0 + kk))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_unit(c);
  const bool has_shared = P.Wg != nullptr && P.I > 0;
  int base = 0;
  if (t == 0 && has_shared) {
    base = atomicAdd(&P.ctr[1], 3);
    for (int q = 0; q < 3; ++q)
      if (base + q < P.I) {
        request_l2(P.Wg + (size_t)(base + q) * H, (size_t)H * 2);
        request_l2(P.Wu + (size_t)(base + q) * H, (size_t)H * 2);
      }
  }
  uint4 gv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = t + kThreads * i;
    gv[i] = (P.gamma != nullptr && v < H8) ? *reinterpret_cast<const uint4*>(P.gamma + (size_t)v * 8)
                                           : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();

  // RMSNorm of the M rows (each row's sum of squares in the RMSNorm kernel's order)
  norm_rows<VPT, MT>(P.h1, M, P.gamma != nullptr, gv, P.eps, H, sx, s_norm, c == 0 ? P.xn : nullptr);
  int pending = base + 2;  // (thread 0)
  __syncthreads();

  // router logit pieces of this CTA's units for every token, then the hand-off
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int u = c + m * G;
    if (m == 1 && u < P.nunits) load_unit(u);
    if (u < P.nunits) {
      const int e = (u % ngrp) * 8 + warp, ks = u / ngrp, k0 = ks * kUnitCols;
      const int kn = min(kUnitCols, H - k0);
      float acc[MT];
#pragma unroll
      for (int q = 0; q < MT; ++q) acc[q] = 0.f;
#pragma unroll
      for (int i = 0; i < kUnitCols / 128; ++i) {
        const int kk = 4 * (lane + 32 * i);
        if (kk < kn) {
#pragma unroll
          for (int q = 0; q < MT; ++q) {
            if (q < M) {
              const uint2 xv = *reinterpret_cast<const uint2*>(&sx[(size_t)q * H + k0 + kk]);
              float a = acc[q];
              a = fmaf(wv[i].x, bf_lo(xv.x), a);
              a = fmaf(wv[i].y, bf_hi(xv.x), a);
              a = fmaf(wv[i].z, bf_lo(xv.y), a);
              a = fmaf(wv[i].w, bf_hi(xv.y), a);
              acc[q] = a;
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < MT; ++q) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
        if (lane == 0 && e < P.E && q < M) P.parts[((size_t)ks * M + q) * P.E + e] = acc[q];
      }
    }
  }
  if (t == 0) {
    s_row[0] = has_shared ? base : P.I;
    s_row[1] = has_shared ? base + 1 : P.I;
  }
  __syncthreads();
  if (t == 0) s_last = atom_add_acq_rel_gpu(&P.ctr[0], 1) == G - 1;
  __syncthreads();
  if (s_last) {
    block_topk_tokens<J, MT>(P.parts, ksplit, M, P.E, P.k, P.idx, P.w, P.scores, P.table);
    if (t == 0) P.ctr[0] = 0;  // leave the workspace reusable
  }

  // shared-expert gate/up rows from the queue, each applied to the M rows
  if (!has_shared) return;
  uint4 wa[2][VPT], wb[2][VPT];
  auto load = [&](uint4(&wr)[2][VPT], int row) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kThreads * i;
        wr[a][i] = v < H8 ? ld_stream((a == 0 ? P.Wg : P.Wu) + (size_t)row * H + (size_t)v * 8, pol)
                          : make_uint4(0, 0, 0, 0);
      }
  };
  int cur = s_row[0], nxt = s_row[1];
  if (cur < P.I) load(wa, cur);
  int buf = 0;
  while (cur < P.I) {
    if (nxt < P.I) load(wb, nxt);
    float g[MT], up[MT];
#pragma unroll
    for (int q = 0; q < MT; ++q) {
      g[q] = 0.f;
      up[q] = 0.f;
      if (q < M) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = t + kThreads * i;
          if (v < H8) {
            const uint4 xv = *reinterpret_cast<const uint4*>(&sx[(size_t)q * H + v * 8]);
            g[q] = dot8(wa[0][i], xv, g[q]);
            up[q] = dot8(wa[1][i], xv, up[q]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        g[q] += __shfl_xor_sync(0xffffffffu, g[q], o);
        up[q] += __shfl_xor_sync(0xffffffffu, up[q], o);
      }
      if (lane == 0) {
        red[buf][warp][2 * q] = g[q];
        red[buf][warp][2 * q + 1] = up[q];
      }
    }
    if (t == 0) {
      s_next[buf] = pending;
      if (pending < P.I) {
        request_l2(P.Wg + (size_t)pending * H, (size_t)H * 2);
        request_l2(P.Wu + (size_t)pending * H, (size_t)H * 2);
        pending = atomicAdd(&P.ctr[1], 1);
      }
    }
    __syncthreads();
    if (t < M) {
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) {
        gs += red[buf][w][2 * t];
        us += red[buf][w][2 * t + 1];
      }
      P.hs[(size_t)t * P.I + cur] = swiglu_bf16(gs, us);
    }
    const int nn = s_next[buf];
    cur = nxt;
    nxt = nn;
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int i = 0; i < VPT; ++i) wa[a][i] = wb[a][i];
    buf ^= 1;
  }
  if (t == 0 && atom_add_acq_rel_gpu(&P.ctr[2], 1) == G - 1) {
    P.ctr[1] = 0;
    P.ctr[2] = 0;
  }
}

// One token: the MoE front in one launch: the routing launch above (RMSNorm,
// router, top-k, routing table), then one row queue over the shared expert's
// gate/up rows followed by the k routed experts' rows. The routing is
// published by the CTA whose arrival completes the last router unit, and it
// waits for nothing. Units go to whichever CTAs are running (take_unit), so
// a CTA that waits for the routing depends only on CTAs that have started,
// however many of the grid's CTAs the SMs can hold beside other kernels.
template <int J, int VPT>
__global__ void __launch_bounds__(kThreads, 2) moe_front_kernel(const RouteSharedParams P) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = P.H, H8 = H >> 3;
  const int ngrp = (P.E + 7) / 8;
  extern __shared__ __align__(16) uint16_t sx[];  // the normalised row [H]
  __shared__ float s_norm[kThreads / 32];
  __shared__ float red[2][kThreads / 32][2];
  __shared__ int s_row[2];
  __shared__ int s_next[2];
  __shared__ int s_last;
  __shared__ int s_ok;
  const uint64_t pol = policy_evict_first();

  float4 wv[kUnitCols / 128];
  auto load_unit = [&](int u) {
    const int e = (u % ngrp) * 8 + warp, k0 = (u / ngrp) * kUnitCols;
    const int kn = min(kUnitCols, H - k0);
#pragma unroll
    for (int i = 0; i < kUnitCols / 128; ++i) {
      const int kk = 4 * (lane + 32 * i);
      wv[i] = (u < P.nunits && e < P.E && kk < kn)
                  ? __ldg(reinterpret_cast<const float4*>(P.Wr + (size_t)e * H + k0 + kk))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  // this CTA's first router unit (take_unit): its fp32 rows load before the wait
  __shared__ int s_unit;
  if (t == 0) s_unit = take_unit(P.ctr, P.nunits, G);
  __syncthreads();
  int u = s_unit;
  load_unit(u);
  // (a grab that races the previous launch's reset finds the queue exhausted
  // or already reset: that launch's CTAs trigger this one's predecessors only
  // after their shared rows)
  int base = 0;
  if (t == 0) {
    base = atomicAdd(&P.ctr[1], 3);
    for (int q = 0; q < 3; ++q)
      if (base + q < P.I) {
        request_l2(P.Wg + (size_t)(base + q) * H, (size_t)H * 2);
        request_l2(P.Wu + (size_t)(base + q) * H, (size_t)H * 2);
      }
  }
  uint4 xr[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = t + kThreads * i;
    xr[i] = (P.gamma != nullptr && v < H8) ? *reinterpret_cast<const uint4*>(P.gamma + (size_t)v * 8)
                                           : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  norm_row<VPT>(P.h1, P.gamma != nullptr, P.eps, H, xr, sx, s_norm, nullptr);
  int pending = base + 2;
  __syncthreads();
  // Router units: the CTA's ticket, then further tickets while units remain.
  // Every computed unit arrives on the hand-off (ctr[0] counts units); the
  // arrival that completes the last unit takes the top-k.
  for (;;) {
    if (u < P.nunits) {
      const int e = (u % ngrp) * 8 + warp, ks = u / ngrp, k0 = ks * kUnitCols;
      const int kn = min(kUnitCols, H - k0);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kUnitCols / 128; ++i) {
        const int kk = 4 * (lane + 32 * i);
        if (kk < kn) {
          const uint2 xv = *reinterpret_cast<const uint2*>(&sx[k0 + kk]);
          acc = fmaf(wv[i].x, bf_lo(xv.x), acc);
          acc = fmaf(wv[i].y, bf_hi(xv.x), acc);
          acc = fmaf(wv[i].z, bf_lo(xv.y), acc);
          acc = fmaf(wv[i].w, bf_hi(xv.y), acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0 && e < P.E) P.parts[(size_t)ks * P.E + e] = acc;
    }
    // The barrier orders the unit's stores before thread 0's acquire-release
    // add; in the last arrival the barrier after it orders every read after it.
    __syncthreads();
    if (t == 0) {
      s_last = u < P.nunits && atom_add_acq_rel_gpu(&P.ctr[0], 1) == P.nunits - 1;
      s_unit = u < P.nunits ? take_unit(P.ctr, P.nunits, G) : P.nunits;
    }
    __syncthreads();
    if (s_last) {
      int se = 0;
      float sw = 0.f;
      block_topk<J, true>(P.parts, (H + kUnitCols - 1) / kUnitCols, 1, 0, P.E, P.k, P.idx, P.w, P.scores, &se, &sw);
      if (warp == 0) {
        write_one_token_table(P.table, P.E, P.k, se);
        __syncwarp();
        if (lane == 0) {
          P.ctr[0] = 0;
          P.ctr[5] = c;                  // this CTA's static share goes to the tail queue
          st_release_gpu(&P.ctr[3], 1);  // the routing is written
        }
      }
    }
    u = s_unit;
    if (u >= P.nunits) break;  // (the last arrival's next ticket is always past the units)
    load_unit(u);
  }

  // Three streams of row pairs, one after the other: the shared expert's
  // rows from the row queue until it runs dry; then this CTA's static
  // contiguous share of the routed rows (7/8 of them split evenly; routed row
  // q is row q mod I of entry q / I, with the one token's row for every
  // problem); then routed rows from a tail queue, so that CTAs that started
  // late or stream slower end together with the rest. Each queue grab is
  // made an iteration before its value is needed. Before its first routed
  // row a CTA waits for the routing (thread 0, acquire, bounded by the
  // wall-clock limit: past it the device error word is raised and the CTA
  // stops); dependents are triggered once the routing is seen, so the down
  // kernel may read it before its dependency wait.
  const int I = P.I, T = P.k * P.I;
  const int bulk = T * 7 / 8 / G, tail0 = G * bulk;
  uint4 wa[2][VPT], wb[2][VPT];
  auto load_rows = [&](uint4(&wr)[2][VPT], const uint16_t* g0, const uint16_t* u0) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kThreads * i;
        wr[a][i] = v < H8 ? ld_stream((a == 0 ? g0 : u0) + (size_t)v * 8, pol) : make_uint4(0, 0, 0, 0);
      }
  };
  auto dot_pair = [&](int b) {
    float g = 0.f, up = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      // the normalised row from shared memory (registers hold the weight stream)
      const int v = t + kThreads * i;
      const uint4 xv = v < H8 ? *reinterpret_cast<const uint4*>(&sx[v * 8]) : make_uint4(0, 0, 0, 0);
      g = dot8(wa[0][i], xv, g);
      up = dot8(wa[1][i], xv, up);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      up += __shfl_xor_sync(0xffffffffu, up, o);
    }
    if (lane == 0) {
      red[b][warp][0] = g;
      red[b][warp][1] = up;
    }
  };
  auto swiglu_out = [&](int b) {  // thread 0, after the barrier
    float gs = 0.f, us = 0.f;
#pragma unroll
    for (int q = 0; q < kThreads / 32; ++q) {
      gs += red[b][q][0];
      us += red[b][q][1];
    }
    return swiglu_bf16(gs, us);
  };
  auto shift = [&]() {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int i = 0; i < VPT; ++i) wa[a][i] = wb[a][i];
  };
  int buf = 0;
  if (t == 0) {
    s_row[0] = base;
    s_row[1] = base + 1;
  }
  __syncthreads();
  {  // the shared expert's rows
    int cur = s_row[0], nxt = s_row[1];
    if (cur < I) load_rows(wa, P.Wg + (size_t)cur * H, P.Wu + (size_t)cur * H);
    while (cur < I) {
      if (nxt < I) load_rows(wb, P.Wg + (size_t)nxt * H, P.Wu + (size_t)nxt * H);
      dot_pair(buf);
      if (t == 0) {
        s_next[buf] = pending;
        if (pending < I) {
          request_l2(P.Wg + (size_t)pending * H, (size_t)H * 2);
          request_l2(P.Wu + (size_t)pending * H, (size_t)H * 2);
          pending = atomicAdd(&P.ctr[1], 1);
        }
      }
      __syncthreads();
      if (t == 0) P.hs[cur] = swiglu_out(buf);
      const int nn = s_next[buf];
      cur = nxt;
      nxt = nn;
      shift();
      buf ^= 1;
    }
  }

  // the routing
  __shared__ const uint16_t* s_g[32];
  __shared__ const uint16_t* s_u[32];
  if (t == 0) {
    // Cross-layer prefetch: a CTA that reaches the wait pulls its slice of the
    // next operator's weights into L2 (memory otherwise idle until the routing).
    if (P.pf_bytes > 0) {
      const size_t off = (size_t)c * P.pf_per;
      if (off < P.pf_bytes) {
        const size_t n = P.pf_bytes - off < P.pf_per ? P.pf_bytes - off : P.pf_per;
        request_l2(P.pf + off, n);
      }
    }
    const unsigned long long t0 = globaltimer();
    int ok = 1;
    while (ld_acquire_gpu(&P.ctr[3]) == 0) {
      if (globaltimer() - t0 > P.wait_ns) {
        atomicOr(P.err, DEV_ERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    s_ok = ok;
  }
  __syncthreads();
  if (s_ok) {
    __shared__ int s_tb, s_cstar;
    if (t < P.k) {
      const long long e = ld_cg_s32(P.table + TableLayout(P.E, P.k).expert() + t);
      s_g[t] = P.Wgb + e * I * H;
      s_u[t] = P.Wub + e * I * H;
    }
    if (t == 0) s_cstar = ld_cg_s32(&P.ctr[5]);
    __syncthreads();
    pdl_trigger();
    const int cstar = s_cstar;
    // tail unit v: the top-k CTA's share first, then the rows after the shares
    auto tail_row = [&](int v) { return v < bulk ? cstar * bulk + v : tail0 + v - bulk; };
    const int ntail = bulk + T - tail0;
    auto rows = [&](int q, const uint16_t*& g0, const uint16_t*& u0) {
      const int e = q / I, r = q - e * I;
      g0 = s_g[e] + (size_t)r * H;
      u0 = s_u[e] + (size_t)r * H;
    };
    int tb = 0;  // (thread 0) the first of three tail units grabbed together, published in s_tb
    const int q0 = c * bulk, q1 = c == cstar ? q0 : q0 + bulk;
    if (q1 - q0 < 4) {
      if (t == 0) {
        tb = atomicAdd(&P.ctr[4], 3);
        s_tb = tb;
      }
      __syncthreads();
    }
    bool wa_loaded = false;
    if (q0 < q1) {  // this CTA's static share
      int e = q0 / I, r = q0 - (q0 / I) * I;
      load_rows(wa, s_g[e] + (size_t)r * H, s_u[e] + (size_t)r * H);
      for (int q = q0; q < q1; ++q) {
        int en = e, rn = r + 1;
        if (rn == I) {
          ++en;
          rn = 0;
        }
        if (q + 1 < q1) {
          load_rows(wb, s_g[en] + (size_t)rn * H, s_u[en] + (size_t)rn * H);
        } else if (s_tb < ntail) {  // the first tail row follows without a gap
          const uint16_t *g0, *u0;
          rows(tail_row(s_tb), g0, u0);
          load_rows(wb, g0, u0);
          wa_loaded = true;
        }
        if (t == 0) {
          if (q + 2 < q1) {  // the row after next into L2
            const int e2 = rn + 1 == I ? en + 1 : en, r2 = rn + 1 == I ? 0 : rn + 1;
            request_l2(s_g[e2] + (size_t)r2 * H, (size_t)H * 2);
            request_l2(s_u[e2] + (size_t)r2 * H, (size_t)H * 2);
          }
          if (q + 3 == q1 && q1 - q0 >= 4) tb = atomicAdd(&P.ctr[4], 3);  // the tail grab
          if (q + 2 == q1 && q1 - q0 >= 4) {
            s_tb = tb;  // published at this iteration's barrier
            for (int v = tb; v < tb + 2 && v < ntail; ++v) {
              const uint16_t *g2, *u2;
              rows(tail_row(v), g2, u2);
              request_l2(g2, (size_t)H * 2);
              request_l2(u2, (size_t)H * 2);
            }
          }
        }
        dot_pair(buf);
        __syncthreads();
        if (t == 0) P.hbuf[q] = swiglu_out(buf);
        e = en;
        r = rn;
        shift();
        buf ^= 1;
      }
    }
    {  // the tail queue
      const int v0 = s_tb;
      int cur = v0, nxt = v0 + 1;
      if (t == 0) pending = v0 + 2;
      const uint16_t *g0, *u0;
      if (cur < ntail && !wa_loaded) {
        rows(tail_row(cur), g0, u0);
        load_rows(wa, g0, u0);
      }
      while (cur < ntail) {
        if (nxt < ntail) {
          rows(tail_row(nxt), g0, u0);
          load_rows(wb, g0, u0);
        }
        dot_pair(buf);
        if (t == 0) {
          s_next[buf] = pending;
          if (pending < ntail) {
            const uint16_t *g2, *u2;
            rows(tail_row(pending), g2, u2);
            request_l2(g2, (size_t)H * 2);
            request_l2(u2, (size_t)H * 2);
            pending = atomicAdd(&P.ctr[4], 1);
          }
        }
        __syncthreads();
        if (t == 0) P.hbuf[tail_row(cur)] = swiglu_out(buf);
        const int nn = s_next[buf];
        cur = nxt;
        nxt = nn;
        shift();
        buf ^= 1;
      }
    }
  }
  if (t == 0 && atom_add_acq_rel_gpu(&P.ctr[2], 1) == G - 1) {
    P.ctr[1] = 0;
    P.ctr[2] = 0;
    P.ctr[3] = 0;
    P.ctr[4] = 0;
  }
}

// Two to four tokens: the MoE front in one launch. The routing and the
// shared gate/up of route_shared_multi_kernel (the M rows normalised into
// shared memory, every CTA's router units for every token, the last CTA's
// top-k of all tokens and entry table; the shared expert's row pairs from the
// queue, each applied to the M rows), then the routed entries' gate/up as in
// moe_front_kernel: once the routing flag is seen, each CTA's static share
// of the M k I row pairs, then the tail queue. Routed row q is row q mod I of
// entry p = q / I (token p / k, its normalised row from shared memory);
// outputs go to hbuf[q] (slot p's row at hbuf + p I).
template <int J, int VPT, int MT>
__global__ void __launch_bounds__(kThreads, 2) moe_front_multi_kernel(const RouteSharedParams P) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = P.H, H8 = H >> 3, M = P.M;
  const int ngrp = (P.E + 7) / 8;
  const int ksplit = (H + kUnitCols - 1) / kUnitCols;
  extern __shared__ __align__(16) uint16_t sx[];  // the normalised rows [MT][H]
  __shared__ float s_norm[MT][kThreads / 32];
  __shared__ float red[2][kThreads / 32][2 * MT];
  __shared__ int s_row[2];
  __shared__ int s_next[2];
  __shared__ int s_last;
  __shared__ int s_ok;
  const uint64_t pol = policy_evict_first();

  float4 wv[kUnitCols / 128];
  auto load_unit = [&](int u) {
    const int e = (u % ngrp) * 8 + warp, k0 = (u / ngrp) * kUnitCols;
    const int kn = min(kUnitCols, H - k0);
#pragma unroll
    for (int i = 0; i < kUnitCols / 128; ++i) {
      const int kk = 4 * (lane + 32 * i);
      wv[i] = (u < P.nunits && e < P.E && kk < kn)
                  ? __ldg(reinterpret_cast<const float4*>(P.Wr + (size_t)e * H + k0 + kk))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  // this CTA's first router unit (take_unit): its fp32 rows load before the wait
  __shared__ int s_unit;
  if (t == 0) s_unit = take_unit(P.ctr, P.nunits, G);
  __syncthreads();
  int u = s_unit;
  load_unit(u);
  // (a grab that races the previous launch's reset finds the queue exhausted
  // or already reset: that launch's CTAs trigger this one's predecessors only
  // after their shared rows)
  int base = 0;
  if (t == 0) {
    base = atomicAdd(&P.ctr[1], 3);
    for (int q = 0; q < 3; ++q)
      if (base + q < P.I) {
        request_l2(P.Wg + (size_t)(base + q) * H, (size_t)H * 2);
        request_l2(P.Wu + (size_t)(base + q) * H, (size_t)H * 2);
      }
  }
  uint4 gv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = t + kThreads * i;
    gv[i] = (P.gamma != nullptr && v < H8) ? *reinterpret_cast<const uint4*>(P.gamma + (size_t)v * 8)
                                           : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();

  // RMSNorm of the M rows (each row's sum of squares in the RMSNorm kernel's order)
  norm_rows<VPT, MT>(P.h1, M, P.gamma != nullptr, gv, P.eps, H, sx, s_norm, nullptr);
  int pending = base + 2;  // (thread 0)
  __syncthreads();

  if (t == 0) {
    s_row[0] = base;
    s_row[1] = base + 1;
  }
  // Router units for every token: the CTA's ticket, then further tickets
  // while units remain. Every computed unit arrives on the hand-off (ctr[0]
  // counts units); the arrival that completes the last unit takes the top-k.
  for (;;) {
    if (u < P.nunits) {
      const int e = (u % ngrp) * 8 + warp, ks = u / ngrp, k0 = ks * kUnitCols;
      const int kn = min(kUnitCols, H - k0);
      float acc[MT];
#pragma unroll
      for (int q = 0; q < MT; ++q) acc[q] = 0.f;
#pragma unroll
      for (int i = 0; i < kUnitCols / 128; ++i) {
        const int kk = 4 * (lane + 32 * i);
        if (kk < kn) {
#pragma unroll
          for (int q = 0; q < MT; ++q) {
            if (q < M) {
              const uint2 xv = *reinterpret_cast<const uint2*>(&sx[(size_t)q * H + k0 + kk]);
              float a = acc[q];
              a = fmaf(wv[i].x, bf_lo(xv.x), a);
              a = fmaf(wv[i].y, bf_hi(xv.x), a);
              a = fmaf(wv[i].z, bf_lo(xv.y), a);
              a = fmaf(wv[i].w, bf_hi(xv.y), a);
              acc[q] = a;
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < MT; ++q) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
        if (lane == 0 && e < P.E && q < M) P.parts[((size_t)ks * M + q) * P.E + e] = acc[q];
      }
    }
    __syncthreads();  // the unit's stores before thread 0's acquire-release add
    if (t == 0) {
      s_last = u < P.nunits && atom_add_acq_rel_gpu(&P.ctr[0], 1) == P.nunits - 1;
      s_unit = u < P.nunits ? take_unit(P.ctr, P.nunits, G) : P.nunits;
    }
    __syncthreads();
    if (s_last) {
      block_topk_tokens<J, MT>(P.parts, ksplit, M, P.E, P.k, P.idx, P.w, P.scores, P.table);
      __syncthreads();  // every warp's entries are written before the release
      if (t == 0) {
        P.ctr[0] = 0;
        P.ctr[5] = c;                  // this CTA's static share goes to the tail queue
        st_release_gpu(&P.ctr[3], 1);  // the routing is written
      }
    }
    u = s_unit;
    if (u >= P.nunits) break;  // (the last arrival's next ticket is always past the units)
    load_unit(u);
  }

  uint4 wa[2][VPT];
  auto load_rows = [&](uint4(&wr)[2][VPT], const uint16_t* g0, const uint16_t* u0) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kThreads * i;
        wr[a][i] = v < H8 ? ld_stream((a == 0 ? g0 : u0) + (size_t)v * 8, pol) : make_uint4(0, 0, 0, 0);
      }
  };
  auto shift = [&](const uint4(&wb)[2][VPT]) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int i = 0; i < VPT; ++i) wa[a][i] = wb[a][i];
  };
  int buf = 0;
  const int I = P.I;
  {  // the shared expert's rows, each applied to the M rows
    int cur = s_row[0], nxt = s_row[1];
    if (cur < I) load_rows(wa, P.Wg + (size_t)cur * H, P.Wu + (size_t)cur * H);
    while (cur < I) {
      uint4 wb[2][VPT];
      if (nxt < I) load_rows(wb, P.Wg + (size_t)nxt * H, P.Wu + (size_t)nxt * H);
      float g[MT], up[MT];
#pragma unroll
      for (int q = 0; q < MT; ++q) {
        g[q] = 0.f;
        up[q] = 0.f;
        if (q < M) {
#pragma unroll
          for (int i = 0; i < VPT; ++i) {
            const int v = t + kThreads * i;
            if (v < H8) {
              const uint4 xv = *reinterpret_cast<const uint4*>(&sx[(size_t)q * H + v * 8]);
              g[q] = dot8(wa[0][i], xv, g[q]);
              up[q] = dot8(wa[1][i], xv, up[q]);
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          g[q] += __shfl_xor_sync(0xffffffffu, g[q], o);
          up[q] += __shfl_xor_sync(0xffffffffu, up[q], o);
        }
        if (lane == 0) {
          red[buf][warp][2 * q] = g[q];
          red[buf][warp][2 * q + 1] = up[q];
        }
      }
      if (t == 0) {
        s_next[buf] = pending;
        if (pending < I) {
          request_l2(P.Wg + (size_t)pending * H, (size_t)H * 2);
          request_l2(P.Wu + (size_t)pending * H, (size_t)H * 2);
          pending = atomicAdd(&P.ctr[1], 1);
        }
      }
      __syncthreads();
      if (t < M) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
          gs += red[buf][w][2 * t];
          us += red[buf][w][2 * t + 1];
        }
        P.hs[(size_t)t * I + cur] = swiglu_bf16(gs, us);
      }
      const int nn = s_next[buf];
      cur = nxt;
      nxt = nn;
      shift(wb);
      buf ^= 1;
    }
  }

  // the routing
  __shared__ const uint16_t* s_g[32];
  __shared__ const uint16_t* s_u[32];
  if (t == 0) {
    // Cross-layer prefetch: a CTA that reaches the wait pulls its slice of the
    // next operator's weights into L2 (memory otherwise idle until the routing).
    if (P.pf_bytes > 0) {
      const size_t off = (size_t)c * P.pf_per;
      if (off < P.pf_bytes) {
        const size_t n = P.pf_bytes - off < P.pf_per ? P.pf_bytes - off : P.pf_per;
        request_l2(P.pf + off, n);
      }
    }
    const unsigned long long t0 = globaltimer();
    int ok = 1;
    while (ld_acquire_gpu(&P.ctr[3]) == 0) {
      if (globaltimer() - t0 > P.wait_ns) {
        atomicOr(P.err, DEV_ERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    s_ok = ok;
  }
  __syncthreads();
  if (s_ok) {
    __shared__ int s_tb, s_cstar;
    const int n = M * P.k;  // entries
    if (t < n) {
      const long long e = ld_cg_s32(P.table + TableLayout(P.E, n).expert() + t);
      s_g[t] = P.Wgb + e * I * H;
      s_u[t] = P.Wub + e * I * H;
    }
    if (t == 0) s_cstar = ld_cg_s32(&P.ctr[5]);
    __syncthreads();
    pdl_trigger();
    const int T = n * I;
    const int bulk = T * 7 / 8 / G, tail0 = G * bulk;
    const int cstar = s_cstar;
    auto tail_row = [&](int v) { return v < bulk ? cstar * bulk + v : tail0 + v - bulk; };
    const int ntail = bulk + T - tail0;
    // one routed row pair: the dot products with its entry's token row, reduced and stored
    auto routed_step = [&](int q, int e) {
      const uint16_t* xrow = sx + (size_t)(e / P.k) * H;
      float g = 0.f, up = 0.f;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kThreads * i;
        const uint4 xv = v < H8 ? *reinterpret_cast<const uint4*>(&xrow[v * 8]) : make_uint4(0, 0, 0, 0);
        g = dot8(wa[0][i], xv, g);
        up = dot8(wa[1][i], xv, up);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        g += __shfl_xor_sync(0xffffffffu, g, o);
        up += __shfl_xor_sync(0xffffffffu, up, o);
      }
      if (lane == 0) {
        red[buf][warp][0] = g;
        red[buf][warp][1] = up;
      }
      __syncthreads();
      if (t == 0) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
          gs += red[buf][w][0];
          us += red[buf][w][1];
        }
        P.hbuf[q] = swiglu_bf16(gs, us);
      }
      buf ^= 1;
    };
    auto rows = [&](int q, const uint16_t*& g0, const uint16_t*& u0) {
      const int e = q / I, r = q - e * I;
      g0 = s_g[e] + (size_t)r * H;
      u0 = s_u[e] + (size_t)r * H;
    };
    int tb = 0;  // (thread 0) the first of three tail rows grabbed together, published in s_tb
    const int q0 = c * bulk, q1 = c == cstar ? q0 : q0 + bulk;
    if (q1 - q0 < 4) {
      if (t == 0) {
        tb = atomicAdd(&P.ctr[4], 3);
        s_tb = tb;
      }
      __syncthreads();
    }
    bool wa_loaded = false;
    if (q0 < q1) {  // this CTA's static share
      int e = q0 / I, r = q0 - (q0 / I) * I;
      load_rows(wa, s_g[e] + (size_t)r * H, s_u[e] + (size_t)r * H);
      for (int q = q0; q < q1; ++q) {
        int en = e, rn = r + 1;
        if (rn == I) {
          ++en;
          rn = 0;
        }
        uint4 wb[2][VPT];
        if (q + 1 < q1) {
          load_rows(wb, s_g[en] + (size_t)rn * H, s_u[en] + (size_t)rn * H);
        } else if (s_tb < ntail) {  // the first tail row follows without a gap
          const uint16_t *g0, *u0;
          rows(tail_row(s_tb), g0, u0);
          load_rows(wb, g0, u0);
          wa_loaded = true;
        }
        if (t == 0) {
          if (q + 2 < q1) {  // the row after next into L2
            const int e2 = rn + 1 == I ? en + 1 : en, r2 = rn + 1 == I ? 0 : rn + 1;
            request_l2(s_g[e2] + (size_t)r2 * H, (size_t)H * 2);
            request_l2(s_u[e2] + (size_t)r2 * H, (size_t)H * 2);
          }
          if (q + 3 == q1 && q1 - q0 >= 4) tb = atomicAdd(&P.ctr[4], 3);  // the tail grab
          if (q + 2 == q1 && q1 - q0 >= 4) {
            s_tb = tb;  // published at this iteration's barrier
            for (int v = tb; v < tb + 2 && v < ntail; ++v) {
              const uint16_t *g2, *u2;
              rows(tail_row(v), g2, u2);
              request_l2(g2, (size_t)H * 2);
              request_l2(u2, (size_t)H * 2);
            }
          }
        }
        routed_step(q, e);
        e = en;
        r = rn;
        shift(wb);
      }
    }
    {  // the tail queue
      const int v0 = s_tb;
      int cur = v0, nxt = v0 + 1;
      if (t == 0) pending = v0 + 2;
      const uint16_t *g0, *u0;
      if (cur < ntail && !wa_loaded) {
        rows(tail_row(cur), g0, u0);
        load_rows(wa, g0, u0);
      }
      while (cur < ntail) {
        uint4 wb[2][VPT];
        if (nxt < ntail) {
          rows(tail_row(nxt), g0, u0);
          load_rows(wb, g0, u0);
        }
        const int b0 = buf;
        if (t == 0) {
          s_next[b0] = pending;
          if (pending < ntail) {
            const uint16_t *g2, *u2;
            rows(tail_row(pending), g2, u2);
            request_l2(g2, (size_t)H * 2);
            request_l2(u2, (size_t)H * 2);
            pending = atomicAdd(&P.ctr[4], 1);
          }
        }
        const int q = tail_row(cur);
        routed_step(q, q / I);
        const int nn = s_next[b0];
        cur = nxt;
        nxt = nn;
        shift(wb);
      }
    }
  }
  if (t == 0 && atom_add_acq_rel_gpu(&P.ctr[2], 1) == G - 1) {
    P.ctr[1] = 0;
    P.ctr[2] = 0;
    P.ctr[3] = 0;
    P.ctr[4] = 0;
  }
}

template <int J>
cudaError_t launch_front_j(dec_handle* h, const RouteSharedParams& P, int vpt, cudaStream_t s) {
  const dim3 g(2 * h->sms), b(kThreads);
  const size_t smem = (size_t)P.H * sizeof(uint16_t);
  if (vpt == 1) return launch_k(h, moe_front_kernel<J, 1>, g, b, smem, s, P);
  if (vpt == 2) return launch_k(h, moe_front_kernel<J, 2>, g, b, smem, s, P);
  return launch_k(h, moe_front_kernel<J, 4>, g, b, smem, s, P);
}

template <int J, int MT>
cudaError_t launch_front_multi(dec_handle* h, const RouteSharedParams& P, int vpt, cudaStream_t s) {
  const dim3 g(2 * h->sms), b(kThreads);
  const size_t smem = (size_t)MT * P.H * sizeof(uint16_t);
  auto go = [&](auto kern) -> cudaError_t {
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    return launch_k(h, kern, g, b, smem, s, P);
  };
  if (vpt == 1) return go(moe_front_multi_kernel<J, 1, MT>);
  if (vpt == 2) return go(moe_front_multi_kernel<J, 2, MT>);
  return go(moe_front_multi_kernel<J, 4, MT>);
}

template <int J, int MT>
cudaError_t launch_multi(dec_handle* h, const RouteSharedParams& P, int vpt, cudaStream_t s) {
  const dim3 g(2 * h->sms), b(kThreads);
  const size_t smem = (size_t)MT * P.H * sizeof(uint16_t);
  auto go = [&](auto kern) -> cudaError_t {
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    return launch_k(h, kern, g, b, smem, s, P);
  };
  if (vpt == 1) return go(route_shared_multi_kernel<J, 1, MT>);
  if (vpt == 2) return go(route_shared_multi_kernel<J, 2, MT>);
  return go(route_shared_multi_kernel<J, 4, MT>);
}

}  // namespace

// Rows of up to 8192 elements (four vectors per thread); E up to 1024; at
// most two router units per CTA; up to 4 tokens (their normalised rows in
// shared memory, two CTAs per SM).
bool route_shared_supported(const dec_handle* h, int M, int H, int E, int k) {
  const long long units = (long long)((E + 7) / 8) * ((H + kUnitCols - 1) / kUnitCols);
  return M >= 1 && M <= 4 && H >= 8 && H % 8 == 0 && H <= 8 * 4 * kThreads && E >= 1 && E <= 1024 && k >= 1 &&
         k <= 16 && k <= E && units <= 2LL * 2 * h->sms && (size_t)(M <= 1 ? 1 : (M <= 2 ? 2 : 4)) * H * 2 <= 100000;
}

cudaError_t launch_route_shared(dec_handle* h, int M, const uint16_t* h1, const uint16_t* gamma, float eps,
                                const float* Wr, int H, int E, int k, uint16_t* xn, float* parts, int* ctr,
                                int32_t* idx, float* w, float* scores, int* table, const uint16_t* Wg_s,
                                const uint16_t* Wu_s, int I, uint16_t* hs, cudaStream_t s) {
  if (M < 2 || !route_shared_supported(h, M, H, E, k)) return cudaErrorInvalidValue;  // (one token: router_select)
  RouteSharedParams P;
  P.M = M;
  P.h1 = h1;
  P.gamma = gamma;
  P.eps = eps;
  P.Wr = Wr;
  P.H = H;
  P.E = E;
  P.k = k;
  P.nunits = ((E + 7) / 8) * ((H + kUnitCols - 1) / kUnitCols);
  P.xn = xn;
  P.parts = parts;
  P.ctr = ctr;
  P.idx = idx;
  P.w = w;
  P.scores = scores;
  P.table = table;
  P.Wg = Wg_s;
  P.Wu = Wu_s;
  P.I = I;
  P.hs = hs;
  const int H8 = H / 8, vpt = H8 <= kThreads ? 1 : (H8 <= 2 * kThreads ? 2 : 4);
  const int Ew = (E + 7) / 8;
  if (M == 2) {
    if (Ew <= 32) return launch_multi<1, 2>(h, P, vpt, s);
    if (Ew <= 64) return launch_multi<2, 2>(h, P, vpt, s);
    return launch_multi<4, 2>(h, P, vpt, s);
  }
  if (Ew <= 32) return launch_multi<1, 4>(h, P, vpt, s);
  if (Ew <= 64) return launch_multi<2, 4>(h, P, vpt, s);
  return launch_multi<4, 4>(h, P, vpt, s);
}

cudaError_t launch_moe_front(dec_handle* h, const uint16_t* h1, const uint16_t* gamma, float eps, const float* Wr,
                             int H, int E, int k, float* parts, int* ctr, int32_t* idx, float* w, float* scores,
                             int* table, const uint16_t* Wg_s, const uint16_t* Wu_s, int I, uint16_t* hs,
                             const uint16_t* Wg, const uint16_t* Wu, uint16_t* hbuf, cudaStream_t s, const void* pf,
                             size_t pf_bytes) {
  if (!route_shared_supported(h, 1, H, E, k) || Wg_s == nullptr || k > 32) return cudaErrorInvalidValue;
  RouteSharedParams P;
  P.M = 1;
  P.h1 = h1;
  P.gamma = gamma;
  P.eps = eps;
  P.Wr = Wr;
  P.H = H;
  P.E = E;
  P.k = k;
  P.nunits = ((E + 7) / 8) * ((H + kUnitCols - 1) / kUnitCols);
  P.xn = nullptr;
  P.parts = parts;
  P.ctr = ctr;
  P.idx = idx;
  P.w = w;
  P.scores = scores;
  P.table = table;
  P.Wg = Wg_s;
  P.Wu = Wu_s;
  P.I = I;
  P.hs = hs;
  P.Wgb = Wg;
  P.Wub = Wu;
  P.hbuf = hbuf;
  P.err = h->d_err;
  P.wait_ns = h->wait_ns;
  P.pf = static_cast<const char*>(pf);
  P.pf_bytes = pf != nullptr ? pf_bytes : 0;
  P.pf_per = (P.pf_bytes / (2 * h->sms) + 15) / 16 * 16;
  const int H8 = H / 8, vpt = H8 <= kThreads ? 1 : (H8 <= 2 * kThreads ? 2 : 4);
  const int Ew = (E + 7) / 8;
  if (Ew <= 32) return launch_front_j<1>(h, P, vpt, s);
  if (Ew <= 64) return launch_front_j<2>(h, P, vpt, s);
  return launch_front_j<4>(h, P, vpt, s);
}

cudaError_t launch_moe_front_multi(dec_handle* h, int M, const uint16_t* h1, const uint16_t* gamma, float eps,
                                   const float* Wr, int H, int E, int k, float* parts, int* ctr, int32_t* idx, float* w,
                                   float* scores, int* table, const uint16_t* Wg_s, const uint16_t* Wu_s, int I,
                                   uint16_t* hs, const uint16_t* Wg, const uint16_t* Wu, uint16_t* hbuf,
                                   cudaStream_t s, const void* pf, size_t pf_bytes) {
  if (M < 2 || M > 4 || !route_shared_supported(h, M, H, E, k) || Wg_s == nullptr || M * k > 32)
    return cudaErrorInvalidValue;
  RouteSharedParams P;
  P.M = M;
  P.h1 = h1;
  P.gamma = gamma;
  P.eps = eps;
  P.Wr = Wr;
  P.H = H;
  P.E = E;
  P.k = k;
  P.nunits = ((E + 7) / 8) * ((H + kUnitCols - 1) / kUnitCols);
  P.xn = nullptr;
  P.parts = parts;
  P.ctr = ctr;
  P.idx = idx;
  P.w = w;
  P.scores = scores;
  P.table = table;
  P.Wg = Wg_s;
  P.Wu = Wu_s;
  P.I = I;
  P.hs = hs;
  P.Wgb = Wg;
  P.Wub = Wu;
  P.hbuf = hbuf;
  P.err = h->d_err;
  P.wait_ns = h->wait_ns;
  P.pf = static_cast<const char*>(pf);
  P.pf_bytes = pf != nullptr ? pf_bytes : 0;
  P.pf_per = (P.pf_bytes / (2 * h->sms) + 15) / 16 * 16;
  const int H8 = H / 8, vpt = H8 <= kThreads ? 1 : (H8 <= 2 * kThreads ? 2 : 4);
  const int Ew = (E + 7) / 8;
  if (M == 2) {
    if (Ew <= 32) return launch_front_multi<1, 2>(h, P, vpt, s);
    if (Ew <= 64) return launch_front_multi<2, 2>(h, P, vpt, s);
    return launch_front_multi<4, 2>(h, P, vpt, s);
  }
  if (Ew <= 32) return launch_front_multi<1, 4>(h, P, vpt, s);
  if (Ew <= 64) return launch_front_multi<2, 4>(h, P, vpt, s);
  return launch_front_multi<4, 4>(h, P, vpt, s);
}

}  // namespace dec
