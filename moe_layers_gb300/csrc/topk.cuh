// Block-wide top-k of one token's router logits (used by the top-k kernel
// and by the one-token routing launches). Requires 256 threads.
#pragma once
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace dec {

constexpr int kTopkSplitsInRegs = 16;  // split partials per expert loaded together (H <= 16384)

// Top-k of token t, one 256-thread block. logits = sum of the split partials
// in split order, s = 1 / (1 + exp(-logit)). Each of the 8 warps takes a
// contiguous eighth of the experts (J per lane, in registers), keeps its local
// top-k by k rounds of warp arg-max (score descending, expert id ascending),
// and warp 0 merges the 8k candidates the same way; weights are the selected
// scores over their sum. All partial-sum loads are issued before any is used.
// CG: read the partials at L2 (written by other CTAs of the running kernel).
// On return lane r < k of warp 0 holds the r-th selection in *sel_e, *sel_w.
template <int J, bool CG>
__device__ __forceinline__ void block_topk(const float* parts, int ks, int M, int t, int E, int k, int32_t* idx,
                                           float* w, float* scores, int* sel_e, float* sel_w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Ew = (E + 7) / 8;
  __shared__ float cv[8][16];
  __shared__ int ci[8][16];
  float sv[J];
  int ev[J];
  bool ok[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int off = lane + 32 * j;
    ev[j] = warp * Ew + off;
    ok[j] = off < Ew && ev[j] < E;
    sv[j] = 0.f;
  }
  auto ld = [&](const float* p) { return CG ? ld_cg_f32(p) : ld_act_f32(p); };
  for (int s0 = 0; s0 < ks; s0 += kTopkSplitsInRegs) {
    float tmp[kTopkSplitsInRegs][J];
#pragma unroll
    for (int q = 0; q < kTopkSplitsInRegs; ++q)
#pragma unroll
      for (int j = 0; j < J; ++j)
        tmp[q][j] = (s0 + q < ks && ok[j]) ? ld(parts + ((size_t)(s0 + q) * M + t) * E + ev[j]) : 0.f;
#pragma unroll
    for (int q = 0; q < kTopkSplitsInRegs; ++q)
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (s0 + q < ks) sv[j] += tmp[q][j];
  }
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (ok[j]) {
      sv[j] = 1.0f / (1.0f + expf(-sv[j]));
      if (scores != nullptr) scores[(size_t)t * E + ev[j]] = sv[j];
    } else {
      sv[j] = -FLT_MAX;
      ev[j] = INT_MAX;
    }
  }
  // k rounds of warp arg-max; returns the r-th selection in lane r.
  auto select = [&](float* v, int* id, int n, float& out_v, int& out_i) {
    for (int r = 0; r < k; ++r) {
      float bv = -FLT_MAX;
      int bi = INT_MAX;
      for (int j = 0; j < n; ++j)
        if (v[j] > bv || (v[j] == bv && id[j] < bi)) {
          bv = v[j];
          bi = id[j];
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      for (int j = 0; j < n; ++j)
        if (id[j] == bi) v[j] = -FLT_MAX;  // ids are unique: only the owner matches
      if (lane == r) {
        out_v = bv;
        out_i = bi;
      }
    }
  };
  float mv = -FLT_MAX;
  int mi = INT_MAX;
  select(sv, ev, J, mv, mi);
  if (lane < k) {
    cv[warp][lane] = mv;
    ci[warp][lane] = mi;
  }
  __syncthreads();
  if (warp == 0) {
    // the 8k candidates, up to four per lane
    float v2[4];
    int i2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = lane + 32 * j;  // candidate index in [0, 8k)
      const int wq = q / k, rq = q - wq * k;
      const bool okq = q < 8 * k;
      v2[j] = okq ? cv[wq][rq] : -FLT_MAX;
      i2[j] = okq ? ci[wq][rq] : INT_MAX;
    }
    float fv = 0.f;
    int fi = 0;
    select(v2, i2, 4, fv, fi);
    float sum = 0.f;
    for (int r = 0; r < k; ++r) sum += __shfl_sync(0xffffffffu, fv, r);
    if (lane < k) {
      idx[(size_t)t * k + lane] = fi;
      w[(size_t)t * k + lane] = fv / sum;
      *sel_e = fi;
      *sel_w = fv / sum;
    }
  }
}

}  // namespace dec

namespace dec {

// One token: the routing table with entry j as problem j on slot j, expert
// sel_e of lane j (< k) of warp 0, U = k. Called by warp 0 only.
__device__ __forceinline__ void write_one_token_table(int* table, int E, int k, int sel_e) {
  const int lane = threadIdx.x & 31;
  const TableLayout L(E, k);
  if (lane < k) {
    table[L.expert() + lane] = sel_e;
    table[L.offset() + lane] = lane;
    table[L.count() + lane] = 1;
    table[L.slot_token() + lane] = 0;
    table[L.entry_slot() + lane] = lane;
  }
  if (lane == 0) table[L.U()] = k;
}

}  // namespace dec

namespace dec {

// Top-k of token t by one warp (up to 8 tokens of a CTA in parallel). Lane l
// holds the experts l, l + 32, ... (JW >= E / 32 per lane). logits = sum of
// the split partials in split order (read at L2: other CTAs wrote them),
// s = 1 / (1 + exp(-logit)), k rounds of warp arg-max (score descending,
// expert id ascending), weights = selected scores over their sum: the rule
// and arithmetic of block_topk. On return lane r < k holds the r-th selection
// in *sel_e, *sel_w (idx, w, scores are written here).
template <int JW>
__device__ __forceinline__ void warp_topk(const float* parts, int ks, int M, int t, int E, int k, int32_t* idx,
                                          float* w, float* scores, int* sel_e, float* sel_w) {
  const int lane = threadIdx.x & 31;
  float sv[JW];
  int ev[JW];
#pragma unroll
  for (int i = 0; i < JW; ++i) {
    ev[i] = lane + 32 * i;
    sv[i] = 0.f;
  }
  for (int s = 0; s < ks; ++s) {
#pragma unroll
    for (int i = 0; i < JW; ++i)
      if (ev[i] < E) sv[i] += __ldcg(parts + ((size_t)s * M + t) * E + ev[i]);
  }
#pragma unroll
  for (int i = 0; i < JW; ++i) {
    if (ev[i] < E) {
      sv[i] = 1.0f / (1.0f + expf(-sv[i]));
      if (scores != nullptr) scores[(size_t)t * E + ev[i]] = sv[i];
    } else {
      sv[i] = -FLT_MAX;
      ev[i] = INT_MAX;
    }
  }
  float fv = 0.f;
  int fi = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < JW; ++i)
      if (sv[i] > bv || (sv[i] == bv && ev[i] < bi)) {
        bv = sv[i];
        bi = ev[i];
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
#pragma unroll
    for (int i = 0; i < JW; ++i)
      if (ev[i] == bi) sv[i] = -FLT_MAX;  // ids are unique: only the owner matches
    if (lane == r) {
      fv = bv;
      fi = bi;
    }
  }
  float sum = 0.f;
  for (int r = 0; r < k; ++r) sum += __shfl_sync(0xffffffffu, fv, r);
  if (lane < k) {
    idx[(size_t)t * k + lane] = fi;
    w[(size_t)t * k + lane] = fv / sum;
  }
  *sel_e = fi;
  *sel_w = fv / sum;
}

// M tokens: the routing table with entry p = t * k + j as problem p on slot p
// (expert idx[t][j], token t), U = M * k. Called by warp t for its token.
__device__ __forceinline__ void write_entry_table(int* table, int E, int M, int k, int t, int sel_e) {
  const int lane = threadIdx.x & 31;
  const TableLayout L(E, M * k);
  if (lane < k) {
    const int p = t * k + lane;
    table[L.expert() + p] = sel_e;
    table[L.offset() + p] = p;
    table[L.count() + p] = 1;
    table[L.slot_token() + p] = t;
    table[L.entry_slot() + p] = p;
  }
  if (t == 0 && lane == 0) table[L.U()] = M * k;
}

}  // namespace dec
