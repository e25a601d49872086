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
// in split order, s = 1 / (1 + exp(-logit)) (thread t owns experts t, t + 256,
// ...; all partial-sum loads are issued before any is used). Warp 0 then
// selects over all E scores from shared memory (lane l holds experts l,
// l + 32, ...): k rounds of arg-max (score descending, expert id ascending),
// each round one warp max of the scores' bit patterns (positive floats order
// as their bits; +1 keeps 0 for "taken") and one warp min of the ids that
// reach it. Weights are the selected scores over their sum. CG: read the
// partials at L2 (written by other CTAs of the running kernel). On return
// lane r < k of warp 0 holds the r-th selection in *sel_e, *sel_w.
template <int J, bool CG>
__device__ __forceinline__ void block_topk(const float* parts, int ks, int M, int t, int E, int k, int32_t* idx,
                                           float* w, float* scores, int* sel_e, float* sel_w) {
  constexpr int JT = J;      // experts per thread (E <= 256 J)
  constexpr int JW = 8 * J;  // experts per lane of warp 0
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float s_sc[256 * J];
  float sv[JT];
#pragma unroll
  for (int j = 0; j < JT; ++j) sv[j] = 0.f;
  auto ld = [&](const float* p) { return CG ? ld_cg_f32(p) : ld_act_f32(p); };
  for (int s0 = 0; s0 < ks; s0 += kTopkSplitsInRegs) {
    float tmp[kTopkSplitsInRegs][JT];
#pragma unroll
    for (int q = 0; q < kTopkSplitsInRegs; ++q)
#pragma unroll
      for (int j = 0; j < JT; ++j) {
        const int e = tid + 256 * j;
        tmp[q][j] = (s0 + q < ks && e < E) ? ld(parts + ((size_t)(s0 + q) * M + t) * E + e) : 0.f;
      }
#pragma unroll
    for (int q = 0; q < kTopkSplitsInRegs; ++q)
#pragma unroll
      for (int j = 0; j < JT; ++j)
        if (s0 + q < ks) sv[j] += tmp[q][j];
  }
#pragma unroll
  for (int j = 0; j < JT; ++j) {
    const int e = tid + 256 * j;
    if (e < E) {
      const float sc = 1.0f / (1.0f + expf(-sv[j]));
      if (scores != nullptr) scores[(size_t)t * E + e] = sc;
      s_sc[e] = sc;
    }
  }
  __syncthreads();
  if (warp == 0) {
    unsigned key[JW];
#pragma unroll
    for (int i = 0; i < JW; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? __float_as_uint(s_sc[e]) + 1u : 0u;
    }
    float fv = 0.f;
    int fi = 0;
    for (int r = 0; r < k; ++r) {
      unsigned bk = 0u;
      int bi = 0;
#pragma unroll
      for (int i = 0; i < JW; ++i)
        if (key[i] > bk) {  // strict: the lowest id among a lane's equal scores
          bk = key[i];
          bi = i;
        }
      const unsigned m = __reduce_max_sync(0xffffffffu, bk);
      const unsigned win = __reduce_min_sync(0xffffffffu, bk == m && m != 0u ? (unsigned)(lane + 32 * bi) : 0xffffffffu);
      if ((int)(win & 31u) == lane) {
#pragma unroll
        for (int i = 0; i < JW; ++i)
          if (i == (int)(win >> 5)) key[i] = 0u;
      }
      if (lane == r) {
        fv = __uint_as_float(m - 1u);
        fi = (int)win;
      }
    }
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
