// Router top-k: the routing-table writers, a warp-level selection, and the
// block-wide top-k of one token (the top-k kernel, the one-token routing
// launches) or of up to four tokens (the few-token routing launch). The block
// functions require 256 threads.
#pragma once
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace dec {

constexpr int kTopkSplitsInRegs = 16;  // split partials per expert loaded together (H <= 16384)

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

// Grouped routing table from the n = M k entries eidx[i] (entry i = token
// i / k, choice i % k) held in shared memory, by a 256-thread block: per
// active expert (ascending id) its first slot and token count; slots ordered
// by (expert, token, choice). Shared scratch: cnt, off, run [E] and stok,
// eslot [n] ints. write: this block writes the table out. On return
// stok[slot] is the slot's token for every thread of the block.
__device__ __forceinline__ void block_route_table(const int* eidx, int n, int k, int E, int* cnt, int* off, int* run,
                                                  int* stok, int* eslot, int* table, bool write) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const TableLayout L(E, n);
  for (int e = tid; e < E; e += blockDim.x) {
    cnt[e] = 0;
    run[e] = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) atomicAdd(&cnt[eidx[i]], 1);
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int s_sum = 0, a_sum = 0;
    for (int e = e0; e < e1; ++e) {
      s_sum += cnt[e];
      a_sum += cnt[e] > 0 ? 1 : 0;
    }
    int s_inc = s_sum, a_inc = a_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vs = __shfl_up_sync(0xffffffffu, s_inc, o);
      const int va = __shfl_up_sync(0xffffffffu, a_inc, o);
      if (lane >= o) {
        s_inc += vs;
        a_inc += va;
      }
    }
    int s_run = s_inc - s_sum, a_run = a_inc - a_sum;
    for (int e = e0; e < e1; ++e) {
      off[e] = s_run;
      if (cnt[e] > 0) {
        if (write) {
          table[L.expert() + a_run] = e;
          table[L.offset() + a_run] = s_run;
          table[L.count() + a_run] = cnt[e];
        }
        ++a_run;
      }
      s_run += cnt[e];
    }
    if (lane == 31 && write) table[L.U()] = a_inc;
  }
  __syncthreads();
  if (warp == 0) {
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const bool valid = i < n;
      const int e = valid ? eidx[i] : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (valid) {
        const int slot = off[e] + run[e] + rank;
        eslot[i] = slot;
        stok[slot] = i / k;
      }
      __syncwarp();
      if (valid && rank == 0) run[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  if (write) {
    for (int i = tid; i < n; i += blockDim.x) {
      table[L.slot_token() + i] = stok[i];
      table[L.entry_slot() + i] = eslot[i];
    }
  }
}

// k rounds of arg-max over E scores in shared memory (score descending,
// expert id ascending), by one warp: lane l holds experts l, l + 32, ... (JW
// per lane, E <= 32 JW). Each round takes the lane's best (a strict > over
// ascending ids keeps the lowest id among equal scores), then one warp max of
// the scores' bit patterns (positive floats order as their bits; +1 keeps 0
// for "taken") and one warp min of the ids that reach it; the owner clears the
// winner. Lane r < k returns the r-th selection in fv, fi; weights are the
// selected scores over their sum, added in selection order. (block_topk below
// runs the same selection inline.)
template <int JW>
__device__ __forceinline__ void warp_select(const float* sc, int E, int k, float& fv, int& fi, float& wt) {
  const int lane = threadIdx.x & 31;
  unsigned key[JW];
#pragma unroll
  for (int i = 0; i < JW; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? __float_as_uint(sc[e]) + 1u : 0u;
  }
  fv = 0.f;
  fi = 0;
  for (int r = 0; r < k; ++r) {
    unsigned bk = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < JW; ++i)
      if (key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    const unsigned m = __reduce_max_sync(0xffffffffu, bk);
    const unsigned win = __reduce_min_sync(0xffffffffu, bk == m && m != 0u ? (unsigned)(lane + 32 * bi) : 0xffffffffu);
    const bool owner = (int)(win & 31u) == lane;
    const int slot = (int)(win >> 5);
#pragma unroll
    for (int i = 0; i < JW; ++i) key[i] = (owner && i == slot) ? 0u : key[i];
    if (lane == r) {
      fv = __uint_as_float(m - 1u);
      fi = (int)win;
    }
  }
  float sum = 0.f;
  for (int r = 0; r < k; ++r) sum += __shfl_sync(0xffffffffu, fv, r);
  wt = fv / sum;
}

// Router scores of tokens t0 .. t0 + nt - 1 (nt <= MT) into shared memory, by
// a 256-thread block: logits = sum of the split partials in split order,
// s = 1 / (1 + exp(-logit)); thread t owns experts t, t + 256, ... (J per
// thread, E <= 256 J) of every token; all of a chunk's partial-sum loads are
// issued before any is used. Partials: parts[(split * M + token) * E + e].
// Writes the scores (when given) and s_sc[m][e] for token t0 + m. CG: read
// the partials at L2 (written by other CTAs of the running kernel).
template <int J, int MT, bool CG>
__device__ __forceinline__ void block_scores(const float* parts, int ks, int M, int t0, int nt, int E,
                                             float* scores, float (*s_sc)[256 * J]) {
  constexpr int KS = MT == 1 ? kTopkSplitsInRegs : 8;  // splits per chunk
  const int tid = threadIdx.x;
  float sv[MT][J];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < J; ++j) sv[m][j] = 0.f;
  auto ld = [&](const float* p) { return CG ? ld_cg_f32(p) : ld_act_f32(p); };
  for (int s0 = 0; s0 < ks; s0 += KS) {
    float tmp[KS][MT][J];
#pragma unroll
    for (int q = 0; q < KS; ++q)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int e = tid + 256 * j;
          tmp[q][m][j] = (s0 + q < ks && m < nt && e < E) ? ld(parts + ((size_t)(s0 + q) * M + t0 + m) * E + e) : 0.f;
        }
#pragma unroll
    for (int q = 0; q < KS; ++q)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (s0 + q < ks) sv[m][j] += tmp[q][m][j];
  }
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = tid + 256 * j;
      if (m < nt && e < E) {
        const float sc = sigmoid_f(sv[m][j]);
        if (scores != nullptr) scores[(size_t)(t0 + m) * E + e] = sc;
        s_sc[m][e] = sc;
      }
    }
}

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
      const float sc = sigmoid_f(sv[j]);
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

// Top-k of the M <= MT tokens of a batch, one 256-thread block: the scores of
// all tokens (block_scores), then warp m selects token m's k experts
// (warp_select) and writes idx, w and its k entries of the routing table (one
// problem per entry, write_entry_table). The rule and arithmetic of
// block_topk, token by token.
template <int J, int MT>
__device__ __forceinline__ void block_topk_tokens(const float* parts, int ks, int M, int E, int k, int32_t* idx,
                                                  float* w, float* scores, int* table) {
  __shared__ float s_sc[MT][256 * J];
  block_scores<J, MT, true>(parts, ks, M, 0, M, E, scores, s_sc);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < M) {
    float fv, wt;
    int fi;
    warp_select<8 * J>(s_sc[warp], E, k, fv, fi, wt);
    if (lane < k) {
      idx[(size_t)warp * k + lane] = fi;
      w[(size_t)warp * k + lane] = wt;
    }
    write_entry_table(table, E, M, k, warp, fi);
  }
}

}  // namespace dec

