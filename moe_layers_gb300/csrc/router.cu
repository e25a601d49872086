// MoE routing: router scores, top-k, the per-expert routing table (with the
// gather of each expert's tokens into contiguous rows), and the final
// weighted combine.
//
// Kimi K3 article, Part 1 §3 "Mejorar la programación de MoE": router scores
// are computed before the experts run, and the expert schedule decides which
// weights are read. The rule (sigmoid scores of fp32 router weights, top-k by
// score with ties to the lower id, weights renormalised over the selected k)
// is the workload's; the pages give no formula.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace dec {

constexpr int kRouterChunk = 1024;  // reduction elements per split (one CTA column)
constexpr int kRouterRows = 8;      // router rows per CTA, one per warp
constexpr int kRouterTok = 4;       // tokens staged in shared memory per pass (8 KB: co-resides with the engine)
// Tokens per CTA (grid z; build-time tunable). Measured (layer step, one box):
// groups of 16 tokens make the router launch faster at 64 tokens (34.0 against
// 40.9 us event-timed) but the step slower at 32 (2418.3 against 2405.4 us):
// the extra CTAs compete for SMs with the shared expert on the side stream.
#ifndef DEC_ROUTER_GROUP
#define DEC_ROUTER_GROUP 64
#endif
constexpr int kRouterGroup = DEC_ROUTER_GROUP;

int router_ksplit(int H) { return (H + kRouterChunk - 1) / kRouterChunk; }

// parts[ks][t][e] = sum over the ks-th chunk of H of x[t][h] * Wr[e][h] (fp32).
// Grid: (ceil(E / 8), ksplit, ceil(M / kRouterGroup)). Each warp owns one
// router row and keeps its chunk of fp32 weights in registers (loaded before
// the dependency wait); the CTA's group of tokens passes through shared
// memory four at a time, the next four tokens' activations loaded into
// registers while the current four are multiplied. Every partial sum is the
// same whatever the grid: the token groups only spread the work over more
// CTAs (the router matrix, 11 MB at the workload's size, is re-read from L2).
__global__ void __launch_bounds__(256) router_kernel(const uint16_t* x, const float* __restrict__ Wr, int M, int H,
                                                     int E, float* parts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterRows + warp;
  const int ks = blockIdx.y;
  const int k0 = ks * kRouterChunk;
  const int kn = min(kRouterChunk, H - k0);
  const int tg0 = blockIdx.z * kRouterGroup, tg1 = min(M, tg0 + kRouterGroup);
  __shared__ __align__(16) uint16_t xs[kRouterTok][kRouterChunk];
  pdl_trigger();
  float4 wv[kRouterChunk / 128];
#pragma unroll
  for (int i = 0; i < kRouterChunk / 128; ++i) {
    const int kk = 4 * (lane + 32 * i);
    wv[i] = (e < E && kk < kn) ? __ldg(reinterpret_cast<const float4*>(Wr + (size_t)e * H + k0 + kk))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  const int kv = kn >> 3;
  // This thread's share of a pass's activation vectors: q = threadIdx.x + 256 j.
  constexpr int kQ = kRouterTok * (kRouterChunk / 8) / 256;
  uint4 xr[kQ];
  auto load_pass = [&](int t0) {
    const int nt = min(kRouterTok, tg1 - t0);
#pragma unroll
    for (int j = 0; j < kQ; ++j) {
      const int q = threadIdx.x + 256 * j;
      const int tt = q / (kRouterChunk / 8), v = q % (kRouterChunk / 8);
      xr[j] = (tt < nt && v < kv) ? ld_act16(x + (size_t)(t0 + tt) * H + k0 + v * 8) : make_uint4(0, 0, 0, 0);
    }
  };
  if (tg0 < tg1) load_pass(tg0);
  for (int t0 = tg0; t0 < tg1; t0 += kRouterTok) {
    const int nt = min(kRouterTok, tg1 - t0);
    __syncthreads();  // the previous pass's readers are done
#pragma unroll
    for (int j = 0; j < kQ; ++j) {
      const int q = threadIdx.x + 256 * j;
      *reinterpret_cast<uint4*>(&xs[q / (kRouterChunk / 8)][(q % (kRouterChunk / 8)) * 8]) = xr[j];
    }
    __syncthreads();
    if (t0 + kRouterTok < tg1) load_pass(t0 + kRouterTok);
    float acc[kRouterTok];
#pragma unroll
    for (int tt = 0; tt < kRouterTok; ++tt) acc[tt] = 0.f;
#pragma unroll
    for (int i = 0; i < kRouterChunk / 128; ++i) {
      const int kk = 4 * (lane + 32 * i);
      if (kk < kn) {
#pragma unroll
        for (int tt = 0; tt < kRouterTok; ++tt) {
          if (tt < nt) {
            const uint2 xv = *reinterpret_cast<const uint2*>(&xs[tt][kk]);
            float a = acc[tt];
            a = fmaf(wv[i].x, bf_lo(xv.x), a);
            a = fmaf(wv[i].y, bf_hi(xv.x), a);
            a = fmaf(wv[i].z, bf_lo(xv.y), a);
            a = fmaf(wv[i].w, bf_hi(xv.y), a);
            acc[tt] = a;
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < kRouterTok; ++tt)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[tt] += __shfl_xor_sync(0xffffffffu, acc[tt], o);
    if (lane == 0 && e < E) {
#pragma unroll
      for (int tt = 0; tt < kRouterTok; ++tt)
        if (tt < nt) parts[((size_t)ks * M + t0 + tt) * E + e] = acc[tt];
    }
  }
}

// One CTA per token (see block_topk).
template <int J>
__global__ void __launch_bounds__(256) topk_kernel(const float* parts, int ks, int M, int E, int k, int32_t* idx,
                                                   float* w, float* scores) {
  pdl_trigger();
  pdl_wait();
  int se;
  float sw;
  block_topk<J, false>(parts, ks, M, blockIdx.x, E, k, idx, w, scores, &se, &sw);
}

// One token: the RMSNorm of the layer's post-attention row, the router logits,
// the top-k and the routing table in one launch (at one token the three
// kernels in a row would each wait on the one before, with the memory idle).
// Grid (ceil(E / 8), ksplit), as router_kernel. Every CTA normalises the row
// itself in the RMSNorm kernel's order (so the normalised row has its bits),
// keeps its chunk of it in shared memory (CTAs of column 0 also write their
// chunk out for the experts) and stores its logit pieces. The last CTA to
// finish (an atomic counter that it resets) runs the top-k and writes the
// routing table of the single token: one problem per selected expert, in
// selection order, problem j on slot j, so every problem reads the same
// normalised row. Without gamma the input row is used as it is.
template <int J>
__global__ void __launch_bounds__(256) router_select_kernel(const uint16_t* xin, const uint16_t* __restrict__ gamma,
                                                            float eps, const float* __restrict__ Wr, int H, int E,
                                                            int k, uint16_t* xn, float* parts, int* counter,
                                                            int32_t* idx, float* w, float* scores, int* table) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e = blockIdx.x * kRouterRows + warp;
  const int ks = blockIdx.y;
  const int k0 = ks * kRouterChunk;
  const int kn = min(kRouterChunk, H - k0);
  const int kv = kn >> 3;
  __shared__ __align__(16) uint16_t xs[kRouterChunk];
  __shared__ float red[8];
  __shared__ int s_last;
  pdl_trigger();
  float4 wv[kRouterChunk / 128];
#pragma unroll
  for (int i = 0; i < kRouterChunk / 128; ++i) {
    const int kk = 4 * (lane + 32 * i);
    wv[i] = (e < E && kk < kn) ? __ldg(reinterpret_cast<const float4*>(Wr + (size_t)e * H + k0 + kk))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // Chunk vector i (of kv) is vector 128 ks + i of the row: in the sum-of-squares
  // pass below thread 128 (ks & 1) + i loads it, as its vector j = ks / 2.
  const int ci = tid & 127;
  const bool owner = (tid >> 7) == (ks & 1) && ci < kv;
  uint4 gv = make_uint4(0, 0, 0, 0);
  if (gamma != nullptr && owner) gv = *reinterpret_cast<const uint4*>(gamma + k0 + (size_t)ci * 8);
  pdl_wait();
  if (gamma != nullptr) {
    // sum of squares over the whole row: up to four vectors per thread loaded
    // together (rows up to 8192), then in ascending order
    const int H8 = H >> 3;
    float ss = 0.f;
    uint4 hv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = tid + 256 * j;
      hv[j] = v < H8 ? ld_act16(xin + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (tid + 256 * j < H8) ss = sumsq8(hv[j], ss);
    for (int v = tid + 1024; v < H8; v += 256) ss = sumsq8(ld_act16(xin + (size_t)v * 8), ss);
    const float r = block_rms_scale<8>(ss, H, eps, red);
    if (owner) {
      const int jj = ks >> 1;
      const uint4 xv = jj == 0 ? hv[0] : jj == 1 ? hv[1] : jj == 2 ? hv[2] : jj == 3 ? hv[3]
                                                                            : ld_act16(xin + k0 + (size_t)ci * 8);
      const uint4 y = norm8(xv, gv, r);
      *reinterpret_cast<uint4*>(&xs[ci * 8]) = y;
      if (blockIdx.x == 0 && xn != nullptr) *reinterpret_cast<uint4*>(xn + k0 + (size_t)ci * 8) = y;
    }
  } else if (tid < kv) {
    *reinterpret_cast<uint4*>(&xs[tid * 8]) = ld_act16(xin + k0 + (size_t)tid * 8);
  }
  __syncthreads();
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kRouterChunk / 128; ++i) {
    const int kk = 4 * (lane + 32 * i);
    if (kk < kn) {
      const uint2 xv = *reinterpret_cast<const uint2*>(&xs[kk]);
      acc = fmaf(wv[i].x, bf_lo(xv.x), acc);
      acc = fmaf(wv[i].y, bf_hi(xv.x), acc);
      acc = fmaf(wv[i].z, bf_lo(xv.y), acc);
      acc = fmaf(wv[i].w, bf_hi(xv.y), acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0 && e < E) parts[(size_t)ks * E + e] = acc;

  // Hand-off to the last CTA: the barrier orders this CTA's stores before
  // thread 0's acquire-release add; in the last CTA the barrier after it
  // orders every thread's reads after the acquire.
  __syncthreads();
  if (tid == 0) s_last = atom_add_acq_rel_gpu(counter, 1) == (int)(gridDim.x * gridDim.y) - 1;
  __syncthreads();
  if (!s_last) return;
  int se = 0;
  float sw = 0.f;
  block_topk<J, true>(parts, gridDim.y, 1, 0, E, k, idx, w, scores, &se, &sw);
  if (table != nullptr && warp == 0) write_one_token_table(table, E, k, se);
  if (tid == 0) *counter = 0;  // leave the workspace reusable
}

// One token: its k entries are k problems, entry j on slot j with expert
// idx[j] (a repeated expert is then simply two problems), U = k. This is the
// table router_select_kernel writes.
__global__ void one_token_table_kernel(const int32_t* idx, int E, int k, int* table) {
  pdl_trigger();
  pdl_wait();
  const TableLayout L(E, k);
  const int j = threadIdx.x;
  if (j < k) {
    table[L.expert() + j] = ld_act_s32(idx + j);
    table[L.offset() + j] = j;
    table[L.count() + j] = 1;
    table[L.slot_token() + j] = 0;
    table[L.entry_slot() + j] = j;
  }
  if (j == 0) table[L.U()] = k;
}

// Routing table from idx[M][k]: per active expert (ascending id) its first
// slot and token count; slots are ordered by (expert, token, j). Every CTA
// rebuilds the table in shared memory (n = M*k <= 1024 entries), CTA 0 writes
// it out, and all CTAs gather x rows into the slot-ordered buffer xs so that
// each expert's tokens are contiguous rows for the TMA loads of the experts.
__global__ void __launch_bounds__(256) route_table_kernel(const int32_t* idx, int M, int k, int E, const uint16_t* x,
                                                          int H, int* table, uint16_t* xs) {
  extern __shared__ int sm[];
  const int n = M * k;
  int* cnt = sm;
  int* off = cnt + E;
  int* run = off + E;
  int* eidx = run + E;
  int* stok = eidx + n;
  int* eslot = stok + n;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  for (int i = tid; i < n; i += blockDim.x) eidx[i] = ld_act_s32(idx + i);
  __syncthreads();
  block_route_table(eidx, n, k, E, cnt, off, run, stok, eslot, table, blockIdx.x == 0);
  // The gather: four 16-byte vectors per thread in flight (all loads of a
  // group issued before its stores), then the remainder one at a time.
  const int H8 = H >> 3;
  const long long total = (long long)n * H8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long q = (long long)blockIdx.x * blockDim.x + tid;
  for (; q + 3 * stride < total; q += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long qu = q + u * stride;
      const int s = (int)(qu / H8), c = (int)(qu - (long long)s * H8);
      v[u] = ld_act16(x + (size_t)stok[s] * H + (size_t)c * 8);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long qu = q + u * stride;
      const int s = (int)(qu / H8), c = (int)(qu - (long long)s * H8);
      *reinterpret_cast<uint4*>(xs + (size_t)s * H + (size_t)c * 8) = v[u];
    }
  }
  for (; q < total; q += stride) {
    const int s = (int)(q / H8), c = (int)(q - (long long)s * H8);
    *reinterpret_cast<uint4*>(xs + (size_t)s * H + (size_t)c * 8) = ld_act16(x + (size_t)stok[s] * H + (size_t)c * 8);
  }
}

// out[t][:] = bf16( sum_j w[t][j] * y[slot(t, j)][:]  (+ ys[t][:])  (+ res[t][:]) ), fp32 sums in that order.
__global__ void __launch_bounds__(256) combine_kernel(const float* y, const int* table, const float* w, int M, int k,
                                                      int E, const float* ys, const uint16_t* res, uint16_t* out,
                                                      int H) {
  const int t = blockIdx.y;
  const int n0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  pdl_trigger();
  pdl_wait();
  if (n0 >= H) return;
  const TableLayout L(E, M * k);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int j = 0; j < k; ++j) {
    const int slot = ld_act_s32(table + L.entry_slot() + t * k + j);
    const float wj = ld_act_f32(w + (size_t)t * k + j);
    const float4 v = ld_act_f4(y + (size_t)slot * H + n0);
    a0 = fmaf(wj, v.x, a0);
    a1 = fmaf(wj, v.y, a1);
    a2 = fmaf(wj, v.z, a2);
    a3 = fmaf(wj, v.w, a3);
  }
  if (ys != nullptr) {
    const float4 v = ld_act_f4(ys + (size_t)t * H + n0);
    a0 += v.x;
    a1 += v.y;
    a2 += v.z;
    a3 += v.w;
  }
  if (res != nullptr) {
    const uint2 r = ld_act8(res + (size_t)t * H + n0);
    a0 += bf_lo(r.x);
    a1 += bf_hi(r.x);
    a2 += bf_lo(r.y);
    a3 += bf_hi(r.y);
  }
  uint2 o;
  o.x = (uint32_t)f2bf(a0) | ((uint32_t)f2bf(a1) << 16);
  o.y = (uint32_t)f2bf(a2) | ((uint32_t)f2bf(a3) << 16);
  *reinterpret_cast<uint2*>(out + (size_t)t * H + n0) = o;
}

// ---------------------------------------------------------------------------- launchers
cudaError_t launch_router(dec_handle* h, const uint16_t* x, const float* Wr, int M, int H, int E, float* parts,
                          cudaStream_t s) {
  const dim3 grid((E + kRouterRows - 1) / kRouterRows, router_ksplit(H), (M + kRouterGroup - 1) / kRouterGroup);
  return launch_k(h, router_kernel, grid, dim3(256), 0, s, x, Wr, M, H, E, parts);
}

cudaError_t launch_topk(dec_handle* h, const float* parts, int ks, int M, int E, int k, int32_t* idx, float* w,
                        float* scores, cudaStream_t s) {
  const int Ew = (E + 7) / 8;
  const dim3 g(M), b(256);
  if (Ew <= 32) return launch_k(h, topk_kernel<1>, g, b, 0, s, parts, ks, M, E, k, idx, w, scores);
  if (Ew <= 64) return launch_k(h, topk_kernel<2>, g, b, 0, s, parts, ks, M, E, k, idx, w, scores);
  return launch_k(h, topk_kernel<4>, g, b, 0, s, parts, ks, M, E, k, idx, w, scores);
}

cudaError_t launch_router_select(dec_handle* h, const uint16_t* x, const uint16_t* gamma, float eps, const float* Wr,
                                 int H, int E, int k, uint16_t* xn, float* parts, int* counter, int32_t* idx,
                                 float* w, float* scores, int* table, cudaStream_t s) {
  const int Ew = (E + 7) / 8;
  const dim3 g((E + kRouterRows - 1) / kRouterRows, router_ksplit(H)), b(256);
  if (Ew <= 32)
    return launch_k(h, router_select_kernel<1>, g, b, 0, s, x, gamma, eps, Wr, H, E, k, xn, parts, counter, idx, w,
                    scores, table);
  if (Ew <= 64)
    return launch_k(h, router_select_kernel<2>, g, b, 0, s, x, gamma, eps, Wr, H, E, k, xn, parts, counter, idx, w,
                    scores, table);
  return launch_k(h, router_select_kernel<4>, g, b, 0, s, x, gamma, eps, Wr, H, E, k, xn, parts, counter, idx, w,
                  scores, table);
}

cudaError_t launch_one_token_table(dec_handle* h, const int32_t* idx, int E, int k, int* table, cudaStream_t s) {
  return launch_k(h, one_token_table_kernel, dim3(1), dim3(32), 0, s, idx, E, k, table);
}

cudaError_t launch_route_table(dec_handle* h, const int32_t* idx, int M, int k, int E, const uint16_t* x, int H,
                               int* table, uint16_t* xs, cudaStream_t s) {
  const int n = M * k;
  const long long vec = (long long)n * (H / 8);
  int grid = (int)std::min<long long>((vec + 255) / 256, (long long)h->sms);
  if (grid < 1) grid = 1;
  const size_t smem = (size_t)(3 * E + 3 * n) * sizeof(int);
  return launch_k(h, route_table_kernel, dim3(grid), dim3(256), smem, s, idx, M, k, E, x, H, table, xs);
}

cudaError_t launch_combine(dec_handle* h, const float* y, const int* table, const float* w, int M, int k, int E,
                           const float* ys, const uint16_t* res, uint16_t* out, int H, cudaStream_t s) {
  const dim3 grid((H / 4 + 255) / 256, M);
  return launch_k(h, combine_kernel, grid, dim3(256), 0, s, y, table, w, M, k, E, ys, res, out, H);
}

}  // namespace dec
