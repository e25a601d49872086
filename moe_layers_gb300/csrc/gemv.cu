// Small-matrix projection kernel: chosen at batch 1, available up to 4 when forced.
//
// Kimi K3 article, Part 1 §1 "Ajustar las formas" (and the aihirek.info
// summary): at batch 1-2 the attention projections use specialised
// small-matrix kernels. With one token every weight byte feeds one FMA, so the
// kernel is a pure weight stream and CUDA cores suffice; it reaches the HBM
// copy rate on GB300. At batch 2 the split-K tcgen05 kernel measured faster
// here, so the automatic choice uses this kernel for one token only.
//
// Layout of the work: the N weight rows are divided into one contiguous,
// equal range per CTA (two 256-thread CTAs per SM), so every SM streams the
// same bytes. Inside a CTA all 256 threads share each row: thread t owns the
// 16-byte column vectors t, t+256, ... of every row, holds the matching
// activation vectors in registers for the whole kernel, and streams weight
// vectors with 128-bit, L1-bypassing, evict-first loads. RB rows are loaded
// per step and the next step's loads are issued before the current step's
// FMAs (8-16 loads in flight per thread). Per-row partial sums are reduced
// with warp shuffles, then across the eight warps through shared memory, in a
// fixed order.
//
// The first rows' weight loads are issued before griddepcontrol.wait, so they
// overlap the previous kernel's tail; activations and the residual are read
// only after it. Beyond the register double buffer, thread 0 keeps about
// `ahead` bytes of the CTA's next rows requested into L2 (bulk prefetches,
// starting before the wait), so that the register loads mostly hit L2 and the
// memory sees many more requests in flight than registers can hold.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dec {

constexpr int kGemvThreads = 256;
// Largest token count that streams 8 weight vectors per thread per step
// (build-time tunable). Two tokens fit it in registers since the dot products
// take bf16 operands directly; measured: the 176 MB projection 26.92 -> 26.32
// us back to back at two tokens.
#ifndef DEC_GEMV_RB8_M
#define DEC_GEMV_RB8_M 2
#endif

template <int M, int VPT>
__global__ void __launch_bounds__(kGemvThreads, 2)
    gemv_kernel(const uint16_t* x, long long ldx, const uint16_t* __restrict__ W, const uint16_t* res, long long ldr,
                uint16_t* y, long long ldy, int N, int K, const uint16_t* __restrict__ gamma, float eps,
                int ahead) {
  // Rows per step: 8 (M <= 2) or 4 weight vectors per thread in flight, kept within 128 registers.
  constexpr int RB = ((M <= DEC_GEMV_RB8_M ? 8 : 4) / VPT) > 0 ? ((M <= DEC_GEMV_RB8_M ? 8 : 4) / VPT) : 1;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K8 = K >> 3;
  const long long G = gridDim.x;
  const int r0 = (int)((long long)blockIdx.x * N / G);
  const int r1 = (int)((long long)(blockIdx.x + 1) * N / G);
  __shared__ float red[2][kGemvThreads / 32][RB * M];
  const uint64_t pol = policy_evict_first();
  pdl_trigger();

  uint4 wa[RB][VPT];
  auto load_rows = [&](uint4(&w)[RB][VPT], int rb) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = t + kGemvThreads * i;
        const int rr = rb + r;
        if (rr < r1 && v < K8)
          w[r][i] = ld_stream(W + (size_t)rr * K + (size_t)v * 8, pol);
        else
          w[r][i] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  if (r0 < r1) load_rows(wa, r0);
  // L2 requests: rows [pf, ...) of this CTA's range are not yet requested.
  const size_t rowb = (size_t)K * sizeof(uint16_t);
  const int ahead_rows = ahead > 0 ? max(RB, (int)((size_t)ahead / rowb)) : 0;
  int pf = r0 + RB;
  auto request = [&](int upto) {
    upto = min(upto, r1);
    if (ahead_rows > 0 && upto > pf) {
      if (t == 0) request_l2(W + (size_t)pf * K, (size_t)(upto - pf) * rowb);
      pf = upto;
    }
  };
  request(r0 + RB + ahead_rows);
  // Optional RMSNorm of the input rows, fused: gains are static weights.
  uint4 gv[VPT];
  if (gamma != nullptr) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = t + kGemvThreads * i;
      gv[i] = (v < K8) ? *reinterpret_cast<const uint4*>(gamma + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
    }
  }

  pdl_wait();
  uint4 xr[M][VPT];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = t + kGemvThreads * i;
      xr[m][i] = (v < K8) ? ld_act16(x + (size_t)m * ldx + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
    }
  if (gamma != nullptr) {
    // a_m = bf16(x_m / sqrt(mean(x_m^2) + eps) * gamma) for every row m, in
    // the reduction order of the stand-alone RMSNorm kernel (the same bits).
    __shared__ float rred[M][kGemvThreads / 32];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float rs =
          block_rms_scale<kGemvThreads / 32>(thread_sumsq<VPT, kGemvThreads>(xr[m], K8), K, eps, rred[m]);
#pragma unroll
      for (int i = 0; i < VPT; ++i) xr[m][i] = norm8(xr[m][i], gv[i], rs);
    }
  }

  int buf = 0;
  for (int rb = r0; rb < r1; rb += RB) {
    uint4 wb[RB][VPT];
    const bool more = rb + RB < r1;
    if (more) load_rows(wb, rb + RB);
    request(rb + 2 * RB + ahead_rows);
    float acc[RB][M];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) a = M == 1 ? dot8_widened(wa[r][i], xr[m][i], a) : dot8(wa[r][i], xr[m][i], a);
        acc[r][m] = a;
      }
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], o);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) red[buf][warp][r * M + m] = acc[r][m];
    }
    __syncthreads();
    if (t < RB * M) {
      const int r = t / M, m = t % M, row = rb + r;
      if (row < r1) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kGemvThreads / 32; ++w) s += red[buf][w][t];
        if (res != nullptr) s += bf2f(ld_act_u16(res + (size_t)m * ldr + row));
        y[(size_t)m * ldy + row] = f2bf(s);
      }
    }
    buf ^= 1;
    if (more) {
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int i = 0; i < VPT; ++i) wa[r][i] = wb[r][i];
    }
  }
}

// Narrow rows (K <= 1024: K / 8 <= TPR <= 128 vectors): TPR threads share a
// row, one 16-byte vector each, so a CTA works on 256 / TPR rows at a time
// instead of leaving most of its threads idle. Each group of TPR threads takes
// RB rows per step (one vector per row per thread; the next step's loads are
// issued before this step's FMAs); groups interleave so that the CTA's
// concurrent rows are adjacent in memory. Groups of up to 32 threads reduce
// with shuffles alone; wider groups add one shared-memory pass over their
// warps. No RMSNorm here (the input projection's rows are wide).
template <int M, int TPR>
__global__ void __launch_bounds__(kGemvThreads, 2)
    gemv_narrow_kernel(const uint16_t* x, long long ldx, const uint16_t* __restrict__ W, const uint16_t* res,
                       long long ldr, uint16_t* y, long long ldy, int N, int K, int ahead) {
  constexpr int NG = kGemvThreads / TPR;  // row groups
  constexpr int RB = M == 1 ? 8 : 4;      // rows per group per step
  constexpr int WPG = TPR > 32 ? TPR / 32 : 1;  // warps per group
  static_assert(TPR >= RB * M, "a group's threads write its RB x M outputs");
  const int t = threadIdx.x, g = t / TPR, j = t % TPR, lane = t & 31;
  const int K8 = K >> 3;
  const long long G = gridDim.x;
  const int r0 = (int)((long long)blockIdx.x * N / G);
  const int r1 = (int)((long long)(blockIdx.x + 1) * N / G);
  constexpr int STEP = NG * RB;  // rows per CTA step
  __shared__ float red[2][kGemvThreads / 32][TPR > 32 ? RB * M : 1];
  const uint64_t pol = policy_evict_first();
  pdl_trigger();

  // row of group g, slot r, in the step starting at rb
  auto row_of = [&](int rb, int r) { return rb + g + NG * r; };
  uint4 wa[RB];
  auto load_rows = [&](uint4(&w)[RB], int rb) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int rr = row_of(rb, r);
      w[r] = (rr < r1 && j < K8) ? ld_stream(W + (size_t)rr * K + (size_t)j * 8, pol) : make_uint4(0, 0, 0, 0);
    }
  };
  if (r0 < r1) load_rows(wa, r0);
  const size_t rowb = (size_t)K * sizeof(uint16_t);
  const int ahead_rows = ahead > 0 ? max(STEP, (int)((size_t)ahead / rowb)) : 0;
  int pf = r0 + STEP;
  auto request = [&](int upto) {
    upto = min(upto, r1);
    if (ahead_rows > 0 && upto > pf) {
      if (t == 0) request_l2(W + (size_t)pf * K, (size_t)(upto - pf) * rowb);
      pf = upto;
    }
  };
  request(r0 + STEP + ahead_rows);
  pdl_wait();
  uint4 xr[M];
#pragma unroll
  for (int m = 0; m < M; ++m) xr[m] = j < K8 ? ld_act16(x + (size_t)m * ldx + (size_t)j * 8) : make_uint4(0, 0, 0, 0);

  int buf = 0;
  for (int rb = r0; rb < r1; rb += STEP) {
    uint4 wb[RB];
    const bool more = rb + STEP < r1;
    if (more) load_rows(wb, rb + STEP);
    request(rb + 2 * STEP + ahead_rows);
    float acc[RB][M];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[r][m] = dot8(wa[r], xr[m], 0.f);
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int o = (TPR < 32 ? TPR : 32) / 2; o > 0; o >>= 1)
          acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], o);
    float val = 0.f;  // thread j < RB * M of the group: output (r, m) = (j / M, j % M)
    if (TPR > 32) {
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
          for (int m = 0; m < M; ++m) red[buf][t >> 5][r * M + m] = acc[r][m];
      }
      __syncthreads();
      if (j < RB * M)
        for (int w = 0; w < WPG; ++w) val += red[buf][g * WPG + w][j];
    } else {
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m)
          if (j == r * M + m) val = acc[r][m];
    }
    if (j < RB * M) {
      const int r = j / M, m = j % M, row = row_of(rb, r);
      if (row < r1) {
        if (res != nullptr) val += bf2f(ld_act_u16(res + (size_t)m * ldr + row));
        y[(size_t)m * ldy + row] = f2bf(val);
      }
    }
    buf ^= 1;
    if (more) {
#pragma unroll
      for (int r = 0; r < RB; ++r) wa[r] = wb[r];
    }
  }
}

bool gemv_supported(int M, int K) { return M >= 1 && M <= 4 && K >= 8 && K % 8 == 0 && K <= 8 * 8 * kGemvThreads; }

template <int M>
static cudaError_t gemv_m(dec_handle* h, const uint16_t* x, long long ldx, const uint16_t* W, const uint16_t* res,
                          long long ldr, uint16_t* y, long long ldy, int N, int K, cudaStream_t s,
                          const uint16_t* gamma, float eps) {
  const int K8 = K / 8;
  const int grid = (int)std::min<long long>((long long)N, 2LL * h->sms);
  const dim3 g(grid > 0 ? grid : 1), b(kGemvThreads);
  const int a = h->l2_ahead;
  if (gamma == nullptr && K8 <= 128) {
    if (K8 <= 16) return launch_k(h, gemv_narrow_kernel<M, 16>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, a);
    if (K8 <= 32) return launch_k(h, gemv_narrow_kernel<M, 32>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, a);
    if (K8 <= 64) return launch_k(h, gemv_narrow_kernel<M, 64>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, a);
    return launch_k(h, gemv_narrow_kernel<M, 128>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, a);
  }
  if (K8 <= kGemvThreads)
    return launch_k(h, gemv_kernel<M, 1>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, gamma, eps, a);
  if (K8 <= 2 * kGemvThreads)
    return launch_k(h, gemv_kernel<M, 2>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, gamma, eps, a);
  if (K8 <= 4 * kGemvThreads)
    return launch_k(h, gemv_kernel<M, 4>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, gamma, eps, a);
  return launch_k(h, gemv_kernel<M, 8>, g, b, 0, s, x, ldx, W, res, ldr, y, ldy, N, K, gamma, eps, a);
}

cudaError_t launch_gemv(dec_handle* h, const uint16_t* x, long long ldx, const uint16_t* W, const uint16_t* res,
                        long long ldr, uint16_t* y, long long ldy, int M, int N, int K, cudaStream_t s,
                        const uint16_t* gamma, float eps) {
  switch (M) {
    case 1: return gemv_m<1>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, gamma, eps);
    case 2: return gemv_m<2>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, gamma, eps);
    case 3: return gemv_m<3>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, gamma, eps);
    case 4: return gemv_m<4>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, gamma, eps);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dec
