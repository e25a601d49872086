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

template <int M, int VPT>
__global__ void __launch_bounds__(kGemvThreads, 2)
    gemv_kernel(const uint16_t* x, long long ldx, const uint16_t* __restrict__ W, const uint16_t* res, long long ldr,
                uint16_t* y, long long ldy, int N, int K, const uint16_t* __restrict__ gamma, float eps,
                int ahead) {
  // Rows per step: 8 (M = 1) or 4 (M > 1) weight vectors per thread in flight, kept within 128 registers.
  constexpr int RB = ((M == 1 ? 8 : 4) / VPT) > 0 ? ((M == 1 ? 8 : 4) / VPT) : 1;
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
        for (int i = 0; i < VPT; ++i) a = dot8(wa[r][i], xr[m][i], a);
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

// ---------------------------------------------------------------- TMA ring kernel
// The same product on a ring of shared-memory stages fed by TMA, one CTA per
// SM. Warp 0 is the producer: one thread issues 1-D bulk copies
// (cp.async.bulk, L2 evict-first) of chunks of RR = 8 / VPT consecutive
// weight rows (at most 32 KB) into a ring of up to 7 stages (about 200 KB in
// flight per SM, beyond what registers can hold, from before the dependency
// wait on). Warps 1-8 (256 consumers) hold the activation rows in registers,
// take each chunk from shared memory (thread t: 16-byte column vectors t,
// t + 256, ... of every row), reduce by warp shuffles and then over the eight
// warps in order (the register kernel's order), and release the stage.
//
// Work split: each CTA first streams its static share of chunks, a
// contiguous range of about 70% of the chunks per CTA; the rest are handed
// out one by one from a ticket counter, so CTAs that started late (as the
// previous kernel's CTAs leave their SMs) or stream slower take fewer and the
// CTAs end together. The counter cycles through D + G values (D dynamic
// chunks, G CTAs): every CTA takes tickets until one fails, so a launch takes
// exactly D + G of them and leaves the counter where it found it. The
// producer triggers dependent launches only after its last ticket, so two
// launches never take tickets from one counter at the same time. Without a
// counter every chunk is static.
constexpr int kRingConsumers = 256;
constexpr int kRingThreads = kRingConsumers + 32;
constexpr int kRingStageBytes = 32768;  // weight bytes per stage (a chunk)
constexpr int kRingBytes = 200 * 1024;  // the ring
constexpr int kRingMaxStages = 8;
constexpr double kRingStaticShare = 0.7;

struct GemvRingParams {
  const uint16_t* x;
  long long ldx;
  const uint16_t* W;
  const uint16_t* res;
  long long ldr;
  uint16_t* y;
  long long ldy;
  int N, K;
  const uint16_t* gamma;
  float eps;
  int C;     // chunks of RR rows
  int S;     // static chunks per CTA (CTA b: chunks b S .. b S + S - 1)
  int D;     // dynamic chunks (S G .. C - 1), from the ticket counter
  int NS;    // ring stages
  int* ctr;  // ticket counter (null: no dynamic chunks)
  int* err;
  unsigned long long wait_ns;
};

template <int M, int VPT>
__global__ void __launch_bounds__(kRingThreads, 1) gemv_ring_kernel(const GemvRingParams P) {
  constexpr int RR = 8 / VPT;  // rows per chunk
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kRingMaxStages], empty[kRingMaxStages];
  __shared__ int s_chunk[kRingMaxStages];
  __shared__ float red[2][kRingConsumers / 32][RR * M];
  __shared__ float rred[M][kRingConsumers / 32];
  __shared__ int s_abort;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = gridDim.x, b = blockIdx.x, NS = P.NS;
  const size_t stage_bytes = (size_t)RR * P.K * sizeof(uint16_t);
  if (t == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&s_abort, P.err, P.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int n = 0;  // fills so far; fill n goes to stage n mod NS
      bool ok = true;
      auto fill = [&](int c) -> bool {  // c < 0: the end mark
        const int st = n % NS, q = n / NS;
        if (q > 0 && !mbar_wait(&empty[st], (uint32_t)((q - 1) & 1), wc)) return false;
        s_chunk[st] = c;
        if (c < 0) {
          mbar_arrive(&full[st]);
        } else {
          const int r0 = c * RR;
          const uint32_t bytes = (uint32_t)(min(RR, P.N - r0) * P.K) * 2u;
          mbar_arrive_expect_tx(&full[st], bytes);
          bulk_load_1d(ring + (size_t)st * stage_bytes, P.W + (size_t)r0 * P.K, bytes, &full[st], pol);
        }
        ++n;
        return true;
      };
      for (int j = 0; j < P.S && ok; ++j) {
        const int c = b * P.S + j;
        if (c >= P.C) break;
        ok = fill(c);
      }
      if (P.ctr != nullptr) {
        unsigned* tk = reinterpret_cast<unsigned*>(P.ctr);
        const unsigned wrap = (unsigned)(P.D + G - 1);
        int d = (int)atomicInc(tk, wrap);
        while (d < P.D) {
          const int dn = (int)atomicInc(tk, wrap);  // in flight while this chunk waits for a stage
          if (ok) ok = fill(P.S * G + d);           // (after an abort: tickets only, the cycle completes)
          d = dn;
        }
      }
      pdl_trigger();
      if (ok) ok = fill(-1);
      if (!ok) {  // no copy may still be in flight when the CTA exits
        for (int i = max(0, n - NS); i < n; ++i)
          mbar_wait_drain(&full[i % NS], (uint32_t)((i / NS) & 1), P.err, P.wait_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int tc = t - 32, cw = warp - 1;
    const int K8 = P.K >> 3;
    uint4 gv[VPT];
    if (P.gamma != nullptr) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tc + kRingConsumers * i;
        gv[i] = v < K8 ? *reinterpret_cast<const uint4*>(P.gamma + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
      }
    }
    pdl_wait();
    uint4 xr[M][VPT];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tc + kRingConsumers * i;
        xr[m][i] = v < K8 ? ld_act16(P.x + (size_t)m * P.ldx + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
      }
    if (P.gamma != nullptr) {
      // a_m = bf16(x_m / sqrt(mean(x_m^2) + eps) * gamma), in the RMSNorm kernel's order
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float rs = block_rms_scale<kRingConsumers / 32>(
            thread_sumsq<VPT, kRingConsumers>(xr[m], K8, 0.f, tc), P.K, P.eps, rred[m], 1, cw);
#pragma unroll
        for (int i = 0; i < VPT; ++i) xr[m][i] = norm8(xr[m][i], gv[i], rs);
      }
    }
    int buf = 0;
    for (int n = 0;; ++n) {
      const int st = n % NS;
      const bool got = mbar_wait(&full[st], (uint32_t)((n / NS) & 1), wc);
      if (!named_bar_and(2, kRingConsumers, got)) break;  // (all consumers leave together)
      const int c = s_chunk[st];
      if (c < 0) break;
      const int r0 = c * RR, rows = min(RR, P.N - r0);
      const uint16_t* ws = reinterpret_cast<const uint16_t*>(ring + (size_t)st * stage_bytes);
      float acc[RR][M];
#pragma unroll
      for (int r = 0; r < RR; ++r) {
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
        if (r < rows) {
#pragma unroll
          for (int i = 0; i < VPT; ++i) {
            const int v = tc + kRingConsumers * i;
            if (v < K8) {
              const uint4 w = *reinterpret_cast<const uint4*>(ws + (size_t)r * P.K + (size_t)v * 8);
#pragma unroll
              for (int m = 0; m < M; ++m) acc[r][m] = dot8(w, xr[m][i], acc[r][m]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RR; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], o);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RR; ++r)
#pragma unroll
          for (int m = 0; m < M; ++m) red[buf][cw][r * M + m] = acc[r][m];
      }
      named_bar_sync(1, kRingConsumers);  // every consumer has read the stage
      if (tc == 0) mbar_arrive(&empty[st]);
      if (tc < RR * M) {
        const int r = tc / M, m = tc % M;
        if (r < rows) {
          float sum = 0.f;
#pragma unroll
          for (int w = 0; w < kRingConsumers / 32; ++w) sum += red[buf][w][tc];
          if (P.res != nullptr) sum += bf2f(ld_act_u16(P.res + (size_t)m * P.ldr + r0 + r));
          P.y[(size_t)m * P.ldy + r0 + r] = f2bf(sum);
        }
      }
      buf ^= 1;
    }
  }
}

template <int M, int VPT>
static cudaError_t gemv_ring_launch(dec_handle* h, const GemvRingParams& P0, cudaStream_t s) {
  constexpr int RR = 8 / VPT;
  GemvRingParams P = P0;
  const size_t stage_bytes = (size_t)RR * P.K * sizeof(uint16_t);
  P.C = (P.N + RR - 1) / RR;
  const int G = std::min(h->sms, P.C);
  P.NS = (int)std::min<size_t>(kRingMaxStages, kRingBytes / stage_bytes);
  if (P.ctr != nullptr) {
    P.S = (int)(kRingStaticShare * P.C / G);
    P.D = P.C - P.S * G;
  } else {
    P.S = (P.C + G - 1) / G;
    P.D = 0;
  }
  const size_t smem = (size_t)P.NS * stage_bytes;
  cudaError_t e = cudaFuncSetAttribute(gemv_ring_kernel<M, VPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(h, gemv_ring_kernel<M, VPT>, dim3(G), dim3(kRingThreads), smem, s, P);
}

bool gemv_supported(int M, int K) { return M >= 1 && M <= 4 && K >= 8 && K % 8 == 0 && K <= 8 * 8 * kGemvThreads; }

template <int M>
static cudaError_t gemv_m(dec_handle* h, const uint16_t* x, long long ldx, const uint16_t* W, const uint16_t* res,
                          long long ldr, uint16_t* y, long long ldy, int N, int K, cudaStream_t s, int* ctr,
                          const uint16_t* gamma, float eps) {
  const int K8 = K / 8;
#ifndef DEC_GEMV_REGISTER_KERNEL
  // (rows above 8192 elements keep the register kernel at three and four tokens)
  if ((gamma != nullptr || K8 > 128) && (K8 <= 4 * kRingConsumers || M <= 2)) {
    GemvRingParams P{};
    P.x = x;
    P.ldx = ldx;
    P.W = W;
    P.res = res;
    P.ldr = ldr;
    P.y = y;
    P.ldy = ldy;
    P.N = N;
    P.K = K;
    P.gamma = gamma;
    P.eps = eps;
    P.ctr = ctr;
    P.err = h->d_err;
    P.wait_ns = h->wait_ns;
    if (K8 <= kRingConsumers) return gemv_ring_launch<M, 1>(h, P, s);
    if (K8 <= 2 * kRingConsumers) return gemv_ring_launch<M, 2>(h, P, s);
    if (K8 <= 4 * kRingConsumers) return gemv_ring_launch<M, 4>(h, P, s);
    return gemv_ring_launch<M, 8>(h, P, s);
  }
#endif
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
                        long long ldr, uint16_t* y, long long ldy, int M, int N, int K, cudaStream_t s, int* ctr,
                        const uint16_t* gamma, float eps) {
  switch (M) {
    case 1: return gemv_m<1>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, ctr, gamma, eps);
    case 2: return gemv_m<2>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, ctr, gamma, eps);
    case 3: return gemv_m<3>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, ctr, gamma, eps);
    case 4: return gemv_m<4>(h, x, ldx, W, res, ldr, y, ldy, N, K, s, ctr, gamma, eps);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dec
