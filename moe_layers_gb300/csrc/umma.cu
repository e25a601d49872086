// Split-K tcgen05 engine for weight-streaming skinny GEMMs (batch 3..64 and
// the experts).
//
// Kimi K3 article, Part 1 §1 "Ajustar las formas": at batch sizes above two
// the projection is a split-K kernel that shares the matrix product among
// more GPU workers. Here a "worker" is an SM: the weight matrix is cut into
// tiles of 128 rows, each tile into k-blocks of 64 x KSUB columns (one ring
// stage each), and the sequence of all (tile, k-block) pairs is divided into
// one contiguous, equal-length range per CTA (one persistent CTA per SM).
// Every SM therefore streams the same number of weight bytes. A tile that
// straddles several ranges is finished by the CTA that holds its first piece
// (the end of that CTA's range): it adds the fp32 partials of all pieces in k
// order (deterministic, no float atomics), its own from its accumulator.
//
// Per CTA: warp 0 issues TMA loads of weight tiles (128 x 64 bf16, 128-byte
// swizzle, evict-first) and activation tiles (16-row boxes) into an smem ring;
// warp 1 issues tcgen05.mma (M = 128 weight rows, N = 16..64 tokens, K = 16)
// into a double-buffered TMEM accumulator; warps 2-5 read the accumulator
// with tcgen05.ld and run the epilogue (bf16 out + residual, SwiGLU, or fp32).
// The weights are the MMA's M operand ("swap AB"), so a batch of one to
// sixty-four tokens fills the N dimension and no weight byte is wasted.
//
// Problems: one dense matrix, or a group of experts read from a device-side
// routing table (expert id, first slot, token count); expert e's rows start at
// e * a_rows_per_prob in a bank tensor that covers all experts.
#include <algorithm>
#include <cstdio>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace dec {

struct EngineParams {
  int K, KB, N, tiles;
  long long a_rows_per_prob;
  int count;           // dense mode: tokens
  const int* table;    // grouped mode: routing table
  int E, n_entries;
  void* out;
  long long ldo;
  const uint16_t* res;
  long long ldr;
  float* partials;
  int slot_floats;     // floats per partial slot (nacc * 128 * cols)
  int cols;            // columns per accumulator in a slot
  int* counters;
  int* err;
  unsigned long long wait_ns;
  int finish;  // split-tile finish: 0 first piece's CTA; 1 the last to publish; 2 as 1, from L2 (test hook)
};

// Shared-memory plan of one engine instantiation. A stage holds KSUB 64-wide
// k sub-blocks of NA weight tiles (128 rows x 64 bf16 = 16 KB each, 128-byte
// swizzle) and of the activation tile (BROWS rows); the SwiGLU kernel loads
// two weight tiles (gate and up) per sub-block. The activation slice is sized
// to the batch, and the
// ring takes as many stages as the 227 KB of shared memory allow: the weight
// bytes in flight per SM are what sets the streaming rate.
// Upper bound on the pieces one tile is split into: at most one per CTA, and
// the grid never exceeds this (checked on the host).
constexpr int kMaxPieces = 256;
// How long the CTA that finishes a split tile waits for the other pieces
// before it publishes its own and leaves the tile to the last publisher.
constexpr uint64_t kFinishWaitNs = 5000;

// 64-wide k sub-blocks per stage, by the stage's activation rows (16 / 32 /
// 64) for single-matrix kernels, and for the SwiGLU pair (build-time
// tunables; the defaults are the measured best). Wider stages read more
// contiguous bytes of each weight row per stage: with 64 activation rows, 4
// sub-blocks (2 stages of 96 KB) stream faster than 2 (4 stages of 48 KB)
// with the same weight bytes in flight; with 16 rows, 3 sub-blocks (4 stages
// of 54 KB) beat 2 and 4. The last k-block of a row may reach past K: those
// columns load as zeros.
#ifndef DEC_ENGINE_KSUB_R16
#define DEC_ENGINE_KSUB_R16 3
#endif
#ifndef DEC_ENGINE_KSUB_R32
#define DEC_ENGINE_KSUB_R32 4
#endif
#ifndef DEC_ENGINE_KSUB_R64
#define DEC_ENGINE_KSUB_R64 4
#endif
#ifndef DEC_ENGINE_KSUB_PAIR
#define DEC_ENGINE_KSUB_PAIR 1
#endif
// Shared memory for the ring and CTAs per SM (build-time tunables): the ring
// takes as many stages as the budget allows; with two CTAs per SM a launch's
// CTAs can start beside the previous launch's and stream their first weights
// while it drains.
#ifndef DEC_ENGINE_SMEM_BUDGET
#define DEC_ENGINE_SMEM_BUDGET (232448 - 1024 - 512 - 8 * kMaxPieces)
#endif
#ifndef DEC_ENGINE_CTAS_PER_SM
#define DEC_ENGINE_CTAS_PER_SM 1
#endif

template <int NA, int BROWS>
struct EngineSmem {
  static constexpr int kKSub = (NA == 2)        ? DEC_ENGINE_KSUB_PAIR
                               : (BROWS == 16) ? DEC_ENGINE_KSUB_R16
                               : (BROWS == 32) ? DEC_ENGINE_KSUB_R32
                                               : DEC_ENGINE_KSUB_R64;
  static constexpr int kBK = kBlockK * kKSub;              // reduction elements per k-block (stage)
  static constexpr int kABox = kTileN * kBlockK * 2;       // 16 KB weight box
  static constexpr int kBBox = BROWS * kBlockK * 2;        // activation box of one sub-block
  static constexpr int kABytes = NA * kKSub * kABox;
  static constexpr int kStageBytes = kABytes + kKSub * kBBox;
  static constexpr int kBudget = DEC_ENGINE_SMEM_BUDGET;  // ring bytes (the opt-in maximum minus slack, barriers, pieces)
  static constexpr int kStages = (kBudget / kStageBytes) < 12 ? (kBudget / kStageBytes) : 12;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kTotal = kMiscOff + 32 + 8 * kMaxPieces + 1024;  // + two piece lists + alignment slack
  static constexpr uint32_t kTmemCols = NA * kMaxCols * 2; // two accumulator buffers
  static_assert(kStages >= 2, "engine ring too shallow");
  static_assert(kTotal <= 232448, "engine shared memory above the opt-in maximum");
  // Offsets inside a stage.
  __device__ static constexpr int a_off(int u, int a) { return (u * NA + a) * kABox; }
  __device__ static constexpr int b_off(int u) { return kABytes + u * kBBox; }
};

__device__ __forceinline__ long long range_start(long long c, long long W, long long G) { return c * W / G; }
// CTA whose range holds k-block index j.
__device__ __forceinline__ long long cta_of(long long j, long long W, long long G) { return ((j + 1) * G - 1) / W; }

struct Prob {
  int e, off, cnt;
};

__device__ __forceinline__ Prob prob_info(const EngineParams& P, int p) {
  if (P.table == nullptr) return Prob{0, 0, P.count};
  const TableLayout L(P.E, P.n_entries);
  return Prob{ld_act_s32(P.table + L.expert() + p), ld_act_s32(P.table + L.offset() + p),
              ld_act_s32(P.table + L.count() + p)};
}

__device__ __forceinline__ long long total_kblocks(const EngineParams& P) {
  const long long nprob = (P.table == nullptr) ? 1 : ld_act_s32(P.table);
  return nprob * P.tiles * P.KB;
}

template <int EPI, int BROWS>
__global__ void __launch_bounds__(kEngineThreads, DEC_ENGINE_CTAS_PER_SM)
    engine_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                  const __grid_constant__ CUtensorMap tmB, const EngineParams P) {
  constexpr int NA = (EPI == EPI_SWIGLU) ? 2 : 1;
  using S = EngineSmem<NA, BROWS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* empty = full + S::kStages;
  uint64_t* tfull = empty + S::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMiscOff + 4);
  volatile int* s_last = reinterpret_cast<volatile int*>(smem + S::kMiscOff + 8);
  // Piece lists of split tiles, two by segment parity: the next segment's list
  // is written while threads may still read the previous one.
  volatile int* s_np = reinterpret_cast<volatile int*>(smem + S::kMiscOff + 12);    // [2]
  volatile int* s_mine = reinterpret_cast<volatile int*>(smem + S::kMiscOff + 20);  // [2]
  int* s_piece = reinterpret_cast<int*>(smem + S::kMiscOff + 32);                   // [2][kMaxPieces]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x, c = blockIdx.x;
  const int KB = P.KB, tiles = P.tiles;

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *s_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tmap_prefetch(&tmA);
    if (NA == 2) tmap_prefetch(&tmA2);
    tmap_prefetch(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, P.err, P.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // weights: read once
      const uint64_t pol_x = policy_evict_last();   // activations: read by every CTA
      long long issued = 0;
      auto load_A = [&](int s, int tau, int kb, long long a_row) {
        uint8_t* st = smem + s * S::kStageBytes;
#pragma unroll
        for (int u = 0; u < S::kKSub; ++u) {
          const int k0 = (kb * S::kKSub + u) * kBlockK;
          tma_load_2d(st + S::a_off(u, 0), &tmA, &full[s], k0, (int)a_row, pol_w);
          if (NA == 2) tma_load_2d(st + S::a_off(u, 1), &tmA2, &full[s], k0, (int)a_row, pol_w);
        }
      };
      auto load_B = [&](int s, int kb, int row0, int nb) {
        uint8_t* st = smem + s * S::kStageBytes;
#pragma unroll
        for (int u = 0; u < S::kKSub; ++u) {
          const int k0 = (kb * S::kKSub + u) * kBlockK;
          for (int b = 0; b < nb; ++b) tma_load_2d(st + S::b_off(u) + b * 2048, &tmB, &full[s], k0, row0 + 16 * b, pol_x);
        }
      };
      if (P.table == nullptr) {
        // Dense: the k-block range is known before the dependency wait, so the
        // first ring's worth of static weights streams in while the previous
        // kernel drains. Activations are loaded only after pdl_wait().
        const long long W = (long long)tiles * KB;
        const long long j0 = range_start(c, W, G), j1 = range_start(c + 1, W, G);
        const int nb = (P.count + 15) >> 4;
        const uint32_t bytes = S::kABytes + S::kKSub * nb * 2048;
        const long long npre = min(j1 - j0, (long long)S::kStages);
        for (long long i = 0; i < npre; ++i) {
          const long long j = j0 + i;
          mbar_arrive_expect_tx(&full[i], bytes);
          load_A((int)i, (int)(j / KB), (int)(j % KB), (j / KB) * kTileN);
        }
        pdl_wait();
        for (long long i = 0; i < j1 - j0; ++i) {
          const long long j = j0 + i;
          const int s = (int)(i % S::kStages);
          const uint32_t ph = (uint32_t)((i / S::kStages) & 1);
          const int kb = (int)(j % KB);
          if (i >= npre) {
            if (!mbar_wait(&empty[s], ph ^ 1u, wc)) break;
            mbar_arrive_expect_tx(&full[s], bytes);
            load_A(s, (int)(j / KB), kb, (j / KB) * kTileN);
          }
          load_B(s, kb, 0, nb);
          issued = i + 1;
        }
      } else {
        pdl_wait();
        const long long W = total_kblocks(P);
        const long long j0 = range_start(c, W, G), j1 = range_start(c + 1, W, G);
        int p_ld = -1;  // the current problem and its table entry
        Prob pr_ld{0, 0, 0};
        for (long long i = 0; i < j1 - j0; ++i) {
          const long long j = j0 + i;
          const int s = (int)(i % S::kStages);
          const uint32_t ph = (uint32_t)((i / S::kStages) & 1);
          const int tau = (int)(j / KB), kb = (int)(j % KB);
          if (tau / tiles != p_ld) {
            p_ld = tau / tiles;
            pr_ld = prob_info(P, p_ld);
          }
          const int nb = (pr_ld.cnt + 15) >> 4;
          if (!mbar_wait(&empty[s], ph ^ 1u, wc)) break;
          mbar_arrive_expect_tx(&full[s], S::kABytes + S::kKSub * nb * 2048);
          load_A(s, tau, kb, (long long)pr_ld.e * P.a_rows_per_prob + (long long)(tau % tiles) * kTileN);
          load_B(s, kb, pr_ld.off, nb);
          issued = i + 1;
        }
      }
      // No copy may still be in flight when the CTA exits: wait for the last
      // ring's worth of loads (all of them have landed on the normal path).
      for (long long i = max(0LL, issued - S::kStages); i < issued; ++i)
        mbar_wait_drain(&full[i % S::kStages], (uint32_t)((i / S::kStages) & 1), P.err, P.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      pdl_wait();
      const long long W = total_kblocks(P);
      const long long j0 = range_start(c, W, G), j1 = range_start(c + 1, W, G);
      uint32_t tphase[2] = {0, 0};
      int buf = 0;
      long long i = 0;
      bool ok = true;
      for (long long j = j0; ok && j < j1;) {
        const int tau = (int)(j / KB), kb0 = (int)(j % KB);
        const int kb1 = (int)min((long long)KB, kb0 + (j1 - j));
        const Prob pr = prob_info(P, tau / tiles);
        const uint32_t idesc = umma_idesc_bf16(kTileN, ((pr.cnt + 15) >> 4) * 16);
        if (!mbar_wait(&tempty[buf], tphase[buf] ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(buf * NA * kMaxCols);
        for (int kb = kb0; kb < kb1; ++kb, ++i) {
          const int s = (int)(i % S::kStages);
          if (!mbar_wait(&full[s], (uint32_t)((i / S::kStages) & 1), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st_addr = smem_u32(smem + s * S::kStageBytes);
#pragma unroll
          for (int u = 0; u < S::kKSub; ++u) {
            const uint32_t a_addr = st_addr + S::a_off(u, 0), b_addr = st_addr + S::b_off(u);
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk) {
              const uint64_t bd = sw128_desc(b_addr + kk * 32);
              const uint32_t acc = (kb > kb0 || u > 0 || kk > 0) ? 1u : 0u;
              umma_bf16(d0, sw128_desc(a_addr + kk * 32), bd, idesc, acc);
              if (NA == 2) umma_bf16(d0 + kMaxCols, sw128_desc(st_addr + S::a_off(u, 1) + kk * 32), bd, idesc, acc);
            }
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
        tphase[buf] ^= 1u;
        buf ^= 1;
        j += kb1 - kb0;
      }
      // Every MMA issued above must complete before TMEM is released.
      umma_commit(done);
      mbar_wait_drain(done, 0, P.err, P.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;              // TMEM lanes 32q..32q+31 are visible to this warp
    const int row = q * 32 + lane;       // row within the 128-row tile
    const int et = threadIdx.x - 64;     // 0..127
    pdl_wait();
    const long long W = total_kblocks(P);
    const long long j0 = range_start(c, W, G), j1 = range_start(c + 1, W, G);
    uint32_t tphase[2] = {0, 0};
    int buf = 0;
    uint16_t* out16 = reinterpret_cast<uint16_t*>(P.out);
    float* out32 = reinterpret_cast<float*>(P.out);

    // Writes columns [ch*16, ch*16 + 16) of this thread's output row n. Residual
    // values are all loaded first (independent loads in flight together), then
    // combined and stored.
    auto emit_chunk = [&](const Prob& pr, int n, int ch, const float (&v0)[16], const float (&v1)[16]) {
      const int jn = min(16, pr.cnt - ch * 16);
      if (EPI == EPI_LINEAR) {
        float r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0.f;
        if (P.res != nullptr) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < jn) r[i] = bf2f(ld_act_u16(P.res + ((long long)pr.off + ch * 16 + i) * P.ldr + n));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < jn) out16[((long long)pr.off + ch * 16 + i) * P.ldo + n] = f2bf(v0[i] + r[i]);
      } else if (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < jn) {
            const float g = v0[i];
            out16[((long long)pr.off + ch * 16 + i) * P.ldo + n] = swiglu_bf16(g, v1[i]);
          }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < jn) out32[((long long)pr.off + ch * 16 + i) * P.ldo + n] = v0[i];
      }
    };

    // The residual rows of a tile can be staged in shared memory with 16-byte copies.
    const bool res_stageable = EPI == EPI_LINEAR && P.res != nullptr &&
                               (reinterpret_cast<uintptr_t>(P.res) & 15) == 0 && (P.ldr & 7) == 0 && (P.N & 7) == 0;
    const bool partials_aligned = (reinterpret_cast<uintptr_t>(P.partials) & 15) == 0;
    constexpr int kOutBytes = (EPI == EPI_F32) ? 4 : 2;
    // Output rows can take 16-byte stores.
    const bool out_vec = (reinterpret_cast<uintptr_t>(P.out) & 15) == 0 && (P.ldo * kOutBytes) % 16 == 0;

    // Copies this thread's row of the accumulator (all tokens, every
    // accumulator) into shared memory laid out like a published partial:
    // [NA][cnt][128] floats from `dst` (consecutive rows: no bank conflicts).
    auto acc_to_smem = [&](float* dst, int cnt, uint32_t taddr) {
      for (int ch = 0; ch < (cnt + 15) >> 4; ++ch) {
        float v0[16], v1[16];
        tmem_ld16(taddr + ch * 16, v0);
        if (NA == 2) tmem_ld16(taddr + kMaxCols + ch * 16, v1);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (ch * 16 + i < cnt) {
            dst[(ch * 16 + i) * kTileN + row] = v0[i];
            if (NA == 2) dst[(cnt + ch * 16 + i) * kTileN + row] = v1[i];
          }
      }
    };

    // Writes eight consecutive outputs (token t of the problem, columns
    // [c, c + 8) with c < N) from their fp32 sums; `rs` holds the tile's staged
    // residual rows ([cnt][128] bf16, column c - n0) or is null.
    auto emit8 = [&](const Prob& pr, int t, int n0, int c, const float (&a0)[8], const float (&a1)[8],
                     const uint16_t* rs) {
      const long long orow = ((long long)pr.off + t) * P.ldo;
      const bool vec = out_vec && c + 8 <= P.N;
      if (EPI == EPI_F32) {
        float* o = reinterpret_cast<float*>(P.out) + orow + c;
        if (vec) {
          reinterpret_cast<float4*>(o)[0] = make_float4(a0[0], a0[1], a0[2], a0[3]);
          reinterpret_cast<float4*>(o)[1] = make_float4(a0[4], a0[5], a0[6], a0[7]);
        } else {
          for (int e = 0; e < 8 && c + e < P.N; ++e) o[e] = a0[e];
        }
        return;
      }
      uint16_t b[8];
      if (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int e = 0; e < 8; ++e) b[e] = swiglu_bf16(a0[e], a1[e]);
      } else {
        float r[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) r[e] = 0.f;
        if (rs != nullptr) {
          const uint4 rv = *reinterpret_cast<const uint4*>(rs + t * kTileN + (c - n0));
          const uint32_t w[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) r[e] = bf2f((uint16_t)(w[e >> 1] >> ((e & 1) * 16)));
        } else if (P.res != nullptr) {
          const uint16_t* rp = P.res + ((long long)pr.off + t) * P.ldr + c;
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (c + e < P.N) r[e] = bf2f(ld_act_u16(rp + e));
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) b[e] = f2bf(a0[e] + r[e]);
      }
      uint16_t* o = reinterpret_cast<uint16_t*>(P.out) + orow + c;
      if (vec) {
        *reinterpret_cast<uint4*>(o) = make_uint4(b[0] | ((uint32_t)b[1] << 16), b[2] | ((uint32_t)b[3] << 16),
                                                  b[4] | ((uint32_t)b[5] << 16), b[6] | ((uint32_t)b[7] << 16));
      } else {
        for (int e = 0; e < 8 && c + e < P.N; ++e) o[e] = b[e];
      }
    };

    // Finishes a split tile from its pieces staged in the ring's shared
    // memory, which is idle once every MMA of the CTA has completed. The
    // partials of every piece but `own` are copied in (16-byte copies through
    // L2) with the tile's residual rows when they can be staged; piece `own`
    // (`own` < 0: none) comes from this CTA's accumulator. Each thread then
    // adds the pieces in k order (the sums of a reduction from the published
    // partials) for eight consecutive columns of one token at a time, and
    // stores them with one 16-byte store.
    auto finish_staged = [&](const Prob& pr, int n0, uint32_t taddr, const int* pieces, int np, int own) {
      const int cnt = pr.cnt;
      const int acc_floats = cnt * kTileN;
      const int piece_floats = NA * acc_floats;
      float* sp = reinterpret_cast<float*>(smem);                                       // [np][NA][cnt][128]
      uint16_t* sr = reinterpret_cast<uint16_t*>(smem + (size_t)np * piece_floats * 4);  // [cnt][128]
      __threadfence();
      for (int p = 0; p < np; ++p) {
        if (p == own) continue;
        const float* src = P.partials + (size_t)pieces[p] * P.slot_floats;
        float* dst = sp + (size_t)p * piece_floats;
#pragma unroll
        for (int a = 0; a < NA; ++a)
          for (int g = et; g < acc_floats / 4; g += 128)
            cp_async16(dst + (size_t)a * acc_floats + g * 4, src + (size_t)a * P.cols * kTileN + g * 4);
      }
      if (res_stageable)
        for (int g = et; g < cnt * (kTileN / 8); g += 128) {  // 8 columns per granule
          const int t = g / (kTileN / 8), c8 = (g % (kTileN / 8)) * 8;
          if (n0 + c8 < P.N) cp_async16(sr + t * kTileN + c8, P.res + ((long long)pr.off + t) * P.ldr + n0 + c8);
        }
      if (own >= 0) acc_to_smem(sp + (size_t)own * piece_floats, cnt, taddr);
      cp_async_wait_all();
      named_bar_sync(1, 128);
      for (int g = et; g < cnt * (kTileN / 8); g += 128) {
        const int t = g / (kTileN / 8), c8 = (g % (kTileN / 8)) * 8;
        if (n0 + c8 >= P.N) continue;
        float a0[8], a1[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a0[e] = a1[e] = 0.f;
        const float* base = sp + t * kTileN + c8;
        // Pieces four at a time: every load of a batch before any add.
        for (int p0 = 0; p0 < np; p0 += 4) {
          float4 x[4][2], y[4][2];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const float4* s4 = reinterpret_cast<const float4*>(base + (size_t)min(p0 + qq, np - 1) * piece_floats);
            x[qq][0] = s4[0];
            x[qq][1] = s4[1];
            if (NA == 2) {
              y[qq][0] = s4[acc_floats / 4];
              y[qq][1] = s4[acc_floats / 4 + 1];
            }
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            if (p0 + qq < np) {
              const float v[8] = {x[qq][0].x, x[qq][0].y, x[qq][0].z, x[qq][0].w,
                                  x[qq][1].x, x[qq][1].y, x[qq][1].z, x[qq][1].w};
#pragma unroll
              for (int e = 0; e < 8; ++e) a0[e] += v[e];
              if (NA == 2) {
                const float u[8] = {y[qq][0].x, y[qq][0].y, y[qq][0].z, y[qq][0].w,
                                    y[qq][1].x, y[qq][1].y, y[qq][1].z, y[qq][1].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) a1[e] += u[e];
              }
            }
        }
        emit8(pr, t, n0, n0 + c8, a0, a1, res_stageable ? sr : nullptr);
      }
    };

    // Publishes this thread's share of a piece's partial from the accumulator
    // staged in shared memory (the ring is idle): 16-byte stores.
    auto publish_staged = [&](float* slot, int cnt, uint32_t taddr) {
      float* sp = reinterpret_cast<float*>(smem);
      acc_to_smem(sp, cnt, taddr);
      named_bar_sync(1, 128);
#pragma unroll
      for (int a = 0; a < NA; ++a)
        for (int g = et; g < cnt * kTileN / 4; g += 128)
          reinterpret_cast<float4*>(slot + (size_t)a * P.cols * kTileN)[g] =
              reinterpret_cast<const float4*>(sp + (size_t)a * cnt * kTileN)[g];
    };

    int seg = 0;  // segments so far (parity selects the piece list)
    for (long long j = j0; j < j1; ++seg) {
      const int tau = (int)(j / KB), kb0 = (int)(j % KB);
      const int kb1 = (int)min((long long)KB, kb0 + (j1 - j));
      const bool first_seg = (j == j0);
      j += kb1 - kb0;
      const bool last_seg = (j == j1);
      const bool whole = (kb0 == 0 && kb1 == KB);
      const int lp = seg & 1;
      int* pieces = s_piece + lp * kMaxPieces;
      if (!whole && et == 0) {
        // The non-empty CTAs that hold pieces of this tile, in k order, their
        // partial slots and this CTA's place among them (computed while the
        // MMAs run: it takes 64-bit divisions).
        const long long kfirst = (long long)tau * KB;
        const long long c_first = cta_of(kfirst, W, G), c_last = cta_of(kfirst + KB - 1, W, G);
        int np = 0, mine = 0;
        for (long long cc = c_first; cc <= c_last; ++cc) {
          const long long st = range_start(cc, W, G);
          if (range_start(cc + 1, W, G) <= st) continue;
          if (cc == c) mine = np;
          if (np < kMaxPieces) pieces[np] = (int)(cc * 2 + ((st >= kfirst) ? 0 : 1));
          ++np;
        }
        s_np[lp] = np;
        s_mine[lp] = mine;
      }
      const bool got = mbar_wait(&tfull[buf], tphase[buf], wc);
      if (!named_bar_and(1, 128, got)) break;  // leave together if any thread gave up
      tc_fence_after();
      const Prob pr = prob_info(P, tau / tiles);
      const int n0 = (tau % tiles) * kTileN;
      const int n = n0 + row;
      const bool valid_row = n < P.N;
      const int nch = (pr.cnt + 15) >> 4;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NA * kMaxCols);
      const size_t piece_bytes = (size_t)NA * pr.cnt * kTileN * 4;
      const size_t res_bytes = res_stageable ? (size_t)pr.cnt * kTileN * 2 : 0;
      if (!whole) {
        if (et == 0) {
          // The CTA that holds the tile's first piece (the end of its range, so
          // its ring is idle by now) finishes the tile: it waits a bounded time
          // for the other pieces, then adds them to its own accumulator without
          // publishing it. Past the bound it publishes like the others, and
          // whichever CTA publishes last finishes the tile.
          const int np = s_np[lp];
          int mode = 0;
          if (P.finish == 0 && s_mine[lp] == 0 && last_seg && partials_aligned && np <= kMaxPieces &&
              (size_t)np * piece_bytes + res_bytes <= (size_t)S::kBarOff) {
            const uint64_t t0 = globaltimer();
            int arrived;
            while ((arrived = ld_acquire_gpu(&P.counters[tau])) < np - 1 && globaltimer() - t0 < kFinishWaitNs) {
            }
            if (arrived == np - 1) mode = 2;
          }
          *s_last = mode;
        }
        named_bar_sync(1, 128);
        if (*s_last == 2) {
          finish_staged(pr, n0, taddr, pieces, s_np[lp], s_mine[lp]);
          tc_fence_before();
          mbar_arrive(&tempty[buf]);
          tphase[buf] ^= 1u;
          buf ^= 1;
          if (et == 0) P.counters[tau] = 0;  // leave the workspace reusable
          continue;
        }
      }
      float* slot = nullptr;
      if (!whole) slot = P.partials + (size_t)(c * 2 + (first_seg ? 0 : 1)) * P.slot_floats;
      if (!whole && last_seg && partials_aligned && piece_bytes <= (size_t)S::kBarOff) {
        publish_staged(slot, pr.cnt, taddr);
      } else {
        for (int ch = 0; ch < nch; ++ch) {
          float v0[16], v1[16];
          tmem_ld16(taddr + ch * 16, v0);
          if (NA == 2) tmem_ld16(taddr + kMaxCols + ch * 16, v1);
          if (whole) {
            if (valid_row) emit_chunk(pr, n, ch, v0, v1);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jc = ch * 16 + i;
              if (jc < pr.cnt) {
                slot[(size_t)jc * kTileN + row] = v0[i];
                if (NA == 2) slot[(size_t)P.cols * kTileN + (size_t)jc * kTileN + row] = v1[i];
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
      tphase[buf] ^= 1u;
      buf ^= 1;
      if (whole) continue;

      // Published piece: the CTA whose arrival completes the count finishes the
      // tile (the first piece's CTA counts only when it gave up waiting).
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0) {
        const int old = atomicAdd(&P.counters[tau], 1);
        *s_last = (old == s_np[lp] - 1) ? 1 : 0;
      }
      named_bar_sync(1, 128);
      if (!*s_last) continue;
      const int np = min(s_np[lp], kMaxPieces);
      if (P.finish <= 1 && last_seg && partials_aligned &&
          (size_t)np * piece_bytes + res_bytes <= (size_t)S::kBarOff) {
        finish_staged(pr, n0, taddr, pieces, np, -1);
      } else {
        __threadfence();
        // The pieces' partials are read RB pieces at a time, every load of a
        // batch issued before any is added (one L2 round trip per batch, not
        // per piece), and added in k order (the same sums as one by one).
        constexpr int RB = (NA == 2) ? 2 : 4;
        for (int ch = 0; ch < nch; ++ch) {
          float a0[16], a1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) a0[i] = a1[i] = 0.f;
          for (int p0 = 0; p0 < np; p0 += RB) {
            float t0[RB][16], t1[RB][16];
#pragma unroll
            for (int q = 0; q < RB; ++q) {
              const int p = p0 + q < np ? p0 + q : p0;
              const float* ps = P.partials + (size_t)pieces[p] * P.slot_floats + (size_t)ch * 16 * kTileN + row;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const bool ok = p0 + q < np && ch * 16 + i < pr.cnt;
                t0[q][i] = ok ? __ldcg(ps + (size_t)i * kTileN) : 0.f;
                if (NA == 2) t1[q][i] = ok ? __ldcg(ps + (size_t)P.cols * kTileN + (size_t)i * kTileN) : 0.f;
              }
            }
#pragma unroll
            for (int q = 0; q < RB; ++q)
              if (p0 + q < np) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (ch * 16 + i < pr.cnt) {
                    a0[i] += t0[q][i];
                    if (NA == 2) a1[i] += t1[q][i];
                  }
              }
          }
          if (valid_row) emit_chunk(pr, n, ch, a0, a1);
        }
      }
      if (et == 0) P.counters[tau] = 0;  // leave the workspace reusable
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

// ---------------------------------------------------------------------------- host side
static bool encode_2d(const dec_handle* h, CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                      uint64_t row_stride_bytes, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {(cuuint32_t)kBlockK, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = h->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int engine_grid(const dec_handle* h) { return h->sms; }

size_t engine_ws_bytes(int grid, int nacc, long long max_tiles) {
  auto al = [](size_t b) { return (b + 255) & ~size_t(255); };
  return al((size_t)2 * grid * nacc * kTileN * kMaxCols * sizeof(float)) + al((size_t)max_tiles * sizeof(int));
}

template <int EPI, int BROWS>
static cudaError_t launch_epi(dec_handle* h, const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb,
                              const EngineParams& P, int grid, cudaStream_t s) {
  constexpr int NA = (EPI == EPI_SWIGLU) ? 2 : 1;
  using S = EngineSmem<NA, BROWS>;
  static bool attr_set = false;  // per process; every device gets the same attribute
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(engine_kernel<EPI, BROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(h, engine_kernel<EPI, BROWS>, dim3(grid), dim3(kEngineThreads), (size_t)S::kTotal, s, ta, ta2, tb,
                  P);
}

// The dense grid never exceeds the number of k-blocks (a CTA per k-block at most).
template <int EPI, int BROWS>
static cudaError_t launch_kb(dec_handle* h, const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb,
                             EngineParams& P, int grid, cudaStream_t s) {
  constexpr int NA = (EPI == EPI_SWIGLU) ? 2 : 1;
  constexpr int BK = EngineSmem<NA, BROWS>::kBK;
  P.KB = (P.K + BK - 1) / BK;
  if (P.table == nullptr) grid = (int)std::min<long long>(grid, (long long)P.tiles * P.KB);
  return launch_epi<EPI, BROWS>(h, ta, ta2, tb, P, grid < 1 ? 1 : grid, s);
}

// Activation rows per stage: the smallest of 16 / 32 / 64 that holds the
// largest token count of any problem in the launch.
template <int EPI>
static cudaError_t launch_rows(dec_handle* h, const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb,
                               EngineParams& P, int max_cols, int grid, cudaStream_t s) {
  if (max_cols <= 16) return launch_kb<EPI, 16>(h, ta, ta2, tb, P, grid, s);
  if (max_cols <= 32) return launch_kb<EPI, 32>(h, ta, ta2, tb, P, grid, s);
  return launch_kb<EPI, 64>(h, ta, ta2, tb, P, grid, s);
}

cudaError_t launch_engine(dec_handle* h, const EngineLaunch& L, cudaStream_t s) {
  CUtensorMap ta, ta2, tb;
  if (!encode_2d(h, &ta, L.A, (uint64_t)L.K, (uint64_t)L.a_rows, (uint64_t)L.K * 2, kTileN))
    return cudaErrorInvalidValue;
  if (L.epi == EPI_SWIGLU) {
    if (!encode_2d(h, &ta2, L.A2, (uint64_t)L.K, (uint64_t)L.a_rows, (uint64_t)L.K * 2, kTileN))
      return cudaErrorInvalidValue;
  } else {
    ta2 = ta;
  }
  if (!encode_2d(h, &tb, L.B, (uint64_t)L.K, (uint64_t)L.b_rows, (uint64_t)L.ldb * 2, 16))
    return cudaErrorInvalidValue;
  const int nacc = (L.epi == EPI_SWIGLU) ? 2 : 1;
  EngineParams P;
  P.K = L.K;
  P.KB = 0;  // set per instantiation (k-block width depends on the stage plan)
  P.N = L.N;
  P.tiles = (L.N + kTileN - 1) / kTileN;
  P.a_rows_per_prob = L.a_rows_per_prob;
  P.count = L.count;
  P.table = L.table;
  P.E = L.E;
  P.n_entries = L.n_entries;
  P.out = L.out;
  P.ldo = L.ldo;
  P.res = L.res;
  P.ldr = L.ldr;
  P.partials = L.partials;
  P.cols = kMaxCols;
  P.slot_floats = nacc * kTileN * kMaxCols;
  P.counters = L.counters;
  P.err = h->d_err;
  P.wait_ns = h->wait_ns;
  P.finish = h->engine_finish;
  const int grid = L.grid > 0 ? L.grid : engine_grid(h);
  if (grid > kMaxPieces) return cudaErrorInvalidConfiguration;
  const int max_cols = L.count;  // dense: the tokens; grouped: the batch, a bound on any expert's tokens
  if (max_cols < 1 || max_cols > kMaxCols) return cudaErrorInvalidValue;
  switch (L.epi) {
    case EPI_LINEAR: return launch_rows<EPI_LINEAR>(h, ta, ta2, tb, P, max_cols, grid, s);
    case EPI_SWIGLU: return launch_rows<EPI_SWIGLU>(h, ta, ta2, tb, P, max_cols, grid, s);
    default: return launch_rows<EPI_F32>(h, ta, ta2, tb, P, max_cols, grid, s);
  }
}

}  // namespace dec
