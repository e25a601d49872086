// Device-side building blocks for sm_103a: bf16 helpers, programmatic
// dependent launch, mbarriers with bounded waits, TMA (bulk tensor) copies,
// L2 cache policies and the tcgen05 tensor-core / tensor-memory instructions.
//
// Every spin on an mbarrier goes through mbar_wait(), which gives up after a
// wall-clock limit (%globaltimer), raises a CTA-wide abort flag and records
// DEV_ERR_TIMEOUT in the handle's device error word. No kernel in this
// library traps or waits without a limit.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#define DEV_ERR_TIMEOUT 1

namespace dec {

// ---------------------------------------------------------------- bf16 <-> fp32
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Round fp32 to bf16, nearest-even (NaN is kept quiet).
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// acc + w_lo * x_lo + w_hi * x_hi for the two bf16 lanes of 32-bit words w
// and x, in that order: fp32 fused multiply-adds on bf16 operands (a product
// of two bf16 values is exact in fp32, so each step is fmaf of the widened
// operands, rounded once) without widening them first.
__device__ __forceinline__ float fma_bf16x2(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

// acc + sum_i w_i * x_i over the 8 bf16 lanes of two 16-byte vectors, lane
// order, one rounding per step. The bf16 operands are widened to fp32 first.
__device__ __forceinline__ float dot8_widened(const uint4& w, const uint4& x, float acc) {
  acc = fmaf(bf_lo(w.x), bf_lo(x.x), acc);
  acc = fmaf(bf_hi(w.x), bf_hi(x.x), acc);
  acc = fmaf(bf_lo(w.y), bf_lo(x.y), acc);
  acc = fmaf(bf_hi(w.y), bf_hi(x.y), acc);
  acc = fmaf(bf_lo(w.z), bf_lo(x.z), acc);
  acc = fmaf(bf_hi(w.z), bf_hi(x.z), acc);
  acc = fmaf(bf_lo(w.w), bf_lo(x.w), acc);
  acc = fmaf(bf_hi(w.w), bf_hi(x.w), acc);
  return acc;
}

// The same sums with fp32 fused multiply-adds on the bf16 operands (the same
// bits). Measured: the MoE fronts, the fused down projections and the
// small-matrix projections at two tokens stream faster this way (layer step
// 167.8 -> 162.9 us at one token, 285.8 -> 273.1 at two), but the
// single-token projection kernel streams slower (4096 x 4096: 6.3 -> 7.0 us),
// so it keeps the widened form. DEC_MIXED_FMA=0 widens everywhere.
#ifndef DEC_MIXED_FMA
#define DEC_MIXED_FMA 1
#endif
__device__ __forceinline__ float dot8(const uint4& w, const uint4& x, float acc) {
#if DEC_MIXED_FMA
  acc = fma_bf16x2(w.x, x.x, acc);
  acc = fma_bf16x2(w.y, x.y, acc);
  acc = fma_bf16x2(w.z, x.z, acc);
  acc = fma_bf16x2(w.w, x.w, acc);
  return acc;
#else
  return dot8_widened(w, x, acc);
#endif
}

// ---------------------------------------------------------------- global loads
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Streaming read of static weights: no L1 allocation, evict-first in L2.
__device__ __forceinline__ uint4 ld_stream(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// Loads of activations: data written by an earlier kernel. They are volatile
// asm so that the compiler can never move them above pdl_wait() (a const
// __restrict__ pointer would let it hoist them, reading stale data while the
// producer still runs). Only static weights use plain or restrict loads.
__device__ __forceinline__ uint4 ld_act16(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_act8(const void* p) {
  uint2 v;
  asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_act_f4(const void* p) {
  float4 v;
  asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float ld_act_f32(const void* p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_act_s32(const void* p) {
  int v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint16_t ld_act_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
  return v;
}
// L2-level loads (.cg, never served from L1) of values that other CTAs of the
// running kernel wrote before a fence and an atomic hand-off, or that a kernel
// two launches back wrote.
__device__ __forceinline__ float ld_cg_f32(const void* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cg_s32(const void* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Device-scope acquire-release fetch-add (CTA hand-offs through a counter).
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- RMSNorm pieces
// Every kernel that normalises a row uses these two, in the same order: the
// sum of squares runs over each thread's 8-element vectors in ascending order,
// element by element, so a row normalised in any of them has the same bits.
__device__ __forceinline__ float sumsq8(const uint4& a, float ss) {
  const uint32_t ws[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = bf_lo(ws[i]), hi = bf_hi(ws[i]);
    ss = fmaf(lo, lo, ss);
    ss = fmaf(hi, hi, ss);
  }
  return ss;
}
// bf16(x * r * gamma) for 8 elements.
__device__ __forceinline__ uint4 norm8(const uint4& a, const uint4& g, float r) {
  const uint32_t ws[4] = {a.x, a.y, a.z, a.w}, gs[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t l = f2bf(bf_lo(ws[i]) * r * bf_lo(gs[i]));
    const uint16_t u = f2bf(bf_hi(ws[i]) * r * bf_hi(gs[i]));
    o[i] = (uint32_t)l | ((uint32_t)u << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// This thread's partial sum of squares over the vectors it holds of a row:
// v[i] is vector t + T i (those below H8), taken in ascending i.
// (tid: the thread's index among the T threads that hold the row.)
template <int NV, int T>
__device__ __forceinline__ float thread_sumsq(const uint4 (&v)[NV], int H8, float ss = 0.f,
                                              int tid = (int)threadIdx.x) {
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (tid + T * i < H8) ss = sumsq8(v[i], ss);
  return ss;
}

// The RMSNorm scale 1 / sqrt(mean(x^2) + eps) of a row of H elements from each
// thread's partial sum of squares, reduced in the one order that every kernel
// here that normalises a row uses: warp shuffles (xor 16, 8, 4, 2, 1), then the
// NW warps' sums in warp order. A row normalised by any of them therefore has
// the same bits. red: NW floats of shared memory that no other thread is
// still reading; one barrier.
// bar: 0 for the whole block (__syncthreads), else the named barrier of the
// NW warps that hold the row; warp: the calling warp's index among them.
template <int NW>
__device__ __forceinline__ float block_rms_scale(float ss, int H, float eps, float* red, int bar = 0,
                                                 int warp = (int)(threadIdx.x >> 5)) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  if (bar == 0)
    __syncthreads();
  else
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(NW * 32) : "memory");
  float tot = 0.f;
#pragma unroll
  for (int q = 0; q < NW; ++q) tot += red[q];
  return rsqrtf(tot / (float)H + eps);
}

// ---------------------------------------------------------------- SwiGLU, sigmoid
// One SwiGLU output from its gate and up sums, rounded once to bf16:
// silu(g) * u = g / (1 + e^-g) * u.
__device__ __forceinline__ uint16_t swiglu_bf16(float g, float u) { return f2bf(g / (1.0f + expf(-g)) * u); }

// Router score of a logit: 1 / (1 + e^-z).
__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: a kernel may start while its predecessor on
// the stream drains. Everything before pdl_wait() may touch only memory that
// no earlier kernel writes (static weights, shared memory, tensor memory).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Barrier over `count` threads that also returns the AND of `pred` over them,
// so that a group leaves a loop together after bounded waits.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait-control block shared by the roles of one CTA.
struct WaitCtl {
  volatile int* abort;  // shared memory flag: some role gave up
  int* err;             // device error word of the handle
  uint64_t limit_ns;
};

// Bounded wait on phase `parity` of an mbarrier. Returns false if the wait ran
// past its limit (which then raises the abort flag and the error word) or if
// another role of the CTA has aborted.
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (*wc.abort) return false;
      if (globaltimer() - t0 > wc.limit_ns) {
        *wc.abort = 1;
        atomicOr(wc.err, DEV_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used when draining in-flight work).
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* err, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0 && globaltimer() - t0 > limit) {
      atomicOr(err, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tmap_prefetch(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completing on `bar`.
// c0 is the inner (contiguous) coordinate in elements and must be a multiple
// of 8 for bf16 (16 bytes); c1 is the row coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}

// 16-byte asynchronous copy global -> shared that allocates in L2 only (both
// addresses 16-byte aligned), and the wait for all of a thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Request [p, p + bytes) into L2 in bulk pieces of at most 32 KB (p and bytes
// multiples of 16). The small-matrix kernels keep their next rows requested
// this way ahead of the register loads: it holds no registers, so far more
// bytes stay in flight than the register double buffer allows.
__device__ __forceinline__ void request_l2(const void* p, size_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (size_t off = 0; off < bytes; off += 32768) {
    const size_t n = bytes - off < 32768 ? bytes - off : 32768;
    bulk_prefetch_l2(c + off, (uint32_t)n);
  }
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO),
// descriptor version 1 (bits 46-47), layout type 2 = SWIZZLE_128B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;    // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;  // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;             // version
  d |= (uint64_t)2 << 61;             // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// shape M x N (M = 64 or 128 with cta_group::1; N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4)                       // D format: F32
         | (1u << 7)                     // A format: BF16
         | (1u << 10)                    // B format: BF16
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape), with
// the wait for the load folded into the same asm block.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace dec
