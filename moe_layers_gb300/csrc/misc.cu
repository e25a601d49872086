// RMSNorm, the L2 prefetch kernel and the two test-hook kernels.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dec {

// y = x / sqrt(mean(x^2) + eps) * gamma, one CTA per row, fp32 math. The
// pre-norm of the decode layer (not named on the pages). Rows of up to 8192
// elements (VPT <= 4 vectors per thread) are read once into registers; longer
// rows are read twice. The sum of squares is accumulated per thread over its
// vectors in ascending order, reduced by warp shuffles, then over the warps in
// order (the small-matrix projection repeats exactly this order when it
// normalises its input itself). y may alias x: each element is written by the
// thread that read it, after the block reduction.
template <int VPT>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* x, const uint16_t* __restrict__ gamma,
                                                      uint16_t* y, int H, float eps) {
  const int tid = threadIdx.x;
  const uint16_t* xr = x + (size_t)blockIdx.x * H;
  uint16_t* yr = y + (size_t)blockIdx.x * H;
  __shared__ float red[8];
  pdl_trigger();
  pdl_wait();
  const int H8 = H >> 3;
  uint4 xv[VPT > 0 ? VPT : 1];
  float ss = 0.f;
  if (VPT > 0) {
#pragma unroll
    for (int j = 0; j < (VPT > 0 ? VPT : 1); ++j) {
      const int v = tid + 256 * j;
      if (v < H8) {
        xv[j] = ld_act16(xr + (size_t)v * 8);
        ss = sumsq8(xv[j], ss);
      }
    }
  } else {
    for (int v = tid; v < H8; v += blockDim.x) ss = sumsq8(ld_act16(xr + (size_t)v * 8), ss);
  }
  const float r = block_rms_scale<8>(ss, H, eps, red);
  auto put = [&](int v, const uint4& a) {
    const uint4 g = *reinterpret_cast<const uint4*>(gamma + (size_t)v * 8);
    *reinterpret_cast<uint4*>(yr + (size_t)v * 8) = norm8(a, g, r);
  };
  if (VPT > 0) {
#pragma unroll
    for (int j = 0; j < (VPT > 0 ? VPT : 1); ++j) {
      const int v = tid + 256 * j;
      if (v < H8) put(v, xv[j]);
    }
  } else {
    for (int v = tid; v < H8; v += blockDim.x) put(v, ld_act16(xr + (size_t)v * 8));
  }
}

// Kimi K3 article, Part 1 §4 "Prefetching": while a phase leaves memory
// bandwidth idle, a kernel on a secondary stream pulls the next operator's
// weights into the cache. Bulk L2 prefetches of 32 KB chunks, evict-last.
__global__ void __launch_bounds__(64) prefetch_kernel(const uint8_t* p, size_t bytes) {
  constexpr size_t kChunk = 32768;
  const size_t nchunks = (bytes + kChunk - 1) / kChunk;
  const uint64_t pol = policy_evict_last();
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < nchunks; q += (size_t)gridDim.x * blockDim.x) {
    const size_t off = q * kChunk;
    const uint32_t sz = (uint32_t)std::min(kChunk, bytes - off);
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p + off), "r"(sz), "l"(pol)
                 : "memory");
  }
}

// Test hook: an mbarrier that nothing arrives on. The bounded wait must give
// up after the limit and record the timeout in the error word.
__global__ void wait_probe_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_flag, err, limit_ns};
    (void)mbar_wait(&bar, 0, wc);
  }
  __syncthreads();
}

// Test hook: a slow producer. Triggers its dependents at once (so a
// programmatically dependent consumer launches early), spins for delay_ns on
// the global timer, then copies.
__global__ void delayed_copy_kernel(uint4* dst, const uint4* src, size_t n16, unsigned long long delay_ns) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < delay_ns) __nanosleep(2000);
  }
  __syncthreads();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// Test hook: one 32-thread CTA per SM on `ctas` SMs (each asks for the whole
// per-block shared memory, so no other CTA fits beside it) that sleeps until
// hold_ns have passed on the global timer, then exits. It writes nothing.
constexpr int kOccupySmem = 227 * 1024;
__global__ void __launch_bounds__(32) occupy_kernel(unsigned long long hold_ns) {
  extern __shared__ uint8_t occupy_smem[];
  if (threadIdx.x == 0) {
    occupy_smem[0] = 0;
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < hold_ns) __nanosleep(4000);
  }
  __syncwarp();
}

cudaError_t launch_occupy(dec_handle* h, int ctas, uint64_t hold_ns, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOccupySmem);
  if (e != cudaSuccess) return e;
  occupy_kernel<<<ctas, 32, kOccupySmem, s>>>((unsigned long long)hold_ns);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(dec_handle* h, const uint16_t* x, const uint16_t* gamma, uint16_t* y, int M, int H,
                           float eps, cudaStream_t s) {
  const int H8 = H / 8;
  if (H8 <= 256) return launch_k(h, rmsnorm_kernel<1>, dim3(M), dim3(256), 0, s, x, gamma, y, H, eps);
  if (H8 <= 512) return launch_k(h, rmsnorm_kernel<2>, dim3(M), dim3(256), 0, s, x, gamma, y, H, eps);
  if (H8 <= 1024) return launch_k(h, rmsnorm_kernel<4>, dim3(M), dim3(256), 0, s, x, gamma, y, H, eps);
  return launch_k(h, rmsnorm_kernel<0>, dim3(M), dim3(256), 0, s, x, gamma, y, H, eps);
}

cudaError_t launch_prefetch(dec_handle* h, const void* p, size_t bytes, int ctas, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  const size_t nchunks = (bytes + 32767) / 32768;
  int grid = (int)std::min<size_t>((size_t)std::max(ctas, 1), (nchunks + 63) / 64);
  if (grid < 1) grid = 1;
  prefetch_kernel<<<grid, 64, 0, s>>>(reinterpret_cast<const uint8_t*>(p), bytes);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(dec_handle* h, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(h->d_err, h->wait_ns);
  return cudaGetLastError();
}

cudaError_t launch_delayed_copy(dec_handle* h, void* dst, const void* src, size_t bytes, uint64_t delay_ns,
                                cudaStream_t s) {
  const size_t n16 = bytes / 16;
  const int grid = (int)std::max<size_t>(1, std::min<size_t>((n16 + 255) / 256, (size_t)h->sms));
  return launch_k(h, delayed_copy_kernel, dim3(grid), dim3(256), 0, s, reinterpret_cast<uint4*>(dst),
                  reinterpret_cast<const uint4*>(src), n16, (unsigned long long)delay_ns);
}

}  // namespace dec
