// Device filler for the seeded synthetic inputs. Same definition as the host
// filler (synth_arith.h); used only to place large synthetic weight banks in
// device memory quickly. The tests check that its bytes equal the host
// filler's.
#include <cstdint>
#include <cuda_runtime.h>

#include "synth_arith.h"

namespace {

__global__ void fill_bf16_kernel(uint16_t* __restrict__ dst, uint64_t n, uint64_t key, uint64_t offset,
                                 double sigma) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = synth_bf16(key, offset + i, sigma);
}

__global__ void fill_f32_kernel(uint32_t* __restrict__ dst, uint64_t n, uint64_t key, uint64_t offset,
                                double sigma) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = synth_f32(key, offset + i, sigma);
}

int grid_for(uint64_t n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  uint64_t blocks = (n + 255) / 256;
  uint64_t cap = (uint64_t)sms * 8;
  return (int)(blocks < cap ? (blocks ? blocks : 1) : cap);
}

}  // namespace

extern "C" int synth_fill_bf16_dev(void* dst, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t offset,
                                   double sigma, void* stream) {
  if (n == 0) return 0;
  fill_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint16_t*)dst, n, synth_key(seed, tensor_id),
                                                                   offset, sigma);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_f32_dev(void* dst, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t offset,
                                  double sigma, void* stream) {
  if (n == 0) return 0;
  fill_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint32_t*)dst, n, synth_key(seed, tensor_id),
                                                                  offset, sigma);
  return (int)cudaGetLastError();
}
