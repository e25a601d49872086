// dec_linear_noalloc: the split-K projection for callers that cannot hand the
// library a workspace. Its scratch (split-K partial sums and per-tile arrival
// counters) lives in one static device array of fixed size instead.
#include <mutex>

#include "internal.h"

using namespace dec;

namespace {

constexpr int kNoAllocMaxCtas = 160;         // persistent CTAs the scratch has partial slots for
constexpr long long kNoAllocMaxTiles = 1024; // 128-row tiles: N <= 131072
constexpr size_t kNoAllocCounterBytes = (size_t)kNoAllocMaxTiles * sizeof(int);  // 4 KiB, first
constexpr size_t kNoAllocPartialBytes =
    (size_t)2 * kNoAllocMaxCtas * kTileN * kMaxCols * sizeof(float);             // 10 MiB
constexpr size_t kNoAllocScratchBytes = kNoAllocCounterBytes + kNoAllocPartialBytes;

// One copy per GPU that loads the library, held until the process exits.
// In host code this name is only a stand-in for the symbol, never a device
// address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `device`, looked up once per device
// with that device current; the caller's current device is restored (a
// failure to restore it is returned as an error).
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[device] == nullptr) {
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (prev != device) {
      const cudaError_t r = cudaSetDevice(prev);
      if (e == cudaSuccess) e = r;
    }
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

// Forget a device's address after a failed call, so that the next call looks
// it up again.
void forget_scratch_address(int device) {
  if (device < 0 || device >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_mu);
  g_scratch_addr[device] = nullptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dec_status dec_linear_noalloc(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W,
                                         const dec_bf16* r, dec_bf16* out, int M, int N, int K,
                                         cudaStream_t stream) {
  if (h == nullptr || x == nullptr || W == nullptr || out == nullptr) return DEC_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W) || !aligned16(out) || (r != nullptr && !aligned16(r)))
    return DEC_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxCols || N < 1 || K < 8 || K % 8 != 0 || ldx < K || ldx % 8 != 0) return DEC_ERR_INVALID_ARG;
  const long long tiles = (N + kTileN - 1) / kTileN;
  if (tiles > kNoAllocMaxTiles) return DEC_ERR_UNSUPPORTED;  // N above the scratch's 131072-row limit

  void* base = nullptr;
  if (scratch_address(h->device, &base) != cudaSuccess) return DEC_ERR_CUDA;
  int* counters = static_cast<int*>(base);
  float* partials = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kNoAllocCounterBytes);

  EngineLaunch L;
  L.epi = EPI_LINEAR;
  L.A = W;
  L.a_rows = N;
  L.B = x;
  L.b_rows = M;
  L.ldb = ldx;
  L.K = K;
  L.N = N;
  L.count = M;
  L.out = out;
  L.ldo = N;
  L.res = r;
  L.ldr = N;
  L.partials = partials;
  L.counters = counters;
  L.grid = h->sms < kNoAllocMaxCtas ? h->sms : kNoAllocMaxCtas;
  h->last_variant = DEC_VARIANT_SPLIT_K;
  cudaError_t e;
  {
    // The array keeps whatever the previous call left; the counters must start at zero.
    LaunchScope scope(h, "linear_noalloc", stream);
    e = cudaMemsetAsync(counters, 0, (size_t)tiles * sizeof(int), stream);
    if (e == cudaSuccess) e = launch_engine(h, L, stream);
  }
  if (e != cudaSuccess) {
    forget_scratch_address(h->device);
    return DEC_ERR_CUDA;
  }
  return DEC_OK;
}
