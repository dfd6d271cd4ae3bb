// noalloc.cu -- fp8gemm_dense_small_m_noalloc: the decode-shape dense GEMM
// (M <= 64) with its split-K scratch in a fixed, statically allocated device
// array instead of a workspace the library obtains with cudaMalloc.
//
// Why: some callers must not have a library allocate device memory behind
// their back -- an inference server that reserves its whole memory budget at
// start-up and treats any later allocation as a failure; a framework whose own
// caching allocator holds the device memory, so a stray cudaMalloc either fails
// or fragments the pool; a latency-critical loop that cannot afford
// cudaMalloc's implicit device-wide synchronisation.  This entry point calls
// no allocating routine at all.  The price is a fixed footprint: the array
// below (kScratchBytes, 10.25 MiB) is created on a GPU when this file's module
// is loaded there -- under CUDA's default lazy loading, by the first call of
// this entry point on that GPU -- and stays until the process exits.
//
// Sharing: every call on a device uses the same array.  Calls that overlap on
// the GPU (for example on two streams at once) race on it and give wrong
// results; serialise them.  The array keeps the last call's contents, so each
// call first clears the part that must start at zero (the per-tile arrival
// counters) with an asynchronous memset on the caller's stream.
//
// The pages this library follows describe no such variant; it exists only for
// the allocation constraint above.
#include <mutex>

#include "common.cuh"

namespace fp8gemm {
namespace {

constexpr int kNoAllocMaxCtas = 160;  // one CTA per SM, up to 160 SMs
constexpr int kNoAllocMaxM = 64;      // activation rows (decode shapes)
constexpr size_t kNoAllocCounterBytes = 256 * 1024;  // one int per 128 output columns
constexpr size_t kScratchBytes =
    kNoAllocCounterBytes + size_t(2) * kNoAllocMaxCtas * kNoAllocMaxM * 128 * sizeof(float);

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device and context with that device current: the first call on each
// device does this set-up (and loads the module that holds the array), so
// that first call belongs before any CUDA stream capture.  After a
// cudaDeviceReset the device has a new context and the address is looked up
// again.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return FP8GEMM_ERR_LAUNCH;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx || ctx == 0) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FP8GEMM_ERR_LAUNCH;
    }
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();
  }
  *out = g_scratch_addr[dev];
  return FP8GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace fp8gemm

using namespace fp8gemm;

extern "C" int fp8gemm_dense_small_m_noalloc(const uint8_t* A, const float* sA, const uint8_t* B,
                                             const float* sB, void* D, int M, int N, int K,
                                             fp8gemm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return FP8GEMM_ERR_SHAPE;
  if (K == 0 || K % 16 != 0) return FP8GEMM_ERR_SHAPE;  // TMA: row strides are 16-B multiples
  if (M == 0 || N == 0) return FP8GEMM_OK;
  const int n_tiles = ceil_div(N, 128);
  if (M > kNoAllocMaxM || size_t(n_tiles) * sizeof(int) > kNoAllocCounterBytes)
    return FP8GEMM_ERR_SCRATCH_LIMIT;
  if (!A || !sA || !B || !sB || !D) return FP8GEMM_ERR_NULL;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D))
    return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = make_launch_ctx(stream, &c)) return r;
  if (c.num_sms > kNoAllocMaxCtas) c.num_sms = kNoAllocMaxCtas;
  if (small_m_workspace_bytes(c.num_sms, N) > kScratchBytes) return FP8GEMM_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  if (int r = scratch_address(&ws)) return r;
  // the arrival counters must start at zero; the partial-sum slots need not
  if (cudaMemsetAsync(ws, 0, size_t(n_tiles) * sizeof(int), stream) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ERR_LAUNCH;
  }
  GemmArgs a{GemmMode::kDense, A, sA, B, sB, nullptr, static_cast<__nv_bfloat16*>(D),
             M, N, K, 1};
  if (launch_gemm_small_m(c, a, ws, kScratchBytes) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ERR_LAUNCH;
  }
  count_kernel_launches(1);
  return FP8GEMM_OK;
}
