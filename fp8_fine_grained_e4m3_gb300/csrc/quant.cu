// quant.cu -- FP32 -> e4m3 quantisers with fine-grained scales.
//
// Rule ("news.rkmt.cn/news/5092" section 5.2: scale = max |x| / 448, one per
// block; "lpnh.cn/news/2822121" section 6.3: round to nearest, not toward
// zero):  amax = max |x| over the block, s = amax / 448 (IEEE FP32 division,
// round to nearest), q = e4m3(x / s) with an IEEE FP32 division and the
// hardware's round-to-nearest-even, saturating conversion.  A block with
// amax = 0 stores s = 0 and zero bytes.  Built without fast-math, so '/'
// here is the correctly rounded division and denormals are kept.
//
// Both kernels are bandwidth-bound (4 bytes read, 1 + 4/128 bytes written
// per element): loads are 16-byte vectors and every warp writes whole 128-byte
// output rows.
//
// Optional saturation count ("blog.hotdry.top: DeepGEMM FP8 GEMM
// fine-grained scaling kernels", section on numerical-stability checks and
// monitoring: track how many FP8 conversions overflow): the number of
// elements of blocks with amax != 0 whose FP32 quotient x / s is not within
// +-limit -- exactly the values the saturating conversion clamps (or, for a
// quotient that is NaN, cannot represent).  With the per-block scale that only
// happens when rounding pushes x / s just past the limit, or when amax / limit
// underflows to 0.  Counted per lane, summed per warp (or CTA) and added once
// to the caller's 64-bit counter, and only in the instances that count.
#include "common.cuh"
#include "f8_convert.cuh"
#include "ptx.cuh"

namespace fp8gemm {
namespace {


constexpr int kQuantUnroll = 4;  // 1x128 blocks per warp (loads kept in flight)

// One warp per group of kQuantUnroll consecutive 1x128 blocks; block b is
// (row b / Kb, K block b % Kb) of the row-major [M, K] input and its scale is
// sX[b].  When K is a multiple of 128 (kRagged false) block b is simply
// elements [128 b, 128 b + 128); otherwise a row's last block holds the
// K % 128 remaining elements (a multiple of 16) and its amax runs over those.
// kPdl: launched as a programmatic dependent of the previous kernel (let the
// next kernel launch at once, then wait for the previous one before the first
// load).
// kCount: add the saturation count to *sat.
template <bool kPdl, bool kRagged, bool kE5M2, bool kCount>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const float* __restrict__ X,
                                                          uint32_t* __restrict__ Q,
                                                          float* __restrict__ sX,
                                                          long long nblocks, int K, int Kb,
                                                          unsigned long long* sat) {
  const long long warp0 =
      ((long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * kQuantUnroll;
  const int lane = threadIdx.x % 32;
  if constexpr (kPdl) {
    // the next kernel may launch before this one's own wait: it still waits
    // for this grid's completion (and so for the kernel before it) before it
    // reads what this one writes
    griddep_launch_dependents();
    griddep_wait();
  }
  float4 v[kQuantUnroll];
  long long e0[kQuantUnroll];  // first element of the block
  bool in[kQuantUnroll];       // this lane's 4 elements exist
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const long long b = warp0 + u;
    if constexpr (kRagged) {
      const long long m = b / Kb;
      const int kb = int(b - m * Kb);
      e0[u] = m * K + kb * kBlockK;
      in[u] = b < nblocks && lane * 4 < K - kb * kBlockK;
    } else {
      e0[u] = b * kBlockK;
      in[u] = b < nblocks;
    }
    v[u] = in[u] ? __ldcs(reinterpret_cast<const float4*>(X + e0[u]) + lane)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  unsigned n_sat = 0;
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const long long b = warp0 + u;
    if (b >= nblocks) break;
    float amax = absmax4(v[u]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, f8_limit<kE5M2>());
    if (in[u]) Q[e0[u] / 4 + lane] = amax != 0.f ? quant4<kE5M2, kCount>(v[u], s, &n_sat) : 0u;
    if (lane == 0) sX[b] = s;
  }
  if constexpr (kCount) {
    n_sat = __reduce_add_sync(0xffffffffu, n_sat);
    if (lane == 0 && n_sat != 0) atomicAdd(sat, (unsigned long long)n_sat);
  }
}

// One CTA (kQ2Threads threads) per 128x128 tile of one [N, K] matrix of the
// batch.  Thread t covers column group t % 32 (4 columns) of rows
// t / 32 + kQ2Warps * i (8 float4).  The FP32 tile (64 KB) is copied into
// shared memory with cp.async rather than held in registers, so three CTAs
// (192 KB of copies in flight) share an SM -- 7168 x 16384 in 94 us against
// 141 with the tile in registers (64 registers a thread, two CTAs).  Each
// thread reads back only the elements it copied, after its own wait.  The
// last K tile may be partial (K % 128 columns, a multiple of 16).
// kCount: add the saturation count to *sat.
constexpr int kQ2Threads = 512;
constexpr int kQ2Warps = kQ2Threads / 32;
constexpr int kQ2Rows = 128 / kQ2Warps;  // rows per thread

template <bool kE5M2, bool kCount>
__global__ void __launch_bounds__(kQ2Threads, 3) quant_128x128_kernel(const float* __restrict__ W,
                                                               uint8_t* __restrict__ Q,
                                                               float* __restrict__ sW, int N,
                                                               int K, unsigned long long* sat) {
  const int Kb = ceil_div(K, kBlockK);
  const int Nb = ceil_div(N, 128);
  const int kb = blockIdx.x;
  const int nb = blockIdx.y;
  const int e = blockIdx.z;
  const int cg = threadIdx.x % 32;
  const int r0 = threadIdx.x / 32;
  const size_t mat = size_t(e) * N * K;
  const bool col_in = cg * 4 < K - kb * kBlockK;  // this thread's 4 columns exist
  extern __shared__ float4 tile4[];  // [128 rows][32 float4]
  __shared__ float red[kQ2Warps];

  // the tile goes to shared memory without passing through registers; each
  // thread later reads back only what it copied
#pragma unroll
  for (int i = 0; i < kQ2Rows; ++i) {
    const int n = nb * 128 + r0 + kQ2Warps * i;
    const bool in = n < N && col_in;
    const float* src = in ? W + mat + size_t(n) * K + kb * kBlockK + cg * 4 : W;
    cp_async_16(smem_addr(&tile4[(r0 + kQ2Warps * i) * 32 + cg]), src, in ? 16u : 0u);
  }
  cp_async_wait_all();
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kQ2Rows; ++i) amax = fmaxf(amax, absmax4(tile4[(r0 + kQ2Warps * i) * 32 + cg]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (cg == 0) red[r0] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQ2Warps; ++w) amax = fmaxf(amax, red[w]);
  const float s = __fdiv_rn(amax, f8_limit<kE5M2>());
  unsigned n_sat = 0;
#pragma unroll
  for (int i = 0; i < kQ2Rows; ++i) {
    const int n = nb * 128 + r0 + kQ2Warps * i;
    if (n < N && col_in) {
      const float4 v = tile4[(r0 + kQ2Warps * i) * 32 + cg];
      uint32_t* dst = reinterpret_cast<uint32_t*>(Q + mat + size_t(n) * K + kb * kBlockK) + cg;
      uint32_t q = 0u;
      if (amax != 0.f) q = quant4<kE5M2, kCount>(v, s, &n_sat);
      *dst = q;
    }
  }
  if (threadIdx.x == 0) sW[(size_t(e) * Nb + nb) * Kb + kb] = s;
  if constexpr (kCount) {
    // amax (and so every thread's path above) is uniform over the CTA
    __shared__ unsigned cnt[kQ2Warps];
    n_sat = __reduce_add_sync(0xffffffffu, n_sat);
    if (cg == 0) cnt[r0] = n_sat;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned t = 0;
#pragma unroll
      for (int w = 0; w < kQ2Warps; ++w) t += cnt[w];
      if (t != 0) atomicAdd(sat, (unsigned long long)t);
    }
  }
}

}  // namespace

namespace {

template <bool kE5M2, bool kCount>
cudaError_t launch_1x128(const LaunchCtx& c, const float* X, uint8_t* Q, float* sX, int M,
                         int K, unsigned long long* sat) {
  const int Kb = ceil_div(K, kBlockK);
  const long long nblocks = (long long)M * Kb;
  if (nblocks == 0) return cudaSuccess;
  const long long per_cta = 8LL * kQuantUnroll;
  const long long grid = (nblocks + per_cta - 1) / per_cta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const bool ragged = K % kBlockK != 0;
  uint32_t* Q4 = reinterpret_cast<uint32_t*>(Q);
  if (grid > 8LL * c.num_sms) {  // more than one wave: plain launch
    if (ragged)
      quant_1x128_kernel<false, true, kE5M2, kCount>
          <<<unsigned(grid), 256, 0, c.stream>>>(X, Q4, sX, nblocks, K, Kb, sat);
    else
      quant_1x128_kernel<false, false, kE5M2, kCount>
          <<<unsigned(grid), 256, 0, c.stream>>>(X, Q4, sX, nblocks, K, Kb, sat);
    return cudaGetLastError();
  }
  // A decode-sized quantisation (one wave) is launched as a programmatic
  // dependent of the previous kernel and lets the next one launch before its
  // own wait, so that its launch, and the prologue of the GEMM after it (with
  // read-only weights: its first weight tiles), overlap the kernel before --
  // two launches from FP32 activations at 1 x 2048 x 7168: 8.9 -> 8.1 us,
  // read-only 8.35 -> 7.4.  (Not for large grids: there every short CTA would
  // pay the dependency wait.)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (ragged)
    return cudaLaunchKernelEx(&cfg, quant_1x128_kernel<true, true, kE5M2, kCount>, X, Q4, sX,
                              nblocks, K, Kb, sat);
  return cudaLaunchKernelEx(&cfg, quant_1x128_kernel<true, false, kE5M2, kCount>, X, Q4, sX,
                            nblocks, K, Kb, sat);
}

}  // namespace

cudaError_t launch_quant_1x128(const LaunchCtx& c, const float* X, uint8_t* Q, float* sX,
                               int M, int K, int fmt, unsigned long long* sat) {
  if (sat != nullptr)
    return fmt == FP8GEMM_FMT_E5M2 ? launch_1x128<true, true>(c, X, Q, sX, M, K, sat)
                                   : launch_1x128<false, true>(c, X, Q, sX, M, K, sat);
  return fmt == FP8GEMM_FMT_E5M2 ? launch_1x128<true, false>(c, X, Q, sX, M, K, nullptr)
                                 : launch_1x128<false, false>(c, X, Q, sX, M, K, nullptr);
}

cudaError_t launch_quant_128x128(const LaunchCtx& c, const float* W, uint8_t* Q, float* sW,
                                 int E, int N, int K, int fmt, unsigned long long* sat) {
  if (E == 0 || N == 0 || K == 0) return cudaSuccess;
  const int Nb = ceil_div(N, 128);
  if (Nb > 65535 || E > 65535) return cudaErrorInvalidValue;
  dim3 grid(ceil_div(K, kBlockK), Nb, E);
  const bool e5 = fmt == FP8GEMM_FMT_E5M2;
  constexpr int kTile = 128 * 128 * 4;  // the FP32 tile in shared memory
  // once per device and context: the attribute belongs to the function in
  // one context, and a cudaDeviceReset gives the device a new one
  static unsigned long long set_in[64] = {};  // context id, per device
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || set_in[dev & 63] != ctx) {
    cudaError_t e = cudaFuncSetAttribute(quant_128x128_kernel<true, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kTile);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(quant_128x128_kernel<false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kTile);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(quant_128x128_kernel<true, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kTile);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(quant_128x128_kernel<false, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kTile);
    if (e != cudaSuccess) return e;
    set_in[dev & 63] = ctx;
  }
  if (sat != nullptr) {
    if (e5)
      quant_128x128_kernel<true, true><<<grid, kQ2Threads, kTile, c.stream>>>(W, Q, sW, N, K, sat);
    else
      quant_128x128_kernel<false, true><<<grid, kQ2Threads, kTile, c.stream>>>(W, Q, sW, N, K, sat);
  } else if (e5) {
    quant_128x128_kernel<true, false><<<grid, kQ2Threads, kTile, c.stream>>>(W, Q, sW, N, K, nullptr);
  } else {
    quant_128x128_kernel<false, false><<<grid, kQ2Threads, kTile, c.stream>>>(W, Q, sW, N, K, nullptr);
  }
  return cudaGetLastError();
}

}  // namespace fp8gemm
