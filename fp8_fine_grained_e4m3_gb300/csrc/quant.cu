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
#include "common.cuh"
#include "ptx.cuh"

namespace fp8gemm {
namespace {

// Two FP32 values -> two e4m3 bytes (lo in the low byte), round to nearest
// even, saturate to +-448.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t quant4(float4 v, float s) {
  const float q0 = __fdiv_rn(v.x, s), q1 = __fdiv_rn(v.y, s);
  const float q2 = __fdiv_rn(v.z, s), q3 = __fdiv_rn(v.w, s);
  return cvt_e4m3x2(q0, q1) | (cvt_e4m3x2(q2, q3) << 16);
}

__device__ __forceinline__ float absmax4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

constexpr int kQuantUnroll = 4;  // 1x128 blocks per warp (loads kept in flight)

// One warp per group of kQuantUnroll consecutive 1x128 blocks.  Block b
// covers elements [128 b, 128 b + 128) of the row-major [M, K] input (K is a
// multiple of 128), and its scale is sX[b].  kPdl: launched as a
// programmatic dependent of the previous kernel (wait for it before the first
// load; let the next kernel launch right away).
template <bool kPdl>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const float4* __restrict__ X,
                                                          uint32_t* __restrict__ Q,
                                                          float* __restrict__ sX,
                                                          long long nblocks) {
  const long long warp0 =
      ((long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * kQuantUnroll;
  const int lane = threadIdx.x % 32;
  if constexpr (kPdl) {
    griddep_wait();
    griddep_launch_dependents();
  }
  float4 v[kQuantUnroll];
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const long long b = warp0 + u;
    v[u] = b < nblocks ? __ldcs(X + b * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const long long b = warp0 + u;
    if (b >= nblocks) break;
    float amax = absmax4(v[u]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, kE4M3Max);
    Q[b * 32 + lane] = amax != 0.f ? quant4(v[u], s) : 0u;
    if (lane == 0) sX[b] = s;
  }
}

// One CTA (256 threads) per 128x128 tile of one [N, K] matrix of the batch.
// Thread t covers column group t % 32 (4 columns) of rows t / 32 + 8 i.
__global__ void __launch_bounds__(256) quant_128x128_kernel(const float* __restrict__ W,
                                                            uint8_t* __restrict__ Q,
                                                            float* __restrict__ sW, int N,
                                                            int K) {
  const int Kb = K / kBlockK;
  const int Nb = ceil_div(N, 128);
  const int kb = blockIdx.x;
  const int nb = blockIdx.y;
  const int e = blockIdx.z;
  const int cg = threadIdx.x % 32;
  const int r0 = threadIdx.x / 32;
  const size_t mat = size_t(e) * N * K;
  __shared__ float red[8];

  float4 v[16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int n = nb * 128 + r0 + 8 * i;
    if (n < N) {
      v[i] = __ldcs(reinterpret_cast<const float4*>(W + mat + size_t(n) * K + kb * kBlockK) + cg);
      amax = fmaxf(amax, absmax4(v[i]));
    } else {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (cg == 0) red[r0] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float s = __fdiv_rn(amax, kE4M3Max);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int n = nb * 128 + r0 + 8 * i;
    if (n < N) {
      uint32_t* dst = reinterpret_cast<uint32_t*>(Q + mat + size_t(n) * K + kb * kBlockK) + cg;
      *dst = amax != 0.f ? quant4(v[i], s) : 0u;
    }
  }
  if (threadIdx.x == 0) sW[(size_t(e) * Nb + nb) * Kb + kb] = s;
}

}  // namespace

cudaError_t launch_quant_1x128(const LaunchCtx& c, const float* X, uint8_t* Q, float* sX,
                               int M, int K) {
  const long long nblocks = (long long)M * (K / kBlockK);
  if (nblocks == 0) return cudaSuccess;
  const long long per_cta = 8LL * kQuantUnroll;
  const long long grid = (nblocks + per_cta - 1) / per_cta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (grid > 8LL * c.num_sms) {  // more than one wave: plain launch
    quant_1x128_kernel<false><<<unsigned(grid), 256, 0, c.stream>>>(
        reinterpret_cast<const float4*>(X), reinterpret_cast<uint32_t*>(Q), sX, nblocks);
    return cudaGetLastError();
  }
  // A decode-sized quantisation (one wave) is launched as a programmatic
  // dependent of the previous kernel, so that its launch, and the prologue of
  // the GEMM after it, overlap the kernel before.  (Not for large grids: there
  // every short CTA would pay the dependency wait.)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_1x128_kernel<true>, reinterpret_cast<const float4*>(X),
                            reinterpret_cast<uint32_t*>(Q), sX, nblocks);
}

cudaError_t launch_quant_128x128(const LaunchCtx& c, const float* W, uint8_t* Q, float* sW,
                                 int E, int N, int K) {
  if (E == 0 || N == 0 || K == 0) return cudaSuccess;
  const int Nb = ceil_div(N, 128);
  if (Nb > 65535 || E > 65535) return cudaErrorInvalidValue;
  dim3 grid(K / kBlockK, Nb, E);
  quant_128x128_kernel<<<grid, 256, 0, c.stream>>>(W, Q, sW, N, K);
  return cudaGetLastError();
}

}  // namespace fp8gemm
