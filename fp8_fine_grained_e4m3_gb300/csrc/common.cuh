// common.cuh -- definitions shared by the kernels and the host launcher.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8gemm.h"

namespace fp8gemm {

constexpr int kBlockK = 128;  // K block of the scaling granularity (= 128 e4m3 bytes)
constexpr int kBlockM = 128;  // rows per tile (= TMEM lanes)
constexpr float kE4M3Max = 448.0f;

// Kernels report device-side conditions through a per-device status word
// (first error wins); the host passes its address to every launch.
__device__ __forceinline__ void raise_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ launch hooks
// Each kernel file exposes one host function that launches its kernels; the
// C ABI in api.cu validates arguments and then calls these.

struct LaunchCtx {
  cudaStream_t stream;
  int num_sms;
  int* status;  // device address of the status word
};

// The quantisers; sat (device, may be null) receives the saturation count.
cudaError_t launch_quant_1x128(const LaunchCtx& c, const float* X, uint8_t* Q, float* sX,
                               int M, int K, int fmt = FP8GEMM_FMT_E4M3,
                               unsigned long long* sat = nullptr);
cudaError_t launch_quant_128x128(const LaunchCtx& c, const float* W, uint8_t* Q, float* sW,
                                 int E, int N, int K, int fmt = FP8GEMM_FMT_E4M3,
                                 unsigned long long* sat = nullptr);

// Problem description for the persistent tensor-core GEMM.
enum class GemmMode : int { kDense = 0, kContiguous = 1, kMasked = 2 };

struct GemmArgs {
  GemmMode mode;
  const uint8_t* A;
  const float* sA;
  const uint8_t* B;
  const float* sB;
  const int32_t* group_info;  // m_indices (contiguous) or masked_m (masked)
  __nv_bfloat16* D;
  int M;      // dense: M; contiguous: M_pad; masked: M_max (rows per expert)
  int N, K;
  int E;      // experts (1 for dense)
  int a_fmt = FP8GEMM_FMT_E4M3;  // operand formats (tensor-core type codes: e4m3 0, e5m2 1)
  int b_fmt = FP8GEMM_FMT_E4M3;
  // Parts per tile along K (persistent tensor-core GEMM, split instance:
  // one cluster of `split` CTAs per tile).  1: whole tiles.
  int split = 1;
  // Time limit of every pipeline wait in the kernel (the launcher fills in
  // the process-wide setting, fp8gemm_set_wait_limit_ns).
  unsigned long long wait_ns = 2000000000ull;
  // The caller's promise (FP8GEMM_FLAG_B_READ_ONLY) that no kernel still
  // running when this one starts writes B or sB: a programmatic dependent may
  // then load weights before waiting for the kernels ahead of it.
  int b_read_only = 0;
  // Persistent tensor-core GEMM: D's tensor map is valid, so whole 32-row
  // bands of a tile leave through shared memory and TMA stores.
  int d_tma = 0;
};

constexpr int kMaxSplit = 8;  // parts (cluster CTAs) per split tile, at most

// The persistent tensor-core GEMM (one launch; the count goes to *launches).
cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmArgs& a, int* launches);
// Up to FP8GEMM_MAX_DENSE_BATCH independent dense problems (host array `p`,
// validated) in one launch of the persistent tensor-core GEMM, tiles handed
// out through `counter` (two zeroed words; each launch leaves them at zero).
cudaError_t launch_gemm_tc_batch(const LaunchCtx& c, const fp8gemm_problem* p, int count,
                                 unsigned int* counter, int* launches);
// The contiguous form in expert-segment order (a one-CTA ordering kernel,
// then the persistent GEMM claiming tiles in that order): the workspace it
// needs (its counters left at zero by every launch), 0 where the form does
// not apply -- then launch_gemm_tc takes the call.
size_t contig_order_workspace_bytes(const LaunchCtx& c, const GemmArgs& a);
cudaError_t launch_gemm_tc_contiguous_ordered(const LaunchCtx& c, const GemmArgs& a, void* ws,
                                              size_t ws_bytes, int* launches);
cudaError_t launch_gemm_small_m(const LaunchCtx& c, const GemmArgs& a, void* workspace,
                                size_t workspace_bytes);
size_t small_m_workspace_bytes(int num_sms, int N);
// The dense decode path: cluster split-K where it fills the SMs (no
// workspace), stream-K through `ws` otherwise.
bool small_m_uses_workspace(const LaunchCtx& c, const GemmArgs& a);
cudaError_t launch_gemm_small_m_any(const LaunchCtx& c, const GemmArgs& a, void* ws,
                                    size_t ws_bytes);
// The dense decode path from FP32 activations X (M <= 64), quantised on load
// inside the GEMM, with Q / sA (both or neither) written too; *taken = false
// when the shape does not qualify (nothing is launched).
cudaError_t launch_gemm_small_m_quant(const LaunchCtx& c, const GemmArgs& a, const float* X,
                                      uint8_t* Q, float* sA, bool* taken);

// Many decode-sized problems from a device-resident table (gemm_table.cu),
// K split over the CTAs (stream-K) through a zeroed workspace of
// table_workspace_bytes bytes whose counters each launch leaves at zero.
size_t table_workspace_bytes(const LaunchCtx& c, int max_M);
cudaError_t launch_gemm_table(const LaunchCtx& c, const fp8gemm_problem* tab, int P, int max_M,
                              void* ws, size_t ws_bytes);

// Fills `c` for the current device and `stream` (SM count, status word);
// returns an fp8gemm_status code.  Defined in api.cu.
int make_launch_ctx(cudaStream_t stream, LaunchCtx* c);
// Adds to the host-side count of kernels enqueued.  Defined in api.cu.
void count_kernel_launches(int n);
// Unique id of the calling thread's current CUDA context, 0 if none: device
// addresses cached per device are valid within one context only.  api.cu.
unsigned long long current_context_id();
// The pipeline-wait time limit kernels launched now get, in ns.  api.cu.
unsigned long long wait_limit_ns();

// Encodes a 2-D K-major uint8 tensor map with 128-byte swizzling:
// rows x cols bytes, box of box_rows x 128 bytes.  Defined in api.cu.
bool make_tmap_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows);
// Encodes a 2-D row-major bf16 tensor map with 64-byte swizzling: rows x
// cols elements, box of box_rows x 32 elements (64 bytes).  False when the
// layout cannot be described (base not 16-byte aligned, cols * 2 not a
// multiple of 16).  Defined in api.cu.
bool make_tmap_bf16_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows);

}  // namespace fp8gemm
