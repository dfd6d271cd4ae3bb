// api.cu -- the C ABI of libfp8gemm.so (declared in include/fp8gemm.h).
//
// Every entry point validates its arguments on the host and only then
// enqueues kernels ("lpnh.cn/news/2822121" section 4.2: do the expensive
// checking and configuration on the host, so the kernel only loops; section
// 6.3, first point: TMA wants 16-byte aligned addresses and strides).
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "common.cuh"

namespace fp8gemm {

// Per-device status word (one instance per device the library is loaded on).
__device__ int g_device_status = 0;
// Where exchange_status leaves the word it took.
__device__ int g_status_taken = 0;

// Reads and clears the status word in one atomic step, so that a condition a
// kernel on another stream raises meanwhile is either returned or kept.
__global__ void exchange_status(int* status) { g_status_taken = atomicExch(status, 0); }

namespace {

std::atomic<unsigned long long> g_launches{0};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

struct DeviceInfo {
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;
  unsigned long long ctx = 0;  // context the device address above belongs to
  bool ok = false;
};

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  unsigned long long ctx = 0;  // context it was allocated in
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::tuple<int, cudaStream_t, int>, Workspace> g_workspaces;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return EncodeTiledFn(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

}  // namespace

// Unique id of the calling thread's current CUDA context (0 if unknown).
// Device addresses cached per device stay valid only within one context: a
// cudaDeviceReset ends the primary context, and the next one gets a new id.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

namespace {

// Looks up (once per device and context) the SM count, compute capability
// and the device address of the status word.
int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
  unsigned long long ctx = current_context_id();
  if (ctx == 0) {  // no context yet on this thread: the runtime creates it
    if (cudaFree(nullptr) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
    ctx = current_context_id();
  }
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_devices.find(dev);
  if (it != g_devices.end() && it->second.ctx != ctx) {
    // a new context on this device: addresses cached for the old one are
    // stale, and so are the old context's workspaces (freed with it)
    g_devices.erase(it);
    for (auto w = g_workspaces.begin(); w != g_workspaces.end();)
      w = std::get<0>(w->first) == dev ? g_workspaces.erase(w) : std::next(w);
    it = g_devices.end();
  }
  if (it == g_devices.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess)
      return FP8GEMM_ERR_LAUNCH;
    d.ok = d.cc_major == 10 && d.cc_minor == 3;
    d.ctx = ctx;
    if (d.ok && cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_device_status) !=
                    cudaSuccess)
      return FP8GEMM_ERR_LAUNCH;
    it = g_devices.emplace(dev, d).first;
  }
  *out = it->second;
  return it->second.ok ? FP8GEMM_OK : FP8GEMM_ERR_ARCH;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int finish(cudaError_t e, int nlaunch) {
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free launch error
    return FP8GEMM_ERR_LAUNCH;
  }
  g_launches += nlaunch;
  return FP8GEMM_OK;
}

// Library-owned device buffers, one per (device, stream, slot), zero-
// initialised.  Slot kWsSplitK: the split-K reduction of the small-M path (its
// counters must start at 0 and are left at 0).  Slot kWsQuantA: quantised
// activations of fp8gemm_dense_quant_a at large M -- a separate buffer, so
// those bytes never land on the counters.
// Slot kWsTable: the stream-K partials and counters of the problem-table GEMM.
// Slot kWsBatch: the tile counters of the batched dense GEMM.  Slot
// kWsContig: the tile counters and tile order of the contiguous form.
enum { kWsSplitK = 0, kWsQuantA = 1, kWsTable = 2, kWsBatch = 3, kWsContig = 4 };

int workspace_for(cudaStream_t s, size_t bytes, void** out, int slot = kWsSplitK) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
  DeviceInfo d;  // drops the workspaces of an ended context first
  if (int r = device_info(&d)) return r;
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, s, slot);
  auto it = g_workspaces.find(key);
  if (it != g_workspaces.end() && it->second.bytes >= bytes) {
    *out = it->second.ptr;
    return FP8GEMM_OK;
  }
  if (it != g_workspaces.end()) {  // grow: the old buffer may still be in use on s
    if (cudaStreamSynchronize(s) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
    cudaFree(it->second.ptr);
    g_workspaces.erase(it);
  }
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
  // zeroed on the stream that will use it: a plain cudaMemset runs on the
  // legacy default stream, which a non-blocking stream does not wait for
  if (cudaMemsetAsync(p, 0, bytes, s) != cudaSuccess) {
    cudaFree(p);
    return FP8GEMM_ERR_LAUNCH;
  }
  g_workspaces[key] = Workspace{p, bytes, d.ctx};
  *out = p;
  return FP8GEMM_OK;
}

constexpr int kSmallM = 64;  // dense calls with M <= this use the swap-AB stream-K kernel

// The persistent tensor-core GEMM (its launch count is 0 for an empty
// problem, else 1).
int run_gemm_tc(const LaunchCtx& c, const GemmArgs& a) {
  int launches = 0;
  const cudaError_t e = launch_gemm_tc(c, a, &launches);
  return finish(e, launches);
}

}  // namespace

bool make_tmap_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0 || cols == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};  // bytes between rows
  const cuuint32_t box[2] = {uint32_t(kBlockK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0 || cols == 0) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (cols * 2) % 16 != 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};  // bytes between rows
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fp8gemm

using namespace fp8gemm;

namespace {

// K granularity: a TMA row stride (K bytes of e4m3) must be a multiple of 16
// bytes.  K need not be a multiple of 128: the last K block is then partial
// and the copies fill its missing columns with zeros.
constexpr int kKAlign = 16;

// Shared shape rules: K a positive multiple of 16, sizes non-negative.
int check_common(int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return FP8GEMM_ERR_SHAPE;
  if (K == 0 || K % kKAlign != 0) return FP8GEMM_ERR_SHAPE;
  return FP8GEMM_OK;
}

int ctx_for(cudaStream_t stream, LaunchCtx* c) {
  DeviceInfo d;
  const int r = device_info(&d);
  if (r != FP8GEMM_OK) return r;
  c->stream = stream;
  c->num_sms = d.num_sms;
  c->status = d.status;
  return FP8GEMM_OK;
}

}  // namespace

namespace fp8gemm {
int make_launch_ctx(cudaStream_t stream, LaunchCtx* c) { return ctx_for(stream, c); }
unsigned long long wait_limit_ns() { return g_wait_ns.load(); }
void count_kernel_launches(int n) { g_launches += n; }
}  // namespace fp8gemm

extern "C" {

int fp8_quant_1x128_ex(const float* X, uint8_t* Q, float* sX, int M, int K, int fmt,
                       unsigned long long* sat_count, fp8gemm_stream_t stream) {
  if (M < 0 || K < 0 || K % kKAlign != 0) return FP8GEMM_ERR_SHAPE;
  if (fmt != FP8GEMM_FMT_E4M3 && fmt != FP8GEMM_FMT_E5M2) return FP8GEMM_ERR_FORMAT;
  if (M == 0 || K == 0) return FP8GEMM_OK;
  if (!X || !Q || !sX) return FP8GEMM_ERR_NULL;
  if (!aligned16(X) || !aligned16(Q) || !aligned16(sX)) return FP8GEMM_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(sat_count) % 8 != 0) return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  return finish(launch_quant_1x128(c, X, Q, sX, M, K, fmt, sat_count), 1);
}

int fp8_quant_1x128_fmt(const float* X, uint8_t* Q, float* sX, int M, int K, int fmt,
                        fp8gemm_stream_t stream) {
  return fp8_quant_1x128_ex(X, Q, sX, M, K, fmt, nullptr, stream);
}

int fp8_quant_1x128(const float* X, uint8_t* Q, float* sX, int M, int K,
                    fp8gemm_stream_t stream) {
  return fp8_quant_1x128_fmt(X, Q, sX, M, K, FP8GEMM_FMT_E4M3, stream);
}

int fp8_quant_128x128_ex(const float* W, uint8_t* Q, float* sW, int E, int N, int K, int fmt,
                         unsigned long long* sat_count, fp8gemm_stream_t stream) {
  if (E < 0 || N < 0 || K < 0 || K % kKAlign != 0) return FP8GEMM_ERR_SHAPE;
  if (fmt != FP8GEMM_FMT_E4M3 && fmt != FP8GEMM_FMT_E5M2) return FP8GEMM_ERR_FORMAT;
  if (E == 0 || N == 0 || K == 0) return FP8GEMM_OK;
  if ((long long)E * N * (long long)K > (1LL << 46)) return FP8GEMM_ERR_SHAPE;
  if (!W || !Q || !sW) return FP8GEMM_ERR_NULL;
  if (!aligned16(W) || !aligned16(Q) || !aligned16(sW)) return FP8GEMM_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(sat_count) % 8 != 0) return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  return finish(launch_quant_128x128(c, W, Q, sW, E, N, K, fmt, sat_count), 1);
}

int fp8_quant_128x128_fmt(const float* W, uint8_t* Q, float* sW, int E, int N, int K, int fmt,
                          fp8gemm_stream_t stream) {
  return fp8_quant_128x128_ex(W, Q, sW, E, N, K, fmt, nullptr, stream);
}

int fp8_quant_128x128(const float* W, uint8_t* Q, float* sW, int E, int N, int K,
                      fp8gemm_stream_t stream) {
  return fp8_quant_128x128_fmt(W, Q, sW, E, N, K, FP8GEMM_FMT_E4M3, stream);
}

int fp8gemm_dense_ex(const uint8_t* A, const float* sA, int a_fmt, const uint8_t* B,
                     const float* sB, int b_fmt, void* D, int M, int N, int K, unsigned flags,
                     fp8gemm_stream_t stream) {
  if (int r = check_common(M, N, K)) return r;
  if ((a_fmt != FP8GEMM_FMT_E4M3 && a_fmt != FP8GEMM_FMT_E5M2) ||
      (b_fmt != FP8GEMM_FMT_E4M3 && b_fmt != FP8GEMM_FMT_E5M2))
    return FP8GEMM_ERR_FORMAT;
  if (flags & ~unsigned(FP8GEMM_FLAG_B_READ_ONLY)) return FP8GEMM_ERR_FLAGS;
  if (M == 0 || N == 0) return FP8GEMM_OK;
  if (!A || !sA || !B || !sB || !D) return FP8GEMM_ERR_NULL;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D))
    return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  GemmArgs a{GemmMode::kDense, A, sA, B, sB, nullptr, static_cast<__nv_bfloat16*>(D),
             M, N, K, 1};
  a.a_fmt = a_fmt;
  a.b_fmt = b_fmt;
  a.b_read_only = (flags & FP8GEMM_FLAG_B_READ_ONLY) ? 1 : 0;
  if (M <= kSmallM) {
    if (!small_m_uses_workspace(c, a)) return finish(launch_gemm_small_m_any(c, a, nullptr, 0), 1);
    const size_t bytes = small_m_workspace_bytes(c.num_sms, N);
    void* ws = nullptr;
    if (int r = workspace_for(stream, bytes, &ws)) return r;
    return finish(launch_gemm_small_m_any(c, a, ws, bytes), 1);
  }
  return run_gemm_tc(c, a);
}

int fp8gemm_dense_fmt(const uint8_t* A, const float* sA, int a_fmt, const uint8_t* B,
                      const float* sB, int b_fmt, void* D, int M, int N, int K,
                      fp8gemm_stream_t stream) {
  return fp8gemm_dense_ex(A, sA, a_fmt, B, sB, b_fmt, D, M, N, K, 0u, stream);
}

int fp8gemm_dense(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, void* D,
                  int M, int N, int K, fp8gemm_stream_t stream) {
  return fp8gemm_dense_fmt(A, sA, FP8GEMM_FMT_E4M3, B, sB, FP8GEMM_FMT_E4M3, D, M, N, K,
                           stream);
}

int fp8gemm_dense_quant_a_ex(const float* X, uint8_t* Q, float* sA, const uint8_t* B,
                             const float* sB, void* D, int M, int N, int K, unsigned flags,
                             fp8gemm_stream_t stream) {
  if (int r = check_common(M, N, K)) return r;
  if (flags & ~unsigned(FP8GEMM_FLAG_B_READ_ONLY)) return FP8GEMM_ERR_FLAGS;
  if (M == 0 || N == 0) return FP8GEMM_OK;
  if (!X || !B || !sB || !D || (Q == nullptr) != (sA == nullptr)) return FP8GEMM_ERR_NULL;
  if (!aligned16(X) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      (Q && (!aligned16(Q) || !aligned16(sA))))
    return FP8GEMM_ERR_ALIGN;
  if ((long long)M * K > (1LL << 46)) return FP8GEMM_ERR_SHAPE;
  if (M <= kSmallM) {
    // decode sizes: one launch that quantises A on load, where the shape allows
    LaunchCtx c;
    if (int r = ctx_for(stream, &c)) return r;
    GemmArgs a{GemmMode::kDense, nullptr, nullptr, B, sB, nullptr, static_cast<__nv_bfloat16*>(D),
               M, N, K, 1};
    a.b_read_only = (flags & FP8GEMM_FLAG_B_READ_ONLY) ? 1 : 0;
    bool taken = false;
    const cudaError_t e = launch_gemm_small_m_quant(c, a, X, Q, sA, &taken);
    if (taken) return finish(e, 1);
  }
  if (!Q) {  // quantised A in the library's buffer: bytes, then (16-B aligned) scales
    const size_t qbytes = (size_t(M) * K + 15) / 16 * 16;
    void* ws = nullptr;
    if (int r = workspace_for(stream, qbytes + size_t(M) * ceil_div(K, kBlockK) * 4, &ws,
                              kWsQuantA))
      return r;
    Q = static_cast<uint8_t*>(ws);
    sA = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + qbytes);
  }
  // the quantiser, then the GEMM as its programmatic dependent: the GEMM's
  // prologue and weight prefetch overlap the quantiser
  if (int r = fp8_quant_1x128(X, Q, sA, M, K, stream)) return r;
  return fp8gemm_dense_ex(Q, sA, FP8GEMM_FMT_E4M3, B, sB, FP8GEMM_FMT_E4M3, D, M, N, K, flags,
                          stream);
}

int fp8gemm_dense_quant_a(const float* X, uint8_t* Q, float* sA, const uint8_t* B,
                          const float* sB, void* D, int M, int N, int K,
                          fp8gemm_stream_t stream) {
  return fp8gemm_dense_quant_a_ex(X, Q, sA, B, sB, D, M, N, K, 0u, stream);
}

int fp8gemm_grouped_table(const fp8gemm_problem* problems, int num_problems, int max_M,
                          fp8gemm_stream_t stream) {
  if (num_problems < 0 || max_M < 1) return FP8GEMM_ERR_SHAPE;
  if (num_problems == 0) return FP8GEMM_OK;
  if (!problems) return FP8GEMM_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(problems) & 7u) return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  const size_t bytes = table_workspace_bytes(c, max_M);
  void* ws = nullptr;
  if (int r = workspace_for(stream, bytes, &ws, kWsTable)) return r;
  return finish(launch_gemm_table(c, problems, num_problems, max_M, ws, bytes), 1);
}

static bool valid_fmt(int f) { return f == FP8GEMM_FMT_E4M3 || f == FP8GEMM_FMT_E5M2; }

int fp8gemm_dense_batch(const fp8gemm_problem* problems, int num_problems,
                        fp8gemm_stream_t stream) {
  if (num_problems < 0 || num_problems > FP8GEMM_MAX_DENSE_BATCH) return FP8GEMM_ERR_SHAPE;
  if (num_problems == 0) return FP8GEMM_OK;
  if (!problems) return FP8GEMM_ERR_NULL;
  bool any = false;
  for (int i = 0; i < num_problems; ++i) {  // every entry is checked before anything runs
    const fp8gemm_problem& q = problems[i];
    if (int r = check_common(q.M, q.N, q.K)) return r;
    if ((long long)q.M * q.K > (1LL << 46) || (long long)q.N * q.K > (1LL << 46))
      return FP8GEMM_ERR_SHAPE;
    if (!valid_fmt(q.formats & 0xff) || !valid_fmt(q.formats >> 8)) return FP8GEMM_ERR_FORMAT;
    if (q.M == 0 || q.N == 0) continue;
    if (!q.A || !q.sA || !q.B || !q.sB || !q.D) return FP8GEMM_ERR_NULL;
    if (!aligned16(q.A) || !aligned16(q.sA) || !aligned16(q.B) || !aligned16(q.sB) ||
        !aligned16(q.D))
      return FP8GEMM_ERR_ALIGN;
    any = true;
  }
  if (!any) return FP8GEMM_OK;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  void* ws = nullptr;
  if (int r = workspace_for(stream, 256, &ws, kWsBatch)) return r;
  int launches = 0;
  const cudaError_t e = launch_gemm_tc_batch(c, problems, num_problems,
                                             static_cast<unsigned int*>(ws), &launches);
  return finish(e, launches);
}

int fp8gemm_grouped_contiguous_fmt(const uint8_t* A, const float* sA, int a_fmt,
                                   const uint8_t* B, const float* sB, int b_fmt,
                                   const int32_t* m_indices, void* D, int M_pad, int N, int K,
                                   int E, fp8gemm_stream_t stream) {
  if (int r = check_common(M_pad, N, K)) return r;
  if (E < 0 || M_pad % kBlockM != 0) return FP8GEMM_ERR_SHAPE;
  if ((long long)E * N > 0x7fffffffLL) return FP8GEMM_ERR_SHAPE;
  if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt)) return FP8GEMM_ERR_FORMAT;
  if (M_pad == 0 || N == 0 || E == 0) return FP8GEMM_OK;
  if (!A || !sA || !B || !sB || !m_indices || !D) return FP8GEMM_ERR_NULL;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) ||
      !aligned16(m_indices) || !aligned16(D))
    return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  GemmArgs a{GemmMode::kContiguous, A, sA, B, sB, m_indices, static_cast<__nv_bfloat16*>(D),
             M_pad, N, K, E};
  a.a_fmt = a_fmt;
  a.b_fmt = b_fmt;
  // a wave or more of whole tiles: in expert-segment order, claimed
  // dynamically (the largest and the smallest experts' tiles side by side)
  if (const size_t bytes = contig_order_workspace_bytes(c, a)) {
    void* ws = nullptr;
    if (int r = workspace_for(stream, bytes, &ws, kWsContig)) return r;
    int launches = 0;
    const cudaError_t e = launch_gemm_tc_contiguous_ordered(c, a, ws, bytes, &launches);
    return finish(e, launches);
  }
  return run_gemm_tc(c, a);
}

int fp8gemm_grouped_contiguous(const uint8_t* A, const float* sA, const uint8_t* B,
                               const float* sB, const int32_t* m_indices, void* D, int M_pad,
                               int N, int K, int E, fp8gemm_stream_t stream) {
  return fp8gemm_grouped_contiguous_fmt(A, sA, FP8GEMM_FMT_E4M3, B, sB, FP8GEMM_FMT_E4M3,
                                        m_indices, D, M_pad, N, K, E, stream);
}

int fp8gemm_grouped_masked_fmt(const uint8_t* A, const float* sA, int a_fmt, const uint8_t* B,
                               const float* sB, int b_fmt, const int32_t* masked_m, void* D,
                               int E, int M_max, int N, int K, fp8gemm_stream_t stream) {
  if (int r = check_common(M_max, N, K)) return r;
  if (E < 0) return FP8GEMM_ERR_SHAPE;
  if ((long long)E * M_max > 0x7fffffffLL || (long long)E * N > 0x7fffffffLL)
    return FP8GEMM_ERR_SHAPE;
  if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt)) return FP8GEMM_ERR_FORMAT;
  if (M_max == 0 || N == 0 || E == 0) return FP8GEMM_OK;
  if (!A || !sA || !B || !sB || !masked_m || !D) return FP8GEMM_ERR_NULL;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) ||
      !aligned16(masked_m) || !aligned16(D))
    return FP8GEMM_ERR_ALIGN;
  LaunchCtx c;
  if (int r = ctx_for(stream, &c)) return r;
  GemmArgs a{GemmMode::kMasked, A, sA, B, sB, masked_m, static_cast<__nv_bfloat16*>(D),
             M_max, N, K, E};
  a.a_fmt = a_fmt;
  a.b_fmt = b_fmt;
  return run_gemm_tc(c, a);
}

int fp8gemm_grouped_masked(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                           const int32_t* masked_m, void* D, int E, int M_max, int N, int K,
                           fp8gemm_stream_t stream) {
  return fp8gemm_grouped_masked_fmt(A, sA, FP8GEMM_FMT_E4M3, B, sB, FP8GEMM_FMT_E4M3, masked_m,
                                    D, E, M_max, N, K, stream);
}

int fp8gemm_get_device_status(fp8gemm_stream_t stream, int* out) {
  if (!out) return FP8GEMM_ERR_NULL;
  DeviceInfo d;
  if (int r = device_info(&d)) return r;
  exchange_status<<<1, 1, 0, stream>>>(d.status);  // after every earlier kernel on stream
  if (cudaGetLastError() != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
  g_launches += 1;
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_taken, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FP8GEMM_ERR_LAUNCH;
  if (v == FP8GEMM_ERR_TIMEOUT) {
    // a launch that gave up may have left a split-K reduction half done, its
    // arrival counters not back at zero: drop every workspace of this device
    // (after the device is idle) so that the next calls start from zeroed ones
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      return FP8GEMM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto w = g_workspaces.begin(); w != g_workspaces.end();) {
      if (std::get<0>(w->first) != dev) {
        ++w;
        continue;
      }
      cudaFree(w->second.ptr);
      w = g_workspaces.erase(w);
    }
  }
  *out = v;
  return FP8GEMM_OK;
}

const char* fp8gemm_strerror(int code) {
  switch (code) {
    case FP8GEMM_OK: return "ok";
    case FP8GEMM_ERR_NULL: return "a required pointer is NULL";
    case FP8GEMM_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case FP8GEMM_ERR_SHAPE: return "unsupported shape (K % 16, M_pad % 128, sign or range)";
    case FP8GEMM_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103a)";
    case FP8GEMM_ERR_LAUNCH: return "CUDA launch or runtime call failed";
    case FP8GEMM_ERR_DEVICE_STATUS: return "device-side input error (expert index or row count)";
    case FP8GEMM_ERR_TIMEOUT: return "a pipeline wait exceeded its time limit";
    case FP8GEMM_ERR_SCRATCH_LIMIT:
      return "problem exceeds the fixed scratch of fp8gemm_dense_small_m_noalloc (M <= 64)";
    case FP8GEMM_ERR_FORMAT: return "unknown FP8 format (FP8GEMM_FMT_E4M3 or FP8GEMM_FMT_E5M2)";
    case FP8GEMM_ERR_FLAGS: return "unknown flag bits (FP8GEMM_FLAG_*)";
    default: return "unknown status";
  }
}

uint64_t fp8gemm_num_kernel_launches(void) { return g_launches.load(); }

int fp8gemm_release_workspaces(fp8gemm_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
  DeviceInfo d;  // forgets workspaces of an ended context (not freed twice)
  if (int r = device_info(&d)) return r;
  std::lock_guard<std::mutex> lk(g_mu);
  bool synced = false;
  int rc = FP8GEMM_OK;
  for (auto w = g_workspaces.begin(); w != g_workspaces.end();) {
    if (std::get<0>(w->first) != dev || std::get<1>(w->first) != stream) {
      ++w;
      continue;
    }
    if (!synced) {  // work already enqueued on the stream may still use it
      if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8GEMM_ERR_LAUNCH;
      synced = true;
    }
    if (cudaFree(w->second.ptr) != cudaSuccess) rc = FP8GEMM_ERR_LAUNCH;
    w = g_workspaces.erase(w);
  }
  return rc;
}

int fp8gemm_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns);
  return FP8GEMM_OK;
}

uint64_t fp8gemm_workspace_bytes(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  uint64_t total = 0;
  for (const auto& w : g_workspaces) total += w.second.bytes;
  return total;
}

}  // extern "C"
