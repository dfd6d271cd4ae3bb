// gemm_small_m.cu -- the dense FP8 block-scaled GEMM for decode-sized M
// (M <= 64), where the weights dominate the bytes moved.
//
// Same arithmetic as gemm_tc.cu (per-K-block tensor-core partial, promoted
// with sA[m, kb] * sB[n/128, kb] into FP32, BF16 out), laid out for small M:
//
// * Swap AB: the weight tile (128 rows of B) is the MMA's M operand and the
//   M <= 64 activation rows, padded to MP in {16, 32, 64}, are its N operand,
//   so the 128-lane MMA is filled by weights instead of by padding.  TMEM lane
//   = output column n, TMEM column = output row m.
// * Stream-K: the (N tile, K block) units are dealt out evenly over one CTA
//   per SM, so every SM streams the same number of weight bytes even when
//   N/128 is far below the SM count ("news.rkmt.cn/news/5092" sections 1.2
//   and 4.2: with M of 1-16, fixed tiles leave most SMs idle; size the work
//   to the SM count).  A CTA whose range ends inside a tile leaves its FP32
//   partial in a workspace slot; the last CTA to finish a tile (one
//   acquire-release atomic per CTA) sums every contributor's partial in CTA
//   order -- a fixed order, so results are deterministic -- writes BF16 and
//   resets the tile's counter for the next launch.
// * Cluster split-K: when the N tiles times a split factor C <= 8 fill most
//   SMs, the C CTAs of a thread-block cluster share one tile's K range
//   instead; each leaves its partial in its own shared memory and, after a
//   cluster barrier, sums a 1/C share of the tile's outputs over the C
//   partials (distributed shared memory, CTA-rank order) and writes it.  No
//   workspace and no atomics; the hardware co-schedules a cluster's CTAs.
// * Programmatic dependent launch: the prologue and an L2 prefetch of the
//   CTA's weight tiles run while the previous kernel in the stream finishes;
//   every load into shared memory, and every access to activations, scales,
//   the workspace and D, waits for it (griddepcontrol.wait).  Shared memory
//   and registers are sized so that two CTAs fit on one SM during that
//   overlap.
//
// CTA layout (192 threads): warps 0-3 promotion/epilogue (thread = TMEM lane
// = output column), warp 4 TMA producer, warp 5 MMA issuer.
#include <cstring>

#include "common.cuh"
#include "f8_convert.cuh"
#include "ptx.cuh"

namespace fp8gemm {
namespace {

constexpr int kCounterBytes = 256 * 1024;  // one int per N tile: N <= 8M columns
constexpr int kMaxMP = 64;
constexpr int kMaxCluster = 16;  // CTAs sharing one tile's K range

template <int MP_>
struct SmCfg {
  static constexpr int MP = MP_;
  // stages: as many as keep two CTAs within one SM's shared memory
  static constexpr int kStages = MP == 16 ? 6 : (MP == 32 ? 5 : 4);
  static constexpr int kThreads = 192;
  static constexpr int kTmaWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kWBytes = 128 * kBlockK;  // weight tile: 16 KB
  static constexpr int kXBytes = MP * kBlockK;   // activation tile
  // TMEM partial buffers: enough that the MMA never waits for promotion on
  // the few K blocks a CTA handles (a partial is only MP columns)
  static constexpr int kTmemBufs = MP == 64 ? 4 : 8;
  static constexpr int kTmemCols = kTmemBufs * MP;  // 128 or 256: two CTAs fit in 512
  static constexpr int kScaleKb = 16;  // K blocks of scales staged per batch
  static constexpr int kBarBytes = 512;
  static constexpr int kAuxBytes = kBarBytes + kScaleKb * (MP + 4) * 4;
  static constexpr size_t kSmemBytes =
      1024 + size_t(kStages) * (kWBytes + kXBytes) + kAuxBytes;
  static_assert(MP == 16 || MP == 32 || MP == 64, "MP");
  static_assert((2 * kStages + 2 * kTmemBufs + 4) * 8 + 16 <= kBarBytes, "barrier area");
  static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
};

struct StreamK {
  long long U;  // units = tiles * Kb
  int G, Kb;
  __device__ long long begin(int c) const { return (long long)c * U / G; }
  __device__ int cta_of(long long u) const { return int(((u + 1) * G - 1) / U); }
};

// Cluster split-K reduction of rows j0, j0 + 4, ... (< r1) of 4 adjacent
// columns col4 .. col4 + 3 (lane c4 of the 128-column partials at `part` in
// the shared memory of ranks 0..C-1), summed in rank order (= K order:
// deterministic) and written to D as BF16; kRows rows a round, all of a
// round's C x kRows 16-byte remote loads issued before any is used.
template <int kRows, int kMaxC>
__device__ __forceinline__ void cluster_reduce_rows4(const float* part, int C, int j0, int r1,
                                                     int col4, int c4, const GemmArgs& args) {
  const float4* src[kMaxC];
#pragma unroll
  for (int r = 0; r < kMaxC; ++r)
    src[r] = reinterpret_cast<const float4*>(map_shared_rank(part, uint32_t(r < C ? r : 0))) + c4;
  const bool vec_ok = args.N % 4 == 0 && col4 + 3 < args.N;
  for (int j = j0; j < r1; j += 4 * kRows) {
    float4 v[kRows][kMaxC];
#pragma unroll
    for (int q = 0; q < kRows; ++q)
#pragma unroll
      for (int r = 0; r < kMaxC; ++r)
        v[q][r] = (r < C && j + 4 * q < r1) ? src[r][(j + 4 * q) * 32]
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
      const int row = j + 4 * q;
      if (row >= r1) continue;
      float4 sum = v[q][0];
#pragma unroll
      for (int r = 1; r < kMaxC; ++r)
        if (r < C) {
          sum.x += v[q][r].x;
          sum.y += v[q][r].y;
          sum.z += v[q][r].z;
          sum.w += v[q][r].w;
        }
      __nv_bfloat16* d = args.D + size_t(row) * args.N + col4;
      const __nv_bfloat162 lo = __float22bfloat162_rn(make_float2(sum.x, sum.y));
      const __nv_bfloat162 hi = __float22bfloat162_rn(make_float2(sum.z, sum.w));
      if (vec_ok) {
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(d) = u;
      } else {
        if (col4 < args.N) d[0] = lo.x;
        if (col4 + 1 < args.N) d[1] = lo.y;
        if (col4 + 2 < args.N) d[2] = hi.x;
        if (col4 + 3 < args.N) d[3] = hi.y;
      }
    }
  }
}

__device__ __forceinline__ void drain_wait_sm(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}

// kQuant (cluster form only, every CTA's K range within the stages): the
// activations arrive as FP32 X (Xf, [M, K]) and the promotion warps quantise
// the CTA's K blocks into the operand stages themselves -- fp8_quant_1x128's
// arithmetic, bit for bit -- instead of the producer loading quantised ones;
// the first tile's cluster also writes Q and sA when Qout is given.
template <class Cfg, bool kClusterSplit, bool kQuant = false>
__global__ void __launch_bounds__(Cfg::kThreads, 2)
    gemm_small_m_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmX, const GemmArgs args,
                        float* ws_partials, int* ws_counters, int* status, int cluster,
                        const float* Xf, uint8_t* Qout, float* sAout) {
  static_assert(!kQuant || kClusterSplit, "quantise-on-load runs in the cluster form");
  constexpr int MP = Cfg::MP;
  constexpr int kStages = Cfg::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smW = smem;
  uint8_t* smX = smem + kStages * Cfg::kWBytes;
  uint8_t* aux = smX + kStages * Cfg::kXBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty_bar = full_bar + kStages;
  constexpr int NB = Cfg::kTmemBufs;
  uint64_t* tfull_bar = full_bar + 2 * kStages;
  uint64_t* tempty_bar = tfull_bar + NB;
  uint64_t* drain_bar = tempty_bar + NB;
  uint64_t* group_bar = drain_bar + 1;
  uint64_t* xq_bar = group_bar + 1;  // kQuant: the operand stages hold the quantised activations
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(group_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_holder + 2);
  // scales of the current batch of K blocks: sa_s[q][j] = sA[j, kb + q], sb_s[q]
  float* sa_s = reinterpret_cast<float*>(aux + Cfg::kBarBytes);
  float* sb_s = sa_s + Cfg::kScaleKb * MP;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int Kb = ceil_div(args.K, kBlockK);  // the last K block may be partial
  const int n_tiles = ceil_div(args.N, 128);
  const StreamK sk{(long long)n_tiles * Kb, int(gridDim.x), Kb};
  // units [u_begin, u_end): the stream-K range, or this CTA's part of its
  // cluster's tile
  const int crank = kClusterSplit ? int(cluster_ctarank()) : 0;
  const long long ctile = (long long)(blockIdx.x / cluster) * Kb;
  const long long u_begin =
      kClusterSplit ? ctile + (long long)crank * Kb / cluster : sk.begin(blockIdx.x);
  const long long u_end =
      kClusterSplit ? ctile + (long long)(crank + 1) * Kb / cluster : sk.begin(blockIdx.x + 1);
  const int n_units = int(u_end - u_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(drain_bar, 1);
    mbar_init(group_bar, 128);
    mbar_init(xq_bar, 4);  // one arrival per promotion warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == Cfg::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmW);
    if (!kQuant) tma_prefetch_desc(&tmX);  // (kQuant: tmX is not a valid map)
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // the next kernel in the stream may start its own prologue now
  griddep_launch_dependents();

  auto fail = [&]() {
    *abort_flag = 1;
    raise_status(status, FP8GEMM_ERR_TIMEOUT);
  };

  if (warp == Cfg::kTmaWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = l2_policy_evict_first();  // weights: read once
      const uint64_t pol_keep = l2_policy_evict_last();     // activations: read by all
      // Pull this CTA's weight tiles towards L2 while the previous kernel in
      // the stream may still be running (a prefetch cannot return stale data);
      // every load into shared memory waits for that kernel.
      // With the caller's promise that no kernel still running writes the
      // weights (args.b_read_only), the first kStages weight tiles go
      // straight into shared memory instead: their full barriers are armed
      // for weights and activations, the activation halves follow the wait.
      const int pre = args.b_read_only ? (n_units < kStages ? n_units : kStages) : 0;
      // bytes a stage's copies bring (kQuant: the weights only)
      constexpr uint32_t kStageTx = Cfg::kWBytes + (kQuant ? 0 : Cfg::kXBytes);
      for (int i = 0; i < n_units; ++i) {
        const long long u = u_begin + i;
        if (i < pre) {  // first use of each stage: nothing to wait for
          mbar_arrive_expect_tx(&full_bar[i], kStageTx);
          tma_load_2d_hint(smW + i * Cfg::kWBytes, &tmW, &full_bar[i], int(u % Kb) * kBlockK,
                           int(u / Kb) * 128, pol_stream);
        } else {
          tma_prefetch_l2_2d(&tmW, int(u % Kb) * kBlockK, int(u / Kb) * 128);
        }
      }
      griddep_wait();
      if (!kQuant)
        for (int i = 0; i < pre; ++i)
          tma_load_2d_hint(smX + i * Cfg::kXBytes, &tmX, &full_bar[i],
                           int((u_begin + i) % Kb) * kBlockK, 0, pol_keep);
      int i = pre;
      for (; i < n_units; ++i) {
        const long long u = u_begin + i;
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(&empty_bar[s], ph ^ 1, abort_flag, args.wait_ns)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], kStageTx);
        tma_load_2d_hint(smW + s * Cfg::kWBytes, &tmW, &full_bar[s], int(u % Kb) * kBlockK,
                         int(u / Kb) * 128, pol_stream);
        if (!kQuant)
          tma_load_2d_hint(smX + s * Cfg::kXBytes, &tmX, &full_bar[s], int(u % Kb) * kBlockK, 0,
                           pol_keep);
      }
      const int n = i < kStages ? i : kStages;  // let in-flight copies land
      for (int j = i - n; j < i; ++j) drain_wait_sm(&full_bar[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // swap-AB: the MMA's A operand is the weights (the GEMM's B), its B
      // operand the activations
      const uint32_t idesc = idesc_f8_f32(128, MP, uint32_t(args.b_fmt), uint32_t(args.a_fmt));
      const uint32_t w_base = smem_addr(smW);
      const uint32_t x_base = smem_addr(smX);
      int i = 0;
      for (; i < n_units; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        const int buf = i % NB;
        const uint32_t tph = (i / NB) & 1;
        if (!mbar_wait(&tempty_bar[buf], tph ^ 1, abort_flag, args.wait_ns) ||
            !mbar_wait(&full_bar[s], ph, abort_flag, args.wait_ns) ||
            (kQuant && i == 0 && !mbar_wait(xq_bar, 0, abort_flag, args.wait_ns))) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * MP;
#pragma unroll
        for (int k = 0; k < kBlockK / 32; ++k) {
          const uint64_t ad = smem_desc_sw128_kmajor(w_base + s * Cfg::kWBytes + k * 32);
          const uint64_t bd = smem_desc_sw128_kmajor(x_base + s * Cfg::kXBytes + k * 32);
          umma_e4m3(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&empty_bar[s]);
        umma_commit(&tfull_bar[buf]);
      }
      if (i > 0) {  // every issued MMA has finished before TMEM is released
        umma_commit(drain_bar);
        drain_wait_sm(drain_bar, 0);
      }
    }
  } else {
    // -------------------------------------------- promotion + epilogue
    const int t = threadIdx.x;  // TMEM lane = column within the N tile
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const int M = args.M;
    const int first_tile = int(u_begin / Kb);
    uint32_t gphase = 0;
    bool ok = true;
    // bounded barrier over the 128 promotion threads
    auto group_sync = [&]() -> bool {
      mbar_arrive(group_bar);
      const bool r = mbar_wait(group_bar, gphase, abort_flag, args.wait_ns);
      gphase ^= 1;
      return r;
    };
    griddep_wait();  // sA, the workspace and D belong to the stream's order
    if constexpr (kQuant) {
      // The CTA's units are K blocks kq0 .. kq0 + n_units - 1 of one tile,
      // unit i in stage i.  Each (unit, row) pair is one 1x128 block: an
      // 8-lane group takes it (16 FP32 values per lane), reduces amax,
      // s = amax / 448, and writes the bytes to the stage's activation slot
      // (row j, 128-byte swizzle: a lane's 16 bytes are one chunk) and s to
      // sa_s[i][j]; rows j >= M are zero.
      const int kq0 = int(u_begin % Kb);
      const int K = args.K;
      const bool publish = Qout != nullptr && u_begin < Kb;  // the first tile's cluster
      // rows M .. MP-1 of every unit's slot: zero bytes, zero scales
      const int zrows = n_units * (MP - M);
      for (int idx = warp * 32 + lane; idx < zrows * 8; idx += 128) {
        const int zr = idx / 8, i = zr / (MP - M), j = M + zr % (MP - M);
        *reinterpret_cast<uint4*>(smX + i * Cfg::kXBytes + j * 128 + (idx % 8) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
        if (idx % 8 == 0) sa_s[i * MP + j] = 0.f;
      }
      // The M real rows: pair p = (unit p / M, row p % M) is one 1x128 block,
      // taken by an 8-lane group (16 values per lane), four pairs per warp
      // and round; K % 16 == 0, so a lane's 16 values are all in or all out.
      const int g = lane >> 3, t8 = lane & 7;
      const int pairs = n_units * M;
      for (int p0 = warp * 4; p0 < pairs; p0 += 16) {
        const int p = p0 + g, i = p / M, j = p % M, kb = kq0 + i;
        const bool have = p < pairs;
        const bool in = have && t8 * 16 < K - kb * kBlockK;
        float4 v[4];
        const float4* src =
            reinterpret_cast<const float4*>(Xf + size_t(j) * K + size_t(kb) * kBlockK + t8 * 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = in ? __ldg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        float amax = fmaxf(fmaxf(absmax4(v[0]), absmax4(v[1])), fmaxf(absmax4(v[2]), absmax4(v[3])));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1)  // within the 8-lane group
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sq = __fdiv_rn(amax, f8_limit<false>());
        const bool nz = amax != 0.f;
        const float sd = nz ? sq : 1.f;  // no division by zero on the way to zero bytes
        uint4 q;
        q.x = nz ? quant4<false>(v[0], sd) : 0u;
        q.y = nz ? quant4<false>(v[1], sd) : 0u;
        q.z = nz ? quant4<false>(v[2], sd) : 0u;
        q.w = nz ? quant4<false>(v[3], sd) : 0u;
        if (have) {
          *reinterpret_cast<uint4*>(smX + i * Cfg::kXBytes + j * 128 + ((t8 ^ (j & 7)) << 4)) = q;
          if (t8 == 0) sa_s[i * MP + j] = sq;
          if (publish) {
            if (in)
              *reinterpret_cast<uint4*>(Qout + size_t(j) * K + size_t(kb) * kBlockK + t8 * 16) = q;
            if (t8 == 0) sAout[size_t(j) * Kb + kb] = sq;
          }
        }
      }
      fence_proxy_async_smem();  // the stores (generic proxy) before the MMAs read them
      __syncwarp();
      if (lane == 0) mbar_arrive(xq_bar);
    }
    int it = 0;
    for (long long u = u_begin; u < u_end && ok;) {
      const int tile = int(u / Kb);
      const int kb0 = int(u % Kb);
      const int kb1 = int(min((long long)Kb, kb0 + (u_end - u)));

      float acc[MP];
#pragma unroll
      for (int j = 0; j < MP; ++j) acc[j] = 0.f;

      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int q = (kb - kb0) % Cfg::kScaleKb;
        if (q == 0) {
          // stage the scales of the next batch of K blocks with independent
          // loads (one latency per batch, not one per K block)
          const int nkb = min(Cfg::kScaleKb, kb1 - kb);
          if (!group_sync()) { fail(); ok = false; break; }  // previous batch consumed
          if (!kQuant)  // (kQuant: the quantisation above wrote sa_s)
            for (int idx = t; idx < MP * nkb; idx += 128) {
              const int j = idx / nkb, qq = idx % nkb;
              sa_s[qq * MP + j] = j < M ? __ldg(args.sA + size_t(j) * Kb + kb + qq) : 0.f;
            }
          if (t < nkb) sb_s[t] = __ldg(args.sB + size_t(tile) * Kb + kb + t);
          if (!group_sync()) { fail(); ok = false; break; }
        }
        const int buf = it % NB;
        const uint32_t tph = (it / NB) & 1;
        if (!mbar_wait(&tfull_bar[buf], tph, abort_flag, args.wait_ns)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_base + buf * MP;
        const float sb = sb_s[q];
        const float* sa_row = sa_s + q * MP;
        if constexpr (MP == 16) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(taddr, r);
          tmem_ld_wait_tied16(r);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[buf]);
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(sa_row + j);
            acc[j] = fmaf(__uint_as_float(r[j]), a4.x * sb, acc[j]);
            acc[j + 1] = fmaf(__uint_as_float(r[j + 1]), a4.y * sb, acc[j + 1]);
            acc[j + 2] = fmaf(__uint_as_float(r[j + 2]), a4.z * sb, acc[j + 2]);
            acc[j + 3] = fmaf(__uint_as_float(r[j + 3]), a4.w * sb, acc[j + 3]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < MP / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c * 32, r);
            tmem_ld_wait_tied(r);
            if (c + 1 == MP / 32) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty_bar[buf]);
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 a4 = *reinterpret_cast<const float4*>(sa_row + c * 32 + j);
              const int o = c * 32 + j;
              acc[o] = fmaf(__uint_as_float(r[j]), a4.x * sb, acc[o]);
              acc[o + 1] = fmaf(__uint_as_float(r[j + 1]), a4.y * sb, acc[o + 1]);
              acc[o + 2] = fmaf(__uint_as_float(r[j + 2]), a4.z * sb, acc[o + 2]);
              acc[o + 3] = fmaf(__uint_as_float(r[j + 3]), a4.w * sb, acc[o + 3]);
            }
          }
        }
      }
      if (!ok) break;

      const int n = tile * 128 + t;
      const bool col_ok = n < args.N;
      bool write = true;
      if (kClusterSplit && !(kb0 == 0 && kb1 == Kb)) {
        // this CTA's partial stays in its own shared memory (the stage area
        // is idle: every load has been consumed); reduced across the cluster
        // below
        float* part = reinterpret_cast<float*>(smW);
#pragma unroll
        for (int j = 0; j < MP; ++j)
          if (j < M) part[j * 128 + t] = acc[j];
        write = false;
      } else if (!(kb0 == 0 && kb1 == Kb)) {
        // split tile: publish this CTA's partial; the last contributor reduces
        const int slot_idx = 2 * blockIdx.x + (tile == first_tile ? 0 : 1);
        float* mine = ws_partials + size_t(slot_idx) * MP * 128;
        if (M >= MP) {
#pragma unroll
          for (int j = 0; j < MP; ++j) mine[j * 128 + t] = acc[j];
        } else {  // only the M real rows are published
#pragma unroll
          for (int j = 0; j < MP; ++j)
            if (j < M) mine[j * 128 + t] = acc[j];
        }
        if (!group_sync()) { fail(); ok = false; break; }
        const int c_first = sk.cta_of((long long)tile * Kb);
        const int c_last = sk.cta_of((long long)(tile + 1) * Kb - 1);
        if (t == 0) {
          // release this CTA's partial (ordered before by the group barrier),
          // acquire the partials of the CTAs that arrived earlier
          const int prev = atomic_add_acq_rel_gpu(ws_counters + tile, 1);
          const int is_last = prev == c_last - c_first;
          if (is_last) ws_counters[tile] = 0;  // ready for the next launch
          *last_flag = is_last;
        }
        if (!group_sync()) { fail(); ok = false; break; }
        write = *last_flag != 0;
        if (!group_sync()) { fail(); ok = false; break; }  // last_flag is reused
        if (write) {
          // sum every contributor's partial in CTA order (fixed order:
          // deterministic); only the M real rows were published
#pragma unroll
          for (int j = 0; j < MP; ++j) acc[j] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const int cs = int(sk.begin(c) / Kb) == tile ? 2 * c : 2 * c + 1;
            const float* p = ws_partials + size_t(cs) * MP * 128;
            if (M >= MP) {
#pragma unroll
              for (int j = 0; j < MP; ++j) acc[j] += __ldcg(p + j * 128 + t);
            } else {
#pragma unroll
              for (int j = 0; j < MP; ++j)
                if (j < M) acc[j] += __ldcg(p + j * 128 + t);
            }
          }
        }
      }
      if (write && col_ok) {
#pragma unroll
        for (int j = 0; j < MP; ++j)
          if (j < M) args.D[size_t(j) * args.N + n] = __float2bfloat16_rn(acc[j]);
      }
      u += kb1 - kb0;
    }
  }

  if (kClusterSplit && cluster > 1) {
    // every CTA of the cluster has its partial in shared memory
    __syncwarp();
    cluster_sync();
    if (warp < 4) {
      // this CTA sums rows [r0, r1) of the tile over the partials of ranks
      // 0..C-1 in rank order (= K order: deterministic); a thread takes 4
      // adjacent columns (16-byte loads through distributed shared memory)
      const int C = cluster;
      const int M = args.M;
      const int r0 = crank * M / C, r1 = (crank + 1) * M / C;
      const int col4 = int(blockIdx.x) / C * 128 + (lane << 2);
      const float* part = reinterpret_cast<const float*>(smW);
      if (C <= 8)
        cluster_reduce_rows4<2, 8>(part, C, r0 + warp, r1, col4, lane, args);
      else
        cluster_reduce_rows4<1, kMaxCluster>(part, C, r0 + warp, r1, col4, lane, args);
    }
    __syncwarp();
    cluster_sync();  // the partners are done reading this CTA's partial
  }

  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// Sets the kernels' launch attributes once per device and context (they
// belong to the functions in one context; a cudaDeviceReset gives the device
// a new one).
template <class Cfg>
cudaError_t prepare_kernels(int dev) {
  static unsigned long long set_in[64] = {};  // context id, per device
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && set_in[dev & 63] == ctx) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_small_m_kernel<Cfg, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Cfg::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_small_m_kernel<Cfg, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_small_m_kernel<Cfg, true>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_small_m_kernel<Cfg, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_small_m_kernel<Cfg, true, true>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) set_in[dev & 63] = ctx;
  return e;
}

// Whether a cluster of C CTAs of the cluster kernel can be resident at all
// (sizes above 8 are not guaranteed); cached per device and C.
template <class Cfg>
bool cluster_fits(int dev, int C) {
  static signed char known[64][kMaxCluster + 1] = {};  // 0 unknown, 1 yes, -1 no
  signed char& k = known[dev & 63][C];
  if (k == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    const bool ok = prepare_kernels<Cfg>(dev) == cudaSuccess &&
                    cudaOccupancyMaxActiveClusters(&n, gemm_small_m_kernel<Cfg, true>, &cfg) ==
                        cudaSuccess &&
                    n > 0;
    if (!ok) cudaGetLastError();  // a refused query leaves no sticky error
    k = ok ? 1 : -1;
  }
  return k > 0;
}

// Split factor C for the cluster form, 0 for stream-K.  First choice: the
// largest portable C <= 8 that keeps tiles * C within two CTAs per SM --
// or, smaller, the largest such C that divides the K blocks evenly (the
// cluster waits for its slowest CTA: 16 K blocks over 4 CTAs beat 3-4 over 5,
// 6.39 -> 6.0 us at 1 x 7168 x 2048); otherwise (few tiles) the largest
// C <= 16 within one CTA per SM.  Either is taken only when tiles * C fills
// at least 70 % of the SMs; below that, and above two tiles per SM, stream-K
// balances better.
template <class Cfg>
int cluster_split(const LaunchCtx& c, int n_tiles, int Kb) {
  const long long fill = 7LL * c.num_sms;  // x10: 70 %
  int best = 0;
  for (int cl = 1; cl <= 8 && cl <= Kb; ++cl)
    if ((long long)n_tiles * cl <= 2LL * c.num_sms) best = cl;
  for (int cl = best; cl >= 2; --cl)
    if (Kb % cl == 0 && (long long)n_tiles * cl * 10 >= fill) return cl;
  if (best > 0 && (long long)n_tiles * best * 10 >= fill) return best;
  best = 0;
  for (int cl = 9; cl <= kMaxCluster && cl <= Kb; ++cl)
    if ((long long)n_tiles * cl <= c.num_sms) best = cl;
  if (best > 0 && (long long)n_tiles * best * 10 >= fill) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cluster_fits<Cfg>(dev, best)) return best;
  }
  return 0;
}

template <class Cfg>
cudaError_t run(const LaunchCtx& c, const GemmArgs& args, void* ws, size_t ws_bytes,
                bool allow_cluster) {
  GemmArgs a = args;
  a.wait_ns = wait_limit_ns();
  const int Kb = ceil_div(a.K, kBlockK);
  const int n_tiles = ceil_div(a.N, 128);
  const long long U = (long long)n_tiles * Kb;
  const int split = allow_cluster ? cluster_split<Cfg>(c, n_tiles, Kb) : 0;
  const int grid = split > 0 ? n_tiles * split : int(U < c.num_sms ? U : c.num_sms);
  if (grid == 0) return cudaSuccess;
  if (split == 0 && (size_t(n_tiles) * 4 > size_t(kCounterBytes) ||
                     ws_bytes < size_t(kCounterBytes) + size_t(2) * grid * Cfg::MP * 128 * 4))
    return cudaErrorInvalidValue;
  CUtensorMap tmW, tmX;
  if (!make_tmap_u8_sw128(&tmW, a.B, uint64_t(a.N), a.K, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&tmX, a.A, uint64_t(a.M), a.K, Cfg::MP)) return cudaErrorInvalidValue;
  int dev = 0;
  cudaGetDevice(&dev);
  if (cudaError_t e = prepare_kernels<Cfg>(dev)) return e;
  int* counters = split > 0 ? nullptr : reinterpret_cast<int*>(ws);
  float* partials =
      split > 0 ? nullptr : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  // launched as a programmatic dependent of the previous kernel in the stream
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = split > 0 ? split : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split > 0 ? 2 : 1;
  if (split > 0)
    return cudaLaunchKernelEx(&cfg, gemm_small_m_kernel<Cfg, true>, tmW, tmX, a, partials,
                              counters, c.status, split, (const float*)nullptr,
                              (uint8_t*)nullptr, (float*)nullptr);
  return cudaLaunchKernelEx(&cfg, gemm_small_m_kernel<Cfg, false>, tmW, tmX, a, partials,
                            counters, c.status, 1, (const float*)nullptr, (uint8_t*)nullptr,
                            (float*)nullptr);
}

// Quantise-on-load: the cluster form when every CTA's K range fits in the
// stages (one stage per K block, none reused), launched as a programmatic
// dependent like run(); *taken = false leaves the call to the caller.
template <class Cfg>
cudaError_t run_quant(const LaunchCtx& c, const GemmArgs& args, const float* X, uint8_t* Q,
                      float* sA, bool* taken) {
  *taken = false;
  GemmArgs a = args;
  a.wait_ns = wait_limit_ns();
  const int Kb = ceil_div(a.K, kBlockK);
  const int n_tiles = ceil_div(a.N, 128);
  const int split = cluster_split<Cfg>(c, n_tiles, Kb);
  // Each (K block, row) of a CTA's range is one 1x128 block for its four
  // promotion warps to quantise before the first MMA, on the critical path,
  // four blocks per warp and round: up to 16 (one round) that costs less than
  // a separate quantiser launch (1 x 7168 x 2048: 6.3 against 7.5 us); at 64
  // (16 rows, four rounds) it costs more (9.1-9.8 against 7.8 us).
  const int units = split < 1 ? 0 : ceil_div(Kb, split);
  if (split < 1 || units > Cfg::kStages || units * a.M > 16) return cudaSuccess;
  *taken = true;
  CUtensorMap tmW, tmX;
  if (!make_tmap_u8_sw128(&tmW, a.B, uint64_t(a.N), a.K, 128)) return cudaErrorInvalidValue;
  memset(&tmX, 0, sizeof(tmX));  // activations come from X, not through a tensor map
  int dev = 0;
  cudaGetDevice(&dev);
  if (cudaError_t e = prepare_kernels<Cfg>(dev)) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles * split);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = split;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_small_m_kernel<Cfg, true, true>, tmW, tmX, a,
                            (float*)nullptr, (int*)nullptr, c.status, split, X, Q, sA);
}

}  // namespace

cudaError_t launch_gemm_small_m_quant(const LaunchCtx& c, const GemmArgs& a, const float* X,
                                      uint8_t* Q, float* sA, bool* taken) {
  *taken = false;
  if (a.M < 1 || a.M > kMaxMP) return cudaSuccess;
  if (a.M <= 16) return run_quant<SmCfg<16>>(c, a, X, Q, sA, taken);
  if (a.M <= 32) return run_quant<SmCfg<32>>(c, a, X, Q, sA, taken);
  return run_quant<SmCfg<64>>(c, a, X, Q, sA, taken);
}

size_t small_m_workspace_bytes(int num_sms, int /*N*/) {
  return size_t(kCounterBytes) + size_t(2) * num_sms * kMaxMP * 128 * 4;
}

cudaError_t launch_gemm_small_m(const LaunchCtx& c, const GemmArgs& a, void* ws,
                                size_t ws_bytes) {
  if (a.M <= 16) return run<SmCfg<16>>(c, a, ws, ws_bytes, false);
  if (a.M <= 32) return run<SmCfg<32>>(c, a, ws, ws_bytes, false);
  return run<SmCfg<64>>(c, a, ws, ws_bytes, false);
}

bool small_m_uses_workspace(const LaunchCtx& c, const GemmArgs& a) {
  const int n_tiles = ceil_div(a.N, 128), Kb = ceil_div(a.K, kBlockK);
  if (a.M <= 16) return cluster_split<SmCfg<16>>(c, n_tiles, Kb) == 0;
  if (a.M <= 32) return cluster_split<SmCfg<32>>(c, n_tiles, Kb) == 0;
  return cluster_split<SmCfg<64>>(c, n_tiles, Kb) == 0;
}

cudaError_t launch_gemm_small_m_any(const LaunchCtx& c, const GemmArgs& a, void* ws,
                                    size_t ws_bytes) {
  if (a.M <= 16) return run<SmCfg<16>>(c, a, ws, ws_bytes, true);
  if (a.M <= 32) return run<SmCfg<32>>(c, a, ws, ws_bytes, true);
  return run<SmCfg<64>>(c, a, ws, ws_bytes, true);
}

}  // namespace fp8gemm
