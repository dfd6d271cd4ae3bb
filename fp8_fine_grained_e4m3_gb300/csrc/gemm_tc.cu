// gemm_tc.cu -- persistent, warp-specialised FP8 block-scaled GEMM on the
// 5th-generation tensor cores (sm_103a), for the dense and the two MoE
// grouped forms.
//
// What it computes (see include/fp8gemm.h): every 128-wide K block is
// contracted on the tensor cores into a fresh FP32 partial in TMEM, then
// "promoted" on the CUDA cores -- multiplied by sA[m, kb] * sB[n/128, kb] and
// added into an FP32 register accumulator ("lpnh.cn/news/2822121" section 2.3:
// the scale product changes per K block, so it cannot wait for the end of the
// K loop; "blog.hotdry.top: DeepGEMM FP8 GEMM fine-grained scaling kernels",
// section "two-level accumulation": first level on the tensor cores, second
// level promoted to FP32 on the CUDA cores).  The result is rounded to BF16
// once, in the epilogue.
//
// CTA layout (384 threads, one CTA per SM, persistent over tiles):
//   warps 0-7  promotion + epilogue: two warpgroups; warpgroup g owns columns
//              [g*BN/2, (g+1)*BN/2) of the tile, thread = tile row (TMEM lane),
//              reading each K block's partial in 64-column TMEM loads
//   warp 8     TMA producer: A tile 128x128 B and B tile BNx128 B per K block
//              into a kStages-deep shared-memory ring (128-byte swizzle)
//   warp 9     MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4 (K = 32)
//              per K block into one of two TMEM partial buffers
//   warps 10-11 idle: they complete the third warpgroup, whose register
//              budget is lowered (setmaxnreg) so the promotion warpgroups can
//              hold a 128-column FP32 accumulator per thread
// Synchronisation is by mbarriers only: full/empty per ring stage, and
// tmem_full/tmem_empty per TMEM buffer, so the tensor cores work on K block
// kb+1 while the promotion warps drain K block kb.  ("lpnh.cn/news/2822121"
// sections 3.1-3.3 and 4.1 describe the Hopper form of this pipeline: TMA
// loads the next block while the matrix instruction consumes the current
// one, with mbarriers between them.)
//
// Split tiles: when every tile fits in one wave (fewer tiles than SMs, as for
// a few hundred rows), most SMs would idle.  A second instance of the kernel
// (kSplit) then gives each tile a cluster of `split` CTAs, CTA r contracting
// the r-th share of the K blocks.  Each CTA stages its FP32 partial in its
// own shared memory (the idle operand ring); after a cluster barrier CTA r
// sums row band r of the tile over the cluster's CTAs, in rank order, through
// distributed shared memory and writes it to D ("news.rkmt.cn/news/5092"
// section 3.2: size the work to the SM count).  Splitting only the last wave
// of a longer run was slower: that wave's parts start cold behind the other
// waves.
//
// Tile order: grouped rasterisation (16 M blocks share each sweep over N) so
// concurrently running CTAs reuse A and B tiles through L2 ("news.rkmt.cn/
// news/5092" section 3.2: size the work to the SM count).  The masked form
// enumerates only tiles that hold valid rows, so no CTA idles on an empty
// expert ("lpnh.cn/news/2822121" section 5.2: skip empty blocks).
//
// Dynamic tile claims: two more instances hand tiles out from a counter
// instead of by CTA index -- a batched launch of independent dense problems
// (kP > 0, fp8gemm_dense_batch) and the contiguous form in expert-segment
// order (kP < 0, after contig_order_kernel) -- so that CTAs which finish
// early take more tiles ("bhfrc.com/news/60211" sections 4.2-4.3: one launch
// over a list of problems).
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8gemm {
namespace {

constexpr int kGroupM = 16;  // M blocks per rasterisation group

template <int BN_, int kStages_>
struct TcCfg {
  static constexpr int BN = BN_;
  static constexpr int kStages = kStages_;
  static constexpr int kPromoWarps = 8;
  static constexpr int kTmaWarp = 8;
  static constexpr int kMmaWarp = 9;
  static constexpr int kThreads = 384;  // 3 warpgroups; warps 10-11 only donate registers
  // Launch cap is 65536 / 384 -> 168 registers.  The producer warpgroup drops
  // to kLowRegs and the two promotion warpgroups rise to kHighRegs (BN = 256:
  // a 128-column accumulator plus a 64-column TMEM chunk per thread):
  // 128*72 + 256*216 = 128*104 + 256*200 = 64512 = 384*168; per sub-partition
  // (one producer and two promotion warps share its 512 registers per lane)
  // low + 2*high <= 512.
  static constexpr uint32_t kLowRegs = BN == 256 ? 72 : 104;
  static constexpr uint32_t kHighRegs = BN == 256 ? 216 : 200;
  static_assert(128 * kLowRegs + 256 * kHighRegs <= 384 * 168, "register split");
  static_assert(kLowRegs + 2 * kHighRegs <= 512, "register split per sub-partition");
  static constexpr int kABytes = kBlockM * kBlockK;  // 16 KB
  static constexpr int kBBytes = BN * kBlockK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kColsPerWG = BN / 2;
  static constexpr int kTmemBufs = 2;       // TMEM partial buffers
  static constexpr int kTmemCols = kTmemBufs * BN;
  static constexpr int kBarBytes = 512;
  // Epilogue staging: two 32-row x 32-column BF16 boxes (2 KB each) per
  // promotion warp, written alternately while TMA stores drain the other.
  static constexpr int kEpiBoxBytes = 32 * 32 * 2;
  static constexpr int kEpiBytes = kPromoWarps * 2 * kEpiBoxBytes;
  static constexpr size_t kSmemBytes =
      1024 + size_t(kStages) * kStageBytes + kEpiBytes + kBarBytes;
  static_assert(kSmemBytes <= 232448, "227 KB of shared memory per CTA");
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM columns must be a power of 2");
  // full/empty per stage, TMEM full/empty, drain, TMEM address + abort flag,
  // and (batched launches) the tile ring: 2 + 2 barriers and 2 slots of 32 B
  static_assert((2 * kStages + 2 * kTmemBufs + 6) * 8 + 64 <= kBarBytes, "barrier area");
};

struct Tile {
  int row0;        // first row in A's (and D's) 2-D row space
  int valid_rows;  // rows of this tile that are real outputs
  int n0;          // first output column
  int b_row0;      // first row in B's 2-D row space (expert * N + n0)
  int e;           // expert (0 for dense)
  int p;           // problem of a batched launch (0 otherwise)
  int kb;          // K blocks of that problem (batched launch only)
  int sb0;         // first sB element of the tile's expert (contiguous order only)
};

// A batched launch (fp8gemm_dense_batch): independent dense problems, each
// with its own tensor maps and sizes, whose tiles form one sequence -- the
// problems one after another, each in the grouped rasterisation order of the
// dense form.  The persistent CTAs take their first tile by index and every
// later one from a counter (the next unclaimed tile when a CTA's producer
// has issued its current tile's loads), so CTAs that finish early take more
// tiles: with the problems ordered by falling K (among equal K, the largest
// and the smallest alternating: launch_gemm_tc_batch), the short tiles of the
// last problems fill the partial last round of the long ones.  The producer hands
// each tile index to the MMA and promotion warps through a two-slot ring in
// shared memory; each role maps the index to its tile itself (handing over
// the mapped fields instead cost the promotion warps a register spill and
// 7 % on 4096x7168x16384).
constexpr int kMaxBatch = FP8GEMM_MAX_DENSE_BATCH;
constexpr int kSmallBatch = 4;  // batches of up to 4 take an instance with 4 slots of parameters

struct BatchProblem {
  const float* sA;
  const float* sB;
  __nv_bfloat16* D;
  int M, N, Kb;
  int num_m, num_n;
  int tile0;  // its first tile in the launch's sequence
  int fmts;   // a_fmt | b_fmt << 8
  int d_tma;  // the D map is valid
};

template <int P>
struct BatchParams {
  CUtensorMap a[P], b[P], d[P];
  BatchProblem prob[P];
  int count;              // problems in use (the rest are never read)
  int total;              // tiles of all problems
  unsigned int* counter;  // [0] tiles claimed past the first round, [1] CTAs done
};
template <>
struct BatchParams<0> {};  // the single-problem instances
// The contiguous form in expert-segment order (kP = -1): its tiles in the
// order contig_order_kernel wrote, claimed like a batched launch's.
template <>
struct BatchParams<-1> {
  unsigned int* counter;  // [0] claims past the first round, [1] CTAs done, [2] tiles, [3] K blocks
  const int4* order;      // tile t: first row, first column, expert, expert's first sB element
};

// Tiles of a launch that claims them dynamically (read after the dependency
// wait: for the contiguous order, the kernel before this one wrote it).
template <int P>
__device__ __forceinline__ int dyn_total(const BatchParams<P>& bp) {
  if constexpr (P > 0) {
    return bp.total;
  } else if constexpr (P < 0) {
    return int(*reinterpret_cast<volatile const unsigned int*>(bp.counter + 2));
  } else {
    return 0;
  }
}

// Tile t of the contiguous form in segment order (t < total).
__device__ __forceinline__ void ordered_tile(const BatchParams<-1>& bp, const GemmArgs& a, int t,
                                             Tile& tile) {
  const int4 o = __ldg(bp.order + t);
  tile.row0 = o.x;
  tile.n0 = o.y;
  tile.e = o.z;
  tile.b_row0 = o.z * a.N + o.y;
  tile.valid_rows = kBlockM;
  tile.p = 0;
  tile.kb = 0;
  tile.sb0 = o.w;
}

// Tile t of a batched launch (t < total).
template <int P>
__device__ __forceinline__ void batch_tile(const BatchParams<P>& bp, int t, int BN, Tile& tile) {
  int p = 0;
#pragma unroll
  for (int q = 1; q < P; ++q)
    if (q < bp.count && t >= bp.prob[q].tile0) p = q;
  const BatchProblem& pr = bp.prob[p];
  t -= pr.tile0;
  const int per_group = kGroupM * pr.num_n;
  const int g = t / per_group;
  const int first_m = g * kGroupM;
  const int gs = min(kGroupM, pr.num_m - first_m);
  const int r = t - g * per_group;
  tile.row0 = (first_m + r % gs) * kBlockM;
  tile.n0 = (r / gs) * BN;
  tile.b_row0 = tile.n0;
  tile.e = 0;
  tile.valid_rows = min(kBlockM, pr.M - tile.row0);
  tile.p = p;
  tile.kb = pr.Kb;
}

// Walks the same tile sequence in every role of every CTA.
struct Scheduler {
  const GemmArgs& a;  // the kernel parameter itself (param space), not a copy
  int num_m, num_n, Kb, total;
  int* status;

  __device__ Scheduler(const GemmArgs& args, int BN, int* st) : a(args) { init(BN, st); }

  __device__ int masked_rows(int e) const {
    int m = __ldg(a.group_info + e);
    if (m < 0 || m > a.M) {
      raise_status(status, FP8GEMM_ERR_DEVICE_STATUS);
      m = m < 0 ? 0 : a.M;
    }
    return m;
  }

  __device__ void init(int BN, int* st) {
    status = st;
    Kb = ceil_div(a.K, kBlockK);  // the last K block may be partial (TMA fills zeros)
    num_n = ceil_div(a.N, BN);
    if (a.mode == GemmMode::kMasked) {
      num_m = ceil_div(a.M, kBlockM);
      int t = 0;
      for (int e = 0; e < a.E; ++e) t += ceil_div(masked_rows(e), kBlockM) * num_n;
      total = t;
    } else {
      num_m = ceil_div(a.M, kBlockM);
      total = num_m * num_n;
    }
  }

  // Returns false when the tile holds no work (contiguous padding block or a
  // bad expert index).
  __device__ bool get(int t, int BN, Tile& tile) const {
    if (a.mode == GemmMode::kMasked) {
      int e = 0;
      int mb_e = 0;
      for (; e < a.E; ++e) {
        mb_e = ceil_div(masked_rows(e), kBlockM);
        const int cnt = mb_e * num_n;
        if (t < cnt) break;
        t -= cnt;
      }
      const int mb = t % mb_e;
      const int nb = t / mb_e;
      tile.e = e;
      tile.row0 = e * a.M + mb * kBlockM;
      tile.valid_rows = min(kBlockM, masked_rows(e) - mb * kBlockM);
      tile.n0 = nb * BN;
      tile.b_row0 = e * a.N + tile.n0;
      return true;
    }
    const int per_group = kGroupM * num_n;
    const int g = t / per_group;
    const int first_m = g * kGroupM;
    const int gs = min(kGroupM, num_m - first_m);
    const int r = t - g * per_group;
    const int mb = first_m + r % gs;
    const int nb = r / gs;
    tile.row0 = mb * kBlockM;
    tile.n0 = nb * BN;
    if (a.mode == GemmMode::kContiguous) {
      const int e = __ldg(a.group_info + tile.row0);
      if (e < 0) return false;
      if (e >= a.E) {
        raise_status(status, FP8GEMM_ERR_DEVICE_STATUS);
        return false;
      }
      tile.e = e;
      tile.valid_rows = kBlockM;
      tile.b_row0 = e * a.N + tile.n0;
      return true;
    }
    tile.e = 0;
    tile.valid_rows = min(kBlockM, a.M - tile.row0);
    tile.b_row0 = tile.n0;
    return true;
  }
};

// Split tiles: a CTA's FP32 partial of its tile, staged row-major in its own
// shared memory (the operand ring, idle once its last K block is contracted).
// Rows are padded by 4 floats: the 8 lanes of each quarter-warp store a float4
// of 8 consecutive rows into 8 distinct bank groups.
template <class Cfg>
struct Stage {
  static constexpr int kPitch = Cfg::BN + 4;  // floats per staged row
  static constexpr size_t kBytes = size_t(kBlockM) * kPitch * 4;
  static_assert(kBytes <= size_t(Cfg::kStages) * Cfg::kStageBytes, "staging fits the ring");
};

// Bounded wait on an mbarrier whose phases may already be complete, with no
// abort check: used only to let in-flight async copies land before exit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}

// kSplit = false: whole tiles, persistent over the CTAs.  kSplit = true (all
// tiles fit in one wave): cluster c of args.split CTAs computes tile c, CTA
// rank r the r-th share of its K blocks.  kP > 0: a batched launch of up to
// kP dense problems (whole tiles; maps, sizes and pointers from `bp`, the
// first three parameters and args' problem fields unused).
template <class Cfg, bool kSplit, int kP = 0>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const GemmArgs args, int* status,
                   const __grid_constant__ BatchParams<kP> bp) {
  constexpr int BN = Cfg::BN;
  constexpr int kStages = Cfg::kStages;
  constexpr bool kBatch = kP > 0;    // independent problems (fp8gemm_dense_batch)
  constexpr bool kOrdered = kP < 0;  // the contiguous form in segment order
  constexpr bool kDyn = kP != 0;     // tiles claimed through the counter and the ring
  static_assert(!(kDyn && kSplit), "dynamic claims take whole tiles");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages * Cfg::kABytes;
  uint8_t* epi = smem + kStages * Cfg::kStageBytes;  // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + Cfg::kEpiBytes);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + kStages;
  uint64_t* tfull_bar = bars + 2 * kStages;
  constexpr int NB = Cfg::kTmemBufs;
  uint64_t* tempty_bar = bars + 2 * kStages + NB;
  uint64_t* drain_bar = bars + 2 * kStages + 2 * NB;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 2 * NB + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // batched launches: the tile ring (slot: a tile index, -1 ends the
  // sequence; 32-byte slots)
  uint64_t* ring_full = bars + 2 * kStages + 2 * NB + 2;
  uint64_t* ring_empty = ring_full + 2;
  int* ring = reinterpret_cast<int*>(ring_full + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], Cfg::kPromoWarps);
    }
    mbar_init(drain_bar, 1);
    if constexpr (kDyn) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ring_full[i], 1);                       // the producer
        mbar_init(&ring_empty[i], 1 + Cfg::kPromoWarps);  // MMA thread + promotion warps
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == Cfg::kTmaWarp && lane == 0) {
    if constexpr (kBatch) {
      for (int q = 0; q < bp.count; ++q) {
        tma_prefetch_desc(&bp.a[q]);
        tma_prefetch_desc(&bp.b[q]);
        if (bp.prob[q].d_tma) tma_prefetch_desc(&bp.d[q]);
      }
    } else {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (args.d_tma) tma_prefetch_desc(&tmD);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_holder;
  // launched as a programmatic dependent: nothing below may read before the
  // stream's earlier work is complete (the prologue above, and the launch
  // itself, overlapped it); the next kernel may launch now -- it waits for
  // this one the same way (one wave: it cannot take an SM this grid needs)
  griddep_wait();
  griddep_launch_dependents();
  const Scheduler sched(args, BN, status);
  const int Kb = sched.Kb;
  // This CTA's tiles, each over K blocks [kb0, kb1): blockIdx.x, + gridDim.x,
  // ... below sched.total; or (kSplit) tile t_begin if t_begin < t_end.  The
  // whole-tile loops read the special registers directly: copies of them kept
  // live through the roles cost registers the promotion warps do not have.
  int t_begin = 0, t_end = 0, kb0 = 0, kb1 = Kb, part = 0;
  if constexpr (kSplit) {
    const int tile_idx = blockIdx.x / args.split;  // clusters span consecutive CTAs
    part = int(cluster_ctarank());
    t_begin = tile_idx;
    t_end = tile_idx < sched.total ? tile_idx + 1 : tile_idx;
    kb0 = part * Kb / args.split;
    kb1 = (part + 1) * Kb / args.split;
  }
  auto first_tile = [&](int tb) { return kSplit ? tb : int(blockIdx.x); };
  auto end_tile = [&](int te) { return kSplit ? te : sched.total; };
  auto tile_step = [&]() { return kSplit ? 1 : int(gridDim.x); };
  auto fail = [&]() {
    *abort_flag = 1;
    raise_status(status, FP8GEMM_ERR_TIMEOUT);
  };
  // Batched launches: the next tile index from the ring (-1 at the end of
  // the sequence or when the wait gave up).  A promotion warp calls it with
  // all lanes (whole_warp: they agree on the outcome, and every lane has read
  // the slot before it is released); the MMA thread alone.
  uint32_t ring_taken = 0;
  auto ring_index = [&](bool whole_warp) -> int {
    const int slot = int(ring_taken & 1);
    bool got = mbar_wait(&ring_full[slot], (ring_taken >> 1) & 1, abort_flag, args.wait_ns);
    if (whole_warp) got = __all_sync(0xffffffffu, got);
    if (!got) {
      fail();
      return -1;
    }
    const int t = ring[slot * 8];
    if (whole_warp) __syncwarp();
    if (lane == 0) mbar_arrive(&ring_empty[slot]);
    ++ring_taken;
    return t;
  };

  // Register budgets change at the top of each role (setmaxnreg, per
  // warpgroup): the producer warpgroup gives registers to the promotion ones.
  if (warp == Cfg::kTmaWarp) {
    // ------------------------------------------------------ TMA producer
    regs_decrease<Cfg::kLowRegs>();
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      if constexpr (kDyn) {
        // first tile by index, then each from the counter once the current
        // tile's loads are issued; every tile is published on the ring, then
        // the end marker
        uint32_t published = 0;
        const int total = dyn_total(bp);
        int t = int(blockIdx.x);
        while (ok) {
          Tile tile;
          const bool have = t < total;
          if (have) {
            if constexpr (kBatch) {
              batch_tile(bp, t, BN, tile);
            } else {
              ordered_tile(bp, args, t, tile);
            }
          }
          const int slot = int(published & 1);
          if (!mbar_wait(&ring_empty[slot], ((published >> 1) & 1) ^ 1, abort_flag,
                         args.wait_ns)) {
            fail();
            break;
          }
          ring[slot * 8] = have ? t : -1;
          mbar_arrive(&ring_full[slot]);
          ++published;
          if (!have) break;
          const CUtensorMap* mA = &tmA;
          const CUtensorMap* mB = &tmB;
          int kb_end = kb1;
          if constexpr (kBatch) {
            mA = &bp.a[tile.p];
            mB = &bp.b[tile.p];
            kb_end = tile.kb;
          }
          for (int kb = 0; kb < kb_end; ++kb, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1;
            if (!mbar_wait(&empty_bar[s], ph ^ 1, abort_flag, args.wait_ns)) {
              fail();
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_bar[s], Cfg::kStageBytes);
            tma_load_2d(smA + s * Cfg::kABytes, mA, &full_bar[s], kb * kBlockK, tile.row0);
            tma_load_2d(smB + s * Cfg::kBBytes, mB, &full_bar[s], kb * kBlockK, tile.b_row0);
          }
          if (ok) t = int(gridDim.x) + int(atomicAdd(bp.counter, 1u));
        }
      }
      for (int t = first_tile(t_begin); !kDyn && t < end_tile(t_end) && ok; t += tile_step()) {
        Tile tile;
        if (!sched.get(t, BN, tile)) continue;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&empty_bar[s], ph ^ 1, abort_flag, args.wait_ns)) {
            fail();
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], Cfg::kStageBytes);
          tma_load_2d(smA + s * Cfg::kABytes, &tmA, &full_bar[s], kb * kBlockK, tile.row0);
          tma_load_2d(smB + s * Cfg::kBBytes, &tmB, &full_bar[s], kb * kBlockK, tile.b_row0);
        }
      }
      // let the last copies into each stage land before the CTA can exit
      const uint32_t n = it < uint32_t(kStages) ? it : uint32_t(kStages);
      for (uint32_t i = it - n; i < it; ++i) drain_wait(&full_bar[i % kStages], (i / kStages) & 1);
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    regs_decrease<Cfg::kLowRegs>();
    if (lane == 0) {
      const uint32_t idesc =
          idesc_f8_f32(kBlockM, BN, uint32_t(args.a_fmt), uint32_t(args.b_fmt));
      const uint32_t a_base = smem_addr(smA);
      const uint32_t b_base = smem_addr(smB);
      uint32_t it = 0;
      bool ok = true;
      for (int t = kDyn ? ring_index(false) : first_tile(t_begin);
           (kDyn ? t >= 0 : t < end_tile(t_end)) && ok;
           t = kDyn ? ring_index(false) : t + tile_step()) {
        Tile tile;
        uint32_t idesc_t = idesc;
        int kb_end = kb1;
        if constexpr (kBatch) {
          batch_tile(bp, t, BN, tile);
          const int f = bp.prob[tile.p].fmts;
          idesc_t = idesc_f8_f32(kBlockM, BN, uint32_t(f & 0xff), uint32_t(f >> 8));
          kb_end = tile.kb;
        } else if constexpr (kOrdered) {
          ordered_tile(bp, args, t, tile);
        } else if (!sched.get(t, BN, tile)) {
          continue;
        }
        for (int kb = kb0; kb < kb_end; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          const int buf = it % NB;
          const uint32_t tph = (it / NB) & 1;
          if (!mbar_wait(&tempty_bar[buf], tph ^ 1, abort_flag, args.wait_ns) ||
              !mbar_wait(&full_bar[s], ph, abort_flag, args.wait_ns)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
          for (int k = 0; k < kBlockK / 32; ++k) {
            const uint64_t ad = smem_desc_sw128_kmajor(a_base + s * Cfg::kABytes + k * 32);
            const uint64_t bd = smem_desc_sw128_kmajor(b_base + s * Cfg::kBBytes + k * 32);
            umma_e4m3(d_tmem, ad, bd, idesc_t, k > 0 ? 1u : 0u);
          }
          umma_commit(&empty_bar[s]);     // stage free once these MMAs finish
          umma_commit(&tfull_bar[buf]);   // partial ready for promotion
        }
      }
      if (it > 0) {  // every issued MMA has finished before TMEM is released
        umma_commit(drain_bar);
        drain_wait(drain_bar, 0);
      }
    }
  } else if (warp < Cfg::kPromoWarps) {
    // ------------------------------------------ promotion + epilogue
    regs_increase<Cfg::kHighRegs>();
    const int wg = warp / 4;                 // column half
    const int row = (warp % 4) * 32 + lane;  // TMEM lane = tile row
    const uint32_t lane_base = uint32_t((warp % 4) * 32) << 16;
    const int Nb = ceil_div(args.N, kBlockK);
    uint32_t it = 0;
    uint32_t n_stores = 0;  // TMA stores this warp has issued (alternates the boxes)
    bool ok = true;
    for (int t = kDyn ? ring_index(true) : first_tile(t_begin);
         (kDyn ? t >= 0 : t < end_tile(t_end)) && ok;
         t = kDyn ? ring_index(true) : t + tile_step()) {
      Tile tile;
      if constexpr (kBatch) {
        batch_tile(bp, t, BN, tile);
      } else if constexpr (kOrdered) {
        ordered_tile(bp, args, t, tile);
      } else if (!sched.get(t, BN, tile)) {
        continue;
      }
      const bool row_ok = row < tile.valid_rows;
      const int col0 = tile.n0 + wg * Cfg::kColsPerWG;  // first column of this warpgroup
      const float* sa_ptr;
      const float* sb_ptr;
      bool cols_ok;
      int kb_end = kb1;
      if constexpr (kBatch) {
        const BatchProblem& pr = bp.prob[tile.p];
        cols_ok = col0 < pr.N;
        sa_ptr = pr.sA + size_t(tile.row0 + row) * tile.kb;
        sb_ptr = pr.sB + size_t(col0 / kBlockK) * tile.kb;
        kb_end = tile.kb;
      } else if constexpr (kOrdered) {
        // the K block count read per tile from the workspace, and the
        // expert's scale offset from the order: kept in registers through
        // the tile loop instead, they made ptxas spill here
        const int kbo = int(*reinterpret_cast<volatile const unsigned int*>(bp.counter + 3));
        cols_ok = col0 < args.N;
        sa_ptr = args.sA + size_t(tile.row0 + row) * kbo;
        sb_ptr = args.sB + tile.sb0 + size_t(col0 / kBlockK) * kbo;
        kb_end = kbo;
      } else {
        cols_ok = col0 < args.N;
        sa_ptr = args.sA + size_t(tile.row0 + row) * Kb;
        sb_ptr = args.sB + (size_t(tile.e) * Nb + col0 / kBlockK) * Kb;
      }

      // FP32 accumulator, two columns per float2 so the promotion runs on the
      // packed FMA (FFMA2)
      float2 acc[Cfg::kColsPerWG / 2];
#pragma unroll
      for (int j = 0; j < Cfg::kColsPerWG / 2; ++j) acc[j] = make_float2(0.f, 0.f);

      float sa_next = row_ok ? __ldg(sa_ptr + kb0) : 0.f;
      float sb_next = cols_ok ? __ldg(sb_ptr + kb0) : 0.f;
      for (int kb = kb0; kb < kb_end; ++kb, ++it) {
        const float sc = sa_next * sb_next;
        if (kb + 1 < kb_end) {
          sa_next = row_ok ? __ldg(sa_ptr + kb + 1) : 0.f;
          sb_next = cols_ok ? __ldg(sb_ptr + kb + 1) : 0.f;
        }
        const int buf = it % NB;
        const uint32_t tph = (it / NB) & 1;
        if (!mbar_wait(&tfull_bar[buf], tph, abort_flag, args.wait_ns)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_base + buf * BN + wg * Cfg::kColsPerWG;
        const float2 sc2 = make_float2(sc, sc);
        // 64-column chunks, one TMEM load each (BN = 256: two per K block).
        // Few wide loads beat many narrow ones: a warp's loads complete one
        // after another, so each costs its own latency.  The TMEM buffer goes
        // back to the MMA warp as soon as the last chunk has landed.
        constexpr int kChunks = Cfg::kColsPerWG / 64;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          uint32_t r[64];
          tmem_ld_32x32b_x64(taddr + c * 64, r);
          tmem_ld_wait_tied(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          reg_tie32(&r[32]);
          if (c + 1 == kChunks) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[buf]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float2 p = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            acc[c * 32 + j] = __ffma2_rn(p, sc2, acc[c * 32 + j]);
          }
        }
      }
      if (!ok) break;
      if constexpr (kSplit) {
        // stage this CTA's partial; the cluster sums and stores it below
        float4* srow = reinterpret_cast<float4*>(smem) + (row * Stage<Cfg>::kPitch +
                                                          wg * Cfg::kColsPerWG) / 4;
#pragma unroll
        for (int j4 = 0; j4 < Cfg::kColsPerWG / 4; ++j4)
          srow[j4] = make_float4(acc[2 * j4].x, acc[2 * j4].y, acc[2 * j4 + 1].x,
                                 acc[2 * j4 + 1].y);
        continue;
      }
      // epilogue: BF16 (round to nearest even).  A warp whose 32 rows are all
      // real outputs stages its band 32 columns at a time in one of its two
      // shared-memory boxes (64-byte swizzle: 16-byte chunk j of row r sits
      // at chunk j ^ (r / 2 % 4)) and one lane stores each box with TMA:
      // whole-line writes that drain while the warp goes on.  Other rows
      // store directly: 16 bytes at a time when rows of D are 16-byte
      // aligned (N % 8 == 0), else element by element.
      const int wrow0 = (warp % 4) * 32;  // first tile row of this warp
      int dN;
      __nv_bfloat16* dD;
      bool d_tma;
      const CUtensorMap* mD;
      if constexpr (kBatch) {
        const BatchProblem& pr = bp.prob[tile.p];
        dN = pr.N;
        dD = pr.D;
        d_tma = pr.d_tma != 0;
        mD = &bp.d[tile.p];
      } else {
        dN = args.N;
        dD = args.D;
        d_tma = args.d_tma != 0;
        mD = &tmD;
      }
      if (d_tma && wrow0 + 32 <= tile.valid_rows) {
        uint8_t* wbox = epi + warp * (2 * Cfg::kEpiBoxBytes);
#pragma unroll
        for (int c = 0; c < Cfg::kColsPerWG / 32; ++c) {
          if (col0 + 32 * c >= dN) break;  // warp-uniform
          uint8_t* box = wbox + (n_stores & 1) * Cfg::kEpiBoxBytes;
          // at most one store pending: the one before it, which used this
          // box, has finished reading it
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2* a4 = acc + 16 * c + 4 * j;
            __nv_bfloat162 p0 = __float22bfloat162_rn(a4[0]);
            __nv_bfloat162 p1 = __float22bfloat162_rn(a4[1]);
            __nv_bfloat162 p2 = __float22bfloat162_rn(a4[2]);
            __nv_bfloat162 p3 = __float22bfloat162_rn(a4[3]);
            uint4 v;
            v.x = *reinterpret_cast<uint32_t*>(&p0);
            v.y = *reinterpret_cast<uint32_t*>(&p1);
            v.z = *reinterpret_cast<uint32_t*>(&p2);
            v.w = *reinterpret_cast<uint32_t*>(&p3);
            *reinterpret_cast<uint4*>(box + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(mD, box, col0 + 32 * c, tile.row0 + wrow0);
            bulk_commit_group();
          }
          ++n_stores;
        }
      } else if (row_ok && dN % 8 != 0) {
        __nv_bfloat16* drow = dD + size_t(tile.row0 + row) * dN + col0;
#pragma unroll
        for (int j = 0; j < Cfg::kColsPerWG / 2; ++j) {
          const __nv_bfloat162 p = __float22bfloat162_rn(acc[j]);
          if (col0 + 2 * j < dN) drow[2 * j] = p.x;
          if (col0 + 2 * j + 1 < dN) drow[2 * j + 1] = p.y;
        }
      } else if (row_ok) {
        __nv_bfloat16* drow = dD + size_t(tile.row0 + row) * dN + col0;
#pragma unroll
        for (int j = 0; j < Cfg::kColsPerWG; j += 8) {
          if (col0 + j < dN) {
            uint4 v;
            __nv_bfloat162 p0 = __float22bfloat162_rn(acc[j / 2 + 0]);
            __nv_bfloat162 p1 = __float22bfloat162_rn(acc[j / 2 + 1]);
            __nv_bfloat162 p2 = __float22bfloat162_rn(acc[j / 2 + 2]);
            __nv_bfloat162 p3 = __float22bfloat162_rn(acc[j / 2 + 3]);
            v.x = *reinterpret_cast<uint32_t*>(&p0);
            v.y = *reinterpret_cast<uint32_t*>(&p1);
            v.z = *reinterpret_cast<uint32_t*>(&p2);
            v.w = *reinterpret_cast<uint32_t*>(&p3);
            *reinterpret_cast<uint4*>(drow + j) = v;
          }
        }
      }
    }
    // this warp's TMA stores have completed before its shared memory can go
    if (lane == 0) bulk_wait_group_all();
  } else {
    regs_decrease<Cfg::kLowRegs>();  // warps 10-11: no work
  }

  if constexpr (kSplit) {
    // every CTA of the cluster has staged its partial (or, on an abort,
    // whatever it holds: the status already says the result is void)
    __syncwarp();
    cluster_sync();
    Tile tile;
    if (warp < Cfg::kPromoWarps && t_begin < t_end && sched.get(t_begin, BN, tile)) {
      // row band [r0, r1) of the tile: summed over the cluster's partials in
      // rank order (deterministic), rounded to BF16, stored along rows
      const int S = args.split;
      const int r0 = part * kBlockM / S, r1 = (part + 1) * kBlockM / S;
      constexpr int kF4 = BN / 4;  // float4s per row
      const float4* mine = reinterpret_cast<const float4*>(smem);
      for (int idx = r0 * kF4 + int(threadIdx.x); idx < r1 * kF4; idx += Cfg::kPromoWarps * 32) {
        const int r = idx / kF4, c4 = idx % kF4;
        const float4* p = mine + r * (Stage<Cfg>::kPitch / 4) + c4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < S; ++q) {
          const float4 w = *map_shared_rank(p, uint32_t(q));
          v.x += w.x;
          v.y += w.y;
          v.z += w.z;
          v.w += w.w;
        }
        const int col = tile.n0 + 4 * c4;
        if (r >= tile.valid_rows || col >= args.N) continue;
        __nv_bfloat16* d = args.D + size_t(tile.row0 + r) * args.N + col;
        const __nv_bfloat162 lo = __float22bfloat162_rn(make_float2(v.x, v.y));
        const __nv_bfloat162 hi = __float22bfloat162_rn(make_float2(v.z, v.w));
        if (args.N % 4 == 0) {  // col + 3 < N and the 8-byte store is aligned
          uint2 u;
          u.x = *reinterpret_cast<const uint32_t*>(&lo);
          u.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(d) = u;
        } else {
          d[0] = lo.x;
          if (col + 1 < args.N) d[1] = lo.y;
          if (col + 2 < args.N) d[2] = hi.x;
          if (col + 3 < args.N) d[3] = hi.y;
        }
      }
    }
    __syncwarp();
    cluster_sync();  // no CTA leaves while another still reads its partial
  }

  __syncthreads();
  if constexpr (kDyn) {
    // every claim of this CTA precedes its count; the last CTA to count
    // leaves both counters at zero for the next launch (which reads them
    // only after this grid has completed)
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(bp.counter + 1, 1u) == gridDim.x - 1) {
        atomicExch(bp.counter, 0u);
        atomicExch(bp.counter + 1, 0u);
      }
    }
  }
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}


// ----------------------------------------- contiguous form in segment order
// One CTA orders the contiguous form's tiles before the GEMM runs them: it
// reads the expert of each 128-row block (m_indices of its first row, as the
// GEMM does), takes each maximal run of blocks of one expert as a segment,
// and lays the segments out largest, smallest, second largest, ... (more
// than kOrderMaxSegs segments: in block order), each segment's tiles in the
// dense form's grouped rasterisation over its own blocks.  Blocks of padding
// (index -1) get no tile; an index >= E sets the status word and its block
// gets no tile.  Tile t of the order: (first row, first column, expert,
// the expert's first sB element).
constexpr int kOrderThreads = 1024;
constexpr int kOrderMaxBlocks = 2048;  // M blocks this ordering takes (larger: block order kernel)
constexpr int kOrderMaxSegs = 256;     // segments it reorders by size

// Exclusive prefix sum over the CTA of one value per thread; *total gets the sum.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d *= 2) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kOrderThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d *= 2) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[kOrderThreads / 32 - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kOrderThreads, 1)
    contig_order_kernel(const int32_t* m_indices, int num_m, int E, int num_n, int BN, int Nb,
                        int Kb, int4* order, unsigned int* counter, int* status) {
  __shared__ int blk[kOrderMaxBlocks];       // expert of each block, -1: no tile
  __shared__ int seg_first[kOrderMaxBlocks];
  __shared__ int seg_len[kOrderMaxBlocks];
  __shared__ int pos_seg[kOrderMaxBlocks];   // segment at each position of the order
  __shared__ int pos_tile0[kOrderMaxBlocks]; // its first tile
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  // m_indices may come from the kernel before this one; the GEMM behind may
  // start its prologue now (it reads the order only after this grid ends)
  griddep_wait();
  griddep_launch_dependents();
  for (int mb = tid; mb < num_m; mb += kOrderThreads) {
    int e = __ldg(m_indices + size_t(mb) * kBlockM);
    if (e >= E) {
      raise_status(status, FP8GEMM_ERR_DEVICE_STATUS);
      e = -1;
    }
    blk[mb] = e < 0 ? -1 : e;
  }
  __syncthreads();
  // segment starts: a block with work whose predecessor holds another expert
  constexpr int kPer = kOrderMaxBlocks / kOrderThreads;
  auto is_start = [&](int mb) {
    return mb < num_m && blk[mb] >= 0 && (mb == 0 || blk[mb - 1] != blk[mb]);
  };
  int mine = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) mine += is_start(tid * kPer + j) ? 1 : 0;
  int S = 0;
  int sid = cta_exclusive_scan(mine, warp_sums, &S);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int mb = tid * kPer + j;
    if (is_start(mb)) {
      int len = 1;
      while (mb + len < num_m && blk[mb + len] == blk[mb]) ++len;
      seg_first[sid] = mb;
      seg_len[sid] = len;
      ++sid;
    }
  }
  __syncthreads();
  // positions: by falling length (ties: segment order), the largest and the
  // smallest alternating
  for (int q = tid; q < S; q += kOrderThreads) {
    int pos = q;
    if (S <= kOrderMaxSegs) {
      const int L = seg_len[q];
      int rank = 0;
      for (int u = 0; u < S; ++u) {
        const int Lu = seg_len[u];
        rank += (Lu > L || (Lu == L && u < q)) ? 1 : 0;
      }
      const int half = (S + 1) / 2;
      pos = rank < half ? 2 * rank : 2 * (S - 1 - rank) + 1;
    }
    pos_seg[pos] = q;
  }
  __syncthreads();
  int tiles_mine[kPer];
  int sum_mine = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int pos = tid * kPer + j;
    tiles_mine[j] = pos < S ? seg_len[pos_seg[pos]] * num_n : 0;
    sum_mine += tiles_mine[j];
  }
  int total = 0;
  int first = cta_exclusive_scan(sum_mine, warp_sums, &total);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int pos = tid * kPer + j;
    if (pos < S) pos_tile0[pos] = first;
    first += tiles_mine[j];
  }
  __syncthreads();
  for (int t = tid; t < total; t += kOrderThreads) {
    int lo = 0, hi = S - 1;  // the last position whose first tile is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (pos_tile0[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int q = pos_seg[lo];
    const int len = seg_len[q], mb0 = seg_first[q];
    const int u = t - pos_tile0[lo];
    const int per_group = kGroupM * num_n;
    const int g = u / per_group;
    const int first_m = g * kGroupM;
    const int gs = min(kGroupM, len - first_m);
    const int r = u - g * per_group;
    order[t] = make_int4((mb0 + first_m + r % gs) * kBlockM, (r / gs) * BN, blk[mb0],
                         blk[mb0] * Nb * Kb);
  }
  if (tid == 0) {
    counter[2] = unsigned(total);
    counter[3] = unsigned(Kb);
  }
}

template <class Cfg, bool kSplit, int kP = 0>
cudaError_t set_smem_attr() {
  // once per device and context: the attribute belongs to the function in
  // one context, and a cudaDeviceReset gives the device a new one
  static unsigned long long set_in[64] = {};  // context id, per device
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && set_in[dev & 63] == ctx) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<Cfg, kSplit, kP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Cfg::kSmemBytes));
  if (e == cudaSuccess) set_in[dev & 63] = ctx;
  return e;
}

// Clusters of `s` split-instance CTAs that can be resident at once (0: none).
template <class Cfg>
int max_clusters(int dev, int s) {
  static int known[64][kMaxSplit + 1] = {};  // 0 unknown, -1 none, else the count
  int& k = known[dev & 63][s];
  if (k == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = s;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<Cfg, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();  // a refused query leaves no sticky error
      n = 0;
    }
    k = n > 0 ? n : -1;
  }
  return k > 0 ? k : 0;
}

// Parts per tile when all `tiles` fit in one wave: as many as leave every
// tile's cluster resident at once, at most kMaxSplit, at least kMinPartKb K
// blocks each, and only for K of kMinSplitKb blocks or more (below that the
// cluster's fixed costs -- staging, two cluster barriers, the exchange --
// ate the gain: neutral at 16 K blocks, 2.4 us slower at 4).  1: whole
// tiles, the persistent instance.
constexpr int kMinSplitKb = 32;
constexpr int kMinPartKb = 4;

template <class Cfg>
int choose_split(const LaunchCtx& c, long long tiles, int Kb) {
  if (tiles >= c.num_sms || Kb < kMinSplitKb) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  long long s = c.num_sms / tiles;
  if (s > Kb / kMinPartKb) s = Kb / kMinPartKb;
  if (s > kMaxSplit) s = kMaxSplit;
  for (; s >= 2; --s)
    if (max_clusters<Cfg>(dev, int(s)) >= tiles) return int(s);
  return 1;
}

template <class Cfg>
cudaError_t run(const LaunchCtx& c, GemmArgs a, int* launches) {
  *launches = 0;
  a.wait_ns = wait_limit_ns();
  CUtensorMap tmA, tmB, tmD;
  const uint64_t a_rows = a.mode == GemmMode::kMasked ? uint64_t(a.E) * a.M : uint64_t(a.M);
  const uint64_t b_rows = uint64_t(a.E) * a.N;
  if (!make_tmap_u8_sw128(&tmA, a.A, a_rows, a.K, kBlockM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&tmB, a.B, b_rows, a.K, Cfg::BN)) return cudaErrorInvalidValue;
  // D has A's row space; without a describable layout (N % 8 != 0, or a base
  // that is not 16-byte aligned) every row takes the direct stores
  memset(&tmD, 0, sizeof(tmD));
  a.d_tma = make_tmap_bf16_sw64(&tmD, a.D, a_rows, uint64_t(a.N), 32) ? 1 : 0;
  if (cudaError_t e = set_smem_attr<Cfg, false>()) return e;
  if (cudaError_t e = set_smem_attr<Cfg, true>()) return e;

  const int num_n = ceil_div(a.N, Cfg::BN);
  const bool masked = a.mode == GemmMode::kMasked;
  // tiles: exact for the dense and contiguous forms; for the masked form an
  // upper bound (the valid rows are on the device; clusters past the valid
  // tiles find no work)
  const long long tiles = (long long)(masked ? a.E : 1) * ceil_div(a.M, kBlockM) * num_n;
  if (tiles == 0) return cudaSuccess;
  a.split = choose_split<Cfg>(c, tiles, ceil_div(a.K, kBlockK));

  if (a.split == 1) {
    // as a programmatic dependent of the previous kernel in the stream (the
    // quantiser of its activations, say): its launch and prologue overlap
    // that kernel's end -- 6 us less per prefill step (quantise A + GEMM, both
    // shapes: 487 against 493 us)
    const int grid = int(tiles < c.num_sms ? tiles : c.num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<Cfg, false>, tmA, tmB, tmD, a,
                                           c.status, BatchParams<0>{}))
      return e;
  } else {
    // one cluster per tile, as a programmatic dependent (its prologue
    // overlaps the end of the stream's earlier work)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles * a.split));
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(a.split);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<Cfg, true>, tmA, tmB, tmD, a,
                                           c.status, BatchParams<0>{}))
      return e;
  }
  *launches = 1;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmArgs& a, int* launches) {
  const bool wide = (a.N % 256 == 0) || a.N >= 2048;
  if (wide) return run<TcCfg<256, 4>>(c, a, launches);
  return run<TcCfg<128, 6>>(c, a, launches);
}

namespace {

// One batched launch with P parameter slots (P = 4: 1.8 KB of kernel
// parameters; P = 32: 14 KB), for the n problems order[0..n) of p.
template <int P>
cudaError_t launch_batch(const LaunchCtx& c, const fp8gemm_problem* p, const int* order, int n,
                         unsigned int* counter, int* launches) {
  using Cfg = TcCfg<256, 4>;
  BatchParams<P> bp;
  memset(&bp, 0, sizeof(bp));
  long long total = 0;
  for (int j = 0; j < n; ++j) {
    const fp8gemm_problem& q = p[order[j]];
    if (!make_tmap_u8_sw128(&bp.a[j], q.A, uint64_t(q.M), uint64_t(q.K), kBlockM))
      return cudaErrorInvalidValue;
    if (!make_tmap_u8_sw128(&bp.b[j], q.B, uint64_t(q.N), uint64_t(q.K), Cfg::BN))
      return cudaErrorInvalidValue;
    BatchProblem& pr = bp.prob[j];
    pr.d_tma = make_tmap_bf16_sw64(&bp.d[j], q.D, uint64_t(q.M), uint64_t(q.N), 32) ? 1 : 0;
    pr.sA = q.sA;
    pr.sB = q.sB;
    pr.D = static_cast<__nv_bfloat16*>(q.D);
    pr.M = q.M;
    pr.N = q.N;
    pr.Kb = ceil_div(q.K, kBlockK);
    pr.num_m = ceil_div(q.M, kBlockM);
    pr.num_n = ceil_div(q.N, Cfg::BN);
    pr.tile0 = int(total);
    pr.fmts = q.formats;
    total += (long long)pr.num_m * pr.num_n;
    if (total > 0x7fffffffLL - 4LL * c.num_sms) return cudaErrorInvalidValue;
  }
  bp.count = n;
  bp.total = int(total);
  bp.counter = counter;
  GemmArgs a{GemmMode::kDense, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0, 0, 1};
  a.wait_ns = wait_limit_ns();
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  if (cudaError_t e = set_smem_attr<Cfg, false, P>()) return e;
  // persistent, one CTA per SM, as a programmatic dependent (see run())
  const int grid = int(total < c.num_sms ? total : c.num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<Cfg, false, P>, unused, unused,
                                         unused, a, c.status, bp))
    return e;
  *launches = 1;
  return cudaSuccess;
}

}  // namespace

size_t contig_order_workspace_bytes(const LaunchCtx& c, const GemmArgs& a) {
  using Cfg = TcCfg<256, 4>;
  const long long num_m = a.M / kBlockM, num_n = ceil_div(a.N, Cfg::BN);
  const bool wide = (a.N % 256 == 0) || a.N >= 2048;  // launch_gemm_tc's BN = 256 instance
  const long long sb_elems = (long long)a.E * ceil_div(a.N, kBlockK) * ceil_div(a.K, kBlockK);
  if (a.mode != GemmMode::kContiguous || !wide || num_m > kOrderMaxBlocks ||
      num_m * num_n < c.num_sms || ceil_div(a.K, kBlockK) < 2 || sb_elems > 0x7fffffffLL)
    return 0;
  return 16 + size_t(num_m * num_n) * sizeof(int4);
}

cudaError_t launch_gemm_tc_contiguous_ordered(const LaunchCtx& c, const GemmArgs& a0, void* ws,
                                              size_t ws_bytes, int* launches) {
  using Cfg = TcCfg<256, 4>;
  *launches = 0;
  const size_t need = contig_order_workspace_bytes(c, a0);
  if (need == 0 || ws_bytes < need) return cudaErrorInvalidValue;
  GemmArgs a = a0;
  a.wait_ns = wait_limit_ns();
  const int num_m = a.M / kBlockM, num_n = ceil_div(a.N, Cfg::BN);
  CUtensorMap tmA, tmB, tmD;
  if (!make_tmap_u8_sw128(&tmA, a.A, uint64_t(a.M), a.K, kBlockM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_sw128(&tmB, a.B, uint64_t(a.E) * a.N, a.K, Cfg::BN))
    return cudaErrorInvalidValue;
  memset(&tmD, 0, sizeof(tmD));
  a.d_tma = make_tmap_bf16_sw64(&tmD, a.D, uint64_t(a.M), uint64_t(a.N), 32) ? 1 : 0;
  if (cudaError_t e = set_smem_attr<Cfg, false, -1>()) return e;
  unsigned int* counter = static_cast<unsigned int*>(ws);
  int4* order = reinterpret_cast<int4*>(static_cast<char*>(ws) + 16);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  // the order, then the GEMM, each as a programmatic dependent of the kernel
  // before it (the GEMM's prologue overlaps the ordering)
  cudaLaunchConfig_t cfg0 = {};
  cfg0.gridDim = dim3(1);
  cfg0.blockDim = dim3(kOrderThreads);
  cfg0.stream = c.stream;
  cfg0.attrs = &attr;
  cfg0.numAttrs = 1;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg0, contig_order_kernel, a.group_info, num_m, a.E,
                                         num_n, Cfg::BN, ceil_div(a.N, kBlockK),
                                         ceil_div(a.K, kBlockK), order, counter, c.status))
    return e;
  *launches = 1;
  const long long bound = (long long)num_m * num_n;  // tiles, padding blocks included
  const int grid = int(bound < c.num_sms ? bound : c.num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = c.stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  BatchParams<-1> bp;
  bp.counter = counter;
  bp.order = order;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<Cfg, false, -1>, tmA, tmB, tmD, a,
                                         c.status, bp))
    return e;
  *launches = 2;
  return cudaSuccess;
}

cudaError_t launch_gemm_tc_batch(const LaunchCtx& c, const fp8gemm_problem* p, int count,
                                 unsigned int* counter, int* launches) {
  *launches = 0;
  if (count < 0 || count > kMaxBatch) return cudaErrorInvalidValue;
  // The problems with work, longest K first, so the long tiles start in the
  // first rounds and the short ones fill the end.  Among problems of equal K
  // the largest and the smallest (by tiles) alternate: a problem with many
  // row blocks reuses each weight tile from L2 and is bound by the tensor
  // cores, one with few streams its weights from HBM, and running the two
  // kinds side by side keeps both busy (32 MoE experts of 8192 Zipf-
  // distributed tokens, N 4096, K 7168: 264.7 us alternated, 273.1 largest
  // first, 279.3 smallest first, 273.4 in expert order).
  int order[kMaxBatch];
  long long tiles[kMaxBatch];
  int n = 0;
  for (int i = 0; i < count; ++i) {
    if (p[i].M <= 0 || p[i].N <= 0) continue;
    tiles[i] = (long long)ceil_div(p[i].M, kBlockM) * ceil_div(p[i].N, 256);
    // insertion: K blocks falling, then tiles falling, then list order
    int j = n++;
    for (; j > 0; --j) {
      const int kb_prev = ceil_div(p[order[j - 1]].K, kBlockK), kb = ceil_div(p[i].K, kBlockK);
      if (kb_prev > kb || (kb_prev == kb && tiles[order[j - 1]] >= tiles[i])) break;
      order[j] = order[j - 1];
    }
    order[j] = i;
  }
  if (n == 0) return cudaSuccess;
  int run_order[kMaxBatch];
  for (int s = 0; s < n;) {  // each run of equal K: largest, smallest, 2nd largest, ...
    int e = s;
    while (e < n && ceil_div(p[order[e]].K, kBlockK) == ceil_div(p[order[s]].K, kBlockK)) ++e;
    int lo = s, hi = e - 1, k = s;
    while (lo <= hi) {
      run_order[k++] = order[lo++];
      if (lo <= hi) run_order[k++] = order[hi--];
    }
    s = e;
  }
  if (n <= kSmallBatch) return launch_batch<kSmallBatch>(c, p, run_order, n, counter, launches);
  return launch_batch<kMaxBatch>(c, p, run_order, n, counter, launches);
}

}  // namespace fp8gemm
