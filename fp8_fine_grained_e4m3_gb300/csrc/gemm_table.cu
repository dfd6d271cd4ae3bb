// gemm_table.cu -- block-scaled FP8 GEMMs of many independent decode-sized
// problems in one launch, each problem's pointers and sizes read from a table
// in device memory (sm_103a).
//
// "bhfrc.com/news/60211" sections 4.2-4.3 and 6: a grouped call takes a list
// of problems whose shape data sit in device memory, so that one captured
// CUDA graph can be replayed with new shapes.  Here the launch shape depends
// only on the problem count and the largest M (the host's arguments); every
// pointer and size comes from the table on the device, and so does every
// check of it.
//
// Per problem p the arithmetic is fp8gemm_dense's (1x128 A scales, 128x128 B
// scales, each K block contracted on the tensor cores and promoted into an
// FP32 accumulator, BF16 out), with each entry's own operand formats (e4m3 or
// e5m2, "lpnh.cn/news/2822121" section 2.1).  The decode layout of
// gemm_small_m.cu: swap-AB (a 128-row weight tile is the MMA's M, up to MP of
// the problem's rows its N), one TMEM partial per K block, promotion per
// output column.  A problem with more rows than MP is taken MP rows at a time:
// its items are (N tile, row chunk), the chunks of one tile consecutive, so
// CTAs running side by side share that weight tile through L2.
//
// What differs: no tensor maps (they would have to be rebuilt per problem on
// the device), so four producer warps fill the 128-byte-swizzled operand
// stages with 16-byte cp.async copies -- zero-filled past a problem's N, M or
// K.  Each producer lane's cp.async.mbarrier.arrive lands on the stage's full
// barrier when that lane's copies have landed; the MMA thread fences the
// generic proxy against the async one before the tensor cores read the stage.
// (One producer warp issued too few copies to keep a stage's 16 KB moving:
// 215 us against 116 us with four, on 16 decode problems of 4096x7168.)
//
// Work division: stream-K.  The (item, K block) units of all problems, in
// table order, are dealt out evenly over the persistent CTAs -- whole items
// over a fixed grid leave the last round mostly idle when there are few
// items per CTA ("news.rkmt.cn/news/5092" section 4.2: size the work to the
// SM count).  A CTA whose range begins or ends inside an item leaves its FP32
// partial in a workspace slot; the last contributor to finish the item (one
// acquire-release atomic per contributor, on a counter owned by the item's
// first CTA) sums every partial in CTA order -- deterministic -- writes BF16
// and resets the counter.  Every role walks the CTA's unit range identically.
#include "common.cuh"
#include "ptx.cuh"

namespace fp8gemm {
namespace {

template <int MP_>
struct TabCfg {
  static constexpr int MP = MP_;
  static constexpr int kStages = 6;
  // two CTAs per SM where they fit (MP = 16): twice the copies in flight
  static constexpr int kCtasPerSm = MP == 16 ? 2 : 1;
  static constexpr int kThreads = 288;
  static constexpr int kLoadWarp = 4;  // warps 4-7 load
  static constexpr int kLoadWarps = 4;
  static constexpr int kMmaWarp = 8;
  static constexpr int kWBytes = 128 * kBlockK;
  static constexpr int kXBytes = MP * kBlockK;
  static constexpr int kTmemBufs = MP == 64 ? 4 : 8;
  static constexpr int kTmemCols = kTmemBufs * MP < 128 ? 128 : kTmemBufs * MP;
  static constexpr int kScaleKb = 16;
  static constexpr int kBarBytes = 512;
  static constexpr int kAuxBytes = kBarBytes + kScaleKb * (MP + 4) * 4;
  static constexpr size_t kSmemBytes =
      1024 + size_t(kStages) * (kWBytes + kXBytes) + kAuxBytes;
  // barriers, then TMEM holder, abort and last flags, and the CTA's range
  static_assert((2 * kStages + 2 * kTmemBufs + 2) * 8 + 16 + 4 * 8 <= kBarBytes, "barrier area");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kCtasPerSm == 1 || kSmemBytes <= 113 * 1024, "two CTAs per SM");
};

// A problem as the kernels use it: its table entry, or an empty problem if
// the entry breaks the contract (then `bad` is set).
struct Prob {
  const uint8_t* A;
  const float* sA;
  const uint8_t* B;
  const float* sB;
  __nv_bfloat16* D;
  int M, N, K, Kb;
  int chunks;  // row chunks of MP rows
  int tiles;   // work items: N tiles x row chunks
  int a_fmt, b_fmt;
  bool bad;
};

__device__ __forceinline__ bool al16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__device__ Prob load_problem(const fp8gemm_problem* tab, int p, int max_M, int MP) {
  Prob r;
  const fp8gemm_problem* e = tab + p;
  r.A = reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(&e->A)));
  r.sA = reinterpret_cast<const float*>(__ldg(reinterpret_cast<const unsigned long long*>(&e->sA)));
  r.B = reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(&e->B)));
  r.sB = reinterpret_cast<const float*>(__ldg(reinterpret_cast<const unsigned long long*>(&e->sB)));
  r.D = reinterpret_cast<__nv_bfloat16*>(__ldg(reinterpret_cast<const unsigned long long*>(&e->D)));
  r.M = __ldg(&e->M);
  r.N = __ldg(&e->N);
  r.K = __ldg(&e->K);
  const int f = __ldg(&e->formats);
  r.a_fmt = f & 0xff;
  r.b_fmt = (f >> 8) & 0xff;
  const bool empty = r.M == 0 || r.N == 0;
  r.bad = r.M < 0 || r.N < 0 || r.M > max_M || r.K <= 0 || r.K % 16 != 0 ||
          r.a_fmt > FP8GEMM_FMT_E5M2 || r.b_fmt > FP8GEMM_FMT_E5M2 || (f >> 16) != 0 ||
          (!empty && (!r.A || !r.sA || !r.B || !r.sB || !r.D || !al16(r.A) || !al16(r.B) ||
                      (reinterpret_cast<uintptr_t>(r.sA) & 3u) ||
                      (reinterpret_cast<uintptr_t>(r.sB) & 3u) ||
                      (reinterpret_cast<uintptr_t>(r.D) & 1u)));
  r.Kb = r.bad ? 0 : ceil_div(r.K, kBlockK);
  r.chunks = (r.bad || empty) ? 0 : ceil_div(r.M, MP);
  r.tiles = (r.bad || empty) ? 0 : ceil_div(r.N, 128) * r.chunks;
  return r;
}

// The (problem, N tile) items of this CTA, in order: item = blockIdx.x +
// j * gridDim.x over the concatenation of every problem's tiles.
// How the table's work is dealt out, the same choice in every CTA: whole
// items round-robin (r[2] = 0), unless that leaves the grid less than 70 %
// busy (fewer items than CTAs, or a last round mostly empty); then the units
// themselves are split evenly (stream-K) over r[2] CTAs -- at most one per
// unit, so that every CTA taking part has a non-empty range -- this CTA's
// being [r[0], r[1]).  r[3]: the table's units.
__device__ void table_range(const fp8gemm_problem* tab, int P, int max_M, int MP, int c, int G,
                            long long r[4]) {
  long long U = 0, I = 0;
  for (int p = 0; p < P; ++p) {
    const Prob q = load_problem(tab, p, max_M, MP);
    U += (long long)q.tiles * q.Kb;
    I += q.tiles;
  }
  r[0] = r[1] = r[2] = 0;
  r[3] = U;
  if (U == 0 || U > 0x7fffffffLL) return;  // more units than 32-bit indices: nothing to do
  const long long rounds = (I + G - 1) / G;
  if (10 * I < 7LL * G * rounds) {  // stream-K
    const long long active = U < G ? U : G;
    r[2] = active;
    if (c < active) {
      r[0] = c * U / active;
      r[1] = (c + 1) * U / active;
    }
    return;
  }
}

// A CTA's units [begin(c), begin(c + 1)) and the CTA holding unit u.
struct Split {
  long long U;
  int G;
  __device__ int begin(int c) const { return int((long long)c * U / G); }
  __device__ int cta_of(int u) const { return int(((long long)(u + 1) * G - 1) / U); }
};

// One item's share of a CTA's unit range: K blocks [kb0, kb1) of the item
// whose first unit is item_u0 (rows m0.., N tile `tile` of problem cur).
struct Seg {
  int tile, m0, kb0, kb1;
  int item_u0;
};

// Walks the problems in table order by unit (or item) index.
struct Walk {
  const fp8gemm_problem* tab;
  int P, max_M, MP;
  int p = -1;
  int first = 0;       // problem p's first unit (the table's units fit in int)
  int first_item = 0;  // and first item
  Prob cur;
  __device__ void advance() {
    first += cur.tiles * cur.Kb;
    first_item += cur.tiles;
    if (++p < P) cur = load_problem(tab, p, max_M, MP);
  }
  __device__ void start() {
    if (p < 0) {
      p = 0;
      if (P > 0) cur = load_problem(tab, 0, max_M, MP);
    }
  }
  // Moves to the problem holding unit u; false past the last one.
  __device__ bool seek(int u) {
    start();
    while (p < P && u >= first + cur.tiles * cur.Kb) advance();
    return p < P;
  }
  // Moves to the problem holding item i; false past the last one.
  __device__ bool seek_item(int i) {
    start();
    while (p < P && i >= first_item + cur.tiles) advance();
    return p < P;
  }
  // The segment that starts at unit u and ends at `end` or the item's end.
  __device__ __forceinline__ Seg segment(int u, int end) const {
    const int rel = u - first;
    const int item = rel / cur.Kb;
    Seg g;
    g.kb0 = rel - item * cur.Kb;
    g.kb1 = min(cur.Kb, g.kb0 + (end - u));
    g.tile = item / cur.chunks;
    g.m0 = (item % cur.chunks) * MP;
    g.item_u0 = first + item * cur.Kb;
    return g;
  }
};

// A CTA's next segment, k counting them: whole items blockIdx.x,
// + gridDim.x, ... (rng[2] == 0), or (stream-K) the next piece of the CTA's
// unit range [rng[0], rng[1]), whose first piece is k == 0.  Every role walks
// the same sequence.
__device__ __forceinline__ bool next_seg(Walk& w, const volatile long long* rng, int& k, int& u,
                                         Seg& g) {
  if (rng[2] == 0) {
    const int item = int(blockIdx.x) + k * int(gridDim.x);
    if (!w.seek_item(item)) return false;
    const int iu = w.first + (item - w.first_item) * w.cur.Kb;
    g = w.segment(iu, iu + w.cur.Kb);
  } else {
    if (k == 0) u = int(rng[0]);
    if (u >= int(rng[1]) || !w.seek(u)) return false;
    g = w.segment(u, int(rng[1]));
    u += g.kb1 - g.kb0;
  }
  ++k;
  return true;
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, Cfg::kCtasPerSm)
    gemm_table_kernel(const fp8gemm_problem* __restrict__ tab, int P, int max_M, int* status,
                      unsigned long long wait_ns, float* ws_partials, int* ws_counters) {
  constexpr int MP = Cfg::MP;
  constexpr int kStages = Cfg::kStages;
  constexpr int NB = Cfg::kTmemBufs;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smW = smem;
  uint8_t* smX = smem + kStages * Cfg::kWBytes;
  uint8_t* aux = smX + kStages * Cfg::kXBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* tfull_bar = full_bar + 2 * kStages;
  uint64_t* tempty_bar = tfull_bar + NB;
  uint64_t* drain_bar = tempty_bar + NB;
  uint64_t* group_bar = drain_bar + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(group_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_holder + 2);
  long long* range_s = reinterpret_cast<long long*>(tmem_holder + 4);  // [4]
  float* sa_s = reinterpret_cast<float*>(aux + Cfg::kBarBytes);
  float* sb_s = sa_s + Cfg::kScaleKb * MP;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 32 * Cfg::kLoadWarps);  // every producer lane
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(drain_bar, 1);
    mbar_init(group_bar, 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  auto fail = [&]() {
    *abort_flag = 1;
    raise_status(status, FP8GEMM_ERR_TIMEOUT);
  };
  griddep_wait();  // the table and the operands belong to the stream's order
  if (threadIdx.x == 0)
    table_range(tab, P, max_M, MP, int(blockIdx.x), int(gridDim.x), const_cast<long long*>(range_s));
  __syncthreads();
  // the range stays in shared memory (read where used): registers are short
  // in the two-CTAs-per-SM configuration
  const volatile long long* rng = range_s;
  // stream-K: an item's contributors are exactly the CTAs from its first to
  // its last unit's (every one of them has a non-empty range)
  auto sk = [&]() { return Split{rng[3], int(rng[2])}; };


  if (warp >= Cfg::kLoadWarp && warp < Cfg::kLoadWarp + Cfg::kLoadWarps) {
    // ------------------------------------------------------ producer
    // 8 lanes per 128-byte row (one 16-byte chunk each), 4 rows per copy
    // instruction; chunk c of tile row r lands at r * 128 + ((c ^ (r % 8)) * 16)
    const int c = lane % 8, r0 = lane / 8 + 4 * (warp - Cfg::kLoadWarp);
    constexpr int kRowStep = 4 * Cfg::kLoadWarps;
    Walk w{tab, P, max_M, MP};
    int i = 0;  // unit (K block) counter
    bool ok = true;
    int k = 0, u = 0;
    Seg g;
    while (ok && next_seg(w, rng, k, u, g)) {
      const Prob& q = w.cur;
      const int tile = g.tile, m0 = g.m0;
      for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&empty_bar[s], ((i / kStages) & 1) ^ 1, abort_flag, wait_ns)) {
          fail();
          ok = false;
          break;
        }
        const bool k_in = kb * kBlockK + c * 16 < q.K;
        const uint32_t w_dst = smem_addr(smW + s * Cfg::kWBytes);
#pragma unroll 4
        for (int r = r0; r < 128; r += kRowStep) {
          const int n = tile * 128 + r;
          const bool in = k_in && n < q.N;
          const uint8_t* src = in ? q.B + size_t(n) * q.K + kb * kBlockK + c * 16 : q.B;
          cp_async_16(w_dst + r * 128 + ((c ^ (r & 7)) << 4), src, in ? 16u : 0u);
        }
        const uint32_t x_dst = smem_addr(smX + s * Cfg::kXBytes);
#pragma unroll
        for (int r = r0; r < MP; r += kRowStep) {
          const bool in = k_in && m0 + r < q.M;
          const uint8_t* src = in ? q.A + size_t(m0 + r) * q.K + kb * kBlockK + c * 16 : q.A;
          cp_async_16(x_dst + r * 128 + ((c ^ (r & 7)) << 4), src, in ? 16u : 0u);
        }
        cp_async_mbar_arrive(&full_bar[s]);  // arrives when this lane's copies land
      }
    }
    cp_async_wait_all();  // this thread's copies have landed before it exits
  } else if (warp == Cfg::kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t w_base = smem_addr(smW);
      const uint32_t x_base = smem_addr(smX);
      Walk w{tab, P, max_M, MP};
      int i = 0;
      bool ok = true;
      int k = 0, u = 0;
      Seg g;
      while (ok && next_seg(w, rng, k, u, g)) {
        // swap-AB: the MMA's A operand is the weights (the problem's B)
        const uint32_t idesc =
            idesc_f8_f32(128, MP, uint32_t(w.cur.b_fmt), uint32_t(w.cur.a_fmt));
        for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
          const int s = i % kStages;
          const int buf = i % NB;
          if (!mbar_wait(&tempty_bar[buf], ((i / NB) & 1) ^ 1, abort_flag, wait_ns) ||
              !mbar_wait(&full_bar[s], (i / kStages) & 1, abort_flag, wait_ns)) {
            fail();
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // the copies (generic proxy) before the MMA's reads
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
      }
      if (i > 0) {  // every issued MMA has finished before TMEM is released
        umma_commit(drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < 200000000ull) {
        }
      }
    }
  } else if (warp < 4) {
    // -------------------------------------------- promotion + epilogue
    const int t = threadIdx.x;  // TMEM lane = column within the N tile
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    uint32_t gphase = 0;
    bool ok = true;
    auto group_sync = [&]() -> bool {
      mbar_arrive(group_bar);
      const bool r = mbar_wait(group_bar, gphase, abort_flag, wait_ns);
      gphase ^= 1;
      return r;
    };
    if (t == 0) {  // report entries that break the contract (once per launch)
      for (int p = blockIdx.x; p < P; p += gridDim.x)
        if (load_problem(tab, p, max_M, MP).bad) raise_status(status, FP8GEMM_ERR_DEVICE_STATUS);
    }
    Walk w{tab, P, max_M, MP};
    int i = 0;
    int k = 0, u = 0;
    Seg g;
    while (ok && next_seg(w, rng, k, u, g)) {
      const Prob& q = w.cur;  // the walk does not move until the next segment
      const bool seg_first = k == 1;  // this CTA's first segment
      const int tile = g.tile, m0 = g.m0;
      const int rows = min(MP, q.M - m0);  // rows of this chunk
      float acc[MP];
#pragma unroll
      for (int j = 0; j < MP; ++j) acc[j] = 0.f;
      for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
        const int qq = (kb - g.kb0) % Cfg::kScaleKb;
        if (qq == 0) {  // stage the next batch of scales
          const int nkb = min(Cfg::kScaleKb, g.kb1 - kb);
          if (!group_sync()) { fail(); ok = false; break; }
          for (int idx = t; idx < MP * nkb; idx += 128) {
            const int j = idx / nkb, b = idx % nkb;
            sa_s[b * MP + j] = j < rows ? __ldg(q.sA + size_t(m0 + j) * q.Kb + kb + b) : 0.f;
          }
          if (t < nkb) sb_s[t] = __ldg(q.sB + size_t(tile) * q.Kb + kb + t);
          if (!group_sync()) { fail(); ok = false; break; }
        }
        const int buf = i % NB;
        if (!mbar_wait(&tfull_bar[buf], (i / NB) & 1, abort_flag, wait_ns)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_base + buf * MP;
        const float sb = sb_s[qq];
        const float* sa_row = sa_s + qq * MP;
        if constexpr (MP == 16) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(taddr, r);
          tmem_ld_wait_tied16(r);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[buf]);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = fmaf(__uint_as_float(r[j]), sa_row[j] * sb, acc[j]);
        } else {
#pragma unroll
          for (int cc = 0; cc < MP / 32; ++cc) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + cc * 32, r);
            tmem_ld_wait_tied(r);
            if (cc + 1 == MP / 32) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty_bar[buf]);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[cc * 32 + j] =
                  fmaf(__uint_as_float(r[j]), sa_row[cc * 32 + j] * sb, acc[cc * 32 + j]);
          }
        }
      }
      if (!ok) break;
      bool write = true;
      if (!(g.kb0 == 0 && g.kb1 == q.Kb)) {
        // part of an item: publish this CTA's partial (the item's real rows);
        // the last contributor sums them all in CTA order
        float* mine = ws_partials + size_t(2 * blockIdx.x + (seg_first ? 0 : 1)) * MP * 128;
#pragma unroll
        for (int j = 0; j < MP; ++j)
          if (j < rows) mine[j * 128 + t] = acc[j];
        if (!group_sync()) { fail(); ok = false; break; }
        const int c_first = sk().cta_of(g.item_u0);
        const int c_last = sk().cta_of(g.item_u0 + q.Kb - 1);
        if (t == 0) {
          // release this CTA's partial (ordered before by the group barrier),
          // acquire those of the contributors that arrived earlier
          const int prev = atomic_add_acq_rel_gpu(ws_counters + c_first, 1);
          const int is_last = prev == c_last - c_first;
          if (is_last) ws_counters[c_first] = 0;  // ready for the next launch
          *last_flag = is_last;
        }
        if (!group_sync()) { fail(); ok = false; break; }
        write = *last_flag != 0;
        if (!group_sync()) { fail(); ok = false; break; }  // last_flag is reused
        if (write) {
#pragma unroll
          for (int j = 0; j < MP; ++j) acc[j] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            // contributor c's slot: its first segment unless the item began
            // after the start of c's range
            const int cs = (c > c_first || g.item_u0 == sk().begin(c)) ? 2 * c : 2 * c + 1;
            const float* pp = ws_partials + size_t(cs) * MP * 128;
#pragma unroll
            for (int j = 0; j < MP; ++j)
              if (j < rows) acc[j] += __ldcg(pp + j * 128 + t);
          }
        }
      }
      const int n = tile * 128 + t;
      if (write && n < q.N) {
#pragma unroll
        for (int j = 0; j < MP; ++j)
          if (j < rows) q.D[size_t(m0 + j) * q.N + n] = __float2bfloat16_rn(acc[j]);
      }
    }
  }

  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// Workspace layout, the same for every configuration so that one per-stream
// buffer can serve them all: the counters (one per CTA of the largest grid,
// two CTAs per SM) first, then the partial slots.  The counters are zero
// between launches; partial slots are written before they are read.
size_t counter_bytes(const LaunchCtx& c) {
  return (size_t(c.num_sms) * 2 * sizeof(int) + 255) / 256 * 256;
}

template <class Cfg>
size_t workspace_bytes(const LaunchCtx& c) {
  const size_t grid = size_t(c.num_sms) * Cfg::kCtasPerSm;
  return counter_bytes(c) + 2 * grid * Cfg::MP * 128 * sizeof(float);
}

template <class Cfg>
cudaError_t run(const LaunchCtx& c, const fp8gemm_problem* tab, int P, int max_M, void* ws,
                size_t ws_bytes) {
  static_assert(Cfg::kCtasPerSm <= 2, "counter region");
  if (ws_bytes < workspace_bytes<Cfg>(c)) return cudaErrorInvalidValue;
  int* counters = static_cast<int*>(ws);
  float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + counter_bytes(c));
  // once per device and context: the attribute belongs to the function in
  // one context, and a cudaDeviceReset gives the device a new one
  static unsigned long long set_in[64] = {};  // context id, per device
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || set_in[dev & 63] != ctx) {
    cudaError_t e = cudaFuncSetAttribute(gemm_table_kernel<Cfg>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(Cfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    set_in[dev & 63] = ctx;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.num_sms * Cfg::kCtasPerSm);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_table_kernel<Cfg>, tab, P, max_M, c.status,
                            wait_limit_ns(), partials, counters);
}

}  // namespace

size_t table_workspace_bytes(const LaunchCtx& c, int max_M) {
  if (max_M <= 16) return workspace_bytes<TabCfg<16>>(c);
  if (max_M <= 32) return workspace_bytes<TabCfg<32>>(c);
  return workspace_bytes<TabCfg<64>>(c);
}

cudaError_t launch_gemm_table(const LaunchCtx& c, const fp8gemm_problem* tab, int P, int max_M,
                              void* ws, size_t ws_bytes) {
  if (max_M <= 16) return run<TabCfg<16>>(c, tab, P, max_M, ws, ws_bytes);
  if (max_M <= 32) return run<TabCfg<32>>(c, tab, P, max_M, ws, ws_bytes);
  return run<TabCfg<64>>(c, tab, P, max_M, ws, ws_bytes);
}

}  // namespace fp8gemm
