/*
 * fp8gemm.h -- C ABI of libfp8gemm.so: FP8 (e4m3) GEMM with fine-grained
 * (1x128 / 128x128) FP32 scales and BF16 output, for GB300 (sm_103a).
 *
 * What is computed.  With A e4m3 [M, K] scaled per 1x128 tile (sA [M, Kb]) and
 * B e4m3 [N, K] scaled per 128x128 tile (sB [Nb, Kb]), Kb = ceil(K/128),
 * Nb = ceil(N/128):
 *
 *   D[m, n] = bf16( sum_kb sA[m, kb] * sB[n/128, kb]
 *                          * sum_{k in block kb} A[m, k] * B[n, k] )
 *
 * -- each 128-wide K block is contracted on the tensor cores, then "promoted":
 * multiplied by its own scale product and added into an FP32 accumulator
 * ("lpnh.cn/news/2822121" section 2.3; granularity from "blog.hotdry.top:
 * DeepGEMM FP8 GEMM fine-grained scaling kernels", sections "fine-grained
 * scaling core design" and "two-level accumulation").  The scale product
 * sA*sB is formed in FP32 and must be finite.
 *
 * Shapes.  K is any positive multiple of 16 (a tensor copy's row stride must
 * be a multiple of 16 bytes); when K is not a multiple of 128 the last K
 * block holds the K % 128 remaining columns -- its scales cover those only,
 * and the GEMM pads the block with zeros.  M and N are any non-negative
 * sizes (the contiguous form keeps M_pad % 128 == 0).  Below, "K/128" in a
 * scale shape means ceil(K/128).
 *
 * Conventions shared by every call:
 *  - Every pointer is a DEVICE pointer owned by the caller; the library keeps
 *    no reference after the call returns.  Matrices are row-major with K
 *    contiguous (D = A * B^T); scale tensors are row-major FP32.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream): it
 *    validates on the host, enqueues, and returns.
 *  - Host-side validation failures return a negative code and enqueue nothing:
 *    FP8GEMM_ERR_NULL (a required pointer is NULL), FP8GEMM_ERR_ALIGN (a base
 *    pointer is not 16-byte aligned), FP8GEMM_ERR_SHAPE (negative size,
 *    K % 16 != 0, K = 0, M_pad % 128 != 0, or a size past INT32 index
 *    range), FP8GEMM_ERR_ARCH (the current device is not compute capability
 *    10.3), FP8GEMM_ERR_LAUNCH (the CUDA launch itself failed).
 *  - Zero-sized problems (M = 0, M_pad = 0, E = 0, or N = 0) succeed and do
 *    nothing.
 *  - Conditions only the device can see (an m_indices entry >= E, a masked_m
 *    entry > M_max or < 0, a pipeline wait that exceeded its time limit) do
 *    not trap: the kernel records FP8GEMM_ERR_DEVICE_STATUS or
 *    FP8GEMM_ERR_TIMEOUT in a per-device status word, skips the offending
 *    tile and finishes.  Read it with fp8gemm_get_device_status().
 *  - Inputs and outputs must not overlap.
 *  - The dense path for M <= 64 may split K across CTAs and reduce partial
 *    sums through a per-(device, stream) workspace that the library allocates
 *    with cudaMalloc on the first such call on that stream (about 10 MB, kept
 *    until released or process exit) and zeroes on that stream; fp8gemm_dense_quant_a at
 *    M > 64 without Q/sA keeps its quantised A in a second per-stream buffer,
 *    and fp8gemm_dense_batch and the ordered contiguous form their tile
 *    counters (and order) in small per-stream buffers.
 *    Such a first call must therefore not happen during CUDA graph capture.
 *    Calls on different streams never share a workspace.  The reduction
 *    order is fixed, so results are deterministic.  A caller that retires a
 *    stream frees its workspaces with fp8gemm_release_workspaces() before
 *    destroying it; fp8gemm_workspace_bytes() reports what is held.
 *  - The dense and grouped paths for M > 64 split each output tile's K loop
 *    over a thread-block cluster when all tiles fit in one wave of the SMs
 *    and K spans at least 32 blocks of 128; the clusters' FP32 partials are
 *    summed in a fixed order through distributed shared memory (no
 *    workspace).  Results stay deterministic for a given shape; a split tile
 *    may differ from the unsplit sum in the last bits of FP32 before the
 *    BF16 rounding.
 */
#ifndef FP8GEMM_H
#define FP8GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8gemm_stream_t; /* same handle as cudaStream_t */

enum fp8gemm_status {
  FP8GEMM_OK = 0,
  FP8GEMM_ERR_NULL = -1,
  FP8GEMM_ERR_ALIGN = -2,
  FP8GEMM_ERR_SHAPE = -3,
  FP8GEMM_ERR_ARCH = -4,
  FP8GEMM_ERR_LAUNCH = -5,
  FP8GEMM_ERR_DEVICE_STATUS = -6,
  FP8GEMM_ERR_TIMEOUT = -7,
  FP8GEMM_ERR_SCRATCH_LIMIT = -8,
  FP8GEMM_ERR_FORMAT = -9,
  FP8GEMM_ERR_FLAGS = -10
};

/* FP8 operand formats of the *_fmt calls ("news.rkmt.cn/news/5092" section
 * 2.1: e4m3 -- 4 exponent, 3 mantissa bits, largest finite 448 -- for
 * activations and weights; e5m2 -- 5 exponent, 2 mantissa bits, IEEE-style
 * infinities and NaNs, largest finite 57344 -- for gradients and other
 * wide-range tensors).  Any other value returns FP8GEMM_ERR_FORMAT. */
enum fp8gemm_format {
  FP8GEMM_FMT_E4M3 = 0,
  FP8GEMM_FMT_E5M2 = 1
};

/*
 * fp8_quant_1x128 -- quantise activations per 1x128 tile (online scaling).
 *
 * Rule ("news.rkmt.cn/news/5092" section 5.2; rounding from
 * "lpnh.cn/news/2822121" section 6.3): for each row m and K block kb,
 *   amax = max |X[m, 128kb : 128kb+128]|,  s = amax / 448  (FP32, IEEE RN),
 *   Q[m, k] = e4m3(X[m, k] / s)  (FP32 IEEE division, then round to nearest
 *   even, saturating at +-448),   sX[m, kb] = s.
 * A block with amax = 0 stores s = 0 and bytes 0x00.  NaN/Inf inputs are
 * outside the contract.
 *
 *   X   f32 [M, K]  (input)         Q  u8 [M, K]  (output, e4m3 bytes)
 *   sX  f32 [M, K/128] (output)     K % 16 == 0; all pointers 16-B aligned.
 */
int fp8_quant_1x128(const float* X, uint8_t* Q, float* sX, int M, int K,
                    fp8gemm_stream_t stream);

/*
 * fp8_quant_128x128 -- quantise weights per 128x128 tile (the offline step
 * that prepares B; same rule, amax over the whole tile; ragged last row tile
 * allowed).  Batched over E independent matrices (E = 1 for a dense B).
 *
 *   W   f32 [E, N, K] (input)       Q  u8 [E, N, K] (output)
 *   sW  f32 [E, ceil(N/128), K/128] (output)
 */
int fp8_quant_128x128(const float* W, uint8_t* Q, float* sW, int E, int N, int K,
                      fp8gemm_stream_t stream);

/*
 * fp8_quant_1x128_fmt / fp8_quant_128x128_fmt -- fp8_quant_1x128 and
 * fp8_quant_128x128 with the output format chosen: the same rule with the
 * format's largest finite value as the limit (s = amax / 448 for e4m3,
 * amax / 57344 for e5m2) and its round-to-nearest-even, saturating encoding.
 * FP8GEMM_FMT_E4M3 gives exactly the bytes and scales of the plain calls.
 */
int fp8_quant_1x128_fmt(const float* X, uint8_t* Q, float* sX, int M, int K, int fmt,
                        fp8gemm_stream_t stream);
int fp8_quant_128x128_fmt(const float* W, uint8_t* Q, float* sW, int E, int N, int K, int fmt,
                          fp8gemm_stream_t stream);

/*
 * fp8_quant_1x128_ex / fp8_quant_128x128_ex -- the _fmt calls with an
 * optional saturation counter, for monitoring FP8 overflow in production
 * ("blog.hotdry.top: DeepGEMM FP8 GEMM fine-grained scaling kernels",
 * section on numerical-stability checks and monitoring, which lists an FP8
 * overflow count among the metrics to watch).
 *
 *   sat_count  device address of a 64-bit counter (8-byte aligned), or NULL.
 *              The call ADDS to it (it is never reset here: zero it once and
 *              it accumulates over calls) the number of elements x of blocks
 *              with amax != 0 whose FP32 quotient x / s is not within
 *              +-limit (448 e4m3, 57344 e5m2) -- the values the saturating
 *              encoding clamps.  With s = amax / limit this happens only when
 *              FP32 rounding pushes x / s just past the limit (one element of
 *              a few percent of Gaussian blocks) or when amax / limit
 *              underflows to 0 (|amax| < about 6e-43 for e4m3; every element
 *              of such a block then counts).  Finite inputs only.
 *   NULL: the bytes, scales and launch of the _fmt call; with a counter the
 *   bytes and scales are the same.  A misaligned counter: FP8GEMM_ERR_ALIGN.
 *   Asynchronous on `stream` like the rest: read the counter after the
 *   stream has reached this call.
 */
int fp8_quant_1x128_ex(const float* X, uint8_t* Q, float* sX, int M, int K, int fmt,
                       unsigned long long* sat_count, fp8gemm_stream_t stream);
int fp8_quant_128x128_ex(const float* W, uint8_t* Q, float* sW, int E, int N, int K, int fmt,
                         unsigned long long* sat_count, fp8gemm_stream_t stream);

/*
 * fp8gemm_dense -- D = A * B^T with block scales ("lpnh.cn/news/2822121"
 * section 4.1 dense main loop; scaling as above).
 *
 *   A  u8 [M, K]   sA f32 [M, K/128]
 *   B  u8 [N, K]   sB f32 [ceil(N/128), K/128]
 *   D  bf16 [M, N] (output, written in full)
 *   M, N >= 0; K > 0, K % 16 == 0.
 */
int fp8gemm_dense(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                  void* D, int M, int N, int K, fp8gemm_stream_t stream);

/*
 * fp8gemm_dense_fmt -- fp8gemm_dense with each operand's format given
 * (a_fmt, b_fmt: FP8GEMM_FMT_*), e.g. an e5m2 gradient against e4m3
 * weights; mixing the formats is allowed ("lpnh.cn/news/2822121" section
 * 2.1).  The tensor cores decode each operand in its own format; scaling,
 * promotion, layouts and limits are those of fp8gemm_dense.  Operand bytes
 * that encode infinity or NaN (e5m2) propagate as in IEEE arithmetic.
 */
int fp8gemm_dense_fmt(const uint8_t* A, const float* sA, int a_fmt, const uint8_t* B,
                      const float* sB, int b_fmt, void* D, int M, int N, int K,
                      fp8gemm_stream_t stream);

/* Flags of fp8gemm_dense_ex. */
enum fp8gemm_flags {
  /* The caller promises that B and sB are not written by any kernel that
   * may still be running when this call's kernel starts (e.g. constant
   * weights).  The decode path (M <= 64), launched as a programmatic
   * dependent of the kernel before it, may then stage its first weight tiles
   * into shared memory while that kernel finishes, instead of waiting for it
   * first; activations, scales of A and D still wait.  Breaking the promise
   * gives results computed from stale weights.  Other paths accept the flag
   * and ignore it. */
  FP8GEMM_FLAG_B_READ_ONLY = 1u
};

/*
 * fp8gemm_dense_ex -- fp8gemm_dense_fmt with flags (FP8GEMM_FLAG_*; 0 gives
 * exactly fp8gemm_dense_fmt).  Unknown flag bits return FP8GEMM_ERR_FLAGS.
 * Arithmetic, layouts and limits are those of fp8gemm_dense.  (The pages
 * describe weights that stay fixed across calls -- quantised once, offline,
 * "lpnh.cn/news/2822121" section 2.3 -- which is what the flag lets the
 * kernel exploit.)
 */
int fp8gemm_dense_ex(const uint8_t* A, const float* sA, int a_fmt, const uint8_t* B,
                     const float* sB, int b_fmt, void* D, int M, int N, int K, unsigned flags,
                     fp8gemm_stream_t stream);

/*
 * fp8gemm_dense_quant_a -- fp8gemm_dense on FP32 activations: A and sA are
 * the 1x128 quantisation of X (fp8_quant_1x128's rule, same bytes and
 * scales), produced on the way into the GEMM ("news.rkmt.cn/news/5092"
 * section 2.3 and "bhfrc.com/news/60211" section 6: the scale work belongs
 * with the producer, not in a separate step of the caller).
 *
 *   X  f32 [M, K]  (input)
 *   Q  u8 [M, K], sA f32 [M, K/128] (optional outputs: both NULL, or both
 *      given to receive the quantised activations, e.g. to reuse them)
 *   B  u8 [N, K]   sB f32 [ceil(N/128), K/128]
 *   D  bf16 [M, N] (output, written in full)
 *   M, N >= 0; K > 0, K % 16 == 0; all pointers 16-B aligned.
 *
 * A few rows (decode shapes where each CTA of the cluster split-K form has at
 * most 16 1x128 blocks of A to quantise, e.g. M <= 4 at K = 2048): one
 * kernel, whose CTAs quantise their own K range of X into their operand
 * stages (same bytes and scales; the first N tile's CTAs also write Q/sA
 * when given).  Otherwise two kernels on `stream`: the quantiser, then the
 * GEMM launched as its programmatic dependent, so the GEMM's launch,
 * prologue and weight prefetch overlap the quantiser; with Q/sA NULL the
 * quantised A then lives in a library-owned per-stream buffer of about
 * M*K*(1 + 4/128) bytes.  Either way D is bit-identical to
 * fp8_quant_1x128 followed by fp8gemm_dense.  Exactly one of Q, sA NULL
 * returns FP8GEMM_ERR_NULL.
 */
int fp8gemm_dense_quant_a(const float* X, uint8_t* Q, float* sA, const uint8_t* B,
                          const float* sB, void* D, int M, int N, int K,
                          fp8gemm_stream_t stream);

/*
 * fp8gemm_dense_quant_a_ex -- fp8gemm_dense_quant_a with flags (as
 * fp8gemm_dense_ex; 0 gives exactly fp8gemm_dense_quant_a).  With
 * FP8GEMM_FLAG_B_READ_ONLY the decode-path GEMM, launched as the
 * quantiser's programmatic dependent, stages its first weight tiles while
 * the quantiser runs -- at decode sizes the quantiser occupies few SMs, so
 * the GEMM's CTAs find room beside it.
 */
int fp8gemm_dense_quant_a_ex(const float* X, uint8_t* Q, float* sA, const uint8_t* B,
                             const float* sB, void* D, int M, int N, int K, unsigned flags,
                             fp8gemm_stream_t stream);

/*
 * fp8gemm_grouped_contiguous -- MoE experts in one launch, each expert's
 * tokens a contiguous row segment of A ("news.rkmt.cn/news/5092" section 5.3;
 * "news.rkmt.cn/news/5092" section 1.2: one launch for many experts).
 *
 *   A  u8 [M_pad, K]          sA f32 [M_pad, K/128]
 *   B  u8 [E, N, K]           sB f32 [E, ceil(N/128), K/128]
 *   m_indices i32 [M_pad] (device): expert of each row, -1 for padding rows
 *   D  bf16 [M_pad, N] (output; padding rows are left unspecified)
 *   M_pad % 128 == 0, and every 128-row block holds rows of a single expert
 *   (segments padded to 128 rows, padding at each segment's end).  Only the
 *   first row's index of each block is read; a block whose first index is -1
 *   is skipped; an index >= E sets FP8GEMM_ERR_DEVICE_STATUS.
 *
 * When the tiles (M_pad/128 x ceil(N/256)) make at least a wave of the SMs,
 * with N % 256 == 0 or N >= 2048, K > 128, M_pad <= 262144 and
 * E * ceil(N/128) * ceil(K/128) < 2^31, the call is two launches: a one-CTA
 * kernel that orders the tiles by expert segment (the experts with the most
 * and the fewest blocks alternating, so the tiles that stream their weights
 * from HBM run beside those that reuse them from L2), then the GEMM taking
 * its tiles in that order.  The order and two tile counters live in a
 * per-(device, stream) workspace of 16 + 16 * tiles bytes that the library
 * allocates and zeroes on the first such call on the stream (not during
 * stream capture; see the conventions above) and that every launch leaves
 * ready for the next.  Results do not depend on the order: each tile's
 * arithmetic is the same.
 */
int fp8gemm_grouped_contiguous(const uint8_t* A, const float* sA, const uint8_t* B,
                               const float* sB, const int32_t* m_indices, void* D,
                               int M_pad, int N, int K, int E, fp8gemm_stream_t stream);

/*
 * fp8gemm_grouped_masked -- MoE experts with per-expert valid-row counts kept
 * in device memory, so the launch shape is fixed and a CUDA graph can be
 * replayed with new counts ("bhfrc.com/news/60211" section 4.3; skipping
 * empty blocks, "lpnh.cn/news/2822121" section 5.2).
 *
 *   A  u8 [E, M_max, K]       sA f32 [E, M_max, K/128]
 *   B  u8 [E, N, K]           sB f32 [E, ceil(N/128), K/128]
 *   masked_m i32 [E] (device): rows of expert e to compute, 0..M_max
 *   D  bf16 [E, M_max, N] (output: rows >= masked_m[e] are NOT written)
 *   A masked_m entry outside [0, M_max] is clamped and sets
 *   FP8GEMM_ERR_DEVICE_STATUS.
 */
int fp8gemm_grouped_masked(const uint8_t* A, const float* sA, const uint8_t* B,
                           const float* sB, const int32_t* masked_m, void* D,
                           int E, int M_max, int N, int K, fp8gemm_stream_t stream);

/*
 * fp8gemm_grouped_contiguous_fmt / fp8gemm_grouped_masked_fmt -- the two
 * grouped forms with each operand's format given (FP8GEMM_FMT_*), as
 * fp8gemm_dense_fmt does for the dense form; all else as the e4m3 calls.
 */
int fp8gemm_grouped_contiguous_fmt(const uint8_t* A, const float* sA, int a_fmt,
                                   const uint8_t* B, const float* sB, int b_fmt,
                                   const int32_t* m_indices, void* D, int M_pad, int N, int K,
                                   int E, fp8gemm_stream_t stream);
int fp8gemm_grouped_masked_fmt(const uint8_t* A, const float* sA, int a_fmt, const uint8_t* B,
                               const float* sB, int b_fmt, const int32_t* masked_m, void* D,
                               int E, int M_max, int N, int K, fp8gemm_stream_t stream);

/*
 * fp8gemm_grouped_table -- many independent dense problems in one launch,
 * each described by an entry of a table in DEVICE memory, for batched decode
 * requests ("bhfrc.com/news/60211" sections 4.2-4.3 and 6: shape data in
 * device memory, so one captured CUDA graph can be replayed with new shapes).
 * The launch depends only on num_problems and max_M; the table (pointers and
 * sizes) is read on the device when the kernel runs, so it may be rewritten
 * between replays of a graph that captured this call.
 *
 * Per entry p (the layouts and arithmetic of fp8gemm_dense_fmt):
 *   A u8 [M, K], sA f32 [M, ceil(K/128)], B u8 [N, K],
 *   sB f32 [ceil(N/128), ceil(K/128)], D bf16 [M, N] (written in full)
 * with 0 <= M <= max_M, N >= 0, K > 0 and K % 16 == 0, A and B 16-byte
 * aligned, sA and sB 4-byte, D 2-byte, and `formats` = a_fmt | (b_fmt << 8)
 * (FP8GEMM_FMT_* each; 0 means e4m3 x e4m3).  An entry with M = 0 or N = 0 is
 * skipped.  An entry that breaks these rules is skipped and sets
 * FP8GEMM_ERR_DEVICE_STATUS (read it with fp8gemm_get_device_status).
 * Entries must not write overlapping D.
 *
 * The kernel is built for decode-sized problems (the padded width is 16, 32
 * or 64 rows, chosen from max_M).  An entry with more rows is processed that
 * many rows at a time -- each 64-row chunk streams the entry's weight tiles
 * again, mostly from L2 -- so large-M problems are served correctly but
 * fp8gemm_dense is the faster call for them.  The (entry, 128-column tile,
 * row chunk, K block) units of the whole table are divided evenly over the
 * CTAs (stream-K): an item whose K range is shared by several CTAs is summed
 * from their FP32 partials in a fixed order, through a per-(device, stream)
 * workspace that the library allocates and zeroes on the first call on the
 * stream (a few MB; not during stream capture, see the conventions above), so
 * results are deterministic for a given table and launch configuration.
 *
 *   problems  device array of num_problems entries, 8-byte aligned
 * Host-side errors: FP8GEMM_ERR_SHAPE (num_problems < 0, max_M < 1),
 * FP8GEMM_ERR_NULL, FP8GEMM_ERR_ALIGN.
 */
typedef struct fp8gemm_problem {
  const uint8_t* A;
  const float* sA;
  const uint8_t* B;
  const float* sB;
  void* D;
  int M, N, K;
  int formats; /* a_fmt | (b_fmt << 8); 0 = e4m3 x e4m3 */
} fp8gemm_problem;

int fp8gemm_grouped_table(const fp8gemm_problem* problems, int num_problems, int max_M,
                          fp8gemm_stream_t stream);

/*
 * fp8gemm_dense_batch -- up to FP8GEMM_MAX_DENSE_BATCH independent dense
 * problems of prefill size in ONE launch of the 128-row tensor-core GEMM (the
 * grouped GEMM of "bhfrc.com/news/60211" sections 4.2-4.3: one launch over a
 * list of problems, each with its own M, N, K; here the list is on the host
 * and fixed at the call) -- several layers' GEMMs, or the experts of a MoE
 * layer whose token counts the host knows (each expert's rows, unpadded, as
 * one entry).  Each problem's output tiles are those fp8gemm_dense computes
 * for it on its whole-tile path; the persistent CTAs take the tiles of all
 * problems from one shared sequence and each CTA its next tile when it
 * finishes the last, so the partial last round of one problem is filled
 * with tiles of the next instead of leaving SMs idle.  The sequence runs the
 * problems with the longest K first; among problems of equal K, the one with
 * the most tiles, then the one with the fewest, then the second most, ...
 * (problems with many row blocks reuse their weight tiles from L2 and keep
 * the tensor cores busy while those with few stream their weights from HBM),
 * each problem's tiles in the dense form's order.  A tile's arithmetic and summation
 * order do not depend on which CTA takes it, so results are deterministic,
 * and bit-identical to fp8gemm_dense_fmt's where that call takes its
 * whole-tile path with 256-column tiles (N % 256 == 0 or N >= 2048, and at
 * least as many tiles as SMs).
 *
 *   problems      HOST array of num_problems entries (read during the call;
 *                 the library keeps no reference), layouts and rules per
 *                 entry as for fp8gemm_grouped_table's entries, except that
 *                 M has no upper bound and sA, sB and D are 16-byte aligned
 *   num_problems  0..FP8GEMM_MAX_DENSE_BATCH
 * The tiles are handed out through two counters in a per-(device, stream)
 * workspace of 256 bytes that the library allocates and zeroes on the first
 * such call on the stream (not during stream capture, see the conventions
 * above); every launch leaves them at zero, so the call may be captured in a
 * graph once the workspace exists.  Two launches of this call on one stream
 * run in stream order and never share the counters at the same time.
 * Entries with M = 0 or N = 0 are skipped.  Host-side errors:
 * FP8GEMM_ERR_SHAPE (num_problems out of range, or an entry with a negative
 * size, K = 0 or K % 16 != 0), FP8GEMM_ERR_FORMAT, FP8GEMM_ERR_NULL,
 * FP8GEMM_ERR_ALIGN; nothing is enqueued then.
 */
#define FP8GEMM_MAX_DENSE_BATCH 32
int fp8gemm_dense_batch(const fp8gemm_problem* problems, int num_problems,
                        fp8gemm_stream_t stream);

/*
 * fp8gemm_dense_small_m_noalloc -- the same computation as fp8gemm_dense for
 * decode-sized M (1..64), for callers that must not have the library allocate
 * device memory: a server that reserves its whole memory budget up front and
 * treats any later allocation as an error, a framework whose own pool owns the
 * device memory, or a latency-critical loop that cannot take cudaMalloc's
 * implicit synchronisation.  (The pages this library follows have no
 * counterpart; this variant exists for that constraint only.)
 *
 * It allocates nothing: its split-K scratch is a fixed array of 10.25 MiB in
 * the library's device image.  The array is created on a GPU when the part of
 * the library that holds it is loaded there -- under CUDA's default lazy
 * module loading, by the first call of this entry point on that GPU -- and
 * stays until the process exits.  That first call on each device also does a
 * one-time set-up (it looks up the array's device address with
 * cudaGetSymbolAddress); later calls reuse the address.  So make the first
 * call on each device during start-up, before the memory budget is fixed and
 * before any CUDA stream capture begins.  After a cudaDeviceReset the next
 * call repeats the set-up in the new context.
 *
 * Arguments, layouts, ownership and results are those of fp8gemm_dense, with
 * these limits: M <= 64 and N <= 8388608 (ceil(N/128) arrival counters must
 * fit), at most 160 SMs used.  Larger problems return
 * FP8GEMM_ERR_SCRATCH_LIMIT and enqueue nothing.
 *
 * All calls on a device share the one scratch array and it keeps the previous
 * call's contents; each call clears what must start at zero with an
 * asynchronous memset on `stream`.  Calls whose execution overlaps on the GPU
 * (e.g. issued on two streams without ordering between them) race on the
 * scratch and produce wrong results: order them.
 */
int fp8gemm_dense_small_m_noalloc(const uint8_t* A, const float* sA, const uint8_t* B,
                                  const float* sB, void* D, int M, int N, int K,
                                  fp8gemm_stream_t stream);

/*
 * fp8gemm_get_device_status -- after every kernel enqueued on `stream` so
 * far, read and clear the current device's status word in one atomic step
 * (a one-thread kernel on `stream`), then synchronise `stream`:
 * *out = FP8GEMM_OK, FP8GEMM_ERR_DEVICE_STATUS or FP8GEMM_ERR_TIMEOUT.  A
 * condition raised meanwhile by a kernel on another stream is either
 * returned here or left for the next read.  On FP8GEMM_ERR_TIMEOUT the call
 * also synchronises the device and frees every library workspace of it (a
 * launch that gave up can leave a split-K reduction's counters mid-count);
 * the next calls allocate fresh, zeroed ones.  Returns FP8GEMM_OK, or
 * FP8GEMM_ERR_NULL / FP8GEMM_ERR_LAUNCH if `out` is NULL or the CUDA calls
 * fail.
 */
int fp8gemm_get_device_status(fp8gemm_stream_t stream, int* out);

/* fp8gemm_strerror -- static description of a status code. */
const char* fp8gemm_strerror(int code);

/* fp8gemm_num_kernel_launches -- kernels this process enqueued through the
 * library so far (all devices); a host-side counter for launch accounting. */
uint64_t fp8gemm_num_kernel_launches(void);

/*
 * fp8gemm_release_workspaces -- free every library-owned workspace of
 * `stream` on the current device (the split-K buffer of the decode path, the
 * quantised-activation buffer of fp8gemm_dense_quant_a, the problem table's
 * partials, and the tile counters and order of fp8gemm_dense_batch and of
 * the ordered contiguous form).  It first
 * synchronises `stream`, since work enqueued there may still use them; the
 * next call that needs a workspace on that stream allocates it again.  Call
 * it before cudaStreamDestroy for streams that are retired: a stream handle
 * that is destroyed and later reused by the runtime would otherwise find its
 * predecessor's buffer.  Not allowed during stream capture.  Returns
 * FP8GEMM_OK, or FP8GEMM_ERR_LAUNCH if a CUDA call fails.
 * (The pages have no counterpart: this is resource management of the
 * library's own buffers.)
 */
int fp8gemm_release_workspaces(fp8gemm_stream_t stream);

/* fp8gemm_workspace_bytes -- bytes of library-owned workspaces currently held
 * (all devices and streams). */
uint64_t fp8gemm_workspace_bytes(void);

/*
 * fp8gemm_set_wait_limit_ns -- time limit, in nanoseconds of the GPU's global
 * timer, of every pipeline wait inside the GEMM kernels launched after this
 * call (process-wide; 0 restores the default of 2 s).  A wait that exceeds
 * it is treated as a deadlock: the CTA stops, lets its copies and tensor-core
 * operations in flight finish, frees its TMEM, exits, and the status word
 * reads FP8GEMM_ERR_TIMEOUT (results of that launch are void).  A short limit
 * makes the failure path observable in tests; production code keeps the
 * default.  The hardware cluster barriers of the split-K forms have no limit
 * of their own; every thread reaches them because every wait before them is
 * bounded.  Returns FP8GEMM_OK.  (The pages have no counterpart: this is the
 * library's deadlock detection.)
 */
int fp8gemm_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* FP8GEMM_H */
