/*
 * gemm_f16 — a barrier-pipelined FP16 GEMM for NVIDIA GB300 (sm_103a).
 *
 *     C = A * B        A: M x K, B: K x N, C: M x N, all row-major IEEE
 *                      binary16; products accumulated in FP32; C rounded to
 *                      binary16 with round-to-nearest-even.
 *
 * The operation is the half-precision GEMM of the "Xe2 ESIMD GEMM" page
 * (sections "Inner-loop rules", "Payload CSE", "Tile walk order",
 * "Correctness testing"), re-designed for Blackwell: its K loop is a ring of
 * shared-memory stages, each guarded by mbarriers whose phase completes when
 * the pending-arrival count and the transaction byte count both reach zero
 * (the "mbarrier State and Operations" page, "Phase Completion Condition"
 * and "Core APIs").  The optional split of the K range across work units is
 * the counterpart of the global split ("GSU") named on the "Insert Cluster
 * Barrier Pass" page, Rule 1; its partial sums are reduced in a fixed order,
 * so split results are bitwise reproducible run to run.
 *
 * Conventions for every entry point below:
 *   - Pointers named A, B, C are DEVICE pointers on the plan's device unless
 *     the name says host (hA, hB, hC).  The caller owns them; the library
 *     never frees them.
 *   - Leading dimensions (lda, ldb, ldc) count elements, not bytes.
 *   - Device pointers must be 16-byte aligned and leading dimensions must be
 *     multiples of 8 elements (the tensor-memory-accelerator's rule for
 *     global addresses and strides); otherwise GEMM_F16_ERR_MISALIGNED.
 *   - Return value: GEMM_F16_OK (0) or a negative gemm_f16_error code.  On
 *     an error no work has been enqueued.
 *   - A plan may be used from one host thread / one stream at a time (it
 *     owns a workspace and a status word that concurrent runs would share).
 *   - Every kernel of a call is launched with programmatic stream
 *     serialisation, and some let the next kernel of the stream start
 *     early: a
 *     kernel the caller launches next on the same stream WITH that launch
 *     attribute must execute griddepcontrol.wait
 *     (cudaGridDependencySynchronize) before it touches the call's results
 *     or operands; kernels, copies and events enqueued without it are
 *     ordered as usual.
 */
#ifndef GEMM_F16_H
#define GEMM_F16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_f16_plan_s *gemm_f16_plan_t;  /* opaque, library-owned */
typedef struct CUstream_st *gemm_f16_stream_t;    /* == cudaStream_t; NULL = legacy default stream */

typedef enum gemm_f16_error {
    GEMM_F16_OK = 0,
    GEMM_F16_ERR_INVALID_ARG = -1,        /* bad size, null pointer, ld too small, bad split_k, bad option */
    GEMM_F16_ERR_MISALIGNED = -2,         /* pointer not 16-byte aligned or ld not a multiple of 8 */
    GEMM_F16_ERR_UNSUPPORTED_DEVICE = -3, /* not a compute-capability 10.3 (sm_103a) device */
    GEMM_F16_ERR_OOM = -4,                /* device or pinned-host allocation failed */
    GEMM_F16_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed (see gemm_f16_last_cuda_error) */
    GEMM_F16_ERR_TIMEOUT = -6,            /* a bounded in-kernel wait expired (reported by gemm_f16_status) */
    GEMM_F16_ERR_SCRATCH_TOO_SMALL = -7   /* gemm_f16_run_noalloc: problem exceeds its fixed scratch */
} gemm_f16_error;

/* Options for gemm_f16_set_option. */
typedef enum gemm_f16_option {
    /* Upper bound, in nanoseconds, of every in-kernel barrier wait.  When a
     * wait runs out the kernel records GEMM_F16_ERR_TIMEOUT, stops issuing
     * work, waits (bounded) for its own copies in flight, frees its tensor
     * memory and returns.  Default 1e9 (1 s).  Must be > 0. */
    GEMM_F16_OPT_TIMEOUT_NS = 1,
    /* Order in which output tiles are handed to the persistent CTAs:
     * 0 = Morton (Z-order, "Xe2 ESIMD GEMM" page, "Tile walk order"), the
     * default; 1 = row-major.  A single-CTA launch whose work units all fit
     * in one wave (one per CTA, all co-resident, so the order cannot change
     * what shares the cache at a time) takes row-major order either way.
     * Results do not depend on it. */
    GEMM_F16_OPT_TILE_ORDER = 2,
    /* TEST ONLY.  If >= 0, the producer of the given work unit expects the
     * bytes of its first stage but issues no copy for it, so that stage's
     * barrier never completes and the bounded waits must run out.  No copy
     * is left in flight.  Default -1 (off). */
    GEMM_F16_OPT_FAULT_UNIT = 3,
    /* Which kernel runs the product: 0 = automatic (the CTA-pair kernel when
     * M > 128 and ceil(M/256) * ceil(N/256) * split_k is at least half the
     * number of co-resident pairs, else the single-CTA kernel; in place of
     * the pair kernel the cluster-of-four kernel, without a repack of A,
     * when A and B are row-major, A's row pitch is not a multiple of 128
     * bytes, N >= 2048, A has at least 2^22 elements, GEMM_F16_OPT_A_REPACK
     * is not 2 and its waves of 36 clusters are no more than the pair
     * kernel's waves),
     * 1 = single-CTA kernel (128-row tiles, tcgen05 cta_group::1),
     * 2 = CTA-pair kernel with 256-row x 256-column tiles (two TMEM
     * accumulators, epilogue overlapped; with one split a partial last wave
     * runs as K halves merged by a second kernel, see gemm_f16_pair_tiles,
     * or as 128-wide tiles), 3 = cluster-of-four kernel: two CTA pairs
     * compute a 256 x 512 cluster tile, each 256 x 256 half as in kernel 2,
     * and share their A rows through multicast copies (each CTA fetches
     * half of the A rows it shares with its counterpart in the other
     * pair), so an SM fetches a quarter fewer bytes per MMA; row-major A
     * and B only (other layouts run kernel 2), no K-halves tail, 36 clusters
     * of four on 152 SMs (GEMM_F16_INFO_MAX_QUADS).  Any other value is
     * GEMM_F16_ERR_INVALID_ARG; 3 without clusters of four (or 2 and 3
     * without pairs) is GEMM_F16_ERR_UNSUPPORTED_DEVICE.
     * Results agree within the usual tolerance; split results are bitwise
     * reproducible for a fixed choice. */
    GEMM_F16_OPT_KERNEL = 4,
    /* Output tile width of the single-CTA kernel: 0 = automatic (a cost
     * model picks 256, 128 or 64 columns so that small problems spread over
     * more SMs), or 256 / 128 / 64.  Narrower tiles get a deeper ring
     * (4 / 6 / 8 stages in the same shared memory).  Results agree within
     * the usual tolerance. */
    GEMM_F16_OPT_TILE_WIDTH = 5,
    /* Most SMs one launch may occupy (0 = all of them), e.g. to leave SMs
     * to work on other streams; the cluster kernels still run one cluster
     * (2 or 4 SMs) when the limit is below that.  The tile schedules are
     * planned for the full device either way.  Also bounds the persistent CTA-pair
     * attention kernel (one cluster of two CTAs per two SMs); the
     * single-CTA attention kernel launches one CTA per 128 query rows and
     * ignores it. */
    GEMM_F16_OPT_SM_LIMIT = 6,
    /* Attention kernel (attn_f16_fwd in attn_f16.h): 0 = automatic (the
     * CTA-pair kernel), 1 = single-CTA kernel (128 query rows, blocks of 64
     * keys), 2 = CTA-pair kernel (256 query rows over two SMs, blocks of
     * 128 keys; persistent: each cluster of two CTAs works through several
     * (batch, head, 256-row) items).  Results agree within the usual
     * tolerance and do not depend on the number of clusters. */
    GEMM_F16_OPT_ATTN_KERNEL = 7,
    /* Key split of the CTA-pair attention kernel: 0 = automatic (when the
     * (batch, head, 256-row) items fill less than half of the co-resident
     * CTA pairs and there are at least four 128-key blocks, each item's
     * keys are cut into up to min(pairs / items, blocks / 2) ranges), n >= 1 =
     * n ranges (capped at the number of key blocks; 1 = no split).  Each
     * range writes a normalised FP32 partial of O with its row offsets and
     * sums to the plan's workspace, and a second kernel merges the ranges
     * in order (bitwise reproducible for a fixed n).  The single-CTA
     * attention kernel ignores it. */
    GEMM_F16_OPT_ATTN_SPLIT = 8,
    /* Repack of A when its row pitch (lda * 2 bytes) is not a multiple of
     * 128 bytes: 0 = automatic (for the CTA-pair kernel when N >= 2048 and
     * A has at least 2^22 elements; not for the cluster-of-four kernel,
     * which fetches half as many A rows per SM), 1 = never, 2 = whenever
     * the pitch is off.  A 128-byte row of an operand copy from such a matrix touches two
     * cache lines, which slows the copies that feed the MMAs (4000 x 4104 x
     * 3000 with lda = 3000: ~20 % longer than with lda = 3008); the repack
     * copies A once into plan-owned rows of whole lines (grown on the
     * stream like the split workspace, kept for later runs) and the product
     * reads that copy.  Results are bit-identical either way. */
    GEMM_F16_OPT_A_REPACK = 9,
    /* Kernel timing records: 0 = off (default), 1 = on.  While on, every
     * gemm_f16_run / gemm_f16_run_ex / gemm_f16_run_host call records a pair
     * of CUDA events on the launch stream directly before and after its
     * product kernel (the single-CTA, pair or cluster-of-four kernel; not
     * the repack of A, the K-halves merge or the split reduction), and every
     * attn_f16_fwd / attn_f16_fwd_host call does the same around its
     * attention kernel (not the merge of key ranges), so that
     * gemm_f16_kernel_time can report the kernels' own durations.  The event
     * between two launches stops a kernel from starting before the previous
     * one on the stream has ended (the programmatic dependent launch that
     * otherwise overlaps their set-up), so timed runs are a little slower
     * back to back.  Nothing is recorded while the stream is being captured
     * into a graph, or once 65536 pairs are waiting to be read.  Events come
     * from a plan-owned pool that grows on demand (cudaEventCreate) and is
     * freed with the plan. */
    GEMM_F16_OPT_KERNEL_TIMING = 10
} gemm_f16_option;

/*
 * Create a plan on CUDA device `device`.  Checks the device (compute
 * capability 10.3), sets the kernels' shared-memory limits and allocates the
 * plan's status word (mapped pinned host memory).  The workspace for split
 * runs and the CTA-pair kernel's work lists are allocated on first use.
 * `*out` receives the plan, or NULL on error.
 */
int gemm_f16_plan(gemm_f16_plan_t *out, int device);

/*
 * Enqueue C = A * B on `stream` (asynchronous; nothing is synchronised).
 *   M, N, K  > 0.
 *   A        device, M x K row-major, row stride lda >= K.
 *   B        device, K x N row-major, row stride ldb >= N.
 *   C        device, M x N row-major, row stride ldc >= N.  Overwritten
 *            (no alpha/beta).  Must not overlap A or B.
 *   split_k  1 = no split requested: one pass over K per output tile, except
 *            that the CTA-pair kernel may run the tiles of a partial last
 *            wave as two K halves whose FP32 sums a second kernel adds
 *            (see gemm_f16_pair_tiles; deterministic).  s > 1 = the K range of
 *            every tile is cut into s contiguous, non-empty ranges of
 *            64-wide k-blocks (range t covers k-blocks
 *            [floor(t*KB/s), floor((t+1)*KB/s)), KB = ceil(K/64)); each
 *            range's FP32 partial tile goes to the plan's workspace and a
 *            second kernel sums the s partials in order t = 0..s-1 in FP32
 *            and rounds once to binary16.  Requires s <= KB.
 * The first run of the CTA-pair kernel for a new shape builds its work list
 * and uploads it (cudaMalloc and a synchronous copy; the single-CTA kernel
 * derives its tile order on the device and needs no list), and a split run,
 * a run with K halves or a repack of A may grow a plan buffer (stream-ordered
 * on `stream`); make one run of each shape before capturing the stream in a
 * graph.
 * Errors found on the device (a wait that timed out) are reported later by
 * gemm_f16_status.
 */
int gemm_f16_run(gemm_f16_plan_t plan, int M, int N, int K,
                 const void *A, int64_t lda, const void *B, int64_t ldb,
                 void *C, int64_t ldc, int split_k, gemm_f16_stream_t stream);

/*
 * Operand storage for gemm_f16_run_ex.  The product is always C = A * B
 * with A of M x K and B of K x N (element (i, k) of A, (k, j) of B); the
 * layout says how each operand sits in memory:
 *   GEMM_F16_LAYOUT_NN  A row-major (M rows of K, stride lda >= K),
 *                       B row-major (K rows of N, stride ldb >= N);
 *   GEMM_F16_LAYOUT_TN  A stored transposed: K rows of M, A(i, k) at
 *                       A[k * lda + i], lda >= M; B as in NN;
 *   GEMM_F16_LAYOUT_NT  A as in NN; B stored transposed: N rows of K,
 *                       B(k, j) at B[j * ldb + k], ldb >= K;
 *   GEMM_F16_LAYOUT_TT  both stored transposed.
 * A transposed operand is read by the same tensor copies with the other
 * dimension innermost and handed to the tensor core with the other major
 * mode: no copy or transpose kernel is run.  These layouts are not in the
 * pages' kernel, whose operands are row-major A and B; they cover the
 * usual "transposed operand" cases of a GEMM library.
 */
enum {
    GEMM_F16_LAYOUT_NN = 0,
    GEMM_F16_LAYOUT_TN = 1,   /* bit 0: A stored K x M */
    GEMM_F16_LAYOUT_NT = 2,   /* bit 1: B stored N x K */
    GEMM_F16_LAYOUT_TT = 3
};

/*
 * gemm_f16_run with an operand layout (above).  gemm_f16_run is
 * gemm_f16_run_ex with GEMM_F16_LAYOUT_NN.  Same semantics, workspace,
 * split-K order and errors; GEMM_F16_ERR_INVALID_ARG also for a layout
 * outside 0..3.
 */
int gemm_f16_run_ex(gemm_f16_plan_t plan, int layout, int M, int N, int K,
                    const void *A, int64_t lda, const void *B, int64_t ldb,
                    void *C, int64_t ldc, int split_k, gemm_f16_stream_t stream);

/*
 * What gemm_f16_run_ex would enqueue for these sizes with the plan's current
 * options, without enqueuing anything (host only):
 *   info[0]  kernel: 1 single-CTA, 2 CTA pair, 3 cluster of four;
 *   info[1]  kernel launches per call: the product, plus one for the split
 *            reduction when split_k > 1, plus one for the repack of A, plus
 *            one for merging the K halves of a partial last wave of pair
 *            tiles (see gemm_f16_pair_tiles);
 *   info[2]  1 if A is repacked first (GEMM_F16_OPT_A_REPACK), else 0;
 *   info[3]  output tile width of the chosen kernel (single-CTA: 256 / 128 /
 *            64 columns; pair: 256).
 * Returns GEMM_F16_OK or GEMM_F16_ERR_INVALID_ARG (null plan or info, sizes
 * or split_k < 1, layout outside 0..3, lda below the stored row length).
 */
int gemm_f16_run_info(gemm_f16_plan_t plan, int layout, int M, int N, int K, int64_t lda,
                      int split_k, int info[4]);

/*
 * Same product with HOST operands: copies hA and hB into plan-owned device
 * buffers, runs gemm_f16_run on them and copies the result into hC.
 * Consecutive calls overlap: the input copies run on a plan-internal stream
 * into one of two alternating device slots, so the next call's input copies
 * proceed while this call's product and result copy (both on `stream`)
 * run.  Hence hA and hB must be ready on the host when the call is made
 * (work enqueued earlier on `stream` is not waited for before they are
 * read); synchronise `stream` before reading hC or reusing hA / hB.
 * Pinned host memory gives asynchronous copies.  Host buffers need no
 * alignment; lda/ldb/ldc >= K/N/N (any value).  The device slots grow on
 * demand (growing synchronises the device) and stay with the plan.  Calls
 * on different streams must be ordered by the caller (one product at a
 * time per plan); a slot's next input copies wait for the result copy of
 * the call that last used it, whatever stream that call ran on.
 */
int gemm_f16_run_host(gemm_f16_plan_t plan, int M, int N, int K,
                      const void *hA, int64_t lda, const void *hB, int64_t ldb,
                      void *hC, int64_t ldc, int split_k,
                      gemm_f16_stream_t stream);

/* Free everything the plan owns (synchronises the plan's device).  NULL is
 * accepted and ignored. */
int gemm_f16_destroy(gemm_f16_plan_t plan);

/*
 * Device-reported status of the runs completed so far, then cleared:
 * GEMM_F16_OK or GEMM_F16_ERR_TIMEOUT.  Synchronises nothing: call it after
 * synchronising the stream of the runs it should cover.
 */
int gemm_f16_status(gemm_f16_plan_t plan);

/* Set a gemm_f16_option (see above).  Applies to later runs. */
int gemm_f16_set_option(gemm_f16_plan_t plan, int option, int64_t value);

/* Read-only plan facts for gemm_f16_get_option. */
enum {
    GEMM_F16_INFO_NUM_SMS = 100,   /* SMs of the plan's device */
    GEMM_F16_INFO_MAX_PAIRS = 101, /* co-resident CTA pairs of the pair kernel (0: unavailable) */
    GEMM_F16_INFO_MAX_QUADS = 102  /* co-resident clusters of four of kernel 3 (0: unavailable) */
};

/* Read an option's current value, or one of the GEMM_F16_INFO_* facts. */
int gemm_f16_get_option(gemm_f16_plan_t plan, int option, int64_t *value);

/*
 * Durations of the kernels timed since the last call (GEMM_F16_OPT_KERNEL_TIMING):
 * waits for each recorded pair's second event (cudaEventSynchronize), adds
 * up the elapsed times, returns the events to the plan's pool and forgets
 * the pairs.  *total_ms receives the sum in milliseconds and *launches the
 * number of timed launches (0 and 0.0 when none was recorded).  Returns
 * GEMM_F16_OK, GEMM_F16_ERR_INVALID_ARG for a null argument, or
 * GEMM_F16_ERR_CUDA if an event cannot be read (the pairs are forgotten
 * either way).
 */
int gemm_f16_kernel_time(gemm_f16_plan_t plan, double *total_ms, int64_t *launches);

/* Static description of an error code (never NULL). */
const char *gemm_f16_strerror(int code);

/* Text of the last CUDA error seen by this host thread (never NULL). */
const char *gemm_f16_last_cuda_error(void);

/*
 * Host-only: what gemm_f16_run_info would report for a plan with default
 * options (automatic kernel, tile width and repack; Morton order) on a device
 * with `num_sms` SMs, `max_pairs` co-resident clusters of two and
 * `max_quads` of four (GEMM_F16_INFO_NUM_SMS / _MAX_PAIRS / _MAX_QUADS of a
 * plan; 152, 76 and 36 on a GB300), so that the automatic choice can be
 * checked without a GPU.  Returns GEMM_F16_OK, or GEMM_F16_ERR_INVALID_ARG
 * for the arguments gemm_f16_run_info rejects, num_sms < 1, negative counts
 * or more clusters than the SMs hold.
 */
int gemm_f16_run_choice(int layout, int M, int N, int K, int64_t lda, int split_k,
                        int num_sms, int max_pairs, int max_quads, int info[4]);

/*
 * Host-only argument check used by gemm_f16_run (no device needed):
 * returns GEMM_F16_OK, GEMM_F16_ERR_INVALID_ARG or GEMM_F16_ERR_MISALIGNED.
 */
int gemm_f16_validate(int M, int N, int K, const void *A, int64_t lda,
                      const void *B, int64_t ldb, const void *C, int64_t ldc,
                      int split_k);

/* Host-only argument check used by gemm_f16_run_ex for `layout`. */
int gemm_f16_validate_ex(int layout, int M, int N, int K, const void *A,
                         int64_t lda, const void *B, int64_t ldb,
                         const void *C, int64_t ldc, int split_k);

/*
 * Host-only: the order in which output tiles of a tiles_m x tiles_n grid
 * are handed out (order 0 = Morton, 1 = row-major).  Writes up to `cap`
 * entries, each (tile_m | tile_n << 16), into `out` and returns the number
 * of tiles (tiles_m * tiles_n), or a negative error code.  tiles_m and
 * tiles_n must be in [1, 65535].
 */
int64_t gemm_f16_tile_order(int tiles_m, int tiles_n, int order,
                            uint32_t *out, int64_t cap);

/*
 * Host-only: the work list of the CTA-pair kernel with full tiles
 * `tile_width` columns wide (must be 256), for an M x N x K product with
 * `pairs` co-resident CTA pairs (see GEMM_F16_INFO_MAX_PAIRS).  Each entry
 * is (pair_row | col128 << 16 | log2(width/128) << 30): rows 256*pair_row ..
 * +255, columns 128*col128 .. +width-1.  Writes up to `cap` entries (`out`
 * may be NULL when cap is 0) and returns the count, or a negative error
 * code.  If `tail_parts` is not NULL it receives 2 when the last
 * (count % pairs) tiles run as two K halves each, else 1.  That happens with
 * split_k 1, 256-wide tiles, at least 32 k-blocks and a partial last wave
 * whose halves fit in one wave (a pair tile of half the width takes about as
 * long as a full one, a tile of half the k-blocks half as long): each half
 * covers a contiguous half of the k-blocks and stores FP32 values in the
 * plan's workspace, and a second kernel writes C = fp16_rn(P0 + P1), so the
 * result is deterministic (not bit-identical to a single pass).
 */
int64_t gemm_f16_pair_tiles(int M, int N, int K, int pairs, int split_k, int order,
                            int tile_width, uint32_t *out, int64_t cap, int *tail_parts);

/* Compile-time tile shape of the kernel: BM x BN output tile, BK k-block. */
int gemm_f16_tile_shape(int *bm, int *bn, int *bk, int *stages);

/*
 * gemm_f16_run_noalloc — the same product as gemm_f16_run, without a plan and
 * without allocating any memory.  (No counterpart in the paper: this is a
 * library convenience.)
 *
 * Who it is for: callers that must not call cudaMalloc/cudaFree, for example
 * code whose device memory is owned by another allocator (a framework's
 * caching pool that has reserved the free HBM, so a direct cudaMalloc can
 * fail), or latency-critical loops where the implicit device-wide
 * synchronisation of cudaMalloc/cudaFree would stall every other stream.
 * gemm_f16_plan allocates (status word, work lists, the split workspace),
 * so such callers cannot use it.
 *
 * Instead of plan-owned buffers this entry point uses one fixed scratch
 * array compiled into the library (a file-scope __device__ array), which
 * every GPU that loads the library holds until the process exits:
 *   GEMM_F16_NOALLOC_SCRATCH_BYTES bytes = a 256-byte status area plus
 *   GEMM_F16_NOALLOC_WS_BYTES of FP32 split partials.
 * The kernel computes each tile's position from its index, so nothing but
 * split partials is kept in the scratch between calls.
 * Limit: for split_k > 1, split_k * M * (N rounded up to 8) * 4 bytes <=
 * GEMM_F16_NOALLOC_WS_BYTES (32 MiB; e.g. 512 x 512 with 16 splits uses 16
 * MiB).  Larger problems return GEMM_F16_ERR_SCRATCH_TOO_SMALL and enqueue
 * nothing.  split_k = 1 uses no scratch beyond the status area.
 *
 * Arguments are those of gemm_f16_run (same validation and error codes),
 * plus `status`: a device-visible int the caller owns, into which the
 * kernel writes GEMM_F16_ERR_TIMEOUT if one of its bounded waits runs out
 * (it is never cleared by this call), or NULL.  With NULL the timeout goes
 * to the scratch's own status word, which only gemm_f16_noalloc_status
 * (below) reads: a caller that passes NULL and never calls it cannot learn
 * of a timeout, after which C is incomplete.  The device is the current
 * CUDA device.
 *
 * The first call on a device (of this function or of
 * gemm_f16_noalloc_status) does a one-time set-up with that device current
 * (shared-memory limit of the kernel, the scratch array's device address via
 * cudaGetSymbolAddress, SM count); make that first call before any stream
 * capture.  Every call shares the one scratch array and it keeps the last
 * call's contents: calls that overlap on the GPU (different streams, or
 * different host threads) race on the split partials and must not be
 * issued concurrently.
 */
#define GEMM_F16_NOALLOC_WS_BYTES (32u << 20)
#define GEMM_F16_NOALLOC_SCRATCH_BYTES (256u + GEMM_F16_NOALLOC_WS_BYTES)
int gemm_f16_run_noalloc(int M, int N, int K, const void *A, int64_t lda,
                         const void *B, int64_t ldb, void *C, int64_t ldc,
                         int split_k, int *status, gemm_f16_stream_t stream);

/*
 * Read and clear the scratch status word that gemm_f16_run_noalloc calls
 * given status == NULL write on the current device: returns 0 if none of
 * them timed out since the last read, GEMM_F16_ERR_TIMEOUT if one did, or a
 * negative error code of its own.  It copies 4 bytes with
 * cudaMemcpyFromSymbol (and clears them with cudaMemcpyToSymbol), which
 * allocates nothing but waits for the device's preceding work on the legacy
 * default stream; call it after the calls it should cover have finished
 * (e.g. after synchronising their stream).  No counterpart in the paper.
 */
int gemm_f16_noalloc_status(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H */
