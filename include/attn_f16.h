/*
 * attn_f16 — scaled dot-product attention forward, head dimension 256, for
 * GB300 (sm_103a).  C ABI, plain pointers and sizes.
 *
 * What it computes, per batch b, head h and query row i:
 *
 *     O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) * V[b,h,j,:]
 *
 * with binary16 Q, K, V, O, FP32 scores, softmax statistics and
 * accumulation, and O rounded to binary16 (round to nearest even).  This is
 * the flash-attention ("SDP") kernel of the "Xe2 Nbarrier Pipelining" page,
 * section "Proven Pattern: SDP Kernel Split Barrier B" (head dimension 256):
 * per block of 64 keys, S = Q K^T, a softmax with a running row maximum,
 * P written to shared memory, then — across the split barrier — the sum
 * update and the next copies while the P V product waits for P.  The page
 * states no mask, so none is applied (every query attends to every key).
 *
 * Uses a gemm_f16 plan (include/gemm_f16.h) for its device, status word
 * and the options GEMM_F16_OPT_TIMEOUT_NS and GEMM_F16_OPT_FAULT_UNIT (here:
 * for the single-CTA kernel the linear index x + gx*(y + gy*z) of the CTA
 * whose first key tile gets no copy, for the CTA-pair kernel the work unit
 * (item * ranges + range) whose first key tile gets no copy from the
 * leader; for the timeout test).  Errors found on the device are reported
 * later by gemm_f16_status.
 */
#ifndef ATTN_F16_H
#define ATTN_F16_H

#include <stdint.h>

#include "gemm_f16.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Head dimension the kernel supports. */
#define ATTN_F16_HEAD_DIM 256

/*
 * Enqueue the attention forward pass on `stream` (asynchronous).
 *   batch, heads      >= 1 and <= 65535 each.
 *   seq_q, seq_kv     >= 1 (query rows, key/value rows per head).
 *   head_dim          must be ATTN_F16_HEAD_DIM (256).
 *   Q, K, V, O        device pointers to binary16, 16-byte aligned; element
 *                     (b, h, i, d) of X is at X[b*xs[0] + h*xs[1] + i*xs[2] + d]
 *                     (d contiguous).  The strides xs[0..2] are in elements,
 *                     positive multiples of 8, with xs[2] >= 256; a stride
 *                     of a dimension of extent 1 is not used.  So both
 *                     [batch, head, seq, 256] and [batch, seq, head, 256]
 *                     storage work.  O is written (every row of every head)
 *                     and must not overlap Q, K or V.
 *   scale             finite; usually 1/sqrt(256) = 0.0625.
 * Returns GEMM_F16_OK, GEMM_F16_ERR_INVALID_ARG (sizes, strides, scale,
 * null pointers), GEMM_F16_ERR_MISALIGNED (pointer or stride alignment) or
 * GEMM_F16_ERR_CUDA (encode or launch failure) or GEMM_F16_ERR_OOM;
 * nothing is enqueued on an error.  Without a key split the call allocates
 * nothing; with one (GEMM_F16_OPT_ATTN_SPLIT, automatic when the
 * (batch, head, 256-row) items are too few to fill the GPU) the CTA-pair
 * kernel writes each key range's normalised FP32 partial of O (256 KB per
 * 256 rows and range) and its row offsets and sums into the plan's
 * workspace, which grows on the stream as needed (as for split GEMM runs),
 * and a second kernel merges the ranges into O.
 */
int attn_f16_fwd(gemm_f16_plan_t plan, int batch, int heads, int seq_q, int seq_kv,
                 int head_dim, const void *Q, const int64_t q_strides[3],
                 const void *K, const int64_t k_strides[3], const void *V,
                 const int64_t v_strides[3], void *O, const int64_t o_strides[3],
                 float scale, gemm_f16_stream_t stream);

/*
 * The same forward pass with HOST operands: hQ [batch, heads, seq_q, 256],
 * hK and hV [batch, heads, seq_kv, 256], hO [batch, heads, seq_q, 256], all
 * contiguous binary16 in host memory (pinned memory gives asynchronous
 * copies).  Q, K, V are copied into one of two plan-owned sets of device
 * buffers on a plan-internal stream, the pass runs on `stream` once they
 * have arrived, and O is copied back on `stream`; consecutive calls
 * alternate the two sets, so one call's input copies overlap the previous
 * call's pass and output copy.  hQ, hK, hV must therefore be ready when the
 * call is made; synchronise `stream` before reading hO or reusing the
 * inputs.  A set grows (after a device synchronisation) when a call needs
 * more room than it has.  Calls on different streams must be ordered by
 * the caller, as for every use of a plan (one pass at a time); the plan
 * orders its own input copies after the output copy of the call that last
 * used the same set, whatever stream that call ran on.  Returns the codes
 * of attn_f16_fwd (the sizes and scale are checked as there; null host
 * pointers give GEMM_F16_ERR_INVALID_ARG).
 */
int attn_f16_fwd_host(gemm_f16_plan_t plan, int batch, int heads, int seq_q, int seq_kv,
                      int head_dim, const void *hQ, const void *hK, const void *hV, void *hO,
                      float scale, gemm_f16_stream_t stream);

/*
 * The number of key ranges attn_f16_fwd would cut each item's keys into for
 * these sizes with this plan's current options (1: no split, one kernel
 * launch; n > 1: the CTA-pair kernel plus the merging kernel).  Enqueues
 * nothing.  Returns GEMM_F16_OK or GEMM_F16_ERR_INVALID_ARG (null pointers,
 * sizes < 1).
 */
int attn_f16_key_ranges(gemm_f16_plan_t plan, int batch, int heads, int seq_q, int seq_kv,
                        int *ranges);

/* Host-only argument check used by attn_f16_fwd (no device needed). */
int attn_f16_validate(int batch, int heads, int seq_q, int seq_kv, int head_dim,
                      const void *Q, const int64_t q_strides[3], const void *K,
                      const int64_t k_strides[3], const void *V,
                      const int64_t v_strides[3], const void *O,
                      const int64_t o_strides[3], float scale);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_F16_H */
