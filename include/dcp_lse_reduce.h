/*
 * dcp_lse_reduce: the LSE-weighted merge of decode-context-parallel (DCP)
 * partial attention outputs, for MLA decode on one GB300 (sm_103a).
 *
 * The operation.
 *   Each of cp context shards j = 0..cp-1 holds a partial attention output
 *   S_j[B, H, D] and its log-sum-exp lse_j[B, H] (base 2 or base e). The
 *   destination r owns heads h in [r*H/cp, (r+1)*H/cp) and merges them:
 *       m       = max_j lse_j[b, h]
 *       w_j     = base^(lse_j[b, h] - m) / sum_k base^(lse_k[b, h] - m)
 *       dst_r[b, i, :]   = sum_j w_j * S_j[b, h, :]        (h = r*H/cp + i)
 *       lse_out_r[b, i]  = m + log_base(sum_k base^(lse_k[b, h] - m))
 *   Sources:
 *   - "[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE reduce"
 *     (sglang #40539), "Motivation" (the exchange is followed by an
 *     LSE-weighted merge) and "Modifications" (the [B, H, D] output is read
 *     in place as a strided [B, H/cp, cp, D] view, head h going to
 *     destination h // (H/cp); the LSE base comes from the attention
 *     backend); "Accuracy Tests" (FlashMLA's [B, H, 1] LSE).
 *   - "[Attention] Add direct symmetric-memory DCP A2A" (vLLM #48897), commit
 *     notes: FP32 LSE weighting for natural-log and base-2 LSEs, fp16 and
 *     bf16 outputs, CUTLASS-style padded token strides, and empty KV shards
 *     that publish LSE = -inf and are skipped by the combine.
 *   - "[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer
 *     memory" (sglang #32851), commit notes: exp(-inf) = 0 for a shard that
 *     owns no tokens; such rows must come out as 0, not NaN.
 *   On one GPU all cp shards are separate device buffers: the kernel reads
 *   them in place, with no pack step and no collective.
 *
 * Numerics. Weights and accumulation in fp32, sources taken in order
 * j = 0..cp-1, output rounded to bf16/fp16 (round to nearest even). A source
 * whose weight is 0 (LSE = -inf, or underflow) is never added, so a NaN
 * payload behind a -inf LSE does not leak. Whether its payload is read
 * depends on the schedule: the default one-(row, head)-per-warp schedule
 * issues every payload load together with the LSE loads (one memory round
 * trip) and drops zero-weight rows before the sum; DCP_FLAG_LSE_FIRST, and
 * seq_lens masking on grids of more than one resident wave, read the LSEs
 * first and never read a zero-weight payload. A (row, head) whose every
 * source is -inf gives an output of 0 and a merged LSE of -inf. The result
 * is bit-identical across calls, launch schedules and graph replays.
 *
 * Ownership. The caller owns every buffer; the library allocates nothing and
 * keeps no per-call state. Sources, LSEs and destinations must not alias.
 *
 * Asynchrony. A call only enqueues one kernel on `stream` (a cudaStream_t;
 * NULL = the legacy default stream of the calling thread's current device).
 * It never synchronises and never copies, so it can be captured in a CUDA
 * graph. The pointer arrays are read on the host during the call and copied
 * by value into the kernel's parameters; they may be freed on return.
 *
 * Errors. 0 on success. A negative DCP_ERR_* code means an argument was
 * rejected on the host and nothing was launched. A positive value is the
 * cudaError_t returned by the launch.
 */
#ifndef DCP_LSE_REDUCE_H
#define DCP_LSE_REDUCE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCP_LSE_REDUCE_CP_MAX 16
#define DCP_LSE_REDUCE_INTERLEAVE_MAX (1 << 24)

/* Element types of the partial outputs and of the merged output. */
#define DCP_DTYPE_BF16 0
#define DCP_DTYPE_F16 1

/* Flags for dcp_lse_reduce_ex. */
#define DCP_FLAG_PDL 1u        /* launch with programmatic dependent launch: the
                                  kernel may start while the previous kernel in
                                  the stream drains; it waits for that kernel's
                                  results before its first load */
#define DCP_FLAG_PRELOAD 2u    /* force the schedule that issues a head's payload
                                  loads together with its LSE loads (available
                                  for D = 512 and cp <= 8; ignored otherwise) */
#define DCP_FLAG_LSE_FIRST 4u  /* force the persistent schedule that reads the
                                  LSEs first and skips zero-weight payloads */
#define DCP_FLAG_PREFETCH 8u   /* each warp brings its first (row, head)'s inputs
                                  into L2 before it waits for the previous kernel
                                  (with DCP_FLAG_PDL: that wait overlaps the
                                  previous kernel's tail). A hint: the values read
                                  are the same; if the previous kernel writes these
                                  inputs, the prefetch only adds reads */

enum {
    DCP_OK = 0,
    DCP_ERR_NULL_POINTER = -1,  /* a required pointer (array or entry) is NULL */
    DCP_ERR_BAD_CP = -2,        /* cp < 1 or cp > DCP_LSE_REDUCE_CP_MAX */
    DCP_ERR_BAD_SHAPE = -3,     /* B < 0, H < 1, or D not a positive multiple of 8 */
    DCP_ERR_HEADS_NOT_DIVISIBLE = -4, /* H % cp != 0 */
    DCP_ERR_BAD_STRIDE = -5,    /* a negative stride, a payload stride that is not a
                                   multiple of 8 elements, or lse_stride < H */
    DCP_ERR_MISALIGNED = -6,    /* a payload pointer not 16-byte aligned, or an LSE
                                   pointer not 4-byte aligned */
    DCP_ERR_BAD_FLAGS = -7,     /* unknown flag bits, or PRELOAD with LSE_FIRST */
    DCP_ERR_BAD_DTYPE = -8,     /* dtype not DCP_DTYPE_BF16 / DCP_DTYPE_F16 */
    DCP_ERR_BAD_BASE = -9,      /* lse_base_e not 0 or 1 */
    DCP_ERR_DEVICE = -10,       /* the current device could not be queried */
    DCP_ERR_BAD_INTERLEAVE = -11 /* seq_lens given with interleave outside [1, 2^24] */
};

/*
 * The merge over contiguous buffers (the layout the pages use).
 *
 *   src_ptrs      host array of cp device pointers; src_ptrs[j] is source j's
 *                 partial output, [B, H, D] contiguous, bf16, 16-byte aligned.
 *   lse_ptrs      host array of cp device pointers; lse_ptrs[j] is source j's
 *                 LSE in fp32, element (b, h) at lse_ptrs[j][b*lse_stride + h]
 *                 ([B, H] and FlashMLA's [B, H, 1] both have lse_stride = H);
 *                 4-byte aligned.
 *   lse_stride    elements between LSE rows; must be >= H.
 *   cp            number of context shards = number of destinations, 1..16.
 *   B             batch rows (decode tokens); B = 0 is a no-op.
 *   H             total heads, a multiple of cp; destination r owns H/cp heads.
 *   D             head (latent) width in elements, a multiple of 8 (MLA: 512).
 *   lse_base_e    1: LSEs are natural logs; 0: base-2 logs. The merged LSE is
 *                 written in the same base.
 *   dst_ptrs      host array of cp device pointers; dst_ptrs[r] is
 *                 destination r's merged output, [B, H/cp, D] contiguous,
 *                 bf16, 16-byte aligned.
 *   lse_out_ptrs  host array of cp device pointers; lse_out_ptrs[r] is
 *                 destination r's merged LSE, [B, H/cp] contiguous fp32.
 *                 The array, or any entry, may be NULL: that LSE is not written.
 *   stream        cudaStream_t on the calling thread's current device.
 */
int dcp_lse_reduce(const void* const* src_ptrs, const float* const* lse_ptrs, int64_t lse_stride,
                   int cp, int64_t B, int H, int D, int lse_base_e,
                   void* const* dst_ptrs, float* const* lse_out_ptrs, void* stream);

/*
 * Strides (in elements) for dcp_lse_reduce_ex. Element (b, h, d) of source j
 * is src_ptrs[j][b*src_row + h*src_head + d]; LSE (b, h) of source j is
 * lse_ptrs[j][b*lse_row + h*lse_head]; element (b, i, d) of destination r is
 * dst_ptrs[r][b*dst_row + i*dst_head + d]; merged LSE (b, i) of destination r
 * is lse_out_ptrs[r][b*lse_out_row + i]. Payload strides must be multiples of
 * 8 elements (16 bytes); all strides must be >= 0.
 */
typedef struct dcp_lse_reduce_layout {
    int64_t src_row, src_head;
    int64_t lse_row, lse_head;
    int64_t dst_row, dst_head;
    int64_t lse_out_row;
} dcp_lse_reduce_layout;

/*
 * The same merge with explicit strides (padded token strides, heads taken from
 * a wider backing array, FlashMLA-style LSE head strides), a dtype
 * (DCP_DTYPE_BF16 or DCP_DTYPE_F16; the output has the input's type),
 * optional masking of empty shards from the rows' context lengths, and launch
 * flags (DCP_FLAG_*). layout = NULL means contiguous buffers with lse_row = H.
 *
 *   seq_lens    NULL, or a device array of B int32 context lengths (4-byte
 *               aligned). The KV of a row is interleaved over the cp shards in
 *               blocks of `interleave` tokens (token t lives on shard
 *               (t / interleave) % cp), so shard j owns a token of a context
 *               of L tokens iff L > j*interleave. A shard that owns none is
 *               empty for that row: its LSE entry is ignored (it may hold
 *               anything) and its payload is never added (nor read, under
 *               the schedule that reads LSEs first; see Numerics). L = 0
 *               gives an output of 0 and a merged LSE of -inf.
 *   interleave  tokens per interleave block, 1..DCP_LSE_REDUCE_INTERLEAVE_MAX
 *               (read only when seq_lens is given).
 *
 * Sources: the pages cited above; "[Attention] Add direct symmetric-memory DCP
 * A2A" (vLLM #48897) commit notes on padded token strides, non-contiguous head
 * storage, fp16/bf16 outputs, and empty-KV-shard masking from the decode
 * seq_lens; "[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer
 * memory" (sglang #32851) commit notes on the KV interleaved across DCP ranks.
 */
int dcp_lse_reduce_ex(const void* const* src_ptrs, const float* const* lse_ptrs,
                      int cp, int64_t B, int H, int D, int lse_base_e, int dtype,
                      void* const* dst_ptrs, float* const* lse_out_ptrs,
                      const dcp_lse_reduce_layout* layout, const int32_t* seq_lens, int interleave,
                      unsigned flags, void* stream);

/* A static, human-readable message for a status code. */
const char* dcp_lse_reduce_strerror(int status);

/* Library version: major*10000 + minor*100 + patch. */
int dcp_lse_reduce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DCP_LSE_REDUCE_H */
