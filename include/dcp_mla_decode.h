/*
 * dcp_mla_decode_partial: the producer of the DCP partials — MLA decode
 * attention of every query head over the tokens one context shard holds,
 * split into up to 16 contiguous token ranges, each giving a partial output
 * and its log-sum-exp. Their LSE-weighted merge (dcp_lse_reduce) is attention
 * over the whole context.
 *
 * The operation. For row b, head h and split s over the shard's first
 * kv_len[b] tokens (split s holds tokens [s*c, min((s+1)*c, kv_len[b])),
 * c = ceil(kv_len[b] / n_split)):
 *     s_t      = scale * <q[b, h, :Dk], kv[b, t, :Dk]>
 *     out_s[b, h, :] = sum_t softmax(s)_t * kv[b, t, :Dv]     (value = first Dv dims)
 *     lse_s[b, h]    = log_base sum_t exp(s_t)
 *   An empty range gives out = 0 and lse = -inf.
 *   Sources:
 *   - "[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer memory"
 *     (sglang #32851), commit notes: under DCP each rank holds an interleaved
 *     share of the latent KV, computes decode attention over the tokens it
 *     owns and returns a partial output with its LSE (trtllm-gen surfaces a
 *     base-2 LSE); attention is invariant under permuting the tokens, so any
 *     split merges back exactly.
 *   - "[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE reduce"
 *     (sglang #40539), "Speed Tests and Profiling": MLA decode with a 512-wide
 *     latent (kv_lora_rank), 16 heads per rank; "Accuracy Tests": FlashMLA's
 *     base-e LSE.
 *   MLA's absorbed form attends with keys of 512 latent + 64 RoPE dims
 *   (Dk = 576) and values of the 512 latent dims (Dv = 512) of the same
 *   cached row; Dk = 512 (no RoPE part) is also taken.
 *
 * Numerics. bf16 inputs, fp32 scores and accumulation (tensor-core MMA),
 * softmax in base 2 with the running maximum taken out, probabilities rounded
 * to bf16 for the value product, output rounded to bf16 (round to nearest
 * even), LSE fp32 in the requested base. Two kernels compute it: one on the
 * 5th-generation tensor cores (tcgen05 MMA into TMEM, operands loaded by TMA)
 * and one on warp-level mma.sync (see DCP_MLA_FLAG_*); they agree within the
 * stated tolerances, not bit for bit.
 *
 * Layout (all contiguous, device memory, caller-owned):
 *   q        [B, H, Dk] bf16, 16-byte aligned
 *   kv       [B, T, Dk] bf16, 16-byte aligned: row b's shard-local tokens
 *   kv_len   [B] int32: tokens of row b held by this shard (clamped to [0, T])
 *   out_ptrs host array of n_split device pointers, each [B, H, Dv] bf16,
 *            16-byte aligned
 *   lse_ptrs host array of n_split device pointers, each [B, H] fp32
 *   status   NULL, or a device int32 the kernel ORs 1 into if a wait for its
 *            own asynchronous copies or MMAs ever exceeds two seconds (20 ms
 *            with DCP_MLA_FLAG_TEST_STALL). Then
 *            the CTA stops issuing copies and MMAs, leaves at the next tile
 *            boundary without writing its outputs (they are not valid), waits
 *            (again at most two seconds each) for what it had issued, frees
 *            its tensor memory and exits: it never hangs.
 *
 * Asynchrony, ownership, errors: as for dcp_lse_reduce (one kernel enqueued
 * on `stream`, nothing allocated, graph-capturable; negative codes are host
 * argument errors with nothing launched, positive codes are cudaError_t).
 */
#ifndef DCP_MLA_DECODE_H
#define DCP_MLA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCP_MLA_SPLIT_MAX 16

enum {
    DCP_MLA_ERR_NULL_POINTER = -101, /* q, kv, kv_len, out_ptrs, lse_ptrs or an entry is NULL */
    DCP_MLA_ERR_BAD_SHAPE = -102,    /* B outside [0, 65535], T < 0, H not a positive multiple of 16,
                                        Dk not 512 or 576, or Dv not 512 */
    DCP_MLA_ERR_BAD_SPLIT = -103,    /* n_split outside [1, DCP_MLA_SPLIT_MAX] */
    DCP_MLA_ERR_MISALIGNED = -104,   /* q, kv or an output not 16-byte aligned, or an LSE or kv_len
                                        pointer not 4-byte aligned */
    DCP_MLA_ERR_BAD_FLAGS = -105,    /* unknown flag bits (DCP_FLAG_PDL, DCP_FLAG_PREFETCH and the flags
                                        below are known; DCP_MLA_FLAG_ONE_KERNEL only by dcp_mla_decode),
                                        or both DCP_MLA_FLAG_MMA_SYNC and DCP_MLA_FLAG_TCGEN05 */
    DCP_MLA_ERR_WORKSPACE = -106,    /* workspace NULL, not 256-byte aligned, or smaller than
                                        dcp_mla_decode_workspace_bytes(...) */
    DCP_MLA_ERR_BAD_CP = -107,       /* cp < 1, cp*n_split > 16, or H not a multiple of cp*n_split */
    DCP_MLA_ERR_SCRATCH_LIMIT = -108, /* dcp_mla_decode_noalloc: the partials need more than
                                         DCP_MLA_NOALLOC_SCRATCH_BYTES */
    DCP_MLA_ERR_SCRATCH_SETUP = -109, /* dcp_mla_decode_noalloc: the scratch array's device address
                                         could not be obtained on the current device */
    DCP_MLA_ERR_TENSOR_MAP = -110     /* a TMA tensor map for q or a cache could not be encoded */
};

/*
 * Flags of the producer and the fused decode (besides DCP_FLAG_PDL = 1). By
 * default the producer runs the tcgen05 kernel (TMEM accumulators, TMA loads)
 * when H is a multiple of 64 and a split holds at least 128 tokens of the
 * cache (ceil(T / n_split) >= 128), or H is a multiple of 32 and a split
 * holds at least 256; otherwise the warp-level mma.sync kernel. These flags
 * force one. Both compute the same partials within the stated tolerances.
 */
#define DCP_MLA_FLAG_MMA_SYNC 2u
#define DCP_MLA_FLAG_TCGEN05 4u
/*
 * dcp_mla_decode only: run the merge inside the producer's launch where the
 * tcgen05 grid fits one wave (see dcp_mla_decode). Slower on GB300 than the
 * default two launches with PDL, so off by default.
 */
#define DCP_MLA_FLAG_ONE_KERNEL 16u
/*
 * For tests of the bounded waits only: every CTA arms the barrier of its
 * first KV tile for 16 bytes more than its copies deliver, so that wait never
 * completes, and every wait of the call gives up after 20 ms instead of two
 * seconds. The call then follows the protocol described under `status`: the
 * status word reads 1 when the call has run on its stream, the outputs are not
 * valid (dcp_mla_decode still merges them), and the kernel exits after about
 * 40 ms per wave of CTAs, leaving the context usable. A CTA whose split holds
 * no token writes its zero output and never waits.
 */
#define DCP_MLA_FLAG_TEST_STALL 32u
/*
 * DCP_FLAG_PREFETCH (8, include/dcp_lse_reduce.h) is also taken by the
 * producer: each CTA of the tcgen05 kernel brings Q and its split's first KV
 * tile into L2 before it waits for the previous kernel (with DCP_FLAG_PDL that
 * wait overlaps the previous kernel's tail). A hint: results are the same.
 * dcp_mla_decode passes it to the producer only, not to its merge (whose
 * inputs the producer has just written).
 */

int dcp_mla_decode_partial(const void* q, const void* kv, const int32_t* kv_len,
                           int64_t B, int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e,
                           int n_split, void* const* out_ptrs, float* const* lse_ptrs,
                           int32_t* status, unsigned flags, void* stream);

/*
 * Dynamic shared memory one CTA of the producer may use for Dk and H (bytes):
 * the larger of the two kernels' needs. -1 for Dk not 512 or 576, or H not a
 * positive multiple of 16.
 */
int dcp_mla_decode_smem_bytes(int Dk, int H);

/*
 * Which kernel dcp_mla_decode_partial (and dcp_mla_decode, per shard) runs
 * for H heads, T cache tokens per row, n_split splits and these flags:
 * DCP_MLA_KERNEL_TCGEN05 or DCP_MLA_KERNEL_MMA_SYNC. Host only; launches
 * nothing. Returns DCP_MLA_ERR_BAD_SHAPE (H not a positive multiple of 16,
 * T < 0), DCP_MLA_ERR_BAD_SPLIT or DCP_MLA_ERR_BAD_FLAGS for arguments the
 * producer would reject for those reasons.
 */
#define DCP_MLA_KERNEL_TCGEN05 1
#define DCP_MLA_KERNEL_MMA_SYNC 2
int dcp_mla_decode_kernel(int H, int64_t T, int n_split, unsigned flags);

/*
 * A split count for cp shards of B rows, H heads and T cache tokens per row on
 * a GPU with num_sms multiprocessors (cudaDevAttrMultiProcessorCount): the
 * largest n_split with cp*n_split <= DCP_MLA_SPLIT_MAX whose producer launch
 * (cp * n_split * head blocks * B CTAs; one per SM for the tcgen05 kernel, as
 * many as fit for the mma.sync kernel) fits in one wave, whose
 * splits hold at least one 128-token tile (ceil(T / n_split) >= 128), and
 * with H a multiple of cp*n_split (as dcp_mla_decode needs); 1 when no larger
 * count qualifies. Use cp = 1 for a single dcp_mla_decode_partial call. Host
 * only; DCP_MLA_ERR_BAD_SHAPE or DCP_MLA_ERR_BAD_CP for invalid arguments.
 */
int dcp_mla_decode_pick_split(int cp, int64_t B, int H, int64_t T, int num_sms);

/*
 * Bytes of caller-provided workspace dcp_mla_decode needs: the cp*n_split
 * partial outputs ([B, H, Dv] bf16 each) and LSEs ([B, H] fp32 each).
 * Returns -1 for a negative or overflowing size.
 */
int64_t dcp_mla_decode_workspace_bytes(int cp, int n_split, int64_t B, int H, int Dv);

/*
 * DCP decode attention on one GPU: dcp_mla_decode_partial over each of cp
 * context shards (kv_ptrs[j], kv_len_ptrs[j]: shard j's [B, T, Dk] cache and
 * [B] token counts, each row's tokens split into n_split ranges), then the
 * LSE-weighted merge (dcp_lse_reduce) of all cp*n_split partials, in which
 * destination r receives heads [r*H/cp, (r+1)*H/cp):
 *   dst_ptrs[r]      [B, H/cp, Dv] bf16, 16-byte aligned
 *   lse_out_ptrs     NULL, or cp pointers to [B, H/cp] fp32 merged LSEs (an
 *                    entry may be NULL)
 *   workspace        device memory of at least
 *                    dcp_mla_decode_workspace_bytes(cp, n_split, B, H, Dv)
 *                    bytes, 256-byte aligned, owned by the caller; its
 *                    contents on entry do not matter. Calls that share a
 *                    workspace must be ordered (one stream, or events).
 * The result is attention over every row's whole context (the union of the
 * shards' tokens): "[DCP] Optimize shared Output, Query, and Indexer/Top-K via
 * peer memory" (sglang #32851), commit notes on the interleaved KV shards and
 * the cross-rank combine; on one GPU the shards are local buffers and the
 * exchange is the merge's strided read. The producer kernel is the one
 * dcp_mla_decode_kernel(H, T, n_split, flags) names, in one launch covering
 * every shard and split.
 *   - By default the merge is a second launch (PDL between the two with
 *     DCP_FLAG_PDL).
 *   - With DCP_MLA_FLAG_ONE_KERNEL, when the producer is the tcgen05 kernel
 *     and its grid (cp * n_split * head blocks * B CTAs) fits in one resident
 *     wave, the merge runs in the same launch instead: a cooperative launch,
 *     in which every CTA writes its partial to the workspace, the grid
 *     synchronises once, and every warp then merges (row, head) units into
 *     the destinations. On GB300 this measured slower than the two launches
 *     (the cooperative launch and the grid-wide sync cost more than the
 *     second launch and its gap under PDL); it is kept for comparison.
 *   Both give bit-identical results (the same arithmetic in the same order).
 * Constraints: cp*n_split <= 16 and H a multiple of cp*n_split and of 16;
 * dst_ptrs 16-byte and lse_out_ptrs 4-byte aligned (DCP_MLA_ERR_MISALIGNED).
 */
int dcp_mla_decode(const void* q, const void* const* kv_ptrs, const int32_t* const* kv_len_ptrs, int cp,
                   int64_t B, int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e, int n_split,
                   void* workspace, int64_t workspace_bytes, void* const* dst_ptrs, float* const* lse_out_ptrs,
                   int32_t* status, unsigned flags, void* stream);

/*
 * Capacity of the library's built-in scratch array used by
 * dcp_mla_decode_noalloc (bytes): 32 MiB.
 */
#define DCP_MLA_NOALLOC_SCRATCH_BYTES (32 << 20)

/*
 * dcp_mla_decode without a workspace argument, for callers that cannot
 * allocate device memory when they run the decode: for instance code inside a
 * host process whose device memory is fully reserved by another allocator at
 * start-up, plug-in or embedded runtimes that forbid allocation after
 * initialisation, or latency-critical paths that cannot afford cudaMalloc's
 * implicit device synchronisation. (The pages this library follows have no
 * counterpart to this call; it is a deployment convenience.)
 *
 * The partial outputs and LSEs live in one scratch array of
 * DCP_MLA_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits. Arguments and
 * results are as for dcp_mla_decode; the call needs
 * dcp_mla_decode_workspace_bytes(cp, n_split, B, H, Dv) <=
 * DCP_MLA_NOALLOC_SCRATCH_BYTES, else it returns DCP_MLA_ERR_SCRATCH_LIMIT
 * and enqueues nothing. It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 * The first call on a device looks up the array's device address on that
 * device (the calling thread's current device) and keeps it; make that first
 * call outside any stream capture. The array becomes resident on a device
 * when the library's code is loaded there, which under CUDA's default lazy
 * module loading can be this first call (or the first call of any producer
 * entry point): that is when the 32 MiB are committed, and if the device has
 * no free memory left by then the call returns DCP_MLA_ERR_SCRATCH_SETUP. So
 * make one warm-up call per device during initialisation, before other
 * allocators reserve the device's memory; a call with B = 0 and otherwise
 * valid arguments launches nothing and does only this set-up. Argument errors
 * are reported as by dcp_mla_decode (a bad shape as DCP_MLA_ERR_BAD_SHAPE)
 * before the scratch limit is checked. The array is shared by every call on a
 * device and keeps the last call's contents (nothing in it has to start at
 * zero); calls whose work overlaps on the GPU — on different streams without
 * ordering between them — race on it and give undefined results.
 */
int dcp_mla_decode_noalloc(const void* q, const void* const* kv_ptrs, const int32_t* const* kv_len_ptrs, int cp,
                           int64_t B, int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e, int n_split,
                           void* const* dst_ptrs, float* const* lse_out_ptrs, int32_t* status, unsigned flags,
                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DCP_MLA_DECODE_H */
