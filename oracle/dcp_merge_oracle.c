/*
 * CPU oracle for the decode-context-parallel (DCP) LSE-weighted merge.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, fp64 statement of
 * what the merge computes. It is loaded by the tests, by the smoke check and
 * by the benchmark's CPU-baseline leg, and by nothing else. It shares no code,
 * header or table with the CUDA library.
 *
 * What it follows:
 *  - "[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE reduce"
 *    (sglang #40539), "Motivation": after the exchange, the head partials are
 *    combined by an LSE-weighted merge. "Modifications": the [B, H, D]
 *    attention output is viewed as [B, H/cp, cp, D] and its LSE as
 *    [B, H/cp, cp]; head h goes to destination h // (H/cp); the LSE base
 *    (2 or e) comes from the attention backend. "Accuracy Tests": FlashMLA's
 *    [B, H, 1] LSE layout.
 *  - "[Attention] Add direct symmetric-memory DCP A2A" (vLLM #48897), commit
 *    notes: received states are combined with FP32 LSE weighting, for
 *    natural-log and base-2 LSEs, fp16 and bf16 outputs; an empty KV shard
 *    publishes LSE = -inf and the combine skips zero-weight sources.
 *  - "[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer memory"
 *    (sglang #32851), commit notes: a shard that owns no tokens contributes
 *    exp(-inf) = 0, and such rows must come out as 0, not NaN.
 *
 * The formula itself (the pages name the merge but do not print it) is the
 * standard split-softmax merge. For destination r, row b and local head
 * i (global head h = r*H/cp + i), with L_j = lse_j[b, h] in natural-log units:
 *     m     = max_j L_j
 *     w_j   = exp(L_j - m) / sum_k exp(L_k - m)
 *     out   = sum_j w_j * S_j[b, h, :]
 *     lse   = m + log(sum_k exp(L_k - m))          (returned in the input base)
 * Readings where the pages are silent: a source whose L_j is -inf has weight
 * exactly 0 and its payload is never read (it may hold NaN); when every
 * source is -inf the output is 0 and the merged LSE is -inf.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_CP_MAX 64

enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F64 = 2 };
enum { ORACLE_LSE_F32 = 0, ORACLE_LSE_F64 = 1 };

/* bfloat16 is the upper half of an IEEE binary32: widen by appending 16 zero
 * bits. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
    }
    return sign ? -mag : mag;
}

static double load_value(int dtype, const void* base, int64_t idx) {
    if (dtype == ORACLE_BF16) return bf16_to_double(((const uint16_t*)base)[idx]);
    if (dtype == ORACLE_F16) return f16_to_double(((const uint16_t*)base)[idx]);
    return ((const double*)base)[idx];
}

static double load_lse(int lse_dtype, const void* base, int64_t idx) {
    if (lse_dtype == ORACLE_LSE_F32) return (double)((const float*)base)[idx];
    return ((const double*)base)[idx];
}

/*
 * Does source (shard) j own any token of a context of `len` tokens? The KV
 * cache is interleaved over the cp shards in blocks of `interleave` tokens:
 * token t belongs to shard (t / interleave) % cp ("[DCP] Optimize shared
 * Output, Query, and Indexer/Top-K via peer memory", commit notes: the latent
 * KV stays interleaved across DCP ranks). Counted token by token.
 */
static int shard_owns_tokens(int64_t len, int j, int cp, int interleave) {
    for (int64_t t = 0; t < len; ++t) {
        if ((t / interleave) % cp == j) return 1; /* found one owned token */
    }
    return 0;
}

/*
 * Merge cp partial outputs for every destination r in [0, cp).
 *
 *   src[j]      source j's partial output, element (b, h, d) at
 *               b*src_row + h*src_head + d  (elements of `dtype`)
 *   lse[j]      source j's LSE, element (b, h) at b*lse_row + h*lse_head
 *   out[r]      destination r's merged output, fp64, element (b, i, d) at
 *               (b*(H/cp) + i)*D + d
 *   lse_out[r]  destination r's merged LSE, fp64, element (b, i) at
 *               b*(H/cp) + i; may be NULL
 *   seq_lens    optional (NULL = no masking): context length of each row. A
 *               source that owns no token of row b's context is empty for
 *               that row: its LSE entry is ignored and it gets weight 0
 *               ("[Attention] Add direct symmetric-memory DCP A2A", commit
 *               notes: the combine masks empty-KV-shard rows given the decode
 *               seq_lens).
 *   interleave  tokens per interleave block (>= 1), used with seq_lens.
 *
 * Returns 0, or -1 on an argument the oracle does not take.
 */
int oracle_dcp_merge(int dtype, const void* const* src, int64_t src_row, int64_t src_head,
                     int lse_dtype, const void* const* lse, int64_t lse_row, int64_t lse_head,
                     int cp, int64_t B, int H, int D, int lse_base_e,
                     const int32_t* seq_lens, int interleave,
                     double* const* out, double* const* lse_out) {
    if (cp < 1 || cp > ORACLE_CP_MAX || B < 0 || H < 1 || D < 1 || H % cp != 0) return -1;
    if (seq_lens && interleave < 1) return -1;
    if (dtype < ORACLE_BF16 || dtype > ORACLE_F64) return -1;
    if (lse_dtype != ORACLE_LSE_F32 && lse_dtype != ORACLE_LSE_F64) return -1;
    const int Hl = H / cp;
    const double to_e = lse_base_e ? 1.0 : log(2.0); /* log b -> natural log */

    for (int r = 0; r < cp; ++r) {
        for (int64_t b = 0; b < B; ++b) {
            for (int i = 0; i < Hl; ++i) {
                const int h = r * Hl + i; /* head h belongs to destination h / Hl */
                double L[ORACLE_CP_MAX];
                double m = -INFINITY;
                for (int j = 0; j < cp; ++j) {
                    if (seq_lens && !shard_owns_tokens(seq_lens[b], j, cp, interleave)) {
                        L[j] = -INFINITY; /* empty shard: its LSE entry is not read */
                    } else {
                        L[j] = load_lse(lse_dtype, lse[j], b * lse_row + (int64_t)h * lse_head) * to_e;
                    }
                    if (L[j] > m) m = L[j];
                }
                double* o = out[r] + (b * Hl + i) * (int64_t)D;
                if (m == -INFINITY) { /* no source holds any token */
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    if (lse_out && lse_out[r]) lse_out[r][b * Hl + i] = -INFINITY;
                    continue;
                }
                double w[ORACLE_CP_MAX];
                double s = 0.0;
                for (int j = 0; j < cp; ++j) {
                    w[j] = (L[j] == -INFINITY) ? 0.0 : exp(L[j] - m);
                    s += w[j];
                }
                for (int j = 0; j < cp; ++j) w[j] /= s;
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int j = 0; j < cp; ++j) {
                        if (w[j] == 0.0) continue; /* zero-weight source: payload not read */
                        acc += w[j] * load_value(dtype, src[j], b * src_row + (int64_t)h * src_head + d);
                    }
                    o[d] = acc;
                }
                if (lse_out && lse_out[r]) lse_out[r][b * Hl + i] = (m + log(s)) / to_e;
            }
        }
    }
    return 0;
}

/* Conversion of one 16-bit pattern, exposed so that the tests can pin it. */
double oracle_half_bits_to_double(int dtype, uint16_t bits) {
    return dtype == ORACLE_F16 ? f16_to_double(bits) : bf16_to_double(bits);
}

int oracle_version(void) { return 1; }
