// LSE-weighted merge of DCP partial attention outputs, sm_103a.
//
// What it computes is stated in include/dcp_lse_reduce.h, with the passages it
// follows ("[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE reduce",
// "Modifications"; "[Attention] Add direct symmetric-memory DCP A2A", commit
// notes; "[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer
// memory", commit notes).
//
// Design. The merge is a pure HBM stream: per (row, head) it reads cp rows of
// D = 512 bf16 (1 KiB each) and cp LSEs, and writes 1 KiB plus one LSE, at
// about 1 flop per byte. There is no contraction, so no tensor cores. One warp
// owns one (row, head) "unit" at a time:
//   * every lane reads the cp LSEs (warp-uniform broadcast loads), so every
//     lane holds the weights without shuffles, and the fp32 sum over sources
//     runs in a fixed order;
//   * each lane moves two 16-byte vectors per source (lane*16 and 512 +
//     lane*16 bytes), so a warp's load of one source row is two fully
//     coalesced 512-byte requests, with 2*cp of them in flight per lane;
//   * stores are 16-byte vectors of packed bf16 (round to nearest even).
// The (row, head) units are walked in source order, so each source is read
// front to back. Head h of row b goes to destination r = h / (H/cp), slot
// i = h % (H/cp): the [B, H/cp, cp, D] strided view, with no pack step.
//
// Two schedules, chosen per call:
//   PRELOAD    one unit per warp; the payload loads are issued together with
//              the LSE loads (one memory round trip), in as many waves of CTAs
//              as the batch needs. The default for D = 512 and cp <= 8.
//   LSE_FIRST  persistent grid (one wave of CTAs); a warp strides over units,
//              reads the next unit's LSEs while the current payload is in
//              flight, and issues payload loads only for sources of nonzero
//              weight, so empty shards cost no payload bytes. Used for other
//              shapes, and with seq_lens masking when the grid would not fit
//              in one resident wave.
// Both give bit-identical results.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "dcp_lse_reduce.h"
#include "dcp_mla_decode.h"

namespace {

constexpr int kCpMax = DCP_LSE_REDUCE_CP_MAX;
constexpr int kMaxThreads = 128;      // CTAs of 2 or 4 warps, chosen per launch
constexpr int kVpl = 2;               // 16-byte vectors per lane per pass (64 chunks = 512 bf16)
constexpr int kChunksPerPass = 32 * kVpl;
constexpr int kMaxUnitsPerLaunch = 1 << 30;  // larger batches run as several launches

// Kernel parameters, sized for at most kMaxCp sources. The scalars a warp needs
// before its first load come first.
template <int kMaxCp>
struct Params {
    int units;                    // (row, head) pairs in this launch: rows * H
    int H, Hl, cp, D;
    int step;                     // warps in the grid = stride between a warp's units
    int step_b, step_r, step_i;   // step = step_b*H + step_r*Hl + step_i, step_r < cp, step_i < Hl
    float lse_scale;              // turns LSE differences into log2 units: 1 or log2(e)
    float log_scale;              // turns log2(sum) into the LSE base: 1 or ln(2)
    int interleave;               // KV tokens per interleave block (with seq_lens)
    int prefetch_first;           // 1: warm L2 with the first unit's inputs before the dependency wait
    const int* seq_lens;          // per-row context length, or null: no masking
    int64_t lse_row, lse_head;    // elements
    int64_t src_row, src_head;    // elements
    int64_t dst_row, dst_head;    // elements
    int64_t lse_out_row;          // elements
    const float* lse[kMaxCp];
    const uint8_t* src[kMaxCp];
    uint8_t* dst[kMaxCp];
    float* lse_out[kMaxCp];
};

// Position of a unit: row b, destination r, local head i (global head r*Hl + i).
struct Pos {
    int b, r, i;
};

template <int kMaxCp>
__device__ __forceinline__ Pos unit_pos(const Params<kMaxCp>& p, int u) {
    Pos q;
    q.b = (int)((unsigned)u / (unsigned)p.H);
    const int h = u - q.b * p.H;
    q.r = (int)((unsigned)h / (unsigned)p.Hl);
    q.i = h - q.r * p.Hl;
    return q;
}

// The unit `step` further on, by carries instead of divisions.
template <int kMaxCp>
__device__ __forceinline__ Pos advance(const Params<kMaxCp>& p, Pos q) {
    q.b += p.step_b;
    q.r += p.step_r;
    q.i += p.step_i;
    if (q.i >= p.Hl) {
        q.i -= p.Hl;
        q.r += 1;
    }
    if (q.r >= p.cp) {
        q.r -= p.cp;
        q.b += 1;
    }
    return q;
}

// ---- PTX helpers -------------------------------------------------------------

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Streaming 16-byte load through the read-only path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const uint8_t* ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ float ld_nc_f32(const float* ptr) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

__device__ __forceinline__ int ld_nc_s32(const int* ptr) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

// L2 prefetches: hints with no effect on the values later loads return. The
// bulk form covers `bytes` (a multiple of 16) from a 16-byte aligned address.
__device__ __forceinline__ void prefetch_l2_bulk(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2_line(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr) : "memory");
}

__device__ __forceinline__ void st_v4(uint8_t* ptr, const uint4& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Hardware (MUFU) base-2 exponential, logarithm and reciprocal, each within
// ~2 ulp; subnormal results flush to zero, so a weight below 2^-126 of the
// largest one counts as zero.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- 16-bit <-> fp32 -----------------------------------------------------------

template <bool kF16>
__device__ __forceinline__ float2 widen2(uint32_t w) {
    if constexpr (kF16) {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    } else {
        // bf16 is the upper half of an fp32: element 2k sits in the low 16 bits
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
}

template <bool kF16>
__device__ __forceinline__ uint32_t narrow2(float lo, float hi) {
    if constexpr (kF16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// ---- per-unit pieces -------------------------------------------------------

constexpr int kNoMask = 0x7fffffff;

// The unit's LSEs, and its row's context length when masking (else kNoMask).
template <int kMaxCp>
__device__ __forceinline__ int load_lses(const Params<kMaxCp>& p, const Pos& q, float (&l)[kMaxCp]) {
    const int64_t off = (int64_t)q.b * p.lse_row + (int64_t)(q.r * p.Hl + q.i) * p.lse_head;
    const int seq = p.seq_lens != nullptr ? ld_nc_s32(p.seq_lens + q.b) : kNoMask;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) l[j] = (j < p.cp) ? ld_nc_f32(p.lse[j] + off) : -INFINITY;
    return seq;
}

// With the KV interleaved over the shards in blocks of `interleave` tokens,
// shard j's first token is j*interleave: it owns a token of a context of `seq`
// tokens iff seq > j*interleave. An empty shard's LSE entry is ignored.
template <int kMaxCp>
__device__ __forceinline__ void mask_empty(const Params<kMaxCp>& p, int seq, float (&l)[kMaxCp]) {
    if (seq == kNoMask) return;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j)
        if ((int64_t)j * p.interleave >= (int64_t)seq) l[j] = -INFINITY;
}

// w_j = 2^((l_j - m)*s) / sum_k 2^((l_k - m)*s), s = 1 for base-2 LSEs and
// log2(e) for natural ones; merged = m + log2(sum) * (1 or ln 2). A row whose
// every source is -inf gets all-zero weights and merged = -inf.
template <int kMaxCp>
__device__ __forceinline__ float lse_weights(const Params<kMaxCp>& p, const float (&l)[kMaxCp],
                                             float (&w)[kMaxCp]) {
    float mx[kMaxCp];
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) mx[j] = l[j];
#pragma unroll
    for (int half = kMaxCp / 2; half >= 1; half /= 2)
#pragma unroll
        for (int j = 0; j < half; ++j) mx[j] = fmaxf(mx[j], mx[j + half]);
    const float m = mx[0];
    if (m == -INFINITY) {
#pragma unroll
        for (int j = 0; j < kMaxCp; ++j) w[j] = 0.f;
        return -INFINITY;
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) {
        const float e = (l[j] == -INFINITY) ? 0.f : ex2_approx((l[j] - m) * p.lse_scale);
        w[j] = e;
        s += e;
    }
    const float inv = rcp_approx(s);  // s is in [1, cp]
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) w[j] *= inv;
    return fmaf(lg2_approx(s), p.log_scale, m);
}

// Issue the payload loads of sources [jb*kSB, jb*kSB + kSB) for one pass.
// kGate: skip sources whose weight is 0 (weights known); otherwise load every
// source j < cp (weights not known yet; zero-weight payloads are dropped later).
template <int kSB, int kMaxCp, int kFixedChunks, bool kGate>
__device__ __forceinline__ void load_batch(const Params<kMaxCp>& p, int64_t src_off, int jb, int pass, int lane,
                                           int nchunks, const float (&w)[kMaxCp], uint4 (&x)[kSB][kVpl]) {
#pragma unroll
    for (int j = 0; j < kSB; ++j) {
        const int jj = jb * kSB + j;
        const bool on = (jj < p.cp) && (!kGate || w[jj] != 0.f);
#pragma unroll
        for (int v = 0; v < kVpl; ++v) {
            const int c = pass * kChunksPerPass + v * 32 + lane;
            const bool in = (kFixedChunks == kChunksPerPass) || (c < nchunks);
            if (on && in) {
                x[j][v] = ld_stream_v4(p.src[jj] + src_off + (int64_t)c * 16);
            } else {
                x[j][v] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
}

template <bool kF16, int kSB, int kMaxCp>
__device__ __forceinline__ void accumulate(int jb, int cp, const float (&w)[kMaxCp], const uint4 (&x)[kSB][kVpl],
                                           float (&acc)[kVpl][8]) {
#pragma unroll
    for (int j = 0; j < kSB; ++j) {
        const int jj = jb * kSB + j;
        if (jj < cp && w[jj] != 0.f) {  // warp-uniform: zero-weight sources are skipped, never multiplied
#pragma unroll
            for (int v = 0; v < kVpl; ++v) {
                const uint32_t q[4] = {x[j][v].x, x[j][v].y, x[j][v].z, x[j][v].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = widen2<kF16>(q[k]);
                    acc[v][2 * k] = fmaf(w[jj], f.x, acc[v][2 * k]);
                    acc[v][2 * k + 1] = fmaf(w[jj], f.y, acc[v][2 * k + 1]);
                }
            }
        }
    }
}

template <int kMaxCp>
__device__ __forceinline__ int64_t src_offset(const Params<kMaxCp>& p, const Pos& q) {
    return ((int64_t)q.b * p.src_row + (int64_t)(q.r * p.Hl + q.i) * p.src_head) * 2;  // bytes
}

// Bring one unit's inputs into L2: lane j < cp takes source j's row (D*2
// bytes, one bulk prefetch), lane 16 + j its LSE line, lane 31 the row's
// context length.
template <int kMaxCp>
__device__ __forceinline__ void prefetch_unit(const Params<kMaxCp>& p, const Pos& q, int lane) {
    if (lane < p.cp) {
        prefetch_l2_bulk(p.src[lane] + src_offset(p, q), (uint32_t)p.D * 2u);
    } else if (lane >= 16 && lane - 16 < p.cp) {
        prefetch_l2_line(p.lse[lane - 16] + (int64_t)q.b * p.lse_row + (int64_t)(q.r * p.Hl + q.i) * p.lse_head);
    } else if (lane == 31 && p.seq_lens != nullptr) {
        prefetch_l2_line(p.seq_lens + q.b);
    }
}

// ---- the kernel ----------------------------------------------------------------

// Register budget for D = 512: keep 7 CTAs of 4 warps resident per SM for up
// to 4 sources (the PRELOAD grid of a 64-head, 64-row call then fits in one
// wave) and 4 CTAs (128 registers) for up to 8 sources.
template <int kMaxCp, int kFixedChunks>
constexpr int min_ctas_per_sm() {
    if (kFixedChunks != kChunksPerPass) return 1;
    return kMaxCp <= 4 ? 7 : (kMaxCp <= 8 ? 4 : 1);
}

template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
__global__ void __launch_bounds__(kMaxThreads, min_ctas_per_sm<kMaxCp, kFixedChunks>())
    lse_merge_kernel(const __grid_constant__ Params<kMaxCp> p) {
    constexpr int kSB = kMaxCp < 8 ? kMaxCp : 8;  // sources per load batch
    constexpr int kNB = kMaxCp / kSB;             // load batches
    static_assert(!kPreload || (kNB == 1 && kFixedChunks == kChunksPerPass),
                  "PRELOAD needs all sources in one batch and one pass");

    const int lane = threadIdx.x & 31;
    int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= p.units) return;  // an exited CTA counts as having released its dependents

    // Index and address arithmetic reads only the parameters, so it runs before
    // the wait and overlaps the previous kernel's tail under PDL: the first
    // unit's LSE and payload addresses are pinned in registers here.
    const int nchunks = kFixedChunks ? kFixedChunks : (p.D >> 3);
    const int npass = (nchunks + kChunksPerPass - 1) / kChunksPerPass;
    Pos q = unit_pos(p, u);
    const float* lp[kMaxCp];
    const uint8_t* sp[kSB];
    const int* slp = p.seq_lens != nullptr ? p.seq_lens + q.b : nullptr;
    {
        const int64_t loff = (int64_t)q.b * p.lse_row + (int64_t)(q.r * p.Hl + q.i) * p.lse_head;
        const int64_t soff = src_offset(p, q) + (int64_t)lane * 16;
#pragma unroll
        for (int j = 0; j < kMaxCp; ++j) {
            lp[j] = p.lse[j] + loff;
            asm volatile("" : "+l"(lp[j]));
        }
#pragma unroll
        for (int j = 0; j < kSB; ++j) {
            sp[j] = p.src[j] + soff;
            asm volatile("" : "+l"(sp[j]));
        }
    }

    // A prefetch only warms L2 (the point of coherence), so it may run before
    // the wait: if the previous kernel writes these inputs, the loads after the
    // wait still see its values.
    if (p.prefetch_first) prefetch_unit(p, q, lane);

    // Inputs may come from the previous kernel in the stream (PDL): wait for it
    // before the first load. Then let the next kernel start its launch.
    pdl_wait();
    pdl_launch_dependents();

    float l[kMaxCp];
    float w[kMaxCp];
    uint4 x[kSB][kVpl];
    int seq = slp != nullptr ? ld_nc_s32(slp) : kNoMask;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) l[j] = (j < p.cp) ? ld_nc_f32(lp[j]) : -INFINITY;
    if constexpr (kPreload) {
        // one pass of 64 chunks: lane's chunks are lane and 32 + lane
#pragma unroll
        for (int j = 0; j < kSB; ++j) {
#pragma unroll
            for (int v = 0; v < kVpl; ++v) {
                x[j][v] = (j < p.cp) ? ld_stream_v4(sp[j] + v * 512) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }

    while (true) {
        const bool more = u + p.step < p.units;
        const Pos qn = advance(p, q);
        const int64_t src_off = src_offset(p, q);
        uint8_t* const dst = p.dst[q.r] + ((int64_t)q.b * p.dst_row + (int64_t)q.i * p.dst_head) * 2;

        mask_empty<kMaxCp>(p, seq, l);
        const float merged = lse_weights<kMaxCp>(p, l, w);

        for (int pass = 0; pass < npass; ++pass) {
            float acc[kVpl][8];
#pragma unroll
            for (int v = 0; v < kVpl; ++v)
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[v][k] = 0.f;
#pragma unroll
            for (int jb = 0; jb < kNB; ++jb) {
                if (jb * kSB >= p.cp) break;
                if (!kPreload) load_batch<kSB, kMaxCp, kFixedChunks, true>(p, src_off, jb, pass, lane, nchunks, w, x);
                // the next unit's LSEs travel while this payload is in flight
                if (pass == 0 && jb == 0 && more) seq = load_lses<kMaxCp>(p, qn, l);
                accumulate<kF16, kSB, kMaxCp>(jb, p.cp, w, x, acc);
            }
#pragma unroll
            for (int v = 0; v < kVpl; ++v) {
                const int c = pass * kChunksPerPass + v * 32 + lane;
                if (kFixedChunks == kChunksPerPass || c < nchunks) {
                    uint4 o;
                    o.x = narrow2<kF16>(acc[v][0], acc[v][1]);
                    o.y = narrow2<kF16>(acc[v][2], acc[v][3]);
                    o.z = narrow2<kF16>(acc[v][4], acc[v][5]);
                    o.w = narrow2<kF16>(acc[v][6], acc[v][7]);
                    st_v4(dst + (int64_t)c * 16, o);
                }
            }
        }
        if (lane == 0 && p.lse_out[q.r] != nullptr) p.lse_out[q.r][(int64_t)q.b * p.lse_out_row + q.i] = merged;

        if (!more) break;
        u += p.step;
        q = qn;
        if constexpr (kPreload) {
            load_batch<kSB, kMaxCp, kFixedChunks, false>(p, src_offset(p, q), 0, 0, lane, nchunks, w, x);
        }
    }
}


// ---- host side -----------------------------------------------------------------

// Everything a launch needs, independent of the source count.
struct Launch {
    const void* const* src;
    const float* const* lse;
    void* const* dst;
    float* const* lse_out;
    int cp, H, D;
    int64_t B;
    bool base_e, f16, fixed512;
    dcp_lse_reduce_layout lay;
    const int32_t* seq_lens;
    int interleave;
    unsigned flags;
    cudaStream_t stream;
    int sms;
};

// Resident CTAs per SM for one instantiation and CTA size, from the occupancy
// calculator (queried once; the value depends only on the kernel).
template <typename K>
int ctas_per_sm(K kernel, int threads, int (&cache)[2]) {
    int& slot = cache[threads == 64 ? 0 : 1];
    int n = __atomic_load_n(&slot, __ATOMIC_RELAXED);
    if (n > 0) return n;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    __atomic_store_n(&slot, n, __ATOMIC_RELAXED);
    return n;
}

template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
int occupancy(int threads) {
    static int cache[2] = {0, 0};
    return ctas_per_sm(lse_merge_kernel<kF16, kMaxCp, kFixedChunks, kPreload>, threads, cache);
}

// The parameters of one launch over rows [b0, b0 + rows), `step` warps apart.
template <int kMaxCp>
Params<kMaxCp> make_params(const Launch& L, int64_t b0, int rows, int step) {
    Params<kMaxCp> p;
    const int H = L.H, Hl = L.H / L.cp;
    p.units = rows * H;
    p.H = H;
    p.Hl = Hl;
    p.cp = L.cp;
    p.D = L.D;
    p.step = step;
    p.step_b = step / H;
    const int sh = step % H;
    p.step_r = sh / Hl;
    p.step_i = sh % Hl;
    p.lse_scale = L.base_e ? 1.4426950408889634f : 1.0f;
    p.log_scale = L.base_e ? 0.6931471805599453f : 1.0f;
    p.interleave = L.interleave;
    p.prefetch_first = (L.flags & DCP_FLAG_PREFETCH) ? 1 : 0;
    p.seq_lens = L.seq_lens != nullptr ? L.seq_lens + b0 : nullptr;
    p.lse_row = L.lay.lse_row;
    p.lse_head = L.lay.lse_head;
    p.src_row = L.lay.src_row;
    p.src_head = L.lay.src_head;
    p.dst_row = L.lay.dst_row;
    p.dst_head = L.lay.dst_head;
    p.lse_out_row = L.lay.lse_out_row;
    for (int j = 0; j < kMaxCp; ++j) {
        const bool on = j < L.cp;
        p.lse[j] = on ? L.lse[j] + b0 * L.lay.lse_row : nullptr;
        p.src[j] = on ? static_cast<const uint8_t*>(L.src[j]) + b0 * L.lay.src_row * 2 : nullptr;
        p.dst[j] = on ? static_cast<uint8_t*>(L.dst[j]) + b0 * L.lay.dst_row * 2 : nullptr;
        float* lo = (on && L.lse_out != nullptr) ? L.lse_out[j] : nullptr;
        p.lse_out[j] = lo != nullptr ? lo + b0 * L.lay.lse_out_row : nullptr;
    }
    return p;
}

template <typename K, typename P>
cudaError_t launch_kernel(const Launch& L, K kernel, const P& p, int ctas, int threads, int smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (L.flags & DCP_FLAG_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
cudaError_t launch_one(const Launch& L, int64_t b0, int rows, int threads, int ctas) {
    const Params<kMaxCp> p = make_params<kMaxCp>(L, b0, rows, ctas * (threads / 32));
    return launch_kernel(L, lse_merge_kernel<kF16, kMaxCp, kFixedChunks, kPreload>, p, ctas, threads, 0);
}

// Pick the schedule and grid for one instantiation family and launch every
// row chunk (a chunk holds at most kMaxUnitsPerLaunch units).
template <bool kF16, int kMaxCp, int kFixedChunks>
cudaError_t launch_cp(const Launch& L) {
    constexpr bool kCanPreload = (kFixedChunks == kChunksPerPass) && (kMaxCp <= 8);
    const int64_t rows_per_launch = kMaxUnitsPerLaunch / L.H;
    for (int64_t b0 = 0; b0 < L.B; b0 += rows_per_launch) {
        const int rows = (int)((L.B - b0) < rows_per_launch ? (L.B - b0) : rows_per_launch);
        const int64_t units = (int64_t)rows * L.H;
        // One unit per warp with the payload loads issued beside the LSE loads
        // (in as many waves as it takes) is the faster stream whenever it is
        // available. The persistent wave that reads LSEs a unit ahead and skips
        // empty sources is kept for seq_lens masking on grids larger than one
        // resident wave, where skipping the masked payloads pays.
        bool preload = false;
        if constexpr (kCanPreload) {
            const int threads = units <= 1024 ? 64 : 128;
            preload = L.seq_lens == nullptr ||
                      units <= (int64_t)L.sms * occupancy<kF16, kMaxCp, kFixedChunks, true>(threads) * (threads / 32);
        }
        if (L.flags & DCP_FLAG_PRELOAD) preload = kCanPreload;
        if (L.flags & DCP_FLAG_LSE_FIRST) preload = false;
        // Small grids spread over more SMs with 2-warp CTAs; larger ones need
        // fewer, larger CTAs.
        const int threads = (preload && units <= 1024) ? 64 : 128;
        const int wpc = threads / 32;
        const int64_t want = (units + wpc - 1) / wpc;
        cudaError_t e;
        if constexpr (kCanPreload) {
            if (preload) {
                e = launch_one<kF16, kMaxCp, kFixedChunks, true>(L, b0, rows, threads, (int)want);
                if (e != cudaSuccess) return e;
                continue;
            }
        }
        const int64_t wave = (int64_t)L.sms * occupancy<kF16, kMaxCp, kFixedChunks, false>(threads);
        e = launch_one<kF16, kMaxCp, kFixedChunks, false>(L, b0, rows, threads, (int)(want < wave ? want : wave));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <bool kF16, int kMaxCp>
cudaError_t launch_d(const Launch& L) {
    return L.fixed512 ? launch_cp<kF16, kMaxCp, kChunksPerPass>(L) : launch_cp<kF16, kMaxCp, 0>(L);
}

template <bool kF16>
cudaError_t launch_dtype(const Launch& L) {
    if (L.cp <= 1) return launch_d<kF16, 1>(L);
    if (L.cp <= 2) return launch_d<kF16, 2>(L);
    if (L.cp <= 4) return launch_d<kF16, 4>(L);
    if (L.cp <= 8) return launch_d<kF16, 8>(L);
    return launch_d<kF16, 16>(L);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int dcp_lse_reduce_ex(const void* const* src_ptrs, const float* const* lse_ptrs,
                                 int cp, int64_t B, int H, int D, int lse_base_e, int dtype,
                                 void* const* dst_ptrs, float* const* lse_out_ptrs,
                                 const dcp_lse_reduce_layout* layout, const int32_t* seq_lens, int interleave,
                                 unsigned flags, void* stream) {
    if (src_ptrs == nullptr || lse_ptrs == nullptr || dst_ptrs == nullptr) return DCP_ERR_NULL_POINTER;
    if (cp < 1 || cp > kCpMax) return DCP_ERR_BAD_CP;
    if (B < 0 || H < 1 || D < 8 || D % 8 != 0) return DCP_ERR_BAD_SHAPE;
    if (H % cp != 0) return DCP_ERR_HEADS_NOT_DIVISIBLE;
    if (dtype != DCP_DTYPE_BF16 && dtype != DCP_DTYPE_F16) return DCP_ERR_BAD_DTYPE;
    if (lse_base_e != 0 && lse_base_e != 1) return DCP_ERR_BAD_BASE;
    if ((flags & ~(DCP_FLAG_PDL | DCP_FLAG_PRELOAD | DCP_FLAG_LSE_FIRST | DCP_FLAG_PREFETCH)) != 0)
        return DCP_ERR_BAD_FLAGS;
    if ((flags & DCP_FLAG_PRELOAD) && (flags & DCP_FLAG_LSE_FIRST)) return DCP_ERR_BAD_FLAGS;
    if (seq_lens != nullptr) {
        if (interleave < 1 || interleave > DCP_LSE_REDUCE_INTERLEAVE_MAX) return DCP_ERR_BAD_INTERLEAVE;
        if (!aligned(seq_lens, 4)) return DCP_ERR_MISALIGNED;
    }

    const int Hl = H / cp;
    dcp_lse_reduce_layout lay;
    if (layout != nullptr) {
        lay = *layout;
    } else {
        lay.src_row = (int64_t)H * D;
        lay.src_head = D;
        lay.lse_row = H;
        lay.lse_head = 1;
        lay.dst_row = (int64_t)Hl * D;
        lay.dst_head = D;
        lay.lse_out_row = Hl;
    }
    if (lay.src_row < 0 || lay.src_head < 0 || lay.lse_row < 0 || lay.lse_head < 0 || lay.dst_row < 0 ||
        lay.dst_head < 0 || lay.lse_out_row < 0)
        return DCP_ERR_BAD_STRIDE;
    if (lay.src_row % 8 || lay.src_head % 8 || lay.dst_row % 8 || lay.dst_head % 8) return DCP_ERR_BAD_STRIDE;

    for (int j = 0; j < cp; ++j) {
        if (src_ptrs[j] == nullptr || lse_ptrs[j] == nullptr || dst_ptrs[j] == nullptr) return DCP_ERR_NULL_POINTER;
        if (!aligned(src_ptrs[j], 16) || !aligned(dst_ptrs[j], 16) || !aligned(lse_ptrs[j], 4))
            return DCP_ERR_MISALIGNED;
        if (lse_out_ptrs != nullptr && lse_out_ptrs[j] != nullptr && !aligned(lse_out_ptrs[j], 4))
            return DCP_ERR_MISALIGNED;
    }
    if (B == 0) return DCP_OK;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1) {
        (void)cudaGetLastError();
        return DCP_ERR_DEVICE;
    }
    Launch L;
    L.src = src_ptrs;
    L.lse = lse_ptrs;
    L.dst = dst_ptrs;
    L.lse_out = lse_out_ptrs;
    L.cp = cp;
    L.H = H;
    L.D = D;
    L.B = B;
    L.base_e = lse_base_e != 0;
    L.f16 = dtype == DCP_DTYPE_F16;
    L.fixed512 = D == 512;
    L.lay = lay;
    L.seq_lens = seq_lens;
    L.interleave = seq_lens != nullptr ? interleave : 1;
    L.flags = flags;
    L.stream = static_cast<cudaStream_t>(stream);
    L.sms = sms;
    const cudaError_t e = L.f16 ? launch_dtype<true>(L) : launch_dtype<false>(L);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    return DCP_OK;
}

extern "C" int dcp_lse_reduce(const void* const* src_ptrs, const float* const* lse_ptrs, int64_t lse_stride,
                              int cp, int64_t B, int H, int D, int lse_base_e,
                              void* const* dst_ptrs, float* const* lse_out_ptrs, void* stream) {
    if (src_ptrs == nullptr || lse_ptrs == nullptr || dst_ptrs == nullptr) return DCP_ERR_NULL_POINTER;
    if (cp < 1 || cp > kCpMax) return DCP_ERR_BAD_CP;
    if (B < 0 || H < 1 || D < 8 || D % 8 != 0) return DCP_ERR_BAD_SHAPE;
    if (H % cp != 0) return DCP_ERR_HEADS_NOT_DIVISIBLE;
    if (lse_stride < H) return DCP_ERR_BAD_STRIDE;
    dcp_lse_reduce_layout lay;
    lay.src_row = (int64_t)H * D;
    lay.src_head = D;
    lay.lse_row = lse_stride;
    lay.lse_head = 1;
    lay.dst_row = (int64_t)(H / cp) * D;
    lay.dst_head = D;
    lay.lse_out_row = H / cp;
    return dcp_lse_reduce_ex(src_ptrs, lse_ptrs, cp, B, H, D, lse_base_e, DCP_DTYPE_BF16, dst_ptrs, lse_out_ptrs,
                             &lay, nullptr, 1, 0u, stream);
}

extern "C" const char* dcp_lse_reduce_strerror(int status) {
    switch (status) {
        case DCP_OK: return "success";
        case DCP_ERR_NULL_POINTER: return "a required pointer (array or entry) is NULL";
        case DCP_ERR_BAD_CP: return "cp must be in [1, 16]";
        case DCP_ERR_BAD_SHAPE: return "B must be >= 0, H >= 1, and D a positive multiple of 8";
        case DCP_ERR_HEADS_NOT_DIVISIBLE: return "H must be a multiple of cp";
        case DCP_ERR_BAD_STRIDE:
            return "strides must be >= 0, payload strides multiples of 8 elements, and lse_stride >= H";
        case DCP_ERR_MISALIGNED: return "payload pointers must be 16-byte aligned and LSE pointers 4-byte aligned";
        case DCP_ERR_BAD_FLAGS: return "unknown flag bits, or DCP_FLAG_PRELOAD together with DCP_FLAG_LSE_FIRST";
        case DCP_ERR_BAD_DTYPE: return "dtype must be DCP_DTYPE_BF16 or DCP_DTYPE_F16";
        case DCP_ERR_BAD_BASE: return "lse_base_e must be 0 (base 2) or 1 (base e)";
        case DCP_ERR_DEVICE: return "could not query the current CUDA device";
        case DCP_ERR_BAD_INTERLEAVE: return "interleave must be in [1, 2^24] when seq_lens is given";
        // the producer and the fused decode (include/dcp_mla_decode.h)
        case DCP_MLA_ERR_NULL_POINTER: return "q, kv, kv_len, out_ptrs, lse_ptrs or an entry is NULL";
        case DCP_MLA_ERR_BAD_SHAPE:
            return "B must be in [0, 65535], T >= 0, H a positive multiple of 16, Dk 512 or 576, Dv 512";
        case DCP_MLA_ERR_BAD_SPLIT: return "n_split must be in [1, 16]";
        case DCP_MLA_ERR_MISALIGNED:
            return "q, kv and outputs must be 16-byte aligned; LSE, kv_len and status 4-byte aligned";
        case DCP_MLA_ERR_BAD_FLAGS: return "unknown flag bits, or DCP_MLA_FLAG_MMA_SYNC together with DCP_MLA_FLAG_TCGEN05";
        case DCP_MLA_ERR_WORKSPACE:
            return "workspace is NULL, not 256-byte aligned, or smaller than dcp_mla_decode_workspace_bytes";
        case DCP_MLA_ERR_BAD_CP: return "cp*n_split must be <= 16 and divide H";
        case DCP_MLA_ERR_SCRATCH_LIMIT:
            return "the partials need more than the built-in 32 MiB scratch (DCP_MLA_NOALLOC_SCRATCH_BYTES)";
        case DCP_MLA_ERR_SCRATCH_SETUP:
            return "the built-in scratch array's device address could not be obtained on this device";
        case DCP_MLA_ERR_TENSOR_MAP: return "a TMA tensor map for q or a cache could not be encoded";
        default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

extern "C" int dcp_lse_reduce_version(void) { return 10000; }
