// Split-KV MLA decode attention over one context shard, sm_103a: the producer
// of the DCP partial outputs and LSEs. What it computes, and the passages it
// follows, are stated in include/dcp_mla_decode.h.
//
// The file holds two kernels and their host side:
//   * mla_partial_kernel, on the warp-level mma.sync tensor path (below);
//   * mla_partial_tc_kernel, on the 5th-generation tensor cores (tcgen05 MMA
//     into TMEM, operands loaded by TMA; its design is stated before it);
//   * the host entry points: the producer (which picks a kernel), the fused
//     DCP decode (producer over every shard, then the merge of
//     dcp_lse_reduce.cu, or with DCP_MLA_FLAG_ONE_KERNEL the merge inside the
//     producer's launch) and its form that allocates nothing.
//
// Design of the mma.sync kernel. One CTA owns (split s, a block of 16*kG
// heads, row b) and walks its token range in tiles of 32 tokens:
//   * Q for the head block and each KV tile land in shared memory by 1-D bulk
//     asynchronous copies (cp.async.bulk, one per row, completing on an
//     mbarrier), into rows padded by 16 bytes so that the 8x8 ldmatrix reads
//     below are free of bank conflicts. Two KV buffers: tile i+2 streams in
//     while tile i+1 is waited for and tile i is consumed.
//   * four warps per group g of 16 heads. For the scores, warp (g, q) takes
//     token half q&1 and Dk half q>>1 (bf16 tensor-core MMA m16n8k16, fp32
//     accumulation; two independent accumulation chains of Dk/32 steps); the
//     upper Dk half hands its partial to the lower half through shared memory,
//     which posts the sum. All four warps then read the 16x32 score tile, run
//     the online softmax in base 2, and multiply the bf16 probabilities by
//     value columns [128q, 128q+128) of the tile (ldmatrix.trans gives the
//     value fragments straight from the token-major rows); the 16x128 fp32
//     output block of a warp lives in registers.
//   * at the end: divide by the running sum, round to bf16, and write the
//     partial output and the LSE (base e or 2).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <cooperative_groups.h>
#include <mutex>

#include "dcp_lse_reduce.h"
#include "dcp_mla_decode.h"

namespace {

constexpr int kDv = 512;
constexpr int kNt = 32;              // tokens per KV tile
constexpr int kSPad = 4;             // fp32 padding of a score row in shared memory
constexpr unsigned kFlagPdl = 1u;
constexpr unsigned kFlagPrefetch = 8u;  // DCP_FLAG_PREFETCH: L2 prefetch of the first tile before the PDL wait
constexpr unsigned kFlagMmaSync = 2u;   // DCP_MLA_FLAG_MMA_SYNC
constexpr unsigned kFlagTcgen05 = 4u;   // DCP_MLA_FLAG_TCGEN05
constexpr unsigned kFlagOneKernel = 16u;  // DCP_MLA_FLAG_ONE_KERNEL (dcp_mla_decode only)
constexpr unsigned kFlagTestStall = 32u;  // DCP_MLA_FLAG_TEST_STALL
// When the tcgen05 kernel is the default. Its MMAs cost about the same per
// instruction whatever the head block (N = 16, 32 or 64), so it pays off with
// 64-head blocks from one full 128-token tile per (row, split), with 32-head
// blocks from two, and never with 16-head blocks, where the mma.sync kernel is
// faster at every measured length.
constexpr int64_t kTcMinTokensH64 = 128;
constexpr int64_t kTcMinTokensH32 = 256;
constexpr long long kWaitLimitNs = 2000000000LL;      // every wait of a call gives up after this
constexpr long long kTestWaitLimitNs = 20000000LL;    // ... or this, with DCP_MLA_FLAG_TEST_STALL

constexpr int kSlots = 16;            // (shard, split) outputs of one launch

struct Params {
    const uint8_t* q;                 // [B, H, Dk] bf16
    const uint8_t* kv[kSlots];        // per shard: [B, T, Dk] bf16
    const int* kv_len[kSlots];        // per shard: [B]
    uint8_t* out[kSlots];             // per (shard, split): [B, H, Dv] bf16
    float* lse[kSlots];               // per (shard, split): [B, H] fp32
    int* status;
    int64_t T;
    int H, n_split;
    float scale_log2;                 // softmax scale * log2(e): scores in base-2 units
    float lse_scale;                  // ln 2 for a natural-log LSE, 1 for base 2
    long long wait_ns;                // limit of every wait (kWaitLimitNs, or kTestWaitLimitNs)
    int stall;                        // DCP_MLA_FLAG_TEST_STALL: the first tile's barrier expects 16 bytes more
};

template <int kDk>
__host__ __device__ constexpr int row_bytes() {
    return (kDk + 8) * 2;  // 16 bytes of padding per row
}

template <int kDk, int kG>
__host__ __device__ constexpr int smem_bytes() {
    return 16 * kG * row_bytes<kDk>() + 2 * kNt * row_bytes<kDk>() + 16 * kG * (kNt + kSPad) * 4 + kG * 2 * 256 * 4 +
           3 * 8 + 16;
}

// ---- PTX helpers -------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ long long global_ns() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// The waits of both kernels. Every thread of a CTA shares one abort
// flag in shared memory: a wait that has not seen its phase after
// limit_ns (the call's wait limit) sets it (and ORs 1 into the status word), and from then on
// every wait of the CTA returns at once. Returns whether the phase completed.
// The kernel stops issuing copies and MMAs, leaves its tile loop at the next
// tile boundary (a barrier vote, so all threads leave together), skips the
// epilogue (the outputs are not valid) and drains the copies and MMAs it
// armed before it frees TMEM and exits.
__device__ __forceinline__ bool mbar_wait_cta(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                              long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            if (status != nullptr) atomicOr(status, 1);
            return false;
        }
    }
    return true;
}
// Bounded wait that ignores the abort flag: the drain before TMEM is freed.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}
// One contiguous global -> shared copy by the bulk-copy engine.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Loads through L2 only (data other CTAs of this grid wrote).
__device__ __forceinline__ float ld_cg_f32(const float* ptr) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}
__device__ __forceinline__ uint4 ld_cg_v4(const uint8_t* ptr) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
    return v;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- the kernel ----------------------------------------------------------------

template <int kDk, int kG>
__global__ void __launch_bounds__(128 * kG, 1) mla_partial_kernel(const __grid_constant__ Params p) {
    constexpr int kHB = 16 * kG;            // heads per CTA
    constexpr int kRow = row_bytes<kDk>();  // padded shared row, bytes
    constexpr int kKHalf = kDk / 32;        // k-steps of 16 in half of Dk
    constexpr int kSRow = kNt + kSPad;      // score row, floats
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* const q_s = smem;
    uint8_t* const kv_s = q_s + kHB * kRow;
    float* const s_s = reinterpret_cast<float*>(kv_s + 2 * kNt * kRow);   // [kHB][kSRow] scores of a tile
    float* const s_part = s_s + kHB * kSRow;                              // [kG][2][16][16] half-Dk partial scores
    uint64_t* const bars = reinterpret_cast<uint64_t*>(s_part + kG * 2 * 256);  // [0] Q, [1], [2] KV buffers
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(bars + 3);  // see mbar_wait_cta
    int* const armed = reinterpret_cast<int*>(bars + 3) + 1;                      // [2]: last tile loaded per buffer

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp % kG;    // head group: heads [16g, 16g+16) of the block
    const int q4 = warp / kG;   // 0..3: value columns [128*q4, +128)
    const int th = q4 & 1;      // score tokens [16*th, +16) of the tile
    const int kh = q4 >> 1;     // score k-steps over Dk half kh
    const int slot = blockIdx.x;            // shard * n_split + split
    const int shard = slot / p.n_split;
    const int split = slot - shard * p.n_split;
    const int h0 = blockIdx.y * kHB;
    const int b = blockIdx.z;
    const int gr = lane >> 2;   // fragment row within the 8-row half
    const int tq = lane & 3;    // fragment column pair

    // Shared-memory set-up reads no input, so it overlaps the previous kernel.
    for (int i = threadIdx.x; i < (2 * kNt * kRow) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(kv_s)[i] = make_uint4(0u, 0u, 0u, 0u);  // stale rows stay finite
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        *abort_flag = 0;
        armed[0] = armed[1] = -1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    pdl_wait();
    pdl_launch_dependents();

    int64_t len = p.kv_len[shard][b];
    len = len < 0 ? 0 : (len > p.T ? p.T : len);
    const int64_t chunk = (len + p.n_split - 1) / p.n_split;
    const int64_t t_begin = (int64_t)split * chunk;
    const int64_t t_end = t_begin + chunk < len ? t_begin + chunk : len;
    const int ntok = t_end > t_begin ? (int)(t_end - t_begin) : 0;

    uint8_t* const out = p.out[slot];
    float* const lse = p.lse[slot];
    const int64_t out_row0 = ((int64_t)b * p.H + h0 + 16 * g) * kDv;  // element index of head row 16g

    if (ntok == 0) {  // empty range: output 0, LSE -inf
        for (int r = 0; r < 16; ++r) {
            uint32_t* o = reinterpret_cast<uint32_t*>(out + (out_row0 + (int64_t)r * kDv + 128 * q4) * 2);
            for (int c = lane; c < 64; c += 32) o[c] = 0u;
        }
        if (q4 == 0 && lane < 16) lse[(int64_t)b * p.H + h0 + 16 * g + lane] = -INFINITY;
        return;
    }
    const int ntiles = (ntok + kNt - 1) / kNt;
    const uint8_t* const kv_row = p.kv[shard] + ((int64_t)b * p.T + t_begin) * kDk * 2;

    auto load_tile = [&](int i, int buf) {
        const int rows = (ntok - i * kNt) < kNt ? (ntok - i * kNt) : kNt;
        uint8_t* dst = kv_s + buf * kNt * kRow;
        // (with the stall test, tile 0's barrier waits for 16 bytes that never come)
        mbar_expect_tx(&bars[1 + buf], (uint32_t)(rows * kDk * 2) + (p.stall && i == 0 ? 16u : 0u));
        for (int r = 0; r < rows; ++r)
            bulk_g2s(dst + r * kRow, kv_row + ((int64_t)i * kNt + r) * kDk * 2, kDk * 2, &bars[1 + buf]);
        armed[buf] = i;
    };
    if (threadIdx.x == 0) {
        mbar_expect_tx(&bars[0], (uint32_t)(kHB * kDk * 2));
        const uint8_t* qrow = p.q + ((int64_t)b * p.H + h0) * kDk * 2;
        for (int r = 0; r < kHB; ++r) bulk_g2s(q_s + r * kRow, qrow + (int64_t)r * kDk * 2, kDk * 2, &bars[0]);
        load_tile(0, 0);
        if (ntiles > 1) load_tile(1, 1);
    }
    (void)mbar_wait_cta(&bars[0], 0, abort_flag, p.status, p.wait_ns);

    // per-lane state: rows gr and gr+8 of the warp's 16 heads
    float m_run[2] = {-INFINITY, -INFINITY};  // running max, base-2 units
    float l_run[2] = {0.f, 0.f};              // running sum of 2^(s - m)
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    // ldmatrix row addresses (bytes within the buffers)
    const uint32_t q_base = smem_u32(q_s) + (16 * g + (lane & 15)) * kRow + (lane >> 4) * 16 + kh * kKHalf * 32;
    const uint32_t k_off =
        (16 * th + (lane & 7) + ((lane >> 4) << 3)) * kRow + ((lane >> 3) & 1) * 16 + kh * kKHalf * 32;
    const uint32_t v_off = ((lane & 7) + (((lane >> 3) & 1) << 3)) * kRow + (128 * q4 + (lane >> 4) * 8) * 2;
    float* const part = s_part + (g * 2 + th) * 256;  // 16 x 16 partial of (group, token half)

    bool aborted = false;  // CTA-uniform: decided by a barrier vote at the end of each tile
    for (int i = 0; i < ntiles; ++i) {
        const int buf = i & 1;
        (void)mbar_wait_cta(&bars[1 + buf], (uint32_t)((i >> 1) & 1), abort_flag, p.status, p.wait_ns);
        const uint32_t kt = smem_u32(kv_s + buf * kNt * kRow);

        // partial scores: 16 heads x 16 tokens over half of Dk
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 6
        for (int ks = 0; ks < kKHalf; ++ks) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(q_base + ks * 32, a0, a1, a2, a3);
            ldsm_x4(kt + k_off + ks * 32, b0, b1, b2, b3);
            mma_bf16(sacc[0], a0, a1, a2, a3, b0, b1);
            mma_bf16(sacc[1], a0, a1, a2, a3, b2, b3);
        }
        // the upper Dk half hands its partial to the lower half, which writes the sum
        if (kh == 1) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                float* r0 = part + gr * 16 + 8 * n + 2 * tq;
                r0[0] = sacc[n][0];
                r0[1] = sacc[n][1];
                r0[128] = sacc[n][2];
                r0[129] = sacc[n][3];
            }
        }
        named_sync(1 + g, 128);
        if (kh == 0) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const float* r0 = part + gr * 16 + 8 * n + 2 * tq;
                float* d0 = s_s + (16 * g + gr) * kSRow + 16 * th + 8 * n + 2 * tq;
                d0[0] = sacc[n][0] + r0[0];
                d0[1] = sacc[n][1] + r0[1];
                d0[8 * kSRow] = sacc[n][2] + r0[128];
                d0[8 * kSRow + 1] = sacc[n][3] + r0[129];
            }
        }
        named_sync(1 + g, 128);

        // the 16 x 32 score tile in accumulator layout, scaled to base 2, masked
        const int valid = (ntok - i * kNt) < kNt ? (ntok - i * kNt) : kNt;
        float sv[4][4];
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int col = 8 * n + 2 * tq;
            const float* r0 = s_s + (16 * g + gr) * kSRow + col;
            const float* r1 = r0 + 8 * kSRow;
            sv[n][0] = col < valid ? r0[0] * p.scale_log2 : -INFINITY;
            sv[n][1] = col + 1 < valid ? r0[1] * p.scale_log2 : -INFINITY;
            sv[n][2] = col < valid ? r1[0] * p.scale_log2 : -INFINITY;
            sv[n][3] = col + 1 < valid ? r1[1] * p.scale_log2 : -INFINITY;
            mx[0] = fmaxf(mx[0], fmaxf(sv[n][0], sv[n][1]));
            mx[1] = fmaxf(mx[1], fmaxf(sv[n][2], sv[n][3]));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float alpha[2], sum[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float m_new = fmaxf(m_run[r], mx[r]);  // finite: every tile has a valid token
            alpha[r] = ex2(m_run[r] - m_new);            // 0 on the first tile
            m_run[r] = m_new;
        }
        uint32_t pa[4][2];  // probabilities as bf16 pairs, accumulator layout
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const float p0 = ex2(sv[n][0] - m_run[0]), p1 = ex2(sv[n][1] - m_run[0]);
            const float p2 = ex2(sv[n][2] - m_run[1]), p3 = ex2(sv[n][3] - m_run[1]);
            sum[0] += p0 + p1;
            sum[1] += p2 + p3;
            pa[n][0] = pack_bf16(p0, p1);
            pa[n][1] = pack_bf16(p2, p3);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 1);
            sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 2);
            l_run[r] = l_run[r] * alpha[r] + sum[r];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
        }

        // O(16 x 128) += P(16 x 32) * V(32 x 128)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t a0 = pa[2 * kk][0], a1 = pa[2 * kk][1], a2 = pa[2 * kk + 1][0], a3 = pa[2 * kk + 1][1];
            const uint32_t vrow = kt + v_off + kk * 16 * kRow;
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vrow + np * 32, b0, b1, b2, b3);
                mma_bf16(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // every warp is done with this KV buffer and the score tile; all threads
        // stop together once any wait gave up
        if (__syncthreads_or(*abort_flag != 0)) {
            aborted = true;
            break;
        }
        if (threadIdx.x == 0 && i + 2 < ntiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            load_tile(i + 2, buf);
        }
    }
    if (aborted) {  // outputs not valid (status says so); no copy may still land in shared memory
        if (threadIdx.x == 0) {
            (void)mbar_wait_drain(&bars[0], 0, p.wait_ns);
            for (int k = 0; k < 2; ++k)
                if (armed[k] >= 0) (void)mbar_wait_drain(&bars[1 + k], (uint32_t)((armed[k] >> 1) & 1), p.wait_ns);
        }
        return;
    }

    // normalise, round to bf16, store; LSE = m + log2(l), in the requested base
    const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
    uint8_t* const o_r0 = out + (out_row0 + (int64_t)gr * kDv + 128 * q4) * 2;
    uint8_t* const o_r1 = o_r0 + 8 * kDv * 2;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int col = 8 * n + 2 * tq;
        *reinterpret_cast<uint32_t*>(o_r0 + col * 2) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
        *reinterpret_cast<uint32_t*>(o_r1 + col * 2) = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
    }
    if (q4 == 0 && tq == 0) {
        float* l = lse + (int64_t)b * p.H + h0 + 16 * g + gr;
        l[0] = (m_run[0] + log2f(l_run[0])) * p.lse_scale;
        l[8] = (m_run[1] + log2f(l_run[1])) * p.lse_scale;
    }
}

// ---- the tcgen05 kernel -------------------------------------------------------------
//
// The same partials on the 5th-generation tensor cores, transposed so that the
// 128 tokens of a tile sit on the MMA's M (TMEM lanes) and a block of kNH heads
// on its N (TMEM columns):
//   S^T[128 x kNH] = K_tile[128 x Dk] . Q^T          (36 MMAs of K = 16 for Dk = 576)
//   O^T[512 x kNH] += V_tile^T[512 x 128] . P^T      (4 row blocks x 8 MMAs)
// Q and each KV tile arrive by TMA in 128-byte-swizzled 64-wide slices; the KV
// slices serve as the K-major A operand of the scores and, read along the
// latent dims, as the M-major A operand of the values. TMEM holds S^T (kNH
// columns) and O^T (4 x kNH columns). A thread owns one token of the tile and
// its heads (all kNH of them, or a quarter when kNH >= 32: then warp w reads
// TMEM lane quadrant w % 4 for head quarter w / 4). The per-head maxima over the tile
// come from a reduce-scatter butterfly across lanes and shared memory, and the
// running maximum moves only when a head's tile maximum exceeds it by more
// than 2^8 (then O^T is rescaled in TMEM), so the rescale is rare. P^T (bf16)
// is written into the RoPE slice's buffer once the scores are done (into its
// own buffer when Dk = 512). The next tile is prefetched into L2 as soon as
// a tile lands, so its reload streams from L2.

constexpr int kTcTok = 128;                  // tokens per tile
constexpr int kTcAtom = kTcTok * 128;        // one 64-wide slice of 128 token rows (bytes)
constexpr int kTcMiscBytes = 2048;

struct TcParams {
    CUtensorMap tm_q;                 // Q as [B*H rows, Dk], box [64, kNH], 128B swizzle
    CUtensorMap tm_kv[kSlots];        // shard caches as [B*T rows, Dk], box [64, 128], 128B swizzle
    const int* kv_len[kSlots];
    uint8_t* out[kSlots];
    float* lse[kSlots];
    int* status;
    int64_t T;
    int H, n_split;
    float scale_log2;
    float lse_scale;
    int prefetch;                     // 1: bring Q and the first KV tile into L2 before the PDL wait
    long long wait_ns;                // limit of every wait (kWaitLimitNs, or kTestWaitLimitNs)
    int stall;                        // DCP_MLA_FLAG_TEST_STALL: the first tile's barrier expects 16 bytes more
    // The merge in the same launch (dcp_mla_decode when the grid is one wave,
    // launched cooperatively): after a grid-wide sync every warp merges (row,
    // head) units of the gridDim.x partials into destination r = h / Hl.
    int merge;
    int Hl;                           // heads per destination (H / cp)
    float merge_lse_scale;            // LSE differences -> log2 units: 1 or log2(e)
    float merge_log_scale;            // log2(sum) -> the LSE base: 1 or ln 2
    uint8_t* dst[kSlots];             // destination r: [B, Hl, Dv] bf16
    float* lse_out[kSlots];           // destination r's merged LSEs [B, Hl], or null
};

template <int kDk, int kNH>
__host__ __device__ constexpr int tc_smem_bytes() {
    return (kDk / 64) * kTcAtom + (kDk / 64) * kNH * 128 + (kDk == 576 ? 0 : 2 * kNH * 128) + kTcMiscBytes + 1024;
}

// byte offset of element (row, col) in a 128-byte-swizzled slice of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int row, int col) {
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((col * 2) >> 4) ^ (row & 7)) << 4) + ((col * 2) & 15);
}
// shared-memory matrix descriptor: 128-byte swizzle, leading / stride byte offsets
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Bring a box of the tensor into L2 ahead of its load (a hint: no shared
// memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* tm, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// 16 consecutive TMEM columns of this warp's 32 lanes -> 16 registers per thread
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Reduce-scatter across the 32 lanes of a warp: kN values per lane in, the
// reduction (max or sum) over all lanes out, lane l keeping the results for
// heads [h0, h0 + max(kN/32, 1)) with h0 = (l / (32 * max(kN/32, 1) / kN)) * max(kN/32, 1).
template <int kN, int kOff, bool kSum>
struct WarpReduceScatter {
    __device__ __forceinline__ static void run(float* v, int lane) {
        if constexpr (kOff > 0) {
            if constexpr (kN > 1) {
                const bool up = (lane & kOff) != 0;
#pragma unroll
                for (int j = 0; j < kN / 2; ++j) {
                    const float send = up ? v[j] : v[j + kN / 2];
                    const float keep = up ? v[j + kN / 2] : v[j];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, kOff);
                    v[j] = kSum ? keep + recv : fmaxf(keep, recv);
                }
                WarpReduceScatter<kN / 2, kOff / 2, kSum>::run(v, lane);
            } else {
                const float recv = __shfl_xor_sync(0xffffffffu, v[0], kOff);
                v[0] = kSum ? v[0] + recv : fmaxf(v[0], recv);
                WarpReduceScatter<1, kOff / 2, kSum>::run(v, lane);
            }
        }
    }
};

// Per-head reduction over the tile's 128 tokens. Each thread holds v[kHW] for
// heads [hb, hb + kHW) of its token (TMEM lane quadrant `quad`); the kNH
// results land in out[kNH] in shared memory (red is a [4][kNH] scratch area).
template <int kNH, int kHW, bool kSum>
__device__ __forceinline__ void cta_reduce_heads(float* v, int quad, int hb, int lane, float* red, float* out) {
    constexpr int kFinal = kHW / 32 > 1 ? kHW / 32 : 1;
    WarpReduceScatter<kHW, 16, kSum>::run(v, lane);
    const int h0 = (lane / (32 * kFinal / kHW)) * kFinal;
#pragma unroll
    for (int e = 0; e < kFinal; ++e) red[quad * kNH + hb + h0 + e] = v[e];
    __syncthreads();
    if (threadIdx.x < kNH) {
        const int h = threadIdx.x;
        const float a = red[h], b = red[kNH + h], c = red[2 * kNH + h], d = red[3 * kNH + h];
        out[h] = kSum ? (a + b) + (c + d) : fmaxf(fmaxf(a, b), fmaxf(c, d));
    }
    __syncthreads();
}


// The merge of the fused decode, one warp per (row, head) unit, with the same
// arithmetic in the same order as dcp_lse_reduce (so the two paths agree bit
// for bit): m = max of the LSEs, e_j = 2^((l_j - m) * s) (0 for -inf), sum
// over j in order, weights e_j / sum by one reciprocal, fp32 FMAs over the
// sources in order j = 0.. (zero weights skipped), round to bf16; merged LSE
// m + log2(sum) * (1 or ln 2), -inf when every source is -inf.
constexpr int kMergeBatch = 8;  // sources whose payloads are in flight together

__device__ __noinline__ void merge_partials(const TcParams& p, int64_t B) {
    constexpr int kMaxSrc = kSlots;
    const int lane = threadIdx.x & 31;
    const int n_src = (int)gridDim.x;
    const int wpc = (int)(blockDim.x >> 5);
    const int64_t cta = ((int64_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    const int64_t total = (int64_t)gridDim.x * gridDim.y * gridDim.z * wpc;
    const int64_t units = B * p.H;
    for (int64_t u = cta * wpc + (threadIdx.x >> 5); u < units; u += total) {
        const int b = (int)(u / p.H), h = (int)(u - (int64_t)b * p.H);
        const int64_t row = (int64_t)b * p.H + h;
        float l[kMaxSrc], w[kMaxSrc];
#pragma unroll
        for (int j = 0; j < kMaxSrc; ++j) l[j] = (j < n_src) ? ld_cg_f32(p.lse[j] + row) : -INFINITY;
        float mx[kMaxSrc];
#pragma unroll
        for (int j = 0; j < kMaxSrc; ++j) mx[j] = l[j];
#pragma unroll
        for (int half = kMaxSrc / 2; half >= 1; half /= 2)
#pragma unroll
            for (int j = 0; j < half; ++j) mx[j] = fmaxf(mx[j], mx[j + half]);
        const float m = mx[0];
        float merged = -INFINITY;
        if (m == -INFINITY) {
#pragma unroll
            for (int j = 0; j < kMaxSrc; ++j) w[j] = 0.f;
        } else {
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxSrc; ++j) {
                const float e = (l[j] == -INFINITY) ? 0.f : ex2((l[j] - m) * p.merge_lse_scale);
                w[j] = e;
                sum += e;
            }
            const float inv = rcp(sum);
#pragma unroll
            for (int j = 0; j < kMaxSrc; ++j) w[j] *= inv;
            merged = fmaf(lg2(sum), p.merge_log_scale, m);
        }
        float acc[2][8];
#pragma unroll
        for (int v = 0; v < 2; ++v)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[v][e] = 0.f;
#pragma unroll
        for (int jb = 0; jb < kMaxSrc; jb += kMergeBatch) {
            if (jb >= n_src) break;
            uint4 x[kMergeBatch][2];
#pragma unroll
            for (int j = 0; j < kMergeBatch; ++j)
#pragma unroll
                for (int v = 0; v < 2; ++v)
                    x[j][v] = (jb + j < n_src && w[jb + j] != 0.f)
                                  ? ld_cg_v4(p.out[jb + j] + row * (kDv * 2) + v * 512 + lane * 16)
                                  : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < kMergeBatch; ++j) {
                const float wj = w[jb + j];
                if (jb + j < n_src && wj != 0.f) {
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const uint32_t q[4] = {x[j][v].x, x[j][v].y, x[j][v].z, x[j][v].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[v][2 * e] = fmaf(wj, __uint_as_float(q[e] << 16), acc[v][2 * e]);
                            acc[v][2 * e + 1] = fmaf(wj, __uint_as_float(q[e] & 0xffff0000u), acc[v][2 * e + 1]);
                        }
                    }
                }
            }
        }
        const int r = h / p.Hl, i = h - r * p.Hl;
        uint8_t* const dst = p.dst[r] + ((int64_t)b * p.Hl + i) * (kDv * 2);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            uint4 o;
            o.x = pack_bf16(acc[v][0], acc[v][1]);
            o.y = pack_bf16(acc[v][2], acc[v][3]);
            o.z = pack_bf16(acc[v][4], acc[v][5]);
            o.w = pack_bf16(acc[v][6], acc[v][7]);
            *reinterpret_cast<uint4*>(dst + v * 512 + lane * 16) = o;
        }
        if (lane == 0 && p.lse_out[r] != nullptr) p.lse_out[r][(int64_t)b * p.Hl + i] = merged;
    }
}

// Threads of the tcgen05 kernel: one per (token, group of heads); with 32 or
// more heads per CTA each token's heads are split over four threads (512
// threads, at most 128 registers each). The softmax and the epilogue are
// latency chains over a thread's heads, so shorter chains on more warps run
// faster; eight groups would spill.
template <int kNH>
__host__ __device__ constexpr int tc_head_groups() { return kNH >= 32 ? 4 : 1; }

template <int kDk, int kNH>
__global__ void __launch_bounds__(128 * tc_head_groups<kNH>(), 1) mla_partial_tc_kernel(const __grid_constant__ TcParams p) {
    constexpr int kHW = kNH / tc_head_groups<kNH>();  // heads per thread
    constexpr int kAtoms = kDk / 64;            // 64-wide slices of a row: 9 (Dk 576) or 8 (Dk 512)
    constexpr int kQAtom = kNH * 128;           // bytes of one Q slice
    constexpr bool kPInRope = kAtoms == 9;      // P^T reuses the RoPE slice's buffer
    constexpr uint32_t kCols = 512;             // TMEM columns: S^T [0, kNH), O^T [kNH, 5 kNH)
    constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kNH >> 3) << 17) |
                                 ((uint32_t)(kTcTok >> 4) << 24);  // fp32 += bf16 x bf16, both K-major
    constexpr uint32_t kIdescO = kIdescS | (1u << 15);             // A read M-major
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* const kv_s = smem;
    uint8_t* const q_s = kv_s + kAtoms * kTcAtom;
    uint8_t* const p_s = kPInRope ? kv_s + 8 * kTcAtom : q_s + kAtoms * kQAtom;
    uint8_t* const misc = kPInRope ? q_s + kAtoms * kQAtom : p_s + 2 * kQAtom;
    uint64_t* const bar_q = reinterpret_cast<uint64_t*>(misc);
    uint64_t* const bar_kv = bar_q + 1;                      // a KV tile has landed
    uint64_t* const bar_s = bar_q + 2;                       // score MMAs of a tile done
    uint64_t* const bar_o = bar_q + 3;                       // value MMAs of a tile done
    uint32_t* const tslot = reinterpret_cast<uint32_t*>(misc + 32);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 36);
    int* const armed = reinterpret_cast<int*>(misc + 40);   // [4]: last tile each barrier was armed for
    float* const red = reinterpret_cast<float*>(misc + 128); // [4][kNH]
    float* const m_s = red + 4 * kNH;                        // running max per head (base-2 units)
    float* const a_s = m_s + kNH;                            // this tile's rescale factor per head
    float* const t_s = a_s + kNH;                            // tile max, then the final sums
    static_assert(128 + 7 * kNH * 4 <= kTcMiscBytes, "misc area");
    constexpr int kArmQ = 0, kArmKv = 1, kArmS = 2, kArmO = 3;  // indices into armed[]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = blockIdx.x;
    const int shard = slot / p.n_split;
    const int split = slot - shard * p.n_split;
    const int h0 = blockIdx.y * kNH;
    const int b = blockIdx.z;

    // set-up that reads no input overlaps the previous kernel
    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(bar_kv, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_q)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_kv[shard])) : "memory");
    }
    if (tid < 4) armed[tid] = -1;
    if (tid == 4) *abort_flag = 0;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid < kNH) m_s[tid] = -INFINITY;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // warp w reads TMEM lane quadrant w % 4 (tokens 32(w%4) .. +31) and
    // handles heads [hb, hb + kHW) of those tokens
    const int quad = warp & 3, tok = tid & 127, hb = (warp >> 2) * kHW;
    const uint32_t tlane = (uint32_t)(32 * quad) << 16;

    // With DCP_FLAG_PREFETCH, Q and the split's first KV tile are brought into
    // L2 before the wait (a hint, so the loads after the wait still see what the
    // previous kernel wrote). The split's start needs kv_len, an input: the
    // prefetch takes the value before the wait, and a stale one only prefetches
    // other rows.
    if (p.prefetch && tid == 32) {
        int64_t len0 = p.kv_len[shard][b];
        len0 = len0 < 0 ? 0 : (len0 > p.T ? p.T : len0);
        const int64_t t0 = (int64_t)split * ((len0 + p.n_split - 1) / p.n_split);
        if (t0 < len0) {
            for (int a = 0; a < kAtoms; ++a) {
                tma_prefetch_2d(&p.tm_q, a * 64, b * p.H + h0);
                tma_prefetch_2d(&p.tm_kv[shard], a * 64, (int)((int64_t)b * p.T + t0));
            }
        }
    }

    pdl_wait();
    pdl_launch_dependents();

    int64_t len = p.kv_len[shard][b];
    len = len < 0 ? 0 : (len > p.T ? p.T : len);
    const int64_t chunk = (len + p.n_split - 1) / p.n_split;
    const int64_t t_begin = (int64_t)split * chunk;
    const int64_t t_end = t_begin + chunk < len ? t_begin + chunk : len;
    const int ntok = t_end > t_begin ? (int)(t_end - t_begin) : 0;
    uint8_t* const out = p.out[slot];
    float* const lse = p.lse[slot];
    const int64_t out_row0 = ((int64_t)b * p.H + h0) * kDv;
    bool aborted = false;  // CTA-uniform: decided by barrier votes

    if (ntok == 0) {  // empty range: output 0, LSE -inf
        for (int i = tid; i < kNH * kDv / 8; i += (int)blockDim.x)
            reinterpret_cast<uint4*>(out + out_row0 * 2)[i] = make_uint4(0u, 0u, 0u, 0u);
        if (tid < kNH) lse[(int64_t)b * p.H + h0 + tid] = -INFINITY;
    } else {
        const int ntiles = (ntok + kTcTok - 1) / kTcTok;
        const int row0 = (int)((int64_t)b * p.T + t_begin);
        if (tid == 0) {
            mbar_expect_tx(bar_q, (uint32_t)(kAtoms * kQAtom));
            for (int a = 0; a < kAtoms; ++a) tma_load_2d(q_s + a * kQAtom, &p.tm_q, a * 64, b * p.H + h0, bar_q);
            armed[kArmQ] = 0;
            // (with the stall test, the first tile's barrier waits for 16 bytes that never come)
            mbar_expect_tx(bar_kv, (uint32_t)(kAtoms * kTcAtom) + (p.stall ? 16u : 0u));
            for (int a = 0; a < kAtoms; ++a) tma_load_2d(kv_s + a * kTcAtom, &p.tm_kv[shard], a * 64, row0, bar_kv);
            armed[kArmKv] = 0;
        }
        float l_part[kHW];  // this thread's token's share of each of its heads' sums
#pragma unroll
        for (int h = 0; h < kHW; ++h) l_part[h] = 0.f;
        (void)mbar_wait_cta(bar_q, 0, abort_flag, p.status, p.wait_ns);

        for (int i = 0; i < ntiles; ++i) {
            // Stop at a tile boundary, all threads together, once any wait gave up.
            if (__syncthreads_or(*abort_flag != 0)) {
                aborted = true;
                break;
            }
            const uint32_t ph = (uint32_t)(i & 1);
            (void)mbar_wait_cta(bar_kv, ph, abort_flag, p.status, p.wait_ns);
            // Start the next tile's DRAM reads now, into L2 (from a thread of another
            // warp than the MMA issuer's), so that its load after this tile's value
            // MMAs streams from L2: every CTA reloads at about the same moment, and
            // from DRAM those loads contend.
            if (tid == 32 && i + 1 < ntiles)
                for (int a = 0; a < kAtoms; ++a) tma_prefetch_2d(&p.tm_kv[shard], a * 64, row0 + (i + 1) * kTcTok);
            if (tid == 0 && !*abort_flag) {  // scores: S^T = K_tile . Q^T
                tc_fence_after();
#pragma unroll 1
                for (int a = 0; a < kAtoms; ++a) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc(smem_u32(kv_s + a * kTcAtom) + kk * 32, 16, 1024);
                        const uint64_t bd = smem_desc(smem_u32(q_s + a * kQAtom) + kk * 32, 16, 1024);
                        umma_f16(tmem, ad, bd, kIdescS, (a | kk) != 0);
                    }
                }
                umma_commit(bar_s);
                armed[kArmS] = i;
            }
            (void)mbar_wait_cta(bar_s, ph, abort_flag, p.status, p.wait_ns);
            tc_fence_after();

            float sv[kHW];
#pragma unroll
            for (int c = 0; c < kHW; c += 16) tmem_ld16(tmem + tlane + hb + c, sv + c);
            tmem_wait_ld();
            const int valid = (ntok - i * kTcTok) < kTcTok ? (ntok - i * kTcTok) : kTcTok;
            const bool live = tok < valid;
#pragma unroll
            for (int h = 0; h < kHW; ++h) sv[h] = live ? sv[h] * p.scale_log2 : -INFINITY;
            // A token past the range gets probability 0. Inside the row's first len
            // cache rows it is another split's token, finite, and adds 0 x V = 0; a
            // row at or past len may hold anything (NaN), so its value row is zeroed.
            // (Chunk order rotated by token: the rows of a warp's tokens lie 128 bytes
            // apart, on the same banks.)
            if (t_begin + (int64_t)i * kTcTok + tok >= len) {
                constexpr int kPerGroup = 8 / tc_head_groups<kNH>();  // latent slices zeroed per thread
#pragma unroll 1
                for (int a = (warp >> 2) * kPerGroup; a < (warp >> 2) * kPerGroup + kPerGroup; ++a) {
                    uint4* row = reinterpret_cast<uint4*>(kv_s + a * kTcAtom + (tok >> 3) * 1024 + (tok & 7) * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) row[(c + tok) & 7] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // The running max moves only when some head's tile max exceeds it by more
            // than 2^8, i.e. when some score does: each thread checks its own, and only
            // then (rarely, after the first tile) are the exact tile maxima reduced.
            bool over = false;
#pragma unroll
            for (int h = 0; h < kHW; h += 4) {
                const float4 mv = *reinterpret_cast<const float4*>(m_s + hb + h);
                over |= (sv[h] > mv.x + 8.f) | (sv[h + 1] > mv.y + 8.f) | (sv[h + 2] > mv.z + 8.f) |
                        (sv[h + 3] > mv.w + 8.f);
            }
            const int any = __syncthreads_or(over);
            if (any) {
                float mx[kHW];
#pragma unroll
                for (int h = 0; h < kHW; ++h) mx[h] = sv[h];
                cta_reduce_heads<kNH, kHW, false>(mx, quad, hb, lane, red, t_s);
                if (tid < kNH) {
                    const float mn = fmaxf(m_s[tid], t_s[tid]);
                    a_s[tid] = ex2(m_s[tid] - mn);
                    m_s[tid] = mn;
                }
                __syncthreads();
            }
            if (any && i > 0) {  // rescale O^T (the previous tile's value MMAs are done)
                (void)mbar_wait_cta(bar_o, (uint32_t)((i - 1) & 1), abort_flag, p.status, p.wait_ns);
                tc_fence_after();
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int c = hb; c < hb + kHW; c += 16) {
                        float ov[16];
                        tmem_ld16(tmem + tlane + kNH + m * kNH + c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) ov[j] *= a_s[c + j];
                        tmem_st16(tmem + tlane + kNH + m * kNH + c, ov);
                    }
                }
                tmem_wait_st();
            }
            // probabilities, this thread's share of the sums, and P^T (bf16, K-major over tokens)
            // (the shared reads all come before the stores, so none waits behind one)
            {
#pragma unroll
                for (int h = 0; h < kHW; h += 4) {
                    const float4 mv = *reinterpret_cast<const float4*>(m_s + hb + h);
                    sv[h] = ex2(sv[h] - mv.x);
                    sv[h + 1] = ex2(sv[h + 1] - mv.y);
                    sv[h + 2] = ex2(sv[h + 2] - mv.z);
                    sv[h + 3] = ex2(sv[h + 3] - mv.w);
                }
                if (any) {
#pragma unroll
                    for (int h = 0; h < kHW; h += 4) {
                        const float4 av = *reinterpret_cast<const float4*>(a_s + hb + h);
                        l_part[h] = l_part[h] * av.x + sv[h];
                        l_part[h + 1] = l_part[h + 1] * av.y + sv[h + 1];
                        l_part[h + 2] = l_part[h + 2] * av.z + sv[h + 2];
                        l_part[h + 3] = l_part[h + 3] * av.w + sv[h + 3];
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < kHW; ++h) l_part[h] += sv[h];
                }
                // P^T row h holds head h over the tile's tokens. Neighbouring lanes hold
                // neighbouring tokens: they swap one value per pair of heads, so each
                // lane converts and stores two tokens of one head in one 4-byte word
                // (the even lane head h, the odd lane head h + 1).
                uint8_t* const prow = p_s + (tok >> 6) * kQAtom;
                const int tl = tok & 62;  // the pair's first token
                const bool odd = (lane & 1) != 0;
#pragma unroll
                for (int h = 0; h < kHW; h += 2) {
                    const float give = odd ? sv[h] : sv[h + 1];
                    const float got = __shfl_xor_sync(0xffffffffu, give, 1);
                    const int hh = hb + h + (odd ? 1 : 0);
                    const __nv_bfloat162 v = odd ? __floats2bfloat162_rn(got, sv[h + 1]) : __floats2bfloat162_rn(sv[h], got);
                    *reinterpret_cast<__nv_bfloat162*>(prow + sw128(hh, tl)) = v;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            __syncthreads();
            if (tid == 0 && !*abort_flag) {  // values: O^T += V_tile^T . P^T, four 128-row blocks of the 512 latent dims
                tc_fence_after();
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = smem_desc(smem_u32(kv_s + 2 * m * kTcAtom) + kk * 2048, kTcAtom, 1024);
                        const uint64_t bd = smem_desc(smem_u32(p_s + (kk >> 2) * kQAtom) + (kk & 3) * 32, 16, 1024);
                        umma_f16(tmem + kNH + m * kNH, ad, bd, kIdescO, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                umma_commit(bar_o);
                armed[kArmO] = i;
                // the next tile reuses every buffer once these MMAs are done
                if (i + 1 < ntiles && mbar_wait_cta(bar_o, ph, abort_flag, p.status, p.wait_ns)) {
                    mbar_expect_tx(bar_kv, (uint32_t)(kAtoms * kTcAtom));
                    for (int a = 0; a < kAtoms; ++a)
                        tma_load_2d(kv_s + a * kTcAtom, &p.tm_kv[shard], a * 64, row0 + (i + 1) * kTcTok, bar_kv);
                    armed[kArmKv] = i + 1;
                }
            }
        }

        if (!aborted) {
            // final sums, then normalise, round to bf16 and store; LSE = m + log2(l)
            (void)mbar_wait_cta(bar_o, (uint32_t)((ntiles - 1) & 1), abort_flag, p.status, p.wait_ns);
            aborted = __syncthreads_or(*abort_flag != 0) != 0;
        }
        if (!aborted) {
            tc_fence_after();
            cta_reduce_heads<kNH, kHW, true>(l_part, quad, hb, lane, red, t_s);
            if (tid < kNH) a_s[tid] = 1.0f / t_s[tid];  // one reciprocal per head, then products
            __syncthreads();
            // The [kNH, 512] output tile is assembled in the KV buffer (free now:
            // every MMA is done and no load is pending), then leaves in one bulk
            // copy: rows h0 .. h0+kNH-1 of out[b] are contiguous.
            __nv_bfloat16* const o_s = reinterpret_cast<__nv_bfloat16*>(kv_s);
            // This thread's latent dim of each 128-row block, all its heads: every
            // TMEM load issued before one wait.
            float ov[4][kHW];
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int c = 0; c < kHW; c += 16) tmem_ld16(tmem + tlane + kNH + m * kNH + hb + c, ov[m] + c);
            tmem_wait_ld();
            // lane = latent dim: neighbouring lanes swap one value per pair of heads,
            // so each lane converts and stores two dims of one head in one word
            const bool odd = (lane & 1) != 0;
#pragma unroll
            for (int j = 0; j < kHW; j += 2) {
                const float2 inv = *reinterpret_cast<const float2*>(a_s + hb + j);  // read once per head pair
                const int hh = hb + j + (odd ? 1 : 0);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int dv = 128 * m + 32 * quad + (lane & ~1);  // the pair's first dim
                    const float x0 = ov[m][j] * inv.x, x1 = ov[m][j + 1] * inv.y;
                    const float got = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
                    *reinterpret_cast<__nv_bfloat162*>(o_s + hh * kDv + dv) =
                        odd ? __floats2bfloat162_rn(got, x1) : __floats2bfloat162_rn(x0, got);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (tid == 0) {
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(out + out_row0 * 2),
                             "r"(smem_u32(o_s)), "r"((uint32_t)(kNH * kDv * 2))
                             : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            if (tid < kNH) lse[(int64_t)b * p.H + h0 + tid] = (m_s[tid] + log2f(t_s[tid])) * p.lse_scale;
            // before the CTA leaves, the copy must have read the tile out of shared
            // memory (its global writes are visible to later kernels once this grid
            // completes); when this grid merges the partials itself, the writes
            // must be complete and ordered before the grid-wide sync
            if (tid == 0) {
                if (p.merge) {
                    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                } else {
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                }
            }
        }
    }
    if (aborted) {
        // A wait gave up (the status word says so; the outputs are not valid).
        // Before TMEM is freed and the CTA leaves, wait (bounded) for every copy
        // and MMA this CTA armed, so none still writes into its shared memory or
        // TMEM.
        __syncthreads();
        if (tid == 0) {
            if (armed[kArmQ] >= 0) (void)mbar_wait_drain(bar_q, 0, p.wait_ns);
            if (armed[kArmKv] >= 0) (void)mbar_wait_drain(bar_kv, (uint32_t)(armed[kArmKv] & 1), p.wait_ns);
            if (armed[kArmS] >= 0) (void)mbar_wait_drain(bar_s, (uint32_t)(armed[kArmS] & 1), p.wait_ns);
            if (armed[kArmO] >= 0) (void)mbar_wait_drain(bar_o, (uint32_t)(armed[kArmO] & 1), p.wait_ns);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
    if (p.merge) {
        // Every CTA reaches this point (each of its waits is bounded and an
        // aborted CTA comes here too) and a cooperative launch keeps every CTA
        // resident, so the grid-wide sync completes.
        __threadfence();
        cooperative_groups::this_grid().sync();
        merge_partials(p, (int64_t)gridDim.z);
    }
}

// ---- host side -----------------------------------------------------------------

template <int kDk, int kG>
cudaError_t launch(const Params& prm, int64_t B, int n_slots, unsigned flags, cudaStream_t stream) {
    constexpr int bytes = smem_bytes<kDk, kG>();
    // The shared-memory opt-in is a per-device attribute of the kernel: set it
    // once per device (setting it again is harmless, so racing callers are fine).
    static int configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(mla_partial_kernel<kDk, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_slots, (unsigned)(prm.H / (16 * kG)), (unsigned)B);
    cfg.blockDim = dim3(128 * kG, 1, 1);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & kFlagPdl) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_partial_kernel<kDk, kG>, prm);
}

template <int kDk>
cudaError_t launch_dk(const Params& prm, int64_t B, int n_slots, unsigned flags, cudaStream_t stream) {
    if (prm.H % 64 == 0) return launch<kDk, 4>(prm, B, n_slots, flags, stream);
    if (prm.H % 32 == 0) return launch<kDk, 2>(prm, B, n_slots, flags, stream);
    return launch<kDk, 1>(prm, B, n_slots, flags, stream);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// cuTensorMapEncodeTiled, from the driver through the runtime (no link to libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            (void)cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A [rows, Dk] bf16 matrix read in [box_rows, 64] boxes with 128-byte swizzle.
bool encode_rows(CUtensorMap* tm, const void* base, int Dk, uint64_t rows, uint32_t box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)Dk, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)Dk * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estride[2] = {1u, 1u};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kDk, int kNH>
cudaError_t launch_tc(const TcParams& prm, int64_t B, int n_slots, unsigned flags, cudaStream_t stream) {
    constexpr int bytes = tc_smem_bytes<kDk, kNH>();
    static int configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(mla_partial_tc_kernel<kDk, kNH>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_slots, (unsigned)(prm.H / kNH), (unsigned)B);
    cfg.blockDim = dim3(128 * tc_head_groups<kNH>(), 1, 1);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (flags & kFlagPdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (prm.merge) {  // the grid-wide sync needs every CTA resident at once
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<kDk, kNH>, prm);
}

// CTAs of the tcgen05 kernel that can be resident at once on the device (the
// limit of a cooperative launch).
template <int kDk, int kNH>
int64_t tc_resident_ctas() {
    constexpr int bytes = tc_smem_bytes<kDk, kNH>();
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (cudaFuncSetAttribute(mla_partial_tc_kernel<kDk, kNH>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mla_partial_tc_kernel<kDk, kNH>,
                                                      128 * tc_head_groups<kNH>(), bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return (int64_t)sms * per_sm;
}

template <int kDk>
int64_t tc_resident_ctas_dk(int H) {
    if (H % 64 == 0) return tc_resident_ctas<kDk, 64>();
    if (H % 32 == 0) return tc_resident_ctas<kDk, 32>();
    return tc_resident_ctas<kDk, 16>();
}

template <int kDk>
cudaError_t launch_tc_dk(const TcParams& prm, int64_t B, int n_slots, unsigned flags, cudaStream_t stream) {
    if (prm.H % 64 == 0) return launch_tc<kDk, 64>(prm, B, n_slots, flags, stream);
    if (prm.H % 32 == 0) return launch_tc<kDk, 32>(prm, B, n_slots, flags, stream);
    return launch_tc<kDk, 16>(prm, B, n_slots, flags, stream);
}

}  // namespace

extern "C" int dcp_mla_decode_smem_bytes(int Dk, int H) {
    if ((Dk != 512 && Dk != 576) || H < 16 || H % 16 != 0) return -1;
    const int g = H % 64 == 0 ? 4 : (H % 32 == 0 ? 2 : 1);
    const int mma = Dk == 576 ? (g == 4 ? smem_bytes<576, 4>() : (g == 2 ? smem_bytes<576, 2>() : smem_bytes<576, 1>()))
                              : (g == 4 ? smem_bytes<512, 4>() : (g == 2 ? smem_bytes<512, 2>() : smem_bytes<512, 1>()));
    const int tc = Dk == 576 ? (g == 4 ? tc_smem_bytes<576, 64>() : (g == 2 ? tc_smem_bytes<576, 32>() : tc_smem_bytes<576, 16>()))
                             : (g == 4 ? tc_smem_bytes<512, 64>() : (g == 2 ? tc_smem_bytes<512, 32>() : tc_smem_bytes<512, 16>()));
    return mma > tc ? mma : tc;
}

namespace {

bool tc_is_default(int H, int64_t tokens_per_split) {
    if (H % 64 == 0) return tokens_per_split >= kTcMinTokensH64;
    if (H % 32 == 0) return tokens_per_split >= kTcMinTokensH32;
    return false;
}

}  // namespace

extern "C" int dcp_mla_decode_kernel(int H, int64_t T, int n_split, unsigned flags) {
    if (H < 16 || H % 16 != 0 || T < 0) return DCP_MLA_ERR_BAD_SHAPE;
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if ((flags & ~(kFlagPdl | kFlagPrefetch | kFlagMmaSync | kFlagTcgen05 | kFlagTestStall)) != 0)
        return DCP_MLA_ERR_BAD_FLAGS;
    if ((flags & kFlagMmaSync) && (flags & kFlagTcgen05)) return DCP_MLA_ERR_BAD_FLAGS;
    if (flags & kFlagTcgen05) return DCP_MLA_KERNEL_TCGEN05;
    if (flags & kFlagMmaSync) return DCP_MLA_KERNEL_MMA_SYNC;
    return tc_is_default(H, (T + n_split - 1) / n_split) ? DCP_MLA_KERNEL_TCGEN05 : DCP_MLA_KERNEL_MMA_SYNC;
}

// CTAs of the mma.sync kernel that fit on one SM (shared memory bound, Dk = 576)
static int mma_ctas_per_sm(int H) {
    constexpr int kSmemPerSm = 228 * 1024, kReserve = 1024;
    const int bytes = H % 64 == 0 ? smem_bytes<576, 4>() : (H % 32 == 0 ? smem_bytes<576, 2>() : smem_bytes<576, 1>());
    const int n = kSmemPerSm / (bytes + kReserve);
    return n > 0 ? n : 1;
}

extern "C" int dcp_mla_decode_pick_split(int cp, int64_t B, int H, int64_t T, int num_sms) {
    if (B < 0 || B > 65535 || T < 0 || H < 16 || H % 16 != 0 || num_sms < 1) return DCP_MLA_ERR_BAD_SHAPE;
    if (cp < 1 || cp > DCP_MLA_SPLIT_MAX || H % cp != 0) return DCP_MLA_ERR_BAD_CP;
    const int64_t blocks = H % 64 == 0 ? H / 64 : (H % 32 == 0 ? H / 32 : H / 16);  // head blocks per row
    const int64_t per_split = (int64_t)cp * blocks * (B > 0 ? B : 1);                // CTAs per split count
    int best = 1;
    for (int n = 2; n * cp <= DCP_MLA_SPLIT_MAX; ++n) {
        const int64_t tokens = (T + n - 1) / n;
        if (tokens < kTcTok) break;                          // at least one 128-token tile per split
        // one wave: one tcgen05 CTA per SM, or as many mma.sync CTAs as fit
        const int64_t wave = (int64_t)num_sms * (tc_is_default(H, tokens) ? 1 : mma_ctas_per_sm(H));
        if (per_split * n > wave) continue;
        if (H % (cp * n) == 0) best = n;                     // the fused merge needs H / (cp * n) heads per source
    }
    return best;
}

namespace {

// The shapes the producer takes (DCP_MLA_ERR_BAD_SHAPE otherwise).
bool shape_ok(int64_t B, int H, int Dk, int Dv, int64_t T) {
    return B >= 0 && B <= 65535 && T >= 0 && H >= 16 && H % 16 == 0 && (Dk == 512 || Dk == 576) && Dv == kDv;
}

// Validate and launch the producer over n_shard shards x n_split splits
// (slot = shard * n_split + split), all in one grid.
// The merge a producer launch may finish with (dcp_mla_decode): cp
// destinations of H / cp heads each.
struct MergeInto {
    void* const* dst;
    float* const* lse_out;
    int cp;
};

// 1 if the producer ran and merged (out == 1), 0 if it ran without merging.
int producer(const void* q, const void* const* kv_ptrs, const int32_t* const* kv_len_ptrs, int n_shard, int64_t B,
             int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e, int n_split, void* const* out_ptrs,
             float* const* lse_ptrs, int32_t* status, unsigned flags, void* stream, const MergeInto* merge = nullptr,
             int* merged = nullptr) {
    if (merged != nullptr) *merged = 0;
    if (q == nullptr || kv_ptrs == nullptr || kv_len_ptrs == nullptr || out_ptrs == nullptr || lse_ptrs == nullptr)
        return DCP_MLA_ERR_NULL_POINTER;
    if (!shape_ok(B, H, Dk, Dv, T)) return DCP_MLA_ERR_BAD_SHAPE;
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if (n_shard < 1 || n_shard * n_split > kSlots) return DCP_MLA_ERR_BAD_CP;
    if ((flags & ~(kFlagPdl | kFlagPrefetch | kFlagMmaSync | kFlagTcgen05 | kFlagTestStall)) != 0)
        return DCP_MLA_ERR_BAD_FLAGS;
    if ((flags & kFlagMmaSync) && (flags & kFlagTcgen05)) return DCP_MLA_ERR_BAD_FLAGS;
    if (!aligned(q, 16) || (status != nullptr && !aligned(status, 4))) return DCP_MLA_ERR_MISALIGNED;
    Params prm;
    for (int k = 0; k < kSlots; ++k) {
        prm.kv[k] = nullptr;
        prm.kv_len[k] = nullptr;
        prm.out[k] = nullptr;
        prm.lse[k] = nullptr;
    }
    for (int j = 0; j < n_shard; ++j) {
        if (kv_ptrs[j] == nullptr || kv_len_ptrs[j] == nullptr) return DCP_MLA_ERR_NULL_POINTER;
        if (!aligned(kv_ptrs[j], 16) || !aligned(kv_len_ptrs[j], 4)) return DCP_MLA_ERR_MISALIGNED;
        prm.kv[j] = static_cast<const uint8_t*>(kv_ptrs[j]);
        prm.kv_len[j] = kv_len_ptrs[j];
    }
    const int n_slots = n_shard * n_split;
    for (int k = 0; k < n_slots; ++k) {
        if (out_ptrs[k] == nullptr || lse_ptrs[k] == nullptr) return DCP_MLA_ERR_NULL_POINTER;
        if (!aligned(out_ptrs[k], 16) || !aligned(lse_ptrs[k], 4)) return DCP_MLA_ERR_MISALIGNED;
        prm.out[k] = static_cast<uint8_t*>(out_ptrs[k]);
        prm.lse[k] = lse_ptrs[k];
    }
    if (B == 0) return 0;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool use_tc = dcp_mla_decode_kernel(H, T, n_split, flags) == DCP_MLA_KERNEL_TCGEN05;
    if (use_tc) {  // the tcgen05 kernel
        TcParams tp;
        const int nh = H % 64 == 0 ? 64 : (H % 32 == 0 ? 32 : 16);
        if (!encode_rows(&tp.tm_q, q, Dk, (uint64_t)B * H, (uint32_t)nh)) return DCP_MLA_ERR_TENSOR_MAP;
        const uint64_t kv_rows = (uint64_t)B * (uint64_t)T > 0 ? (uint64_t)B * (uint64_t)T : 1;
        if (kv_rows > 0x7fffffffull) return DCP_MLA_ERR_BAD_SHAPE;
        for (int j = 0; j < kSlots; ++j) {
            tp.kv_len[j] = prm.kv_len[j];
            tp.out[j] = prm.out[j];
            tp.lse[j] = prm.lse[j];
            if (j < n_shard) {
                if (!encode_rows(&tp.tm_kv[j], kv_ptrs[j], Dk, kv_rows, (uint32_t)kTcTok)) return DCP_MLA_ERR_TENSOR_MAP;
            } else {
                tp.tm_kv[j] = tp.tm_q;
            }
        }
        tp.status = status;
        tp.T = T;
        tp.H = H;
        tp.n_split = n_split;
        tp.scale_log2 = scale * 1.4426950408889634f;
        tp.lse_scale = lse_base_e ? 0.6931471805599453f : 1.0f;
        tp.prefetch = (flags & kFlagPrefetch) ? 1 : 0;
        tp.wait_ns = (flags & kFlagTestStall) ? kTestWaitLimitNs : kWaitLimitNs;
        tp.stall = (flags & kFlagTestStall) ? 1 : 0;
        tp.merge = 0;
        tp.Hl = H;
        tp.merge_lse_scale = lse_base_e ? 1.4426950408889634f : 1.0f;
        tp.merge_log_scale = lse_base_e ? 0.6931471805599453f : 1.0f;
        for (int j = 0; j < kSlots; ++j) {
            tp.dst[j] = nullptr;
            tp.lse_out[j] = nullptr;
        }
        // The merge joins this launch when the grid fits in one resident wave
        // (a cooperative launch then keeps every CTA resident for the grid-wide
        // sync); otherwise the caller launches the merge separately.
        if (merge != nullptr) {
            const int64_t ctas = (int64_t)n_slots * (H / (H % 64 == 0 ? 64 : (H % 32 == 0 ? 32 : 16))) * B;
            const int64_t resident = Dk == 576 ? tc_resident_ctas_dk<576>(H) : tc_resident_ctas_dk<512>(H);
            if (ctas <= resident && merge->cp <= kSlots) {
                tp.merge = 1;
                tp.Hl = H / merge->cp;
                for (int j = 0; j < merge->cp; ++j) {
                    tp.dst[j] = static_cast<uint8_t*>(merge->dst[j]);
                    tp.lse_out[j] = merge->lse_out != nullptr ? merge->lse_out[j] : nullptr;
                }
            }
        }
        const cudaError_t e = Dk == 576 ? launch_tc_dk<576>(tp, B, n_slots, flags & kFlagPdl, st)
                                        : launch_tc_dk<512>(tp, B, n_slots, flags & kFlagPdl, st);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return (int)e;
        }
        if (merged != nullptr) *merged = tp.merge;
        return 0;
    }
    prm.q = static_cast<const uint8_t*>(q);
    prm.status = status;
    prm.T = T;
    prm.H = H;
    prm.n_split = n_split;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.lse_scale = lse_base_e ? 0.6931471805599453f : 1.0f;
    prm.wait_ns = (flags & kFlagTestStall) ? kTestWaitLimitNs : kWaitLimitNs;
    prm.stall = (flags & kFlagTestStall) ? 1 : 0;
    const cudaError_t e = Dk == 576 ? launch_dk<576>(prm, B, n_slots, flags & kFlagPdl, st)
                                    : launch_dk<512>(prm, B, n_slots, flags & kFlagPdl, st);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    return 0;
}

constexpr int64_t kWsAlign = 256;
int64_t round_up(int64_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

}  // namespace

extern "C" int dcp_mla_decode_partial(const void* q, const void* kv, const int32_t* kv_len,
                                      int64_t B, int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e,
                                      int n_split, void* const* out_ptrs, float* const* lse_ptrs,
                                      int32_t* status, unsigned flags, void* stream) {
    if (kv == nullptr || kv_len == nullptr) return DCP_MLA_ERR_NULL_POINTER;
    const void* kvp[1] = {kv};
    const int32_t* lenp[1] = {kv_len};
    return producer(q, kvp, lenp, 1, B, H, Dk, Dv, T, scale, lse_base_e, n_split, out_ptrs, lse_ptrs, status, flags,
                    stream);
}

extern "C" int64_t dcp_mla_decode_workspace_bytes(int cp, int n_split, int64_t B, int H, int Dv) {
    if (cp < 1 || n_split < 1 || B < 0 || H < 1 || Dv < 1 || B > (int64_t(1) << 31)) return -1;
    const int64_t n = (int64_t)cp * n_split;
    return n * (round_up(B * H * (int64_t)Dv * 2) + round_up(B * H * 4));
}

extern "C" int dcp_mla_decode(const void* q, const void* const* kv_ptrs, const int32_t* const* kv_len_ptrs, int cp,
                              int64_t B, int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e, int n_split,
                              void* workspace, int64_t workspace_bytes, void* const* dst_ptrs,
                              float* const* lse_out_ptrs, int32_t* status, unsigned flags, void* stream) {
    if (kv_ptrs == nullptr || kv_len_ptrs == nullptr || dst_ptrs == nullptr) return DCP_MLA_ERR_NULL_POINTER;
    if (!shape_ok(B, H, Dk, Dv, T)) return DCP_MLA_ERR_BAD_SHAPE;
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if (cp < 1 || cp * n_split > DCP_LSE_REDUCE_CP_MAX || H % (cp * n_split) != 0) return DCP_MLA_ERR_BAD_CP;
    const int64_t need = dcp_mla_decode_workspace_bytes(cp, n_split, B, H, Dv);
    if (need < 0) return DCP_MLA_ERR_BAD_SHAPE;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) != 0 ||
        workspace_bytes < need)
        return DCP_MLA_ERR_WORKSPACE;
    for (int j = 0; j < cp; ++j)
        if (dst_ptrs[j] == nullptr) return DCP_MLA_ERR_NULL_POINTER;
    const int n_src = cp * n_split;
    const int64_t out_bytes = round_up(B * H * (int64_t)Dv * 2), lse_bytes = round_up(B * H * 4);
    uint8_t* const ws = static_cast<uint8_t*>(workspace);
    // partials of shard j, split s in slot j*n_split + s: outputs first, then LSEs
    void* part_out[kSlots];
    float* part_lse[kSlots];
    for (int k = 0; k < n_src; ++k) {
        part_out[k] = ws + k * out_bytes;
        part_lse[k] = reinterpret_cast<float*>(ws + n_src * out_bytes + k * lse_bytes);
    }
    // With DCP_MLA_FLAG_ONE_KERNEL, and when the producer's grid is one wave of
    // tcgen05 CTAs, the merge runs in the producer's launch after a grid-wide
    // sync; otherwise the producer and the merge are two launches.
    const bool one = (flags & kFlagOneKernel) != 0;
    for (int j = 0; j < cp; ++j)
        if (!aligned(dst_ptrs[j], 16) || (lse_out_ptrs != nullptr && lse_out_ptrs[j] != nullptr &&
                                          !aligned(lse_out_ptrs[j], 4)))
            return DCP_MLA_ERR_MISALIGNED;
    const MergeInto into{dst_ptrs, lse_out_ptrs, cp};
    int merged = 0;
    int rc = producer(q, kv_ptrs, kv_len_ptrs, cp, B, H, Dk, Dv, T, scale, lse_base_e, n_split, part_out, part_lse,
                      status, flags & ~kFlagOneKernel, stream, one ? &into : nullptr, &merged);
    if (rc != 0 || B == 0 || merged) return rc;

    // Merge source k into head block k of width H/n_src: block k lies in
    // destination k / n_split at local head (k % n_split) * H/n_src.
    const int Hl = H / cp, Hs = H / n_src;
    void* dst[kSlots];
    float* lout[kSlots];
    for (int k = 0; k < n_src; ++k) {
        const int r = k / n_split, off = (k % n_split) * Hs;
        dst[k] = static_cast<uint8_t*>(dst_ptrs[r]) + (int64_t)off * Dv * 2;
        lout[k] = (lse_out_ptrs != nullptr && lse_out_ptrs[r] != nullptr) ? lse_out_ptrs[r] + off : nullptr;
    }
    dcp_lse_reduce_layout lay;
    lay.src_row = (int64_t)H * Dv;
    lay.src_head = Dv;
    lay.lse_row = H;
    lay.lse_head = 1;
    lay.dst_row = (int64_t)Hl * Dv;
    lay.dst_head = Dv;
    lay.lse_out_row = Hl;
    return dcp_lse_reduce_ex(part_out, part_lse, n_src, B, H, Dv, lse_base_e, DCP_DTYPE_BF16, dst, lout, &lay, nullptr,
                             1, flags & kFlagPdl, stream);
}

// ---- the no-allocation variant -----------------------------------------------------

namespace {

// Scratch for dcp_mla_decode_noalloc: the partials of one call. Host code must
// not use this name as an address; it takes the device address from
// cudaGetSymbolAddress on each device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[DCP_MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int dcp_mla_decode_noalloc(const void* q, const void* const* kv_ptrs, const int32_t* const* kv_len_ptrs,
                                      int cp, int64_t B, int H, int Dk, int Dv, int64_t T, float scale,
                                      int lse_base_e, int n_split, void* const* dst_ptrs, float* const* lse_out_ptrs,
                                      int32_t* status, unsigned flags, void* stream) {
    // the same argument checks as dcp_mla_decode, in the same order, before the
    // scratch limit: a bad shape reports itself, not as too large
    if (kv_ptrs == nullptr || kv_len_ptrs == nullptr || dst_ptrs == nullptr) return DCP_MLA_ERR_NULL_POINTER;
    if (!shape_ok(B, H, Dk, Dv, T)) return DCP_MLA_ERR_BAD_SHAPE;
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if (cp < 1 || cp * n_split > DCP_LSE_REDUCE_CP_MAX || H % (cp * n_split) != 0) return DCP_MLA_ERR_BAD_CP;
    const int64_t need = dcp_mla_decode_workspace_bytes(cp, n_split, B, H, Dv);
    if (need < 0) return DCP_MLA_ERR_BAD_SHAPE;
    if (need > (int64_t)DCP_MLA_NOALLOC_SCRATCH_BYTES) return DCP_MLA_ERR_SCRATCH_LIMIT;
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return DCP_MLA_ERR_SCRATCH_SETUP;
    return dcp_mla_decode(q, kv_ptrs, kv_len_ptrs, cp, B, H, Dk, Dv, T, scale, lse_base_e, n_split, scratch,
                          DCP_MLA_NOALLOC_SCRATCH_BYTES, dst_ptrs, lse_out_ptrs, status, flags, stream);
}
