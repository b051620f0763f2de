// Split-KV MLA decode attention over one context shard, sm_103a: the producer
// of the DCP partial outputs and LSEs. What it computes, and the passages it
// follows, are stated in include/dcp_mla_decode.h.
//
// Design. One CTA owns (split s, a block of 16*kG heads, row b) and walks its
// token range in tiles of 32 tokens:
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
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "dcp_lse_reduce.h"
#include "dcp_mla_decode.h"

namespace {

constexpr int kDv = 512;
constexpr int kNt = 32;              // tokens per KV tile
constexpr int kSPad = 4;             // fp32 padding of a score row in shared memory
constexpr unsigned kFlagPdl = 1u;
constexpr long long kWaitLimitNs = 2000000000LL;

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
};

template <int kDk>
__host__ __device__ constexpr int row_bytes() {
    return (kDk + 8) * 2;  // 16 bytes of padding per row
}

template <int kDk, int kG>
__host__ __device__ constexpr int smem_bytes() {
    return 16 * kG * row_bytes<kDk>() + 2 * kNt * row_bytes<kDk>() + 16 * kG * (kNt + kSPad) * 4 + kG * 2 * 256 * 4 +
           3 * 8;
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
// Wait for a phase of an mbarrier, giving up after kWaitLimitNs: then the
// status word records it and the caller carries on (the outputs are invalid,
// but the kernel ends).
__device__ __forceinline__ void mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return;
    const long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            if (status != nullptr) atomicOr(status, 1);
            return;
        }
    }
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
        mbar_expect_tx(&bars[1 + buf], (uint32_t)(rows * kDk * 2));
        for (int r = 0; r < rows; ++r)
            bulk_g2s(dst + r * kRow, kv_row + ((int64_t)i * kNt + r) * kDk * 2, kDk * 2, &bars[1 + buf]);
    };
    if (threadIdx.x == 0) {
        mbar_expect_tx(&bars[0], (uint32_t)(kHB * kDk * 2));
        const uint8_t* qrow = p.q + ((int64_t)b * p.H + h0) * kDk * 2;
        for (int r = 0; r < kHB; ++r) bulk_g2s(q_s + r * kRow, qrow + (int64_t)r * kDk * 2, kDk * 2, &bars[0]);
        load_tile(0, 0);
        if (ntiles > 1) load_tile(1, 1);
    }
    mbar_wait(&bars[0], 0, p.status);

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

    for (int i = 0; i < ntiles; ++i) {
        const int buf = i & 1;
        mbar_wait(&bars[1 + buf], (uint32_t)((i >> 1) & 1), p.status);
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
        __syncthreads();  // every warp is done with this KV buffer and the score tile
        if (threadIdx.x == 0 && i + 2 < ntiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            load_tile(i + 2, buf);
        }
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

}  // namespace

extern "C" int dcp_mla_decode_smem_bytes(int Dk, int H) {
    const int g = H % 64 == 0 ? 4 : (H % 32 == 0 ? 2 : 1);
    if (Dk == 576) return g == 4 ? smem_bytes<576, 4>() : (g == 2 ? smem_bytes<576, 2>() : smem_bytes<576, 1>());
    if (Dk == 512) return g == 4 ? smem_bytes<512, 4>() : (g == 2 ? smem_bytes<512, 2>() : smem_bytes<512, 1>());
    return -1;
}

namespace {

// Validate and launch the producer over n_shard shards x n_split splits
// (slot = shard * n_split + split), all in one grid.
int producer(const void* q, const void* const* kv_ptrs, const int32_t* const* kv_len_ptrs, int n_shard, int64_t B,
             int H, int Dk, int Dv, int64_t T, float scale, int lse_base_e, int n_split, void* const* out_ptrs,
             float* const* lse_ptrs, int32_t* status, unsigned flags, void* stream) {
    if (q == nullptr || kv_ptrs == nullptr || kv_len_ptrs == nullptr || out_ptrs == nullptr || lse_ptrs == nullptr)
        return DCP_MLA_ERR_NULL_POINTER;
    if (B < 0 || B > 65535 || T < 0 || H < 16 || H % 16 != 0 || (Dk != 512 && Dk != 576) || Dv != kDv)
        return DCP_MLA_ERR_BAD_SHAPE;
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if (n_shard < 1 || n_shard * n_split > kSlots) return DCP_MLA_ERR_BAD_CP;
    if ((flags & ~kFlagPdl) != 0) return DCP_MLA_ERR_BAD_FLAGS;
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
    prm.q = static_cast<const uint8_t*>(q);
    prm.status = status;
    prm.T = T;
    prm.H = H;
    prm.n_split = n_split;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.lse_scale = lse_base_e ? 0.6931471805599453f : 1.0f;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = Dk == 576 ? launch_dk<576>(prm, B, n_slots, flags, st)
                                    : launch_dk<512>(prm, B, n_slots, flags, st);
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
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if (cp < 1 || cp * n_split > DCP_LSE_REDUCE_CP_MAX || H < 1 || H % (cp * n_split) != 0) return DCP_MLA_ERR_BAD_CP;
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
    int rc = producer(q, kv_ptrs, kv_len_ptrs, cp, B, H, Dk, Dv, T, scale, lse_base_e, n_split, part_out, part_lse,
                      status, flags, stream);
    if (rc != 0 || B == 0) return rc;

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
                             1, flags & DCP_FLAG_PDL, stream);
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
    if (n_split < 1 || n_split > DCP_MLA_SPLIT_MAX) return DCP_MLA_ERR_BAD_SPLIT;
    if (cp < 1 || cp * n_split > DCP_LSE_REDUCE_CP_MAX || H < 1 || H % (cp * n_split) != 0) return DCP_MLA_ERR_BAD_CP;
    const int64_t need = dcp_mla_decode_workspace_bytes(cp, n_split, B, H, Dv);
    if (need < 0) return DCP_MLA_ERR_BAD_SHAPE;
    if (need > (int64_t)DCP_MLA_NOALLOC_SCRATCH_BYTES) return DCP_MLA_ERR_SCRATCH_LIMIT;
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return DCP_MLA_ERR_SCRATCH_SETUP;
    return dcp_mla_decode(q, kv_ptrs, kv_len_ptrs, cp, B, H, Dk, Dv, T, scale, lse_base_e, n_split, scratch,
                          DCP_MLA_NOALLOC_SCRATCH_BYTES, dst_ptrs, lse_out_ptrs, status, flags, stream);
}
