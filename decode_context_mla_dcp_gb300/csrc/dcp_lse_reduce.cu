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
//              the LSE loads (one memory round trip). Used when every warp of
//              the grid fits on the GPU at once: small batches, latency-bound.
//   LSE_FIRST  persistent grid (one wave of CTAs); a warp strides over units,
//              reads the next unit's LSEs while the current payload is in
//              flight, and issues payload loads only for sources of nonzero
//              weight, so empty shards cost no payload bytes.
// Both give bit-identical results.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "dcp_lse_reduce.h"

namespace {

constexpr int kCpMax = DCP_LSE_REDUCE_CP_MAX;
constexpr int kWarps = 4;             // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kVpl = 2;               // 16-byte vectors per lane per pass (64 chunks = 512 bf16)
constexpr int kChunksPerPass = 32 * kVpl;

struct Params {
    const uint8_t* src[kCpMax];
    const float* lse[kCpMax];
    uint8_t* dst[kCpMax];
    float* lse_out[kCpMax];
    int64_t src_row, src_head;   // elements
    int64_t lse_row, lse_head;   // elements
    int64_t dst_row, dst_head;   // elements
    int64_t lse_out_row;         // elements
    int64_t units;               // B * H
    int H, Hl, D, cp;
    int base_e;
};

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

__device__ __forceinline__ void st_v4(uint8_t* ptr, const uint4& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
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

template <int kMaxCp>
__device__ __forceinline__ void load_lses(const Params& p, int64_t u, float (&l)[kMaxCp]) {
    const int64_t b = u / p.H;
    const int64_t h = u - b * p.H;
    const int64_t off = b * p.lse_row + h * p.lse_head;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) l[j] = (j < p.cp) ? ld_nc_f32(p.lse[j] + off) : -INFINITY;
}

// w_j = base^(l_j - m) / sum_k base^(l_k - m); merged = m + log_base(sum).
// A row whose every source is -inf gets all-zero weights and merged = -inf.
template <int kMaxCp>
__device__ __forceinline__ float lse_weights(const float (&l)[kMaxCp], int base_e, float (&w)[kMaxCp]) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) m = fmaxf(m, l[j]);
    if (m == -INFINITY) {
#pragma unroll
        for (int j = 0; j < kMaxCp; ++j) w[j] = 0.f;
        return -INFINITY;
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) {
        const float e = (l[j] == -INFINITY) ? 0.f : (base_e ? expf(l[j] - m) : exp2f(l[j] - m));
        w[j] = e;
        s += e;
    }
#pragma unroll
    for (int j = 0; j < kMaxCp; ++j) w[j] = w[j] / s;
    return m + (base_e ? logf(s) : log2f(s));
}

// Issue the payload loads of sources [jb*kSB, jb*kSB + kSB) for one pass.
// kGate: skip sources whose weight is 0 (weights known); otherwise load every
// source j < cp (weights not known yet; zero-weight payloads are dropped later).
template <int kSB, int kMaxCp, int kFixedChunks, bool kGate>
__device__ __forceinline__ void load_batch(const Params& p, int64_t src_off, int jb, int pass, int lane,
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

// ---- the kernel ----------------------------------------------------------------

template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
__global__ void __launch_bounds__(kThreads) lse_merge_kernel(const __grid_constant__ Params p) {
    constexpr int kSB = kMaxCp < 8 ? kMaxCp : 8;  // sources per load batch
    constexpr int kNB = kMaxCp / kSB;             // load batches
    static_assert(!kPreload || (kNB == 1 && kFixedChunks == kChunksPerPass),
                  "PRELOAD needs all sources in one batch and one pass");

    const int lane = threadIdx.x & 31;
    const int64_t step = (int64_t)gridDim.x * kWarps;
    int64_t u = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);

    // Inputs may come from the previous kernel in the stream (PDL): wait for it
    // before the first load. Let the next kernel start its launch right away.
    pdl_wait();
    pdl_launch_dependents();
    if (u >= p.units) return;

    const int nchunks = kFixedChunks ? kFixedChunks : (p.D >> 3);
    const int npass = (nchunks + kChunksPerPass - 1) / kChunksPerPass;

    float l[kMaxCp];
    float w[kMaxCp];
    uint4 x[kSB][kVpl];
    load_lses<kMaxCp>(p, u, l);
    if constexpr (kPreload) {
        const int64_t b = u / p.H;
        const int64_t h = u - b * p.H;
        load_batch<kSB, kMaxCp, kFixedChunks, false>(p, (b * p.src_row + h * p.src_head) * 2, 0, 0, lane,
                                                     nchunks, w, x);
    }

    while (true) {
        const int64_t un = u + step;
        const int64_t b = u / p.H;
        const int h = (int)(u - b * p.H);
        const int r = h / p.Hl;
        const int i = h - r * p.Hl;
        const int64_t src_off = (b * p.src_row + (int64_t)h * p.src_head) * 2;  // bytes
        uint8_t* const dst = p.dst[r] + (b * p.dst_row + (int64_t)i * p.dst_head) * 2;

        const float merged = lse_weights<kMaxCp>(l, p.base_e, w);

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
                if (pass == 0 && jb == 0 && un < p.units) load_lses<kMaxCp>(p, un, l);
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
        if (lane == 0 && p.lse_out[r] != nullptr) p.lse_out[r][b * p.lse_out_row + i] = merged;

        if (un >= p.units) break;
        u = un;
        if constexpr (kPreload) {
            const int64_t bn = u / p.H;
            const int64_t hn = u - bn * p.H;
            load_batch<kSB, kMaxCp, kFixedChunks, false>(p, (bn * p.src_row + hn * p.src_head) * 2, 0, 0, lane,
                                                         nchunks, w, x);
        }
    }
}

// ---- host side -----------------------------------------------------------------

using KernelFn = void (*)(Params);

template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
KernelFn kernel_ptr() {
    return reinterpret_cast<KernelFn>(&lse_merge_kernel<kF16, kMaxCp, kFixedChunks, kPreload>);
}

// Resident CTAs per SM for one instantiation, from the occupancy calculator
// (queried once per instantiation; the value depends only on the kernel).
template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
int ctas_per_sm() {
    static int cached = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &n, lse_merge_kernel<kF16, kMaxCp, kFixedChunks, kPreload>, kThreads, 0) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = 1;
        }
        return n;
    }();
    return cached;
}

struct Choice {
    KernelFn fn;
    int occupancy;
};

template <bool kF16, int kMaxCp, int kFixedChunks, bool kPreload>
Choice make_choice() {
    return Choice{kernel_ptr<kF16, kMaxCp, kFixedChunks, kPreload>(),
                  ctas_per_sm<kF16, kMaxCp, kFixedChunks, kPreload>()};
}

template <bool kF16, int kMaxCp>
Choice choose_cp(bool fixed512, bool preload) {
    if (fixed512) {
        if constexpr (kMaxCp <= 8) {
            if (preload) return make_choice<kF16, kMaxCp, kChunksPerPass, true>();
        }
        return make_choice<kF16, kMaxCp, kChunksPerPass, false>();
    }
    return make_choice<kF16, kMaxCp, 0, false>();
}

template <bool kF16>
Choice choose(int cp, bool fixed512, bool preload) {
    if (cp <= 1) return choose_cp<kF16, 1>(fixed512, preload);
    if (cp <= 2) return choose_cp<kF16, 2>(fixed512, preload);
    if (cp <= 4) return choose_cp<kF16, 4>(fixed512, preload);
    if (cp <= 8) return choose_cp<kF16, 8>(fixed512, preload);
    return choose_cp<kF16, 16>(fixed512, preload);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int dcp_lse_reduce_ex(const void* const* src_ptrs, const float* const* lse_ptrs,
                                 int cp, int64_t B, int H, int D, int lse_base_e, int dtype,
                                 void* const* dst_ptrs, float* const* lse_out_ptrs,
                                 const dcp_lse_reduce_layout* layout, unsigned flags, void* stream) {
    if (src_ptrs == nullptr || lse_ptrs == nullptr || dst_ptrs == nullptr) return DCP_ERR_NULL_POINTER;
    if (cp < 1 || cp > kCpMax) return DCP_ERR_BAD_CP;
    if (B < 0 || H < 1 || D < 8 || D % 8 != 0) return DCP_ERR_BAD_SHAPE;
    if (H % cp != 0) return DCP_ERR_HEADS_NOT_DIVISIBLE;
    if (dtype != DCP_DTYPE_BF16 && dtype != DCP_DTYPE_F16) return DCP_ERR_BAD_DTYPE;
    if (lse_base_e != 0 && lse_base_e != 1) return DCP_ERR_BAD_BASE;
    if ((flags & ~(DCP_FLAG_PDL | DCP_FLAG_PRELOAD | DCP_FLAG_LSE_FIRST)) != 0) return DCP_ERR_BAD_FLAGS;
    if ((flags & DCP_FLAG_PRELOAD) && (flags & DCP_FLAG_LSE_FIRST)) return DCP_ERR_BAD_FLAGS;

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

    Params p;
    for (int j = 0; j < kCpMax; ++j) {
        p.src[j] = nullptr;
        p.lse[j] = nullptr;
        p.dst[j] = nullptr;
        p.lse_out[j] = nullptr;
    }
    for (int j = 0; j < cp; ++j) {
        if (src_ptrs[j] == nullptr || lse_ptrs[j] == nullptr || dst_ptrs[j] == nullptr) return DCP_ERR_NULL_POINTER;
        if (!aligned(src_ptrs[j], 16) || !aligned(dst_ptrs[j], 16) || !aligned(lse_ptrs[j], 4))
            return DCP_ERR_MISALIGNED;
        if (lse_out_ptrs != nullptr && lse_out_ptrs[j] != nullptr && !aligned(lse_out_ptrs[j], 4))
            return DCP_ERR_MISALIGNED;
        p.src[j] = static_cast<const uint8_t*>(src_ptrs[j]);
        p.lse[j] = lse_ptrs[j];
        p.dst[j] = static_cast<uint8_t*>(dst_ptrs[j]);
        p.lse_out[j] = lse_out_ptrs != nullptr ? lse_out_ptrs[j] : nullptr;
    }
    if (B == 0) return DCP_OK;

    p.src_row = lay.src_row;
    p.src_head = lay.src_head;
    p.lse_row = lay.lse_row;
    p.lse_head = lay.lse_head;
    p.dst_row = lay.dst_row;
    p.dst_head = lay.dst_head;
    p.lse_out_row = lay.lse_out_row;
    p.units = B * (int64_t)H;
    p.H = H;
    p.Hl = Hl;
    p.D = D;
    p.cp = cp;
    p.base_e = lse_base_e;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1) {
        (void)cudaGetLastError();
        return DCP_ERR_DEVICE;
    }

    const bool fixed512 = (D == 512);
    const bool f16 = (dtype == DCP_DTYPE_F16);
    // The PRELOAD schedule needs every source in one load batch and D = 512.
    const bool preload_ok = fixed512 && cp <= 8;
    // Probe the persistent schedule's occupancy to size both grids.
    const Choice persistent = f16 ? choose<true>(cp, fixed512, false) : choose<false>(cp, fixed512, false);
    const int64_t wave_units = (int64_t)sms * persistent.occupancy * kWarps;
    bool preload;
    if (flags & DCP_FLAG_PRELOAD) {
        preload = preload_ok;
    } else if (flags & DCP_FLAG_LSE_FIRST) {
        preload = false;
    } else {
        preload = preload_ok && p.units <= wave_units;
    }
    const Choice c = preload ? (f16 ? choose<true>(cp, fixed512, true) : choose<false>(cp, fixed512, true))
                             : persistent;
    const int64_t want_ctas = (p.units + kWarps - 1) / kWarps;
    const int64_t wave_ctas = (int64_t)sms * c.occupancy;
    const int64_t ctas = preload ? want_ctas : (want_ctas < wave_ctas ? want_ctas : wave_ctas);
    const unsigned grid = (unsigned)(ctas < 0x7fffffff ? ctas : 0x7fffffff);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & DCP_FLAG_PDL) ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, c.fn, p);
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
                             &lay, 0u, stream);
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
        default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

extern "C" int dcp_lse_reduce_version(void) { return 10000; }
