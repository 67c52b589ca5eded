// sage_prep.cu - preparation kernels: K channel statistics, K smoothing,
// INT8 Q/K and FP8 V quantization (Experiment Log, "Phase 0 Import And
// Verification": Q/K preparation, K smoothing, INT8 quantization, FP8 V).
//
// Two forms compute the same bytes.  The default is three plain launches
// (below).  The one-launch form, prep_onepass, reads every element of Q, K
// and V from HBM once: its CTAs walk a fixed queue of work
// items: per head, the chunk statistics of K and V, then its Q blocks, and the
// K/V quantization items of the head `lag` places earlier in the queue.  By
// the time a head's K/V items come up, its statistics are done and its K and
// V are still in L2 from the statistics pass, so the quantization pass reads
// them from L2.  The last statistics item of a head reduces the chunk
// partials in the pinned order (the finalize step) and publishes a ready
// flag; the head's K/V items wait for that flag (bounded).  CTAs take items
// from an atomic counter, so an item is only taken by a running CTA; a
// statistics item never waits, and a K/V item waits only for statistics
// items taken before it, so every wait ends without any assumption about
// how many CTAs are resident.  Measured on GB300 it is slower than the three
// launches (0.21 against 0.16 ms on 24 heads of 16K tokens): a statistics
// item walks its 64-token chunks in the pinned order, one thread per chunk
// and 8 channels, and holds its CTA for longer than the queue takes to move
// several heads on, so a head's K/V items either wait for it or come too
// late to find K and V in L2.
//
// The three plain launches:
//   1. prep_stats_q   per 64-token chunk: ordered FP32 K column sums and V
//                     column |max| (16 chunks per block); and, independent
//                     of those, the INT8 quantization of every 128-row Q block
//   2. prep_finalize  per (b,h) and 16 channels: chunk sums in order -> K
//                     mean; V amax -> v_scale and its inverse
//   3. prep_kv        K blocks (64 rows of K - mean) and V tiles (64 tokens,
//                     written transposed: token index fastest)
// Loaded BF16 data stays packed in registers (8 values per 16-byte word) and
// is widened on use, which keeps register use low enough for several blocks
// per SM and enough bytes in flight to stream HBM.  Every kernel is
// instantiated for head dimensions 64 and 128: a thread owns 8 channels, so a
// row takes D/8 threads and the 256 threads of a block cover 2048/D rows.
#include <atomic>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "sage_internal.h"
#include "sage_quant.cuh"

namespace sage {
namespace {

// Thread layout for head dimension D (256 threads per block, 8 channels each).
template <int D>
struct PrepShape {
    static_assert(D == 64 || D == 128, "head dimension");
    static constexpr int kGroups = D / 8;                 // threads per row
    static constexpr int kRowsPerPass = 256 / kGroups;    // rows a block covers at once
    static constexpr int kStatChunks = kRowsPerPass;      // 64-token chunks per statistics block
    static constexpr int kQPasses = kBQS / kRowsPerPass;  // passes over a 128-row Q block
    static constexpr int kKPasses = kBKS / kRowsPerPass;  // passes over a 64-row K block
    static constexpr int kVTokens = 8192 / D;             // tokens per V tile (64 or 128)
    static constexpr int kTokGroups = kVTokens / 4;       // threads per channel group, 4 tokens each
    static constexpr int kVStride = kTokGroups + 4;       // words per transposed row (+4 pad)
};

__device__ __forceinline__ int clamp_len(const int32_t* lens, int b, int n) {
    if (lens == nullptr) return n;
    int v = lens[b];
    return v < 0 ? 0 : (v > n ? n : v);
}

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
    return r;
}

// Store the INT8 codes of one row's 8 channels as FP16 images (and as INT8
// bytes when requested).
__device__ __forceinline__ void store_row_codes(const int (&c)[8], uint16_t* img, int8_t* bytes, int64_t off) {
    *reinterpret_cast<uint4*>(img + off) = pack_half_codes(c);
    if (bytes != nullptr) {
        uint2 bv;
        bv.x = (uint32_t)(c[0] & 0xFF) | ((uint32_t)(c[1] & 0xFF) << 8) |
               ((uint32_t)(c[2] & 0xFF) << 16) | ((uint32_t)(c[3] & 0xFF) << 24);
        bv.y = (uint32_t)(c[4] & 0xFF) | ((uint32_t)(c[5] & 0xFF) << 8) |
               ((uint32_t)(c[6] & 0xFF) << 16) | ((uint32_t)(c[7] & 0xFF) << 24);
        *reinterpret_cast<uint2*>(bytes + off) = bv;
    }
}

// ---------------------------------------------------------------------------
// 1. Chunk statistics and Q quantization.
// ---------------------------------------------------------------------------
// Statistics: thread (chunk slot cl, channel group dg) owns 8 channels of one
// 64-token chunk and walks its tokens in ascending order, so every partial
// sum is the FP32 left-to-right sum the contract pins.
template <int D>
__device__ __forceinline__ void chunk_stats(const PrepParams& p, int b, int h, int c) {
    const int dg = threadIdx.x % PrepShape<D>::kGroups;
    const int lk = clamp_len(p.kv_len, b, p.Nkv);
    const int d0 = dg * 8;
    const int t0 = c * kMeanChunk;
    const int t1 = min(t0 + kMeanChunk, lk);
    float s[8], a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { s[i] = 0.f; a[i] = 0.f; }
    const uint16_t* kp = p.k + b * p.ksb + h * p.ksh + d0;
    const uint16_t* vp = p.v + b * p.vsb + h * p.vsh + d0;
    int t = t0;
    for (; t + 4 <= t1; t += 4) {
        uint4 ku[4], vu[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            ku[u] = ldg16(kp + (int64_t)(t + u) * p.ksn);
            vu[u] = ldg16(vp + (int64_t)(t + u) * p.vsn);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float kx[8], vx[8];
            unpack8(ku[u], kx);
            unpack8(vu[u], vx);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                s[i] = __fadd_rn(s[i], kx[i]);
                a[i] = fmaxf(a[i], fabsf(vx[i]));
            }
        }
    }
    for (; t < t1; ++t) {
        float kx[8], vx[8];
        unpack8(ldg16(kp + (int64_t)t * p.ksn), kx);
        unpack8(ldg16(vp + (int64_t)t * p.vsn), vx);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            s[i] = __fadd_rn(s[i], kx[i]);
            a[i] = fmaxf(a[i], fabsf(vx[i]));
        }
    }
    const int64_t o = (((int64_t)b * p.H + h) * p.n_chunks + c) * D + d0;
    float4* ps = reinterpret_cast<float4*>(p.psum + o);
    float4* pa = reinterpret_cast<float4*>(p.pamax + o);
    ps[0] = make_float4(s[0], s[1], s[2], s[3]);
    ps[1] = make_float4(s[4], s[5], s[6], s[7]);
    pa[0] = make_float4(a[0], a[1], a[2], a[3]);
    pa[1] = make_float4(a[4], a[5], a[6], a[7]);
}

// Q block: rows [r0, r0+128), one INT8 scale for the whole block.
template <int D>
__device__ __forceinline__ void quant_q_block(const PrepParams& p, int b, int h, int qb, float* red) {
    using Sh = PrepShape<D>;
    const int bh = b * p.H + h;
    const int tid = threadIdx.x;
    const int lq = clamp_len(p.q_len, b, p.Nq);
    const int dg = tid % Sh::kGroups, rs = tid / Sh::kGroups;
    const int d0 = dg * 8, r0 = qb * kBQS;
    uint4 xr[Sh::kQPasses];
    float amax = 0.f;
    const uint16_t* qp = p.q + b * p.qsb + h * p.qsh + d0;
#pragma unroll
    for (int i = 0; i < Sh::kQPasses; ++i) {
        const int r = r0 + rs + Sh::kRowsPerPass * i;
        xr[i] = (r < lq) ? ldg16(qp + (int64_t)r * p.qsn) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < Sh::kQPasses; ++i) amax = absmax8(xr[i], amax);
    amax = block_max_256(amax, red);
    const float inv = int8_inv(amax);
    if (tid == 0) p.q_scale[(int64_t)bh * p.nq_blocks + qb] = int8_scale(amax);
#pragma unroll
    for (int i = 0; i < Sh::kQPasses; ++i) {
        const int r = r0 + rs + Sh::kRowsPerPass * i;
        if (r >= p.Nq) continue;
        float x[8];
        unpack8(xr[i], x);
        int c[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = (r < lq) ? int8_code(x[e], inv) : 0;
        store_row_codes(c, p.q16, p.q8, ((int64_t)bh * p.Nq + r) * D + d0);
    }
}

template <int D>
__global__ void __launch_bounds__(256, 3) prep_stats_q_kernel(const PrepParams p) {
    using Sh = PrepShape<D>;
    __shared__ float red[8];
    const int b = blockIdx.z, h = p.h_begin + (int)blockIdx.y;
    const int n_stat_blocks = (p.n_chunks + Sh::kStatChunks - 1) / Sh::kStatChunks;
    if ((int)blockIdx.x < n_stat_blocks) {
        const int c = blockIdx.x * Sh::kStatChunks + (threadIdx.x / Sh::kGroups);
        if (c < p.n_chunks) chunk_stats<D>(p, b, h, c);
    } else {
        quant_q_block<D>(p, b, h, blockIdx.x - n_stat_blocks, red);
    }
}

// ---------------------------------------------------------------------------
// 2. Per-(b,h) finalisation.  A block owns 16 channels of one head: its 256
// threads stage the chunk partials of those channels in shared memory (256
// chunks per pass, every load in flight at once), then one thread per
// channel adds them strictly in ascending chunk order.
// ---------------------------------------------------------------------------
constexpr int kFinChannels = 16;
constexpr int kFinChunks = 256;            // chunks staged per pass

template <int D>
__global__ void __launch_bounds__(256) prep_finalize_kernel(const PrepParams p) {
    __shared__ __align__(16) float st_sum[kFinChunks * kFinChannels];
    __shared__ __align__(16) float st_max[kFinChunks * kFinChannels];
    const int b = blockIdx.z, h = p.h_begin + (int)blockIdx.y, d0 = blockIdx.x * kFinChannels;
    const int lk = clamp_len(p.kv_len, b, p.Nkv);
    const int nc = (lk + kMeanChunk - 1) / kMeanChunk;
    const int64_t base = ((int64_t)b * p.H + h) * p.n_chunks * D + d0;
    const int quad = threadIdx.x & 3, lane_c = threadIdx.x >> 2;       // 4 float4 per chunk row, 64 chunk lanes
    float total = 0.f, amax = 0.f;
    for (int c0 = 0; c0 < nc; c0 += kFinChunks) {
        const int n = min(kFinChunks, nc - c0);
#pragma unroll
        for (int i = 0; i < kFinChunks / 64; ++i) {
            const int c = lane_c + 64 * i;
            if (c < n) {
                const int64_t g = base + (int64_t)(c0 + c) * D + quad * 4;
                reinterpret_cast<float4*>(st_sum)[c * 4 + quad] = __ldcg(reinterpret_cast<const float4*>(p.psum + g));
                reinterpret_cast<float4*>(st_max)[c * 4 + quad] = __ldcg(reinterpret_cast<const float4*>(p.pamax + g));
            }
        }
        __syncthreads();
        if (threadIdx.x < kFinChannels) {
            for (int c = 0; c < n; ++c) {
                total = __fadd_rn(total, st_sum[c * kFinChannels + threadIdx.x]);
                amax = fmaxf(amax, st_max[c * kFinChannels + threadIdx.x]);
            }
        }
        __syncthreads();
    }
    if (threadIdx.x < kFinChannels) {
        const int64_t o = ((int64_t)b * p.H + h) * D + d0 + threadIdx.x;
        p.k_mean[o] = lk > 0 ? __fdiv_rn(total, (float)lk) : 0.f;
        p.v_scale[o] = amax > 0.f ? __fdiv_rn(amax, p.sv) : 0.f;
        p.v_inv[o] = amax > 0.f ? __fdiv_rn(p.sv, amax) : 0.f;
    }
}

// ---------------------------------------------------------------------------
// 3. K and V quantization.  blockIdx.x selects the work item: K blocks first,
// then V tiles.  256 threads.
// ---------------------------------------------------------------------------
// K block: rows [r0, r0+64) of K - mean, one INT8 scale for the block.
template <int D>
__device__ __forceinline__ void quant_k_block(const PrepParams& p, int b, int h, int kb, float* red) {
    using Sh = PrepShape<D>;
    const int bh = b * p.H + h;
    const int tid = threadIdx.x;
    const int lk = clamp_len(p.kv_len, b, p.Nkv);
    const int dg = tid % Sh::kGroups, rs = tid / Sh::kGroups;
    const int d0 = dg * 8, r0 = kb * kBKS;
    float mean[8];
    {
        const float4* mp = reinterpret_cast<const float4*>(p.k_mean + (int64_t)bh * D + d0);
        const float4 m0 = mp[0], m1 = mp[1];
        mean[0] = m0.x; mean[1] = m0.y; mean[2] = m0.z; mean[3] = m0.w;
        mean[4] = m1.x; mean[5] = m1.y; mean[6] = m1.z; mean[7] = m1.w;
    }
    uint4 xr[Sh::kKPasses];
    const uint16_t* kp = p.k + b * p.ksb + h * p.ksh + d0;
#pragma unroll
    for (int i = 0; i < Sh::kKPasses; ++i) {
        const int r = r0 + rs + Sh::kRowsPerPass * i;
        xr[i] = (r < lk) ? ldg16(kp + (int64_t)r * p.ksn) : make_uint4(0, 0, 0, 0);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < Sh::kKPasses; ++i) {
        const int r = r0 + rs + Sh::kRowsPerPass * i;
        if (r < lk) {
            float x[8];
            unpack8(xr[i], x);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(__fsub_rn(x[e], mean[e])));
        }
    }
    amax = block_max_256(amax, red);
    const float inv = int8_inv(amax);
    if (tid == 0) p.k_scale[(int64_t)bh * p.nk_blocks + kb] = int8_scale(amax);
#pragma unroll
    for (int i = 0; i < Sh::kKPasses; ++i) {
        const int r = r0 + rs + Sh::kRowsPerPass * i;
        if (r >= p.Nkv) continue;
        float x[8];
        unpack8(xr[i], x);
        int c[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = (r < lk) ? int8_code(__fsub_rn(x[e], mean[e]), inv) : 0;
        store_row_codes(c, p.k16, p.k8, ((int64_t)bh * p.Nkv + r) * D + d0);
    }
}

// V tile: tokens [t0, t0 + 8192/D) -> e4m3 per channel, stored [d][token].
template <int D>
__device__ __forceinline__ void quant_v_tile(const PrepParams& p, int b, int h, int vt, uint32_t* vtile) {
    using Sh = PrepShape<D>;
    const int bh = b * p.H + h;
    const int tid = threadIdx.x;
    const int lk = clamp_len(p.kv_len, b, p.Nkv);
    const int tq = tid % Sh::kTokGroups, dg = tid / Sh::kTokGroups;   // 4 tokens x 8 channels per thread
    const int d0 = dg * 8, t0 = vt * Sh::kVTokens;
    float inv[8];
    {
        const float4* ip = reinterpret_cast<const float4*>(p.v_inv + (int64_t)bh * D + d0);
        const float4 i0 = ip[0], i1 = ip[1];
        inv[0] = i0.x; inv[1] = i0.y; inv[2] = i0.z; inv[3] = i0.w;
        inv[4] = i1.x; inv[5] = i1.y; inv[6] = i1.z; inv[7] = i1.w;
    }
    const uint16_t* vp = p.v + b * p.vsb + h * p.vsh + d0;
    uint4 xr[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = t0 + tq * 4 + u;
        xr[u] = (t < lk) ? ldg16(vp + (int64_t)t * p.vsn) : make_uint4(0, 0, 0, 0);
    }
    uint32_t word[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) word[e] = 0u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = t0 + tq * 4 + u;
        float x[8];
        unpack8(xr[u], x);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const bool live = (t < lk) && (inv[e] > 0.f);
            const __nv_fp8_storage_t c =
                __nv_cvt_float_to_fp8(__fmul_rn(x[e], inv[e]), __NV_SATFINITE, __NV_E4M3);
            word[e] |= (live ? (uint32_t)c : 0u) << (8 * u);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) vtile[(d0 + e) * Sh::kVStride + tq] = word[e];
    __syncthreads();
    constexpr int kParts = Sh::kVTokens / 16;           // 16-token chunks per channel row
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int chunk = tid + 256 * k;                // D rows x kParts chunks = 512
        const int d = chunk / kParts, part = chunk % kParts;
        const int t = t0 + part * 16;
        if (t < p.nkv_pad) {
            const uint4 w = *reinterpret_cast<const uint4*>(&vtile[d * Sh::kVStride + part * 4]);
            *reinterpret_cast<uint4*>(p.v8t + ((int64_t)bh * D + d) * p.nkv_pad + t) = w;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256, 4) prep_kv_kernel(const PrepParams p) {
    __shared__ float red[8];
    __shared__ __align__(16) uint32_t vtile[D * PrepShape<D>::kVStride];   // [d][words of 4 tokens + 4 pad]
    const int b = blockIdx.z, h = p.h_begin + (int)blockIdx.y;
    if ((int)blockIdx.x < p.nk_blocks) quant_k_block<D>(p, b, h, blockIdx.x, red);
    else quant_v_tile<D>(p, b, h, blockIdx.x - p.nk_blocks, vtile);
}

// ---------------------------------------------------------------------------
// One-pass preparation.
// ---------------------------------------------------------------------------
constexpr int kItemBlocks = 4;             // Q / K blocks or V tiles per work item
constexpr int kPrepCtasPerSm = 3;

// Shape of the work queue: rounds of R items; round r holds the statistics
// and Q items of head r and the K/V items of head r - lag.
struct PrepQueue {
    int nheads;          // B * h_count heads, in (b, h) order of the range
    int nS, nQ, nK, nV;  // items of each kind per head
    int R, lag, total;
    uint32_t epoch;      // this launch's value of the ready flags
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* a) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* a, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long prep_globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Per-(b,h) reduction of the chunk partials (the same pinned order as
// prep_finalize): threads [0, D) each add one channel's chunk sums in
// ascending chunk order; threads [D, 2D) take the V amax (order-free).
template <int D>
__device__ __forceinline__ void finalize_head(const PrepParams& p, int b, int h) {
    const int lk = clamp_len(p.kv_len, b, p.Nkv);
    const int nc = (lk + kMeanChunk - 1) / kMeanChunk;
    const int64_t bh = (int64_t)b * p.H + h;
    const int t = threadIdx.x;
    if (t < 2 * D) {
        const int d = t % D;
        const float* src = (t < D ? p.psum : p.pamax) + bh * p.n_chunks * D + d;
        float acc = 0.f;
        int c = 0;
        for (; c + 8 <= nc; c += 8) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = __ldcg(src + (int64_t)(c + u) * D);
#pragma unroll
            for (int u = 0; u < 8; ++u) acc = t < D ? __fadd_rn(acc, x[u]) : fmaxf(acc, x[u]);
        }
        for (; c < nc; ++c) {
            const float x = __ldcg(src + (int64_t)c * D);
            acc = t < D ? __fadd_rn(acc, x) : fmaxf(acc, x);
        }
        const int64_t o = bh * D + d;
        if (t < D) {
            p.k_mean[o] = lk > 0 ? __fdiv_rn(acc, (float)lk) : 0.f;
        } else {
            p.v_scale[o] = acc > 0.f ? __fdiv_rn(acc, p.sv) : 0.f;
            p.v_inv[o] = acc > 0.f ? __fdiv_rn(p.sv, acc) : 0.f;
        }
        __threadfence();
    }
}

// Wait (thread 0, bounded) until head bh's statistics are published.
__device__ __forceinline__ bool wait_head_ready(const PrepParams& p, const PrepQueue& q, int64_t bh, int* flag) {
    if (threadIdx.x == 0) {
        const uint32_t* ready = p.ready + bh;
        bool ok = ld_acquire_u32(ready) == q.epoch;
        if (!ok) {
            const unsigned long long t0 = prep_globaltimer();
            while (!(ok = ld_acquire_u32(ready) == q.epoch)) {
                __nanosleep(128);
                if (prep_globaltimer() - t0 > 1000000000ull) break;
            }
            if (!ok && p.status != nullptr && atomicCAS(p.status, 0, -4 /* SAGE_ERR_TIMEOUT */) == 0) {
                p.status[1] = (int)blockIdx.x;
                p.status[2] = 5;              // role: preparation
                p.status[3] = (int)bh;
            }
        }
        *flag = ok;
    }
    __syncthreads();
    return *flag != 0;
}

template <int D>
__device__ __forceinline__ void process_item(const PrepParams& p, const PrepQueue& q, int i, float* red,
                                             uint32_t* vtile, int* flag_s, int n_vtiles) {
    using Sh = PrepShape<D>;
    int& flag = *flag_s;
    {
        const int r = i / q.R, o = i % q.R;
        int kind, hi, sub;
        if (o < q.nS) { kind = 0; hi = r; sub = o; }
        else if (o < q.nS + q.nQ) { kind = 1; hi = r; sub = o - q.nS; }
        else if (o < q.nS + q.nQ + q.nK) { kind = 2; hi = r - q.lag; sub = o - q.nS - q.nQ; }
        else { kind = 3; hi = r - q.lag; sub = o - q.nS - q.nQ - q.nK; }
        if (hi < 0 || hi >= q.nheads) return;
        const int b = hi / p.h_count, h = p.h_begin + hi % p.h_count;
        const int64_t bh = (int64_t)b * p.H + h;
        if (kind == 0) {
            const int c = sub * Sh::kStatChunks + (threadIdx.x / Sh::kGroups);
            if (c < p.n_chunks) chunk_stats<D>(p, b, h, c);
            __threadfence();                  // partials visible before the count
            __syncthreads();
            if (threadIdx.x == 0) {
                // count this head's finished statistics items; the count word
                // holds (epoch << 32) | count, so stale words of other launches
                // read as zero
                unsigned long long* w = p.stats_done + bh;
                unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w), seen;
                unsigned long long n;
                do {
                    n = ((old >> 32) == q.epoch) ? (old & 0xFFFFFFFFull) : 0ull;
                    seen = old;
                    old = atomicCAS(w, seen, ((unsigned long long)q.epoch << 32) | (n + 1));
                } while (old != seen);
                __threadfence();
                flag = (int)(n + 1 == (unsigned long long)q.nS);
            }
            __syncthreads();
            if (flag) {                       // last statistics item of the head
                finalize_head<D>(p, b, h);
                __syncthreads();
                if (threadIdx.x == 0) st_release_u32(p.ready + bh, q.epoch);
            }
        } else if (kind == 1) {
#pragma unroll 1
            for (int j = 0; j < kItemBlocks; ++j) {
                const int qb = sub * kItemBlocks + j;
                if (qb < p.nq_blocks) quant_q_block<D>(p, b, h, qb, red);
                __syncthreads();
            }
        } else {
            if (!wait_head_ready(p, q, bh, &flag)) return;
#pragma unroll 1
            for (int j = 0; j < kItemBlocks; ++j) {
                const int blk = sub * kItemBlocks + j;
                if (kind == 2) {
                    if (blk < p.nk_blocks) quant_k_block<D>(p, b, h, blk, red);
                } else {
                    if (blk < n_vtiles) quant_v_tile<D>(p, b, h, blk, vtile);
                }
                __syncthreads();
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256, kPrepCtasPerSm) prep_onepass_kernel(const PrepParams p, const PrepQueue q) {
    using Sh = PrepShape<D>;
    __shared__ float red[8];
    __shared__ __align__(16) uint32_t vtile[D * Sh::kVStride];
    __shared__ int flag;
    __shared__ int next_item;
    const int n_vtiles = (p.nkv_pad + Sh::kVTokens - 1) / Sh::kVTokens;
    int* const counter = p.queue + p.h_begin;
    if (threadIdx.x == 0) next_item = atomicAdd(counter, 1);
    for (;;) {
        __syncthreads();                      // next_item written; the previous item's reads of flag, red, vtile done
        const int i = next_item;
        if (i >= q.total) break;
        __syncthreads();                      // every thread has read next_item
        // take the next item now; its index is needed only after this one
        int taken = 0;
        if (threadIdx.x == 0) taken = atomicAdd(counter, 1);
        process_item<D>(p, q, i, red, vtile, &flag, n_vtiles);
        if (threadIdx.x == 0) next_item = taken;
    }
}

std::atomic<uint32_t> g_prep_epoch{0};

template <int D>
cudaError_t launch_prep_d(const PrepParams& p, bool with_q, cudaStream_t s, int* launches);

template <int D>
cudaError_t launch_prep_onepass(const PrepParams& p, bool with_q, cudaStream_t s, int* launches) {
    using Sh = PrepShape<D>;
    static int grid_max[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (grid_max[dev] == 0) {
        int n = 0, per = 0;
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, prep_onepass_kernel<D>, 256, 0)) != cudaSuccess)
            return e;
        grid_max[dev] = n * (per > 0 ? per : 1);
    }
    const int64_t heads = (int64_t)p.B * p.h_count;
    if (heads > (1 << 24)) return launch_prep_d<D>(p, with_q, s, launches);   // queue indices stay in int
    PrepQueue q{};
    q.nheads = (int)heads;
    q.nS = (p.n_chunks + Sh::kStatChunks - 1) / Sh::kStatChunks;
    q.nQ = with_q ? (p.nq_blocks + kItemBlocks - 1) / kItemBlocks : 0;
    q.nK = (p.nk_blocks + kItemBlocks - 1) / kItemBlocks;
    q.nV = ((p.nkv_pad + Sh::kVTokens - 1) / Sh::kVTokens + kItemBlocks - 1) / kItemBlocks;
    q.R = q.nS + q.nQ + q.nK + q.nV;
    // The CTAs work on about grid/R consecutive rounds at a time; the K/V
    // items of a head come that many rounds (plus one) after its statistics.
    q.lag = p.prep_lag > 0 ? p.prep_lag : (grid_max[dev] + q.R - 1) / q.R + 1;
    q.lag = q.lag < q.nheads ? q.lag : q.nheads;
    q.total = (q.nheads + q.lag) * q.R;
    uint32_t ep;
    do { ep = ++g_prep_epoch; } while (ep == 0);
    q.epoch = ep;
    // the queue counter of this head range starts at zero
    if ((e = cudaMemsetAsync(p.queue + p.h_begin, 0, sizeof(int), s)) != cudaSuccess) return e;
    const int grid = q.total < grid_max[dev] ? q.total : grid_max[dev];
    prep_onepass_kernel<D><<<grid, 256, 0, s>>>(p, q);
    *launches = 1;
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_prep_d(const PrepParams& p, bool with_q, cudaStream_t s, int* launches) {
    using Sh = PrepShape<D>;
    *launches = 0;
    {
        // Q blocks follow the statistics blocks in the grid; without Q they are
        // simply not launched
        const int n_stat_blocks = (p.n_chunks + Sh::kStatChunks - 1) / Sh::kStatChunks;
        dim3 grid((unsigned)(n_stat_blocks + (with_q ? p.nq_blocks : 0)), (unsigned)p.h_count, (unsigned)p.B);
        prep_stats_q_kernel<D><<<grid, 256, 0, s>>>(p);
        ++*launches;
    }
    {
        dim3 grid((unsigned)(D / kFinChannels), (unsigned)p.h_count, (unsigned)p.B);
        prep_finalize_kernel<D><<<grid, 256, 0, s>>>(p);
        ++*launches;
    }
    {
        const int n_vtiles = (p.nkv_pad + Sh::kVTokens - 1) / Sh::kVTokens;
        dim3 grid((unsigned)(p.nk_blocks + n_vtiles), (unsigned)p.h_count, (unsigned)p.B);
        prep_kv_kernel<D><<<grid, 256, 0, s>>>(p);
        ++*launches;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const PrepParams& p, bool with_q, cudaStream_t s, int* launches, bool one_pass) {
    *launches = 0;
    if (p.D != 64 && p.D != 128) return cudaErrorInvalidValue;
    if (one_pass && p.stats_done != nullptr)
        return p.D == 64 ? launch_prep_onepass<64>(p, with_q, s, launches)
                         : launch_prep_onepass<128>(p, with_q, s, launches);
    if (p.D == 64) return launch_prep_d<64>(p, with_q, s, launches);
    return launch_prep_d<128>(p, with_q, s, launches);
}

}  // namespace sage
