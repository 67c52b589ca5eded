// sage_attn.cu - fused quantized attention for sm_103a.
//
// One CTA computes one 128-row query tile of one (b, h) head.  It follows the
// numerical contract's stage order (Experiment Log, "Phase 0 Import And
// Verification": QK traversal, online softmax, FP8 V/P, two-level PV
// accumulation, final conversion, ragged tails) with the state split that
// "Phase 1 State-Ownership Decision" argues for: QK/softmax state and
// PV/output state live in different warps, and every KV tile is processed in
// strict order with a per-tile rescale of the FP32 running output (RO).
//
// Warp roles (576 threads).  Each query row is split between two threads of
// two warps that see the same tensor-memory lane quarter: "half" 0 owns key
// columns 0-63 of every tile (one 64-key K scale block) and output channels
// 0-63, half 1 owns columns 64-127 and channels 64-127.
//   warps 0-7   softmax: S from tensor memory, half-row max, exchange of the
//               two half maxima through shared memory, alpha = 2^(m_old -
//               m_new), p*448 = 2^(S*f - m_new + log2 448) (packed FP32 pair
//               FMAs), half-row sums, e4m3 packing of P into tensor memory
//   warps 8-15  correction: RO[row, 64 channels] in registers; per tile
//               RO = RN(RN(RO * alpha) + fp16(PV)); epilogue 1/l, V scale, BF16
//   warp 16     TMA producer: Q once, then K (FP16 integer codes) and V (e4m3,
//               token-fastest) tiles through 3-deep rings
//   warp 17     tensor-memory allocator and single-thread tcgen05 issuer:
//               S_t = Q K_t^T (kind::f16, exact for INT8 codes: |sum| < 2^21
//               < 2^24) and PV_t = P_t V_t (kind::f8f6f4 with an FP16
//               accumulator -- the "FP16 PV" level of the two-level
//               accumulation -- P read from tensor memory)
//
// Tensor memory (512 columns x 128 lanes): three S buffers [0,384), the e4m3
// P of a tile overwriting the first 32 columns of its S buffer (4 values per
// 32-bit column), and one PV buffer [384,512) of FP16 tile sums (one per
// column).  Three S/P buffers let QK run two tiles ahead of PV, so the
// softmax of tile t+1 never waits for the PV MMA of tile t-1.  The BKV = 64
// form instead has two S/P buffers [0,256) and two PV buffers [256,512), one
// per 64-key epoch, so the PV of an epoch waits only for the drain of the
// same epoch one tile earlier.
//
// Every mbarrier wait is bounded (sage_ptx.cuh); a wait that runs out records
// SAGE_ERR_TIMEOUT in the device status words, raises a CTA-wide abort flag,
// lets the other roles leave their loops, drains the copies and MMAs in
// flight, frees tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "sage_internal.h"
#include "sage_ptx.cuh"
#include "sage_quant.cuh"

namespace sage {
namespace {

constexpr int kThreads = 576;
constexpr int kWarpProducer = 16;
constexpr int kWarpMma = 17;
constexpr int kNK = 3;              // K ring depth
constexpr int kNV = 3;              // V ring depth
constexpr int kNS = 3;              // S/P buffers in tensor memory
constexpr uint32_t kHalfBytes = 128 * 128;      // 64 FP16 channels (one 128-byte swizzle row) x 128 rows

enum Bar : uint32_t {
    B_QFULL = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + kNK,
    B_VFULL = B_KEMPTY + kNK,
    B_VEMPTY = B_VFULL + kNV,
    B_SFULL = B_VEMPTY + kNV,   // [3] S/P buffers
    B_SFREE = B_SFULL + kNS,
    B_PFULL = B_SFREE + kNS,
    B_PVFULL = B_PFULL + kNS,   // PV buffer 0 (the only one except with BKV = 64)
    B_PVFREE = B_PVFULL + 1,
    B_AFULL = B_PVFREE + 1,     // [4]: alpha slots (the BKV = 64 and paired forms use two)
    B_AFREE = B_AFULL + 4,      // [2]: alpha slot read (BKV = 64 and paired forms)
    B_XM = B_AFREE + 2,         // [buf][quarter]: the two halves of 32 rows exchanged maxima
    B_LFULL = B_XM + 8,
    B_DRAIN = B_LFULL + 1,
    B_QREADY = B_DRAIN + 1,     // fused Q: codes written over the BF16 tile
    B_COUNT = B_QREADY + 1
};

// Shared-memory map for head dimension D (offsets from a 1024-byte aligned
// base).  Q and K tiles hold 128 rows of FP16 codes as D/64 column blocks of
// kHalfBytes; a V tile holds D channel rows of 128 e4m3 tokens.
// Paired CTAs (kPair) hold only their half of each K tile (64 keys) and of
// each V tile (D/2 channels).
template <int D, bool kPair = false>
struct Smem {
    static_assert(D == 64 || D == 128, "head dimension");
    static constexpr uint32_t kTileQBytes = 128 * D * 2;
    static constexpr uint32_t kKRows = kPair ? 64 : 128;        // keys of a K stage
    static constexpr uint32_t kKBlock = kKRows * 128;          // one 64-channel column block of a K stage
    static constexpr uint32_t kTileKBytes = kKRows * D * 2;
    static constexpr uint32_t kTileVBytes = 128 * (kPair ? D / 2 : D);
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + kTileQBytes;
    static constexpr uint32_t OFF_V = OFF_K + kNK * kTileKBytes;
    static constexpr uint32_t OFF_BAR = OFF_V + kNV * kTileVBytes;
    static constexpr uint32_t OFF_ALPHA = OFF_BAR + ((B_COUNT * 8 + 15) / 16) * 16;   // float [4 slot][128] or [2 buf][2 epoch][128]
    static constexpr uint32_t OFF_XM = OFF_ALPHA + 4 * 128 * 4;                       // float [2 buf][2 half][128]
    static constexpr uint32_t OFF_L = OFF_XM + 4 * 128 * 4;                           // float [2 half][128]
    static constexpr uint32_t OFF_VS = OFF_L + 2 * 128 * 4;                           // float [D]
    static constexpr uint32_t OFF_TMEM = OFF_VS + 128 * 4;                            // u32
    static constexpr uint32_t OFF_ABORT = OFF_TMEM + 16;                              // int
    static constexpr uint32_t OFF_RED = OFF_ABORT + 16;                               // float [16]
    static constexpr uint32_t kSmemUsed = OFF_RED + 64;
    static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;                          // + alignment slack
};

constexpr uint32_t TM_S = 0;        // S buffer b (0..2) at column 128*b
constexpr uint32_t TM_PV = 384;     // PV buffer (D FP16 tile sums, one per column); BKV = 64: 256 + 128*epoch
// P of tile t is written over the first 32 columns of S buffer t%2 once both
// halves of every row have read their S values; the next QK into that buffer
// is issued after the PV MMA that reads P, and tcgen05.mma executes in issue
// order.
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2SP = 8.807354922057604f;   // log2(448)

enum Role { R_SOFTMAX = 1, R_CORRECT = 2, R_PRODUCER = 3, R_MMA = 4 };

__device__ __forceinline__ int clamp_len(const int32_t* lens, int b, int n) {
    if (lens == nullptr) return n;
    int v = lens[b];
    return v < 0 ? 0 : (v > n ? n : v);
}

__device__ __forceinline__ void record_failure(const AttnParams& p, volatile int* abort_flag, int role, int tile) {
    *abort_flag = 1;
    if (atomicCAS(p.status, 0, -4 /* SAGE_ERR_TIMEOUT */) == 0) {
        p.status[1] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
        p.status[2] = role;
        p.status[3] = tile;
    }
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// kCausal: key j is visible to query i iff j <= i + (Lk - Lq); a CTA visits
// only the KV tiles up to the diagonal of its last row, and rows that see no
// key are written as zero.
// kFusedQ: tm_q maps the caller's BF16 Q (4-D: channel, row, head, batch) and
// the CTA quantizes its own 128-row Q block (one INT8 scale block) in place in
// shared memory before the first QK; its scale goes to p.q_scale_out.
// kCkpt: a single CTA (p.ck.b, p.ck.h, p.ck.qtile) also writes its per-tile
// stage values (running max, rescale, running sums, P bytes, FP16 PV sums,
// FP32 running output, reciprocal) to p.ck.
// kB64: the BKV = 64 contract.  Each 128-key S tile is two online-softmax
// epochs: keys 0-63 (half 0) then keys 64-127 (half 1), each with its own
// running maximum, rescale and FP16 PV sum (two PV groups of K = 64 through
// the one PV accumulator) and its own RO update.
// kPair: a cluster of two CTAs computes two adjacent query tiles of one head
// with shared MMAs (tcgen05 .cta_group::2, M = 256).  Rank 0 issues every MMA
// for both; each CTA loads its own Q tile, one half of every K tile (64 keys)
// and one half of every V tile (D/2 channels), and holds its own S, P, PV,
// softmax and correction state.  Loads of both CTAs complete on rank 0's
// barriers; rank 0's commits arrive on both CTAs' barriers; the P-ready and
// PV-consumed arrivals of both CTAs' warps go to rank 0.
template <int D, bool kCapture, bool kCausal, bool kFusedQ, bool kCkpt = false, bool kB64 = false,
          bool kPair = false, bool kTmaOut = false>
__global__ void __launch_bounds__(kThreads, 1)
sage_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const AttnParams p) {
    static_assert(!kPair || (!kCapture && !kFusedQ && !kCkpt && !kB64), "paired CTAs: default and causal forms");
    using L = Smem<D, kPair>;
    constexpr uint32_t kKBlock = L::kKBlock;
    constexpr uint32_t kTileQBytes = L::kTileQBytes, kTileKBytes = L::kTileKBytes, kTileVBytes = L::kTileVBytes;
    constexpr uint32_t OFF_Q = L::OFF_Q, OFF_K = L::OFF_K, OFF_V = L::OFF_V, OFF_BAR = L::OFF_BAR;
    constexpr uint32_t OFF_ALPHA = L::OFF_ALPHA, OFF_XM = L::OFF_XM, OFF_L = L::OFF_L, OFF_VS = L::OFF_VS;
    constexpr uint32_t OFF_TMEM = L::OFF_TMEM, OFF_ABORT = L::OFF_ABORT, OFF_RED = L::OFF_RED;
    constexpr int kDH = D / 2;                              // output channels per correction thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw_base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t rank = 0;                                      // kPair: rank in the CTA pair
    int qtile;
    if constexpr (kPair) {
        rank = cluster_ctarank();
        const int npairs = (int)(gridDim.x >> 1);
        const int pi = kCausal ? npairs - 1 - (int)(blockIdx.x >> 1) : (int)(blockIdx.x >> 1);
        qtile = 2 * pi + (int)rank;
    } else {
        // causal: the longest query tiles start first
        qtile = kCkpt ? p.ck.qtile : (kCausal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x);
    }
    const int h = kCkpt ? p.ck.h : p.h_begin + (int)blockIdx.y, b = kCkpt ? p.ck.b : (int)blockIdx.z;
    const int bh = b * p.H + h;
    const int q0 = qtile * 128;
    const int lq = clamp_len(p.q_len, b, p.Nq);
    const int lk = clamp_len(p.kv_len, b, p.Nkv);
    // a pair takes every decision below from its first tile so both CTAs agree
    const int qg0 = kPair ? (qtile & ~1) * 128 : q0;        // first row of the CTA group
    constexpr int kGroupRows = kPair ? 256 : 128;
    if (qg0 >= lq) return;                                  // no valid row in this CTA group
    const int diag = lk - lq;                               // causal: row i sees keys j <= i + diag
    // keys any row of this CTA group can see
    const int kv_end = kCausal ? min(lk, min(qg0 + kGroupRows - 1, lq - 1) + diag + 1) : lk;

    if (kv_end <= 0) {                                      // no keys: rows are zero
        if (!kCapture && threadIdx.x < 128) {
            const int r = q0 + threadIdx.x;
            if (r < lq) {
                uint4* dst = reinterpret_cast<uint4*>(p.o + b * p.osb + h * p.osh + (int64_t)r * p.osn);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int T = (kv_end + 127) / 128;                     // KV tiles

    auto bar = [&](uint32_t i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
    float* alpha_s = reinterpret_cast<float*>(sgen + OFF_ALPHA);
    float* l_s = reinterpret_cast<float*>(sgen + OFF_L);
    float* vs_s = reinterpret_cast<float*>(sgen + OFF_VS);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + OFF_ABORT);
    const uint32_t peer_abort = kPair ? mapa_rank(sbase + OFF_ABORT, rank ^ 1u) : 0u;
    // waits, commits and failure reports of this kernel form
    auto bwait = [&](uint32_t bb, uint32_t par, const volatile int* af) -> bool {
        if constexpr (kPair) return mbar_wait_cluster(bb, par, af);
        else return mbar_wait(bb, par, af);
    };
    // A wait taken by all 32 lanes of a warp: one warp-wide vote per poll.
    auto wwait = [&](uint32_t bb, uint32_t par, const volatile int* af) -> bool {
        if constexpr (kPair) return __all_sync(0xffffffffu, bwait(bb, par, af));
        else return mbar_wait_warp(bb, par, af);
    };
    // Waits off the critical chain (the producer's ring-slot waits, the alpha
    // wait of the BKV = 64 and paired forms) sleep between checks; the others
    // spin.
    auto swait = [&](uint32_t bb, uint32_t par, const volatile int* af) -> bool {
        if constexpr (kPair) return mbar_wait_cluster(bb, par, af);
        else return mbar_wait_sleep(bb, par, af);
    };
    auto commit = [&](uint32_t bb) {
        if constexpr (kPair) mma_commit2(bb);
        else mma_commit(bb);
    };
    // BKV = 64 (not paired): two PV buffers, one per epoch, so that the PV of
    // epoch e waits only for the drain of epoch e of the previous tile; the
    // S/P buffers are then two.
    constexpr bool kDB = kB64 && !kPair;
    // The MMA issuer's order makes four handshakes implied in the one-CTA
    // forms:
    // - S-free (forms that issue PV): QK(t+2) reuses the S/P buffer of tile
    //   t-1, and the same thread issued PV(t-1) after P-full(t-1), which the
    //   softmax arrives only once it has read S(t-1).  The capture form issues
    //   no PV and keeps the handshake; the BKV = 64 form never needed it.
    // - alpha-free (forms with one alpha per tile), with four alpha slots: the
    //   correction reads alpha(t) before it arrives PV-free(t); PV(t+1) waits
    //   for that, QK(t+4) is issued after PV(t+1), and the softmax writes
    //   alpha(t+4) only after S-full(t+4).
    // - K-empty (three S/P buffers): a K stage is free once the QK that read it
    //   has completed, and with as many S/P buffers as K stages that QK's
    //   commit is S-full of the same index; the producer waits on it.
    // - V-empty (one PV commit per tile): a V stage is free once PV of the
    //   tile that used it has completed, i.e. at PV-full of that tile.  The
    //   single PV-full barrier may have run ahead of the producer by one more
    //   phase, in which case the producer waits one tile longer than needed;
    //   PV(t-1) never depends on V(t), so it cannot wait forever.
    constexpr bool kSFree = kCapture;
    constexpr bool kRing4 = !kB64 && !kPair;
    constexpr bool kKSlotBySFull = !kDB && !kPair && (kNS == kNK);
    constexpr bool kVSlotByPVFull = !kB64 && !kPair && !kCapture;
    static_assert(!(kB64 && kFusedQ), "the BKV = 64 form has no fused Q prologue (its scratch holds PV barriers)");
    constexpr int kNSb = kDB ? 2 : kNS;
    auto tm_pv = [&](int j) -> uint32_t { return kDB ? 256u + 128u * (uint32_t)j : TM_PV; };
    // PV buffer j's barriers; buffer 1's (BKV = 64 only) live in the scratch of
    // the fused-Q prologue, which that form never runs
    auto pv_full = [&](int j) -> uint32_t { return (kDB && j) ? sbase + OFF_RED : bar(B_PVFULL); };
    auto pv_free = [&](int j) -> uint32_t { return (kDB && j) ? sbase + OFF_RED + 8u : bar(B_PVFREE); };
    auto fail = [&](int role, int tile) {
        record_failure(p, abort_flag, role, tile);
        if constexpr (kPair) st_cluster_u32(peer_abort, 1u);  // the peer leaves its loops too
    };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar(B_QFULL), 1);
        for (int i = 0; i < kNK; ++i) { mbar_init(bar(B_KFULL + i), 1); mbar_init(bar(B_KEMPTY + i), 1); }
        for (int i = 0; i < kNV; ++i) { mbar_init(bar(B_VFULL + i), 1); mbar_init(bar(B_VEMPTY + i), 1); }
        for (int i = 0; i < kNS; ++i) {
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_SFREE + i), 256);     // every softmax thread
            mbar_init(bar(B_PFULL + i), kPair ? 16 : 256);   // every softmax thread / warp of both CTAs
        }
        mbar_init(bar(B_PVFULL), 1);
        mbar_init(bar(B_PVFREE), kPair ? 16 : 256);       // every correction thread / warp of both CTAs
        if constexpr (kDB) {
            mbar_init(pv_full(1), 1);
            mbar_init(pv_free(1), 256);
        }
        for (int i = 0; i < 8; ++i) mbar_init(bar(B_XM + i), 64);    // both halves of 32 rows
        for (int i = 0; i < 4; ++i) mbar_init(bar(B_AFULL + i), 128);   // softmax half 0 (writes alpha)
        for (int i = 0; i < 2; ++i) mbar_init(bar(B_AFREE + i), 256);   // every correction thread
        mbar_init(bar(B_LFULL), 256);             // every softmax thread
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_QREADY), 512);            // every softmax and correction thread (fused Q)
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        if constexpr (kPair) {
            tmem_alloc2(sbase + OFF_TMEM, kTmemCols);
            tmem_relinquish2();
        } else {
            tmem_alloc(sbase + OFF_TMEM, kTmemCols);
            tmem_relinquish();
        }
    }
    if (warp == kWarpProducer && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        if (!kCapture) tma_prefetch_desc(&tm_v);
        if (kTmaOut) tma_prefetch_desc(&tm_o);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();               // the peer's barriers exist before remote traffic
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    float fused_qs = 0.f;                                   // fused Q: this block's INT8 scale
    if constexpr (kFusedQ) {
        if (warp < 16) {
            // The softmax and correction warps quantize the CTA's Q block in
            // place: the BF16 tile and the FP16 code tile have the same element
            // size and the same 128-byte swizzle, so each 16-byte chunk keeps
            // its address; the swizzle permutes chunks within a row, so a
            // chunk's row is its byte offset / 128 within its 64-channel block.
            const int ct = threadIdx.x;                     // 0..511
            constexpr int kChunks = (int)(kTileQBytes / 16 / 512);
            const bool got = wwait(bar(B_QFULL), 0, abort_flag);
            if (!got && lane == 0) fail(R_SOFTMAX, -1);
            uint4 xq[kChunks];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < kChunks; ++i) {
                const uint32_t off = (uint32_t)(ct + 512 * i) * 16u;
                const int r = (int)((off % kHalfBytes) / 128u);
                xq[i] = got ? *reinterpret_cast<const uint4*>(sgen + OFF_Q + off) : make_uint4(0, 0, 0, 0);
                if (q0 + r < lq) amax = absmax8(xq[i], amax);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            float* red = reinterpret_cast<float*>(sgen + OFF_RED);
            if (lane == 0) red[warp] = amax;
            named_bar_sync(6, 512);                         // every softmax/correction thread, unconditionally
            amax = red[0];
#pragma unroll
            for (int i = 1; i < 16; ++i) amax = fmaxf(amax, red[i]);
            const float inv = int8_inv(amax);
            fused_qs = int8_scale(amax);
            if (ct == 0) p.q_scale_out[(int64_t)bh * p.nq_blocks + qtile] = fused_qs;
#pragma unroll
            for (int i = 0; i < kChunks; ++i) {
                const uint32_t off = (uint32_t)(ct + 512 * i) * 16u;
                const int r = (int)((off % kHalfBytes) / 128u);
                float x[8];
                unpack8(xq[i], x);
                int c[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) c[e] = (q0 + r < lq) ? int8_code(x[e], inv) : 0;
                *reinterpret_cast<uint4*>(sgen + OFF_Q + off) = pack_half_codes(c);
            }
            fence_proxy_async_smem();                       // codes visible to the tensor core
            mbar_arrive(bar(B_QREADY));
        }
    }

    if (warp < 8) {
        // ===================================================== softmax
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        float* xm = reinterpret_cast<float*>(sgen + OFF_XM);    // [buf][half][row]
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        const float qs = kFusedQ ? fused_qs : p.q_scale[(int64_t)bh * p.nq_blocks + qtile];
        // this half's 64-key scale block of tile t is 2t + half; load one tile ahead
        const float* kscale = p.k_scale + (int64_t)bh * p.nk_blocks;
        float ks_next = (half * 64 < lk) ? kscale[half] : 0.f;
        int s3 = 0, s3ph = 0;                               // S/P buffer of tile t and its phase
        const int T_sm = ok ? T : 0;
        for (int t = 0; t < T_sm; ++t, s3 = (s3 == kNSb - 1) ? 0 : s3 + 1, s3ph ^= (s3 == 0) ? 1 : 0) {
            const int sb = t & 1;
            const float ks = ks_next;
            const int kb_next = 2 * (t + 1) + half;
            ks_next = (kb_next * 64 < lk) ? kscale[kb_next] : 0.f;
            const float f = __fmul_rn(__fmul_rn(qs, ks), p.c);
            if (!wwait(bar(B_SFULL + s3), s3ph, abort_flag)) {
                if (lane == 0) fail(R_SOFTMAX, t);
                ok = false;
                break;
            }
            tc_fence_after();
            // The half row's 64 scores; every form but the capture takes their
            // maximum from the load itself (tcgen05.ld.red), which replaces a
            // 16-instruction max loop on the softmax's critical chain.
            uint32_t s0[32], s1[32];
            float mx_ld = -INFINITY;
            if constexpr (kCapture) {
                tmem_ld32(tmem + lane_base + TM_S + s3 * 128 + half * 64, s0);
                tmem_ld32(tmem + lane_base + TM_S + s3 * 128 + half * 64 + 32, s1);
            } else {
                tmem_ld64_max(tmem + lane_base + TM_S + s3 * 128 + half * 64, s0, s1, mx_ld);
            }
            tmem_wait_ld();
            tc_fence_before();
            if constexpr (kSFree) mbar_arrive(bar(B_SFREE + s3));
            // valid columns of this half (may be <= 0); causal: per row
            const int lim = (kCausal ? min(lk, q0 + row + diag + 1) : lk) - t * 128 - half * 64;
            const bool full = kCausal ? __all_sync(0xffffffffu, lim >= 64) : (lim >= 64);

            if (kCapture) {
                const int r = q0 + row;
                if (r < lq) {
                    int32_t* dst = p.s_out + ((int64_t)bh * p.Nq + r) * p.Nkv + t * 128 + half * 64;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (i < lim) dst[i] = (int32_t)__uint_as_float(s0[i]);
                        if (i + 32 < lim) dst[i + 32] = (int32_t)__uint_as_float(s1[i]);
                    }
                }
                continue;
            }

            // half-row maximum of the raw integer scores: the load's own when
            // all 64 columns are valid, else over the valid columns only
            float mx;
            if (full) {
                mx = mx_ld;
            } else {
                mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if (i < lim) mx = fmaxf(mx, __uint_as_float(s0[i]));
                    if (i + 32 < lim) mx = fmaxf(mx, __uint_as_float(s1[i]));
                }
            }
            // scaling by f >= 0 is monotone in every rounding, so this is the
            // maximum of the scaled scores of the half row
            const float mt = (mx == -INFINITY) ? -INFINITY : __fmul_rn(mx, f);
            xm[(sb * 2 + half) * 128 + row] = mt;
            // The two halves of these 32 rows meet here.  Both have read their S
            // values (tcgen05.wait::ld + fence before the s_free arrival), so
            // after this barrier either half may overwrite S columns with P.
            mbar_arrive(bar(B_XM + sb * 4 + quarter));
            if (!wwait(bar(B_XM + sb * 4 + quarter), (t >> 1) & 1, abort_flag)) {
                if (lane == 0) fail(R_SOFTMAX, t);
                ok = false;
                break;
            }
            tc_fence_after();
            const float mt_a = xm[(sb * 2 + 0) * 128 + row], mt_b = xm[(sb * 2 + 1) * 128 + row];
            float m_new = fmaxf(m_run, fmaxf(mt_a, mt_b));
            // causal: a row that has seen no key yet keeps m = -inf; measure from
            // 0 so that alpha = 0 and every p = 0 instead of NaN
            if (kCausal && m_new == -INFINITY) m_new = 0.f;
            float alpha = ex2_approx(m_run - m_new);        // first tile: 2^-inf = 0
            float nb = kLog2SP - m_new;                     // P is produced pre-scaled by 448
            float alpha_b = 1.f;                            // kB64: rescale of the second epoch
            if constexpr (kB64) {
                // epoch A (keys 0-63) ends at mA = max(m, max_A), epoch B
                // (keys 64-127) at m_new = max(mA, max_B)
                float m_a = fmaxf(m_run, mt_a);
                const bool none_a = kCausal && (m_a == -INFINITY);
                if (none_a) m_a = 0.f;
                alpha = ex2_approx(m_run - m_a);
                alpha_b = none_a ? 0.f : ex2_approx(m_a - m_new);
                nb = kLog2SP - (half == 0 ? m_a : m_new);
            }

            uint32_t pk[16];
            float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
            auto quad = [&](const uint32_t (&src)[32], int i, int col, bool masked) {
                float e0, e1, e2, e3;
                fma2_bc(e0, e1, __uint_as_float(src[i]), __uint_as_float(src[i + 1]), f, nb);
                fma2_bc(e2, e3, __uint_as_float(src[i + 2]), __uint_as_float(src[i + 3]), f, nb);
                if (masked) {
                    e0 = (col + 0 < lim) ? e0 : -INFINITY;
                    e1 = (col + 1 < lim) ? e1 : -INFINITY;
                    e2 = (col + 2 < lim) ? e2 : -INFINITY;
                    e3 = (col + 3 < lim) ? e3 : -INFINITY;
                }
                e0 = ex2_approx(e0); e1 = ex2_approx(e1); e2 = ex2_approx(e2); e3 = ex2_approx(e3);
                add2(sa0, sa1, e0, e1);
                add2(sb0, sb1, e2, e3);
                pk[col >> 2] = pack_e4m3x4(e0, e1, e2, e3);
            };
            if (full) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) { quad(s0, i, i, false); quad(s1, i, i + 32, false); }
            } else {
#pragma unroll
                for (int i = 0; i < 32; i += 4) { quad(s0, i, i, true); quad(s1, i, i + 32, true); }
            }
            const float tile_sum = (sa0 + sa1) + (sb0 + sb1);

            tmem_st16(tmem + lane_base + TM_S + s3 * 128 + half * 16, pk);
            if constexpr (kCkpt) {
                uint4* dp = reinterpret_cast<uint4*>(p.ck.p8 + ((int64_t)t * 128 + row) * 128 + half * 64);
#pragma unroll
                for (int i = 0; i < 4; ++i) dp[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                if (half == 0) {
                    p.ck.m[t * 128 + row] = m_new;
                    p.ck.alpha[t * 128 + row] = alpha;
                }
            }
            tmem_wait_st();
            // P-ready first: the PV MMA needs only P; the alpha hand-off to the
            // correction (which may wait for its slot) follows
            tc_fence_before();
            if constexpr (kPair) {                          // one arrival per warp, on rank 0's barrier
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_rank(bar(B_PFULL + s3), 0));
            } else {
                mbar_arrive(bar(B_PFULL + s3));
            }
            if (half == 0) {
                if constexpr (kRing4) {
                    alpha_s[(t & 3) * 128 + row] = alpha;
                    mbar_arrive(bar(B_AFULL + (t & 3)));
                } else {
                    if (t >= 2 && !wwait(bar(B_AFREE + sb), ((t >> 1) - 1) & 1, abort_flag)) {
                        if (lane == 0) fail(R_SOFTMAX, t);
                        ok = false;
                        break;
                    }
                    alpha_s[(sb * 2) * 128 + row] = alpha;
                    if (kB64) alpha_s[(sb * 2 + 1) * 128 + row] = alpha_b;
                    mbar_arrive(bar(B_AFULL + sb));
                }
            }
            if constexpr (kB64) {
                // half 0's keys join in epoch A, half 1's in epoch B
                l_run = half == 0 ? __fmul_rn(fmaf(l_run, alpha, tile_sum), alpha_b)
                                  : fmaf(__fmul_rn(l_run, alpha), alpha_b, tile_sum);
            } else {
                l_run = fmaf(l_run, alpha, tile_sum);
            }
            m_run = (kCausal && l_run == 0.f) ? -INFINITY : m_new;
            if constexpr (kCkpt) p.ck.l[(t * 2 + half) * 128 + row] = l_run;
        }
        if (!kCapture && ok) {
            l_s[half * 128 + row] = l_run;
            mbar_arrive(bar(B_LFULL));
        }
    } else if (warp < 16) {
        // ===================================================== correction + epilogue
        if (!kCapture) {
            const int quarter = (warp - 8) & 3, half = (warp - 8) >> 2;
            const int row = quarter * 32 + lane;
            const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
            if (half == 0 && row < D) vs_s[row] = p.v_scale[(int64_t)bh * D + row];
            named_bar_sync(5, 256);
            float ro[kDH];
#pragma unroll
            for (int i = 0; i < kDH; ++i) ro[i] = 0.f;
            bool ok = true;
            for (int t = 0; t < T; ++t) {
                const int sb = t & 1;
                const bool got_alpha = kRing4 ? wwait(bar(B_AFULL + (t & 3)), (t >> 2) & 1, abort_flag)
                                              : swait(bar(B_AFULL + sb), (t >> 1) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, got_alpha)) {
                    if (lane == 0) fail(R_CORRECT, t);
                    ok = false;
                    break;
                }
                const float alpha_a = kRing4 ? alpha_s[(t & 3) * 128 + row] : alpha_s[(sb * 2) * 128 + row];
                const float alpha_b = kB64 ? alpha_s[(sb * 2 + 1) * 128 + row] : 1.f;
                if constexpr (!kRing4) mbar_arrive(bar(B_AFREE + sb));
#pragma unroll 1
                for (int e = 0; e < (kB64 ? 2 : 1); ++e) {  // PV epochs of this tile
                    const float alpha = e ? alpha_b : alpha_a;
                    const bool unit = __all_sync(0xffffffffu, alpha == 1.0f);   // RN(RO * 1) == RO
                    const int pj = kDB ? e : 0;                 // PV buffer of this epoch
                    // RO = RN(RN(RO * alpha) + PV16): the product first, as one
                    // warp-uniform block skipped when alpha is 1 for the whole
                    // warp, and before the wait for PV
                    if (!unit) {
#pragma unroll
                        for (int i = 0; i < kDH; i += 2) mul2_s(ro[i], ro[i + 1], alpha);
                    }
                    if (!wwait(pv_full(pj), kDB ? (t & 1) : (kB64 ? e : (t & 1)), abort_flag)) {
                        if (lane == 0) fail(R_CORRECT, t);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kDH / 32; ++c) {
                        uint32_t v[16];                         // FP16 tile sums, two per register
                        tmem_ld32_pack16(tmem + lane_base + tm_pv(pj) + half * kDH + c * 32, v);
                        tmem_wait_ld();
                        if (c == kDH / 32 - 1) {
                            tc_fence_before();
                            if constexpr (kPair) {          // one arrival per warp, on rank 0's barrier
                                __syncwarp();
                                if (lane == 0) mbar_arrive_cluster(mapa_rank(bar(B_PVFREE), 0));
                            } else {
                                mbar_arrive(pv_free(pj));
                            }
                        }
                        if constexpr (kCkpt) {
                            uint4* dp = reinterpret_cast<uint4*>(p.ck.pv16 + ((int64_t)t * 128 + row) * D + half * kDH +
                                                                 c * 32);
#pragma unroll
                            for (int i = 0; i < 4; ++i) dp[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) add_f16x2_to(ro[c * 32 + 2 * i], ro[c * 32 + 2 * i + 1], v[i]);
                    }
                }
                if (!ok) break;
                if constexpr (kCkpt) {
                    float4* dp = reinterpret_cast<float4*>(p.ck.ro + ((int64_t)t * 128 + row) * D + half * kDH);
#pragma unroll
                    for (int i = 0; i < kDH / 4; ++i) dp[i] = make_float4(ro[4 * i], ro[4 * i + 1], ro[4 * i + 2], ro[4 * i + 3]);
                }
            }
            // Two epilogue forms, the same bytes.  Default: each thread writes
            // its row's channels with 16-byte stores.  kTmaOut (a separate
            // instantiation of the default and causal forms): a tile whose 128
            // rows are all valid (or valid up to Nq, where the tensor map
            // clips) is staged in shared memory and leaves through one TMA
            // store; a partial tile of a shorter batch item is still written
            // row by row, so rows >= q_len are never touched.  The TMA form
            // measured slower on GB300: the CTA waits for the store to read
            // shared memory before it can exit.
            const bool tma_out = kTmaOut && ((q0 + 128 <= lq) || (lq == p.Nq));
            if (ok && wwait(bar(B_LFULL), 0, abort_flag)) {
                // l carries the 448 scale of P, so (RO / l) * v_scale is the output
                const float l_row = l_s[row] + l_s[128 + row];
                // causal rows that saw no key have l = 0 and RO = 0: write zeros
                const float rl = (kCausal && l_row == 0.f) ? 0.f : __frcp_rn(l_row);
                if (kCkpt && half == 0) p.ck.recip[row] = rl;
                const int r = q0 + row;
                if (tma_out || r < lq) {
                    uint4* dst = reinterpret_cast<uint4*>(p.o + b * p.osb + h * p.osh + (int64_t)r * p.osn +
                                                          half * kDH);
#pragma unroll
                    for (int i = 0; i < kDH / 8; ++i) {
                        uint32_t w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int d = i * 8 + j * 2;
                            const float o0 = __fmul_rn(__fmul_rn(ro[d], rl), vs_s[half * kDH + d]);
                            const float o1 = __fmul_rn(__fmul_rn(ro[d + 1], rl), vs_s[half * kDH + d + 1]);
                            const __nv_bfloat162 pr = __floats2bfloat162_rn(o0, o1);
                            w[j] = *reinterpret_cast<const uint32_t*>(&pr);
                        }
                        if (tma_out) {
                            // channel c = half*kDH + 8i sits in 64-channel box c/64, 16-byte
                            // chunk (c%64)/8 of its 128-byte row, XOR-swizzled by row % 8;
                            // the K ring is free: every MMA has completed
                            const int c = half * kDH + i * 8;
                            const uint32_t off = (uint32_t)(c / 64) * kHalfBytes + (uint32_t)row * 128u +
                                                 ((uint32_t)(((c % 64) / 8) ^ (row & 7)) << 4);
                            *reinterpret_cast<uint4*>(sgen + OFF_K + off) = make_uint4(w[0], w[1], w[2], w[3]);
                        } else {
                            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (tma_out) fence_proxy_async_smem();      // staged rows visible to the TMA
            } else if (ok) {
                if (lane == 0) fail(R_CORRECT, T);
            }
            // Every correction thread reaches this barrier (each wait above is
            // bounded; tma_out is uniform over the CTA); the store is issued
            // only when no role has failed.
            if constexpr (kTmaOut) {
                if (tma_out) named_bar_sync(7, 256);
                if (tma_out && threadIdx.x == 256 && *abort_flag == 0) {
#pragma unroll
                    for (int hh = 0; hh < D / 64; ++hh)
                        tma_store_4d(&tm_o, sbase + OFF_K + hh * kHalfBytes, hh * 64, q0, h, b);
                    tma_store_commit();
                    tma_store_wait_read();                  // shared memory read before the CTA exits
                }
            }
        }
    } else if (warp == kWarpProducer) {
        // ===================================================== TMA producer
        if (lane == 0) {
            const uint32_t sQ = sbase + OFF_Q;
            int last_k[kNK], last_v[kNV];
            for (int i = 0; i < kNK; ++i) last_k[i] = -1;
            for (int i = 0; i < kNV; ++i) last_v[i] = -1;
            bool ok = true;
            // kPair: rank 0 expects the bytes of both CTAs; both complete on rank 0's barrier
            const uint32_t qfull = kPair ? mapa_rank(bar(B_QFULL), 0) : bar(B_QFULL);
            if (rank == 0) mbar_arrive_expect_tx(bar(B_QFULL), (kPair ? 2 : 1) * kTileQBytes);
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh) {
                if constexpr (kFusedQ)
                    tma_load_4d(sQ + hh * kHalfBytes, &tm_q, hh * 64, q0, h, b, bar(B_QFULL));
                else if constexpr (kPair)
                    tma_load_3d_pair(sQ + hh * kHalfBytes, &tm_q, hh * 64, q0, bh, qfull);
                else
                    tma_load_3d(sQ + hh * kHalfBytes, &tm_q, hh * 64, q0, bh, bar(B_QFULL));
            }
            auto load_k = [&](int t) -> bool {
                const int st = t % kNK;
                if (t >= kNK && !swait(kKSlotBySFull ? bar(B_SFULL + st) : bar(B_KEMPTY + st), ((t / kNK) - 1) & 1,
                                       abort_flag))
                    return false;
                const uint32_t dst = sbase + OFF_K + st * kTileKBytes;
                if (rank == 0) mbar_arrive_expect_tx(bar(B_KFULL + st), (kPair ? 2 : 1) * kTileKBytes);
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh) {
                    if constexpr (kPair)                    // keys [t*128 + 64*rank, +64)
                        tma_load_3d_pair(dst + hh * kKBlock, &tm_k, hh * 64, t * 128 + 64 * (int)rank, bh,
                                         mapa_rank(bar(B_KFULL + st), 0));
                    else
                        tma_load_3d(dst + hh * kHalfBytes, &tm_k, hh * 64, t * 128, bh, bar(B_KFULL + st));
                }
                last_k[st] = t;
                return true;
            };
            auto load_v = [&](int t) -> bool {
                const int st = t % kNV;
                if (t >= kNV && !swait(kVSlotByPVFull ? bar(B_PVFULL) : bar(B_VEMPTY + st),
                                       kVSlotByPVFull ? ((t - kNV) & 1) : (((t / kNV) - 1) & 1), abort_flag))
                    return false;
                const uint32_t dst = sbase + OFF_V + st * kTileVBytes;
                if (rank == 0) mbar_arrive_expect_tx(bar(B_VFULL + st), (kPair ? 2 : 1) * kTileVBytes);
                if (p.fault_mode != 1) {
                    if constexpr (kPair)                    // channels [rank*D/2, +D/2)
                        tma_load_3d_pair(dst, &tm_v, t * 128, (int)rank * (D / 2), bh,
                                         mapa_rank(bar(B_VFULL + st), 0));
                    else
                        tma_load_3d(dst, &tm_v, t * 128, 0, bh, bar(B_VFULL + st));
                }
                last_v[st] = t;
                return true;
            };
            // Loads follow the MMA issuer's consumption order: K0, K1, then
            // K(t+2), V(t) for every tile t.
            ok = load_k(0);
            if (ok && T > 1) ok = load_k(1);
            if (!ok) fail(R_PRODUCER, 0);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 2 < T) ok = load_k(t + 2);
                if (ok && !kCapture) ok = load_v(t);
                if (!ok) fail(R_PRODUCER, t);
            }
            // Drain: every copy issued must land before the CTA may exit.  A pair's
            // copies complete on rank 0's barriers: rank 0 drains for both, and
            // the closing cluster barrier keeps rank 1 alive until then.
            const int zero = 0;
            const volatile int* no_abort = &zero;
            if (rank == 0) {
                bwait(bar(B_QFULL), 0, no_abort);
                for (int i = 0; i < kNK; ++i)
                    if (last_k[i] >= 0) bwait(bar(B_KFULL + i), (last_k[i] / kNK) & 1, no_abort);
                if (p.fault_mode != 1)
                    for (int i = 0; i < kNV; ++i)
                        if (last_v[i] >= 0) bwait(bar(B_VFULL + i), (last_v[i] / kNV) & 1, no_abort);
            }
        }
    } else {
        // ===================================================== MMA issuer
        if (lane == 0 && rank == 0) {
            constexpr uint32_t kM = kPair ? 256u : 128u;                  // rows of both CTAs of a pair
            constexpr uint32_t kIdescQK = idesc_f32acc(0u, kM, 128u);     // F16 x F16 -> F32
            constexpr uint32_t kIdescPV = idesc_f16acc(0u, kM, (uint32_t)D);   // E4M3 x E4M3 -> F16
            const uint32_t sQ = sbase + OFF_Q;
            bool ok = bwait(bar(kFusedQ ? B_QREADY : B_QFULL), 0, abort_flag);
            int fail_tile = 0;
            // Shared-memory descriptors are built once.  Their start-address field
            // holds (address >> 4) in the low 14 bits; every operand lies below
            // 256 KB, so adding (byte offset >> 4) never carries out of the field.
            const uint64_t dQ = sdesc_sw128(sQ);
            const uint64_t dK = sdesc_sw128(sbase + OFF_K);
            const uint64_t dV = sdesc_sw128(sbase + OFF_V);
            int k_st = 0, k_ph = 0, v_st = 0, v_ph = 0;   // ring stage and phase of the next K / V tile
            int qb = 0, qph = 0;                          // S/P buffer (and phase) of the next QK
            int pb = 0, pph = 0;                          // S/P buffer (and phase) of the next PV
            // QK runs two tiles ahead of PV: with three S/P buffers, QK(t+2)
            // reuses the buffer of tile t-1, whose S the softmax has read and
            // whose P the PV MMA issued before it (same thread, in order) reads.
            auto issue_qk = [&](int t) -> bool {
                if (!bwait(bar(B_KFULL + k_st), k_ph, abort_flag)) return false;
                // only the capture form waits for S-free (see kSFree)
                if (kSFree && t >= kNS && !bwait(bar(B_SFREE + qb), qph ^ 1, abort_flag)) return false;
                tc_fence_after();
                const uint64_t bK = dK + (uint64_t)(k_st * (kTileKBytes >> 4));
                const uint32_t dS = tmem + TM_S + qb * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off_a = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    const uint32_t off_b = ((kk >> 2) * kKBlock + (kk & 3) * 32) >> 4;
                    if constexpr (kPair)
                        mma2_f16_ss(dS, dQ + off_a, bK + off_b, kIdescQK, kk > 0 ? 1u : 0u);
                    else
                        mma_f16_ss(dS, dQ + off_a, bK + off_b, kIdescQK, kk > 0 ? 1u : 0u);
                }
                commit(bar(B_SFULL + qb));
                if constexpr (!kKSlotBySFull) commit(bar(B_KEMPTY + k_st));
                if (++k_st == kNK) { k_st = 0; k_ph ^= 1; }
                if (++qb == kNSb) { qb = 0; qph ^= 1; }
                return true;
            };
            // The operands that are almost always ready are checked first, so
            // that only the wait for P sits between the softmax and the PV MMA.
            auto issue_pv = [&](int t) -> bool {
                if (!bwait(bar(B_VFULL + v_st), v_ph, abort_flag)) return false;
                const uint64_t bV = dV + (uint64_t)(v_st * (kTileVBytes >> 4));
                const uint32_t aP = tmem + TM_S + pb * 128;
                constexpr int kEpochs = kB64 ? 2 : 1, kSteps = 4 / kEpochs;   // K = 32 steps per epoch
#pragma unroll
                for (int e = 0; e < kEpochs; ++e) {
                    const int n = t * kEpochs + e;                           // PV accumulator use
                    const int pj = kDB ? e : 0;
                    if (kDB ? (t >= 1 && !bwait(pv_free(pj), (t - 1) & 1, abort_flag))
                            : (n >= 1 && !bwait(bar(B_PVFREE), (n - 1) & 1, abort_flag)))
                        return false;
                    if (e == 0 && !bwait(bar(B_PFULL + pb), pph, abort_flag)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < kSteps; ++j) {
                        const int kk = e * kSteps + j;
                        if constexpr (kPair)
                            mma2_f8_ts(tmem + tm_pv(pj), aP + kk * 8, bV + (uint64_t)(kk * (32 >> 4)), kIdescPV,
                                       j > 0 ? 1u : 0u);
                        else
                            mma_f8_ts(tmem + tm_pv(pj), aP + kk * 8, bV + (uint64_t)(kk * (32 >> 4)), kIdescPV,
                                      j > 0 ? 1u : 0u);
                    }
                    commit(pv_full(pj));
                }
                if constexpr (!kVSlotByPVFull) commit(bar(B_VEMPTY + v_st));
                if (++v_st == kNV) { v_st = 0; v_ph ^= 1; }
                if (++pb == kNSb) { pb = 0; pph ^= 1; }
                return true;
            };
            if (ok) ok = issue_qk(0);
            if (ok && T > 1) ok = issue_qk(1);
            for (int t = 0; t < T && ok; ++t) {
                fail_tile = t;
                if constexpr (kDB) {
                    // PV(t) first: QK(t+2) reuses the S/P buffer whose P it reads
                    ok = issue_pv(t);
                    if (ok && t + 2 < T) ok = issue_qk(t + 2);
                } else {
                    if (t + 2 < T) ok = issue_qk(t + 2);
                    if (ok && !kCapture) ok = issue_pv(t);
                }
            }
            if (!ok) fail(R_MMA, fail_tile);
            // Drain: all MMAs issued by this thread complete before teardown.
            commit(bar(B_DRAIN));
            const int zero = 0;
            bwait(bar(B_DRAIN), 0, &zero);
        } else if (kPair && lane == 0) {
            // rank 1: rank 0's MMAs read this CTA's shared memory and write its
            // tensor memory; they finish before it frees either
            const int zero = 0;
            bwait(bar(B_DRAIN), 0, &zero);
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();               // no remote traffic past this point
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        if constexpr (kPair) tmem_dealloc2(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool kCapture, bool kCausal, bool kFusedQ = false, bool kCkpt = false, bool kB64 = false,
          bool kTmaOut = false>
cudaError_t launch_one(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t s) {
    static bool attr_set[64] = {};                          // per device, per instantiation
    constexpr uint32_t kSmemBytes = Smem<D>::kSmemBytes;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(sage_attn_kernel<D, kCapture, kCausal, kFusedQ, kCkpt, kB64, false, kTmaOut>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const dim3 grid = kCkpt ? dim3(1, 1, 1) : dim3((unsigned)((p.Nq + 127) / 128), (unsigned)p.h_count, (unsigned)p.B);
    sage_attn_kernel<D, kCapture, kCausal, kFusedQ, kCkpt, kB64, false, kTmaOut>
        <<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

// Paired form: clusters of two CTAs over an even number of query tiles.
template <int D, bool kCausal>
cudaError_t launch_pair(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& to, cudaStream_t s) {
    static bool attr_set[64] = {};
    constexpr uint32_t kSmemBytes = Smem<D, true>::kSmemBytes;
    auto kernel = sage_attn_kernel<D, false, kCausal, false, false, false, true>;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const unsigned pairs = (unsigned)((p.Nq + 255) / 256);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, (unsigned)p.h_count, (unsigned)p.B);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& to, const AttnMode& m, cudaStream_t s) {
    if (m.pair) {
        if (m.capture || m.fused_q || m.bkv64) return cudaErrorInvalidValue;
        return m.causal ? launch_pair<D, true>(p, tq, tk, tv, to, s) : launch_pair<D, false>(p, tq, tk, tv, to, s);
    }
    if (m.capture) return launch_one<D, true, false>(p, tq, tk, tv, to, s);   // S does not depend on BKV
    if (m.bkv64) {
        if (m.fused_q) return cudaErrorInvalidValue;
        return m.causal ? launch_one<D, false, true, false, false, true>(p, tq, tk, tv, to, s)
                        : launch_one<D, false, false, false, false, true>(p, tq, tk, tv, to, s);
    }
    if (m.fused_q)
        return m.causal ? launch_one<D, false, true, true>(p, tq, tk, tv, to, s)
                        : launch_one<D, false, false, true>(p, tq, tk, tv, to, s);
    if (p.tma_out)                                          // the TMA-store epilogue form
        return m.causal ? launch_one<D, false, true, false, false, false, true>(p, tq, tk, tv, to, s)
                        : launch_one<D, false, false, false, false, false, true>(p, tq, tk, tv, to, s);
    return m.causal ? launch_one<D, false, true>(p, tq, tk, tv, to, s) : launch_one<D, false, false>(p, tq, tk, tv, to, s);
}

}  // namespace

cudaError_t launch_attn(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, const AttnMode& mode, cudaStream_t s,
                        int* launches) {
    *launches = 1;
    if (p.D == 128) return launch_d<128>(p, tq, tk, tv, to, mode, s);
    if (p.D == 64) return launch_d<64>(p, tq, tk, tv, to, mode, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_checkpoints(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& to, bool causal, cudaStream_t s) {
    if (p.D == 128)
        return causal ? launch_one<128, false, true, false, true>(p, tq, tk, tv, to, s)
                      : launch_one<128, false, false, false, true>(p, tq, tk, tv, to, s);
    if (p.D == 64)
        return causal ? launch_one<64, false, true, false, true>(p, tq, tk, tv, to, s)
                      : launch_one<64, false, false, false, true>(p, tq, tk, tv, to, s);
    return cudaErrorInvalidValue;
}

}  // namespace sage
