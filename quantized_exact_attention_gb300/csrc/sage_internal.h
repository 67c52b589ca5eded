// sage_internal.h - contract constants and kernel parameter blocks shared by
// the library's translation units (host and device).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>

namespace sage {

// Contract tile constants.  The pages name the stages but give no numbers;
// these are the readings the whole library is built on.
constexpr int kBQS = 128;        // rows per INT8 Q scale block (one 128-row query tile)
constexpr int kBKS = 64;         // rows per INT8 K scale block (64-key K/V slots)
constexpr int kBKV = 128;        // keys per online-softmax tile and per inner PV sum
constexpr int kMeanChunk = 64;   // tokens per chunk of the pinned K-mean summation
constexpr float kSV = 1.125f;    // V is scaled so |v| <= 1.125: 128 * 448 * 1.125 <= FP16 max
constexpr float kSP = 448.0f;    // P is scaled by the e4m3 maximum

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t nkv_pad_of(int64_t nkv) { return ceil_div(nkv, 16) * 16; }

struct PrepParams {
    const uint16_t* q;  // BF16 bit patterns
    const uint16_t* k;
    const uint16_t* v;
    int64_t qsb, qsh, qsn, ksb, ksh, ksn, vsb, vsh, vsn;   // element strides
    int B, H, Nq, Nkv, D, nkv_pad;         // D: head dimension, 64 or 128
    int h_begin, h_count;                  // heads [h_begin, h_begin + h_count) are processed
    int nq_blocks, nk_blocks, n_chunks;    // ceil(Nq/128), ceil(Nkv/64), ceil(Nkv/64)
    const int32_t* q_len;                  // device [B] or null
    const int32_t* kv_len;
    uint16_t* q16;
    uint16_t* k16;
    uint8_t* v8t;
    int8_t* q8;                            // optional
    int8_t* k8;                            // optional
    float* q_scale;
    float* k_scale;
    float* v_scale;
    float* k_mean;
    float* psum;                           // workspace [B,H,n_chunks,D]
    float* pamax;                          // workspace [B,H,n_chunks,D]
    float* v_inv;                          // workspace [B,H,D]
    unsigned long long* stats_done;        // workspace [B,H]: (launch epoch << 32) | finished statistics items
    uint32_t* ready;                       // workspace [B,H]: launch epoch once the head's statistics are final
    int* queue;                            // workspace [H]: one-pass work counter of the range starting at head h
    int* status;                           // device status words (a bounded wait that ran out)
    int prep_lag;                          // one-pass queue lag in heads; <= 0: chosen from the grid
    float sv;                              // target |v| of the V codes: 144 / BKV (1.125 or 2.25)
};

// Workspace bytes: chunk sums and maxima [B,H,chunks,D], V inverse scales
// [B,H,D] (floats), then the one-pass synchronisation words (12 B per head)
// and work counters (4 B per head), 16 B per head in all, then a slot for the
// per-item lengths [2][B] int32 that the host-memory entries stage there
// (rounded up to 16 B).
inline size_t prep_workspace_core(int64_t bh, int64_t nchunks, int64_t D) {
    return (size_t)(2 * bh * nchunks * D * 4 + bh * D * 4 + bh * 16);
}
inline size_t prep_workspace_bytes(int64_t B, int64_t H, int64_t nchunks, int64_t D) {
    return prep_workspace_core(B * H, nchunks, D) + (size_t)((8 * B + 15) / 16) * 16;
}
// The lengths slot: q_len at [0, B), kv_len at [B, 2B).
inline int32_t* prep_lens_slot(void* ws, int64_t B, int64_t H, int64_t nchunks, int64_t D) {
    return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + prep_workspace_core(B * H, nchunks, D));
}
// Point the workspace fields of p (whose B, H, D and n_chunks are set) at a
// workspace of that size.
inline void set_prep_workspace(PrepParams& p, void* ws) {
    const int64_t bh = (int64_t)p.B * p.H;
    float* f = static_cast<float*>(ws);
    const int64_t part = bh * p.n_chunks * p.D;
    p.psum = f;
    p.pamax = f + part;
    p.v_inv = f + 2 * part;
    p.stats_done = reinterpret_cast<unsigned long long*>(f + 2 * part + bh * p.D);
    p.ready = reinterpret_cast<uint32_t*>(p.stats_done + bh);
    p.queue = reinterpret_cast<int*>(p.ready + bh);
}

// Stage checkpoints of one query tile (see sage_attn_checkpoints).
struct CkptParams {
    float* m;          // [T][128]        running max after tile t
    float* l;          // [T][2][128]     each half row's running sum after tile t
    float* alpha;      // [T][128]        rescale factor of tile t
    uint8_t* p8;       // [T][128][128]   e4m3 P bytes of tile t (row-major, key fastest)
    uint16_t* pv16;    // [T][128][D]     FP16 PV tile sums
    float* ro;         // [T][128][D]     FP32 running output after tile t
    float* recip;      // [128]           1/l
    int b, h, qtile;   // the query tile (its CTA is the only one launched)
};

struct AttnParams {
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    const int32_t* q_len;
    const int32_t* kv_len;
    uint16_t* o;                           // BF16 bit patterns
    int64_t osb, osh, osn;
    int32_t* s_out;                        // QK checkpoint output (capture kernel only)
    int B, H, Nq, Nkv, D;                  // D: head dimension, 64 or 128
    int h_begin, h_count;                  // heads [h_begin, h_begin + h_count) are processed
    int nq_blocks, nk_blocks;
    float c;                               // fp32(sm_scale * log2(e))
    int* status;                           // device status words
    int fault_mode;                        // test hook: 0 = none
    int tma_out;                           // 1: full output tiles leave through a TMA store (measured slower)
    float* q_scale_out;                    // fused Q only: per-block Q scales written by the kernel
    CkptParams ck;                         // checkpoint kernel only
};

// Device status word layout: [0] first error code, [1] block id, [2] role, [3] tile.
constexpr int kStatusWords = 4;

int* device_status_ptr();                  // per-device address of the status words
void set_last_launch_count(int n);         // what sage_last_launch_count() reports next

// with_q = false: K/V statistics and quantization only (Q is quantized by the
// attention kernel of the fused entry point).
// one_pass: the single launch that reads K and V once, instead of the three
// plain launches (same bytes; measured slower on GB300).
cudaError_t launch_prep(const PrepParams& p, bool with_q, cudaStream_t s, int* launches, bool one_pass = false);
// Which form of the attention kernel to launch.
struct AttnMode {
    bool capture = false;   // QK checkpoint only (int32 scores)
    bool causal = false;    // causal mask
    bool fused_q = false;   // tq maps BF16 Q and each CTA quantizes its own Q block
    bool bkv64 = false;     // BKV = 64 contract: two 64-key softmax/PV epochs per 128-key tile
    bool pair = false;      // clusters of two CTAs sharing M = 256 MMAs (default and causal forms);
                            // tk / tv then map half tiles (64 keys; D/2 channels)
};
// to maps the BF16 output view (box 64 channels x 128 rows, 128-byte
// swizzle) for the TMA-store epilogue; unused by the capture form.
cudaError_t launch_attn(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, const AttnMode& mode, cudaStream_t s,
                        int* launches);
// One CTA (p.ck.b, p.ck.h, p.ck.qtile) of the attention kernel, writing its
// stage checkpoints besides its output rows.
cudaError_t launch_attn_checkpoints(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& to, bool causal, cudaStream_t s);

}  // namespace sage
