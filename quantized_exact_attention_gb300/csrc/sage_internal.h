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
    float sv;                              // target |v| of the V codes: 144 / BKV (1.125 or 2.25)
};

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
    float* q_scale_out;                    // fused Q only: per-block Q scales written by the kernel
    CkptParams ck;                         // checkpoint kernel only
};

// Device status word layout: [0] first error code, [1] block id, [2] role, [3] tile.
constexpr int kStatusWords = 4;

int* device_status_ptr();                  // per-device address of the status words

// with_q = false: K/V statistics and quantization only (Q is quantized by the
// attention kernel of the fused entry point).
cudaError_t launch_prep(const PrepParams& p, bool with_q, cudaStream_t s, int* launches);
// Which form of the attention kernel to launch.
struct AttnMode {
    bool capture = false;   // QK checkpoint only (int32 scores)
    bool causal = false;    // causal mask
    bool fused_q = false;   // tq maps BF16 Q and each CTA quantizes its own Q block
    bool bkv64 = false;     // BKV = 64 contract: two 64-key softmax/PV epochs per 128-key tile
    bool pair = false;      // clusters of two CTAs sharing M = 256 MMAs (default and causal forms);
                            // tk / tv then map half tiles (64 keys; D/2 channels)
};
cudaError_t launch_attn(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const AttnMode& mode, cudaStream_t s, int* launches);
// One CTA (p.ck.b, p.ck.h, p.ck.qtile) of the attention kernel, writing its
// stage checkpoints besides its output rows.
cudaError_t launch_attn_checkpoints(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, bool causal, cudaStream_t s);

}  // namespace sage
