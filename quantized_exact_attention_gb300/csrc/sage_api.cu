// sage_api.cu - the C ABI declared in include/sage_gb300.h: argument checks,
// TMA descriptor encoding and kernel dispatch.  No allocation, no sync on the
// compute entry points.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "sage_gb300.h"
#include "sage_internal.h"

namespace sage {

// Device status words, one copy per device that loads the library.
__device__ int g_status_words[kStatusWords];

namespace {

int* g_status_ptr[64] = {};
std::mutex g_mu;
thread_local int g_last_launches = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D tiled map over a [z][y][x] array with a 128-byte swizzled box.
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t x, uint64_t y, uint64_t z,
               uint64_t stride_y_bytes, uint64_t stride_z_bytes, uint32_t box_x, uint32_t box_y) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {x, y, z};
    cuuint64_t strides[2] = {stride_y_bytes, stride_z_bytes};
    cuuint32_t box[3] = {box_x, box_y, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D tiled map over a BF16 [B][H][N][D] view with arbitrary element strides
// (channel fastest), box 64 channels x 128 rows, 128-byte swizzle.
bool encode_bf16_view(CUtensorMap* m, const void* base, uint64_t D, uint64_t N, uint64_t H, uint64_t B,
                      int64_t sn, int64_t sh, int64_t sb) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {D, N, H, B};
    cuuint64_t strides[3] = {(cuuint64_t)sn * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
    cuuint32_t box[4] = {64, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_shape(int B, int H, int Nq, int Nkv, int D) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nkv <= 0) return SAGE_ERR_ARG;
    if (B > 65535 || H > 65535 || Nq > (1 << 24) || Nkv > (1 << 24)) return SAGE_ERR_ARG;
    if (D != 64 && D != 128) return SAGE_ERR_UNSUPPORTED;
    return SAGE_OK;
}

int check_tensor(const sage_tensor* t) {
    if (t == nullptr || t->ptr == nullptr) return SAGE_ERR_ARG;
    if (!aligned16(t->ptr)) return SAGE_ERR_UNSUPPORTED;
    if ((t->stride_b % 8) || (t->stride_h % 8) || (t->stride_n % 8)) return SAGE_ERR_UNSUPPORTED;
    if (t->stride_b < 0 || t->stride_h < 0 || t->stride_n < 0) return SAGE_ERR_UNSUPPORTED;
    return SAGE_OK;
}

int check_prep_buffers(const sage_prep_buffers* p, bool need_workspace, const sage_sizes& sz) {
    if (p == nullptr) return SAGE_ERR_ARG;
    if (!p->q16 || !p->k16 || !p->v8t || !p->q_scale || !p->k_scale || !p->v_scale || !p->k_mean)
        return SAGE_ERR_ARG;
    const void* ptrs[] = {p->q16, p->k16, p->v8t, p->q_scale, p->k_scale, p->v_scale, p->k_mean};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SAGE_ERR_UNSUPPORTED;
    if ((p->q8 && !aligned16(p->q8)) || (p->k8 && !aligned16(p->k8))) return SAGE_ERR_UNSUPPORTED;
    if (need_workspace) {
        if (!p->workspace || !aligned16(p->workspace)) return SAGE_ERR_ARG;
        if (p->workspace_bytes < sz.workspace) return SAGE_ERR_ARG;
    }
    return SAGE_OK;
}

int status_from(cudaError_t e) { return e == cudaSuccess ? SAGE_OK : SAGE_ERR_LAUNCH; }

int fault_mode_for_next_launch = 0;
int g_prep_one_pass = 0;        // sage_debug_prep_mode: 1 = the one-launch preparation
int g_prep_lag = 0;             // sage_debug_prep_mode: one-pass queue lag (0 = from the grid)
int g_tma_epilogue = 0;         // sage_debug_epilogue_mode: 1 = TMA-store epilogue

}  // namespace

int* device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_words) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(ptr);
    }
    return g_status_ptr[dev];
}

void set_last_launch_count(int n) { g_last_launches = n; }

}  // namespace sage

using namespace sage;

extern "C" {

int sage_buffer_sizes(int B, int H, int Nq, int Nkv, int D, sage_sizes* out) {
    if (out == nullptr) return SAGE_ERR_ARG;
    const int rc = check_shape(B, H, Nq, Nkv, D);
    if (rc != SAGE_OK) return rc;
    const int64_t bh = (int64_t)B * H;
    const int64_t pad = nkv_pad_of(Nkv);
    const int64_t nchunks = ceil_div(Nkv, kMeanChunk);
    out->q16 = (size_t)(bh * Nq * D * 2);
    out->k16 = (size_t)(bh * Nkv * D * 2);
    out->v8t = (size_t)(bh * D * pad);
    out->q_scale = (size_t)(bh * ceil_div(Nq, kBQS) * 4);
    out->k_scale = (size_t)(bh * ceil_div(Nkv, kBKS) * 4);
    out->v_scale = (size_t)(bh * D * 4);
    out->k_mean = (size_t)(bh * D * 4);
    out->q8 = (size_t)(bh * Nq * D);
    out->k8 = (size_t)(bh * Nkv * D);
    // partial sums + partial amax [B,H,chunks,D], the V inverse scales [B,H,D]
    // and 16 bytes of synchronisation words per head
    out->workspace = prep_workspace_bytes(B, H, nchunks, D);
    out->nkv_pad = pad;
    return SAGE_OK;
}

static int prep_common(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v, int B, int H, int Nq,
                       int Nkv, int D, const int32_t* q_len, const int32_t* kv_len, float sv,
                       const sage_prep_buffers* out, void* stream, int h_begin = 0, int h_count = -1) {
    int rc = check_shape(B, H, Nq, Nkv, D);
    if (rc != SAGE_OK) return rc;
    if ((rc = check_tensor(q)) != SAGE_OK || (rc = check_tensor(k)) != SAGE_OK || (rc = check_tensor(v)) != SAGE_OK)
        return rc;
    sage_sizes sz;
    sage_buffer_sizes(B, H, Nq, Nkv, D, &sz);
    if ((rc = check_prep_buffers(out, true, sz)) != SAGE_OK) return rc;

    PrepParams p{};
    p.q = static_cast<const uint16_t*>(q->ptr);
    p.k = static_cast<const uint16_t*>(k->ptr);
    p.v = static_cast<const uint16_t*>(v->ptr);
    p.qsb = q->stride_b; p.qsh = q->stride_h; p.qsn = q->stride_n;
    p.ksb = k->stride_b; p.ksh = k->stride_h; p.ksn = k->stride_n;
    p.vsb = v->stride_b; p.vsh = v->stride_h; p.vsn = v->stride_n;
    p.B = B; p.H = H; p.h_begin = h_begin; p.h_count = h_count < 0 ? H : h_count;
    p.Nq = Nq; p.Nkv = Nkv; p.D = D; p.sv = sv;
    p.nkv_pad = (int)sz.nkv_pad;
    p.nq_blocks = (int)ceil_div(Nq, kBQS);
    p.nk_blocks = (int)ceil_div(Nkv, kBKS);
    p.n_chunks = (int)ceil_div(Nkv, kMeanChunk);
    p.q_len = q_len; p.kv_len = kv_len;
    p.q16 = out->q16; p.k16 = out->k16; p.v8t = out->v8t;
    p.q8 = out->q8; p.k8 = out->k8;
    p.q_scale = out->q_scale; p.k_scale = out->k_scale; p.v_scale = out->v_scale; p.k_mean = out->k_mean;
    set_prep_workspace(p, out->workspace);
    p.status = device_status_ptr();
    p.prep_lag = g_prep_lag;
    int launches = 0;
    rc = status_from(launch_prep(p, true, static_cast<cudaStream_t>(stream), &launches, g_prep_one_pass != 0));
    if (rc == SAGE_OK) g_last_launches = launches;
    return rc;
}

// S_V of the BKV contract (R6): 144 / BKV; 0 for an unsupported tile length.
static float sv_of_bkv(int bkv) { return bkv == 128 ? kSV : (bkv == 64 ? 2.0f * kSV : 0.f); }

int sage_prep_qkv(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v, int B, int H, int Nq,
                  int Nkv, int D, const int32_t* q_len, const int32_t* kv_len, const sage_prep_buffers* out,
                  void* stream) {
    return prep_common(q, k, v, B, H, Nq, Nkv, D, q_len, kv_len, kSV, out, stream);
}

int sage_prep_qkv_bkv(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v, int B, int H, int Nq,
                      int Nkv, int D, const int32_t* q_len, const int32_t* kv_len, int bkv,
                      const sage_prep_buffers* out, void* stream) {
    const float sv = sv_of_bkv(bkv);
    if (sv == 0.f) return SAGE_ERR_UNSUPPORTED;
    return prep_common(q, k, v, B, H, Nq, Nkv, D, q_len, kv_len, sv, out, stream);
}

static int attn_common(const sage_prep_buffers* in, const sage_tensor* o, int32_t* s_out, int B, int H, int Nq,
                       int Nkv, int D, const int32_t* q_len, const int32_t* kv_len, float sm_scale,
                       void* stream, bool capture, bool causal, const CkptParams* ck = nullptr,
                       bool bkv64 = false, int h_begin = 0, int h_count = -1, bool pairs = false) {
    int rc = check_shape(B, H, Nq, Nkv, D);
    if (rc != SAGE_OK) return rc;
    sage_sizes sz;
    sage_buffer_sizes(B, H, Nq, Nkv, D, &sz);
    if ((rc = check_prep_buffers(in, false, sz)) != SAGE_OK) return rc;
    if (capture) {
        if (s_out == nullptr) return SAGE_ERR_ARG;
    } else if ((rc = check_tensor(o)) != SAGE_OK) {
        return rc;
    }
    int* status = device_status_ptr();
    if (status == nullptr) return SAGE_ERR_LAUNCH;

    const uint64_t bh = (uint64_t)B * H;
    // CTA pairs serve the default and causal forms; each CTA of a pair loads
    // half of every K tile (64 keys) and of every V tile (D/2 channels)
    const bool pair = pairs && !capture && ck == nullptr && !bkv64;
    CUtensorMap tq, tk, tv, to;
    // Q/K code images: boxes of 64 channels (128 bytes, one swizzle row) x 128
    // rows (K: 64 rows when paired); V^T: boxes of 128 tokens x D (D/2) channels;
    // O (the TMA-store epilogue): boxes of 64 channels x 128 rows.
    const uint64_t d = (uint64_t)D;
    if (!encode_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, in->q16, d, (uint64_t)Nq, bh, d * 2,
                   (uint64_t)Nq * d * 2, 64, 128) ||
        !encode_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, in->k16, d, (uint64_t)Nkv, bh, d * 2,
                   (uint64_t)Nkv * d * 2, 64, pair ? 64 : 128) ||
        !encode_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, in->v8t, (uint64_t)sz.nkv_pad, d, bh,
                   (uint64_t)sz.nkv_pad, (uint64_t)sz.nkv_pad * d, 128, (uint32_t)(pair ? D / 2 : D)))
        return encode_fn() ? SAGE_ERR_UNSUPPORTED : SAGE_ERR_DRIVER;
    if (capture)
        to = tq;                                           // no output
    else if (!encode_bf16_view(&to, o->ptr, d, (uint64_t)Nq, (uint64_t)H, (uint64_t)B, o->stride_n, o->stride_h,
                               o->stride_b))
        return encode_fn() ? SAGE_ERR_UNSUPPORTED : SAGE_ERR_DRIVER;

    AttnParams p{};
    p.q_scale = in->q_scale; p.k_scale = in->k_scale; p.v_scale = in->v_scale;
    p.q_len = q_len; p.kv_len = kv_len;
    if (!capture) {
        p.o = static_cast<uint16_t*>(const_cast<void*>(o->ptr));
        p.osb = o->stride_b; p.osh = o->stride_h; p.osn = o->stride_n;
    }
    p.s_out = s_out;
    p.B = B; p.H = H; p.h_begin = h_begin; p.h_count = h_count < 0 ? H : h_count;
    p.Nq = Nq; p.Nkv = Nkv; p.D = D;
    p.nq_blocks = (int)ceil_div(Nq, kBQS);
    p.nk_blocks = (int)ceil_div(Nkv, kBKS);
    const double scale = sm_scale > 0.f ? (double)sm_scale : 1.0 / std::sqrt((double)D);
    p.c = (float)(scale * (1.0 / std::log(2.0)));
    p.status = status;
    p.fault_mode = fault_mode_for_next_launch;
    p.tma_out = g_tma_epilogue;
    fault_mode_for_next_launch = 0;
    int launches = 0;
    if (ck != nullptr) {
        p.ck = *ck;
        rc = status_from(launch_attn_checkpoints(p, tq, tk, tv, to, causal, static_cast<cudaStream_t>(stream)));
        launches = 1;
    } else {
        AttnMode mode;
        mode.capture = capture;
        mode.causal = causal;
        mode.bkv64 = bkv64;
        mode.pair = pair;
        rc = status_from(launch_attn(p, tq, tk, tv, to, mode, static_cast<cudaStream_t>(stream), &launches));
    }
    if (rc == SAGE_OK) g_last_launches = launches;
    return rc;
}

int sage_attn_fwd(const sage_prep_buffers* in, const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                  const int32_t* q_len, const int32_t* kv_len, float sm_scale, void* stream) {
    return attn_common(in, o, nullptr, B, H, Nq, Nkv, D, q_len, kv_len, sm_scale, stream, false, false);
}

int sage_attn_fwd_causal(const sage_prep_buffers* in, const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                         const int32_t* q_len, const int32_t* kv_len, float sm_scale, void* stream) {
    return attn_common(in, o, nullptr, B, H, Nq, Nkv, D, q_len, kv_len, sm_scale, stream, false, true);
}

int sage_attn_fwd_pairs(const sage_prep_buffers* in, const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                        const int32_t* q_len, const int32_t* kv_len, float sm_scale, int causal, void* stream) {
    return attn_common(in, o, nullptr, B, H, Nq, Nkv, D, q_len, kv_len, sm_scale, stream, false, causal != 0,
                       nullptr, false, 0, -1, true);
}

int sage_attn_fwd_bkv(const sage_prep_buffers* in, const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                      const int32_t* q_len, const int32_t* kv_len, float sm_scale, int bkv, int causal,
                      void* stream) {
    if (bkv != 64 && bkv != 128) return SAGE_ERR_UNSUPPORTED;
    return attn_common(in, o, nullptr, B, H, Nq, Nkv, D, q_len, kv_len, sm_scale, stream, false, causal != 0,
                       nullptr, bkv == 64);
}

int sage_attn_checkpoints(const sage_prep_buffers* in, const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                          const int32_t* q_len, const int32_t* kv_len, float sm_scale, int causal, int b, int h,
                          int qtile, const sage_checkpoints* ck, void* stream) {
    if (ck == nullptr || !ck->m || !ck->l || !ck->alpha || !ck->p8 || !ck->pv16 || !ck->ro || !ck->recip)
        return SAGE_ERR_ARG;
    const void* ptrs[] = {ck->m, ck->l, ck->alpha, ck->p8, ck->pv16, ck->ro, ck->recip};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return SAGE_ERR_UNSUPPORTED;
    if (b < 0 || b >= B || h < 0 || h >= H || qtile < 0 || (int64_t)qtile * 128 >= Nq) return SAGE_ERR_ARG;
    CkptParams c{};
    c.m = ck->m; c.l = ck->l; c.alpha = ck->alpha; c.p8 = ck->p8; c.pv16 = ck->pv16; c.ro = ck->ro;
    c.recip = ck->recip;
    c.b = b; c.h = h; c.qtile = qtile;
    return attn_common(in, o, nullptr, B, H, Nq, Nkv, D, q_len, kv_len, sm_scale, stream, false, causal != 0, &c);
}

int sage_qk_int32(const sage_prep_buffers* in, int32_t* s, int B, int H, int Nq, int Nkv, int D,
                  const int32_t* q_len, const int32_t* kv_len, void* stream) {
    return attn_common(in, nullptr, s, B, H, Nq, Nkv, D, q_len, kv_len, 0.f, stream, true, false);
}

int sage_attention(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v, const sage_tensor* o,
                   int B, int H, int Nq, int Nkv, int D, const int32_t* q_len, const int32_t* kv_len,
                   float sm_scale, int causal, const sage_prep_buffers* buf, void* stream) {
    int rc = check_shape(B, H, Nq, Nkv, D);
    if (rc != SAGE_OK) return rc;
    if ((rc = check_tensor(q)) != SAGE_OK || (rc = check_tensor(k)) != SAGE_OK ||
        (rc = check_tensor(v)) != SAGE_OK || (rc = check_tensor(o)) != SAGE_OK)
        return rc;
    sage_sizes sz;
    sage_buffer_sizes(B, H, Nq, Nkv, D, &sz);
    if (buf == nullptr || !buf->k16 || !buf->v8t || !buf->q_scale || !buf->k_scale || !buf->v_scale ||
        !buf->k_mean || !buf->workspace)
        return SAGE_ERR_ARG;
    const void* ptrs[] = {buf->k16, buf->v8t, buf->q_scale, buf->k_scale, buf->v_scale, buf->k_mean,
                          buf->workspace};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return SAGE_ERR_UNSUPPORTED;
    if (buf->k8 && !aligned16(buf->k8)) return SAGE_ERR_UNSUPPORTED;
    if (buf->workspace_bytes < sz.workspace) return SAGE_ERR_ARG;
    int* status = device_status_ptr();
    if (status == nullptr) return SAGE_ERR_LAUNCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // K/V preparation only
    PrepParams pp{};
    pp.k = static_cast<const uint16_t*>(k->ptr);
    pp.v = static_cast<const uint16_t*>(v->ptr);
    pp.ksb = k->stride_b; pp.ksh = k->stride_h; pp.ksn = k->stride_n;
    pp.vsb = v->stride_b; pp.vsh = v->stride_h; pp.vsn = v->stride_n;
    pp.B = B; pp.H = H; pp.h_begin = 0; pp.h_count = H; pp.Nq = Nq; pp.Nkv = Nkv; pp.D = D; pp.sv = kSV;
    pp.nkv_pad = (int)sz.nkv_pad;
    pp.nq_blocks = (int)ceil_div(Nq, kBQS);
    pp.nk_blocks = (int)ceil_div(Nkv, kBKS);
    pp.n_chunks = (int)ceil_div(Nkv, kMeanChunk);
    pp.q_len = q_len; pp.kv_len = kv_len;
    pp.k16 = buf->k16; pp.v8t = buf->v8t; pp.k8 = buf->k8;
    pp.k_scale = buf->k_scale; pp.v_scale = buf->v_scale; pp.k_mean = buf->k_mean;
    set_prep_workspace(pp, buf->workspace);
    pp.status = status;
    pp.prep_lag = g_prep_lag;
    int prep_launches = 0;
    if ((rc = status_from(launch_prep(pp, false, s, &prep_launches, g_prep_one_pass != 0))) != SAGE_OK) return rc;

    // attention with the Q quantization in its prologue
    const uint64_t bh = (uint64_t)B * H, d = (uint64_t)D;
    CUtensorMap tq, tk, tv, to;
    if (!encode_bf16_view(&tq, q->ptr, d, (uint64_t)Nq, (uint64_t)H, (uint64_t)B, q->stride_n, q->stride_h,
                          q->stride_b) ||
        !encode_bf16_view(&to, o->ptr, d, (uint64_t)Nq, (uint64_t)H, (uint64_t)B, o->stride_n, o->stride_h,
                          o->stride_b) ||
        !encode_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, buf->k16, d, (uint64_t)Nkv, bh, d * 2,
                   (uint64_t)Nkv * d * 2, 64, 128) ||
        !encode_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, buf->v8t, (uint64_t)sz.nkv_pad, d, bh,
                   (uint64_t)sz.nkv_pad, (uint64_t)sz.nkv_pad * d, 128, (uint32_t)D))
        return encode_fn() ? SAGE_ERR_UNSUPPORTED : SAGE_ERR_DRIVER;
    AttnParams p{};
    p.k_scale = buf->k_scale; p.v_scale = buf->v_scale;
    p.q_scale_out = buf->q_scale;
    p.q_len = q_len; p.kv_len = kv_len;
    p.o = static_cast<uint16_t*>(const_cast<void*>(o->ptr));
    p.osb = o->stride_b; p.osh = o->stride_h; p.osn = o->stride_n;
    p.B = B; p.H = H; p.h_begin = 0; p.h_count = H; p.Nq = Nq; p.Nkv = Nkv; p.D = D;
    p.nq_blocks = pp.nq_blocks;
    p.nk_blocks = pp.nk_blocks;
    const double scale = sm_scale > 0.f ? (double)sm_scale : 1.0 / std::sqrt((double)D);
    p.c = (float)(scale * (1.0 / std::log(2.0)));
    p.status = status;
    p.fault_mode = fault_mode_for_next_launch;
    p.tma_out = g_tma_epilogue;
    fault_mode_for_next_launch = 0;
    int launches = 0;
    AttnMode mode;
    mode.causal = causal != 0;
    mode.fused_q = true;
    rc = status_from(launch_attn(p, tq, tk, tv, to, mode, s, &launches));
    if (rc == SAGE_OK) g_last_launches = launches + prep_launches;
    return rc;
}

// A host length clamped to [0, n] (NULL array: n), as the kernels clamp
// the device copies.
static int host_len(const int32_t* lens, int b, int n) {
    if (lens == nullptr) return n;
    return lens[b] < 0 ? 0 : (lens[b] > n ? n : lens[b]);
}

// Host-memory entries: stage per-item lengths given as host arrays (NULL: all
// valid) into the workspace's lengths slot on `s`, and point *q_dev/*kv_dev
// at the device copies (NULL when the host array was NULL).  The kernels
// clamp the staged values.
static int stage_host_lens(const sage_prep_buffers* buf, int B, int H, int Nq, int Nkv, int D,
                           const int32_t* q_len, const int32_t* kv_len, cudaStream_t s,
                           const int32_t** q_dev, const int32_t** kv_dev) {
    *q_dev = *kv_dev = nullptr;
    if (q_len == nullptr && kv_len == nullptr) return SAGE_OK;
    if (buf == nullptr || buf->workspace == nullptr) return SAGE_ERR_ARG;
    sage_sizes sz;
    sage_buffer_sizes(B, H, Nq, Nkv, D, &sz);
    if (buf->workspace_bytes < sz.workspace) return SAGE_ERR_ARG;
    int32_t* slot = prep_lens_slot(buf->workspace, B, H, ceil_div(Nkv, kMeanChunk), D);
    // pageable sources: the copies are staged before cudaMemcpyAsync returns
    if ((q_len && cudaMemcpyAsync(slot, q_len, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s) != cudaSuccess) ||
        (kv_len && cudaMemcpyAsync(slot + B, kv_len, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s) != cudaSuccess))
        return SAGE_ERR_LAUNCH;
    if (q_len) *q_dev = slot;
    if (kv_len) *kv_dev = slot + B;
    return SAGE_OK;
}

int sage_attention_host(const sage_copy* inputs, int n_inputs, const sage_tensor* q, const sage_tensor* k,
                        const sage_tensor* v, const sage_prep_buffers* buf, const sage_tensor* o,
                        const sage_copy* output, int B, int H, int Nq, int Nkv, int D,
                        const int32_t* q_len, const int32_t* kv_len, float sm_scale, void* stream) {
    if (inputs == nullptr || n_inputs <= 0 || output == nullptr) return SAGE_ERR_ARG;
    int rc = check_shape(B, H, Nq, Nkv, D);
    if (rc != SAGE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int32_t *q_dev = nullptr, *kv_dev = nullptr;
    if ((rc = stage_host_lens(buf, B, H, Nq, Nkv, D, q_len, kv_len, s, &q_dev, &kv_dev)) != SAGE_OK) return rc;
    for (int i = 0; i < n_inputs; ++i) {
        if (!inputs[i].host || !inputs[i].device) return SAGE_ERR_ARG;
        if (cudaMemcpyAsync(inputs[i].device, inputs[i].host, inputs[i].bytes, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return SAGE_ERR_LAUNCH;
    }
    rc = sage_prep_qkv(q, k, v, B, H, Nq, Nkv, D, q_dev, kv_dev, buf, stream);
    if (rc != SAGE_OK) return rc;
    const int prep_launches = g_last_launches;
    rc = sage_attn_fwd(buf, o, B, H, Nq, Nkv, D, q_dev, kv_dev, sm_scale, stream);
    if (rc != SAGE_OK) return rc;
    g_last_launches += prep_launches;
    if (!output->host || !output->device) return SAGE_ERR_ARG;
    if (cudaMemcpyAsync(const_cast<void*>(output->host), output->device, output->bytes, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess)
        return SAGE_ERR_LAUNCH;
    return SAGE_OK;
}

// Copy rows [0, host_len(lens, b, n)) of heads [h0, h0 + nh) of a [B, H, n, D]
// BF16 tensor (element strides of t; the same physical layout on both sides)
// with 2-D copies.
static int copy_heads(void* dst, const void* src, const sage_tensor* t, int B, const int32_t* lens, int n, int D,
                      int h0, int nh, cudaMemcpyKind kind, cudaStream_t s) {
    const int64_t sb = t->stride_b, sh = t->stride_h, sn = t->stride_n;
    for (int b = 0; b < B; ++b) {
        const int N = host_len(lens, b, n);
        if (N <= 0) continue;
        const int64_t off = (b * sb + (int64_t)h0 * sh) * 2;
        char* d = static_cast<char*>(dst) + off;
        const char* c = static_cast<const char*>(src) + off;
        cudaError_t e;
        if (sh == D && sn >= (int64_t)nh * D)          // a row holds the head range contiguously
            e = cudaMemcpy2DAsync(d, sn * 2, c, sn * 2, (size_t)nh * D * 2, (size_t)N, kind, s);
        else if (sn == D && sh >= (int64_t)N * D)      // each head's valid rows are one contiguous block
            e = cudaMemcpy2DAsync(d, sh * 2, c, sh * 2, (size_t)N * D * 2, (size_t)nh, kind, s);
        else {
            e = cudaSuccess;
            for (int h = 0; h < nh && e == cudaSuccess; ++h)
                e = cudaMemcpy2DAsync(d + h * sh * 2, sn * 2, c + h * sh * 2, sn * 2, (size_t)D * 2, (size_t)N, kind,
                                      s);
        }
        if (e != cudaSuccess) return SAGE_ERR_LAUNCH;
    }
    return SAGE_OK;
}

// Streams and events of the overlapped host entry, created once per device.
struct OverlapStreams {
    cudaStream_t s[3] = {};
    cudaEvent_t start = nullptr, done[3] = {};
    bool ready = false;
};
static OverlapStreams g_overlap[64];

static OverlapStreams* overlap_streams() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    OverlapStreams& o = g_overlap[dev];
    if (!o.ready) {
        for (int i = 0; i < 3; ++i)
            if (cudaStreamCreateWithFlags(&o.s[i], cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&o.done[i], cudaEventDisableTiming) != cudaSuccess)
                return nullptr;
        if (cudaEventCreateWithFlags(&o.start, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        o.ready = true;
    }
    return &o;
}

int sage_attention_host_overlapped(const sage_tensor* q_host, const sage_tensor* k_host, const sage_tensor* v_host,
                                   const sage_tensor* o_host, const sage_tensor* q, const sage_tensor* k,
                                   const sage_tensor* v, const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                                   const int32_t* q_len, const int32_t* kv_len, float sm_scale, int causal,
                                   int head_groups, const sage_prep_buffers* buf, void* stream) {
    int rc = check_shape(B, H, Nq, Nkv, D);
    if (rc != SAGE_OK) return rc;
    if (head_groups < 1 || head_groups > H) return SAGE_ERR_ARG;
    const sage_tensor* hs[4] = {q_host, k_host, v_host, o_host};
    const sage_tensor* ds[4] = {q, k, v, o};
    for (int i = 0; i < 4; ++i) {
        if (hs[i] == nullptr || hs[i]->ptr == nullptr) return SAGE_ERR_ARG;
        if ((rc = check_tensor(ds[i])) != SAGE_OK) return rc;
        if (hs[i]->stride_b != ds[i]->stride_b || hs[i]->stride_h != ds[i]->stride_h ||
            hs[i]->stride_n != ds[i]->stride_n)
            return SAGE_ERR_ARG;
    }
    OverlapStreams* os = overlap_streams();
    if (os == nullptr) return SAGE_ERR_LAUNCH;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    const int32_t *q_dev = nullptr, *kv_dev = nullptr;
    if ((rc = stage_host_lens(buf, B, H, Nq, Nkv, D, q_len, kv_len, user, &q_dev, &kv_dev)) != SAGE_OK) return rc;
    if (cudaEventRecord(os->start, user) != cudaSuccess) return SAGE_ERR_LAUNCH;
    for (int i = 0; i < 3; ++i)
        if (cudaStreamWaitEvent(os->s[i], os->start, 0) != cudaSuccess) return SAGE_ERR_LAUNCH;
    int launches = 0;
    for (int g = 0; g < head_groups && rc == SAGE_OK; ++g) {
        const int h0 = (int)((int64_t)H * g / head_groups), h1 = (int)((int64_t)H * (g + 1) / head_groups);
        cudaStream_t s = os->s[g % 3];
        if ((rc = copy_heads(const_cast<void*>(q->ptr), q_host->ptr, q, B, q_len, Nq, D, h0, h1 - h0,
                             cudaMemcpyHostToDevice, s)) != SAGE_OK ||
            (rc = copy_heads(const_cast<void*>(k->ptr), k_host->ptr, k, B, kv_len, Nkv, D, h0, h1 - h0,
                             cudaMemcpyHostToDevice, s)) != SAGE_OK ||
            (rc = copy_heads(const_cast<void*>(v->ptr), v_host->ptr, v, B, kv_len, Nkv, D, h0, h1 - h0,
                             cudaMemcpyHostToDevice, s)) != SAGE_OK)
            break;
        rc = prep_common(q, k, v, B, H, Nq, Nkv, D, q_dev, kv_dev, kSV, buf, s, h0, h1 - h0);
        if (rc != SAGE_OK) break;
        launches += g_last_launches;
        rc = attn_common(buf, o, nullptr, B, H, Nq, Nkv, D, q_dev, kv_dev, sm_scale, s, false, causal != 0,
                         nullptr, false, h0, h1 - h0);
        if (rc != SAGE_OK) break;
        launches += g_last_launches;
        rc = copy_heads(const_cast<void*>(o_host->ptr), o->ptr, o, B, q_len, Nq, D, h0, h1 - h0,
                        cudaMemcpyDeviceToHost, s);
    }
    // the caller's stream resumes after every group, also on an error
    for (int i = 0; i < 3; ++i) {
        if (cudaEventRecord(os->done[i], os->s[i]) != cudaSuccess) return SAGE_ERR_LAUNCH;
        if (cudaStreamWaitEvent(user, os->done[i], 0) != cudaSuccess) return SAGE_ERR_LAUNCH;
    }
    if (rc == SAGE_OK) g_last_launches = launches;
    return rc;
}

int sage_get_device_status(void) {
    int* st = device_status_ptr();
    if (st == nullptr) return SAGE_ERR_LAUNCH;
    if (cudaDeviceSynchronize() != cudaSuccess) return SAGE_ERR_LAUNCH;
    int words[kStatusWords] = {0, 0, 0, 0};
    if (cudaMemcpy(words, st, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return SAGE_ERR_LAUNCH;
    const int zero[kStatusWords] = {0, 0, 0, 0};
    if (cudaMemcpy(st, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SAGE_ERR_LAUNCH;
    return words[0];
}

const char* sage_status_string(int code) {
    switch (code) {
        case SAGE_OK: return "ok";
        case SAGE_ERR_ARG: return "invalid argument";
        case SAGE_ERR_UNSUPPORTED: return "unsupported shape, alignment or stride";
        case SAGE_ERR_LAUNCH: return "CUDA launch error";
        case SAGE_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case SAGE_ERR_DRIVER: return "driver entry point cuTensorMapEncodeTiled unavailable";
        case SAGE_ERR_SCRATCH: return "problem needs more scratch than the no-allocation entry point holds";
        default: return "unknown status";
    }
}

int sage_last_launch_count(void) { return g_last_launches; }

// Test hook (not part of the public header): the next sage_attn_fwd launch
// withholds one V tile copy so its consumer's bounded wait runs out.
int sage_debug_inject_fault(int mode) {
    fault_mode_for_next_launch = mode;
    return SAGE_OK;
}

// Test hook: preparation form for later calls (process-wide, tests only).
// one_pass = 1 selects the single launch that reads K and V once instead of
// the three plain launches; lag > 0 fixes its queue lag in heads.
int sage_debug_epilogue_mode(int tma_store) {
    g_tma_epilogue = tma_store != 0;
    return SAGE_OK;
}

int sage_debug_prep_mode(int one_pass, int lag) {
    g_prep_one_pass = one_pass != 0;
    g_prep_lag = lag > 0 ? lag : 0;
    return SAGE_OK;
}

}  // extern "C"
