// sage_noalloc.cu - preparation entry point for callers that cannot allocate.
//
// sage_prep_qkv needs a caller-provided scratch buffer (per-chunk K sums,
// per-chunk V maxima, V inverse scales).  Some callers cannot obtain one: an
// inference-engine plugin whose enqueue hook is handed only its input and
// output pointers, or host code running while the device memory pool is
// fully committed or locked, must not call cudaMalloc.  For them this file
// keeps the scratch in a fixed device array that every GPU which loads the
// library holds until the process exits; the caller still passes all inputs
// and outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  The preparation kernels write every scratch word they later
// read, so nothing has to be cleared between calls.  Calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on
// the array.
#include <mutex>

#include "sage_gb300.h"
#include "sage_internal.h"

namespace sage {
namespace {

// 16 MiB.  A problem needs 1 KiB per (b, h, 64-token chunk) plus 512 B per
// (b, h): B*H*ceil(Nkv/64) up to about 16,000, e.g. 24 heads of 16K tokens
// (6,144 chunk rows, 6.3 MB) or 256 heads of 2K tokens (8,192, 8.5 MB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) float g_prep_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
float* g_scratch_dev[64] = {};

// Device address of g_prep_scratch on the current device; looked up once per
// device with that device current.  Host code must never pass the symbol
// itself to a kernel: on the host it names a stand-in, not device memory.
float* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_dev[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_prep_scratch) != cudaSuccess) return nullptr;
        g_scratch_dev[dev] = static_cast<float*>(ptr);
    }
    return g_scratch_dev[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_view(const sage_tensor* t) {
    if (t == nullptr || t->ptr == nullptr) return SAGE_ERR_ARG;
    if (!aligned16(t->ptr) || (t->stride_b % 8) || (t->stride_h % 8) || (t->stride_n % 8) ||
        t->stride_b < 0 || t->stride_h < 0 || t->stride_n < 0)
        return SAGE_ERR_UNSUPPORTED;
    return SAGE_OK;
}

}  // namespace
}  // namespace sage

using namespace sage;

extern "C" size_t sage_prep_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" int sage_prep_qkv_noalloc(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                                     int B, int H, int Nq, int Nkv, int D,
                                     const int32_t* q_len, const int32_t* kv_len,
                                     const sage_prep_buffers* out, void* stream) {
    sage_sizes sz;
    int rc = sage_buffer_sizes(B, H, Nq, Nkv, D, &sz);
    if (rc != SAGE_OK) return rc;
    if (sz.workspace > kNoAllocScratchBytes) return SAGE_ERR_SCRATCH;
    if ((rc = check_view(q)) != SAGE_OK || (rc = check_view(k)) != SAGE_OK || (rc = check_view(v)) != SAGE_OK)
        return rc;
    if (out == nullptr || !out->q16 || !out->k16 || !out->v8t || !out->q_scale || !out->k_scale ||
        !out->v_scale || !out->k_mean)
        return SAGE_ERR_ARG;
    const void* ptrs[] = {out->q16, out->k16, out->v8t, out->q_scale, out->k_scale, out->v_scale, out->k_mean};
    for (const void* p : ptrs)
        if (!aligned16(p)) return SAGE_ERR_UNSUPPORTED;
    if ((out->q8 && !aligned16(out->q8)) || (out->k8 && !aligned16(out->k8))) return SAGE_ERR_UNSUPPORTED;

    float* scratch = scratch_for_current_device();
    if (scratch == nullptr) return SAGE_ERR_LAUNCH;

    PrepParams p{};
    p.q = static_cast<const uint16_t*>(q->ptr);
    p.k = static_cast<const uint16_t*>(k->ptr);
    p.v = static_cast<const uint16_t*>(v->ptr);
    p.qsb = q->stride_b; p.qsh = q->stride_h; p.qsn = q->stride_n;
    p.ksb = k->stride_b; p.ksh = k->stride_h; p.ksn = k->stride_n;
    p.vsb = v->stride_b; p.vsh = v->stride_h; p.vsn = v->stride_n;
    p.B = B; p.H = H; p.h_begin = 0; p.h_count = H; p.Nq = Nq; p.Nkv = Nkv; p.D = D; p.sv = kSV;
    p.nkv_pad = (int)sz.nkv_pad;
    p.nq_blocks = (int)ceil_div(Nq, kBQS);
    p.nk_blocks = (int)ceil_div(Nkv, kBKS);
    p.n_chunks = (int)ceil_div(Nkv, kMeanChunk);
    p.q_len = q_len; p.kv_len = kv_len;
    p.q16 = out->q16; p.k16 = out->k16; p.v8t = out->v8t;
    p.q8 = out->q8; p.k8 = out->k8;
    p.q_scale = out->q_scale; p.k_scale = out->k_scale; p.v_scale = out->v_scale; p.k_mean = out->k_mean;
    set_prep_workspace(p, scratch);
    p.status = device_status_ptr();
    int launches = 0;
    if (launch_prep(p, true, static_cast<cudaStream_t>(stream), &launches) != cudaSuccess) return SAGE_ERR_LAUNCH;
    set_last_launch_count(launches);
    return SAGE_OK;
}
