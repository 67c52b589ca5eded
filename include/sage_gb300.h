/*
 * sage_gb300.h - C ABI of the GB300 (sm_103a) quantized exact attention library.
 *
 * The library implements the numerical contract whose stages the Experiment
 * Log lists under "Phase 0 Import And Verification": Q/K preparation, K
 * smoothing, INT8 quantization, QK traversal, online softmax, FP8 V/P,
 * two-level PV accumulation, final conversion and ragged tails; with the
 * strict tile order, exact FP8 score bytes and per-tile RO rescaling named
 * under "Phase 1 State-Ownership Decision", and the checkpoint list (QK, m,
 * d, FP8 probability, rescale, FP16 PV, FP32 RO, reciprocal, BF16 output) of
 * "Phase 2B Fixed Aligned Numerical Prototype".  Strided NHD views of a fused
 * projection buffer are accepted directly (Experiment Registry, "Complete
 * Registry", row qkv-direct-sageattention-layout); the library never makes a
 * padded copy (row layout-direct-q-padding-32) and never allocates on the hot
 * path (row layout-dynamic-to-hot-allocation).
 *
 * Conventions for every entry point:
 *  - All buffers are caller-owned.  Device pointers must be device memory of
 *    the current CUDA device; host pointers (sage_attention_host only) should
 *    be pinned for asynchronous copies.  The library allocates nothing, frees
 *    nothing and does not synchronize, except sage_get_device_status.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued on it; results are ready when the stream completes.
 *  - Return value: SAGE_OK (0) when the work was enqueued, or a negative
 *    SAGE_ERR_* code when arguments were rejected (nothing enqueued) or the
 *    launch failed.  Errors found on the device (a bounded wait that ran out)
 *    are recorded in a device status word read by sage_get_device_status.
 *  - Head dimension D = 64 or 128.  Q, K, V and O are BF16.
 */
#ifndef SAGE_GB300_H
#define SAGE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum sage_status {
    SAGE_OK = 0,
    SAGE_ERR_ARG = -1,          /* null pointer, non-positive size, bad length */
    SAGE_ERR_UNSUPPORTED = -2,  /* D not 64 or 128, misaligned pointer or stride */
    SAGE_ERR_LAUNCH = -3,       /* CUDA reported an error at launch */
    SAGE_ERR_TIMEOUT = -4,      /* device: a bounded wait inside a kernel ran out */
    SAGE_ERR_DRIVER = -5,       /* driver entry point for TMA descriptors missing */
    SAGE_ERR_SCRATCH = -6       /* problem needs more scratch than the fixed buffer
                                   of sage_prep_qkv_noalloc holds */
};

/* Logical [B, H, N, D] BF16 tensor given by its element strides; the D stride
 * is 1.  NHD ([B,N,H,D]) and HND ([B,H,N,D]) layouts and strided views into a
 * fused QKV buffer are all described this way.  ptr and the three strides
 * (in bytes) must be multiples of 16 bytes. */
typedef struct {
    const void* ptr;
    int64_t stride_b;
    int64_t stride_h;
    int64_t stride_n;
} sage_tensor;

/* Outputs of sage_prep_qkv / inputs of sage_attn_fwd (all device memory).
 * Sizes are given by sage_buffer_sizes.  Nkv_pad = Nkv rounded up to 16.
 *   q16     fp16 [B, H, Nq, D]      INT8 Q codes held as exact FP16 integers
 *   k16     fp16 [B, H, Nkv, D]     INT8 codes of the smoothed K, as FP16
 *   v8t     e4m3 [B, H, D, Nkv_pad] FP8 V codes, token index fastest
 *   q_scale f32  [B, H, ceil(Nq/128)]  per 128-row Q block
 *   k_scale f32  [B, H, ceil(Nkv/64)]  per 64-row K block
 *   v_scale f32  [B, H, D]          per channel
 *   k_mean  f32  [B, H, D]          channel mean removed from K
 *   q8, k8  int8 [B, H, Nq|Nkv, D]  optional INT8 code bytes (NULL: skipped)
 *   workspace                       scratch of sage_buffer_sizes().workspace (its last
 *                                   8*B bytes, rounded up to 16, are the lengths slot of
 *                                   the host-memory entries)
 * Rows at or beyond a batch item's valid length are written as code 0 and
 * scales of blocks holding no valid row are 0, so no uninitialised byte is
 * ever read by sage_attn_fwd. */
typedef struct {
    uint16_t* q16;
    uint16_t* k16;
    uint8_t* v8t;
    float* q_scale;
    float* k_scale;
    float* v_scale;
    float* k_mean;
    int8_t* q8;
    int8_t* k8;
    void* workspace;
    size_t workspace_bytes;
} sage_prep_buffers;

typedef struct {
    size_t q16, k16, v8t, q_scale, k_scale, v_scale, k_mean, q8, k8, workspace;
    int64_t nkv_pad;
} sage_sizes;

/* Byte sizes of every buffer of sage_prep_buffers for a problem shape.
 * Returns SAGE_ERR_ARG / SAGE_ERR_UNSUPPORTED for bad shapes. */
int sage_buffer_sizes(int B, int H, int Nq, int Nkv, int D, sage_sizes* out);

/* Preparation (Experiment Log, "Phase 0 Import And Verification": Q/K
 * preparation, K smoothing, INT8 quantization, FP8 V).  Three kernel
 * launches: K/V channel statistics with the Q quantization, the per-head
 * finalize, and the K/V quantization.
 *  q, k, v : BF16 inputs [B,H,Nq,D], [B,H,Nkv,D], [B,H,Nkv,D] (device).
 *  q_len, kv_len : device int32 [B] valid lengths (<= Nq, <= Nkv), or NULL
 *                  for all rows valid.  Out-of-range lengths are clamped.
 *  out : device buffers, filled completely (see sage_prep_buffers).
 * Steps: per (b,h,channel) mean of the valid keys in a fixed order (chunks of
 * 64 tokens summed in order, chunk sums in order, one division); K - mean;
 * per-block amax, scale = amax/127, codes rne(x*127/amax); V per channel to
 * e4m3 with scale amax/1.125.  Calls on the same workspace must be ordered
 * (one stream, or events): the workspace holds the call's statistics and its
 * synchronisation words. */
int sage_prep_qkv(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                  int B, int H, int Nq, int Nkv, int D,
                  const int32_t* q_len, const int32_t* kv_len,
                  const sage_prep_buffers* out, void* stream);

/* Fused attention (QK traversal through FP32 running output and BF16
 * conversion).  `in` holds the output of sage_prep_qkv for the same shape and
 * lengths.  o : BF16 [B,H,Nq,D] output (device); rows >= q_len[b] are not
 * written; rows of a batch item with kv_len = 0 are written as zero.
 * sm_scale <= 0 selects 1/sqrt(D).  One kernel: per 128-row query tile, a TMA
 * producer warp, a single-thread tcgen05 MMA issuer (QK on FP16 integer codes
 * with FP32 accumulation, PV as e4m3 x e4m3 with P taken from tensor memory),
 * a softmax warpgroup and a correction/epilogue warpgroup. */
int sage_attn_fwd(const sage_prep_buffers* in, const sage_tensor* o,
                  int B, int H, int Nq, int Nkv, int D,
                  const int32_t* q_len, const int32_t* kv_len,
                  float sm_scale, void* stream);

/* Causal form of sage_attn_fwd (the pages describe only the non-causal
 * path; this is the same contract with a mask).  Query i of batch item b sees
 * key j iff j <= i + (kv_len[b] - q_len[b]): the diagonal runs through the
 * last query and the last key, so j <= i when the lengths are equal.  Rows
 * that see no key are written as zero.  Arguments, layouts, ownership and
 * errors are those of sage_attn_fwd.  Each query tile reads only the KV
 * tiles up to its diagonal; hidden keys inside a tile are masked, and a row's
 * result equals the non-causal result over the keys it sees. */
int sage_attn_fwd_causal(const sage_prep_buffers* in, const sage_tensor* o,
                         int B, int H, int Nq, int Nkv, int D,
                         const int32_t* q_len, const int32_t* kv_len,
                         float sm_scale, void* stream);

/* One call from BF16 Q/K/V to the BF16 output, with the Q preparation fused
 * into the attention kernel (the pages run preparation and attention as
 * separate stages; fusing them skips the round trip of the Q codes through
 * device memory).
 *  q, k, v : BF16 [B,H,Nq,D], [B,H,Nkv,D], [B,H,Nkv,D] views (device), as for
 *            sage_prep_qkv; o : BF16 [B,H,Nq,D] output (device), as for
 *            sage_attn_fwd.
 *  causal  : 0 = the sage_attn_fwd contract, 1 = the sage_attn_fwd_causal one.
 *  buf     : k16, v8t, k_scale, v_scale, k_mean, workspace (and k8 if not
 *            NULL) are filled as by sage_prep_qkv; q16 and q8 are not used
 *            and may be NULL.  q_scale receives the Q block scales of every
 *            query tile that has a valid row and at least one visible key.
 * Enqueues the K/V preparation (three kernels) and one attention kernel whose
 * CTAs load their 128-row BF16 Q block, compute its INT8 scale and codes with
 * the same arithmetic as sage_prep_qkv, and write the codes over the block in
 * shared memory before the first QK.  The output is bit-identical to
 * sage_prep_qkv followed by sage_attn_fwd / sage_attn_fwd_causal. */
int sage_attention(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                   const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                   const int32_t* q_len, const int32_t* kv_len, float sm_scale, int causal,
                   const sage_prep_buffers* buf, void* stream);

/* The "QK" checkpoint: exact integer scores S[b,h,i,j] = sum_d q8*k8 from the
 * same tensor-core path sage_attn_fwd uses, written as int32 to
 * s [B, H, Nq, Nkv] (device, row-major).  Entries with i >= q_len[b] or
 * j >= kv_len[b] are not written. */
int sage_qk_int32(const sage_prep_buffers* in, int32_t* s,
                  int B, int H, int Nq, int Nkv, int D,
                  const int32_t* q_len, const int32_t* kv_len, void* stream);

/* The BKV = 64 form of the contract, matching the 64-key epochs of Experiment
 * Log, "Phase 2A" (64-key K/V slots): the online-softmax tile and the inner
 * FP16 PV sum cover 64 keys, and V is quantized to |v| <= S_V = 144/64 = 2.25
 * so that 64 * 448 * S_V stays within the FP16 range.  bkv = 128 gives the
 * default contract (identical to sage_prep_qkv / sage_attn_fwd[_causal]);
 * any other value returns SAGE_ERR_UNSUPPORTED.  Prepare and attend with the
 * same bkv: only V's codes and scales depend on it.  Other arguments,
 * layouts and errors as for sage_prep_qkv and sage_attn_fwd; causal as for
 * sage_attn_fwd_causal. */
int sage_prep_qkv_bkv(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                      int B, int H, int Nq, int Nkv, int D,
                      const int32_t* q_len, const int32_t* kv_len, int bkv,
                      const sage_prep_buffers* out, void* stream);
int sage_attn_fwd_bkv(const sage_prep_buffers* in, const sage_tensor* o,
                      int B, int H, int Nq, int Nkv, int D,
                      const int32_t* q_len, const int32_t* kv_len, float sm_scale,
                      int bkv, int causal, void* stream);

/* Stage checkpoints of one query tile (device buffers, caller-owned).  T is
 * the number of 128-key tiles the tile visits: ceil(kv_len/128), or up to its
 * diagonal for the causal form; size every buffer for T = ceil(Nkv/128).
 * Scale conventions: m, alpha, p8, pv16 and ro are the contract's values (m in
 * the log2 domain of the scaled scores); l and recip carry the 448 scale of P,
 * i.e. l = 448 * sum(p) and recip = 1 / (448 * sum(p)). */
typedef struct {
    float* m;          /* [T][128]       running maximum after tile t */
    float* l;          /* [T][2][128]    running sum of each half row (keys 0-63, 64-127 of every
                                         tile) after tile t; the row's l is their sum */
    float* alpha;      /* [T][128]       rescale factor 2^(m_old - m_new) of tile t */
    uint8_t* p8;       /* [T][128][128]  e4m3 P bytes of tile t, key index fastest */
    uint16_t* pv16;    /* [T][128][D]    FP16 PV tile sums (bit patterns) */
    float* ro;         /* [T][128][D]    FP32 running output after tile t */
    float* recip;      /* [128]          reciprocal of the final l */
} sage_checkpoints;

/* The checkpoint list of Experiment Log, "Phase 2B Fixed Aligned Numerical
 * Prototype" (QK, m, d, FP8 probability, rescale, FP16 PV, FP32 RO,
 * reciprocal) for one query tile: runs the attention kernel of sage_attn_fwd
 * (causal = 0) or sage_attn_fwd_causal (causal = 1) as a single CTA for query
 * rows [128*qtile, 128*qtile + 128) of head (b, h), writing that tile's output
 * rows to o as usual and its stage values to ck (rows >= q_len hold
 * don't-care values).  The QK checkpoint is sage_qk_int32.  Arguments as for
 * sage_attn_fwd; SAGE_ERR_ARG for a NULL checkpoint buffer or an out-of-range
 * (b, h, qtile), SAGE_ERR_UNSUPPORTED for a buffer not 16-byte aligned. */
int sage_attn_checkpoints(const sage_prep_buffers* in, const sage_tensor* o,
                          int B, int H, int Nq, int Nkv, int D,
                          const int32_t* q_len, const int32_t* kv_len, float sm_scale, int causal,
                          int b, int h, int qtile, const sage_checkpoints* ck, void* stream);

/* One host<->device region copied with one cudaMemcpyAsync. */
typedef struct {
    const void* host;
    void* device;
    size_t bytes;
} sage_copy;

/* End-to-end call from host memory: copies every `inputs` region host->device,
 * runs sage_prep_qkv and sage_attn_fwd on the device views q, k, v, o (which
 * point into those regions), then copies `output` device->host, all on
 * `stream`, without synchronizing.
 *  q_len, kv_len : HOST int32 [B] valid lengths (clamped to [0, Nq] and
 *                  [0, Nkv]), or NULL for all rows valid.  They are copied
 *                  on `stream` into the lengths slot at the end of
 *                  buf->workspace.  Pageable arrays are staged before the
 *                  call returns and may be reused at once; pinned arrays are
 *                  read when the stream reaches the copy and must not change
 *                  before then.  Rows >= q_len[b] of the device output are
 *                  not written; the `output` region is copied back as given. */
int sage_attention_host(const sage_copy* inputs, int n_inputs,
                        const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                        const sage_prep_buffers* buf, const sage_tensor* o,
                        const sage_copy* output,
                        int B, int H, int Nq, int Nkv, int D,
                        const int32_t* q_len, const int32_t* kv_len, float sm_scale, void* stream);

/* The CTA-pair launch form of sage_attn_fwd (causal = 0) and
 * sage_attn_fwd_causal (causal = 1): adjacent query tiles run as clusters of
 * two CTAs sharing each tensor-core instruction (tcgen05 .cta_group::2, 256
 * rows), each CTA loading half of every K and V tile.  Both forms compute the
 * same values in the same order, so the output is bit-identical to the
 * one-CTA form's.  Arguments, layouts and errors as for sage_attn_fwd.  On
 * GB300 the paired form is slower for this kernel (every tile's PV waits for
 * P-ready arrivals from both CTAs, which cross SMs); the other entry points
 * always use one CTA per 128-row query tile. */
int sage_attn_fwd_pairs(const sage_prep_buffers* in, const sage_tensor* o,
                        int B, int H, int Nq, int Nkv, int D,
                        const int32_t* q_len, const int32_t* kv_len,
                        float sm_scale, int causal, void* stream);

/* End-to-end call from host memory with the copies overlapped with the
 * compute.  The heads of a problem are independent (K mean, quantization
 * scales and attention are all per (b, h)), so the call splits the heads into
 * head_groups contiguous ranges and, for each range on one of three internal
 * streams, copies its Q/K/V rows host->device, prepares them, runs the
 * attention and copies its output rows device->host; the copies of one range
 * overlap the kernels of the others.
 *  q_host, k_host, v_host, o_host : host (pinned) tensors with the same
 *            element strides as the device tensors q, k, v, o ([B,H,N,D]
 *            views, BF16); only the logical elements are copied, one 2-D
 *            copy per batch item and tensor when the heads of a row, or the
 *            rows of a head, are contiguous.
 *  causal  : 0 or 1 as for sage_attention.
 *  head_groups : 1 .. H.
 *  q_len, kv_len : HOST int32 [B] valid lengths, or NULL for all valid, as
 *            for sage_attention_host; only rows [0, q_len[b]) of Q and O and
 *            [0, kv_len[b]) of K and V are copied, so host output rows at or
 *            beyond q_len[b] are left untouched.
 *  buf     : full-size buffers as for sage_prep_qkv (each range uses its own
 *            heads' slices).
 * The work is ordered after prior work on `stream` and later work on
 * `stream` waits for all of it; the call does not synchronize.  The internal
 * streams and events are created on the first call on a device and kept.
 * The output equals sage_prep_qkv + sage_attn_fwd[_causal] on the same
 * inputs bit for bit.  SAGE_ERR_ARG for a NULL host pointer, mismatched
 * strides or head_groups out of range. */
int sage_attention_host_overlapped(const sage_tensor* q_host, const sage_tensor* k_host,
                                   const sage_tensor* v_host, const sage_tensor* o_host,
                                   const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                                   const sage_tensor* o, int B, int H, int Nq, int Nkv, int D,
                                   const int32_t* q_len, const int32_t* kv_len,
                                   float sm_scale, int causal, int head_groups,
                                   const sage_prep_buffers* buf, void* stream);

/* Synchronizes the device, returns the first error a kernel recorded since
 * the last call (SAGE_OK if none) and clears it. */
int sage_get_device_status(void);

/* Static description of a status code. */
const char* sage_status_string(int code);

/* Number of kernel launches the last successful sage_prep_qkv / sage_attn_fwd
 * call enqueued (for launch accounting). */
int sage_last_launch_count(void);

/* Preparation for callers that cannot allocate device memory.  The paper has
 * no counterpart: this is a deployment variant of sage_prep_qkv.  Some
 * callers cannot call cudaMalloc for the scratch sage_prep_qkv needs, for
 * example a plugin of an inference engine whose enqueue hook receives only
 * its input and output pointers, or host code that runs while the device
 * memory pool is fully committed.  This entry point takes the same arguments
 * and fills the same outputs bit for bit, but ignores out->workspace and uses
 * a fixed 16 MiB device array inside the library instead, which every GPU that
 * loads the library holds until the process exits.  Its V codes and scales
 * are those of the default BKV = 128 contract (|v| <= 1.125): pair it with
 * sage_attn_fwd, sage_attn_fwd_causal or sage_attn_fwd_bkv(bkv = 128), not
 * with the BKV = 64 form, whose V scaling differs.
 *  - Allocates nothing (no cudaMalloc/cudaFree, no allocating library call).
 *  - The first call on a device looks up that device's address of the array
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - All calls on a device share the array, which keeps the last call's
 *    contents; the kernels write every scratch word before reading it, so no
 *    clearing is needed.  Calls whose kernels may overlap on the GPU (e.g. on
 *    unordered streams) race on the array: order them.
 *  - Returns SAGE_ERR_SCRATCH, enqueueing nothing, when the problem needs more
 *    than sage_prep_noalloc_capacity() bytes of scratch (the workspace size
 *    sage_buffer_sizes reports). */
int sage_prep_qkv_noalloc(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                          int B, int H, int Nq, int Nkv, int D,
                          const int32_t* q_len, const int32_t* kv_len,
                          const sage_prep_buffers* out, void* stream);

/* Bytes of scratch available to sage_prep_qkv_noalloc (16 MiB). */
size_t sage_prep_noalloc_capacity(void);

/* Test hook for the failure-detection tests: mode 1 makes the next
 * sage_attn_fwd launch withhold its V tile copies, so the MMA issuer's
 * bounded wait runs out, the kernel records SAGE_ERR_TIMEOUT, releases its
 * tensor memory and returns; mode 0 restores normal launches.  Use only on
 * a problem of one or a few query tiles (each CTA waits about one second). */
int sage_debug_inject_fault(int mode);

/* Test hook for the preparation tests and measurements (process-wide; not
 * for production use): one_pass = 1 makes later preparation calls use a
 * single launch that reads K and V from HBM once (a work queue in which each
 * head's K/V quantization trails its channel statistics, re-reading K and V
 * from L2) instead of the default three launches (statistics and Q,
 * finalize, K/V quantization); both compute the same bytes, and the single
 * launch is the slower of the two on GB300.  lag > 0 fixes how many heads the
 * K/V items trail their statistics (0: chosen from the grid size). */
int sage_debug_prep_mode(int one_pass, int lag);

/* Test hook for the attention tests and measurements (process-wide; not for
 * production use): tma_store = 1 makes later sage_attn_fwd and
 * sage_attn_fwd_causal launches (the other forms are unaffected) write each
 * output tile whose rows are all valid through a TMA store of the BF16 tile
 * staged in shared memory (a partial tile of a shorter batch item is still
 * written row by row); 0 (default) writes every row with per-thread 16-byte
 * stores.  Both write the same bytes; the TMA form is the slower one on
 * GB300. */
int sage_debug_epilogue_mode(int tma_store);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_GB300_H */
