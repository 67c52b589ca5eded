"""GB300 (sm_103a) quantized exact attention: Python binding of libsage_gb300.so.

This module only marshals arguments for the C ABI declared in
``include/sage_gb300.h``; every step of the computation runs in the CUDA
kernels of the shared library.  PyTorch is used to allocate device memory and
to hand over CUDA streams.  There is no CPU fallback: if the compiled library
is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import functools
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsage_gb300.so")

SAGE_OK = 0
SAGE_ERR_ARG = -1
SAGE_ERR_UNSUPPORTED = -2
SAGE_ERR_LAUNCH = -3
SAGE_ERR_TIMEOUT = -4
SAGE_ERR_DRIVER = -5
SAGE_ERR_SCRATCH = -6

D_HEAD = 128
HEAD_DIMS = (64, 128)       # head dimensions the kernels are built for

# Names the header declares (checked by the CPU tests against the .so exports).
EXPORTED = ("sage_buffer_sizes", "sage_prep_qkv", "sage_attn_fwd", "sage_attn_fwd_causal", "sage_attention",
            "sage_attn_checkpoints", "sage_prep_qkv_bkv", "sage_attn_fwd_bkv", "sage_attn_fwd_pairs",
            "sage_attention_host_overlapped",
            "sage_qk_int32",
            "sage_attention_host", "sage_get_device_status", "sage_status_string",
            "sage_last_launch_count", "sage_debug_inject_fault", "sage_debug_prep_mode",
            "sage_debug_epilogue_mode", "sage_prep_qkv_noalloc",
            "sage_prep_noalloc_capacity")


class SageError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class sage_tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_h", ctypes.c_int64), ("stride_n", ctypes.c_int64)]


class sage_prep_buffers(ctypes.Structure):
    _fields_ = [("q16", ctypes.c_void_p), ("k16", ctypes.c_void_p), ("v8t", ctypes.c_void_p),
                ("q_scale", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("k_mean", ctypes.c_void_p),
                ("q8", ctypes.c_void_p), ("k8", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class sage_sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("q16", "k16", "v8t", "q_scale", "k_scale", "v_scale", "k_mean", "q8", "k8",
                 "workspace")] + [("nkv_pad", ctypes.c_int64)]


class sage_checkpoints(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("m", "l", "alpha", "p8", "pv16", "ro", "recip")]


class sage_copy(ctypes.Structure):
    _fields_ = [("host", ctypes.c_void_p), ("device", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsage_gb300.so not found at {path}; run quantized_exact_attention_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    i, vp, f = ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    lib.sage_buffer_sizes.argtypes = [i, i, i, i, i, P(sage_sizes)]
    lib.sage_prep_qkv.argtypes = [P(sage_tensor), P(sage_tensor), P(sage_tensor), i, i, i, i, i, vp, vp,
                                  P(sage_prep_buffers), vp]
    lib.sage_attn_fwd.argtypes = [P(sage_prep_buffers), P(sage_tensor), i, i, i, i, i, vp, vp, f, vp]
    lib.sage_attn_fwd_causal.argtypes = lib.sage_attn_fwd.argtypes
    lib.sage_prep_qkv_bkv.argtypes = [P(sage_tensor), P(sage_tensor), P(sage_tensor), i, i, i, i, i, vp, vp, i,
                                      P(sage_prep_buffers), vp]
    lib.sage_attn_fwd_bkv.argtypes = [P(sage_prep_buffers), P(sage_tensor), i, i, i, i, i, vp, vp, f, i, i, vp]
    lib.sage_attn_checkpoints.argtypes = [P(sage_prep_buffers), P(sage_tensor), i, i, i, i, i, vp, vp, f, i,
                                          i, i, i, P(sage_checkpoints), vp]
    lib.sage_attention.argtypes = [P(sage_tensor), P(sage_tensor), P(sage_tensor), P(sage_tensor),
                                   i, i, i, i, i, vp, vp, f, i, P(sage_prep_buffers), vp]
    lib.sage_qk_int32.argtypes = [P(sage_prep_buffers), vp, i, i, i, i, i, vp, vp, vp]
    lib.sage_attention_host.argtypes = [P(sage_copy), i, P(sage_tensor), P(sage_tensor), P(sage_tensor),
                                        P(sage_prep_buffers), P(sage_tensor), P(sage_copy),
                                        i, i, i, i, i, vp, vp, f, vp]
    lib.sage_get_device_status.argtypes = []
    lib.sage_status_string.argtypes = [i]
    lib.sage_status_string.restype = ctypes.c_char_p
    lib.sage_last_launch_count.argtypes = []
    lib.sage_debug_inject_fault.argtypes = [i]
    lib.sage_debug_prep_mode.argtypes = [i, i]
    lib.sage_debug_epilogue_mode.argtypes = [i]
    lib.sage_debug_prep_mode.restype = ctypes.c_int
    lib.sage_attn_fwd_pairs.argtypes = [P(sage_prep_buffers), P(sage_tensor), i, i, i, i, i, vp, vp, f, i, vp]
    lib.sage_attention_host_overlapped.argtypes = [P(sage_tensor)] * 8 + [i, i, i, i, i, vp, vp, f, i, i,
                                                                          P(sage_prep_buffers), vp]
    lib.sage_prep_qkv_noalloc.argtypes = lib.sage_prep_qkv.argtypes
    lib.sage_prep_noalloc_capacity.argtypes = []
    for name in EXPORTED:
        if name not in ("sage_status_string", "sage_prep_noalloc_capacity"):
            getattr(lib, name).restype = ctypes.c_int
    lib.sage_prep_noalloc_capacity.restype = ctypes.c_size_t
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().sage_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != SAGE_OK:
        raise SageError(rc, what)


# torch's raw current-stream accessor (a handle without a Stream object); the
# public torch.cuda.current_stream() costs several microseconds per call
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(torch.cuda.current_device()) or None
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def tensor_desc(t: torch.Tensor) -> sage_tensor:
    """Describe a logical [B, H, N, D] BF16 view (any strides, D stride 1)."""
    if t.dim() != 4 or t.dtype != torch.bfloat16 or t.stride(3) != 1:
        raise ValueError("expected a [B, H, N, D] bfloat16 view with unit D stride")
    return sage_tensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def buffer_sizes(B: int, H: int, Nq: int, Nkv: int, D: int = D_HEAD) -> sage_sizes:
    s = sage_sizes()
    _check(load_library().sage_buffer_sizes(B, H, Nq, Nkv, D, ctypes.byref(s)), "sage_buffer_sizes")
    return s


@dataclass(frozen=True)
class PrepBuffers:
    """Device buffers of sage_prep_buffers, allocated by torch.  Frozen: the C
    struct of their addresses is built once and reused by every call."""
    q16: torch.Tensor
    k16: torch.Tensor
    v8t: torch.Tensor
    q_scale: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    k_mean: torch.Tensor
    q8: torch.Tensor | None
    k8: torch.Tensor | None
    workspace: torch.Tensor
    nkv_pad: int

    @functools.cached_property
    def _c(self) -> sage_prep_buffers:
        ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
        return sage_prep_buffers(ptr(self.q16), ptr(self.k16), ptr(self.v8t), ptr(self.q_scale),
                                 ptr(self.k_scale), ptr(self.v_scale), ptr(self.k_mean),
                                 ptr(self.q8), ptr(self.k8), ptr(self.workspace),
                                 self.workspace.numel())

    def c_struct(self) -> sage_prep_buffers:
        return self._c


def alloc_prep_buffers(B, H, Nq, Nkv, device="cuda", int8_codes=False, D=D_HEAD) -> PrepBuffers:
    sz = buffer_sizes(B, H, Nq, Nkv, D)
    pad = int(sz.nkv_pad)
    e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
    return PrepBuffers(
        q16=e((B, H, Nq, D), torch.float16), k16=e((B, H, Nkv, D), torch.float16),
        v8t=e((B, H, D, pad), torch.uint8),
        q_scale=e((B, H, (Nq + 127) // 128), torch.float32),
        k_scale=e((B, H, (Nkv + 63) // 64), torch.float32),
        v_scale=e((B, H, D), torch.float32), k_mean=e((B, H, D), torch.float32),
        q8=e((B, H, Nq, D), torch.int8) if int8_codes else None,
        k8=e((B, H, Nkv, D), torch.int8) if int8_codes else None,
        workspace=e((int(sz.workspace),), torch.uint8), nkv_pad=pad)


def _lens(x):
    if x is None:
        return None
    assert x.dtype == torch.int32 and x.is_cuda
    return x.data_ptr()


def sage_prep_qkv(q, k, v, bufs: PrepBuffers, q_len=None, kv_len=None, stream=None, bkv: int = 128):
    """Enqueue the preparation kernels on [B,H,N,D] BF16 views q, k, v.
    bkv = 64 prepares for the BKV = 64 contract (sage_prep_qkv_bkv)."""
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    qs, ks, vs, pb = tensor_desc(q), tensor_desc(k), tensor_desc(v), bufs.c_struct()
    lib = load_library()
    if bkv == 128:
        rc = lib.sage_prep_qkv(ctypes.byref(qs), ctypes.byref(ks), ctypes.byref(vs), B, H, Nq, Nkv, D,
                               _lens(q_len), _lens(kv_len), ctypes.byref(pb), _stream_ptr(stream))
    else:
        rc = lib.sage_prep_qkv_bkv(ctypes.byref(qs), ctypes.byref(ks), ctypes.byref(vs), B, H, Nq, Nkv, D,
                                   _lens(q_len), _lens(kv_len), int(bkv), ctypes.byref(pb), _stream_ptr(stream))
    _check(rc, "sage_prep_qkv")


def sage_prep_qkv_noalloc(q, k, v, bufs: PrepBuffers, q_len=None, kv_len=None, stream=None):
    """Like sage_prep_qkv, for callers that cannot allocate device memory:
    the library's fixed scratch array is used instead of bufs.workspace."""
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    qs, ks, vs, pb = tensor_desc(q), tensor_desc(k), tensor_desc(v), bufs.c_struct()
    rc = load_library().sage_prep_qkv_noalloc(ctypes.byref(qs), ctypes.byref(ks), ctypes.byref(vs), B, H, Nq,
                                              Nkv, D, _lens(q_len), _lens(kv_len), ctypes.byref(pb),
                                              _stream_ptr(stream))
    _check(rc, "sage_prep_qkv_noalloc")


def sage_prep_noalloc_capacity() -> int:
    return int(load_library().sage_prep_noalloc_capacity())


def sage_attn_fwd(bufs: PrepBuffers, o, q_len=None, kv_len=None, sm_scale: float = 0.0, stream=None,
                  Nkv: int | None = None, causal: bool = False, bkv: int = 128, pairs: bool = False):
    """Enqueue the fused attention kernel; o is a [B,H,Nq,D] BF16 view.
    causal=True calls sage_attn_fwd_causal (key j visible to query i iff
    j <= i + kv_len - q_len); bkv = 64 calls sage_attn_fwd_bkv; pairs=True
    calls sage_attn_fwd_pairs (the CTA-pair launch form)."""
    B, H, Nq, D = o.shape
    Nkv = bufs.k16.shape[2] if Nkv is None else Nkv
    os_, pb = tensor_desc(o), bufs.c_struct()
    lib = load_library()
    if pairs:
        if bkv != 128:
            raise ValueError("the CTA-pair form serves the BKV = 128 contract only")
        rc = lib.sage_attn_fwd_pairs(ctypes.byref(pb), ctypes.byref(os_), B, H, Nq, Nkv, D, _lens(q_len),
                                     _lens(kv_len), float(sm_scale), 1 if causal else 0, _stream_ptr(stream))
        _check(rc, "sage_attn_fwd_pairs")
        return
    if bkv != 128:
        rc = lib.sage_attn_fwd_bkv(ctypes.byref(pb), ctypes.byref(os_), B, H, Nq, Nkv, D, _lens(q_len),
                                   _lens(kv_len), float(sm_scale), int(bkv), 1 if causal else 0,
                                   _stream_ptr(stream))
        _check(rc, "sage_attn_fwd_bkv")
        return
    fn = lib.sage_attn_fwd_causal if causal else lib.sage_attn_fwd
    rc = fn(ctypes.byref(pb), ctypes.byref(os_), B, H, Nq, Nkv, D,
            _lens(q_len), _lens(kv_len), float(sm_scale), _stream_ptr(stream))
    _check(rc, "sage_attn_fwd_causal" if causal else "sage_attn_fwd")


def sage_attention(q, k, v, o, bufs: PrepBuffers, q_len=None, kv_len=None, sm_scale: float = 0.0,
                   causal: bool = False, stream=None):
    """Enqueue K/V preparation plus the attention kernel that quantizes its own
    Q blocks, on [B,H,N,D] BF16 views q, k, v and output view o."""
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    qs, ks, vs, os_, pb = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(o), bufs.c_struct()
    rc = load_library().sage_attention(ctypes.byref(qs), ctypes.byref(ks), ctypes.byref(vs), ctypes.byref(os_),
                                       B, H, Nq, Nkv, D, _lens(q_len), _lens(kv_len), float(sm_scale),
                                       1 if causal else 0, ctypes.byref(pb), _stream_ptr(stream))
    _check(rc, "sage_attention")


def sage_attn_checkpoints(bufs: PrepBuffers, o, b: int, h: int, qtile: int, q_len=None, kv_len=None,
                          sm_scale: float = 0.0, causal: bool = False, stream=None, Nkv: int | None = None):
    """Run one query tile as a single CTA and return its stage checkpoints
    (dict of device tensors: m, l, alpha, p8, pv16, ro, recip; see the header)."""
    B, H, Nq, D = o.shape
    Nkv = bufs.k16.shape[2] if Nkv is None else Nkv
    T = (Nkv + 127) // 128
    dev = o.device
    z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=dev)  # noqa: E731
    ck = dict(m=z((T, 128), torch.float32), l=z((T, 2, 128), torch.float32), alpha=z((T, 128), torch.float32),
              p8=z((T, 128, 128), torch.uint8), pv16=z((T, 128, D), torch.float16),
              ro=z((T, 128, D), torch.float32), recip=z((128,), torch.float32))
    cs = sage_checkpoints(*[ck[n].data_ptr() for n in ("m", "l", "alpha", "p8", "pv16", "ro", "recip")])
    os_, pb = tensor_desc(o), bufs.c_struct()
    rc = load_library().sage_attn_checkpoints(ctypes.byref(pb), ctypes.byref(os_), B, H, Nq, Nkv, D,
                                              _lens(q_len), _lens(kv_len), float(sm_scale), 1 if causal else 0,
                                              b, h, qtile, ctypes.byref(cs), _stream_ptr(stream))
    _check(rc, "sage_attn_checkpoints")
    return ck


def sage_qk_int32(bufs: PrepBuffers, s: torch.Tensor, q_len=None, kv_len=None, stream=None):
    """Enqueue the QK checkpoint kernel; s is int32 [B, H, Nq, Nkv] contiguous."""
    B, H, Nq, Nkv = s.shape
    assert s.dtype == torch.int32 and s.is_contiguous()
    pb = bufs.c_struct()
    rc = load_library().sage_qk_int32(ctypes.byref(pb), s.data_ptr(), B, H, Nq, Nkv, bufs.q16.shape[3],
                                      _lens(q_len), _lens(kv_len), _stream_ptr(stream))
    _check(rc, "sage_qk_int32")


def _host_lens(x, B):
    """A host int32 [B] array for the host-memory entries (None stays None)."""
    if x is None:
        return None
    vals = [int(v) for v in (x.tolist() if hasattr(x, "tolist") else x)]
    if len(vals) != B:
        raise ValueError(f"expected {B} lengths")
    return (ctypes.c_int32 * B)(*vals)


def sage_attention_host(host_phys, dev_phys, views_of, bufs: PrepBuffers, o_dev, o_host,
                        sm_scale: float = 0.0, stream=None, q_len=None, kv_len=None):
    """End-to-end call: copy host buffers in, prep + attention, copy O out.

    host_phys / dev_phys: matching lists of pinned-host / device tensors
    holding the physical inputs; views_of(dev_phys) -> (q, k, v) [B,H,N,D]
    views; o_dev / o_host: device output view and its pinned host twin
    (same physical layout, contiguous); q_len / kv_len: per-item lengths as
    host sequences (None: all valid).
    """
    q, k, v = views_of(dev_phys)
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    n = len(host_phys)
    copies = (sage_copy * n)(*[sage_copy(h.data_ptr(), d.data_ptr(), h.numel() * h.element_size())
                              for h, d in zip(host_phys, dev_phys)])
    out = sage_copy(o_host.data_ptr(), o_dev.data_ptr(), o_host.numel() * o_host.element_size())
    qs, ks, vs, os_, pb = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(o_dev), bufs.c_struct()
    rc = load_library().sage_attention_host(copies, n, ctypes.byref(qs), ctypes.byref(ks), ctypes.byref(vs),
                                            ctypes.byref(pb), ctypes.byref(os_), ctypes.byref(out),
                                            B, H, Nq, Nkv, D, _host_lens(q_len, B), _host_lens(kv_len, B),
                                            float(sm_scale), _stream_ptr(stream))
    _check(rc, "sage_attention_host")


def sage_attention_host_overlapped(q_host, k_host, v_host, o_host, q, k, v, o, bufs: PrepBuffers,
                                   sm_scale: float = 0.0, causal: bool = False, head_groups: int = 4,
                                   stream=None, q_len=None, kv_len=None):
    """End-to-end call with copies overlapped with compute: host views
    q_host.. (pinned, same strides as the device views q..), per head range
    copy in, prep, attention, copy out; q_len / kv_len: per-item lengths as
    host sequences (None: all valid; only valid rows are copied)."""
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    descs = [tensor_desc(t) for t in (q_host, k_host, v_host, o_host, q, k, v, o)]
    pb = bufs.c_struct()
    rc = load_library().sage_attention_host_overlapped(*[ctypes.byref(d) for d in descs], B, H, Nq, Nkv, D,
                                                       _host_lens(q_len, B), _host_lens(kv_len, B),
                                                       float(sm_scale), 1 if causal else 0, int(head_groups),
                                                       ctypes.byref(pb), _stream_ptr(stream))
    _check(rc, "sage_attention_host_overlapped")


def sage_get_device_status() -> int:
    return int(load_library().sage_get_device_status())


def sage_last_launch_count() -> int:
    return int(load_library().sage_last_launch_count())


def sage_debug_inject_fault(mode: int):
    _check(load_library().sage_debug_inject_fault(int(mode)), "sage_debug_inject_fault")


def sage_debug_epilogue_mode(tma_store: bool = False):
    """Test hook: write full output tiles through a TMA store (True) or row by
    row (False, the default) in later attention launches."""
    _check(load_library().sage_debug_epilogue_mode(1 if tma_store else 0), "sage_debug_epilogue_mode")


def sage_debug_prep_mode(one_pass: bool = False, lag: int = 0):
    """Test hook: select the one-launch preparation (one_pass=True, queue lag
    `lag` heads, 0 = from the grid) or the default three launches for later calls."""
    _check(load_library().sage_debug_prep_mode(1 if one_pass else 0, int(lag)), "sage_debug_prep_mode")


def attention(q, k, v, q_len=None, kv_len=None, sm_scale: float = 0.0, out=None, int8_codes=False,
              stream=None, causal: bool = False, fused: bool = True):
    """Attention on [B,H,N,D] BF16 CUDA views; returns (o, bufs).  fused=True
    uses sage_attention (Q quantized inside the attention kernel); False runs
    sage_prep_qkv then sage_attn_fwd (every code buffer filled)."""
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    bufs = alloc_prep_buffers(B, H, Nq, Nkv, q.device, int8_codes=int8_codes, D=D)
    if out is None:
        out = torch.zeros((B, Nq, H, D), dtype=torch.bfloat16, device=q.device).permute(0, 2, 1, 3)
    if fused:
        sage_attention(q, k, v, out, bufs, q_len, kv_len, sm_scale, causal, stream)
    else:
        sage_prep_qkv(q, k, v, bufs, q_len, kv_len, stream)
        sage_attn_fwd(bufs, out, q_len, kv_len, sm_scale, stream, Nkv=Nkv, causal=causal)
    return out, bufs
