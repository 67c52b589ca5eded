"""C ABI checks that need no GPU: the library builds, loads, exports every
function the header declares, sizes buffers and rejects bad arguments on the
host before any CUDA call."""
import ctypes
import os
import re

import pytest

import quantized_exact_attention_gb300 as S
from quantized_exact_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return S.load_library()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sage_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("sage_prep_qkv", "sage_attn_fwd", "sage_qk_int32", "sage_attention_host",
                     "sage_get_device_status", "sage_buffer_sizes"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) <= set(S.EXPORTED)


def test_buffer_sizes(lib):
    s = S.buffer_sizes(2, 16, 1000, 777)
    assert s.nkv_pad == 784
    assert s.q16 == 2 * 16 * 1000 * 128 * 2
    assert s.k16 == 2 * 16 * 777 * 128 * 2
    assert s.v8t == 2 * 16 * 128 * 784
    assert s.q_scale == 2 * 16 * 8 * 4 and s.k_scale == 2 * 16 * 13 * 4
    # chunk sums and maxima, V inverse scales, 16 B of one-pass words per head,
    # the host entries' lengths slot (2 x B int32, rounded up to 16 B)
    assert s.workspace == 2 * (2 * 16 * 13 * 128 * 4) + 2 * 16 * 128 * 4 + 2 * 16 * 16 + 16
    s64 = S.buffer_sizes(2, 16, 1000, 777, D=64)
    assert s64.q16 == 2 * 16 * 1000 * 64 * 2 and s64.v8t == 2 * 16 * 64 * 784
    assert s64.workspace == 2 * (2 * 16 * 13 * 64 * 4) + 2 * 16 * 64 * 4 + 2 * 16 * 16 + 16


@pytest.mark.parametrize("shape,code", [((0, 1, 1, 1, 128), S.SAGE_ERR_ARG),
                                        ((1, 1, 1, 0, 128), S.SAGE_ERR_ARG),
                                        ((1, 1, 1, 1, 96), S.SAGE_ERR_UNSUPPORTED),
                                        ((1, 1, 1, 1, 256), S.SAGE_ERR_UNSUPPORTED)])
def test_buffer_sizes_rejects_bad_shapes(lib, shape, code):
    s = S.sage_sizes()
    assert lib.sage_buffer_sizes(*shape, ctypes.byref(s)) == code


def _fake_tensor(ptr=0x10000, sb=128 * 128, sh=128, sn=128 * 4):
    return S.sage_tensor(ptr, sb, sh, sn)


def _fake_bufs(**over):
    vals = dict(q16=0x20000, k16=0x30000, v8t=0x40000, q_scale=0x50000, k_scale=0x60000,
                v_scale=0x70000, k_mean=0x80000, q8=None, k8=None, workspace=0x90000,
                workspace_bytes=1 << 30)
    vals.update(over)
    return S.sage_prep_buffers(**vals)


def _prep(lib, q=None, k=None, v=None, bufs=None, shape=(1, 4, 256, 256, 128)):
    q, k, v = q or _fake_tensor(), k or _fake_tensor(), v or _fake_tensor()
    bufs = bufs or _fake_bufs()
    return lib.sage_prep_qkv(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), *shape, None, None,
                             ctypes.byref(bufs), None)


def test_prep_rejects_bad_arguments_before_touching_the_gpu(lib):
    assert _prep(lib, q=_fake_tensor(ptr=0)) == S.SAGE_ERR_ARG
    assert _prep(lib, k=_fake_tensor(ptr=0x10008)) == S.SAGE_ERR_UNSUPPORTED      # not 16-B aligned
    assert _prep(lib, v=_fake_tensor(sn=100)) == S.SAGE_ERR_UNSUPPORTED          # stride not 16-B multiple
    assert _prep(lib, bufs=_fake_bufs(q16=None)) == S.SAGE_ERR_ARG
    assert _prep(lib, bufs=_fake_bufs(workspace_bytes=16)) == S.SAGE_ERR_ARG
    assert _prep(lib, bufs=_fake_bufs(k_scale=0x60004)) == S.SAGE_ERR_UNSUPPORTED
    assert _prep(lib, shape=(1, 4, 256, 256, 96)) == S.SAGE_ERR_UNSUPPORTED
    assert _prep(lib, shape=(1, 0, 256, 256, 128)) == S.SAGE_ERR_ARG
    assert lib.sage_prep_qkv(None, None, None, 1, 1, 1, 1, 128, None, None, None, None) == S.SAGE_ERR_ARG


def test_attn_rejects_bad_arguments_before_touching_the_gpu(lib):
    o = _fake_tensor(ptr=0x10004)
    b = _fake_bufs()
    assert lib.sage_attn_fwd(ctypes.byref(b), ctypes.byref(o), 1, 1, 128, 128, 128, None, None,
                             0.0, None) == S.SAGE_ERR_UNSUPPORTED
    assert lib.sage_attn_fwd(ctypes.byref(b), None, 1, 1, 128, 128, 128, None, None, 0.0,
                             None) == S.SAGE_ERR_ARG
    assert lib.sage_qk_int32(ctypes.byref(b), None, 1, 1, 128, 128, 128, None, None, None) == S.SAGE_ERR_ARG
    assert lib.sage_attention_host(None, 0, None, None, None, None, None, None, 1, 1, 1, 1, 128, None, None,
                                   0.0, None) == S.SAGE_ERR_ARG


def test_fused_entry_and_causal_reject_bad_arguments_before_touching_the_gpu(lib):
    t, o = _fake_tensor(), _fake_tensor()
    b = _fake_bufs(q16=None)                                   # q16/q8 are not used by the fused entry

    def call(q=t, k=t, v=t, out=o, bufs=b, shape=(1, 4, 256, 256, 128), causal=0):
        return lib.sage_attention(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(out), *shape,
                                  None, None, 0.0, causal, ctypes.byref(bufs), None)

    assert call(q=_fake_tensor(ptr=0)) == S.SAGE_ERR_ARG
    assert call(out=_fake_tensor(ptr=0x10004)) == S.SAGE_ERR_UNSUPPORTED
    assert call(v=_fake_tensor(sh=12)) == S.SAGE_ERR_UNSUPPORTED
    assert call(bufs=_fake_bufs(k16=None)) == S.SAGE_ERR_ARG
    assert call(bufs=_fake_bufs(workspace_bytes=16)) == S.SAGE_ERR_ARG
    assert call(bufs=_fake_bufs(v8t=0x40008)) == S.SAGE_ERR_UNSUPPORTED
    assert call(shape=(1, 4, 256, 256, 96)) == S.SAGE_ERR_UNSUPPORTED
    assert call(shape=(1, 4, 0, 256, 128), causal=1) == S.SAGE_ERR_ARG
    assert lib.sage_attention(None, None, None, None, 1, 1, 1, 1, 128, None, None, 0.0, 0, None,
                              None) == S.SAGE_ERR_ARG
    o_bad = _fake_tensor(ptr=0x10004)
    assert lib.sage_attn_fwd_causal(ctypes.byref(_fake_bufs()), ctypes.byref(o_bad), 1, 1, 128, 128, 64, None,
                                    None, 0.0, None) == S.SAGE_ERR_UNSUPPORTED


def test_overlapped_host_entry_rejects_bad_arguments_before_touching_the_gpu(lib):
    t = _fake_tensor()
    b = _fake_bufs()

    def call(hq=t, dq=t, groups=4, shape=(1, 8, 256, 256, 128)):
        tens = [hq, t, t, t, dq, t, t, t]
        return lib.sage_attention_host_overlapped(*[ctypes.byref(x) for x in tens], *shape, None, None, 0.0, 0,
                                                  groups, ctypes.byref(b), None)

    assert call(groups=0) == S.SAGE_ERR_ARG
    assert call(groups=9) == S.SAGE_ERR_ARG                     # more ranges than heads
    assert call(hq=_fake_tensor(ptr=0)) == S.SAGE_ERR_ARG
    assert call(hq=_fake_tensor(sn=128 * 8)) == S.SAGE_ERR_ARG  # host strides differ from the device view's
    assert call(dq=_fake_tensor(ptr=0x10004)) == S.SAGE_ERR_UNSUPPORTED
    assert call(shape=(1, 8, 256, 256, 96)) == S.SAGE_ERR_UNSUPPORTED


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert S.status_string(code) not in ("", "unknown status")
    assert S.status_string(-99) == "unknown status"
