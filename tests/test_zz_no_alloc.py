"""The no-allocation preparation entry point against the regular one.

sage_prep_qkv_noalloc exists for callers that cannot call cudaMalloc (an
engine plugin handed only input and output pointers, code running while the
device memory pool is fully committed): it keeps its scratch in a fixed
device array inside the library instead of a caller-provided workspace.  Its
outputs must equal those of sage_prep_qkv bit for bit (the tolerance every
preparation test here uses), on consecutive calls that reuse the array with
different shapes.  This file is named so pytest collects it last.
"""
import ctypes
import dataclasses

import pytest
import torch

import quantized_exact_attention_gb300 as S
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

FIELDS = ("q16", "k16", "v8t", "q_scale", "k_scale", "v_scale", "k_mean", "q8", "k8")


def _prep_both(w):
    run = G.GpuRun(w, int8_codes=True)                        # regular entry point, own workspace
    run.prep()
    ref = {f: getattr(run.bufs, f).clone() for f in FIELDS}
    nb = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", int8_codes=True, D=w.D)
    for f in FIELDS:                                          # poison the outputs first
        getattr(nb, f).fill_(0x5A if getattr(nb, f).dtype in (torch.uint8, torch.int8) else 7)
    S.sage_prep_qkv_noalloc(run.q, run.k, run.v, nb, run.q_len, run.kv_len)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    return ref, nb


def _assert_equal(ref, nb):
    for f in FIELDS:
        got = getattr(nb, f)
        assert torch.equal(got.view(torch.uint8) if got.dtype != torch.uint8 else got,
                           ref[f].view(torch.uint8) if ref[f].dtype != torch.uint8 else ref[f]), f


@pytest.mark.gpu
def test_noalloc_prep_matches_regular_prep_on_two_calls_in_a_row():
    G.ensure_built()
    first = W.make_config(3)                                  # varlen, 2 x 16 heads of 1000 tokens
    second = W.make_custom(B=1, H=24, Nq=2048, Nkv=3000, seed=31, layout="hnd",
                           k_offset_std=2.0)
    third = W.make_custom(B=2, H=6, Nq=500, Nkv=1300, D=64, seed=34, layout="hnd",   # D = 64, varlen
                          k_offset_std=2.0, q_len=[500, 77], kv_len=[1300, 640])
    for w in (first, second, third):
        ref, nb = _prep_both(w)
        _assert_equal(ref, nb)


@pytest.mark.gpu
def test_noalloc_prep_ignores_the_callers_workspace():
    # a NULL workspace of 0 bytes is accepted, and a poisoned workspace passed
    # in is left untouched: the scratch is the library's own array
    G.ensure_built()
    w = W.make_custom(B=2, H=8, Nq=700, Nkv=900, D=64, seed=33, layout="hnd", k_offset_std=2.0,
                      q_len=[700, 333], kv_len=[900, 401])
    run = G.GpuRun(w, int8_codes=True)
    run.prep()
    ref = {f: getattr(run.bufs, f).clone() for f in FIELDS}
    for workspace in (torch.empty(0, dtype=torch.uint8, device="cuda"),
                      torch.full_like(run.bufs.workspace, 0xA5)):
        nb = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", int8_codes=True, D=64)
        nb = dataclasses.replace(nb, workspace=workspace)
        S.sage_prep_qkv_noalloc(run.q, run.k, run.v, nb, run.q_len, run.kv_len)
        torch.cuda.synchronize()
        assert S.sage_get_device_status() == S.SAGE_OK
        assert S.sage_last_launch_count() == 3          # the three preparation kernels
        _assert_equal(ref, nb)
        assert workspace.numel() == 0 or bool((workspace == 0xA5).all())


@pytest.mark.gpu
def test_noalloc_prep_feeds_the_attention_kernel():
    G.ensure_built()
    w = W.make_custom(B=2, H=3, Nq=300, Nkv=333, seed=32, q_len=[300, 129], kv_len=[333, 65])
    run = G.GpuRun(w, int8_codes=False).prep().attn()
    expect = run.out_bits().copy()
    fresh = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda")
    S.sage_prep_qkv_noalloc(run.q, run.k, run.v, fresh, run.q_len, run.kv_len)
    run.bufs = fresh
    run.attn()
    assert (run.out_bits() == expect).all()


def test_noalloc_rejects_problems_beyond_its_scratch():
    G.ensure_built()
    lib = S.load_library()
    cap = S.sage_prep_noalloc_capacity()
    assert cap == 16 << 20
    # 1024 heads of 16K tokens need 1024*256 chunk rows x 1 KiB = 256 MiB of scratch
    sz = S.buffer_sizes(1, 1024, 128, 16384)
    assert sz.workspace > cap
    t = S.sage_tensor(0x10000, 0, 128, 128 * 1024)
    b = S.sage_prep_buffers(0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000, 0x80000, None, None,
                            None, 0)
    rc = lib.sage_prep_qkv_noalloc(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), 1, 1024, 128, 16384,
                                   128, None, None, ctypes.byref(b), None)
    assert rc == S.SAGE_ERR_SCRATCH
    assert "scratch" in S.status_string(rc)
