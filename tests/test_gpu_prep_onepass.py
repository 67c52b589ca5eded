"""The one-launch preparation against the default three-launch form.

The one-launch form (selected with the preparation test hook) is a single
kernel whose CTAs take work items from a queue: a head's channel statistics, its Q blocks, and the K/V quantization of
a head some places earlier in the queue (so that its K and V are re-read from
L2), with the K mean reduced in the pinned order by the last statistics item
of each head.  The three plain launches (statistics and Q, finalize, K/V)
compute the same bytes; the two are compared bit for bit on every output
buffer, with the queue lag at its default, at 1 (K/V items right behind their
statistics, so they wait) and larger than the head count (all statistics
first), on poisoned workspaces and on two calls in a row.
"""
import dataclasses

import pytest
import torch

import quantized_exact_attention_gb300 as S
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

FIELDS = ("q16", "k16", "v8t", "q_scale", "k_scale", "v_scale", "k_mean", "q8", "k8")

EXTRA = {
    "d64_varlen_hnd": dict(B=3, H=5, Nq=700, Nkv=900, D=64, seed=141, layout="hnd", k_offset_std=2.0,
                           q_len=[700, 1, 333], kv_len=[900, 0, 65]),
    "one_token": dict(B=1, H=3, Nq=1, Nkv=1, seed=142),
    "long_kv_few_heads": dict(B=1, H=2, Nq=300, Nkv=9000, seed=143, k_offset_std=3.0),
}


def _workload(name):
    return W.make_config(name) if isinstance(name, int) else W.make_custom(**EXTRA[name])


def _prep(run, one_pass, lag=0, poison=None):
    nb = S.alloc_prep_buffers(run.w.B, run.w.H, run.w.Nq, run.w.Nkv, "cuda", int8_codes=True, D=run.w.D)
    for f in FIELDS:
        getattr(nb, f).view(torch.uint8).fill_(0x5A)
    if poison is not None:
        nb.workspace.fill_(poison)
    S.sage_debug_prep_mode(one_pass, lag)
    try:
        S.sage_prep_qkv(run.q, run.k, run.v, nb, run.q_len, run.kv_len)
        torch.cuda.synchronize()
    finally:
        S.sage_debug_prep_mode(False, 0)
    assert S.sage_get_device_status() == S.SAGE_OK
    return nb


def _same(a, b):
    for f in FIELDS:
        x, y = getattr(a, f), getattr(b, f)
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), f


@pytest.mark.parametrize("name", [1, 2, 3, 4, 5, *sorted(EXTRA)])
def test_one_launch_matches_three_launches(name):
    run = G.GpuRun(_workload(name))
    ref = _prep(run, one_pass=False)
    for lag, poison in ((0, None), (1, 0xFF), (1000, 0x00)):
        got = _prep(run, one_pass=True, lag=lag, poison=poison)
        _same(ref, got)
        assert S.sage_last_launch_count() == 1


def test_two_calls_in_a_row_share_a_workspace():
    # the second call on the same workspace sees the first call's words
    w = _workload(3)
    run = G.GpuRun(w)
    ref = _prep(run, one_pass=False)
    nb = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", int8_codes=True)
    S.sage_debug_prep_mode(True, 0)
    try:
        for _ in range(3):
            S.sage_prep_qkv(run.q, run.k, run.v, nb, run.q_len, run.kv_len)
        torch.cuda.synchronize()
    finally:
        S.sage_debug_prep_mode(False, 0)
    assert S.sage_get_device_status() == S.SAGE_OK
    _same(ref, nb)
    # a different shape on the same workspace bytes
    w2 = W.make_custom(B=1, H=4, Nq=500, Nkv=1500, seed=144)
    run2 = G.GpuRun(w2)
    ref2 = _prep(run2, one_pass=False)
    nb2 = S.alloc_prep_buffers(w2.B, w2.H, w2.Nq, w2.Nkv, "cuda", int8_codes=True)
    nb2 = dataclasses.replace(nb2, workspace=nb.workspace[:nb2.workspace.numel()])
    S.sage_debug_prep_mode(True, 0)
    try:
        S.sage_prep_qkv(run2.q, run2.k, run2.v, nb2, run2.q_len, run2.kv_len)
        torch.cuda.synchronize()
    finally:
        S.sage_debug_prep_mode(False, 0)
    _same(ref2, nb2)
