"""The end-to-end entries from host memory.  sage_attention_host_overlapped:
per head range, host->device copies, preparation, attention and
device->host copies on internal streams; heads are independent problems, so
its output must equal the device path bit for bit.  Both host entries take
per-item lengths as host arrays; with ragged lengths only valid rows are
computed (and, for the overlapped entry, copied), and the output is compared
with the oracle."""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CASES = {
    "cfg2_nhd_4groups": (dict(W.CONFIGS[2]), 4, False),
    "hnd_odd_groups": (dict(B=2, H=5, Nq=300, Nkv=260, seed=110, layout="hnd", k_offset_std=2.0), 3, False),
    "fused_layout_causal": (dict(B=1, H=6, Nq=640, Nkv=640, seed=111, layout="nhd_fused"), 6, True),
    "d64_one_group": (dict(B=1, H=4, Nq=384, Nkv=384, seed=112, D=64), 1, False),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_overlapped_host_entry_matches_device_path(name):
    spec, groups, causal = CASES[name]
    w = W.make_custom(**spec)
    ref = G.GpuRun(w).prep().attn(causal=causal).out_bits()
    host_phys = [t.contiguous().pin_memory() for t in w.phys]
    dev_phys = [torch.zeros_like(t, device="cuda") for t in w.phys]
    o_host = torch.full((w.B, w.Nq, w.H, w.D), 3.0, dtype=torch.bfloat16).pin_memory()
    o_dev = torch.zeros((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    qh, kh, vh = w.views(host_phys)
    qd, kd, vd = w.views(dev_phys)
    bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", D=w.D)
    S.sage_attention_host_overlapped(qh, kh, vh, o_host.permute(0, 2, 1, 3), qd, kd, vd, o_dev.permute(0, 2, 1, 3),
                                     bufs, causal=causal, head_groups=groups)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    got = o_host.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


VARLEN = {
    "ragged_workload": dict(W.CONFIGS[3]),
    "hnd_empty_item": dict(B=3, H=4, Nq=300, Nkv=420, seed=113, layout="hnd", k_offset_std=2.0,
                           q_len=[300, 0, 129], kv_len=[420, 77, 0]),
}


def _oracle_bits(w):
    q, k, v = G.logical_f32(w)
    return O.attention(O.prepare(q, k, v, w.q_len, w.kv_len))


@pytest.mark.parametrize("name", sorted(VARLEN))
def test_overlapped_host_entry_with_lengths(name):
    w = W.make_custom(**VARLEN[name])
    ref = G.GpuRun(w).prep().attn().out_bits()
    host_phys = [t.contiguous().pin_memory() for t in w.phys]
    dev_phys = [torch.zeros_like(t, device="cuda") for t in w.phys]
    o_host = torch.full((w.B, w.Nq, w.H, w.D), 3.0, dtype=torch.bfloat16).pin_memory()
    o_dev = torch.zeros((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    qh, kh, vh = w.views(host_phys)
    qd, kd, vd = w.views(dev_phys)
    bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", D=w.D)
    S.sage_attention_host_overlapped(qh, kh, vh, o_host.permute(0, 2, 1, 3), qd, kd, vd, o_dev.permute(0, 2, 1, 3),
                                     bufs, head_groups=3, q_len=w.q_len, kv_len=w.kv_len)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    got = o_host.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy().view(np.uint16)
    orc = _oracle_bits(w)
    three = O.f32_to_bf16_bits(np.float32([3.0]))[0]
    for b in range(w.B):
        lq = w.qlens[b]
        assert np.array_equal(got[b, :, :lq], ref[b, :, :lq])       # the device path, bit for bit
        assert G.within_tolerance(got[b, :, :lq], orc[b, :, :lq])   # and the oracle
        assert np.all(got[b, :, lq:] == three)                      # rows past q_len never copied back


def test_sequential_host_entry_with_lengths():
    w = W.make_custom(**VARLEN["ragged_workload"])
    ref = G.GpuRun(w).prep().attn().out_bits()
    host_phys = [t.contiguous().pin_memory() for t in w.phys]
    dev_phys = [torch.zeros_like(t, device="cuda") for t in w.phys]
    o_dev = torch.zeros((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    o_host = torch.empty_like(o_dev, device="cpu").pin_memory()
    bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", D=w.D)
    S.sage_attention_host(host_phys, dev_phys, w.views, bufs, o_dev.permute(0, 2, 1, 3), o_host,
                          q_len=w.q_len, kv_len=w.kv_len)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    got = o_host.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy().view(np.uint16)
    orc = _oracle_bits(w)
    for b in range(w.B):
        lq = w.qlens[b]
        assert np.array_equal(got[b, :, :lq], ref[b, :, :lq])
        assert G.within_tolerance(got[b, :, :lq], orc[b, :, :lq])
        assert np.all(got[b, :, lq:] == 0)                          # device rows past q_len stay as zeroed
