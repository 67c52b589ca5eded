"""The end-to-end entry with copies overlapped with compute
(sage_attention_host_overlapped): per head range, host->device copies,
preparation, attention and device->host copies on internal streams.  Heads are
independent problems, so its output must equal the device path bit for bit."""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
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
