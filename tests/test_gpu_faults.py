"""Failure detection without a GPU fault.

The test hook makes the next attention launch withhold its V tile copies, so
the MMA issuer's bounded mbarrier wait runs out (about one second).  The
kernel must record SAGE_ERR_TIMEOUT in the device status words, let every
role leave its loop, drain its copies and MMAs, free tensor memory and
return; the CUDA context must stay usable, so the next launch is correct.
No trap, no bad address, no endless loop is involved.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu


def test_withheld_copy_times_out_and_context_survives():
    w = W.make_custom(1, 1, 128, 256, seed=40)                 # one CTA, two KV tiles
    run = G.GpuRun(w).prep()
    assert S.sage_get_device_status() == S.SAGE_OK
    out = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    S.sage_debug_inject_fault(1)
    S.sage_attn_fwd(run.bufs, out)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_ERR_TIMEOUT
    assert S.sage_get_device_status() == S.SAGE_OK            # read-and-clear
    # the context is intact: a normal launch still matches the oracle
    run.attn()
    q, k, v = G.logical_f32(w)
    ref = O.attention(O.prepare(q, k, v))
    assert G.within_tolerance(run.out_bits(), ref)
