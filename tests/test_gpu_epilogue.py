"""The two output epilogues of the attention kernel write the same bytes.

Default: every correction thread writes its row's channels with 16-byte
stores.  Selected by the epilogue test hook (for the default and causal
forms): a tile whose 128 rows are all valid is staged in shared memory
(128-byte swizzle) and written by one TMA store; partial tiles of shorter
batch items are still written row by row.  Each is run both ways on a
pre-filled output and compared bit for bit; rows at or past q_len must keep
the fill value.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

SHAPES = {
    "koffset_nhd": dict(W.CONFIGS[2]),
    "ragged_varlen": dict(W.CONFIGS[3]),
    "hnd_partial_last_tile": dict(B=2, H=3, Nq=300, Nkv=520, seed=150, layout="hnd", k_offset_std=2.0),
    "d64_varlen": dict(B=2, H=4, Nq=384, Nkv=300, D=64, seed=151, q_len=[384, 200], kv_len=[300, 129]),
    "fused_qkv_layout": dict(B=1, H=4, Nq=512, Nkv=512, seed=152, layout="nhd_fused"),
}
FORMS = {"default": {}, "causal": dict(causal=True)}        # the forms the TMA epilogue serves


def _run(w, form, tma):
    run = G.GpuRun(w)
    run.prep(bkv=form.get("bkv", 128))
    base = torch.full((w.B, w.Nq, w.H, w.D), 9.0, dtype=torch.bfloat16, device="cuda")
    out = base.permute(0, 2, 1, 3)
    S.sage_debug_epilogue_mode(tma)
    try:
        if form.get("fused"):
            S.sage_attention(run.q, run.k, run.v, out, run.bufs, run.q_len, run.kv_len)
        else:
            S.sage_attn_fwd(run.bufs, out, run.q_len, run.kv_len, Nkv=w.Nkv, causal=form.get("causal", False),
                            bkv=form.get("bkv", 128), pairs=form.get("pairs", False))
        torch.cuda.synchronize()
    finally:
        S.sage_debug_epilogue_mode(False)
    assert S.sage_get_device_status() == S.SAGE_OK
    return out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("form", sorted(FORMS))
@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_tma_store_epilogue_writes_the_same_bytes(shape, form):
    w = W.make_custom(**SHAPES[shape])
    rows = _run(w, FORMS[form], False)
    tma = _run(w, FORMS[form], True)
    assert np.array_equal(rows, tma)
    nine = O.f32_to_bf16_bits(np.float32([9.0]))[0]
    for b in range(w.B):
        assert np.all(tma[b, :, w.qlens[b]:] == nine)
