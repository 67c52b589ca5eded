"""GPU edge cases for every form of the path besides the default one: causal,
the one-call entry (Q quantized in the attention kernel), BKV = 64, D = 64 and
CTA pairs, on tiny and ragged shapes and on varlen batches with empty items.

Each case compares the output with the oracle of the same form; rows past a
query length must keep the canary the output was filled with, and rows that
see no key (kv_len = 0, or hidden by the causal mask) must be zero.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CANARY = np.uint16(0x4040)   # bf16 3.0

FORMS = {
    "causal": dict(causal=True),
    "fused": dict(fused=True),
    "fused_causal": dict(fused=True, causal=True),
    "bkv64": dict(bkv=64),
    "d64": dict(D=64),
    "d64_causal": dict(D=64, causal=True),
    "pairs": dict(pairs=True),
    "pairs_causal": dict(pairs=True, causal=True),
}

SHAPES = {
    "1x1": dict(B=1, H=1, Nq=1, Nkv=1),
    "63x65": dict(B=1, H=1, Nq=63, Nkv=65),
    "129x191": dict(B=1, H=2, Nq=129, Nkv=191),
    "300x1": dict(B=1, H=1, Nq=300, Nkv=1),
    "1x300": dict(B=1, H=1, Nq=1, Nkv=300),
    "varlen_empty": dict(B=3, H=2, Nq=200, Nkv=260, q_len=[0, 130, 200], kv_len=[100, 0, 257]),
}


def _run_form(w, form):
    causal = form.get("causal", False)
    bkv = form.get("bkv", 128)
    run = G.GpuRun(w)
    base = torch.full((w.B, w.Nq, w.H, w.D), 3.0, dtype=torch.bfloat16, device="cuda")
    out = base.permute(0, 2, 1, 3)
    if form.get("fused"):
        S.sage_attention(run.q, run.k, run.v, out, run.bufs, run.q_len, run.kv_len, causal=causal)
    else:
        run.prep(bkv=bkv)
        S.sage_attn_fwd(run.bufs, out, run.q_len, run.kv_len, Nkv=w.Nkv, causal=causal, bkv=bkv,
                        pairs=form.get("pairs", False))
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    return out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("form", sorted(FORMS))
def test_form_edge_case(form, shape):
    f = FORMS[form]
    spec = dict(SHAPES[shape], seed=120 + len(shape), k_offset_std=1.0, D=f.get("D", 128))
    w = W.make_custom(**spec)
    got = _run_form(w, f)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len, bkv=f.get("bkv", 128))
    causal = f.get("causal", False)
    ref = O.attention(prep, causal=causal)
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        assert G.within_tolerance(got[b, :, :lq], ref[b, :, :lq]), G.out_metrics(got[b, :, :lq], ref[b, :, :lq])
        # rows that see no key: all of them when kv_len = 0; with the causal
        # mask also rows i with i + (kv_len - q_len) < 0
        hidden = np.full(lq, lk == 0)
        if causal:
            hidden |= np.arange(lq) + (lk - lq) < 0
        assert np.all(got[b, :, :lq][:, hidden] == 0)
        assert np.all(got[b, :, lq:] == CANARY), "rows beyond q_len were written"
