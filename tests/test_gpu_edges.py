"""GPU edge cases: ragged and tiny shapes, empty lengths, layouts, canaries.

Every case compares the full output and every preparation buffer with the
oracle; rows past a query length must keep the canary value the output
buffer was filled with.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CANARY = 3.0     # bf16 0x4040


def _check(w):
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len)
    run = G.GpuRun(w).prep().attn(fill=CANARY)
    G.compare_prep(run, prep)
    ref = O.attention(prep)
    got = run.out_bits()
    canary = np.uint16(0x4040)
    for b in range(w.B):
        lq = w.qlens[b]
        ex, rel, ma = G.out_metrics(got[b, :, :lq], ref[b, :, :lq])
        assert ex <= 0 and rel <= G.OUT_REL_L2, (w.name, b, ma, rel)
        if w.kvlens[b] == 0:
            assert np.all(got[b, :, :lq] == 0)
        assert np.all(got[b, :, lq:] == canary), "rows beyond q_len were written"
    s = run.qk()
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        for h in range(w.H):
            ref_s = O.qk_scores(prep.q8[b, h][:lq], prep.k8[b, h][:lk])
            assert np.array_equal(s[b, h, :lq, :lk].cpu().numpy().astype(np.int64), ref_s)


SHAPES = [(1, 1, 1, 1), (1, 1, 63, 65), (1, 2, 64, 64), (1, 1, 65, 127), (1, 1, 127, 129),
          (1, 1, 129, 191), (1, 2, 191, 777), (1, 1, 777, 63), (1, 1, 300, 1), (1, 3, 256, 384)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes(shape):
    B, H, Nq, Nkv = shape
    _check(W.make_custom(B, H, Nq, Nkv, seed=100 + Nq + Nkv, k_offset_std=2.0))


@pytest.mark.parametrize("layout", ["nhd", "hnd", "nhd_fused"])
def test_layouts(layout):
    _check(W.make_custom(2, 3, 200, 200, seed=7, layout=layout, k_offset_std=1.0))


def test_varlen_with_empty_items():
    w = W.make_custom(4, 2, 300, 260, seed=9, q_len=[300, 0, 131, 17], kv_len=[260, 100, 0, 129],
                      k_offset_std=2.0)
    _check(w)


def test_outlier_block_scales():
    _check(W.make_custom(2, 2, 384, 384, seed=10, outlier_frac=0.01, layout="hnd"))


def test_sm_scale_argument():
    w = W.make_custom(1, 2, 200, 300, seed=11)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v)
    run = G.GpuRun(w).prep()
    out = torch.zeros((1, 200, 2, 128), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    S.sage_attn_fwd(run.bufs, out, sm_scale=0.05)
    torch.cuda.synchronize()
    got = out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ref = O.attention(prep, sm_scale=0.05)
    assert G.within_tolerance(got, ref)
