"""Large and extreme shapes against the oracle: one head of 128K tokens with
ragged tails at the very end, 4096 short heads in one launch (the grid's head
and batch dimensions), and head dimension 64 at 64K tokens.

Preparation outputs are compared bit for bit everywhere; the attention output
on sampled query rows (the first, a middle and the last query tiles, which
cover the ragged tail) and on sampled heads, within the output tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CASES = {
    # 1024 query tiles x 1024 key tiles in one head; the last query tile and
    # the last key tile are both partial
    "one_head_128k_ragged": dict(B=1, H=1, Nq=131072, Nkv=131072, seed=160, layout="hnd", k_offset_std=2.0,
                                 q_len=[131071], kv_len=[130001]),
    # 4096 (b, h) heads of 64 tokens: grid y = 64 heads, z = 64 batch items
    "heads_4096_short": dict(B=64, H=64, Nq=64, Nkv=64, seed=161, layout="nhd", k_offset_std=1.0),
    "d64_two_heads_64k": dict(B=1, H=2, Nq=65536, Nkv=65536, D=64, seed=162, layout="hnd"),
}


def _rows(lq):
    tiles = sorted({0, (lq // 128) // 2, (lq - 1) // 128})
    rows = np.concatenate([np.arange(t * 128, min(t * 128 + 128, lq)) for t in tiles])
    return rows


@pytest.mark.parametrize("name", sorted(CASES))
def test_large_shape_matches_oracle(name):
    w = W.make_custom(**CASES[name])
    run = G.GpuRun(w).prep().attn(fill=5.0)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len)
    G.compare_prep(run, prep)
    out = run.out_bits()
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    if len(heads) > 16:
        rng = np.random.default_rng(0)
        heads = [heads[i] for i in sorted(rng.choice(len(heads), 16, replace=False))]
    five = O.f32_to_bf16_bits(np.float32([5.0]))[0]
    for b, h in heads:
        lq = w.qlens[b]
        rows = _rows(lq)
        ref, _ = O.attention_rows(prep, b, h, rows)
        assert G.within_tolerance(out[b, h][rows], ref), (b, h)
        assert np.all(out[b, h, lq:] == five)            # rows past q_len never written
    del run
    torch.cuda.empty_cache()
