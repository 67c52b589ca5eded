"""CTA pairs (two adjacent 128-row query tiles sharing each tcgen05 MMA, 256
rows per instruction) against one CTA per query tile.

The pair form computes the same products in the same order (S is exact; the
FP16 PV accumulation runs the same K steps), so its output must be
bit-identical to the one-CTA form, and within the oracle tolerance.  Cases
cover an odd number of query tiles (the last pair's second CTA has no row),
varlen batches, causal masks and D = 64.
"""
import numpy as np
import pytest

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CASES = {
    "three_tiles": (dict(B=1, H=2, Nq=300, Nkv=400, seed=100, k_offset_std=2.0), False),
    "varlen": (dict(W.CONFIGS[3]), False),
    "causal_odd": (dict(B=1, H=2, Nq=520, Nkv=520, seed=101), True),
    "causal_varlen": (dict(B=2, H=2, Nq=700, Nkv=700, seed=102, q_len=[700, 257], kv_len=[700, 400]), True),
    "d64": (dict(B=1, H=3, Nq=640, Nkv=520, seed=103, D=64), False),
    "d64_causal_long_q": (dict(B=1, H=2, Nq=520, Nkv=300, seed=104, D=64), True),
}


def _run(w, causal, pairing):
    return G.GpuRun(w).prep().attn(fill=9.0, causal=causal, pairs=pairing).out_bits()


@pytest.mark.parametrize("name", sorted(CASES))
def test_pair_form_matches_single_cta_form(name):
    spec, causal = CASES[name]
    w = W.make_custom(**spec)
    paired = _run(w, causal, True)
    single = _run(w, causal, False)
    assert np.array_equal(paired, single)
    q, k, v = G.logical_f32(w)
    ref = O.attention(O.prepare(q, k, v, w.q_len, w.kv_len), causal=causal)
    nine = O.f32_to_bf16_bits(np.float32([9.0]))[0]
    for b in range(w.B):
        lq = w.qlens[b]
        assert G.within_tolerance(paired[b, :, :lq], ref[b, :, :lq])
        assert np.all(paired[b, :, lq:] == nine)


def test_pair_form_on_the_long_workload():
    w = W.make_config(4)
    assert np.array_equal(_run(w, False, True), _run(w, False, False))
