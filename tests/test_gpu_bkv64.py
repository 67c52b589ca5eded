"""The BKV = 64 contract variant on the GPU against the oracle (reading R16:
64-key online-softmax tiles and inner FP16 PV sums, S_V = 2.25; the 64-key
epochs of Experiment Log, "Phase 2A").  Bars as for the main contract:
bit-exact V codes and scales (the only preparation outputs that change),
BF16 output within max(1e-2, one BF16 ulp) per element and rel-L2 <= 5e-3.
"""
import numpy as np
import pytest

from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CASES = {
    "cfg1": (dict(W.CONFIGS[1]), False),
    "cfg2": (dict(W.CONFIGS[2]), False),
    "cfg3_varlen": (dict(W.CONFIGS[3]), False),
    "ragged_odd_tail": (dict(B=1, H=3, Nq=300, Nkv=333, seed=90, k_offset_std=2.0), False),   # last tile 77 keys
    "tail_in_first_epoch": (dict(B=1, H=2, Nq=256, Nkv=300, seed=91), False),               # last tile 44 keys
    "causal": (dict(B=2, H=2, Nq=520, Nkv=520, seed=92, q_len=[520, 200], kv_len=[520, 333]), True),
    "d64": (dict(B=1, H=3, Nq=400, Nkv=450, seed=93, D=64), False),
    "d64_causal": (dict(B=1, H=2, Nq=384, Nkv=384, seed=94, D=64), True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bkv64_parity(name):
    spec, causal = CASES[name]
    w = W.make_custom(**spec)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len, bkv=64)
    run = G.GpuRun(w).prep(bkv=64)
    G.compare_prep(run, prep)
    run.attn(fill=5.0, causal=causal, bkv=64)
    got = run.out_bits()
    ref = O.attention(prep, causal=causal)
    five = O.f32_to_bf16_bits(np.float32([5.0]))[0]
    for b in range(w.B):
        lq = w.qlens[b]
        assert G.within_tolerance(got[b, :, :lq], ref[b, :, :lq]), G.out_metrics(got[b, :, :lq], ref[b, :, :lq])
        assert np.all(got[b, :, lq:] == five)
    # the BKV = 128 oracle is a different contract: its output differs
    if name == "cfg2":
        ref128 = O.attention(O.prepare(q, k, v, w.q_len, w.kv_len))
        assert not np.array_equal(ref, ref128)
