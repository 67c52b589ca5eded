"""The one-call entry point (sage_attention): Q preparation fused into the
attention kernel.  Each CTA quantizes its own 128-row Q block (one INT8 scale
block) with the preparation arithmetic, so the output must be bit-identical to
sage_prep_qkv followed by sage_attn_fwd, its Q scales bit-identical to the
oracle's, and the K/V buffers identical to the two-call path.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

CASES = {
    "cfg1_single_tile": dict(W.CONFIGS[1]),
    "cfg2_koffset": dict(W.CONFIGS[2]),
    "cfg3_varlen": dict(W.CONFIGS[3]),
    "hnd_ragged_q": dict(B=2, H=3, Nq=333, Nkv=520, seed=70, layout="hnd", q_len=[333, 200], kv_len=[520, 129]),
    "d64_varlen": dict(B=2, H=2, Nq=400, Nkv=400, seed=71, D=64, q_len=[400, 130], kv_len=[256, 400]),
}


def _both(w, causal):
    two = G.GpuRun(w).prep().attn(fill=3.0, causal=causal)
    one = G.GpuRun(w)
    base = torch.full((w.B, w.Nq, w.H, w.D), 3.0, dtype=torch.bfloat16, device="cuda")
    out = base.permute(0, 2, 1, 3)
    S.sage_attention(one.q, one.k, one.v, out, one.bufs, one.q_len, one.kv_len, causal=causal)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    one.out = out
    return two, one


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_entry_matches_two_calls_bit_for_bit(name, causal):
    w = W.make_custom(**CASES[name])
    two, one = _both(w, causal)
    assert np.array_equal(one.out_bits(), two.out_bits())
    for buf in ("k16", "v8t", "k_scale", "v_scale", "k_mean"):
        assert torch.equal(getattr(one.bufs, buf), getattr(two.bufs, buf)), buf
    # Q scales written by the attention kernel == the oracle's, for every query
    # tile with a valid row and a visible key
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len)
    qs = one.bufs.q_scale.cpu().numpy()
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        for t in range((lq + 127) // 128):
            last = min(t * 128 + 127, lq - 1)
            sees = lk > 0 and (not causal or last + lk - lq >= 0)
            if sees:
                assert qs[b, :, t].view(np.uint32).tolist() == prep.q_scale[b, :, t].view(np.uint32).tolist()


def test_fused_entry_full_size_bench_workload():
    w = W.make_config(4)
    two, one = _both(w, False)
    assert np.array_equal(one.out_bits(), two.out_bits())
    assert torch.equal(one.bufs.q_scale, two.bufs.q_scale)
    del one, two
    torch.cuda.empty_cache()
