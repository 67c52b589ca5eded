"""GPU path vs the oracle for head dimension 64 and for the causal form.

Neither is on the pages (they describe D = 128, non-causal); both run the same
contract (Experiment Log, "Phase 0 Import And Verification" stages).  Causal
reading: query i sees key j iff j <= i + (kv_len - q_len); rows that see no
key are zero.  Bars as in the main parity tests: bit-exact codes, scales and
integer QK scores; BF16 output within max(1e-2, one BF16 ulp) per element and
relative L2 <= 5e-3.
"""
import numpy as np
import pytest
import torch

from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

D64_CASES = {
    "d64_single_tile": dict(B=1, H=2, Nq=128, Nkv=192, seed=60, D=64),
    "d64_varlen_ragged": dict(B=2, H=3, Nq=700, Nkv=700, seed=61, D=64, k_offset_std=3.0,
                              q_len=[700, 333], kv_len=[700, 451]),
    "d64_hnd_1024": dict(B=1, H=4, Nq=1024, Nkv=1024, seed=62, D=64, layout="hnd", k_offset_std=2.0),
}

CAUSAL_CASES = {
    "causal_equal_640": dict(B=1, H=2, Nq=640, Nkv=640, seed=63, k_offset_std=2.0),
    "causal_short_q": dict(B=1, H=2, Nq=300, Nkv=520, seed=64),
    "causal_long_q": dict(B=1, H=2, Nq=520, Nkv=300, seed=65),           # rows 0..219 see no key
    "causal_varlen": dict(B=2, H=2, Nq=700, Nkv=700, seed=66, k_offset_std=2.0,
                          q_len=[700, 257], kv_len=[700, 400]),
    "causal_d64_equal": dict(B=1, H=3, Nq=600, Nkv=600, seed=67, D=64),
    "causal_d64_varlen": dict(B=2, H=2, Nq=450, Nkv=450, seed=68, D=64, q_len=[450, 129],
                              kv_len=[300, 450]),
}


def _case(spec):
    w = W.make_custom(**spec)
    q, k, v = G.logical_f32(w)
    return w, O.prepare(q, k, v, w.q_len, w.kv_len)


def _check_rows(w, gpu_bits, ref_bits):
    for b in range(w.B):
        lq = w.qlens[b]
        assert G.within_tolerance(gpu_bits[b, :, :lq], ref_bits[b, :, :lq]), G.out_metrics(
            gpu_bits[b, :, :lq], ref_bits[b, :, :lq])


@pytest.mark.parametrize("name", sorted(D64_CASES))
def test_d64_prep_and_qk_bit_exact(name):
    w, prep = _case(D64_CASES[name])
    run = G.GpuRun(w).prep()
    G.compare_prep(run, prep)
    s = run.qk().cpu().numpy()
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        for h in range(w.H):
            ref = O.qk_scores(prep.q8[b, h][:lq], prep.k8[b, h][:lk])
            assert np.array_equal(s[b, h, :lq, :lk], ref)


@pytest.mark.parametrize("name", sorted(D64_CASES))
def test_d64_attention_parity(name):
    w, prep = _case(D64_CASES[name])
    run = G.GpuRun(w).prep().attn(fill=7.0)
    got = run.out_bits()
    _check_rows(w, got, O.attention(prep))
    seven = O.f32_to_bf16_bits(np.float32([7.0]))[0]
    for b in range(w.B):
        assert np.all(got[b, :, w.qlens[b]:] == seven)               # rows >= q_len untouched


@pytest.mark.parametrize("name", sorted(CAUSAL_CASES))
def test_causal_attention_parity(name):
    w, prep = _case(CAUSAL_CASES[name])
    run = G.GpuRun(w).prep().attn(fill=7.0, causal=True)
    got = run.out_bits()
    ref = O.attention(prep, causal=True)
    _check_rows(w, got, ref)
    seven = O.f32_to_bf16_bits(np.float32([7.0]))[0]
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        hidden = np.arange(lq) + (lk - lq) < 0                        # rows that see no key
        assert np.all(got[b, :, :lq][:, hidden] == 0)
        assert np.all(got[b, :, lq:] == seven)


def test_causal_long_sequence_sampled_tiles():
    # 8K tokens: each query tile reads only the KV tiles up to its diagonal;
    # compare the first, a middle and the last query tile of two heads
    w = W.make_custom(B=1, H=4, Nq=8192, Nkv=8192, seed=69, layout="nhd_fused", k_offset_std=2.0)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v)
    run = G.GpuRun(w, int8_codes=False).prep().attn(causal=True)
    got = run.out_bits()
    rows = np.concatenate([np.arange(t * 128, t * 128 + 128) for t in (0, 31, 63)])
    for h in (0, 3):
        ref = O.attention_rows(prep, 0, h, rows, causal=True)[0]
        assert G.within_tolerance(got[0, h, rows], ref), G.out_metrics(got[0, h, rows], ref)
    del run
    torch.cuda.empty_cache()
