"""Exactness of the production kernel's integer scores, seen through its output.

The QK checkpoint (sage_qk_int32) reads scores from a separate capture form of
the attention kernel; this test checks the default form's scores through an
output that a score error of one unit would change by O(1).

Construction (codes known exactly, no rounding anywhere before QK):
- Q and K values are integers times 2^-7 with a +-127 in every scale block,
  so every block scale is 2^-7 and every INT8 code is the integer itself;
- keys come in quads (k, k', -k, -k'), which makes every channel sum of K
  exactly zero in the pinned chunk order, so smoothing changes nothing;
- k' equals k except one code larger in the last channel, where every query
  has code 1; so in every quad the best key's runner-up scores exactly 1 less;
- sm_scale is chosen so that f = q_scale * k_scale * c = 4 in the log2
  domain: the runner-up gets weight 2^-4 against the best key, and a score
  off by one at the top would move that weight to 2^-8 or to 1.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

U = 2.0 ** -7
SM_SCALE = 2.0 ** 16 / 1.4426950408889634       # c = 2^16 (to FP32 rounding), so f = 2^-14 * c ~ 4


def _codes(seed=170, B=1, H=2, Nq=256, Nkv=512, D=128):
    rng = np.random.default_rng(seed)
    qc = rng.integers(-60, 61, (B, H, Nq, D))
    qc[..., D - 1] = 1                                  # the tie-breaking channel
    qc[..., ::128, 0] = 127                             # every 128-row Q block holds a 127
    base = rng.integers(-120, 121, (B, H, Nkv // 4, D))
    base[..., ::16, 0] = 127                            # every 64-key block holds a 127
    twin = base.copy()
    twin[..., D - 1] += 1
    kc = np.stack([base, twin, -base, -twin], axis=3).reshape(B, H, Nkv, D)
    v = rng.standard_normal((B, H, Nkv, D)).astype(np.float32)
    return qc, kc, v


def _workload():
    qc, kc, v = _codes()
    B, H, Nq, D = qc.shape
    Nkv = kc.shape[2]
    t = [torch.from_numpy((x * U).astype(np.float32)).to(torch.bfloat16) for x in (qc, kc)]
    t.append(torch.from_numpy(v).to(torch.bfloat16))
    return W.Workload("sharp_quads_B1_H2_Nq256_Nkv512", B, H, Nq, Nkv, D, "hnd", tuple(t), None, None), qc, kc


def test_construction_gives_exact_codes_and_unit_margins():
    w, qc, kc = _workload()
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v)
    assert np.array_equal(prep.q8, qc) and np.array_equal(prep.k8, kc)     # codes are the integers
    assert np.all(prep.k_mean == 0) and np.all(prep.q_scale == U) and np.all(prep.k_scale == U)
    f = np.float32(np.float32(U) * np.float32(U)) * O.score_factor_c(SM_SCALE)
    assert abs(float(f) - 4.0) < 1e-3
    margins = []
    for h in range(w.H):
        s = O.qk_scores(prep.q8[0, h], prep.k8[0, h])
        top = s.max(axis=1)
        second = np.where(s < top[:, None], s, np.iinfo(np.int64).min).max(axis=1)
        margins.append(top - second)
    margins = np.concatenate(margins)
    assert np.mean(margins == 1) > 0.95                  # nearly every row has a runner-up one below


@pytest.mark.gpu
def test_production_kernel_scores_are_exact_at_the_top():
    w, _, _ = _workload()
    run = G.GpuRun(w).prep()
    base = torch.zeros((w.B, w.H, w.Nq, w.D), dtype=torch.bfloat16, device="cuda")
    S.sage_attn_fwd(run.bufs, base, sm_scale=SM_SCALE)                     # the default form
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    got = base.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v)
    for h in range(w.H):
        ref, _ = O.attention_rows(prep, 0, h, np.arange(w.Nq), sm_scale=SM_SCALE)
        assert G.within_tolerance(got[0, h], ref), h


def test_a_one_unit_score_error_at_the_top_is_beyond_the_tolerance():
    # the power of the GPU check: moving each row's best score by one unit
    # either way (planted in the oracle) takes the output outside the bar
    w, _, _ = _workload()
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v)
    ref = O.bf16_bits_to_f32(O.attention_rows(prep, 0, 0, np.arange(w.Nq), sm_scale=SM_SCALE)[0])
    for shift in (-1, 1):
        alt = O.bf16_bits_to_f32(_shifted_top_score(prep, 0, shift))
        assert not G.within_tolerance(O.f32_to_bf16_bits(alt), O.f32_to_bf16_bits(ref))
        assert np.abs(alt - ref).max() > 0.1


def _shifted_top_score(prep, h, shift):
    """Oracle output with each row's best key's score moved by `shift` units
    (a planted score error, on the CPU)."""
    p2 = O.Prepared(prep.q8.copy(), prep.k8.copy(), prep.v8, prep.q_scale, prep.k_scale, prep.v_scale,
                    prep.k_mean, prep.q_len, prep.kv_len, prep.bkv)
    s = O.qk_scores(prep.q8[0, h], prep.k8[0, h])
    rows = np.arange(s.shape[0])
    outs = []
    for i in rows:
        j = int(np.argmax(s[i]))
        # an error of `shift` in S[i, j]: shift the key's last-channel code,
        # where this query's code is 1 (one score unit per code unit)
        k8 = prep.k8.copy()
        k8[0, h, j, -1] = np.int8(int(k8[0, h, j, -1]) + shift)
        p2.k8 = k8
        out, _ = O.attention_rows(p2, 0, h, np.array([i]), sm_scale=SM_SCALE)
        outs.append(out[0])
    return np.stack(outs)
