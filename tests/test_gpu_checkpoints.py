"""Stage checkpoints of one query tile against the oracle (Experiment Log,
"Phase 2B Fixed Aligned Numerical Prototype" lists the checkpoints QK, m, d,
FP8 probability, rescale, FP16 PV, FP32 RO and reciprocal).

Each stage is checked where its inputs are pinned:
  m       bit-exact vs the oracle (a maximum of RN(S * f), order-free)
  alpha   vs the oracle's exact exp2 within ex2.approx error (same argument);
          below 2^-126 the GPU's flush to zero is accepted
  P8      e4m3 codes adjacent to the oracle's, and rarely different
  PV16    within four FP16 roundings of the exact sum of the GPU's own P bytes
          times the V codes (the tensor core accumulates 4 K-steps in FP16)
  RO      bit-exact replay of RO = RN(RN(RO * alpha) + PV16) from the GPU's
          own alpha and PV16
  l       448 * the oracle's sum of p, within FP32 summation error
  recip   bit-exact RN(1 / l) of the GPU's l; the output row bit-exact from
          RO, recip and v_scale
QK itself is the bit-exact sage_qk_int32 checkpoint of the main parity tests.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G

pytestmark = pytest.mark.gpu

F32 = np.float32
CASES = {
    "cfg1": (dict(W.CONFIGS[1]), (0, 0, 0), False),
    "cfg2_head5_tile3": (dict(W.CONFIGS[2]), (0, 5, 3), False),
    "varlen_tail": (dict(B=2, H=2, Nq=500, Nkv=700, seed=80, k_offset_std=2.0, q_len=[500, 300],
                         kv_len=[700, 333]), (1, 1, 2), False),
    "causal_diag": (dict(B=1, H=2, Nq=640, Nkv=640, seed=81), (0, 1, 3), True),
    "d64": (dict(B=1, H=2, Nq=384, Nkv=520, seed=82, D=64, k_offset_std=3.0), (0, 1, 1), False),
    "cfg3_varlen_item1": (dict(W.CONFIGS[3]), (1, 9, 6), False),
    "cfg4_long_tile64": (dict(W.CONFIGS[4]), (0, 7, 64), False),
    "cfg5_outliers": (dict(W.CONFIGS[5]), (11, 4, 9), False),
}


def _f16_ulp(x):
    a = np.maximum(np.abs(x), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(a)) - 10)


@pytest.mark.parametrize("name", sorted(CASES))
def test_stage_checkpoints(name):
    spec, (b, h, qt), causal = CASES[name]
    w = W.make_custom(**spec)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len)
    run = G.GpuRun(w).prep()
    out = torch.zeros((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    ck = S.sage_attn_checkpoints(run.bufs, out, b, h, qt, run.q_len, run.kv_len, causal=causal, Nkv=w.Nkv)
    torch.cuda.synchronize()
    assert S.sage_get_device_status() == S.SAGE_OK
    ck = {n: t.cpu().numpy() for n, t in ck.items()}

    lq, lk = w.qlens[b], w.kvlens[b]
    rows = np.arange(qt * 128, min(qt * 128 + 128, lq))
    vis = O.visible_keys(prep, b, rows, causal)
    live = vis > 0
    rows, rl = rows[live], np.nonzero(live)[0]                # rl: row index within the tile
    ref = O.Checkpoints()
    O.attention_rows(prep, b, h, rows, checkpoints=ref, causal=causal)
    T = len(ref.m)
    v_dec = O.e4m3_decode(prep.v8[b, h])
    ro = np.zeros((len(rows), w.D), F32)
    p8_diff = p8_total = 0
    for t in range(T):
        width = min(128, int(vis.max()) - t * 128)
        # m: bit-exact
        assert np.array_equal(ck["m"][t, rl].view(np.uint32), ref.m[t].view(np.uint32)), f"m tile {t}"
        # alpha: ex2.approx of the same argument; the GPU flushes results below
        # the FP32 normal range (2^-126) to zero where the oracle keeps subnormals
        a_g, a_r = ck["alpha"][t, rl].astype(np.float64), ref.alpha[t].astype(np.float64)
        tol = np.where(a_r < 2.0 ** -126, 2.0 ** -126, 2.0 ** -21 * a_r)
        assert np.all(np.abs(a_g - a_r) <= tol), f"alpha tile {t}"
        # P8: adjacent codes, rare differences; columns beyond the visible keys are 0
        g8 = ck["p8"][t, rl, :width].astype(np.int32)
        r8 = ref.p8[t].astype(np.int32)
        assert np.all(np.abs((g8 & 0x7F) - (r8 & 0x7F)) <= 1), f"P8 tile {t}"
        assert np.all(ck["p8"][t, rl, width:] == 0)
        p8_diff += int(np.count_nonzero(g8 != r8))
        p8_total += g8.size
        # PV16: exact sum of the GPU's own P bytes times V, within a few FP16
        # roundings at the size of the partial sums of the four 32-key K-steps
        pv_g = ck["pv16"][t, rl].astype(np.float64)
        pd = O.e4m3_decode(ck["p8"][t, rl, :width])
        vd = v_dec[t * 128:t * 128 + width]
        partial = np.stack([pd[:, :j] @ vd[:j] for j in range(32, width + 32, 32)])
        exact = partial[-1]
        scale = np.abs(partial).max(axis=0)
        assert np.all(np.abs(pv_g - exact) <= 8 * _f16_ulp(scale) + 1e-12), f"PV16 tile {t}"
        # RO: bit-exact replay from the GPU's alpha and PV16
        ro = ((ro * ck["alpha"][t, rl][:, None]).astype(F32) + ck["pv16"][t, rl].astype(F32)).astype(F32)
        assert np.array_equal(ck["ro"][t, rl].view(np.uint32), ro.view(np.uint32)), f"RO tile {t}"
    assert p8_diff <= max(2, 1e-3 * p8_total), (p8_diff, p8_total)
    # l: 448 * sum(p) of the oracle
    l_g = ck["l"][T - 1, 0, rl].astype(F32) + ck["l"][T - 1, 1, rl].astype(F32)
    assert np.allclose(l_g, 448.0 * ref.l[-1].astype(np.float64), rtol=2e-5)
    # reciprocal and output: bit-exact from the GPU's own l, RO and v_scale
    recip = (F32(1.0) / l_g).astype(F32)
    assert np.array_equal(ck["recip"][rl].view(np.uint32), recip.view(np.uint32))
    o = ((ro * recip[:, None]).astype(F32) * prep.v_scale[b, h][None, :]).astype(F32)
    got = out[b, h, rows].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, O.f32_to_bf16_bits(o))
