"""Pins for the oracle's causal masking (reading R15) and head dimension 64.

Neither is on the pages; both are adjacent uses of the same contract (the
attention stages of Experiment Log, "Phase 0 Import And Verification").  The
causal reading: key j is visible to query i iff j <= i + (Lk - Lq); rows that
see no key are zero.  Checked against FP64 masked softmax attention, a closed
form for the first row, and the equality with a shorter key range.
"""
import dataclasses
import math

import numpy as np
import pytest

from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests.test_oracle_attention import _dequant_v, _logical, _metrics, fp64_attention

F32 = np.float32


def fp64_causal_attention(q, k, v, sm_scale=None):
    """softmax(Q K^T * scale + mask) V in float64; key j visible to query i iff
    j <= i + (Lk - Lq); rows with no visible key are zero."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    lq, lk = q.shape[-2], k.shape[-2]
    sm_scale = 1 / math.sqrt(q.shape[-1]) if sm_scale is None else sm_scale
    s = np.einsum("bhid,bhjd->bhij", q, k) * sm_scale
    vis = np.arange(lk)[None, :] <= np.arange(lq)[:, None] + (lk - lq)
    s = np.where(vis, s, -np.inf)
    out = np.zeros(q.shape[:-1] + (v.shape[-1],))
    live = vis.any(1)
    sl = s[..., live, :]
    sl = sl - sl.max(-1, keepdims=True)
    p = np.exp(sl)
    p /= p.sum(-1, keepdims=True)
    out[..., live, :] = np.einsum("bhij,bhjd->bhid", p, v)
    return out


@pytest.mark.parametrize("lq,lk,d", [(300, 300, 128), (200, 333, 128), (333, 200, 128), (257, 257, 64),
                                     (130, 390, 64)])
def test_causal_close_to_fp64_masked_attention(lq, lk, d):
    w = W.make_custom(B=1, H=2, Nq=lq, Nkv=lk, seed=40 + lq + d, k_offset_std=2.0, D=d)
    q, k, v = _logical(w)
    out = O.bf16_bits_to_f32(O.attention(O.prepare(q, k, v), causal=True))
    ref = fp64_causal_attention(q, k, v)
    hidden = ~np.any(np.arange(lk)[None, :] <= np.arange(lq)[:, None] + (lk - lq), axis=1)
    assert np.all(out[:, :, hidden] == 0)                     # R15: rows that see nothing
    cos, rel = _metrics(out, ref)
    assert cos >= 0.999 and rel <= 5e-2


def test_causal_first_row_is_its_first_value():
    # Lq = Lk: row 0 sees key 0 only -> p = 1, P8 = 448, PV = 448 * v8 exactly
    w = W.make_custom(B=1, H=3, Nq=200, Nkv=200, seed=44)
    q, k, v = _logical(w)
    prep = O.prepare(q, k, v)
    for h in range(3):
        row = O.attention_rows(prep, 0, h, np.array([0]), causal=True)[1][0]
        exact = _dequant_v(prep, 0, h, 1)[0]
        ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64) * 2 ** 16
        assert np.all(np.abs(row - exact) <= ulp)


@pytest.mark.parametrize("lq,lk", [(260, 260), (200, 333), (333, 200)])
def test_causal_row_equals_attention_over_its_visible_prefix(lq, lk):
    # R15: fully hidden tiles change nothing, so a causal row is bit-identical to
    # the non-causal row computed with kv_len cut to the keys it sees (same codes)
    w = W.make_custom(B=1, H=1, Nq=lq, Nkv=lk, seed=45, k_offset_std=2.0)
    q, k, v = _logical(w)
    prep = O.prepare(q, k, v)
    rows = np.array(sorted({0, 1, 63, 127, 128, 129, lq // 2, lq - 2, lq - 1}))
    causal = O.attention_rows(prep, 0, 0, rows, causal=True)[0]
    for n, i in enumerate(rows):
        vis = int(O.visible_keys(prep, 0, np.array([i]), True)[0])
        if vis == 0:
            assert np.all(causal[n] == 0)
            continue
        cut = dataclasses.replace(prep, kv_len=np.array([vis]))
        assert np.array_equal(causal[n], O.attention_rows(cut, 0, 0, np.array([i]))[0][0])


def test_causal_is_noncausal_when_every_key_is_visible():
    # one query row placed after all keys (Lq = 1): the mask hides nothing
    w = W.make_custom(B=1, H=2, Nq=1, Nkv=300, seed=46)
    q, k, v = _logical(w)
    prep = O.prepare(q, k, v)
    assert np.array_equal(O.attention(prep, causal=True), O.attention(prep))


@pytest.mark.parametrize("cfg_d", [64])
def test_d64_close_to_fp64_attention(cfg_d):
    w = W.make_custom(B=1, H=4, Nq=384, Nkv=320, seed=47, k_offset_std=3.0, D=cfg_d)
    q, k, v = _logical(w)
    out = O.bf16_bits_to_f32(O.attention(O.prepare(q, k, v)))
    cos, rel = _metrics(out, fp64_attention(q, k, v))
    assert cos >= 0.999 and rel <= 5e-2


def test_d64_single_key_gives_dequantized_value_row():
    rng = np.random.default_rng(48)
    q = rng.standard_normal((1, 2, 150, 64)).astype(F32)
    k = rng.standard_normal((1, 2, 1, 64)).astype(F32)
    v = rng.standard_normal((1, 2, 1, 64)).astype(F32)
    prep = O.prepare(q, k, v)
    out = O.bf16_bits_to_f32(O.attention(prep))
    for h in range(2):
        exact = _dequant_v(prep, 0, h, 1)[0]
        ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64) * 2 ** 16
        assert np.all(np.abs(out[0, h] - exact[None, :]) <= ulp[None, :])


# --- BKV = 64 contract variant (R16) ------------------------------------------
@pytest.mark.parametrize("cfg", [2, 3])
def test_bkv64_close_to_fp64_attention(cfg):
    w = W.make_config(cfg)
    if cfg == 3:
        w = W.make_custom(B=2, H=3, Nq=500, Nkv=500, seed=49, k_offset_std=2.0, q_len=[500, 301],
                          kv_len=[500, 377])
    q, k, v = _logical(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len, bkv=64)
    out = O.bf16_bits_to_f32(O.attention(prep))
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        cos, rel = _metrics(out[b:b + 1, :, :lq], fp64_attention(q[b:b + 1, :, :lq], k[b:b + 1, :, :lk],
                                                                  v[b:b + 1, :, :lk]))
        assert cos >= 0.999 and rel <= 5e-2


def test_bkv64_v_scale_and_tiles():
    # S_V doubles with half the tile; every V code then covers |v| <= 2.25
    w = W.make_custom(B=1, H=1, Nq=128, Nkv=300, seed=50)
    q, k, v = _logical(w)
    p128, p64 = O.prepare(q, k, v), O.prepare(q, k, v, bkv=64)
    assert np.array_equal(p128.v_scale.view(np.uint32), (p64.v_scale * F32(2)).view(np.uint32))
    assert np.abs(O.e4m3_decode(p64.v8)).max() <= 2.25
    assert np.array_equal(p128.q8, p64.q8) and np.array_equal(p128.k8, p64.k8)
    ck = O.Checkpoints()
    O.attention_rows(p64, 0, 0, np.arange(128), checkpoints=ck)
    assert len(ck.m) == 5                                      # ceil(300 / 64) tiles
    assert max(np.abs(pv).max() for pv in ck.pv16) <= 64 * 448 * 2.25
    assert np.all((ck.p8[0] == 0x7E).any(axis=1))             # p = 1 at each row's first-tile max


def test_bkv64_single_key_gives_dequantized_value_row():
    rng = np.random.default_rng(51)
    q = rng.standard_normal((1, 2, 70, 128)).astype(F32)
    k = rng.standard_normal((1, 2, 1, 128)).astype(F32)
    v = rng.standard_normal((1, 2, 1, 128)).astype(F32)
    prep = O.prepare(q, k, v, bkv=64)
    out = O.bf16_bits_to_f32(O.attention(prep))
    for h in range(2):
        exact = _dequant_v(prep, 0, h, 1)[0]
        ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64) * 2 ** 16
        assert np.all(np.abs(out[0, h] - exact[None, :]) <= ulp[None, :])
