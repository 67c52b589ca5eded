"""Planted mistakes in the oracle must fail at least one pin.

Each case swaps one oracle helper or constant for a plausible wrong version
(on the CPU, through monkeypatch) and runs the pin that should catch it.
A pin that still passes would mean the oracle is not pinned at that point.
"""
import numpy as np
import pytest

from oracle import sage_oracle as O
from tests import test_oracle_attention as TA
from tests import test_oracle_causal as TC
from tests import test_oracle_formats as TF
from tests import test_oracle_prep as TP


_ENCODE = O.e4m3_encode


def _ties_away(x):
    # round-half-away-from-zero instead of ties-to-even
    xv = np.asarray(x, np.float64)
    out = _ENCODE(xv)
    below = np.abs(O.e4m3_decode(out))
    up = _ENCODE(np.nextafter(np.abs(xv), np.inf)) & 0x7F
    d_out = np.abs(np.abs(xv) - below)
    d_up = np.abs(O.e4m3_decode(up) - np.abs(xv))
    tie = (d_out > 0) & (d_up == d_out) & (O.e4m3_decode(up) > below)
    return np.where(tie, (up | (out & 0x80)).astype(np.uint8), out).astype(np.uint8)


_VISIBLE = O.visible_keys
_QUANT_V = O.quantize_v_fp8


def _v_scale_ignores_tile(v, valid, s_v=None):
    # the BKV = 64 variant quantizing V with the BKV = 128 target magnitude
    return _QUANT_V(v, valid, None)


def _causal_top_left(prep, b, rows, causal):
    # diagonal through (0, 0) instead of through the last query and last key
    if not causal:
        return _VISIBLE(prep, b, rows, causal)
    return np.clip(np.asarray(rows, np.int64) + 1, 0, int(prep.kv_len[b]))


def _causal_strict(prep, b, rows, causal):
    # j < i + (Lk - Lq): the diagonal key itself hidden
    return np.maximum(_VISIBLE(prep, b, rows, causal) - (1 if causal else 0), 0)


def _mean_over_channels(k, kv_len):
    lead = k.shape[:-2]
    m = np.asarray(k[..., :max(kv_len, 1), :], np.float32).mean(axis=-1)       # wrong axis
    return np.broadcast_to(m[..., :1], lead + (k.shape[-1],)).astype(np.float32)


MUTATIONS = {
    "natural_exp_instead_of_exp2": (
        lambda mp: mp.setattr(O, "exp2_f32", lambda x: np.exp(np.asarray(x, np.float64)).astype(np.float32)),
        lambda: TA.test_oracle_close_to_fp64_attention(2)),
    "score_factor_without_log2e": (
        lambda mp: mp.setattr(O, "score_factor_c", lambda s: np.float32(s)),
        lambda: TA.test_oracle_close_to_fp64_attention(2)),
    "k_mean_over_wrong_axis": (
        lambda mp: mp.setattr(O, "k_channel_mean", _mean_over_channels),
        TP.test_smoothed_keys_have_zero_channel_mean),
    "e4m3_ties_away_from_zero": (
        lambda mp: mp.setattr(O, "e4m3_encode", _ties_away),
        TF.test_e4m3_encode_midpoints_and_neighbours_match_torch),
    "v_scaled_to_e4m3_max": (
        lambda mp: mp.setattr(O, "S_V", 448.0),
        TA.test_checkpoints_follow_online_softmax_invariants),
    "k_scale_block_128": (
        lambda mp: mp.setattr(O, "BKS", 128),
        TP.test_prepare_shapes_and_varlen_padding),
    "q_scale_block_64": (
        lambda mp: mp.setattr(O, "BQS", 64),
        TP.test_prepare_shapes_and_varlen_padding),
    "causal_diagonal_top_left": (
        lambda mp: mp.setattr(O, "visible_keys", _causal_top_left),
        lambda: TC.test_causal_close_to_fp64_masked_attention(200, 333, 128)),
    "causal_diagonal_key_hidden": (
        lambda mp: mp.setattr(O, "visible_keys", _causal_strict),
        TC.test_causal_first_row_is_its_first_value),
    "bkv64_keeps_bkv128_v_scale": (
        lambda mp: mp.setattr(O, "quantize_v_fp8", _v_scale_ignores_tile),
        TC.test_bkv64_v_scale_and_tiles),
    "kv_tile_256": (
        lambda mp: mp.setattr(O, "BKV", 256),
        TA.test_checkpoints_follow_online_softmax_invariants),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    plant, pin = MUTATIONS[name]
    pin()                                   # the pin passes on the real oracle
    plant(monkeypatch)
    with pytest.raises((AssertionError, FloatingPointError, ValueError, IndexError)):
        pin()
