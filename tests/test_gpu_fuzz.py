"""Seeded randomized sweep over shapes, varlen lengths and every form of the
path, each compared with the oracle of the same form.

The cases are drawn once from a fixed seed, so the sweep is the same on
every run.  Each draws the form (default, causal, one-call entry, BKV = 64,
D = 64, D = 64 with BKV = 64, CTA pairs and their causal variants), batch
and head counts, query and key lengths (1-384, spanning several tiles and a
ragged tail), the physical layout (NHD or HND) and, for half the cases,
per-item q_len / kv_len between 0 and the buffer length.  The checks are those of the edge-case tests: the
output within the tolerance, rows that see no key zero, rows past q_len left
untouched.
"""
import random

import numpy as np
import pytest

from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import workloads as W
from tests import gpu_support as G
from tests.test_gpu_edges_forms import CANARY, FORMS, _run_form

pytestmark = pytest.mark.gpu

FUZZ_FORMS = {"default": {}, **FORMS, "bkv64_causal": dict(bkv=64, causal=True),
              "d64_bkv64": dict(D=64, bkv=64)}


def _draw_cases(n=40, seed=2026):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        form = rng.choice(sorted(FUZZ_FORMS))
        B, H = rng.randint(1, 3), rng.randint(1, 3)
        Nq, Nkv = rng.randint(1, 384), rng.randint(1, 384)
        varlen = rng.random() < 0.5
        spec = dict(B=B, H=H, Nq=Nq, Nkv=Nkv, seed=1000 + i, layout=rng.choice(["nhd", "hnd"]),
                    k_offset_std=rng.choice([0.0, 1.0, 3.0]))
        if varlen:
            spec["q_len"] = [rng.randint(0, Nq) for _ in range(B)]
            spec["kv_len"] = [rng.randint(0, Nkv) for _ in range(B)]
        cases.append((f"{i:02d}_{form}_B{B}H{H}_{Nq}x{Nkv}{'_varlen' if varlen else ''}", form, spec))
    return cases


CASES = _draw_cases()


@pytest.mark.parametrize("name,form,spec", CASES, ids=[c[0] for c in CASES])
def test_random_case_matches_oracle(name, form, spec):
    f = FUZZ_FORMS[form]
    w = W.make_custom(**spec, D=f.get("D", 128))
    got = _run_form(w, f)
    q, k, v = G.logical_f32(w)
    prep = O.prepare(q, k, v, w.q_len, w.kv_len, bkv=f.get("bkv", 128))
    causal = f.get("causal", False)
    ref = O.attention(prep, causal=causal)
    for b in range(w.B):
        lq, lk = w.qlens[b], w.kvlens[b]
        assert G.within_tolerance(got[b, :, :lq], ref[b, :, :lq]), G.out_metrics(got[b, :, :lq], ref[b, :, :lq])
        hidden = np.full(lq, lk == 0)
        if causal:
            hidden |= np.arange(lq) + (lk - lq) < 0
        assert np.all(got[b, :, :lq][:, hidden] == 0)
        assert np.all(got[b, :, lq:] == CANARY), "rows beyond q_len were written"
