"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
on a seeded workload and run the oracle on the same BF16 bytes."""
from __future__ import annotations

import functools

import numpy as np
import torch

import quantized_exact_attention_gb300 as S
from oracle import sage_oracle as O
from quantized_exact_attention_gb300 import build as B
from quantized_exact_attention_gb300 import workloads as W

OUT_MAX_ABS = 1e-2      # BF16 output vs oracle: max |difference| ...
OUT_REL_L2 = 5e-3       # BF16 output vs oracle: ||difference|| / ||oracle||
# ... except where one BF16 ulp of the oracle value exceeds 1e-2 (|o| >= 2):
# two correct implementations that round slightly different FP32 values to
# BF16 can land one ulp apart there, so the bound is max(1e-2, 1 ulp).


def ensure_built():
    B.build()
    S.load_library()


def logical_f32(w: W.Workload):
    """Oracle inputs: float32 [B, H, N, D] copies of the workload's BF16 values."""
    return [t.float().numpy() for t in w.views()]


@functools.lru_cache(maxsize=4)
def oracle_prep(w_key):
    w = _WORKLOADS[w_key]
    q, k, v = logical_f32(w)
    return O.prepare(q, k, v, w.q_len, w.kv_len)


_WORKLOADS: dict = {}


def register(w: W.Workload) -> str:
    _WORKLOADS[w.name] = w
    return w.name


class GpuRun:
    """Device copies of a workload plus its prep buffers and output."""

    def __init__(self, w: W.Workload, int8_codes=True):
        ensure_built()
        self.w = w
        self.phys = w.to("cuda")
        self.q, self.k, self.v = w.views(self.phys)
        self.q_len = (torch.tensor(w.q_len, dtype=torch.int32, device="cuda")
                      if w.q_len is not None else None)
        self.kv_len = (torch.tensor(w.kv_len, dtype=torch.int32, device="cuda")
                       if w.kv_len is not None else None)
        self.bufs = S.alloc_prep_buffers(w.B, w.H, w.Nq, w.Nkv, "cuda", int8_codes=int8_codes, D=w.D)
        self.out = None

    def prep(self, bkv=128):
        S.sage_prep_qkv(self.q, self.k, self.v, self.bufs, self.q_len, self.kv_len, bkv=bkv)
        torch.cuda.synchronize()
        return self

    def attn(self, fill=None, causal=False, bkv=128, pairs=False):
        w = self.w
        base = torch.empty((w.B, w.Nq, w.H, w.D), dtype=torch.bfloat16, device="cuda")
        if fill is None:
            base.zero_()
        else:
            base.fill_(fill)
        self.out = base.permute(0, 2, 1, 3)
        S.sage_attn_fwd(self.bufs, self.out, self.q_len, self.kv_len, Nkv=w.Nkv, causal=causal, bkv=bkv,
                        pairs=pairs)
        torch.cuda.synchronize()
        assert S.sage_get_device_status() == S.SAGE_OK
        return self

    def qk(self):
        w = self.w
        s = torch.zeros((w.B, w.H, w.Nq, w.Nkv), dtype=torch.int32, device="cuda")
        S.sage_qk_int32(self.bufs, s, self.q_len, self.kv_len)
        torch.cuda.synchronize()
        assert S.sage_get_device_status() == S.SAGE_OK
        return s

    def out_bits(self) -> np.ndarray:
        return self.out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def compare_prep(run: GpuRun, prep: O.Prepared):
    """Bit-exact comparison of every preparation output; returns nothing, asserts."""
    w = run.w
    b = run.bufs
    lq, lk = w.qlens, w.kvlens
    q16 = b.q16.float().cpu().numpy()
    k16 = b.k16.float().cpu().numpy()
    assert np.array_equal(q16, prep.q8.astype(np.float32)), "FP16 Q code images differ"
    assert np.array_equal(k16, prep.k8.astype(np.float32)), "FP16 K code images differ"
    if b.q8 is not None:
        assert np.array_equal(b.q8.cpu().numpy(), prep.q8), "INT8 Q bytes differ"
        assert np.array_equal(b.k8.cpu().numpy(), prep.k8), "INT8 K bytes differ"
    v8 = b.v8t.cpu().numpy().transpose(0, 1, 3, 2)[:, :, :w.Nkv, :]
    assert np.array_equal(v8, prep.v8), "FP8 V bytes differ"
    assert np.all(b.v8t.cpu().numpy()[..., w.Nkv:] == 0), "V padding not zero"
    for name in ("q_scale", "k_scale", "v_scale", "k_mean"):
        g = getattr(b, name).cpu().numpy()
        o = getattr(prep, name)
        assert g.shape == o.shape, name
        assert np.array_equal(g.view(np.uint32), o.view(np.uint32)), f"{name} differs"
    del lq, lk


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (8 significand bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def out_metrics(gpu_bits: np.ndarray, ref_bits: np.ndarray):
    """(excess, rel_l2, max_abs): excess = max(|g-r| - max(1e-2, ulp(r))) must be <= 0."""
    g = O.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    r = O.bf16_bits_to_f32(ref_bits).astype(np.float64)
    if g.size == 0:
        return 0.0, 0.0, 0.0
    diff = np.abs(g - r)
    excess = float((diff - np.maximum(OUT_MAX_ABS, bf16_ulp(r))).max())
    den = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / den) if den > 0 else float(np.linalg.norm(g - r))
    return excess, rel, float(diff.max())


def literal_bar_audit(gpu_bits: np.ndarray, ref_bits: np.ndarray):
    """Elements whose |difference| exceeds the literal max-abs 1e-2 bar.

    Returns (count, all_adjacent): all_adjacent is True when every such
    element is exactly one BF16 step away from the oracle value (neighbouring
    bit patterns of the same sign) and the oracle value has |o| >= 2, where
    one BF16 step (>= 2^-6 = 0.0156) is itself larger than 1e-2.
    """
    g = O.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    r = O.bf16_bits_to_f32(ref_bits).astype(np.float64)
    over = np.abs(g - r) > OUT_MAX_ABS
    n = int(np.count_nonzero(over))
    if n == 0:
        return 0, True
    gb = gpu_bits[over].astype(np.int32)
    rb = ref_bits[over].astype(np.int32)
    same_sign = (gb & 0x8000) == (rb & 0x8000)
    adjacent = same_sign & (np.abs(gb - rb) == 1)
    large = np.abs(r[over]) >= 2.0
    return n, bool(np.all(adjacent & large))


def within_tolerance(gpu_bits, ref_bits):
    excess, rel, _ = out_metrics(gpu_bits, ref_bits)
    return excess <= 0.0 and rel <= OUT_REL_L2
