"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out in memory; it holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it.  Every tensor is drawn on the CPU with a seeded
``torch.Generator`` in float32 and rounded once to BF16, so the same BF16
bytes go to the GPU and to the oracle.

The pages measure on private model fixtures that are not available, so these
shapes and value distributions stand in for them:

  1  single aligned tile: B=1,H=1,Nq=128,Nkv=192, N(0,1), NHD
  2  B=1,H=8,N=1024; Q,V N(0,1); K N(0,1) + per-(h,d) offset N(0,3^2), NHD
  3  B=2,H=16,Nmax=1000, item 1 has Nq=Nkv=777 (varlen); N(0,1);
     K + per-(b,h,d) offset N(0,2^2), NHD
  4  B=1,H=24,N=16384; Q,K N(0,1), K + per-(h,d) offset N(0,2^2), V N(0,1);
     strided NHD views into one fused [B,N,3,H,D] projection buffer
  5  B=16,H=16,N=2048; N(0,1); 1% of Q and 1% of K entries (independent
     Bernoulli(0.01) masks) multiplied by 20; HND

All tensors are exposed as logical [B, H, N, D] views (possibly strided) over
a physical buffer, which is what the C ABI takes (element strides, D unit).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

D_HEAD = 128


@dataclass
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nkv: int
    D: int
    layout: str                 # "nhd", "hnd" or "nhd_fused"
    phys: tuple                 # physical buffers (q, k, v) or (qkv,)
    q_len: list | None          # per-batch valid query rows (None: all Nq)
    kv_len: list | None         # per-batch valid keys (None: all Nkv)

    # logical [B, H, N, D] views over the physical buffers
    def views(self, phys=None):
        phys = self.phys if phys is None else phys
        if self.layout == "nhd":
            return tuple(t.permute(0, 2, 1, 3) for t in phys)
        if self.layout == "hnd":
            return tuple(phys)
        if self.layout == "nhd_fused":
            (qkv,) = phys
            return tuple(qkv[:, :, i].permute(0, 2, 1, 3) for i in range(3))
        raise ValueError(self.layout)

    def to(self, device):
        return tuple(t.to(device) for t in self.phys)

    @property
    def qlens(self):
        return list(self.q_len) if self.q_len is not None else [self.Nq] * self.B

    @property
    def kvlens(self):
        return list(self.kv_len) if self.kv_len is not None else [self.Nkv] * self.B

    def ops(self) -> int:
        """4 * H * D * sum_b Lq_b * Lk_b  (QK^T and PV multiply-adds, 2 ops each)."""
        return 4 * self.H * self.D * sum(a * b for a, b in zip(self.qlens, self.kvlens))


def _randn(g, shape):
    return torch.randn(shape, generator=g, dtype=torch.float32)


def _bf16(x):
    return x.to(torch.bfloat16)


def make_custom(B, H, Nq, Nkv, seed, layout="nhd", k_offset_std=0.0, q_len=None,
                kv_len=None, outlier_frac=0.0, outlier_mult=20.0, D=D_HEAD,
                name=None) -> Workload:
    """General generator used by the named configs and by the tests.

    Draw order (fixed): Q, K, V as float32 N(0,1) in logical [B, H, N, D]
    order; then the K channel offset [B, H, D] (or [1, H, D] broadcast when
    B == 1) times k_offset_std; then the outlier masks for Q and K.
    """
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (B, H, Nq, D))
    k = _randn(g, (B, H, Nkv, D))
    v = _randn(g, (B, H, Nkv, D))
    if k_offset_std:
        k = k + _randn(g, (B, H, 1, D)) * k_offset_std
    if outlier_frac:
        mq = torch.rand((B, H, Nq, D), generator=g) < outlier_frac
        mk = torch.rand((B, H, Nkv, D), generator=g) < outlier_frac
        q = torch.where(mq, q * outlier_mult, q)
        k = torch.where(mk, k * outlier_mult, k)
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    if layout == "hnd":
        phys = (q.contiguous(), k.contiguous(), v.contiguous())
    elif layout == "nhd":
        phys = tuple(t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v))
    elif layout == "nhd_fused":
        assert Nq == Nkv
        qkv = torch.stack([t.permute(0, 2, 1, 3) for t in (q, k, v)], dim=2).contiguous()
        phys = (qkv,)
    else:
        raise ValueError(layout)
    return Workload(name or f"custom_B{B}_H{H}_Nq{Nq}_Nkv{Nkv}", B, H, Nq, Nkv, D,
                    layout, phys, q_len, kv_len)


CONFIGS = {
    1: dict(B=1, H=1, Nq=128, Nkv=192, seed=0, layout="nhd",
            name="single_tile_B1_H1_Nq128_Nkv192_D128"),
    2: dict(B=1, H=8, Nq=1024, Nkv=1024, seed=1, layout="nhd", k_offset_std=3.0,
            name="koffset3_B1_H8_N1024_D128"),
    3: dict(B=2, H=16, Nq=1000, Nkv=1000, seed=2, layout="nhd", k_offset_std=2.0,
            q_len=[1000, 777], kv_len=[1000, 777], name="varlen_B2_H16_N1000_777_D128"),
    4: dict(B=1, H=24, Nq=16384, Nkv=16384, seed=3, layout="nhd_fused", k_offset_std=2.0,
            name="long_dit_B1_H24_N16384_D128_strided_nhd"),
    5: dict(B=16, H=16, Nq=2048, Nkv=2048, seed=4, layout="hnd", outlier_frac=0.01,
            name="outlier_B16_H16_N2048_D128_hnd"),
}


def make_config(i: int) -> Workload:
    return make_custom(**CONFIGS[i])
