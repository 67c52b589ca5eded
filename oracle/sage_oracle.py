"""CPU oracle of the quantized exact attention contract (test infrastructure).

This module is TEST INFRASTRUCTURE.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The CUDA library never calls it and shares no code with it; the two sides
meet only through the seeded inputs and the bytes they produce.

What it computes
----------------
The numerical contract of SageAttention2-style quantized exact attention as
the source pages list its stages (Experiment Log, "Phase 0 Import And
Verification": Q/K preparation, K smoothing, INT8 quantization, QK traversal,
online softmax, FP8 V/P, two-level PV accumulation, final conversion, ragged
tails) and as the later phases name its checkpoints (Experiment Log, "Phase 2B
Fixed Aligned Numerical Prototype": QK, m, d, FP8 probability, rescale, FP16
PV, FP32 RO, reciprocal, final BF16 output; "Phase 1 State-Ownership
Decision": strict tile order, exact FP8 score bytes, per-tile RO rescaling).

The pages give the stages but none of their constants.  Every constant,
granularity and rounding choice below is a reading, tagged R1..R16 and listed
with its justification in the design notes:

  R3  K channel mean: FP32, chunks of 64 valid tokens summed in ascending
      order, chunk sums added in ascending order, one IEEE division.
  R4  smoothed K = K - mean in FP32, no re-rounding to BF16.
  R5  INT8 Q per 128-row block, INT8 K per 64-row block, symmetric
      [-127, 127], scale = amax/127, code = rne(x * (127/amax)).
  R6  FP8 V per (b, h, channel): v_scale = amax/S_V, code =
      e4m3_rne_satfinite(v * (S_V/amax)), S_V = 144/BKV = 1.125.
  R7  e4m3 is OCP E4M3 (bias 7, max 448, no infinities).
  R8  score factor f = (q_scale * k_scale) * c, c = fp32(sm_scale*log2(e)).
  R9  online softmax over KV tiles of BKV = 128 keys, strictly ascending;
      l sums the FP32 probabilities before quantization.
  R10 P8 = e4m3(p * 448).
  R11 PV tile sum exact, rounded once to FP16.
  R12 RO = RO * alpha + PV16 in FP32 every tile.
  R13 out = bf16((RO * (1/l)) * (v_scale/448)).
  R14 rows of a query with no keys are zero.
  R15 causal masking (not on the pages; an adjacent use): key j is visible
      to query i of a batch item iff j <= i + (Lk - Lq), i.e. the diagonal is
      aligned to the last query and the last key (j <= i when Lq = Lk).  A
      row that sees no key is zero, as in R14.  A tile whose keys are all
      hidden from a row changes nothing for it (alpha = exp2(0) = 1, p = 0),
      so the row's result is the non-causal one over its visible prefix.
  R16 a second contract variant with BKV = 64 (the pages' 64-key epochs):
      the online-softmax tile and the inner PV sum cover 64 keys and
      S_V = 144/64 = 2.25, so the FP16 bound BKV * S_P * S_V <= 65504 holds
      at the same margin.  Q/K blocks are unchanged.

Precision: every step is carried out in the precision the contract names
(FP32 via numpy float32 arithmetic, which rounds each operation to nearest
even and never contracts a*b+c); exact steps use float64 where float64 is
provably exact (integer QK sums < 2^53, e4m3 products on a 2^-18 grid).
exp2 is computed in float64 and rounded once to FP32.

Parity status: the pages print no worked example and no usable golden values
(their locked output hash has no published inputs), so this oracle is pinned
by brute force, closed forms, invariants and FP64 attention instead; see the
``-m "not gpu"`` tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# Contract constants (readings; the pages give none of these numbers).
# ---------------------------------------------------------------------------
D_HEAD = 128          # head dimension of every workload on the pages (Q128 x KV192 x D128)
BQS = 128             # R5: Q scale block (matches the Q128 tile of VEA-B)
BKS = 64              # R5: K scale block (matches the 64-key K/V slots of the probe)
BKV = 128             # R9: KV tile of the online softmax and of the inner PV sum
MEAN_CHUNK = 64       # R3: chunk length of the pinned K-mean summation order
S_P = 448.0           # R10: P is scaled by the e4m3 maximum before quantization
S_V = 144.0 / BKV     # R6: keeps BKV * S_P * S_V <= 65504 (FP16 range of the tile sum)
E4M3_MAX = 448.0

F32 = np.float32


# ---------------------------------------------------------------------------
# Number formats (R7 and the BF16/FP16 conversions)
# ---------------------------------------------------------------------------
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float32, exactly (BF16 is the top half of FP32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns, round to nearest, ties to even (finite inputs).

    Dropping the low 16 bits rounds toward zero; adding 0x7FFF plus the LSB of
    the kept half first turns that into round-to-nearest-even on the magnitude.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return (r & np.uint64(0xFFFF)).astype(np.uint16)


def _e4m3_magnitudes() -> np.ndarray:
    """The 127 finite non-negative E4M3 magnitudes, indexed by their 7-bit code.

    OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits (bias 7),
    3 mantissa bits.  Exponent field 0 holds subnormals m/8 * 2^-6; the code
    S.1111.111 is NaN and there is no infinity, so the largest finite value
    is 1.75 * 2^8 = 448.
    """
    mags = np.empty(127, dtype=np.float64)
    for code in range(127):
        e = code >> 3
        m = code & 7
        if e == 0:
            mags[code] = (m / 8.0) * 2.0 ** -6
        else:
            mags[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return mags


_E4M3_MAG = _e4m3_magnitudes()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 byte -> float64 value (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag_code = c & 0x7F
    sign = np.where((c & 0x80) != 0, -1.0, 1.0)
    out = np.full(c.shape, np.nan, dtype=np.float64)
    finite = mag_code != 0x7F
    out[finite] = sign[finite] * _E4M3_MAG[mag_code[finite]]
    return out


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Real value -> E4M3 byte, round to nearest with ties to even, saturating.

    The input is taken as an exact real (float32 or float64 values).  The
    result is the representable value nearest to |x|; on a tie the code with
    an even mantissa (even code) wins; magnitudes beyond 448 saturate to 448
    ("satfinite").  NaN maps to 0x7F.  The sign of zero is kept.
    """
    xv = np.asarray(x, dtype=np.float64)
    sign = np.signbit(xv)
    a = np.abs(xv)
    nan = np.isnan(xv)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    hi = np.searchsorted(_E4M3_MAG, a, side="left")          # first magnitude >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_MAG[hi] - a
    d_lo = a - _E4M3_MAG[lo]
    exact = d_hi == 0.0
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(exact, hi, np.where(pick_lo, lo, hi)).astype(np.uint8)
    code = np.where(sign, code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def f16_round(x: np.ndarray) -> np.ndarray:
    """Real (float64) -> nearest IEEE binary16 (ties to even); returns float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def exp2_f32(x: np.ndarray) -> np.ndarray:
    """2**x of a float32 argument, computed in float64 and rounded once to float32."""
    with np.errstate(over="ignore", under="ignore"):
        return np.exp2(np.asarray(x, dtype=np.float32).astype(np.float64)).astype(F32)


# ---------------------------------------------------------------------------
# Preparation: K smoothing, INT8 Q/K, FP8 V  (Phase 0: "Q/K preparation,
# K smoothing, INT8 quantization ... FP8 V")
# ---------------------------------------------------------------------------
def k_channel_mean(k: np.ndarray, kv_len: int) -> np.ndarray:
    """Per-channel mean of keys over their valid tokens (R3).

    k: float32 [..., N, D] (leading axes are independent heads; only the first
    kv_len rows of each are valid).  Order: the valid tokens are cut into
    chunks of 64; each chunk is summed from 0.0 in ascending token order in
    FP32; the chunk sums are added from 0.0 in ascending chunk order in FP32;
    the total is divided by kv_len once.  kv_len = 0 gives 0.
    """
    lead = k.shape[:-2]
    d = k.shape[-1]
    if kv_len == 0:
        return np.zeros(lead + (d,), dtype=F32)
    total = np.zeros(lead + (d,), dtype=F32)
    for c0 in range(0, kv_len, MEAN_CHUNK):
        s = np.zeros(lead + (d,), dtype=F32)
        for t in range(c0, min(c0 + MEAN_CHUNK, kv_len)):
            s = (s + k[..., t, :]).astype(F32)
        total = (total + s).astype(F32)
    return (total / F32(kv_len)).astype(F32)


def quantize_int8_blocks(x: np.ndarray, valid: int, block: int):
    """Per-block symmetric INT8 quantization of one head's rows (R5).

    x: float32 [N, D].  Rows [valid, N) are not part of any block: their codes
    are 0.  Block b covers valid rows [b*block, min((b+1)*block, valid)).
    Returns (codes int8 [N, D], scales float32 [ceil(N/block)]); scales of
    blocks holding no valid row are 0.
    """
    n, d = x.shape
    codes = np.zeros((n, d), dtype=np.int8)
    scales = np.zeros((n + block - 1) // block, dtype=F32)
    for b in range(len(scales)):
        r0, r1 = b * block, min((b + 1) * block, valid)
        if r1 <= r0:
            continue
        blk = x[r0:r1]
        amax = F32(np.max(np.abs(blk)))
        if amax == 0:
            continue
        scales[b] = F32(amax / F32(127.0))
        inv = F32(F32(127.0) / amax)
        q = np.rint((blk * inv).astype(F32))
        codes[r0:r1] = np.clip(q, -127, 127).astype(np.int8)
    return codes, scales


def quantize_v_fp8(v: np.ndarray, valid: int, s_v: float | None = None):
    """Per-channel FP8 e4m3 quantization of one head's values (R6).

    v: float32 [N, D].  Per channel d over the valid rows: amax = max |v|,
    v_scale = amax / S_V, code = e4m3_rne_satfinite(v * (S_V / amax)).
    Rows [valid, N) get code 0; channels with amax = 0 get scale 0, codes 0.
    s_v: the target magnitude S_V (default: the BKV = 128 contract's).
    Returns (codes uint8 [N, D], v_scale float32 [D]).
    """
    s_v = S_V if s_v is None else s_v
    n, d = v.shape
    codes = np.zeros((n, d), dtype=np.uint8)
    scale = np.zeros(d, dtype=F32)
    if valid == 0:
        return codes, scale
    vv = v[:valid]
    amax = np.max(np.abs(vv), axis=0).astype(F32)
    nz = amax > 0
    safe = np.where(nz, amax, F32(1.0)).astype(F32)
    inv = (F32(s_v) / safe).astype(F32)
    scale = np.where(nz, (amax / F32(s_v)).astype(F32), F32(0.0)).astype(F32)
    scaled = (vv * inv[None, :]).astype(F32)
    c = e4m3_encode(scaled)
    codes[:valid] = np.where(nz[None, :], c, np.uint8(0))
    return codes, scale


@dataclass
class Prepared:
    """Output of the preparation stage for a [B, H, N, D] problem."""
    q8: np.ndarray        # int8  [B, H, Nq, D]
    k8: np.ndarray        # int8  [B, H, Nkv, D]
    v8: np.ndarray        # uint8 [B, H, Nkv, D]  (e4m3 bytes, token-major)
    q_scale: np.ndarray   # f32   [B, H, ceil(Nq/128)]
    k_scale: np.ndarray   # f32   [B, H, ceil(Nkv/64)]
    v_scale: np.ndarray   # f32   [B, H, D]
    k_mean: np.ndarray    # f32   [B, H, D]
    q_len: np.ndarray     # int   [B]
    kv_len: np.ndarray    # int   [B]
    bkv: int = 128        # keys per online-softmax tile / inner PV sum (R9, R16)


def prepare(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_len=None, kv_len=None,
            smooth_k: bool = True, bkv: int | None = None) -> Prepared:
    """Quantize float32 [B, H, N, D] Q/K/V (values exactly representable in BF16).

    smooth_k=False skips the K mean subtraction (used only to show what the
    smoothing step buys; the contract always smooths).  bkv: the contract's
    KV tile (128, or 64 for R16); S_V scales inversely with it.
    """
    bkv = BKV if bkv is None else int(bkv)
    s_v = S_V * BKV / bkv
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    q_len = np.full(B, Nq) if q_len is None else np.asarray(q_len)
    kv_len = np.full(B, Nkv) if kv_len is None else np.asarray(kv_len)
    q8 = np.zeros((B, H, Nq, D), np.int8)
    k8 = np.zeros((B, H, Nkv, D), np.int8)
    v8 = np.zeros((B, H, Nkv, D), np.uint8)
    qs = np.zeros((B, H, (Nq + BQS - 1) // BQS), F32)
    ks = np.zeros((B, H, (Nkv + BKS - 1) // BKS), F32)
    vs = np.zeros((B, H, D), F32)
    km = np.zeros((B, H, D), F32)
    for b in range(B):
        lq, lk = int(q_len[b]), int(kv_len[b])
        kf_all = k[b].astype(F32)
        means = k_channel_mean(kf_all, lk) if smooth_k else np.zeros((H, D), F32)
        for h in range(H):
            qf = q[b, h].astype(F32)
            vf = v[b, h].astype(F32)
            q8[b, h], qs[b, h] = quantize_int8_blocks(qf, lq, BQS)
            km[b, h] = means[h]
            ksm = (kf_all[h] - means[h][None, :]).astype(F32)
            k8[b, h], ks[b, h] = quantize_int8_blocks(ksm, lk, BKS)
            v8[b, h], vs[b, h] = quantize_v_fp8(vf, lk, s_v)
    return Prepared(q8, k8, v8, qs, ks, vs, km, q_len, kv_len, bkv)


# ---------------------------------------------------------------------------
# Attention: QK traversal, online softmax, FP8 P, two-level PV, final
# conversion  (Phase 0 stage list; Phase 1 strict tile order and per-tile RO
# rescale; Phase 2B checkpoints)
# ---------------------------------------------------------------------------
def qk_scores(q8: np.ndarray, k8: np.ndarray) -> np.ndarray:
    """Exact integer scores S[i, j] = sum_d q8[i, d] * k8[j, d] (R8), as int64.

    The float64 matrix product is exact here: every partial sum is an integer
    of magnitude <= 128 * 127 * 127 < 2^53.
    """
    s = q8.astype(np.float64) @ k8.astype(np.float64).T
    return s.astype(np.int64)


def score_factor_c(sm_scale: float) -> np.float32:
    """c = fp32(sm_scale * log2(e)), the product taken in float64 (R8)."""
    return F32(float(sm_scale) * (1.0 / math.log(2.0)))


@dataclass
class Checkpoints:
    """Per-tile stage values for the rows of one attention_rows call (Phase 2B list)."""
    m: list = field(default_factory=list)
    l: list = field(default_factory=list)
    alpha: list = field(default_factory=list)
    p8: list = field(default_factory=list)
    pv16: list = field(default_factory=list)
    ro: list = field(default_factory=list)
    recip: np.ndarray | None = None


def visible_keys(prep: Prepared, b: int, rows: np.ndarray, causal: bool) -> np.ndarray:
    """Number of keys [0, n) each query row sees (R14; R15 when causal)."""
    lk = int(prep.kv_len[b])
    rows = np.asarray(rows, dtype=np.int64)
    if not causal:
        return np.full(len(rows), lk, dtype=np.int64)
    lq = int(prep.q_len[b])
    return np.clip(rows + (lk - lq) + 1, 0, lk)


def attention_rows(prep: Prepared, b: int, h: int, rows: np.ndarray,
                   sm_scale: float | None = None, checkpoints: Checkpoints | None = None,
                   causal: bool = False):
    """Output rows of one (b, h) head: float32 values of the BF16 result.

    rows: query indices (all < q_len[b]).  Returns (out_bf16_bits uint16
    [len(rows), D], out float32 [len(rows), D]).  causal: R15 masking.
    """
    rows = np.asarray(rows, dtype=np.int64)
    D = prep.q8.shape[-1]
    nr = len(rows)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    c = score_factor_c(sm_scale)
    vis = visible_keys(prep, b, rows, causal)
    if nr == 0:
        return np.zeros((0, D), np.uint16), np.zeros((0, D), F32)
    if np.any(vis == 0):                          # R14/R15: rows that see no key are zero
        bits = np.zeros((nr, D), np.uint16)
        live = vis > 0
        if np.any(live):
            bits[live] = attention_rows(prep, b, h, rows[live], sm_scale, checkpoints, causal)[0]
        return bits, bf16_bits_to_f32(bits)
    lk = int(vis.max())                           # keys [lk, kv_len) are hidden from every row

    q_sc = prep.q_scale[b, h][rows // BQS]                      # [nr]
    S = qk_scores(prep.q8[b, h][rows], prep.k8[b, h][:lk])      # [nr, lk] exact ints
    v_dec = e4m3_decode(prep.v8[b, h][:lk])                     # [lk, D] float64

    m = np.full(nr, -np.inf, dtype=F32)
    l = np.zeros(nr, dtype=F32)
    ro = np.zeros((nr, D), dtype=F32)
    bkv = prep.bkv
    for j0 in range(0, lk, bkv):                                # strict ascending tile order
        j1 = min(j0 + bkv, lk)
        cols = np.arange(j0, j1)
        k_sc = prep.k_scale[b, h][cols // BKS]                  # [w]
        f = ((q_sc[:, None] * k_sc[None, :]).astype(F32) * c).astype(F32)
        s2 = (S[:, j0:j1].astype(F32) * f).astype(F32)          # exact int -> f32, one rounding
        s2 = np.where(cols[None, :] < vis[:, None], s2, F32(-np.inf)).astype(F32)   # R15 mask
        m_new = np.maximum(m, np.max(s2, axis=1)).astype(F32)
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isneginf(m), F32(0.0), exp2_f32((m - m_new).astype(F32))).astype(F32)
        p = exp2_f32((s2 - m_new[:, None]).astype(F32))        # [nr, w]
        tile_sum = np.zeros(nr, dtype=F32)
        for t in range(p.shape[1]):                             # ascending FP32 sum
            tile_sum = (tile_sum + p[:, t]).astype(F32)
        l = ((l * alpha).astype(F32) + tile_sum).astype(F32)
        p8 = e4m3_encode((p * F32(S_P)).astype(F32))
        pv = f16_round(e4m3_decode(p8) @ v_dec[j0:j1])          # exact, then one FP16 rounding
        ro = ((ro * alpha[:, None]).astype(F32) + pv.astype(F32)).astype(F32)
        m = m_new
        if checkpoints is not None:
            checkpoints.m.append(m.copy())
            checkpoints.l.append(l.copy())
            checkpoints.alpha.append(alpha.copy())
            checkpoints.p8.append(p8.copy())
            checkpoints.pv16.append(pv.copy())
            checkpoints.ro.append(ro.copy())
    r = (F32(1.0) / l).astype(F32)
    dq = (prep.v_scale[b, h] / F32(S_P)).astype(F32)            # [D]
    o = ((ro * r[:, None]).astype(F32) * dq[None, :]).astype(F32)
    bits = f32_to_bf16_bits(o)
    if checkpoints is not None:
        checkpoints.recip = r
    return bits, bf16_bits_to_f32(bits)


def attention(prep: Prepared, sm_scale: float | None = None, causal: bool = False):
    """Full output [B, H, Nq, D] as BF16 bits (uint16); rows >= q_len are 0."""
    B, H, Nq, D = prep.q8.shape
    out = np.zeros((B, H, Nq, D), dtype=np.uint16)
    for b in range(B):
        lq = int(prep.q_len[b])
        rows = np.arange(lq)
        for h in range(H):
            out[b, h, :lq] = attention_rows(prep, b, h, rows, sm_scale, causal=causal)[0]
    return out
