"""Seeded synthetic inputs for the EB sampler: logits of a stand-in denoiser.

This module holds none of the sampler's arithmetic.  It only produces inputs: logits
[B, L, V] with a Gaussian background and one planted peak per canvas position, the
initial mask of a single-step workload, and (for the fused unembedding workload) the
hidden states and unembedding matrix.  Both the CPU oracle (through the tests) and the
CUDA library (through ``eb_synth.device``) consume exactly the same values: the CUDA
generator in ``csrc/eb_synth.cu`` is bit-identical to the numpy one here, which a GPU
test checks.

Generator definition (every floating-point operation is one IEEE binary32 operation
with round-to-nearest-even, in the order written; no fused multiply-add):

* Philox4x32-10 (Salmon et al., SC'11), key = (low, high) 32 bits of the seed,
  counter = (v // 4, p, s, stream << 24 | b).  Streams: 2 = background normals,
  3 = per-position peak token / height, 4 = initial-mask ranking.
* uniform u(w) = ((w >> 9) + 1/2) * 2^-23, exact in binary32, in [2^-24, 1 - 2^-24].
* Box-Muller on the word pairs (w0, w1) -> entries 4k, 4k+1 and (w2, w3) -> 4k+2, 4k+3:
  n = sqrt(-2 ln u(w_even)) * (cos, sin)(2 pi u(w_odd)), with ln from the atanh series
  after a Cody-Waite ln 2 split, and sin / cos from Taylor series after an octant
  reduction (see ``_ln`` and ``_sincos_2pi``).
* per-position parameters from stream 3, counter (0, p, 0, 3 << 24 | b): peak token
  t_p = (w0 * V) >> 32, peak uniform u_p = u(w1).
* logit x[b, p, v] = sigma * n[b, p, v], plus h_p(s) at v == t_p, where
  h_p(s) = ((base_scale * u_p) + base_lo) + growth_b * s.
* bfloat16 outputs are rounded to nearest even from binary32.

Workloads (seeded, synthetic; shapes of a 256-position canvas and a 262144-entry
vocabulary):
  ``cfg0``  B=1, L=256, V=4096 fp32, sigma 3, peak 2 + 0.3 s, all positions masked.
  ``cfg1``  B=1, L=256, V=262144 bf16, sigma 2.5, peak U(0,12), 128 of 256 masked, s=0.
  ``cfg2``  B=1, L=256, V=262144 bf16, sigma 3, peak U(0,4) + 0.3 s.
  ``cfg3``  B=8, L=256, V=262144 bf16, sigma 3, peak U(0,4) + r_b s,
            r_b in (0.1, 0.2, 0.4, 0.8)[b % 4], canvas b keyed by seed b.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

STREAM_NORMAL = 2
STREAM_POSITION = 3
STREAM_MASK = 4
STREAM_UNEMBED_H = 5
STREAM_UNEMBED_COL = 6
STREAM_UNEMBED_W = 7

_F = np.float32
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox(c0, c1, c2, c3, seed: int):
    """Vectorised Philox4x32-10 over counter arrays (any broadcastable shapes)."""
    c0 = np.asarray(c0, np.uint64) & _MASK32
    c1 = np.asarray(c1, np.uint64) & _MASK32
    c2 = np.asarray(c2, np.uint64) & _MASK32
    c3 = np.asarray(c3, np.uint64) & _MASK32
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = seed & 0xFFFFFFFF
    k1 = (seed >> 32) & 0xFFFFFFFF
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
        p0 = _M0 * c0
        p1 = _M1 * c2
        n0 = (p1 >> np.uint64(32)) ^ c1 ^ np.uint64(k0)
        n1 = p1 & _MASK32
        n2 = (p0 >> np.uint64(32)) ^ c3 ^ np.uint64(k1)
        n3 = p0 & _MASK32
        c0, c1, c2, c3 = n0, n1, n2, n3
    return (c0.astype(np.uint32), c1.astype(np.uint32), c2.astype(np.uint32),
            c3.astype(np.uint32))


def uniform(w) -> np.ndarray:
    """u(w) = ((w >> 9) + 1/2) * 2^-23 in binary32 (exact)."""
    w = np.asarray(w, np.uint32)
    return ((w >> np.uint32(9)).astype(_F) + _F(0.5)) * _F(2.0 ** -23)


# binary32 constants of the ln / sin / cos series, given by bit pattern (they are the
# series coefficients 1/3, 1/5, ..., -1/6, 1/120, ... and sqrt(2), ln 2, pi/4 rounded to
# binary32; ln 2 is split Cody-Waite style into a 16-bit head and a tail)
def _f32bits(b: int) -> np.float32:
    return np.array([b], np.uint32).view(_F)[0]


_SQRT2 = _f32bits(0x3FB504F3)
_C3, _C5, _C7, _C9 = (_f32bits(0x3EAAAAAB), _f32bits(0x3E4CCCCD), _f32bits(0x3E124925),
                      _f32bits(0x3DE38E39))
_LN2_HI, _LN2_LO = _f32bits(0x3F317200), _f32bits(0x35BFBE8E)
_PI4 = _f32bits(0x3F490FDB)
_S3, _S5, _S7, _S9 = (_f32bits(0xBE2AAAAB), _f32bits(0x3C088889), _f32bits(0xB9500D01),
                      _f32bits(0x3638EF1D))
_K2, _K4, _K6, _K8, _K10 = (_f32bits(0xBF000000), _f32bits(0x3D2AAAAB), _f32bits(0xBAB60B61),
                            _f32bits(0x37D00D01), _f32bits(0xB493F27E))


def _ln(x: np.ndarray) -> np.ndarray:
    """Natural log of binary32 x in (0, 1): x = 2^e f with f in [sqrt(1/2), sqrt(2)),
    ln f = 2 atanh(s), s = (f - 1)/(f + 1), series to s^9; ln x = e ln2 + ln f."""
    x = np.asarray(x, _F)
    bits = x.view(np.uint32)
    e = ((bits >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int32) - 127
    f = ((bits & np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)).view(_F)
    big = f > _SQRT2
    f = np.where(big, f * _F(0.5), f).astype(_F)
    e = np.where(big, e + 1, e)
    s = (f - _F(1.0)) / (f + _F(1.0))
    z = s * s
    t = _C9 * z
    t = t + _C7
    t = t * z
    t = t + _C5
    t = t * z
    t = t + _C3
    a = s + s
    lnf = a + a * (z * t)
    ef = e.astype(_F)
    return ef * _LN2_HI + (ef * _LN2_LO + lnf)


def _sincos_2pi(u: np.ndarray):
    """(cos, sin)(2 pi u) for binary32 u in (0, 1): octant o = floor(8u), reduced angle
    phi * pi/4 with phi = frac(8u) (even o) or 1 - frac(8u) (odd o), Taylor series."""
    u = np.asarray(u, _F)
    t = u * _F(8.0)
    o = t.astype(np.int32)
    f = t - o.astype(_F)
    odd = (o & 1) == 1
    phi = np.where(odd, _F(1.0) - f, f).astype(_F)
    a = phi * _PI4
    a2 = a * a
    q = _S9 * a2
    q = q + _S7
    q = q * a2
    q = q + _S5
    q = q * a2
    q = q + _S3
    q = q * a2
    sn = a + a * q
    c = _K10 * a2
    c = c + _K8
    c = c * a2
    c = c + _K6
    c = c * a2
    c = c + _K4
    c = c * a2
    c = c + _K2
    c = c * a2
    cs = _F(1.0) + c
    # octant table: (cos, sin) of 2 pi u in terms of (cs, sn) = (cos, sin)(phi pi/4)
    swap = (o == 1) | (o == 2) | (o == 5) | (o == 6)
    cos_mag = np.where(swap, sn, cs)
    sin_mag = np.where(swap, cs, sn)
    cos_neg = (o >= 2) & (o <= 5)
    sin_neg = o >= 4
    cosv = np.where(cos_neg, -cos_mag, cos_mag).astype(_F)
    sinv = np.where(sin_neg, -sin_mag, sin_mag).astype(_F)
    return cosv, sinv


def normals(seed: int, b: int, p, s: int, V: int) -> np.ndarray:
    """Background normals n[b, p, v] for the given positions p (array), shape [len(p), V]."""
    return _normal_rows(seed, p, s, (STREAM_NORMAL << 24) | b, V)


def _normal_rows(seed: int, rows, c2: int, c3: int, cols: int) -> np.ndarray:
    """Box-Muller normals of counters (k, row, c2, c3), k = column // 4: [len(rows), cols]."""
    p = np.atleast_1d(np.asarray(rows, np.int64))
    V = cols
    nk = (V + 3) // 4
    k = np.arange(nk, dtype=np.uint64)[None, :]
    pc = p.astype(np.uint64)[:, None]
    w0, w1, w2, w3 = philox(k, pc, np.uint64(c2), np.uint64(c3), seed)
    r0 = np.sqrt(_ln(uniform(w0)) * _F(-2.0))
    r1 = np.sqrt(_ln(uniform(w2)) * _F(-2.0))
    c0, s0 = _sincos_2pi(uniform(w1))
    c1, s1 = _sincos_2pi(uniform(w3))
    out = np.empty((p.shape[0], nk, 4), _F)
    out[:, :, 0] = r0 * c0
    out[:, :, 1] = r0 * s0
    out[:, :, 2] = r1 * c1
    out[:, :, 3] = r1 * s1
    return out.reshape(p.shape[0], nk * 4)[:, :V]


def position_params(seed: int, b: int, L: int, V: int):
    """(t_p int64 [L], u_p float32 [L]): peak token and peak-height uniform."""
    p = np.arange(L, dtype=np.uint64)
    w0, w1, _, _ = philox(np.uint64(0), p, np.uint64(0), np.uint64((STREAM_POSITION << 24) | b), seed)
    t = ((w0.astype(np.uint64) * np.uint64(V)) >> np.uint64(32)).astype(np.int64)
    return t, uniform(w1)


def initial_mask(seed: int, b: int, L: int, n_masked: int) -> np.ndarray:
    """u8 [L]: the n_masked positions with the smallest stream-4 words (ties: lower p)."""
    p = np.arange(L, dtype=np.uint64)
    w0, _, _, _ = philox(np.uint64(0), p, np.uint64(0), np.uint64((STREAM_MASK << 24) | b), seed)
    order = np.lexsort((np.arange(L), w0))
    m = np.zeros(L, np.uint8)
    m[order[:n_masked]] = 1
    return m


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 to bfloat16 (nearest even), returned as uint16 bit patterns."""
    bits = np.ascontiguousarray(x, _F).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return ((bits + bias) >> np.uint32(16)).astype(np.uint16)


def to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 to OCP FP8 e4m3 (nearest, ties to even; magnitudes above the largest
    finite value 448 saturate to it; NaN stays NaN), returned as uint8 codes.  Normal codes
    hold (1 + m/8) 2^(e-7) for exponent field e in 1..15 (m < 7 when e = 15); subnormal codes
    m/8 2^-6, so below 2^-6 the grid is 2^-9."""
    x = np.ascontiguousarray(x, _F)
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    a = np.abs(x).astype(np.float64)                       # exact
    a = np.where(np.isfinite(a), a, 1e6)                   # inf / NaN: fixed up below
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # correct log2's rounding at exact powers of two
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= a, e + 1, e)
    e = np.maximum(e, -6.0)                                  # the subnormal grid below 2^-6
    q = np.rint(np.ldexp(a, (3 - e).astype(np.int64)))       # 8..16 (normal) or 0..8 (subnormal)
    e = np.where(q >= 16, e + 1, e)
    q = np.where(q >= 16, q / 2, q)
    normal = q >= 8
    code = np.where(normal, ((e + 7) * 8 + (q - 8)), q)
    code = np.where(a > 448.0, 0x7E, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return (code.astype(np.uint8) | np.where(np.isnan(x), np.uint8(0), sign)).astype(np.uint8)


def e4m3_bits_to_f32(c: np.ndarray) -> np.ndarray:
    """Exact binary32 values of e4m3 codes (NaN for S.1111.111)."""
    c = np.asarray(c, np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e, m = (c >> 3) & 15, c & 7
    v = np.where(e == 0, np.ldexp(m.astype(np.float64), -9), np.ldexp((8 + m).astype(np.float64), e - 10))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return (s * v).astype(_F)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(_F)


@dataclass(frozen=True)
class Peaked:
    """Recipe of a peaked-logit workload (see the module docstring)."""
    B: int
    L: int
    V: int
    dtype: str            # "f32", "bf16" or "fp8" (e4m3)
    sigma: float
    base_lo: float
    base_scale: float
    growth: tuple         # per canvas b (length B)
    seeds: tuple          # per canvas b (length B)

    def peak_height(self, b: int, u_p: np.ndarray, s: int) -> np.ndarray:
        h = _F(self.base_scale) * u_p
        h = h + _F(self.base_lo)
        g = _F(self.growth[b]) * _F(s)
        return (h + g).astype(_F)

    def rows(self, b: int, p, s: int) -> np.ndarray:
        """Logits of canvas b, positions p (array), step s -> [len(p), V] (f32 or bf16 bits)."""
        p = np.atleast_1d(np.asarray(p, np.int64))
        seed = int(self.seeds[b])
        n = normals(seed, b, p, s, self.V)
        x = (n * _F(self.sigma)).astype(_F)
        t, u = position_params(seed, b, self.L, self.V)
        h = self.peak_height(b, u, s)
        idx = np.arange(p.shape[0])
        x[idx, t[p]] = x[idx, t[p]] + h[p]
        if self.dtype == "bf16":
            return to_bf16_bits(x)
        return to_e4m3_bits(x) if self.dtype == "fp8" else x

    def logits(self, s: int, rows_per_chunk: int = 16) -> np.ndarray:
        """Full logits [B, L, V] at step s."""
        dt = {"bf16": np.uint16, "fp8": np.uint8}.get(self.dtype, _F)
        out = np.empty((self.B, self.L, self.V), dt)
        for b in range(self.B):
            for p0 in range(0, self.L, rows_per_chunk):
                p = np.arange(p0, min(self.L, p0 + rows_per_chunk))
                out[b, p0:p0 + p.shape[0]] = self.rows(b, p, s)
        return out


def cfg0(seed: int = 0, L: int = 256, V: int = 4096) -> Peaked:
    return Peaked(1, L, V, "f32", 3.0, 2.0, 0.0, (0.3,), (seed,))


def cfg1(seed: int = 0, L: int = 256, V: int = 262144) -> Peaked:
    return Peaked(1, L, V, "bf16", 2.5, 0.0, 12.0, (0.0,), (seed,))


def cfg1_mask(seed: int = 0, L: int = 256) -> np.ndarray:
    """Initial mask [1, L] of the single-step workload: a random half of the positions."""
    return initial_mask(seed, 0, L, L // 2)[None, :]


def cfg2(seed: int = 0, L: int = 256, V: int = 262144) -> Peaked:
    return Peaked(1, L, V, "bf16", 3.0, 0.0, 4.0, (0.3,), (seed,))


def cfg_stop(seed: int = 7, L: int = 256, V: int = 262144) -> Peaked:
    """The early-stop loop: one canvas whose peaks (sigma 1, U(12, 14) + 0.5 s) soon dominate,
    so that the mean entropy falls below the stop threshold while positions are still masked
    and the adaptive stop ends the loop (after 9 of at most 48 steps for seed 7)."""
    return Peaked(1, L, V, "bf16", 1.0, 12.0, 2.0, (0.5,), (seed,))


CFG3_RATES = (0.1, 0.2, 0.4, 0.8)


def cfg3(B: int = 8, L: int = 256, V: int = 262144) -> Peaked:
    return Peaked(B, L, V, "bf16", 3.0, 0.0, 4.0,
                  tuple(CFG3_RATES[b % 4] for b in range(B)), tuple(range(B)))


# ------------------------------------------------------------------ fused unembedding inputs

def unembed_h_rows(seed: int, rows, K: int) -> np.ndarray:
    """Hidden states h[m, :] = N(0,1) for rows m (array) as bf16 bits [len(rows), K];
    counters (j // 4, m, 0, 5 << 24)."""
    n = _normal_rows(seed, rows, 0, STREAM_UNEMBED_H << 24, K)
    return to_bf16_bits((n * _F(1.0)).astype(_F))


def unembed_bias_columns(seed: int, rows, V: int) -> np.ndarray:
    """Column c_k = (w0 * V) >> 32 of counter (0, k, 0, 6 << 24) that carries row k's bias."""
    rows = np.atleast_1d(np.asarray(rows, np.uint64))
    w0, _, _, _ = philox(np.uint64(0), rows, np.uint64(0), np.uint64(STREAM_UNEMBED_COL << 24), seed)
    return ((w0.astype(np.uint64) * np.uint64(V)) >> np.uint64(32)).astype(np.int64)


def unembed_W_rows(seed: int, rows, V: int, sigma_w: float = 0.02, bias: float = 0.05) -> np.ndarray:
    """Unembedding rows W[k, :] = sigma_w N(0,1) plus `bias` at column c_k, for rows k (array),
    as bf16 bits [len(rows), V]; counters (v // 4, k, 0, 7 << 24)."""
    rows = np.atleast_1d(np.asarray(rows, np.int64))
    x = (_normal_rows(seed, rows, 0, STREAM_UNEMBED_W << 24, V) * _F(sigma_w)).astype(_F)
    c = unembed_bias_columns(seed, rows, V)
    idx = np.arange(rows.shape[0])
    x[idx, c] = (x[idx, c] + _F(bias)).astype(_F)
    return to_bf16_bits(x)


@dataclass(frozen=True)
class Unembed:
    """Recipe of the fused unembedding workload: h [B*L, K] ~ N(0,1), W [K, V] ~
    N(0, sigma_w^2) with +bias planted at one seeded column per row of W, both bf16."""
    B: int
    L: int
    K: int
    V: int
    seed: int = 0
    sigma_w: float = 0.02
    bias: float = 0.05

    @property
    def M(self) -> int:
        return self.B * self.L

    def h(self) -> np.ndarray:
        return unembed_h_rows(self.seed, np.arange(self.M), self.K)

    def W(self, rows_per_chunk: int = 64) -> np.ndarray:
        out = np.empty((self.K, self.V), np.uint16)
        for k0 in range(0, self.K, rows_per_chunk):
            k = np.arange(k0, min(self.K, k0 + rows_per_chunk))
            out[k0:k0 + k.shape[0]] = unembed_W_rows(self.seed, k, self.V, self.sigma_w, self.bias)
        return out


def cfg4(B: int = 4, L: int = 256, K: int = 2048, V: int = 262144, seed: int = 0) -> Unembed:
    return Unembed(B, L, K, V, seed)
