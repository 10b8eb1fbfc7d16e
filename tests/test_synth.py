"""CPU checks of the seeded input generator (eb_synth): its Philox against the published
known-answer vectors, its binary32 ln / sin / cos against numpy, its normals against the
normal law, and its bfloat16 rounding against torch's conversion."""
import os

import numpy as np
import scipy.stats
import torch

import eb_synth as S


def test_generator_philox_known_answers(golden_dir):
    with open(os.path.join(golden_dir, "philox4x32_10_kat.txt")) as f:
        rows = [[int(t, 16) for t in line.split()] for line in f
                if line.strip() and not line.startswith("#")]
    for r in rows:
        seed = r[4] | (r[5] << 32)
        out = S.philox(r[0], r[1], r[2], r[3], seed)
        assert [int(x) for x in out] == r[6:10]


def test_ln_and_sincos_accuracy():
    rng = np.random.default_rng(0)
    w = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    u = S.uniform(w)
    ref = np.log(u.astype(np.float64))
    assert np.max(np.abs(S._ln(u) - ref) / np.abs(ref)) < 5e-7
    c, s = S._sincos_2pi(u)
    th = 2 * np.pi * u.astype(np.float64)
    assert np.max(np.abs(c - np.cos(th))) < 3e-7
    assert np.max(np.abs(s - np.sin(th))) < 3e-7


def test_uniform_extremes_exact():
    assert S.uniform(np.uint32(0)) == np.float32(2.0 ** -24)
    assert S.uniform(np.uint32(0xFFFFFFFF)) == np.float32(1 - 2.0 ** -24)


def test_normals_follow_normal_law():
    n = S.normals(5, 0, np.arange(8), 3, 8192).ravel()
    stat, pval = scipy.stats.kstest(n, "norm")
    assert pval > 1e-3
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(100000) * 7).astype(np.float32)
    x[:5] = [0.0, -0.0, 1.0, 65504.0, 1e-30]
    ours = S.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == ref).all()


def test_workload_shapes_and_peaks():
    cfg = S.cfg0(0, L=8, V=64)
    x = cfg.logits(5)
    assert x.shape == (1, 8, 64) and x.dtype == np.float32
    t, u = S.position_params(0, 0, 8, 64)
    assert ((0 <= t) & (t < 64)).all()
    # the planted peak is sigma*n + (2 + 0.3*5) at t_p
    n = S.normals(0, 0, np.arange(8), 5, 64) * np.float32(3.0)
    h = np.float32(2.0) + np.float32(0.3) * np.float32(5)
    assert np.array_equal(x[0, np.arange(8), t], (n[np.arange(8), t] + h).astype(np.float32))
    m = S.cfg1_mask(0, L=256)
    assert m.shape == (1, 256) and m.sum() == 128
    c3 = S.cfg3(B=8, L=4, V=32)
    assert c3.growth == (0.1, 0.2, 0.4, 0.8, 0.1, 0.2, 0.4, 0.8) and c3.seeds == tuple(range(8))
    xb = c3.logits(2)
    assert xb.dtype == np.uint16 and xb.shape == (8, 4, 32)


def test_rows_subset_equals_full():
    cfg = S.cfg2(3, L=16, V=1000)
    full = cfg.logits(7)
    sub = cfg.rows(0, np.array([2, 9, 15]), 7)
    assert np.array_equal(full[0, [2, 9, 15]], sub)


def test_e4m3_rounding_matches_torch_inside_the_range():
    """Nearest-even rounding to e4m3 agrees with torch's float8_e4m3fn cast wherever no
    saturation is involved (|x| <= 448), subnormals included."""
    rng = np.random.default_rng(2)
    x = np.concatenate([(rng.standard_normal(200000) * 40).astype(np.float32),
                        (rng.standard_normal(50000) * 0.01).astype(np.float32),
                        np.float32([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 1.0625, 232.0])])
    x = x[np.abs(x) <= 448]
    ours = S.to_e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == ref).all()


def test_e4m3_rounding_by_brute_force_and_saturation():
    """Against the definition: the nearest finite e4m3 value, ties to the even code; above 448
    saturation; every finite code round-trips."""
    codes = np.arange(256, dtype=np.uint8)
    vals = S.e4m3_bits_to_f32(codes).astype(np.float64)
    finite = ~np.isnan(vals)
    assert np.array_equal(S.to_e4m3_bits(vals[finite].astype(np.float32))[vals[finite] != 0],
                          codes[finite][vals[finite] != 0])
    fc, fv = codes[finite], vals[finite]
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-0.05, 0.05, 20000)]).astype(np.float32)
    got = S.to_e4m3_bits(x)
    for xi, gi in zip(x[:4000].astype(np.float64), got[:4000]):
        d = np.abs(fv - xi)
        best = np.nonzero(d == d.min())[0]
        cand = fc[best]
        if len(cand) > 1:                      # a tie: the even mantissa, the same sign as x
            cand = [c for c in cand if (c & 1) == 0 and ((c >> 7) == (xi < 0) or (c & 0x7F) == 0)]
        assert gi in cand or (gi & 0x7F) == 0 and xi == 0
    sat = S.to_e4m3_bits(np.float32([449.0, 464.0, 1e6, np.inf, -500.0, -np.inf, np.nan]))
    assert sat.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]
