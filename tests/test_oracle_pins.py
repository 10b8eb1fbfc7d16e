"""Pins of the CPU oracle against facts that do not come from the oracle itself:
published known-answer vectors, closed forms, library routines, brute force and
hand-built cases of the sampler rules (DiffusionGemma model card, "Best practices"
section 1, "Diffusion sampling settings").  CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from eb_synth import to_bf16_bits


# ---------------------------------------------------------------- Philox4x32-10

def test_philox_known_answers(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(t, 16) for t in line.split()])
    assert len(rows) == 3
    for r in rows:
        out = oracle.philox4x32_10(r[0:4], r[4:6])
        assert [int(x) for x in out] == r[6:10]


def test_philox_is_a_bijection_of_the_counter_on_a_sample():
    # distinct counters under one key give distinct 128-bit outputs (Philox is a bijection)
    seen = set()
    for c in range(2000):
        seen.add(tuple(int(x) for x in oracle.philox4x32_10([c, 7, 0, 1 << 24], [5, 0])))
    assert len(seen) == 2000


# ---------------------------------------------------------------- uniforms / Gumbel

def test_uniform_range_and_resolution():
    assert oracle.uniform(0) == 0.5 / 2 ** 23
    assert oracle.uniform(0x7FFFFF) == 1.0 - 0.5 / 2 ** 23
    assert oracle.uniform(0xFF800000) == 0.5 / 2 ** 23   # only the low 23 bits count
    assert 0.0 < oracle.uniform(0x12345678) < 1.0


def test_gumbel_noise_distribution_ks():
    # the per-entry noise the sampler draws is standard Gumbel (scipy's gumbel_r)
    g = np.array([oracle.gumbel(oracle.gumbel_word(3, 0, p, 0, v))
                  for p in range(40) for v in range(500)])
    stat, pval = scipy.stats.kstest(g, "gumbel_r")
    assert pval > 1e-3, (stat, pval)


# ---------------------------------------------------------------- temperature

def test_temperature_schedule_endpoints_and_linearity():
    assert oracle.temperature(0) == pytest.approx(0.8, abs=1e-15)
    assert oracle.temperature(47) == pytest.approx(0.4, abs=1e-15)
    d = [oracle.temperature(s + 1) - oracle.temperature(s) for s in range(47)]
    assert np.allclose(d, -0.4 / 47, atol=1e-15)
    assert oracle.temperature(5, max_steps=1) == 0.8


# ---------------------------------------------------------------- entropy closed forms

@pytest.mark.parametrize("V,expected", [(8, 2.0794415416798357), (4096, 8.317766166719343),
                                        (262144, 12.476649250079015)])
def test_uniform_logits_entropy_is_ln_V(V, expected):
    assert expected == pytest.approx(math.log(V), abs=1e-15)
    x = np.zeros(V, np.float32)
    H, A, Y, gap = oracle.row(x, 0.8, True, seed=1)
    assert H == pytest.approx(expected, abs=1e-9)
    assert A == 0                      # first index on equality
    assert 0 <= Y < V
    xb = to_bf16_bits(np.full(V, 1.5, np.float32))
    H2, A2, _, _ = oracle.row(xb, 0.8, False)
    assert H2 == pytest.approx(expected, abs=1e-9) and A2 == 0


def test_dominant_peak_entropy_zero_and_sample_is_peak():
    V = 4096
    rng = np.random.default_rng(0)
    x = rng.standard_normal(V).astype(np.float32)
    x[1234] = 1.0e4
    xb = to_bf16_bits(x)
    assert np.asarray(xb[1234]).astype(np.uint32) << 16 == np.float32(9984.0).view(np.uint32)
    for arr in (x, xb):
        H, A, Y, gap = oracle.row(arr, 0.8, True, seed=2, p=3)
        assert H < 1e-12 and A == 1234 and Y == 1234


@pytest.mark.parametrize("k", [1, 2, 3, 7])
def test_k_equal_top_logits_rest_minus_inf(k):
    V = 64
    x = np.full(V, -np.inf, np.float32)
    top = [5, 17, 18, 40, 41, 50, 63][:k]
    x[top] = 2.0
    H, A, Y, gap = oracle.row(x, 0.6, True, seed=9, p=1)
    assert H == pytest.approx(math.log(k), abs=1e-12)
    assert A == top[0]
    assert Y in top


@pytest.mark.parametrize("d,T", [(0.0, 0.8), (1.0, 0.8), (3.0, 0.4), (-2.5, 0.55)])
def test_two_logit_binary_entropy(d, T):
    x = np.array([0.0, d], np.float64)
    q = 1.0 / (1.0 + math.exp(-d / T))
    expected = -(q * math.log(q) + (1 - q) * math.log(1 - q))
    H, A, _, _ = oracle.row(x, T, False)
    assert H == pytest.approx(expected, abs=1e-13)
    assert A == (1 if d > 0 else 0)


def test_entropy_matches_scipy_on_random_rows():
    rng = np.random.default_rng(5)
    for V, T in [(100, 0.8), (4096, 0.4), (5000, 0.63)]:
        x = (3.0 * rng.standard_normal(V)).astype(np.float64)
        H, A, _, _ = oracle.row(x, T, False)
        expected = scipy.stats.entropy(scipy.special.softmax(x / T))
        assert H == pytest.approx(expected, abs=1e-10)
        assert A == int(np.argmax(x))


def test_shift_invariance():
    rng = np.random.default_rng(6)
    x = np.round(rng.standard_normal(1000) * 64) / 64          # exact in binary64 after +c
    H0, A0, Y0, _ = oracle.row(x, 0.8, True, seed=4, p=7, s=3)
    H1, A1, Y1, _ = oracle.row(x + 96.0, 0.8, True, seed=4, p=7, s=3)
    assert H1 == pytest.approx(H0, abs=1e-12)
    assert (A0, Y0) == (A1, Y1)


def test_argmax_first_index_on_ties():
    x = np.array([1.0, 3.0, 2.0, 3.0, 3.0], np.float32)
    _, A, _, _ = oracle.row(x, 0.8, False)
    assert A == 1


# ---------------------------------------------------------------- Gumbel-max sampling

def test_gumbel_max_frequencies_chi_square():
    # V=8 fixed logits, 2^20 independent draws (distinct (b, p, s) counters); the
    # sampled-token frequencies must follow softmax(x / T).
    V, T = 8, 0.7
    x = np.array([0.3, -1.0, 1.2, 0.0, 2.0, -0.5, 0.9, 1.5], np.float64)
    B, L = 64, 4096
    logits = np.broadcast_to(x, (B, L, V)).copy()
    counts = np.zeros(V, np.int64)
    for s in range(4):
        st = oracle.State.fresh(B, L)
        res = oracle.step(logits, st, s, oracle.Params(max_steps=48, seed=11), temperature=T)
        counts += np.bincount(res.Y.ravel(), minlength=V)
    p = scipy.special.softmax(x / T)
    chi2, pval = scipy.stats.chisquare(counts, counts.sum() * p)
    assert pval > 1e-3, (chi2, pval, counts)


def test_low_temperature_sample_is_argmax():
    rng = np.random.default_rng(8)
    x = rng.standard_normal(512).astype(np.float64)
    H, A, Y, _ = oracle.row(x, 1e-4, True, seed=1, p=2)
    assert Y == A


def test_unmasked_rows_do_not_sample():
    H, A, Y, gap = oracle.row(np.zeros(16, np.float32), 0.8, False)
    assert Y == -1 and math.isinf(gap)


# ---------------------------------------------------------------- selection

def _brute_force_max_subset(H, mask, bound):
    """Largest subset S of the masked positions with sum(H_S) - max(H_S) <= bound."""
    idx = [p for p in range(len(H)) if mask[p]]
    best = 0
    for r in range(1, len(idx) + 1):
        for sub in itertools.combinations(idx, r):
            hs = [H[p] for p in sub]
            if sum(hs) - max(hs) <= bound:
                best = max(best, r)
    return best


def test_selection_brute_force_V8_L4_all_masks():
    # canvases of L=4 positions over V=8, entropies from real rows (oracle.row), every
    # mask pattern: the prefix rule accepts as many positions as the best subset, and
    # exactly the k lowest-entropy masked positions.
    rng = np.random.default_rng(12)
    bound = 0.1
    for trial in range(60):
        scale = rng.choice([0.5, 2.0, 6.0, 12.0])
        H = []
        for p in range(4):
            x = np.zeros(8)
            x[rng.integers(8)] = scale * rng.uniform(0.5, 1.5)
            x += rng.standard_normal(8) * 0.5
            H.append(oracle.row(x, 0.8, False)[0])
        H = np.array(H)
        for bits in range(16):
            mask = np.array([(bits >> p) & 1 for p in range(4)], np.uint8)
            acc, k, _, _ = oracle.select(H, mask, bound)
            n = int(mask.sum())
            if n == 0:
                assert k == 0 and acc.sum() == 0
                continue
            assert k >= 1
            assert k == _brute_force_max_subset(H, mask, bound)
            masked = [p for p in range(4) if mask[p]]
            lowest = sorted(masked, key=lambda p: (H[p], p))[:k]
            assert sorted(np.nonzero(acc)[0].tolist()) == sorted(lowest)


def test_selection_hand_cases():
    H = np.array([0.05, 0.04, 0.3, 0.01, 0.02])
    acc, k, smargin, omargin = oracle.select(H, np.ones(5, np.uint8), 0.1)
    # sorted: 0.01(p3) 0.02(p4) 0.04(p1) 0.05(p0) 0.3(p2); sums before: 0 .01 .03 .07 .12
    assert k == 4 and acc.tolist() == [1, 1, 0, 1, 1]
    assert smargin == pytest.approx(0.02, abs=1e-15)
    assert omargin == pytest.approx(0.25, abs=1e-15)
    # a single huge entropy is still accepted (at least one position per step)
    acc, k, _, _ = oracle.select(np.array([9.0, 8.0, 7.0]), np.ones(3, np.uint8), 0.1)
    assert k == 1 and acc.tolist() == [0, 0, 1]
    # equal entropies: lower position first
    acc, k, _, _ = oracle.select(np.array([1.0, 1.0, 1.0]), np.ones(3, np.uint8), 0.1)
    assert acc.tolist() == [1, 0, 0]
    # unmasked positions never selected, bound inclusive (sum 0.0625 + 0.03125 <= 0.09375)
    acc, k, _, _ = oracle.select(np.array([0.0, 0.0625, 0.03125, 0.5]), np.array([0, 1, 1, 1], np.uint8),
                                 0.09375)
    assert acc.tolist() == [0, 1, 1, 1]


# ---------------------------------------------------------------- stop / finalize

def _peaked(B, L, V, tokens, height=40.0):
    x = np.zeros((B, L, V), np.float32)
    for b in range(B):
        for p in range(L):
            x[b, p, tokens[b][p]] = height
    return x


def test_no_stop_at_step_zero_then_adaptive_stop_at_step_one():
    B, L, V = 1, 16, 32
    toks = [[(3 * p + 1) % V for p in range(L)]]
    x = _peaked(B, L, V, toks)
    st = oracle.State.fresh(B, L)
    prm = oracle.Params(entropy_bound=-1.0)       # accept exactly one position per step
    r0 = oracle.step(x, st, 0, prm)
    assert st.status[0] == oracle.RUNNING and r0.committed[0] == 1
    assert r0.mean_entropy[0] < 0.005
    r1 = oracle.step(x, st, 1, prm)
    assert st.status[0] == oracle.ADAPTIVE and st.steps_taken[0] == 2
    assert r1.committed[0] == L - 1
    assert st.tokens[0].tolist() == toks[0] and st.mask.sum() == 0


def test_argmax_flip_blocks_stop():
    B, L, V = 1, 8, 16
    toks = [[p for p in range(L)]]
    st = oracle.State.fresh(B, L)
    prm = oracle.Params(entropy_bound=-1.0)
    oracle.step(_peaked(B, L, V, toks), st, 0, prm)
    toks2 = [list(toks[0])]
    toks2[0][5] = 15
    oracle.step(_peaked(B, L, V, toks2), st, 1, prm)
    assert st.status[0] == oracle.RUNNING
    oracle.step(_peaked(B, L, V, toks2), st, 2, prm)
    assert st.status[0] == oracle.ADAPTIVE and st.steps_taken[0] == 3


def test_stop_threshold_is_strict():
    B, L, V = 1, 8, 16
    rng = np.random.default_rng(3)
    x = _peaked(B, L, V, [[p for p in range(L)]], height=6.0) + \
        rng.standard_normal((B, L, V)).astype(np.float32) * 0.1
    x[0, :, :] = x[0, 0, :]        # all rows equal
    probe = oracle.State.fresh(B, L)
    r = oracle.step(x, probe, 1, oracle.Params(stop_entropy=0.0))
    mean = float(r.mean_entropy[0])
    assert 0 < mean
    for thr, expect in [(mean, oracle.RUNNING), (np.nextafter(mean, 1.0), oracle.ADAPTIVE)]:
        st = oracle.State.fresh(B, L)
        st.prev_argmax[:] = r.A
        oracle.step(x, st, 1, oracle.Params(stop_entropy=float(thr), entropy_bound=-1.0))
        assert st.status[0] == expect


def test_cap_finalizes_with_argmax():
    B, L, V = 1, 6, 10
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((B, L, V)) * 4).astype(np.float32)
    st = oracle.State.fresh(B, L)
    prm = oracle.Params(max_steps=3, entropy_bound=-1.0)
    for s in range(3):
        r = oracle.step(x + np.float32(s), st, s, prm)
    assert st.status[0] == oracle.CAP and st.steps_taken[0] == 3
    assert st.mask.sum() == 0
    fin = r.selected[0].astype(bool)
    assert fin.sum() == L - 2
    assert (st.tokens[0][fin] == r.A[0][fin]).all()


def test_complete_when_mask_empties():
    B, L, V = 2, 5, 12
    x = _peaked(B, L, V, [[1, 2, 3, 4, 5], [6, 7, 8, 9, 10]])
    st = oracle.State.fresh(B, L)
    st.mask[1, :] = 0
    st.tokens[1, :] = 0
    st.status[1] = oracle.COMPLETE
    r = oracle.step(x, st, 0, oracle.Params())
    assert st.status.tolist() == [oracle.COMPLETE, oracle.COMPLETE]
    assert st.steps_taken[0] == 1 and r.committed[0] == L
    assert st.tokens[0].tolist() == [1, 2, 3, 4, 5]
    assert np.isnan(r.H[1]).all()       # stopped canvases are not touched


def test_unselected_positions_are_remasked():
    B, L, V = 1, 10, 50
    rng = np.random.default_rng(10)
    x = (rng.standard_normal((B, L, V)) * 2).astype(np.float32)
    st = oracle.State.fresh(B, L)
    r = oracle.step(x, st, 0, oracle.Params())
    assert r.committed[0] == 1
    sel = r.selected[0].astype(bool)
    assert (st.tokens[0][~sel] == -1).all() and (st.mask[0][~sel] == 1).all()
    assert (st.tokens[0][sel] == r.Y[0][sel]).all()


# ---------------------------------------------------------------- unembedding product

def test_unembed_logits_one_hot_rows_and_brute_force():
    from eb_synth import to_bf16_bits
    rng = np.random.default_rng(21)
    K, V = 24, 40
    W = to_bf16_bits(rng.standard_normal((K, V)).astype(np.float32) * 0.5)
    Wf = oracle.bf16_to_f64(W)
    # a one-hot hidden state selects one row of W exactly
    h = np.zeros((3, K), np.float32)
    h[0, 5] = 1.0
    h[1, 0] = 1.0
    h[2, K - 1] = -2.0
    out = oracle.unembed_logits(to_bf16_bits(h), W)
    assert np.array_equal(out[0], Wf[5]) and np.array_equal(out[1], Wf[0])
    assert np.array_equal(out[2], -2.0 * Wf[K - 1])
    # brute-force triple loop on random bf16 inputs
    hb = to_bf16_bits(rng.standard_normal((4, K)).astype(np.float32))
    hf = oracle.bf16_to_f64(hb)
    got = oracle.unembed_logits(hb, W)
    for m in range(4):
        for v in range(V):
            ref = 0.0
            for k in range(K):
                ref += hf[m, k] * Wf[k, v]
            assert abs(got[m, v] - ref) <= 1e-12 * (1 + abs(ref))


def test_bf16_to_f64_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F7F], np.uint16)
    vals = oracle.bf16_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[2] == 0.0
    assert vals[3] == 3.140625 and vals[4] == float(np.float32(3.3895313892515355e38))


# ---------------------------------------------------------------- reading variants (flags)

def test_masked_only_stop_statistics_ignore_committed_positions():
    """STOP_MASKED_ONLY: the mean entropy and the argmax-stability test run over the positions
    still masked.  Committed positions with uniform rows (H = ln 16) and a changed argmax block
    the default stop but not the variant."""
    B, L, V = 1, 8, 16
    x = _peaked(B, L, V, [[p + 8 for p in range(L)]])
    x[0, :4, :] = 0.0                                # committed positions: uniform, H = ln 16
    st0 = oracle.State.fresh(B, L)
    st0.mask[0, :4] = 0
    st0.tokens[0, :4] = 3
    st0.prev_argmax[0, :] = [5, 5, 5, 5, 12, 13, 14, 15]   # A = 0 at the uniform rows
    runs = {}
    for flags in (0, oracle.STOP_MASKED_ONLY):
        st = st0.copy()
        r = oracle.step(x, st, 1, oracle.Params(flags=flags, entropy_bound=-1.0))
        runs[flags] = (st, r)
    st, r = runs[0]
    assert st.status[0] == oracle.RUNNING
    assert r.mean_entropy[0] == pytest.approx(4 * np.log(16) / 8, rel=1e-12)
    st, r = runs[oracle.STOP_MASKED_ONLY]
    assert st.status[0] == oracle.ADAPTIVE and st.steps_taken[0] == 2
    assert r.mean_entropy[0] < 1e-12
    assert st.tokens[0].tolist() == [3, 3, 3, 3, 12, 13, 14, 15]


def test_finalize_sampled_takes_the_sampled_token_at_stop_and_cap():
    """FINALIZE_SAMPLED: positions finalised by the adaptive stop or the step cap take Y, the
    Gumbel-max sample, instead of the argmax A."""
    B, L, V = 1, 12, 10
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((B, L, V)) * 0.5).astype(np.float32)
    # adaptive stop at step 1 (threshold above every mean, argmax stable)
    for flags, key in ((0, "A"), (oracle.FINALIZE_SAMPLED, "Y")):
        probe = oracle.State.fresh(B, L)
        r0 = oracle.step(x, probe, 1, oracle.Params(stop_entropy=0.0))
        st = oracle.State.fresh(B, L)
        st.prev_argmax[:] = r0.A
        r = oracle.step(x, st, 1, oracle.Params(stop_entropy=100.0, flags=flags))
        assert st.status[0] == oracle.ADAPTIVE
        assert (st.tokens == getattr(r, key)).all()
        assert (r.Y != r.A).sum() >= 3          # the two readings differ here
    # cap after three one-position steps
    for flags, key in ((0, "A"), (oracle.FINALIZE_SAMPLED, "Y")):
        st = oracle.State.fresh(B, L)
        prm = oracle.Params(max_steps=3, entropy_bound=-1.0, flags=flags)
        for s in range(3):
            r = oracle.step(x + np.float32(s), st, s, prm)
        assert st.status[0] == oracle.CAP
        fin = r.selected[0].astype(bool)
        assert fin.sum() == L - 2
        assert (st.tokens[0][fin] == getattr(r, key)[0][fin]).all()
        assert (r.Y[0][fin] != r.A[0][fin]).sum() >= 3


# ---------------------------------------------------------------- block driver

def test_blocks_run_alone_equal_the_batch_loop():
    """Block k run on its own with Philox canvas id k reproduces canvas k of the loop over all
    blocks at once, and the id is what makes it so: the same block under id 0 samples
    differently."""
    import eb_synth
    cfg = eb_synth.Peaked(3, 16, 256, "f32", 3.0, 0.0, 4.0, (0.4, 0.8, 0.2), (7, 8, 9))
    op = oracle.Params(seed=2)
    st = oracle.run_loop(lambda s, _st: cfg.logits(s), 3, 16, op)
    tok, steps, status = oracle.run_blocks(lambda k, s: cfg.logits(s)[k], 3, 16, op)
    assert np.array_equal(tok, st.tokens)
    assert np.array_equal(steps, st.steps_taken) and np.array_equal(status, st.status)
    x = cfg.logits(0)[1:2]
    r_own = oracle.step(x, oracle.State.fresh(1, 16), 0, op, canvas_ids=[1])
    r_zero = oracle.step(x, oracle.State.fresh(1, 16), 0, op, canvas_ids=[0])
    r_batch = oracle.step(cfg.logits(0)[:2], oracle.State.fresh(2, 16), 0, op)
    assert np.array_equal(r_own.Y[0], r_batch.Y[1])
    assert (r_own.Y[0] != r_zero.Y[0]).sum() >= 4


# ---------------------------------------------------------------- e4m3 logits

def test_e4m3_decoding_known_values():
    """OCP FP8 e4m3: bias 7, 3 mantissa bits, subnormals below 2^-6, no infinities,
    S.1111.111 is NaN."""
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0,
             0xFE: -448.0}
    for code, value in known.items():
        assert oracle.e4m3_value(code) == value, hex(code)
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) == -1.0


def test_e4m3_row_equals_its_decoded_values():
    """A row of e4m3 codes gives exactly the statistics of the binary64 values they encode."""
    from eb_synth import e4m3_bits_to_f32
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, 4096).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                     # no NaN in this row
    a = oracle.row(codes, 0.8, True, 3, 0, 7, 2)
    b = oracle.row(e4m3_bits_to_f32(codes).astype(np.float64), 0.8, True, 3, 0, 7, 2)
    assert a[0] == b[0] and a[1] == b[1] and a[2] == b[2]


def test_raw_entropy_stop_statistic():
    """STOP_RAW_ENTROPY: the stop rule averages the entropy of the raw logits (T = 1).  A peak of
    9 over 15 zeros has a raw entropy of about 0.019 nats but a shaped one (T = 0.79 at step 1)
    of about 0.002, so the default stops and the variant does not; selection is unchanged."""
    B, L, V = 1, 8, 16
    x = _peaked(B, L, V, [[p + 1 for p in range(L)]], height=9.0)
    raw_h = oracle.row(x[0, 0], 1.0, False)[0]
    shaped_h = oracle.row(x[0, 0], oracle.temperature(1), False)[0]
    assert shaped_h < 0.005 < raw_h
    for flags, expect in ((0, oracle.ADAPTIVE), (oracle.STOP_RAW_ENTROPY, oracle.RUNNING)):
        st = oracle.State.fresh(B, L)
        st.prev_argmax[:] = [[p + 1 for p in range(L)]]
        r = oracle.step(x, st, 1, oracle.Params(flags=flags, entropy_bound=-1.0))
        assert st.status[0] == expect
        assert r.mean_entropy[0] == pytest.approx(raw_h if flags else shaped_h, rel=1e-12)
        assert r.H[0, 0] == pytest.approx(shaped_h, rel=1e-12)


def test_raw_and_masked_only_statistics_combine():
    """STOP_RAW_ENTROPY | STOP_MASKED_ONLY: the mean of the raw-logit entropies over the
    positions still masked."""
    B, L, V = 1, 8, 16
    x = _peaked(B, L, V, [[p + 1 for p in range(L)]], height=9.0)
    x[0, :4, :] = 0.0                                        # committed rows: uniform
    st = oracle.State.fresh(B, L)
    st.mask[0, :4] = 0
    st.tokens[0, :4] = 3
    r = oracle.step(x, st, 1, oracle.Params(flags=oracle.STOP_RAW_ENTROPY | oracle.STOP_MASKED_ONLY,
                                            entropy_bound=-1.0))
    raw_h = oracle.row(x[0, 4], 1.0, False)[0]
    assert r.mean_entropy[0] == pytest.approx(raw_h, rel=1e-12)


def test_entropy_against_50_digit_arithmetic():
    """H = ln S - T'/S of the shaped logits, against the definition -sum p ln p evaluated with
    50 significant digits (mpmath), on rows with a wide logit range, at two temperatures."""
    import mpmath
    mpmath.mp.dps = 50
    rng = np.random.default_rng(21)
    for T in (0.8, 0.4):
        for scale in (1.0, 12.0):
            x = (rng.standard_normal(257) * scale).astype(np.float32)
            H = oracle.row(x, T, False)[0]
            z = [mpmath.mpf(float(v)) / mpmath.mpf(T) for v in x]
            m = max(z)
            w = [mpmath.e ** (zi - m) for zi in z]
            s = mpmath.fsum(w)
            ref = -mpmath.fsum((wi / s) * mpmath.log(wi / s) for wi in w)
            assert abs(H - float(ref)) <= 1e-12 * max(1.0, float(ref)), (T, scale, H, float(ref))
