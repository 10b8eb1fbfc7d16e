"""GPU-vs-oracle parity of the EB sampler step and loop, through the C ABI.

Every input is seeded and synthetic (eb_synth).  The oracle always receives the numpy
generator's values; the GPU receives the CUDA generator's values, which
``test_generator_bit_exact`` shows to be the same bits (or an H2D copy of the numpy ones).
"""
import numpy as np
import pytest
import torch

import canvas_sampler_step_b300 as eb
import eb_synth
import eb_synth.device as synth_dev
import oracle
from parity import (ORDER_TOL, STOP_TOL, Report, compare_step, device_logits, host_state, params_pair,
                    to_device_logits, H_TOL)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eb.build()
    synth_dev.build()
    eb.lib()
    synth_dev.lib()


def _dtype(cfg):
    return {"f32": eb.EB_F32, "bf16": eb.EB_BF16, "fp8": eb.EB_FP8_E4M3}[cfg.dtype]


# ------------------------------------------------------------------ generator

@pytest.mark.parametrize("cfg,rows", [
    (eb_synth.cfg0(0, L=16, V=4096), None),
    (eb_synth.cfg1(3, L=8, V=262144), None),
    (eb_synth.Peaked(2, 5, 1001, "f32", 3.0, 1.0, 2.0, (0.3, 0.7), (11, 12)), None),
    (eb_synth.Peaked(2, 5, 1001, "bf16", 3.0, 1.0, 2.0, (0.3, 0.7), (11, 12)), None),
    (eb_synth.cfg3(B=8, L=256, V=262144), [0, 77, 255]),
    (eb_synth.Peaked(2, 5, 1001, "fp8", 3.0, 1.0, 2.0, (0.3, 0.7), (11, 12)), None),
    (eb_synth.Peaked(1, 4, 65536, "fp8", 60.0, 400.0, 200.0, (0.0,), (13,)), None),   # saturation
])
def test_generator_bit_exact(cfg, rows):
    view = {"f32": np.uint32, "bf16": np.uint16, "fp8": np.uint8}[cfg.dtype]
    for s in (0, 7):
        dev = device_logits(cfg, s).cpu().numpy()
        for b in range(cfg.B):
            p = np.arange(cfg.L) if rows is None else np.array(rows)
            host = cfg.rows(b, p, s)
            assert np.array_equal(dev[b, p].view(view), host.view(view)), (b, s)


def test_generator_skips_stopped_canvases():
    cfg = eb_synth.cfg3(B=4, L=4, V=64)
    out = torch.full((4, 4, 64), 7, dtype=torch.int16, device="cuda")
    status = torch.tensor([0, 1, 0, 2], dtype=torch.int32, device="cuda")
    synth_dev.logits(synth_dev.Recipe.of(cfg), 3, out, status)
    o = out.cpu().numpy()
    assert (o[1] == 7).all() and (o[3] == 7).all() and not (o[0] == 7).all()


# ------------------------------------------------------------------ one step

def _run_step(cfg, step, mask=None, seed=5, temperature=0.0, state=None, **kw):
    gp, op = params_pair(seed=seed, **kw)
    x = cfg.logits(step)
    c = eb.Canvas(cfg.B, cfg.L, cfg.V, _dtype(cfg), mask=mask)
    ost = oracle.State.fresh(cfg.B, cfg.L, mask)
    if state is not None:
        state(c, ost)
    running = ost.status == oracle.RUNNING
    c.step(gp, to_device_logits(x), step, temperature)
    res = oracle.step(x, ost, step, op, temperature=float(np.float32(temperature)))
    return host_state(c), res, ost, running


CASES = [
    # (recipe, step, mask density)  -- vector paths, several tiles per row, ragged tails
    (eb_synth.cfg0(0, L=256, V=4096), 0, 1.0),
    (eb_synth.cfg0(0, L=256, V=4096), 9, 0.7),
    (eb_synth.Peaked(3, 64, 20000, "bf16", 2.5, 0.0, 12.0, (0.0, 0.0, 0.0), (1, 2, 3)), 0, 0.5),
    (eb_synth.Peaked(2, 100, 2048, "bf16", 3.0, 4.0, 2.0, (0.3, 0.3), (4, 5)), 20, 0.8),
    # scalar paths: V not a multiple of the 16-byte vector
    (eb_synth.Peaked(2, 16, 4099, "f32", 3.0, 2.0, 0.0, (0.3, 0.3), (6, 7)), 3, 1.0),
    (eb_synth.Peaked(1, 40, 12347, "bf16", 2.5, 0.0, 12.0, (0.0,), (8,)), 0, 0.5),
    # e4m3 logits: 16 per vector, a ragged tail (20000 = 1250 vectors), and the scalar path
    (eb_synth.Peaked(2, 64, 4096, "fp8", 2.5, 0.0, 12.0, (0.0, 0.0), (14, 15)), 0, 0.5),
    (eb_synth.Peaked(2, 48, 20000, "fp8", 3.0, 4.0, 2.0, (0.3, 0.3), (16, 17)), 12, 0.8),
    (eb_synth.Peaked(1, 32, 4099, "fp8", 3.0, 2.0, 0.0, (0.3,), (18,)), 3, 1.0),
    # tiny rows and a non-power-of-two canvas
    (eb_synth.Peaked(1, 1000, 8, "f32", 1.0, 3.0, 0.0, (0.0,), (9,)), 2, 0.9),
    (eb_synth.Peaked(4, 1, 1, "f32", 1.0, 0.0, 0.0, (0.0,) * 4, (1, 2, 3, 4)), 0, 1.0),
]


@pytest.mark.parametrize("cfg,step,density", CASES)
def test_step_parity(cfg, step, density):
    rng = np.random.default_rng(step + cfg.V)
    mask = (rng.random((cfg.B, cfg.L)) < density).astype(np.uint8)
    mask[:, 0] = 1
    g, res, ost, running = _run_step(cfg, step, mask=mask)
    rep = Report()
    compare_step(g, res, ost, running, rep, ctx=f"V={cfg.V}")
    assert rep.canvas_ties <= max(1, cfg.B // 4)


def test_step_parity_low_entropy_many_accepted():
    # peaks so high that most entropies are ~0: selection accepts long prefixes
    cfg = eb_synth.Peaked(2, 256, 4096, "f32", 1.0, 30.0, 10.0, (0.0, 0.0), (3, 4))
    g, res, ost, running = _run_step(cfg, 4)
    rep = Report()
    compare_step(g, res, ost, running, rep)
    assert res.committed.min() > 1


@pytest.mark.parametrize("seed", range(10))
def test_step_parity_single_step_workload_full_size(seed):
    """B=1, L=256, V=262144 bf16, 128 of 256 masked, T=0.8 (the benchmarked step)."""
    cfg = eb_synth.cfg1(seed)
    mask = eb_synth.cfg1_mask(seed)
    x = cfg.logits(0)
    dev = device_logits(cfg, 0)
    assert torch.equal(dev.cpu(), torch.from_numpy(x.view(np.int16)))
    gp, op = params_pair(seed=seed)
    c = eb.Canvas(1, 256, 262144, eb.EB_BF16, mask=mask)
    ost = oracle.State.fresh(1, 256, mask)
    c.step(gp, dev, 0, 0.8)
    res = oracle.step(x, ost, 0, op, temperature=float(np.float32(0.8)))
    rep = Report()
    compare_step(host_state(c), res, ost, np.array([True]), rep, ctx=f"seed {seed}")
    assert rep.max_h_err < H_TOL


def test_step_parity_single_step_workload_e4m3_full_size():
    """The benchmarked step with its logits rounded to e4m3 (64 MiB): only about 250 distinct
    values, so most argmax comparisons are exact ties that the first index settles."""
    import dataclasses
    cfg = dataclasses.replace(eb_synth.cfg1(0), dtype="fp8")
    mask = eb_synth.cfg1_mask(0)
    x = cfg.logits(0)
    dev = device_logits(cfg, 0)
    assert np.array_equal(dev.cpu().numpy(), x)
    gp, op = params_pair(seed=0)
    c = eb.Canvas(1, 256, 262144, eb.EB_FP8_E4M3, mask=mask)
    ost = oracle.State.fresh(1, 256, mask)
    c.step(gp, dev, 0, 0.8)
    res = oracle.step(x, ost, 0, op, temperature=float(np.float32(0.8)))
    rep = Report()
    compare_step(host_state(c), res, ost, np.array([True]), rep, ctx="e4m3")
    assert rep.max_h_err < H_TOL


# ------------------------------------------------------------------ the loop

def _host_copy(cfg, dev, s, rng):
    """The device generator's logits of step s as the oracle's input, with two rows of a running
    canvas checked against the numpy generator (the whole-array equality of the two generators
    is test_generator_bit_exact's; the numpy generator alone takes ~10 s per canvas-step at
    V = 262144)."""
    view = {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8}[cfg.dtype]
    x = dev.cpu().numpy().view(view)
    b = int(rng.integers(cfg.B))
    p = rng.choice(cfg.L, 2, replace=False)
    return x, (b, p)


def _lockstep(cfg, params_kw=None, mask=None, device_generator=False, label="", resync_ties=False):
    """Run eb_sampler_step step by step next to the oracle; compare every step until a
    counted tie lets the trajectories part, then keep running the GPU alone.  Returns
    (report, GPU state after every step, canvas, oracle state, canvases parted by a tie).
    ``device_generator``: the oracle takes the CUDA generator's bits (full-size loops).
    ``resync_ties``: at a counted tie the GPU's step is checked for validity and the oracle
    adopts the GPU's canvas state, so that no canvas parts and every step is compared."""
    gp, op = params_pair(seed=cfg.seeds[0], **(params_kw or {}))
    c = eb.Canvas(cfg.B, cfg.L, cfg.V, _dtype(cfg), mask=mask, max_steps=gp.max_steps)
    ost = oracle.State.fresh(cfg.B, cfg.L, mask)
    rep = Report(label=label)
    hist = []
    parted = set()
    rng = np.random.default_rng(1234)
    for s in range(gp.max_steps):
        st_before = c.status.cpu().numpy()
        if not (st_before == eb.EB_RUNNING).any():
            break
        dev = device_logits(cfg, s, c.status)
        if device_generator:
            x, (bc, pc) = _host_copy(cfg, dev, s, rng)
            if st_before[bc] == eb.EB_RUNNING:
                view = {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8}[cfg.dtype]
                assert np.array_equal(x[bc, pc].view(view), cfg.rows(bc, pc, s).view(view)), (s, bc, pc)
        else:
            x = cfg.logits(s)
        c.step(gp, dev, s, 0.0)
        g = host_state(c)
        hist.append(g)
        running = ost.status == oracle.RUNNING
        mask_before = ost.mask.copy()
        res = oracle.step(x, ost, s, op)
        # canvases whose trajectories parted after a counted tie are no longer compared
        view = running & (st_before == eb.EB_RUNNING)
        for b in parted:
            view[b] = False
        tied = compare_step(g, res, ost, view, rep, ctx=f"step {s}")
        if resync_ties:
            for b in tied:
                _check_tied_step(g, res, ost, mask_before, b, ctx=f"step {s}")
                _adopt(ost, g, b)
        else:
            parted |= tied
    return rep, hist, c, ost, parted


def _check_tied_step(g, res, ost, mask_before, b, ctx=""):
    """At a counted tie the GPU's step must still be a valid one: it commits only positions that
    were masked; unless the stop decision itself tied, its commit count is within one of the
    oracle's, and no committed position has an entropy above an uncommitted masked one by more
    than the order tolerance."""
    sel = g["selected"][b].astype(bool)
    was = mask_before[b].astype(bool)
    assert not (sel & ~was).any(), f"{ctx} canvas {b}: committed an unmasked position"
    stopped = g["status"][b] != eb.EB_RUNNING or ost.status[b] != oracle.RUNNING
    if stopped and res.stop_margin[b] < STOP_TOL:
        return
    assert abs(int(g["committed"][b]) - int(res.committed[b])) <= 1, (ctx, b, g["committed"][b], res.committed[b])
    rest = was & ~sel
    if sel.any() and rest.any() and g["status"][b] == eb.EB_RUNNING:
        H = g["entropy"][b].astype(np.float64)
        assert H[sel].max() <= H[rest].min() + ORDER_TOL, (ctx, b)


def _adopt(ost, g, b):
    """The oracle continues from the GPU's canvas state b (after a tie the GPU's choice is as
    good as the oracle's), so that the following steps are still compared."""
    for k in ("mask", "tokens", "prev_argmax", "status", "steps_taken"):
        getattr(ost, k)[b] = g[k][b]


def test_loop_parity_pr1_workload():
    """B=1, L=256, V=4096 fp32, up to 48 steps, seed 0: lockstep with the oracle."""
    cfg = eb_synth.cfg0(0)
    rep, hist, c, *_ = _lockstep(cfg)
    assert rep.canvases >= 10
    # the whole loop through eb_sample_canvas reproduces the stepwise run bit for bit
    gp, _ = params_pair(seed=0)
    c2 = eb.Canvas(1, 256, 4096, eb.EB_F32, max_steps=48)
    buf = torch.empty((1, 256, 4096), dtype=torch.float32, device="cuda")
    recipe = synth_dev.Recipe.of(cfg)
    import ctypes
    ran = c2.run(gp, synth_dev.callback_address(), ctypes.addressof(recipe), buf)
    g2 = host_state(c2)
    last = hist[-1]
    for k in ("tokens", "mask", "status", "steps_taken", "prev_argmax"):
        assert np.array_equal(g2[k], last[k]), k
    assert ran == 48 or g2["status"][0] != eb.EB_RUNNING
    assert g2["mask"].sum() == 0 and (g2["tokens"] >= 0).all()


def test_loop_parity_mixed_batch_small():
    """B=8 canvases with per-canvas growth rates (easy / hard), V=2048 bf16."""
    cfg = eb_synth.Peaked(8, 64, 2048, "bf16", 3.0, 0.0, 4.0, eb_synth.cfg3().growth,
                          tuple(range(8)))
    rep, hist, c, *_ = _lockstep(cfg)
    st = hist[-1]["status"]
    assert (st != eb.EB_RUNNING).all()
    assert rep.canvases > 50


def test_loop_adaptive_stop_parity():
    """Dominant, fixed peaks: the entropy is ~0 everywhere and the argmax never moves, so every
    canvas stops adaptively at step 1 and its still-masked positions take the argmax.  Which
    position step 0 commits is an order tie (all entropies ~0), but every committed token is
    the peak either way: stop reason, stop step and final tokens match the oracle's."""
    cfg = eb_synth.Peaked(3, 128, 4096, "f32", 1.0, 40.0, 0.0, (0.0, 0.0, 0.0), (21, 22, 23))
    gp, op = params_pair(seed=21, entropy_bound=-1.0)
    rep, hist, c, *_ = _lockstep(cfg, params_kw={"entropy_bound": -1.0})
    final = hist[-1]
    assert (final["status"] == eb.EB_STOP_ADAPTIVE).all()
    assert (final["steps_taken"] == 2).all()
    assert final["mask"].sum() == 0
    # step 0 committed one position per canvas, step 1 the remaining 127
    assert hist[0]["committed"].tolist() == [1, 1, 1]
    assert hist[1]["committed"].tolist() == [127, 127, 127]
    ost = oracle.run_loop(lambda s, st: cfg.logits(s), 3, 128, op)
    assert ost.status.tolist() == [oracle.ADAPTIVE] * 3 and ost.steps_taken.tolist() == [2, 2, 2]
    assert np.array_equal(final["tokens"], ost.tokens)


def test_loop_cap_and_complete_parity():
    """Noisy logits that never settle: with the bound at -1 exactly one position commits per
    step, so a 5-step run ends at the cap with the rest filled by the argmax, while a canvas of
    4 positions completes at step 3; both match the oracle."""
    cfg = eb_synth.Peaked(1, 16, 512, "f32", 3.0, 0.0, 0.0, (0.0,), (31,))
    rep, hist, c, *_ = _lockstep(cfg, params_kw={"entropy_bound": -1.0, "max_steps": 5})
    assert hist[-1]["status"][0] == eb.EB_STOP_CAP and hist[-1]["steps_taken"][0] == 5
    assert hist[-1]["committed"][0] == 16 - 4
    cfg2 = eb_synth.Peaked(1, 4, 512, "f32", 3.0, 0.0, 0.0, (0.0,), (32,))
    rep2, hist2, c2, *_ = _lockstep(cfg2, params_kw={"entropy_bound": -1.0})
    assert hist2[-1]["status"][0] == eb.EB_STOP_COMPLETE and hist2[-1]["steps_taken"][0] == 4


def test_step_parity_longest_canvas():
    """L = 1024 positions (the largest canvas the selection kernel takes) with many
    low-entropy positions: the general (shared-memory) sort path."""
    cfg = eb_synth.Peaked(1, 1024, 256, "f32", 1.0, 25.0, 10.0, (0.0,), (41,))
    g, res, ost, running = _run_step(cfg, 0)
    rep = Report()
    compare_step(g, res, ost, running, rep)
    assert res.committed[0] > 32


def test_step_parity_beyond_the_weighted_partition():
    """B*L = 17 x 256 = 4352 rows exceed the weighted partition's 4096-row limit, so the
    closed-form uniform partition runs instead; it skips a halted canvas by its status."""
    cfg = eb_synth.Peaked(17, 256, 1024, "f32", 3.0, 0.0, 4.0, (0.0,) * 17, tuple(range(17)))
    rng = np.random.default_rng(3)
    mask = (rng.random((17, 256)) < 0.5).astype(np.uint8)
    mask[:, 0] = 1

    def halt(c, ost):
        c.status[5] = eb.EB_STOP_CAP
        ost.status[5] = oracle.CAP

    g, res, ost, running = _run_step(cfg, 0, mask=mask, state=halt)
    assert not running[5]
    rep = Report()
    compare_step(g, res, ost, running, rep, ctx="uniform partition")
    assert rep.canvases == 16 and rep.canvas_ties <= 4
    assert g["status"][5] == eb.EB_STOP_CAP and np.array_equal(g["mask"][5], mask[5])


def _check_loop_against_oracle(cfg, rep, hist, ost, parted):
    """Steps to stop, stop reason and final tokens of every canvas equal the oracle's, except
    for canvases whose trajectories parted at a counted tie; the ties stay rare."""
    final = hist[-1]
    assert (final["status"] != eb.EB_RUNNING).all() and final["mask"].sum() == 0
    for b in range(cfg.B):
        if b in parted:
            continue
        assert final["status"][b] == ost.status[b], (b, final["status"][b], ost.status[b])
        assert final["steps_taken"][b] == ost.steps_taken[b], (b, final["steps_taken"][b], ost.steps_taken[b])
        assert np.array_equal(final["tokens"][b], ost.tokens[b]), b
    assert rep.row_ties <= max(2, rep.rows // 1000), rep.line()
    assert rep.canvas_ties <= max(2, rep.canvases // 10), rep.line()


def _loop_in_one_call(cfg, gp, final):
    """eb_sample_canvas with the stand-in denoiser reproduces the stepwise run bit for bit."""
    import ctypes
    c2 = eb.Canvas(cfg.B, cfg.L, cfg.V, _dtype(cfg), max_steps=gp.max_steps)
    buf = torch.empty((cfg.B, cfg.L, cfg.V), dtype=torch.int16, device="cuda")
    recipe = synth_dev.Recipe.of(cfg)
    c2.run(gp, synth_dev.callback_address(), ctypes.addressof(recipe), buf, poll_every=4)
    g2 = host_state(c2)
    for k in ("tokens", "status", "steps_taken"):
        assert np.array_equal(g2[k], final[k]), k


def test_loop_full_size_adaptive_one_canvas():
    """The full adaptive loop: B=1, L=256, V=262144 bf16, up to 48 steps, logits regenerated
    every step (sigma 3, peak U(0,4) + 0.3 s).  Every step is compared with the oracle element by
    element, and the steps to stop, stop reason and tokens equal the oracle's."""
    cfg = eb_synth.cfg2()
    rep, hist, c, ost, parted = _lockstep(cfg, device_generator=True, label="full adaptive loop, B=1",
                                          resync_ties=True)
    _check_loop_against_oracle(cfg, rep, hist, ost, parted)
    assert rep.canvases == len(hist)            # every step was compared
    committed = [int(h["committed"][0]) for h in hist]
    assert sum(committed) == 256 and all(k >= 1 for k in committed[:-1])
    _loop_in_one_call(cfg, params_pair(seed=0)[0], hist[-1])


def test_loop_full_size_adaptive_stop():
    """The early-stop loop at full size (B=1, 256 x 262144 bf16, sigma 1, peaks U(12, 14) +
    0.5 s): the mean entropy falls below 0.005 with positions still masked, so the adaptive stop
    ends the loop well before the cap, and the still-masked positions take the argmax.  Every
    step is compared with the oracle; the stop step, stop reason and tokens equal the oracle's."""
    cfg = eb_synth.cfg_stop()
    rep, hist, c, ost, parted = _lockstep(cfg, device_generator=True, label="early stop, B=1",
                                          resync_ties=True)
    _check_loop_against_oracle(cfg, rep, hist, ost, parted)
    final = hist[-1]
    assert final["status"][0] == eb.EB_STOP_ADAPTIVE, final["status"]
    assert final["steps_taken"][0] < 48
    committed = [int(h["committed"][0]) for h in hist]
    assert committed[-1] > 1 and sum(committed) == 256     # the stop commits the rest at once
    _loop_in_one_call(cfg, params_pair(seed=cfg.seeds[0])[0], hist[-1])


def test_loop_full_size_batch_of_eight():
    """B=8, L=256, V=262144 bf16, rates (0.1, 0.2, 0.4, 0.8), up to 48 steps: every step of every
    running canvas compared with the oracle element by element, steps to stop per canvas equal
    to the oracle's, and eb_sample_canvas equal to the stepwise run."""
    cfg = eb_synth.cfg3()
    rep, hist, c, ost, parted = _lockstep(cfg, device_generator=True, label="mixed batch, B=8",
                                          resync_ties=True)
    _check_loop_against_oracle(cfg, rep, hist, ost, parted)
    assert rep.canvases >= 8 * 20
    _loop_in_one_call(cfg, params_pair(seed=0)[0], hist[-1])


# ------------------------------------------------------------------ edge cases

def test_empty_batch_is_noop():
    gp, _ = params_pair()
    eb.eb_sampler_step(gp, 0, 256, 4096, eb.EB_F32, None, 0, 0.0, None, None, None, None, None,
                       None, None, None, None, None, None, None, 0)


def test_all_unmasked_canvas_completes_without_commit():
    cfg = eb_synth.cfg0(0, L=32, V=512)
    g, res, ost, running = _run_step(cfg, 0, mask=np.zeros((1, 32), np.uint8))
    assert g["status"][0] == eb.EB_STOP_COMPLETE and g["committed"][0] == 0
    assert (g["sampled"] == -1).all()
    rep = Report()
    compare_step(g, res, ost, running, rep)


def test_stopped_canvases_untouched():
    cfg = eb_synth.Peaked(3, 16, 256, "f32", 2.0, 1.0, 0.0, (0.0,) * 3, (1, 1, 1))

    def prep(c, ost):
        c.status[1] = eb.EB_STOP_CAP
        ost.status[1] = oracle.CAP
    g, res, ost, running = _run_step(cfg, 1, state=prep)
    assert g["status"][1] == eb.EB_STOP_CAP and (g["mask"][1] == 1).all()
    rep = Report()
    compare_step(g, res, ost, running, rep)


def test_nonfinite_logits_set_status_bit():
    for bad in (np.nan, np.inf, -np.inf):
        x = np.zeros((2, 8, 64), np.float32)
        x[1, 3, 5] = bad
        c = eb.Canvas(2, 8, 64, eb.EB_F32)
        gp, _ = params_pair()
        c.step(gp, to_device_logits(x), 0, 0.0)
        g = host_state(c)
        assert g["status"][1] & eb.EB_STATUS_NONFINITE
        assert g["status"][0] == eb.EB_RUNNING
        assert (g["mask"][1] == 1).all() and (g["tokens"][1] == -1).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_excluded_tokens_k_point_entropy(dtype):
    # k equal top logits and the rest -1e30 (excluded): H = ln k, the sample is one of the
    # k, the argmax the first of them -- the oracle's k-point closed form with -inf
    x = np.full((1, 4, 4096), -1.0e30, np.float32)
    tops = {0: [5], 1: [7, 900], 2: [1, 2, 3], 3: list(range(100, 4096, 64))}
    for p, t in tops.items():
        x[0, p, t] = 1.5
    if dtype == "bf16":
        x = eb_synth.to_bf16_bits(x)
    c = eb.Canvas(1, 4, 4096, eb.EB_BF16 if dtype == "bf16" else eb.EB_F32)
    gp, _ = params_pair(entropy_bound=-1.0)
    c.step(gp, to_device_logits(x), 0, 0.0)
    g = host_state(c)
    for p, t in tops.items():
        assert abs(g["entropy"][0, p] - np.log(len(t))) < H_TOL
        assert g["argmax"][0, p] == t[0]
        assert g["sampled"][0, p] in t


def test_deterministic_repeat():
    cfg = eb_synth.Peaked(2, 64, 50000, "bf16", 2.5, 0.0, 12.0, (0.0, 0.0), (1, 2))
    x = to_device_logits(cfg.logits(0))
    outs = []
    for _ in range(2):
        c = eb.Canvas(2, 64, 50000, eb.EB_BF16)
        gp, _ = params_pair(seed=3)
        c.step(gp, x, 0, 0.8)
        outs.append(host_state(c))
    for k in outs[0]:
        assert np.array_equal(outs[0][k], outs[1][k], equal_nan=True), k


def test_callback_failure_aborts_loop():
    c = eb.Canvas(1, 8, 64, eb.EB_F32)
    buf = torch.zeros((1, 8, 64), dtype=torch.float32, device="cuda")
    calls = []

    @eb.LOGITS_FN
    def fn(user, step, tokens, status, logits, stream):
        calls.append(step)
        return 0 if step < 2 else 1

    gp, _ = params_pair()
    with pytest.raises(eb.EbError) as ei:
        c.run(gp, fn, None, buf)
    assert ei.value.status == eb.EB_ERR_CALLBACK
    assert calls == [0, 1, 2]


def test_resume_reproduces_uninterrupted_run():
    cfg = eb_synth.cfg0(1, L=64, V=1024)
    recipe = synth_dev.Recipe.of(cfg)
    import ctypes
    gp, _ = params_pair(seed=1, max_steps=12)
    buf = torch.empty((1, 64, 1024), dtype=torch.float32, device="cuda")
    full = eb.Canvas(1, 64, 1024, eb.EB_F32, max_steps=12)
    full.run(gp, synth_dev.callback_address(), ctypes.addressof(recipe), buf)
    part = eb.Canvas(1, 64, 1024, eb.EB_F32, max_steps=12)
    gp5, _ = params_pair(seed=1, max_steps=12)
    # first 5 steps via the step API, then resume the loop at step 5
    for s in range(5):
        synth_dev.logits(recipe, s, buf, part.status)
        part.step(gp5, buf, s)
    part.run(gp, synth_dev.callback_address(), ctypes.addressof(recipe), buf, start_step=5)
    a, b = host_state(full), host_state(part)
    for k in ("tokens", "status", "steps_taken", "prev_argmax"):
        assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------- reading variants (flags)

def _variant_step(x, flags, step=1, mask=None, prev=None, **prm):
    B, L, V = x.shape
    gp, op = params_pair(seed=13, flags=flags, **prm)
    c = eb.Canvas(B, L, V, eb.EB_F32, mask=mask)
    ost = oracle.State.fresh(B, L, mask)
    if prev is not None:
        c.prev_argmax.copy_(torch.as_tensor(prev, dtype=torch.int32))
        ost.prev_argmax[:] = prev
    c.step(gp, to_device_logits(x), step, 0.0)
    g = host_state(c)
    res = oracle.step(x, ost, step, op)
    rep = Report()
    compare_step(g, res, ost, np.ones(B, bool), rep, ctx=f"flags {flags}")
    return g, res, ost, rep


def test_stop_masked_only_parity():
    """Committed positions with uniform rows (H = ln V) and a changed argmax block the default
    stop; with EB_FLAG_STOP_MASKED_ONLY only the still-masked, sharply peaked positions count,
    so the canvases stop.  GPU and oracle agree under both readings."""
    B, L, V = 2, 64, 512
    x = np.zeros((B, L, V), np.float32)
    peak = (np.arange(L) * 7 + 3) % V
    for b in range(B):
        x[b, np.arange(L), peak] = 40.0
    mask = np.ones((B, L), np.uint8)
    mask[:, : L // 2] = 0
    x[:, : L // 2, :] = 0.0
    prev = np.broadcast_to(np.where(np.arange(L) < L // 2, 5, peak), (B, L)).astype(np.int32)
    g, res, ost, _ = _variant_step(x, 0, mask=mask, prev=prev, entropy_bound=-1.0)
    assert (g["status"] == eb.EB_RUNNING).all() and (ost.status == oracle.RUNNING).all()
    g, res, ost, _ = _variant_step(x, eb.EB_FLAG_STOP_MASKED_ONLY, mask=mask, prev=prev, entropy_bound=-1.0)
    assert (g["status"] == eb.EB_STOP_ADAPTIVE).all() and (ost.status == oracle.ADAPTIVE).all()
    assert (g["mean_entropy"] < 1e-6).all()
    assert np.array_equal(g["tokens"], ost.tokens)


def test_finalize_sampled_parity_at_stop_and_cap():
    """EB_FLAG_FINALIZE_SAMPLED: the positions an adaptive stop or the step cap finalises take
    the sampled token; GPU and oracle agree, and the tokens differ from the argmax."""
    B, L, V = 2, 48, 512
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((B, L, V)) * 0.5).astype(np.float32)
    probe = oracle.State.fresh(B, L)
    r0 = oracle.step(x, probe, 1, params_pair(seed=13)[1])
    g, res, ost, rep = _variant_step(x, eb.EB_FLAG_FINALIZE_SAMPLED, prev=r0.A, stop_entropy=100.0)
    assert (g["status"] == eb.EB_STOP_ADAPTIVE).all()
    assert (g["tokens"] == g["sampled"]).all()
    assert (g["tokens"] != g["argmax"]).sum() >= 10
    cfg = eb_synth.Peaked(1, 16, 512, "f32", 3.0, 0.0, 0.0, (0.0,), (31,))
    rep, hist, c, *_ = _lockstep(cfg, params_kw={"entropy_bound": -1.0, "max_steps": 5,
                                             "flags": eb.EB_FLAG_FINALIZE_SAMPLED})
    last = hist[-1]
    assert last["status"][0] == eb.EB_STOP_CAP
    fin = last["selected"][0].astype(bool)
    assert (last["tokens"][0][fin] == last["sampled"][0][fin]).all()


def test_raw_entropy_stop_parity():
    """EB_FLAG_STOP_RAW_ENTROPY: the stop statistic from a second pass at T = 1.  Peaks of 12
    over 511 zeros stop the default (shaped entropy ~0.002) but not the variant (raw ~0.041);
    both match the oracle, and a lockstep loop with the flag matches it step by step."""
    B, L, V = 2, 64, 512
    x = np.zeros((B, L, V), np.float32)
    peak = (np.arange(L) * 5 + 1) % V
    for b in range(B):
        x[b, np.arange(L), peak] = 12.0
    prev = np.broadcast_to(peak, (B, L)).astype(np.int32)
    g, res, ost, _ = _variant_step(x, 0, prev=prev, entropy_bound=-1.0)
    assert (g["status"] == eb.EB_STOP_ADAPTIVE).all() and (ost.status == oracle.ADAPTIVE).all()
    g, res, ost, _ = _variant_step(x, eb.EB_FLAG_STOP_RAW_ENTROPY, prev=prev, entropy_bound=-1.0)
    assert (g["status"] == eb.EB_RUNNING).all() and (ost.status == oracle.RUNNING).all()
    assert np.abs(g["mean_entropy"] - res.mean_entropy).max() < 1e-4
    rep, hist, c, *_ = _lockstep(eb_synth.cfg0(0, L=64, V=4096), params_kw={"flags": eb.EB_FLAG_STOP_RAW_ENTROPY})
    assert rep.canvases >= 10
