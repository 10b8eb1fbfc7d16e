"""The block driver with continuous batching (eb_sample_blocks).

Ten blocks of 32 positions run on fewer slots than blocks, with peaks that grow at different
rates, so that blocks stop after different step counts and slots are refilled while the
others keep denoising.  Block k must come out exactly as canvas k of the plain denoising loop
over all blocks at once (the same canvas id in the Gumbel noise, the same stand-in denoiser
canvas), and as the oracle's run of that block on its own.  The configuration's closest
selection prefix sum stays 2e-4 from the bound and its closest perturbed-score gap 2e-5, so no
tie rule is needed.
"""
import ctypes

import numpy as np
import pytest
import torch

import canvas_sampler_step_b300 as eb
import eb_synth
import eb_synth.device as synth_dev
import oracle
from parity import params_pair

pytestmark = pytest.mark.gpu

N, L, V = 10, 32, 4096
RATES = (0.1, 0.2, 0.4, 0.8)


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eb.build()
    synth_dev.build()
    eb.lib()
    synth_dev.lib()


def _cfg():
    return eb_synth.Peaked(N, L, V, "f32", 3.0, 0.0, 4.0, tuple(RATES[k % 4] for k in range(N)),
                           tuple(100 + k for k in range(N)))


def _run_blocks(cfg, slots, params, poll_every=4):
    recipe = synth_dev.Recipe.of(cfg)
    logits = torch.empty((slots, L, V), dtype=torch.float32, device="cuda")
    ws_bytes = eb.eb_blocks_workspace_bytes(slots, L, V, eb.EB_F32)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    toks = torch.full((N, L), -7, dtype=torch.int32, device="cuda")
    steps = torch.zeros(N, dtype=torch.int32, device="cuda")
    status = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    it = eb.eb_sample_blocks(params, slots, L, V, eb.EB_F32, synth_dev.block_callback_address(),
                             ctypes.addressof(recipe), logits, N, toks, steps, status, ws, ws_bytes,
                             poll_every)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), steps.cpu().numpy(), status.cpu().numpy(), it


@pytest.fixture(scope="module")
def batch_loop():
    """Canvas k of the plain loop over all N blocks at once."""
    cfg = _cfg()
    gp, _ = params_pair(seed=5)
    recipe = synth_dev.Recipe.of(cfg)
    c = eb.Canvas(N, L, V, eb.EB_F32, max_steps=gp.max_steps)
    buf = torch.empty((N, L, V), dtype=torch.float32, device="cuda")
    c.run(gp, synth_dev.callback_address(), ctypes.addressof(recipe), buf)
    torch.cuda.synchronize()
    return c.tokens.cpu().numpy(), c.steps_taken.cpu().numpy(), c.status.cpu().numpy()


@pytest.mark.parametrize("slots", [4, 1, 16])
def test_blocks_equal_the_batch_loop(batch_loop, slots):
    """4 slots (refills), 1 slot (one block after the other), 16 slots (idle from the start)."""
    gp, _ = params_pair(seed=5)
    toks, steps, status, it = _run_blocks(_cfg(), slots, gp)
    btoks, bsteps, bstatus = batch_loop
    assert np.array_equal(status, bstatus)
    assert np.array_equal(steps, bsteps)
    assert np.array_equal(toks, btoks)
    assert len(set(steps.tolist())) > 3              # blocks stopped at different steps
    # the driver stops once every block is done, within one polling interval
    lower = int(np.ceil(steps.sum() / slots)) if slots <= N else int(steps.max())
    assert lower <= it <= steps.sum() + 4


def test_blocks_match_the_oracle():
    gp, op = params_pair(seed=5)
    cfg = _cfg()
    toks, steps, status, _ = _run_blocks(cfg, 4, gp)
    otoks, osteps, ostatus = oracle.run_blocks(lambda k, s: cfg.logits(s)[k], N, L, op)
    assert np.array_equal(status, ostatus)
    assert np.array_equal(steps, osteps)
    assert np.array_equal(toks, otoks)


def test_slot_generator_matches_the_batch_generator():
    """Slot b holding block k at step s receives exactly canvas k's logits at step s."""
    cfg = _cfg()
    recipe = synth_dev.Recipe.of(cfg)
    slot_block = torch.tensor([3, -1, 7, 0], dtype=torch.int32, device="cuda")
    slot_step = torch.tensor([5, 9, 0, 12], dtype=torch.int32, device="cuda")
    out = torch.full((4, L, V), 123.0, dtype=torch.float32, device="cuda")
    synth_dev.slot_logits(recipe, slot_block, slot_step, out)
    got = out.cpu().numpy()
    for b, (k, s) in enumerate(zip(slot_block.tolist(), slot_step.tolist())):
        if k < 0:
            assert (got[b] == 123.0).all()
        else:
            assert np.array_equal(got[b], cfg.logits(s)[k])


def test_blocks_on_e4m3_logits_equal_the_batch_loop():
    """The block driver on e4m3 logits (16 per vector, per-slot steps): block k again equals
    canvas k of the plain loop over all blocks at once."""
    import dataclasses
    cfg = dataclasses.replace(_cfg(), dtype="fp8")
    gp, _ = params_pair(seed=5)
    recipe = synth_dev.Recipe.of(cfg)
    logits = torch.empty((4, L, V), dtype=torch.uint8, device="cuda")
    ws_bytes = eb.eb_blocks_workspace_bytes(4, L, V, eb.EB_FP8_E4M3)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    toks = torch.full((N, L), -7, dtype=torch.int32, device="cuda")
    steps = torch.zeros(N, dtype=torch.int32, device="cuda")
    status = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    eb.eb_sample_blocks(gp, 4, L, V, eb.EB_FP8_E4M3, synth_dev.block_callback_address(),
                        ctypes.addressof(recipe), logits, N, toks, steps, status, ws, ws_bytes, 4)
    c = eb.Canvas(N, L, V, eb.EB_FP8_E4M3, max_steps=gp.max_steps)
    buf = torch.empty((N, L, V), dtype=torch.uint8, device="cuda")
    c.run(gp, synth_dev.callback_address(), ctypes.addressof(recipe), buf)
    torch.cuda.synchronize()
    assert np.array_equal(status.cpu().numpy(), c.status.cpu().numpy())
    assert np.array_equal(steps.cpu().numpy(), c.steps_taken.cpu().numpy())
    assert np.array_equal(toks.cpu().numpy(), c.tokens.cpu().numpy())
