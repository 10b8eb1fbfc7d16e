"""The sampler step for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc. A process may have reserved all device memory up front for
its own pool, a plugin may run inside a runtime that owns every allocation, or a hot loop may be
unable to afford an allocation's implicit synchronisation. ``eb_sampler_step_noalloc`` serves
them: it keeps its scratch in a fixed device array inside the library, for at most 8192 canvas
positions. This test calls it through the C ABI twice in a row, on the same canvases and on two
consecutive steps. Each call's outputs and canvas state must match those of ``eb_sampler_step``
run with a caller-allocated workspace. It also checks that a batch above the fixed size is
refused before any work is done.

The file name sorts last, so a run that stops at the first failure has already run every other
test.
"""
import numpy as np
import pytest
import torch

import canvas_sampler_step_b300 as eb
import eb_synth
import eb_synth.device as synth_dev
from parity import H_TOL, host_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eb.build()
    synth_dev.build()
    eb.lib()
    synth_dev.lib()


def _noalloc_step(c: eb.Canvas, params, logits, step):
    eb.eb_sampler_step_noalloc(params, c.B, c.L, c.V, c.dtype, logits, step, 0.0, c.mask, c.tokens,
                               c.prev_argmax, c.status, c.steps_taken, c.entropy, c.argmax,
                               c.sampled, c.selected, c.committed, c.mean_entropy)


def test_noalloc_step_matches_workspace_step_on_two_calls():
    cfg = eb_synth.Peaked(2, 256, 65536, "bf16", 2.5, 0.0, 12.0, (0.3, 0.3), (4, 5))
    params = eb.eb_default_params(seed=9)
    mask = np.stack([eb_synth.initial_mask(4, b, 256, 128) for b in range(2)])
    ref = eb.Canvas(2, 256, 65536, eb.EB_BF16, mask=mask)
    fixed = eb.Canvas(2, 256, 65536, eb.EB_BF16, mask=mask)
    for step in (0, 1):
        x = torch.empty((2, 256, 65536), dtype=torch.int16, device="cuda")
        synth_dev.logits(synth_dev.Recipe.of(cfg), step, x)
        ref.step(params, x, step)
        _noalloc_step(fixed, params, x, step)
        a, b = host_state(ref), host_state(fixed)
        assert np.abs(a["entropy"] - b["entropy"]).max() <= H_TOL, step
        for k in ("argmax", "sampled", "selected", "mask", "tokens", "prev_argmax", "status",
                  "committed"):
            assert np.array_equal(a[k], b[k]), (step, k)
        assert (b["committed"] >= 1).all()


def test_noalloc_step_at_the_fixed_size_with_the_raw_entropy_pass():
    """B * L = 8 x 1024 = 8192 positions, the largest batch the fixed array holds, with
    EB_FLAG_STOP_RAW_ENTROPY, whose second streaming pass keeps its partial states in the
    upper half of the array: two calls in a row equal eb_sampler_step on a caller-allocated
    workspace."""
    B, L, V = 8, 1024, 256
    cfg = eb_synth.Peaked(B, L, V, "bf16", 3.0, 0.0, 4.0, (0.3,) * B, tuple(range(20, 20 + B)))
    params = eb.eb_default_params(seed=11, flags=eb.EB_FLAG_STOP_RAW_ENTROPY)
    rng = np.random.default_rng(8)
    mask = (rng.random((B, L)) < 0.6).astype(np.uint8)
    mask[:, 0] = 1
    ref = eb.Canvas(B, L, V, eb.EB_BF16, mask=mask)
    fixed = eb.Canvas(B, L, V, eb.EB_BF16, mask=mask)
    for step in (0, 1):
        x = torch.empty((B, L, V), dtype=torch.int16, device="cuda")
        synth_dev.logits(synth_dev.Recipe.of(cfg), step, x)
        ref.step(params, x, step)
        _noalloc_step(fixed, params, x, step)
        a, b = host_state(ref), host_state(fixed)
        assert np.abs(a["entropy"] - b["entropy"]).max() <= H_TOL, step
        assert np.abs(a["mean_entropy"] - b["mean_entropy"]).max() <= H_TOL, step
        for k in ("argmax", "sampled", "selected", "mask", "tokens", "prev_argmax", "status",
                  "committed"):
            assert np.array_equal(a[k], b[k]), (step, k)


def test_noalloc_step_rejects_batches_above_the_fixed_scratch():
    params = eb.eb_default_params()
    c = eb.Canvas(1, 16, 64, eb.EB_F32)
    with pytest.raises(eb.EbError) as ei:
        # 9 x 1024 positions > 8192: refused before anything is read or launched
        eb.eb_sampler_step_noalloc(params, 9, 1024, 64, eb.EB_F32, c.entropy, 0, 0.0, c.mask,
                                   c.tokens, c.prev_argmax, c.status, c.steps_taken, c.entropy,
                                   c.argmax, c.sampled, c.selected, c.committed, c.mean_entropy)
    assert ei.value.status == eb.EB_ERR_UNSUPPORTED
    with pytest.raises(eb.EbError) as ei:
        # one position beyond the fixed size (8193 = 8193 x 1) is refused too
        eb.eb_sampler_step_noalloc(params, 8193, 1, 64, eb.EB_F32, c.entropy, 0, 0.0, c.mask,
                                   c.tokens, c.prev_argmax, c.status, c.steps_taken, c.entropy,
                                   c.argmax, c.sampled, c.selected, c.committed, c.mean_entropy)
    assert ei.value.status == eb.EB_ERR_UNSUPPORTED
