"""CPU checks of the C ABI: the shared libraries load and export every function their
headers declare; argument validation rejects bad calls before touching a device; the
parameter defaults are the model card's settings (DiffusionGemma model card, "Best
practices" section 1)."""
import ctypes
import os
import re

import numpy as np
import pytest

import canvas_sampler_step_b300 as eb
import eb_synth.device as synth_dev

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(eb_\w+)\s*\(", text))
    # typedef'd function-pointer types are not symbols
    names -= set(re.findall(r"\(\s*\*\s*(eb_\w+)\s*\)", text))
    return names


@pytest.fixture(scope="module")
def libs():
    eb.build()
    synth_dev.build()
    return eb.lib(), synth_dev.lib()


def test_every_declared_symbol_is_exported(libs):
    sampler, synth = libs
    decl = _declared("eb_sampler.h")
    assert {"eb_sampler_step", "eb_sample_canvas", "eb_workspace_bytes"} <= decl
    for name in decl:
        assert hasattr(sampler, name), name
    for name in _declared("eb_synth.h"):
        assert hasattr(synth, name), name
    assert set(eb.EXPORTED) <= decl


def test_checked_build_exports_the_same_symbols(libs):
    """The checked debug build (-DEB_CHECKS) is the same library with device bounds checks: it
    exports every declared function, says it is the checked build, and the normal one does
    not (neither call needs a device)."""
    eb.build_checks()
    checked = ctypes.CDLL(eb.CHECKS_LIB_PATH)
    for name in _declared("eb_sampler.h"):
        assert hasattr(checked, name), name
    checked.eb_checks_enabled.restype = ctypes.c_int
    assert checked.eb_checks_enabled() == 1
    assert not eb.eb_checks_enabled() or os.environ.get("EB_SAMPLER_LIB")
    assert eb.eb_check_word() == 0 or eb.eb_checks_enabled()


def test_default_params_are_the_recommended_settings(libs):
    p = eb.eb_default_params()
    assert p.max_steps == 48
    assert p.t_start == np.float32(0.8) and p.t_end == np.float32(0.4)
    assert p.entropy_bound == np.float32(0.1) and p.stop_entropy == np.float32(0.005)
    assert eb.eb_temperature(p, 0) == np.float32(0.8)
    assert abs(eb.eb_temperature(p, 47) - 0.4) < 1e-7
    temps = [eb.eb_temperature(p, s) for s in range(48)]
    assert all(a > b for a, b in zip(temps, temps[1:]))


def test_workspace_bytes(libs):
    assert eb.eb_workspace_bytes(1, 256, 262144, eb.EB_BF16) % 256 == 0
    assert eb.eb_workspace_bytes(8, 256, 262144, eb.EB_BF16) > eb.eb_workspace_bytes(1, 256, 262144, eb.EB_BF16)
    assert eb.eb_workspace_bytes(-1, 256, 16, eb.EB_F32) == 0


FAKE = 0x100000   # never dereferenced: every call below fails validation first


def _step(**kw):
    args = dict(params=eb.eb_default_params(), B=1, L=256, V=4096, dtype=eb.EB_F32, logits=FAKE,
                step=0, temperature=0.0, mask=FAKE, tokens=FAKE, prev_argmax=FAKE, status=FAKE,
                steps_taken=None, entropy=FAKE, argmax=FAKE, sampled=FAKE, selected=FAKE,
                committed=None, mean_entropy=None, workspace=FAKE, workspace_bytes=1 << 30,
                stream=0)
    args.update(kw)
    return eb.eb_sampler_step(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(L=0), eb.EB_ERR_INVALID),
    (dict(L=1025), eb.EB_ERR_INVALID),
    (dict(V=0), eb.EB_ERR_INVALID),
    (dict(B=-1), eb.EB_ERR_INVALID),
    (dict(dtype=7), eb.EB_ERR_INVALID),
    (dict(logits=None), eb.EB_ERR_INVALID),
    (dict(mask=None), eb.EB_ERR_INVALID),
    (dict(entropy=None), eb.EB_ERR_INVALID),
    (dict(workspace=None), eb.EB_ERR_WORKSPACE),
    (dict(workspace=FAKE + 8), eb.EB_ERR_WORKSPACE),
    (dict(workspace_bytes=16), eb.EB_ERR_WORKSPACE),
    (dict(step=48), eb.EB_ERR_INVALID),
    (dict(step=-1), eb.EB_ERR_INVALID),
    (dict(temperature=float("nan")), eb.EB_ERR_INVALID),
])
def test_invalid_arguments_rejected_before_launch(libs, kw, status):
    with pytest.raises(eb.EbError) as ei:
        _step(**kw)
    assert ei.value.status == status
    assert eb.lib().eb_last_error().decode()


def test_invalid_params_rejected(libs):
    for field, value in (("max_steps", 0), ("t_start", 0.0), ("t_end", -1.0), ("flags", 16),
                         ("flags", 0x80000001), ("entropy_bound", float("inf"))):
        p = eb.eb_default_params()
        setattr(p, field, value)
        with pytest.raises(eb.EbError) as ei:
            _step(params=p)
        assert ei.value.status == eb.EB_ERR_INVALID


def test_loop_rejects_missing_callback(libs):
    with pytest.raises(eb.EbError) as ei:
        eb.eb_sample_canvas(eb.eb_default_params(), 1, 16, 64, eb.EB_F32, 0, None, FAKE, 0, FAKE,
                            FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                            1 << 30, 0, 0)
    assert ei.value.status == eb.EB_ERR_INVALID


def test_status_strings(libs):
    for s in range(6):
        assert eb.lib().eb_status_string(s)


def test_block_driver_rejects_bad_arguments(libs):
    p = eb.eb_default_params()
    ws = eb.eb_blocks_workspace_bytes(2, 32, 64, eb.EB_F32)
    assert ws > eb.eb_workspace_bytes(2, 32, 64, eb.EB_F32) and ws % 256 == 0
    assert eb.eb_blocks_workspace_bytes(0, 32, 64, eb.EB_F32) == 0
    cases = [
        (dict(B=0), eb.EB_ERR_INVALID),
        (dict(n_blocks=-1), eb.EB_ERR_INVALID),
        (dict(logits_fn=0), eb.EB_ERR_INVALID),
        (dict(block_tokens=None), eb.EB_ERR_INVALID),
        (dict(workspace_bytes=16), eb.EB_ERR_WORKSPACE),
        (dict(workspace=FAKE + 8), eb.EB_ERR_WORKSPACE),
        (dict(L=1025, workspace_bytes=1 << 40), eb.EB_ERR_INVALID),
    ]
    for kw, status in cases:
        args = dict(params=p, B=2, L=32, V=64, dtype=eb.EB_F32, logits_fn=FAKE, user=None, logits=FAKE,
                    n_blocks=3, block_tokens=FAKE, block_steps=None, block_status=None,
                    workspace=FAKE, workspace_bytes=ws, poll_every=0, stream=0)
        args.update(kw)
        with pytest.raises(eb.EbError) as ei:
            eb.eb_sample_blocks(**args)
        assert ei.value.status == status, kw
