"""Parity cases run on the checked debug build of the sampler library (-DEB_CHECKS).

Run as a child process by ``test_gpu_checks.py`` with EB_SAMPLER_LIB naming the checked
library, so that this process loads it instead of the normal build.  It runs step cases of the
streaming paths (vector, scalar, e4m3, uniform partition, the full-size single step) and a
short loop next to the oracle, exactly as the parity tests do, and then requires that no
device bounds check failed: the check word is 0 and no canvas carries EB_STATUS_CHECK.
Prints "checked build ok" on success; any failure raises.
"""
import os
import sys

import numpy as np
import torch

_TESTS = os.path.dirname(os.path.abspath(__file__))
sys.path[:0] = [os.path.dirname(_TESTS), _TESTS]

import canvas_sampler_step_b300 as eb  # noqa: E402
import eb_synth  # noqa: E402
import test_gpu_parity as tp  # noqa: E402
from parity import Report, compare_step  # noqa: E402


def main():
    assert eb.eb_checks_enabled(), f"{eb.LIB_PATH} is not the checked build"
    eb.eb_check_word(clear=True)
    statuses = []
    for cfg, step, density in tp.CASES:
        rng = np.random.default_rng(step + cfg.V)
        mask = (rng.random((cfg.B, cfg.L)) < density).astype(np.uint8)
        mask[:, 0] = 1
        g, res, ost, running = tp._run_step(cfg, step, mask=mask)
        compare_step(g, res, ost, running, Report(), ctx=f"checked build, V={cfg.V}")
        statuses.append(g["status"])
    # the uniform partition: 17 x 256 rows, more than the weighted partition takes
    cfg = eb_synth.Peaked(17, 256, 1024, "f32", 3.0, 0.0, 4.0, (0.0,) * 17, tuple(range(17)))
    g, res, ost, running = tp._run_step(cfg, 0)
    compare_step(g, res, ost, running, Report(), ctx="checked build, uniform partition")
    statuses.append(g["status"])
    # the full-size single step
    cfg = eb_synth.cfg1(0)
    g, res, ost, running = tp._run_step(cfg, 0, mask=eb_synth.cfg1_mask(0), seed=0, temperature=0.8)
    compare_step(g, res, ost, running, Report(), ctx="checked build, single step")
    statuses.append(g["status"])
    # a short loop of a mixed batch, every step next to the oracle
    cfg = eb_synth.Peaked(4, 64, 2048, "bf16", 3.0, 0.0, 4.0, (0.1, 0.2, 0.4, 0.8), (0, 1, 2, 3))
    rep, hist, *_ = tp._lockstep(cfg, label="checked build, loop")
    statuses.extend(h["status"] for h in hist)
    torch.cuda.synchronize()
    word = eb.eb_check_word()
    assert word == 0, f"bounds checks failed: word {word:#x}"
    for st in statuses:
        assert not (np.asarray(st) & eb.EB_STATUS_CHECK).any(), st
    print("checked build ok")


if __name__ == "__main__":
    main()
