"""Shared helpers of the GPU-vs-oracle parity tests.

Tolerances (the sampler step's contract):
  * entropy H within 1e-4 nats (absolute);
  * argmax, sampled token, selected positions, mask, tokens, status and stop step
    bit-exact, except tie cases, which are counted: a masked row whose two best
    perturbed scores differ by < 1e-6 relative (the oracle's `gap`), a canvas where a
    prefix sum of sorted entropies lies within 1e-5 of the bound, a canvas whose
    acceptance cut separates two entropies closer than 2e-5 (a rounding difference can
    swap them), and a canvas whose mean entropy is within 1e-6 of the stop threshold while
    its argmax is stable.
"""
from __future__ import annotations

import os
from dataclasses import dataclass, field

import numpy as np
import torch

import canvas_sampler_step_b300 as eb
import eb_synth
import eb_synth.device as synth_dev
import oracle

H_TOL = 1e-4
GAP_TOL = 1e-6
SUM_TOL = 1e-5
ORDER_TOL = 2e-5
STOP_TOL = 1e-6


def to_device_logits(x: np.ndarray, device="cuda") -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def host_state(c: eb.Canvas) -> dict:
    torch.cuda.synchronize()
    return {k: getattr(c, k).cpu().numpy() for k in
            ("mask", "tokens", "prev_argmax", "status", "steps_taken", "entropy", "argmax",
             "sampled", "selected", "committed", "mean_entropy")}


# Every Report made while a test runs is kept here with that test's id; conftest.py prints one
# line per report at the end of the session (and writes them to $EB_TIE_REPORT if set), so
# that the tie counts of every parity case are reported.
REPORTS: list = []


@dataclass
class Report:
    rows: int = 0
    canvases: int = 0
    row_ties: int = 0
    canvas_ties: int = 0
    tied_canvases: set = field(default_factory=set)
    max_h_err: float = 0.0
    label: str = ""

    def __post_init__(self):
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        REPORTS.append((test, self))

    def line(self) -> str:
        return (f"rows {self.rows}, row ties {self.row_ties}; canvases {self.canvases}, canvas ties "
                f"{self.canvas_ties}; max |dH| {self.max_h_err:.3g}")


def compare_step(g: dict, res: oracle.StepResult, ost: oracle.State, running_before: np.ndarray,
                 rep: Report, ctx: str = "", atie: np.ndarray | None = None,
                 ytie_extra: np.ndarray | None = None) -> set:
    """Compare one GPU step (host copies ``g``) with the oracle's result ``res`` / state
    ``ost``.  Returns the set of canvases that hit a tie at this step.  ``atie`` / ``ytie_extra``
    ([B, L] bool, optional) mark rows where the GPU's logits themselves carry a rounding
    error (the fused product) large enough to swap the argmax / the sample: those rows are
    counted as ties too, and a canvas holding one is not compared beyond its rows."""
    B, L = res.H.shape
    tied = set()
    for b in range(B):
        if not running_before[b]:
            continue
        rep.canvases += 1
        rep.rows += L
        herr = np.abs(g["entropy"][b].astype(np.float64) - res.H[b])
        rep.max_h_err = max(rep.max_h_err, float(herr.max()))
        assert herr.max() <= H_TOL, f"{ctx} canvas {b}: entropy error {herr.max():.3g}"
        a_ok = g["argmax"][b] == res.A[b]
        if atie is not None:
            rep.row_ties += int((atie[b] & ~a_ok).sum())
            a_ok |= atie[b]
        assert a_ok.all(), f"{ctx} canvas {b}: argmax differs at {np.nonzero(~a_ok)[0][:8]}"
        ytie = res.gap[b] < GAP_TOL
        if ytie_extra is not None:
            ytie = ytie | ytie_extra[b]
        rep.row_ties += int(ytie.sum())
        ok_y = (g["sampled"][b] == res.Y[b]) | ytie
        assert ok_y.all(), f"{ctx} canvas {b}: sampled token differs at {np.nonzero(~ok_y)[0][:8]}"
        ctie = (res.sum_margin[b] < SUM_TOL or res.order_margin[b] < ORDER_TOL
                or res.stop_margin[b] < STOP_TOL)
        if atie is not None and (atie[b] & (g["argmax"][b] != res.A[b])).any():
            ctie = True     # a swapped argmax feeds the stop test and the finalisation
        if ctie:
            rep.canvas_ties += 1
            tied.add(b)
            continue
        # selection / re-mask / commit / stop: exact except tokens at sampled-token ties
        for k in ("selected", "mask"):
            ref = res.selected[b] if k == "selected" else ost.mask[b]
            assert np.array_equal(g[k][b], ref), f"{ctx} canvas {b}: {k} differs"
        tok_ok = (g["tokens"][b] == ost.tokens[b]) | ytie
        assert tok_ok.all(), f"{ctx} canvas {b}: tokens differ at {np.nonzero(~tok_ok)[0][:8]}"
        assert g["status"][b] == ost.status[b], f"{ctx} canvas {b}: status {g['status'][b]} vs {ost.status[b]}"
        if ost.status[b] != oracle.RUNNING:
            assert g["steps_taken"][b] == ost.steps_taken[b], f"{ctx} canvas {b}: stop step differs"
        assert g["committed"][b] == res.committed[b], f"{ctx} canvas {b}: committed count differs"
    rep.tied_canvases |= tied
    return tied


def params_pair(seed=0, **kw):
    """Matching (GPU, oracle) parameter objects."""
    gp = eb.eb_default_params(seed=seed)
    op = oracle.Params(seed=seed)
    for k, v in kw.items():
        setattr(gp, k, v)
        setattr(op, k, v)
    # the oracle runs the schedule in binary64 from the binary32 endpoints the GPU uses
    op.t_start = float(np.float32(gp.t_start))
    op.t_end = float(np.float32(gp.t_end))
    op.entropy_bound = float(np.float32(gp.entropy_bound))
    op.stop_entropy = float(np.float32(gp.stop_entropy))
    return gp, op


def device_logits(cfg: eb_synth.Peaked, step: int, status=None) -> torch.Tensor:
    dt = {"f32": torch.float32, "bf16": torch.int16, "fp8": torch.uint8}[cfg.dtype]
    out = torch.empty((cfg.B, cfg.L, cfg.V), dtype=dt, device="cuda")
    synth_dev.logits(synth_dev.Recipe.of(cfg), step, out, status)
    return out
