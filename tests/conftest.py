import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """One line per parity report: the tie counts of every GPU-vs-oracle comparison (a tie is a
    case the contract exempts from bit-exactness: a top-2 perturbed-score gap below 1e-6 relative,
    a prefix sum within 1e-5 of the bound, an acceptance cut between entropies closer than 2e-5,
    or a mean entropy within 1e-6 of the stop threshold)."""
    try:
        from parity import REPORTS
    except Exception:
        return
    used = [(t, r) for t, r in REPORTS if r.rows or r.canvases]
    if not used:
        return
    terminalreporter.section("parity tie counts")
    lines = []
    for test, rep in used:
        name = test + (f" [{rep.label}]" if rep.label else "")
        lines.append(f"{name}: {rep.line()}")
    for line in lines:
        terminalreporter.write_line(line)
    tot = [sum(getattr(r, k) for _, r in used) for k in ("rows", "row_ties", "canvases", "canvas_ties")]
    terminalreporter.write_line(
        f"total: rows {tot[0]}, row ties {tot[1]}; canvases {tot[2]}, canvas ties {tot[3]}; "
        f"max |dH| {max(r.max_h_err for _, r in used):.3g}")
    path = os.environ.get("EB_TIE_REPORT")
    if path:
        with open(path, "w") as f:
            f.write("\n".join(lines) + "\n")
