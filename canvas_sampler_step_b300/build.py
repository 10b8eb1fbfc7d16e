"""In-tree build of libeb_sampler.so for sm_103a (nvcc; no JIT cache)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "eb_sampler.cu")
HDR = os.path.join(ROOT, "include", "eb_sampler.h")
LIB_PATH = os.path.join(PKG, "libeb_sampler.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
         "-Xlinker", "-rpath,/usr/local/cuda/lib64"]


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def nvcc_shared(src: str, out: str, include_dir: str, deps, extra=(), force: bool = False,
                verbose: bool = False) -> str:
    if not force and not _stale(out, list(deps) + [src]):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, *FLAGS, "-I", include_dir, *extra, "-o", tmp, src]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


CHECKS_LIB_PATH = os.path.join(PKG, "libeb_sampler_checks.so")


def build(force: bool = False, verbose: bool = False) -> str:
    return nvcc_shared(SRC, LIB_PATH, os.path.join(ROOT, "include"), [HDR], force=force,
                       verbose=verbose)


def build_checks(force: bool = False, verbose: bool = False) -> str:
    """The checked debug build (-DEB_CHECKS): device bounds checks that record a status bit
    instead of trapping (eb_check_word in the header)."""
    return nvcc_shared(SRC, CHECKS_LIB_PATH, os.path.join(ROOT, "include"), [HDR], extra=["-DEB_CHECKS"],
                       force=force, verbose=verbose)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
