"""ctypes binding of libeb_synth.so: the CUDA side of the seeded input generator (see the
package docstring and include/eb_synth.h).  It produces the same bits as the numpy
generator in ``eb_synth``."""
from __future__ import annotations

import ctypes
import os

from . import Peaked

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
SRC = os.path.join(_HERE, "csrc", "eb_synth.cu")
HDR = os.path.join(_ROOT, "include", "eb_synth.h")
LIB_PATH = os.path.join(_HERE, "libeb_synth.so")
MAX_B = 64
EXPORTED = ("eb_synth_logits", "eb_synth_logits_callback", "eb_synth_unembed_inputs",
            "eb_synth_slot_logits", "eb_synth_block_callback")


def build(force: bool = False, verbose: bool = False) -> str:
    from canvas_sampler_step_b300.build import nvcc_shared
    return nvcc_shared(SRC, LIB_PATH, os.path.join(_ROOT, "include"), [HDR], force=force,
                       verbose=verbose)


class Recipe(ctypes.Structure):
    """Mirror of eb_synth_recipe."""
    _fields_ = [("B", ctypes.c_int32), ("L", ctypes.c_int32), ("V", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("sigma", ctypes.c_float), ("base_lo", ctypes.c_float),
                ("base_scale", ctypes.c_float), ("growth", ctypes.c_float * MAX_B),
                ("seed", ctypes.c_uint64 * MAX_B)]

    @staticmethod
    def of(cfg: Peaked) -> "Recipe":
        if cfg.B > MAX_B:
            raise ValueError(f"B={cfg.B} > {MAX_B}")
        r = Recipe()
        r.B, r.L, r.V = cfg.B, cfg.L, cfg.V
        r.dtype = {"f32": 0, "bf16": 1, "fp8": 2}[cfg.dtype]
        r.sigma, r.base_lo, r.base_scale = cfg.sigma, cfg.base_lo, cfg.base_scale
        for b in range(cfg.B):
            r.growth[b] = cfg.growth[b]
            r.seed[b] = int(cfg.seeds[b])
        return r


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with eb_synth.device.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        L.eb_synth_logits.argtypes = [ctypes.POINTER(Recipe), ctypes.c_int, P, P, P]
        L.eb_synth_logits.restype = ctypes.c_int
        L.eb_synth_logits_callback.argtypes = [P, ctypes.c_int, P, P, P, P]
        L.eb_synth_logits_callback.restype = ctypes.c_int
        L.eb_synth_unembed_inputs.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_float, ctypes.c_float, P, P, P]
        L.eb_synth_unembed_inputs.restype = ctypes.c_int
        L.eb_synth_slot_logits.argtypes = [ctypes.POINTER(Recipe), ctypes.c_int, P, P, P, P]
        L.eb_synth_slot_logits.restype = ctypes.c_int
        L.eb_synth_block_callback.argtypes = [P, ctypes.c_int, P, P, P, P, P]
        L.eb_synth_block_callback.restype = ctypes.c_int
        _lib = L
    return _lib


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    return stream if isinstance(stream, int) else (stream.cuda_stream or None)


def logits(recipe: Recipe, step: int, out, status=None, stream=None) -> None:
    """Fill the device tensor ``out`` [B, L, V] (float32, or bfloat16/int16/uint16 bits)."""
    rc = lib().eb_synth_logits(ctypes.byref(recipe), step,
                               status.data_ptr() if status is not None else None,
                               out.data_ptr(), _stream(stream))
    if rc != 0:
        raise RuntimeError(f"eb_synth_logits failed ({rc})")


def callback_address() -> int:
    """Address of eb_synth_logits_callback (an eb_logits_fn; user = Recipe*)."""
    return ctypes.cast(lib().eb_synth_logits_callback, ctypes.c_void_p).value


def unembed_inputs(seed: int, M: int, K: int, V: int, sigma_w: float, bias: float, h, W,
                   stream=None) -> None:
    rc = lib().eb_synth_unembed_inputs(seed, M, K, V, sigma_w, bias, h.data_ptr(), W.data_ptr(),
                                       _stream(stream))
    if rc != 0:
        raise RuntimeError(f"eb_synth_unembed_inputs failed ({rc})")


def slot_logits(recipe: Recipe, slot_block, slot_step, out, stream=None) -> None:
    """Fill slot b of ``out`` [B_slots, L, V] with recipe canvas slot_block[b] at slot_step[b]."""
    rc = lib().eb_synth_slot_logits(ctypes.byref(recipe), int(slot_block.numel()), slot_block.data_ptr(),
                                    slot_step.data_ptr(), out.data_ptr(), _stream(stream))
    if rc != 0:
        raise RuntimeError(f"eb_synth_slot_logits failed ({rc})")


def block_callback_address() -> int:
    """Address of eb_synth_block_callback (an eb_block_logits_fn; user = Recipe*)."""
    return ctypes.cast(lib().eb_synth_block_callback, ctypes.c_void_p).value
