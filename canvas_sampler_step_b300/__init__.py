"""Python binding of libeb_sampler.so, the B300 (sm_103a) Entropy-Bounded (EB) denoising
sampler of DiffusionGemma (model card, "Best practices" section 1, "Diffusion sampling
settings").

Argument marshalling only: every step of the sampler runs in the library's CUDA kernels.
Tensors are passed by ``data_ptr()``; PyTorch is used for device memory and streams.  The
entry points keep the C names and argument order of ``include/eb_sampler.h``.  There is no
CPU fallback: if the shared library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import CHECKS_LIB_PATH, build, build_checks  # noqa: F401
from .build import LIB_PATH as _DEFAULT_LIB_PATH

# The library this process loads: libeb_sampler.so, or another build of the same sources named
# by EB_SAMPLER_LIB (for instance the checked build, CHECKS_LIB_PATH).
LIB_PATH = os.environ.get("EB_SAMPLER_LIB") or _DEFAULT_LIB_PATH

EB_OK, EB_ERR_INVALID, EB_ERR_CUDA, EB_ERR_UNSUPPORTED, EB_ERR_WORKSPACE, EB_ERR_CALLBACK = range(6)
EB_F32, EB_BF16, EB_FP8_E4M3 = 0, 1, 2
EB_RUNNING, EB_STOP_ADAPTIVE, EB_STOP_COMPLETE, EB_STOP_CAP = 0, 1, 2, 3
EB_STATUS_NONFINITE = 0x100
EB_STATUS_TIMEOUT = 0x200
EB_SLOT_IDLE = 0x400
EB_STATUS_CHECK = 0x800
EB_FLAG_DIAG_STALL = 1
EB_FLAG_STOP_MASKED_ONLY = 2
EB_FLAG_FINALIZE_SAMPLED = 4
EB_FLAG_STOP_RAW_ENTROPY = 8

EXPORTED = ("eb_default_params", "eb_temperature", "eb_workspace_bytes", "eb_sampler_step",
            "eb_sample_canvas", "eb_status_string", "eb_last_error", "eb_set_profile_events",
            "eb_unembed_workspace_bytes", "eb_unembed_sample", "eb_unembed_logits",
            "eb_sampler_step_noalloc", "eb_blocks_workspace_bytes", "eb_sample_blocks",
            "eb_checks_enabled", "eb_check_word")


class EbParams(ctypes.Structure):
    """Mirror of eb_params."""
    _fields_ = [("max_steps", ctypes.c_int32), ("t_start", ctypes.c_float),
                ("t_end", ctypes.c_float), ("entropy_bound", ctypes.c_float),
                ("stop_entropy", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("seed", ctypes.c_uint64)]


LOGITS_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


class EbError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: the CUDA library must be built "
                           "(canvas_sampler_step_b300.build()); there is no CPU path")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.eb_default_params.argtypes = [ctypes.POINTER(EbParams)]
    L.eb_default_params.restype = i32
    L.eb_temperature.argtypes = [ctypes.POINTER(EbParams), i32]
    L.eb_temperature.restype = ctypes.c_float
    L.eb_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.eb_workspace_bytes.restype = sz
    L.eb_sampler_step.argtypes = ([ctypes.POINTER(EbParams), i32, i32, i32, i32, P, i32, ctypes.c_float]
                                  + [P] * 11 + [P, sz, P])
    L.eb_sampler_step.restype = i32
    L.eb_sample_canvas.argtypes = ([ctypes.POINTER(EbParams), i32, i32, i32, i32, P, P, P, i32]
                                   + [P] * 11 + [P, sz, i32, ctypes.POINTER(ctypes.c_int), P])
    L.eb_sample_canvas.restype = i32
    L.eb_status_string.argtypes = [i32]
    L.eb_status_string.restype = ctypes.c_char_p
    L.eb_last_error.argtypes = []
    L.eb_last_error.restype = ctypes.c_char_p
    L.eb_checks_enabled.argtypes = []
    L.eb_checks_enabled.restype = i32
    L.eb_check_word.argtypes = [i32]
    L.eb_check_word.restype = ctypes.c_uint32
    L.eb_set_profile_events.argtypes = [P, P]
    L.eb_set_profile_events.restype = i32
    L.eb_unembed_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.eb_unembed_workspace_bytes.restype = sz
    L.eb_unembed_sample.argtypes = ([ctypes.POINTER(EbParams), i32, i32, i32, i32, P, P, i32,
                                     ctypes.c_float] + [P] * 11 + [P, sz, P])
    L.eb_unembed_sample.restype = i32
    L.eb_unembed_logits.argtypes = [i32, i32, i32, P, P, P, P]
    L.eb_unembed_logits.restype = i32
    L.eb_sampler_step_noalloc.argtypes = ([ctypes.POINTER(EbParams), i32, i32, i32, i32, P, i32,
                                           ctypes.c_float] + [P] * 11 + [P])
    L.eb_sampler_step_noalloc.restype = i32
    L.eb_blocks_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.eb_blocks_workspace_bytes.restype = sz
    L.eb_sample_blocks.argtypes = ([ctypes.POINTER(EbParams), i32, i32, i32, i32, P, P, P, i32, P, P, P,
                                    P, sz, i32, ctypes.POINTER(ctypes.c_int), P])
    L.eb_sample_blocks.restype = i32
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check(status: int):
    if status != EB_OK:
        raise EbError(status, lib().eb_last_error().decode() or lib().eb_status_string(status).decode())


def eb_checks_enabled() -> bool:
    """True for the checked debug build (device bounds checks, EB_STATUS_CHECK)."""
    return bool(lib().eb_checks_enabled())


def eb_check_word(clear: bool = False) -> int:
    """The checked build's device word of failed bounds checks (0 in the normal build)."""
    return int(lib().eb_check_word(1 if clear else 0))


def eb_default_params(seed: int = 0, **overrides) -> EbParams:
    p = EbParams()
    _check(lib().eb_default_params(ctypes.byref(p)))
    p.seed = seed
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


def eb_temperature(params: EbParams, step: int) -> float:
    return float(lib().eb_temperature(ctypes.byref(params), step))


def eb_workspace_bytes(B: int, L: int, V: int, dtype: int) -> int:
    return int(lib().eb_workspace_bytes(B, L, V, dtype))


def eb_sampler_step(params: EbParams, B: int, L: int, V: int, dtype: int, logits, step: int,
                    temperature: float, mask, tokens, prev_argmax, status, steps_taken,
                    entropy, argmax, sampled, selected, committed, mean_entropy,
                    workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib().eb_sampler_step(ctypes.byref(params), B, L, V, dtype, _ptr(logits), step,
                                 float(temperature), _ptr(mask), _ptr(tokens), _ptr(prev_argmax),
                                 _ptr(status), _ptr(steps_taken), _ptr(entropy), _ptr(argmax),
                                 _ptr(sampled), _ptr(selected), _ptr(committed),
                                 _ptr(mean_entropy), _ptr(workspace), workspace_bytes,
                                 _stream(stream)))


def eb_sample_canvas(params: EbParams, B: int, L: int, V: int, dtype: int, logits_fn, user,
                     logits, start_step: int, mask, tokens, prev_argmax, status, steps_taken,
                     committed_per_step, mean_entropy_per_step, entropy, argmax, sampled,
                     selected, workspace, workspace_bytes: int, poll_every: int = 0,
                     stream=None) -> int:
    """``logits_fn`` is a C function address (int) or a LOGITS_FN instance.  Returns the
    number of sampler steps enqueued."""
    fn = logits_fn if isinstance(logits_fn, int) else ctypes.cast(logits_fn, ctypes.c_void_p).value
    ran = ctypes.c_int(0)
    _check(lib().eb_sample_canvas(ctypes.byref(params), B, L, V, dtype, fn, _ptr(user),
                                  _ptr(logits), start_step, _ptr(mask), _ptr(tokens),
                                  _ptr(prev_argmax), _ptr(status), _ptr(steps_taken),
                                  _ptr(committed_per_step), _ptr(mean_entropy_per_step),
                                  _ptr(entropy), _ptr(argmax), _ptr(sampled), _ptr(selected),
                                  _ptr(workspace), workspace_bytes, poll_every,
                                  ctypes.byref(ran), _stream(stream)))
    return ran.value


def eb_blocks_workspace_bytes(B: int, L: int, V: int, dtype: int) -> int:
    return int(lib().eb_blocks_workspace_bytes(B, L, V, dtype))


def eb_sample_blocks(params: EbParams, B: int, L: int, V: int, dtype: int, logits_fn, user, logits,
                     n_blocks: int, block_tokens, block_steps, block_status, workspace,
                     workspace_bytes: int, poll_every: int = 0, stream=None) -> int:
    """Block driver over B slots; ``logits_fn`` is a C function address of an
    eb_block_logits_fn.  Returns the number of iterations enqueued."""
    fn = logits_fn if isinstance(logits_fn, int) else ctypes.cast(logits_fn, ctypes.c_void_p).value
    ran = ctypes.c_int(0)
    _check(lib().eb_sample_blocks(ctypes.byref(params), B, L, V, dtype, fn, _ptr(user), _ptr(logits),
                                  n_blocks, _ptr(block_tokens), _ptr(block_steps), _ptr(block_status),
                                  _ptr(workspace), workspace_bytes, poll_every, ctypes.byref(ran),
                                  _stream(stream)))
    return ran.value


def eb_sampler_step_noalloc(params: EbParams, B: int, L: int, V: int, dtype: int, logits,
                            step: int, temperature: float, mask, tokens, prev_argmax, status,
                            steps_taken, entropy, argmax, sampled, selected, committed,
                            mean_entropy, stream=None) -> None:
    """eb_sampler_step with the library's fixed scratch instead of a caller workspace (for
    callers that cannot allocate device memory; B * L <= 8192, calls must not overlap)."""
    _check(lib().eb_sampler_step_noalloc(ctypes.byref(params), B, L, V, dtype, _ptr(logits), step,
                                         float(temperature), _ptr(mask), _ptr(tokens),
                                         _ptr(prev_argmax), _ptr(status), _ptr(steps_taken),
                                         _ptr(entropy), _ptr(argmax), _ptr(sampled),
                                         _ptr(selected), _ptr(committed), _ptr(mean_entropy),
                                         _stream(stream)))


def eb_unembed_workspace_bytes(B: int, L: int, K: int, V: int) -> int:
    return int(lib().eb_unembed_workspace_bytes(B, L, K, V))


def eb_unembed_sample(params: EbParams, B: int, L: int, K: int, V: int, h, W, step: int,
                      temperature: float, mask, tokens, prev_argmax, status, steps_taken,
                      entropy, argmax, sampled, selected, committed, mean_entropy,
                      workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib().eb_unembed_sample(ctypes.byref(params), B, L, K, V, _ptr(h), _ptr(W), step,
                                   float(temperature), _ptr(mask), _ptr(tokens),
                                   _ptr(prev_argmax), _ptr(status), _ptr(steps_taken),
                                   _ptr(entropy), _ptr(argmax), _ptr(sampled), _ptr(selected),
                                   _ptr(committed), _ptr(mean_entropy), _ptr(workspace),
                                   workspace_bytes, _stream(stream)))


def eb_unembed_logits(M: int, K: int, V: int, h, W, logits, stream=None) -> None:
    _check(lib().eb_unembed_logits(M, K, V, _ptr(h), _ptr(W), _ptr(logits), _stream(stream)))


def eb_set_profile_events(k1_begin, k1_end) -> None:
    """torch.cuda.Event pair (or raw cudaEvent_t ints) around the next row-statistics launch."""
    def ev(e):
        if e is None or isinstance(e, int):
            return e or None
        return e.cuda_event or None
    _check(lib().eb_set_profile_events(ev(k1_begin), ev(k1_end)))


class Canvas:
    """Device buffers of B canvases (allocated with torch): state, per-step outputs and
    the workspace.  ``mask`` [B, L] (u8) gives the initial mask (default: all masked)."""

    def __init__(self, B: int, L: int, V: int, dtype: int, device="cuda", mask=None,
                 max_steps: int = 48):
        import torch
        self.B, self.L, self.V, self.dtype = B, L, V, dtype
        dev = torch.device(device)
        if mask is None:
            self.mask = torch.ones((B, L), dtype=torch.uint8, device=dev)
        else:
            self.mask = torch.as_tensor(mask, dtype=torch.uint8).to(dev).clone()
        self.tokens = torch.where(self.mask.bool(), -1, 0).to(torch.int32)
        self.prev_argmax = torch.full((B, L), -1, dtype=torch.int32, device=dev)
        self.status = torch.zeros(B, dtype=torch.int32, device=dev)
        self.steps_taken = torch.zeros(B, dtype=torch.int32, device=dev)
        self.entropy = torch.zeros((B, L), dtype=torch.float32, device=dev)
        self.argmax = torch.zeros((B, L), dtype=torch.int32, device=dev)
        self.sampled = torch.zeros((B, L), dtype=torch.int32, device=dev)
        self.selected = torch.zeros((B, L), dtype=torch.uint8, device=dev)
        self.committed = torch.zeros(B, dtype=torch.int32, device=dev)
        self.mean_entropy = torch.zeros(B, dtype=torch.float32, device=dev)
        self.committed_per_step = torch.zeros((B, max_steps), dtype=torch.int32, device=dev)
        self.mean_entropy_per_step = torch.full((B, max_steps), float("nan"),
                                                dtype=torch.float32, device=dev)
        self.ws_bytes = eb_workspace_bytes(B, L, V, dtype)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)

    def step(self, params: EbParams, logits, step: int, temperature: float = 0.0, stream=None):
        eb_sampler_step(params, self.B, self.L, self.V, self.dtype, logits, step, temperature,
                        self.mask, self.tokens, self.prev_argmax, self.status, self.steps_taken,
                        self.entropy, self.argmax, self.sampled, self.selected, self.committed,
                        self.mean_entropy, self.workspace, self.ws_bytes, stream)

    def unembed_step(self, params: EbParams, h, W, K: int, step: int, temperature: float = 0.0,
                     workspace=None, stream=None):
        """One fused unembedding + sampler step: logits = h W never leave the chip.  Uses a
        workspace of eb_unembed_workspace_bytes (allocated on first use unless given)."""
        import torch
        need = eb_unembed_workspace_bytes(self.B, self.L, K, self.V)
        if workspace is None:
            if getattr(self, "_uws", None) is None or self._uws.numel() < need:
                self._uws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.mask.device)
            workspace = self._uws
        eb_unembed_sample(params, self.B, self.L, K, self.V, h, W, step, temperature, self.mask,
                          self.tokens, self.prev_argmax, self.status, self.steps_taken,
                          self.entropy, self.argmax, self.sampled, self.selected,
                          self.committed, self.mean_entropy, workspace, need, stream)

    def run(self, params: EbParams, logits_fn, user, logits, start_step: int = 0,
            poll_every: int = 0, stream=None) -> int:
        return eb_sample_canvas(params, self.B, self.L, self.V, self.dtype, logits_fn, user,
                                logits, start_step, self.mask, self.tokens, self.prev_argmax,
                                self.status, self.steps_taken, self.committed_per_step,
                                self.mean_entropy_per_step, self.entropy, self.argmax,
                                self.sampled, self.selected, self.workspace, self.ws_bytes,
                                poll_every, stream)
