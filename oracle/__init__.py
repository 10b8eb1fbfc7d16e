"""CPU oracle of the Entropy-Bounded (EB) denoising sampler (DiffusionGemma).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It is the plain, slow statement
of the sampler's rules (DiffusionGemma model card, "Best practices" section 1,
"Diffusion sampling settings"), written in C (binary64, OpenMP over rows) in
``eb_oracle.c`` and wrapped here with ctypes.  It shares no code with the CUDA library.

Functions
---------
philox4x32_10(ctr, key)    -- the counter-based generator (Salmon et al., SC'11)
gumbel_word / uniform / gumbel -- the per-entry Gumbel noise the sampler draws
temperature(step, ...)     -- linear 0.8 -> 0.4 logit-shaping schedule
row(x, T, masked, ...)     -- entropy, argmax and Gumbel-max sample of one row
select(H, mask, bound)     -- entropy-bounded prefix selection of one canvas
step(...)                  -- one full sampler step over B canvases (stats, stop test,
                              selection, re-mask, complete / cap)
unembed_logits(h, W)       -- the decoder's unembedding product h W in binary64 (the logits
                              the fused path feeds to the sampler without storing them)
run_loop(...)              -- the <= 48-step denoising loop with per-canvas stop
run_blocks(...)            -- the block driver's result: every block through its own loop

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` except the
readings the pages leave open (shaped-entropy stop statistic, mean over all positions,
argmax finalisation at stop / cap), which are "parity unpinned" by the pages.  The two
alternative readings selectable by ``Params.flags`` (stop statistics over the masked positions
only, sampled-token finalisation) are pinned by hand-built cases like the default ones.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "eb_oracle.c")
_LIB = os.path.join(_HERE, "libeb_oracle.so")

RUNNING, ADAPTIVE, COMPLETE, CAP = 0, 1, 2, 3
DTYPE_F32, DTYPE_BF16, DTYPE_F64, DTYPE_E4M3 = 0, 1, 2, 3

_lib = None


def build(force: bool = False) -> str:
    """Compile eb_oracle.c into libeb_oracle.so (gcc -O2, no fast-math, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i32, i64, u64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
    lib.eb_oracle_philox4x32_10.argtypes = [P, P, P]
    lib.eb_oracle_philox4x32_10.restype = None
    lib.eb_oracle_gumbel_word.argtypes = [u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64]
    lib.eb_oracle_gumbel_word.restype = ctypes.c_uint32
    lib.eb_oracle_uniform.argtypes = [ctypes.c_uint32]
    lib.eb_oracle_uniform.restype = f64
    lib.eb_oracle_gumbel.argtypes = [ctypes.c_uint32]
    lib.eb_oracle_gumbel.restype = f64
    lib.eb_oracle_temperature.argtypes = [ctypes.c_int, ctypes.c_int, f64, f64]
    lib.eb_oracle_temperature.restype = f64
    lib.eb_oracle_row.argtypes = [P, ctypes.c_int, i64, f64, ctypes.c_int, u64, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, P, P, P, P]
    lib.eb_oracle_row.restype = None
    lib.eb_oracle_select.argtypes = [ctypes.c_int, P, P, f64, P, P, P]
    lib.eb_oracle_select.restype = ctypes.c_int
    lib.eb_oracle_step.argtypes = [ctypes.c_int, ctypes.c_int, i64, ctypes.c_int, P,
                                   ctypes.c_int, f64, ctypes.c_int, f64, f64, f64, f64, u64,
                                   ctypes.c_uint32, P,
                                   P, P, P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.eb_oracle_step.restype = None
    lib.eb_oracle_e4m3_value.argtypes = [ctypes.c_int]
    lib.eb_oracle_e4m3_value.restype = ctypes.c_double
    lib.eb_oracle_num_threads.argtypes = []
    lib.eb_oracle_num_threads.restype = ctypes.c_int
    lib.eb_oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.eb_oracle_set_num_threads.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().eb_oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().eb_oracle_set_num_threads(int(n))


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().eb_oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def gumbel_word(seed: int, b: int, p: int, s: int, v: int) -> int:
    return int(_load().eb_oracle_gumbel_word(seed, b, p, s, v))


def uniform(w: int) -> float:
    return float(_load().eb_oracle_uniform(w))


def gumbel(w: int) -> float:
    return float(_load().eb_oracle_gumbel(w))


def temperature(step: int, max_steps: int = 48, t_start: float = 0.8, t_end: float = 0.4) -> float:
    return float(_load().eb_oracle_temperature(step, max_steps, t_start, t_end))


_schedule = temperature


def _logits_array(x: np.ndarray):
    """Accepts float32, float64, bfloat16 carried as uint16 bits, or e4m3 codes as uint8."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, DTYPE_F32
    if x.dtype == np.uint16:
        return x, DTYPE_BF16
    if x.dtype == np.float64:
        return x, DTYPE_F64
    if x.dtype == np.uint8:
        return x, DTYPE_E4M3
    raise TypeError(f"logits must be float32, float64, uint16 (bf16 bits) or uint8 (e4m3 codes), got {x.dtype}")


def e4m3_value(code: int) -> float:
    """Exact value of one OCP FP8 e4m3 code (NaN for S.1111.111)."""
    return float(_load().eb_oracle_e4m3_value(int(code)))


def row(x: np.ndarray, T: float, masked: bool, seed: int = 0, b: int = 0, p: int = 0, s: int = 0):
    """(H, A, Y, gap) of one row of logits; see eb_oracle_row."""
    x, dt = _logits_array(x)
    H = np.zeros(1, np.float64)
    A = np.zeros(1, np.int32)
    Y = np.zeros(1, np.int32)
    gap = np.zeros(1, np.float64)
    _load().eb_oracle_row(_ptr(x), dt, x.shape[-1], float(T), int(bool(masked)), seed, b, p, s,
                          _ptr(H), _ptr(A), _ptr(Y), _ptr(gap))
    return float(H[0]), int(A[0]), int(Y[0]), float(gap[0])


def select(H: np.ndarray, mask: np.ndarray, bound: float = 0.1):
    """Entropy-bounded selection of one canvas -> (accept[L] u8, k, sum_margin, order_margin)."""
    H = np.ascontiguousarray(H, dtype=np.float64)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    L = H.shape[0]
    acc = np.zeros(L, np.uint8)
    sm = np.zeros(1, np.float64)
    om = np.zeros(1, np.float64)
    k = _load().eb_oracle_select(L, _ptr(H), _ptr(mask), float(bound), _ptr(acc), _ptr(sm), _ptr(om))
    return acc, int(k), float(sm[0]), float(om[0])


@dataclass
class Params:
    """Sampler settings; defaults are the model card's recommended values."""
    max_steps: int = 48
    t_start: float = 0.8
    t_end: float = 0.4
    entropy_bound: float = 0.1
    stop_entropy: float = 0.005
    seed: int = 0
    flags: int = 0            # reading variants: STOP_MASKED_ONLY, FINALIZE_SAMPLED, STOP_RAW_ENTROPY


# Reading variants of the stop / finalisation rules (Params.flags bits)
STOP_MASKED_ONLY = 2          # stop statistics over the still-masked positions only
FINALIZE_SAMPLED = 4          # positions finalised at stop / cap take the sampled token
STOP_RAW_ENTROPY = 8          # stop statistics on the entropy of the raw logits (T = 1)


@dataclass
class State:
    """Canvas state for B canvases of L positions."""
    mask: np.ndarray          # [B, L] u8, 1 = masked
    tokens: np.ndarray        # [B, L] i32, -1 while masked
    prev_argmax: np.ndarray   # [B, L] i32, -1 before the first step
    status: np.ndarray        # [B] i32
    steps_taken: np.ndarray   # [B] i32

    @staticmethod
    def fresh(B: int, L: int, mask: np.ndarray | None = None) -> "State":
        m = np.ones((B, L), np.uint8) if mask is None else np.ascontiguousarray(mask, np.uint8).copy()
        tok = np.where(m == 1, -1, 0).astype(np.int32)
        return State(m, tok, np.full((B, L), -1, np.int32), np.zeros(B, np.int32),
                     np.zeros(B, np.int32))

    def copy(self) -> "State":
        return State(self.mask.copy(), self.tokens.copy(), self.prev_argmax.copy(),
                     self.status.copy(), self.steps_taken.copy())


@dataclass
class StepResult:
    H: np.ndarray
    A: np.ndarray
    Y: np.ndarray
    gap: np.ndarray
    selected: np.ndarray
    committed: np.ndarray
    mean_entropy: np.ndarray
    sum_margin: np.ndarray
    order_margin: np.ndarray
    stop_margin: np.ndarray
    temperature: float = field(default=0.0)


def step(logits: np.ndarray, state: State, step_index: int, params: Params = Params(),
         temperature: float = 0.0, canvas_ids=None) -> StepResult:
    """One EB sampler step over logits [B, L, V]; updates ``state`` in place.  ``canvas_ids``
    ([B] ints, default 0..B-1) are the canvases' ids in the Gumbel noise's Philox counter."""
    x, dt = _logits_array(logits)
    B, L, V = x.shape
    st = state
    for name in ("mask", "tokens", "prev_argmax", "status", "steps_taken"):
        arr = getattr(st, name)
        if not arr.flags["C_CONTIGUOUS"]:
            setattr(st, name, np.ascontiguousarray(arr))
    H = np.zeros((B, L), np.float64)
    A = np.zeros((B, L), np.int32)
    Y = np.zeros((B, L), np.int32)
    gap = np.zeros((B, L), np.float64)
    sel = np.zeros((B, L), np.uint8)
    committed = np.zeros(B, np.int32)
    meanH = np.zeros(B, np.float64)
    sm = np.zeros(B, np.float64)
    om = np.zeros(B, np.float64)
    stm = np.zeros(B, np.float64)
    ids = None if canvas_ids is None else np.ascontiguousarray(canvas_ids, np.int32)
    if ids is not None and ids.shape != (B,):
        raise ValueError("canvas_ids must have one entry per canvas")
    _load().eb_oracle_step(B, L, V, dt, _ptr(x), int(step_index), float(temperature),
                           params.max_steps, params.t_start, params.t_end, params.entropy_bound,
                           params.stop_entropy, params.seed, params.flags,
                           _ptr(ids) if ids is not None else None,
                           _ptr(st.mask), _ptr(st.tokens), _ptr(st.prev_argmax), _ptr(st.status),
                           _ptr(st.steps_taken), _ptr(H), _ptr(A), _ptr(Y), _ptr(gap), _ptr(sel),
                           _ptr(committed), _ptr(meanH), _ptr(sm), _ptr(om), _ptr(stm))
    T = temperature if temperature > 0 else _schedule(
        step_index, params.max_steps, params.t_start, params.t_end)
    return StepResult(H, A, Y, gap, sel, committed, meanH, sm, om, stm, T)


def run_loop(logits_fn, B: int, L: int, params: Params = Params(), state: State | None = None,
             start_step: int = 0, on_step=None, canvas_ids=None) -> State:
    """The denoising loop: for s in [start_step, max_steps) while any canvas runs,
    logits_fn(s, state) -> [B, L, V] logits, then one sampler step.  ``on_step(s, result,
    state)`` sees every step's result (for lockstep comparison)."""
    st = State.fresh(B, L) if state is None else state
    for s in range(start_step, params.max_steps):
        if not np.any(st.status == RUNNING):
            break
        res = step(logits_fn(s, st), st, s, params, canvas_ids=canvas_ids)
        if on_step is not None:
            on_step(s, res, st)
    return st


def run_blocks(block_logits_fn, n_blocks: int, L: int, params: Params = Params()):
    """What the block driver computes, block by block: block k is a fresh all-masked canvas of L
    positions, with k as its Philox canvas id, run through the denoising loop on its own
    (block_logits_fn(k, s) -> [L, V] logits of block k at its step s).  The slots and the order
    in which they take blocks do not enter.  Returns (tokens [n, L], steps [n], status [n])."""
    tokens = np.zeros((n_blocks, L), np.int32)
    steps = np.zeros(n_blocks, np.int32)
    status = np.zeros(n_blocks, np.int32)
    for k in range(n_blocks):
        st = run_loop(lambda s, _st, k=k: block_logits_fn(k, s)[None], 1, L, params,
                      canvas_ids=[k])
        tokens[k], steps[k], status[k] = st.tokens[0], st.steps_taken[0], st.status[0]
    return tokens, steps, status


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact binary64 values of bfloat16 bit patterns (uint16)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def unembed_logits(h_bits: np.ndarray, W_bits: np.ndarray) -> np.ndarray:
    """logits = h W in binary64 for bf16 h [M, K] and W [K, V] (bit patterns).  The sampler
    step consumes the decoder's full-vocabulary logits of every canvas position (DiffusionGemma
    model card, "Best practices" section 1); the fused path computes them as this product.
    numpy's matmul serves as the (library) dot-product step; every product of two bfloat16
    values is exact in binary64, so the only rounding is binary64 accumulation."""
    return bf16_to_f64(h_bits) @ bf16_to_f64(W_bits)
