"""Seeded synthetic inputs for the pruned gated-MLP (POP) workloads.

This package only draws random numbers: it holds none of the FFN arithmetic.
The oracle tests, the GPU parity tests and the benchmark all take their inputs
from here, so both sides see identical bf16 bytes.

The recipe follows the workload shapes of the POP notes (papernotes.org, "POP:
Online Structural Pruning...", main-experiment and ablation tables: LLaMA-2-7B
FFN D=4096, D_FF=11008) and of batch-wise adaptive pruning (bittide page,
Section 3.1, eq. (1): gated MLP with Wg, W1 in R^{D_FF x D}, W2 in R^{D x D_FF}):

* weights Wg, W1, W2 ~ N(0, 0.02^2), rounded to bf16;
* a per-dimension scale c_d = exp(N(0, 1)) (log-normal, drawn once per run)
  that gives the activations outlier channels;
* prompt and decode activations x = N(0, 1) * c_d, rounded to bf16;
* MoE router logits ~ N(0, 1) (float64, not rounded).

Every tensor has its own counter stream (seed, tensor id), so a decode input
for step t can be drawn without drawing steps 0..t-1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()

# tensor kinds (bits 24..31 of the tensor id); the layer sits in bits 32..47
# and the decode step in bits 0..23.
KIND_WG, KIND_W1, KIND_W2, KIND_SCALE, KIND_PROMPT, KIND_DECODE, KIND_ROUTER, KIND_ROUTER_DECODE = range(1, 9)


def tensor_id(kind: int, layer: int = 0, step: int = 0) -> int:
    assert 0 <= step < (1 << 24) and 0 <= layer < (1 << 16)
    return (layer << 32) | (kind << 24) | step


def build(force: bool = False) -> str:
    """Compiles libsynth.so next to synth.c (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal_f64.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
            lib.synth_scaled_rows_bf16.argtypes = [u64, u64, u64, i64, i64, vp, vp]
            lib.synth_round_bf16.argtypes = [i64, vp, vp]
            for f in (lib.synth_normal_f64, lib.synth_normal_bf16, lib.synth_scaled_rows_bf16, lib.synth_round_bf16):
                f.restype = None
            _lib = lib
    return _lib


def normal_f64(seed: int, tid: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal_f64(seed, tid, offset, n, out.ctypes.data)
    return out


def normal_bf16(seed: int, tid: int, shape, std: float = 1.0, mean: float = 0.0, offset: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of mean + std * N(0, 1)."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(seed, tid, offset, out.size, mean, std, out.ctypes.data)
    return out


def round_bf16(a) -> np.ndarray:
    """Rounds float64 values to bf16 bit patterns (round to nearest even)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().synth_round_bf16(a.size, a.ctypes.data, out.ctypes.data)
    return out


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(u: np.ndarray) -> np.ndarray:
    return bf16_to_f32(u).astype(np.float64)


# ---------------------------------------------------------------- workload recipe

WEIGHT_STD = 0.02


def ffn_weights(seed: int, D: int, N: int, layer: int = 0):
    """(Wg [N, D], W1 [N, D], W2 [D, N]) as bf16 bit patterns, N(0, 0.02^2)."""
    Wg = normal_bf16(seed, tensor_id(KIND_WG, layer), (N, D), std=WEIGHT_STD)
    W1 = normal_bf16(seed, tensor_id(KIND_W1, layer), (N, D), std=WEIGHT_STD)
    W2 = normal_bf16(seed, tensor_id(KIND_W2, layer), (D, N), std=WEIGHT_STD)
    return Wg, W1, W2


def dim_scales(seed: int, D: int) -> np.ndarray:
    """Per-dimension log-normal scales c_d = exp(N(0, 1)), float64, shared by prompt and decode."""
    return np.exp(normal_f64(seed, tensor_id(KIND_SCALE), D))


def scaled_rows(seed: int, tid: int, rows: int, scales: np.ndarray) -> np.ndarray:
    scales = np.ascontiguousarray(scales, dtype=np.float64)
    cols = scales.shape[0]
    out = np.empty((rows, cols), dtype=np.uint16)
    _load().synth_scaled_rows_bf16(seed, tid, 0, rows, cols, scales.ctypes.data, out.ctypes.data)
    return out


def prompt(seed: int, M: int, scales: np.ndarray, layer: int = 0) -> np.ndarray:
    """Prompt activations X [M, D] = bf16(N(0, 1) * c_d)."""
    return scaled_rows(seed, tensor_id(KIND_PROMPT, layer), M, scales)


def decode_input(seed: int, step: int, B: int, scales: np.ndarray, layer: int = 0) -> np.ndarray:
    """Fresh decode activations x_t [B, D] = bf16(N(0, 1) * c_d) for step t."""
    return scaled_rows(seed, tensor_id(KIND_DECODE, layer, step), B, scales)


def router_logits(seed: int, tokens: int, E: int, step: int | None = None) -> np.ndarray:
    """MoE router logits [tokens, E] ~ N(0, 1) (float64)."""
    tid = tensor_id(KIND_ROUTER) if step is None else tensor_id(KIND_ROUTER_DECODE, 0, step)
    return normal_f64(seed, tid, tokens * E).reshape(tokens, E)
