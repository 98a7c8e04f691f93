"""Seeded synthetic inputs for the MoE layer workloads.

This module is shared by the CPU oracle side and the CUDA side: it holds the
workload shapes and the counter-based normal generator (``synth.cpp``), and
none of the layer's arithmetic.  Every tensor is drawn from its own stream
(seed, tensor id), so any slice (one expert's weights, a block of tokens) can
be regenerated on its own without drawing the rest.

Tensor ids: X=1, W_r=2, W13=3, W2=4, dY=5, sel_bias=6, W13_s=7, W2_s=8.
The skewed workload's logit_bias is a closed-form ramp, not a random draw.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cpp")
_LIB = os.path.join(_HERE, "libmoe_synth.so")
_lock = threading.Lock()
_lib = None

TID_X, TID_WR, TID_W13, TID_W2, TID_DY, TID_SEL_BIAS, TID_W13S, TID_W2S = 1, 2, 3, 4, 5, 6, 7, 8


def build(force: bool = False) -> str:
    """Compile synth.cpp into libmoe_synth.so (host code only, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, dbl, dbl, ctypes.c_void_p, i32]
            lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, dbl, dbl, ctypes.c_void_p, i32]
            lib.synth_words.argtypes = [u64, u64, u64, i64, ctypes.c_void_p]
            _lib = lib
    return _lib


def fill_normal_bf16(ptr: int, n: int, seed: int, tid: int, std: float, start: int = 0,
                     mean: float = 0.0, nthreads: int = 0) -> None:
    """Write n bf16 values (elements [start, start+n) of stream (seed, tid)) to host address ptr."""
    _load().synth_normal_bf16(seed, tid, start, n, mean, std, ptr, nthreads)


def fill_normal_f32(ptr: int, n: int, seed: int, tid: int, std: float, start: int = 0,
                    mean: float = 0.0, nthreads: int = 0) -> None:
    _load().synth_normal_f32(seed, tid, start, n, mean, std, ptr, nthreads)


def normal_bf16(n: int, seed: int, tid: int, std: float, start: int = 0) -> np.ndarray:
    """bf16 values as raw uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    fill_normal_bf16(out.ctypes.data, n, seed, tid, std, start)
    return out


def normal_f32(n: int, seed: int, tid: int, std: float, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    fill_normal_f32(out.ctypes.data, n, seed, tid, std, start)
    return out


def words(n: int, seed: int, tid: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_words(seed, tid, start, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and routing recipe of one synthetic MoE layer."""
    name: str
    T: int
    H: int
    E: int
    k: int
    F: int
    F_shared: int = 0
    score_fn: int = 0          # 0 softmax, 1 sigmoid
    renorm: int = 1
    gate_scale: float = 1.0
    n_group: int = 1
    topk_group: int = 1
    sel_bias: bool = False     # selection-only per-expert bias, N(0, 0.1)
    skew: bool = False         # Zipf-shaped logit_bias ramp
    fp8: bool = False
    x_std: float = 1.0
    w_std: float = 0.02
    wr_std: float = 0.02
    dy_std: float = 1.0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=128, E=8, k=2, F=256),
    "mixtral": Workload("mixtral", T=4096, H=4096, E=8, k=2, F=14336),
    "qwen3": Workload("qwen3", T=16384, H=4096, E=128, k=8, F=1536),
    "dsv3": Workload("dsv3", T=8192, H=7168, E=256, k=8, F=2048, F_shared=2048, score_fn=1,
                     renorm=1, gate_scale=2.5, n_group=8, topk_group=4, sel_bias=True),
    "dsv3-fp8": Workload("dsv3-fp8", T=8192, H=7168, E=256, k=8, F=2048, F_shared=2048, score_fn=1,
                         renorm=1, gate_scale=2.5, n_group=8, topk_group=4, sel_bias=True, fp8=True),
    "skew": Workload("skew", T=32768, H=4096, E=64, k=4, F=2048, skew=True),
    # profiling stand-in: the Mixtral-style layer with a narrower FFN (same per-tile
    # shapes along K for FC1, 0.4 GB of expert weights: larger than L2, small enough
    # for a multi-pass profiler capture)
    "mixtral-small": Workload("mixtral-small", T=4096, H=4096, E=8, k=2, F=2048),
    # profiling stand-in with the Qwen3-style layer's router (X of 134 MB, 128 experts,
    # top-8) and a narrow FFN, so that the whole layer holds a few GB
    "qwen3-small": Workload("qwen3-small", T=16384, H=4096, E=128, k=8, F=128),
    # profiling stand-in with the DeepSeek-V3-style layer's routing (the router weight's
    # spread scaled so the logits keep their spread at the narrower H) and therefore its
    # per-expert row counts, with a narrower H and FFN: 1.6 GB of expert weights
    "dsv3-mid": Workload("dsv3-mid", T=8192, H=2048, E=256, k=8, F=512, F_shared=512, score_fn=1,
                         renorm=1, gate_scale=2.5, n_group=8, topk_group=4, sel_bias=True,
                         wr_std=0.02 * math.sqrt(7168 / 2048)),
    # the same stand-in with FP8 expert GEMMs
    "dsv3-mid-fp8": Workload("dsv3-mid-fp8", T=8192, H=2048, E=256, k=8, F=512, F_shared=512, score_fn=1,
                             renorm=1, gate_scale=2.5, n_group=8, topk_group=4, sel_bias=True,
                             wr_std=0.02 * math.sqrt(7168 / 2048), fp8=True),
    # profiling stand-in with DeepSeek-V3-style routing and small expert segments
    # (about 64 rows per expert): 2.8 GB of expert weights, small enough for a full capture
    "dsv3-small": Workload("dsv3-small", T=2048, H=7168, E=256, k=8, F=256, F_shared=256, score_fn=1,
                           renorm=1, gate_scale=2.5, n_group=8, topk_group=4, sel_bias=True),
}

SKEW_BETA = 2.0
SKEW_EMPTY = 8


def skew_logit_bias(E: int, beta: float = SKEW_BETA, n_empty: int = SKEW_EMPTY) -> np.ndarray:
    """Zipf(1.2)-shaped preference ramp: -beta*1.2*ln(e+1); the last n_empty experts get -1e4."""
    b = np.array([-beta * 1.2 * math.log(e + 1) for e in range(E)], dtype=np.float32)
    if n_empty:
        b[E - n_empty:] = -1.0e4
    return b


def host_inputs(w: Workload, seed: int = 0, weights: bool = True) -> dict:
    """All inputs of workload w as numpy arrays (bf16 tensors as uint16 bit patterns).

    Meant for sizes that fit comfortably in host memory (the oracle-sized cases).
    """
    T, H, E, F = w.T, w.H, w.E, w.F
    d = {
        "X": normal_bf16(T * H, seed, TID_X, w.x_std).reshape(T, H),
        "W_r": normal_f32(E * H, seed, TID_WR, w.wr_std).reshape(E, H),
        "dY": normal_bf16(T * H, seed, TID_DY, w.dy_std).reshape(T, H),
        "logit_bias": skew_logit_bias(E) if w.skew else None,
        "sel_bias": normal_f32(E, seed, TID_SEL_BIAS, 0.1) if w.sel_bias else None,
    }
    if weights:
        d["W13"] = normal_bf16(E * 2 * F * H, seed, TID_W13, w.w_std).reshape(E, 2 * F, H)
        d["W2"] = normal_bf16(E * H * F, seed, TID_W2, w.w_std).reshape(E, H, F)
        if w.F_shared:
            Fs = w.F_shared
            d["W13_s"] = normal_bf16(2 * Fs * H, seed, TID_W13S, w.w_std).reshape(2 * Fs, H)
            d["W2_s"] = normal_bf16(H * Fs, seed, TID_W2S, w.w_std).reshape(H, Fs)
    return d
