"""CPU oracle of the dropless top-k MoE layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never calls it and shares no code with it.

The arithmetic lives in ``moe_oracle.cpp`` (plain C++, double accumulation);
this module only builds it with g++ and marshals numpy arrays through ctypes.
See the header of ``moe_oracle.cpp`` for the readings of the pages it takes
and for what pins each part.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


class OraCfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32), ("F_shared", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("renorm", ctypes.c_int32),
                ("gate_scale", ctypes.c_double), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("group_score", ctypes.c_int32),
                ("align", ctypes.c_int32), ("BM", ctypes.c_int32), ("mirror", ctypes.c_int32),
                ("nthreads", ctypes.c_int32), ("fp8", ctypes.c_int32), ("gated", ctypes.c_int32)]


def build(force: bool = False) -> str:
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
            _lib = ctypes.CDLL(build())
            _lib.ora_dispatch.restype = ctypes.c_int
            _lib.ora_dispatch_capacity.restype = ctypes.c_int
            _lib.ora_dispatch_priority.restype = ctypes.c_int
    return _lib


def cfg(w, mirror: bool = True, align: int = 128, BM: int = 128, nthreads: int = 0,
        group_score: int = 0, fp8: bool | None = None, gated: bool = False) -> OraCfg:
    """Oracle configuration from a moe_synth.Workload (fp8 defaults to the workload's flag).
    gated: routed experts take their gate before the down projection (the memory-efficient
    path's form of the same function; it only moves the mirror-mode roundings)."""
    f8 = getattr(w, "fp8", False) if fp8 is None else fp8
    return OraCfg(w.T, w.H, w.E, w.k, w.F, w.F_shared, w.score_fn, w.renorm, float(w.gate_scale),
                  w.n_group, w.topk_group, group_score, align, BM, 1 if mirror else 0, nthreads, 1 if f8 else 0,
                  1 if gated else 0)


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint16)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def router(c: OraCfg, X, W_r, logit_bias=None):
    """logits = X W_r^T (+ logit_bias) and scores (softmax over E or sigmoid), both float64 [T,E]."""
    logits = np.empty((c.T, c.E), np.float64)
    scores = np.empty((c.T, c.E), np.float64)
    _load().ora_router(ctypes.byref(c), _p(_u16(X)), _p(_f32(W_r)), _p(_f32(logit_bias)),
                       _p(logits), _p(scores))
    return logits, scores


def select(c: OraCfg, logits, scores, sel_bias=None):
    """Top-k experts per token, [T,k] int32.  float32 inputs select in float32, float64 in float64."""
    idx = np.empty((c.T, c.k), np.int32)
    if logits.dtype == np.float32:
        _load().ora_select_f32(ctypes.byref(c), _p(_f32(logits)), _p(_f32(scores)), _p(_f32(sel_bias)),
                               _p(idx))
    else:
        _load().ora_select_f64(ctypes.byref(c), _p(np.ascontiguousarray(logits, np.float64)),
                               _p(np.ascontiguousarray(scores, np.float64)), _p(_f32(sel_bias)), _p(idx))
    return idx


def gates(c: OraCfg, logits, topk_idx):
    g = np.empty((c.T, c.k), np.float64)
    _load().ora_gates(ctypes.byref(c), _p(np.ascontiguousarray(logits, np.float64)),
                      _p(np.ascontiguousarray(topk_idx, np.int32)), _p(g))
    return g


def dispatch(c: OraCfg, topk_idx, R: int | None = None, capacity: int | None = None, priority=None):
    """counts [E], offsets [E+1], tile_offsets [E+1], row_id_map [T,k], slot_src [R].

    capacity: each expert keeps at most `capacity` assignments, dropped ones get
    row_id_map -1 and counts are the kept counts.  Without `priority` the first ones
    in token order are kept; with priority [T,k] the ones of largest priority (equal
    priorities to the earlier assignment), their rows still in token order."""
    if R is None:
        R = c.T * c.k + c.E * (c.align - 1)
    counts = np.empty(c.E, np.int32)
    offsets = np.empty(c.E + 1, np.int32)
    tiles = np.empty(c.E + 1, np.int32)
    rim = np.empty((c.T, c.k), np.int32)
    src = np.full(R, -2, np.int32)
    cap = 2 ** 31 - 1 if capacity is None else int(capacity)
    pr = None if priority is None else np.ascontiguousarray(priority, np.float64)
    rc = _load().ora_dispatch_priority(ctypes.byref(c), _p(np.ascontiguousarray(topk_idx, np.int32)),
                                       ctypes.c_int32(cap), _p(pr), _p(counts), _p(offsets), _p(tiles), _p(rim),
                                       _p(src), ctypes.c_int64(R))
    if rc != 0:
        raise ValueError("permuted rows exceed R")
    return dict(counts=counts, offsets=offsets, tile_offsets=tiles, row_id_map=rim, slot_src=src)


def tokens(c: OraCfg, inp: dict, topk_idx, logits, gates_, tok_list=None, want_bwd=True, kept=None):
    """Per-token forward/backward: Y [n,H], dX [n,H], dgates [n,k], dlogits [n,E] (float64).

    kept: optional [T,k] mask; an assignment with kept == 0 (dropped by capacity)
    adds nothing to Y and gets no gradient."""
    if tok_list is None:
        tok_list = np.arange(c.T, dtype=np.int64)
    tok_list = np.ascontiguousarray(tok_list, np.int64)
    n = len(tok_list)
    Y = np.empty((n, c.H), np.float64)
    dX = np.empty((n, c.H), np.float64) if want_bwd else None
    dg = np.empty((n, c.k), np.float64) if want_bwd else None
    dl = np.empty((n, c.E), np.float64) if want_bwd else None
    kp = None if kept is None else np.ascontiguousarray(kept, np.int32)
    _load().ora_tokens_kept(ctypes.byref(c), _p(_u16(inp["X"])), _p(_u16(inp["W13"])), _p(_u16(inp["W2"])),
                       _p(_u16(inp.get("W13_s"))), _p(_u16(inp.get("W2_s"))), _p(_f32(inp["W_r"])),
                       _p(np.ascontiguousarray(topk_idx, np.int32)),
                       _p(np.ascontiguousarray(logits, np.float64)),
                       _p(np.ascontiguousarray(gates_, np.float64)),
                       _p(_u16(inp["dY"])) if want_bwd else None, ctypes.c_int64(n), _p(tok_list),
                       _p(Y), _p(dX), _p(dg), _p(dl), _p(kp))
    return dict(Y=Y, dX=dX, dgates=dg, dlogits=dl)


def expert_wgrad(c: OraCfg, inp: dict, topk_idx, gates_, expert: int, kept=None):
    """dW13 [2F,H] and dW2 [H,F] (float64) of one expert; expert=-1 is the shared expert.
    kept: optional [T,k] mask of the assignments that were not dropped."""
    F = c.F_shared if expert < 0 else c.F
    dW13 = np.empty((2 * F, c.H), np.float64)
    dW2 = np.empty((c.H, F), np.float64)
    kp = None if kept is None else np.ascontiguousarray(kept, np.int32)
    _load().ora_expert_wgrad_kept(ctypes.byref(c), _p(_u16(inp["X"])), _p(_u16(inp["W13"])), _p(_u16(inp["W2"])),
                                  _p(_u16(inp.get("W13_s"))), _p(_u16(inp.get("W2_s"))),
                                  _p(np.ascontiguousarray(topk_idx, np.int32)),
                                  _p(np.ascontiguousarray(gates_, np.float64)), _p(_u16(inp["dY"])),
                                  ctypes.c_int32(expert), _p(dW13), _p(dW2), _p(kp))
    return dW13, dW2


def expert_wgrad_cols(c: OraCfg, inp: dict, topk_idx, gates_, expert: int, cols, kept=None):
    """The weight gradients of one expert at a few FFN indices f in `cols`, equal to the
    corresponding entries of expert_wgrad at a fraction of its cost: dW13 rows f and F+f
    ([2*len(cols), H]: gate rows, then up rows) and dW2 columns f ([H, len(cols)])."""
    cols = np.ascontiguousarray(cols, np.int32)
    nc = len(cols)
    dW13r = np.empty((2 * nc, c.H), np.float64)
    dW2c = np.empty((c.H, nc), np.float64)
    kp = None if kept is None else np.ascontiguousarray(kept, np.int32)
    _load().ora_expert_wgrad_cols(ctypes.byref(c), _p(_u16(inp["X"])), _p(_u16(inp["W13"])), _p(_u16(inp["W2"])),
                                  _p(_u16(inp.get("W13_s"))), _p(_u16(inp.get("W2_s"))),
                                  _p(np.ascontiguousarray(topk_idx, np.int32)),
                                  _p(np.ascontiguousarray(gates_, np.float64)), _p(_u16(inp["dY"])),
                                  ctypes.c_int32(expert), ctypes.c_int32(nc), _p(cols), _p(dW13r), _p(dW2c), _p(kp))
    return dW13r, dW2c


def router_dlogits(c: OraCfg, logits, topk_idx, gates_, dgates):
    """dlogits [T,E] (float64): the gates' exact gradient w.r.t. the logits for the given
    selection, applied to dgates [T,k]."""
    dl = np.empty((c.T, c.E), np.float64)
    _load().ora_router_dlogits(ctypes.byref(c), _p(np.ascontiguousarray(logits, np.float64)),
                               _p(np.ascontiguousarray(topk_idx, np.int32)),
                               _p(np.ascontiguousarray(gates_, np.float64)),
                               _p(np.ascontiguousarray(dgates, np.float64)), _p(dl))
    return dl


def router_wgrad(c: OraCfg, X, dlogits):
    """dW_r [E,H] and dlogit_bias [E] (float64) from the dlogits of all T tokens."""
    dWr = np.empty((c.E, c.H), np.float64)
    dlb = np.empty(c.E, np.float64)
    _load().ora_router_wgrad(ctypes.byref(c), _p(_u16(X)), _p(np.ascontiguousarray(dlogits, np.float64)),
                             _p(dWr), _p(dlb))
    return dWr, dlb


def e4m3(x):
    """FP8 E4M3 round-to-nearest-even of float64 values (|x| <= 448)."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty_like(x)
    _load().ora_e4m3(_p(x), _p(out), ctypes.c_int64(x.size))
    return out


def qdq_blocks(x, blk=128):
    """Quantize-dequantize consecutive blocks of `blk` values with power-of-two block scales."""
    x = np.ascontiguousarray(x, np.float64).ravel()
    out = np.empty_like(x)
    _load().ora_qdq_blocks(_p(x), _p(out), ctypes.c_int64(x.size), ctypes.c_int(blk))
    return out


def qdq_weights(W):
    """128x128 block quantize-dequantize of a stack of bf16 matrices (returned as bf16 bits)."""
    W = np.ascontiguousarray(W, np.uint16)
    rows, cols = W.shape[-2], W.shape[-1]
    nmat = int(np.prod(W.shape[:-2])) if W.ndim > 2 else 1
    out = np.empty_like(W)
    _load().ora_qdq_weight_blocks(_p(W), ctypes.c_int64(nmat), ctypes.c_int(rows), ctypes.c_int(cols), _p(out))
    return out


def fp8_inputs(inp: dict) -> dict:
    """The inputs with every expert weight replaced by its 128x128-block FP8 quantize-dequantize."""
    out = dict(inp)
    for k in ["W13", "W2", "W13_s", "W2_s"]:
        if out.get(k) is not None:
            out[k] = qdq_weights(out[k])
    return out


def round_bf16(x):
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty_like(x)
    _load().ora_round_bf16(_p(x), _p(out), ctypes.c_int64(x.size))
    return out


def full_layer(w, inp: dict, mirror: bool = True, sel_scores=None, nthreads: int = 0, capacity=None,
               drop_by_gate: bool = False, gated: bool = False):
    """Whole-layer forward and backward for every token and every expert (small cases).

    sel_scores: optional (logits_f32, scores_f32) from another implementation;
    when given, the selection runs on them in float32 (identical-scores rule).
    """
    c = cfg(w, mirror=mirror, nthreads=nthreads, gated=gated)
    if c.fp8:
        inp = fp8_inputs(inp)
    logits, scores = router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    if sel_scores is None:
        idx = select(c, logits, scores, inp.get("sel_bias"))
    else:
        idx = select(c, sel_scores[0], sel_scores[1], inp.get("sel_bias"))
    g = gates(c, logits, idx)
    d = dispatch(c, idx, capacity=capacity, priority=g if drop_by_gate else None)
    kept = None if capacity is None else (d["row_id_map"] >= 0).astype(np.int32)
    tk = tokens(c, inp, idx, logits, g, kept=kept)
    dW13 = np.empty((c.E, 2 * c.F, c.H))
    dW2 = np.empty((c.E, c.H, c.F))
    for e in range(c.E):
        dW13[e], dW2[e] = expert_wgrad(c, inp, idx, g, e, kept=kept)
    dWr, dlb = router_wgrad(c, inp["X"], tk["dlogits"])
    out = dict(logits=logits, scores=scores, topk_idx=idx, gates=g, Y=tk["Y"], dX=tk["dX"],
               dgates=tk["dgates"], dlogits=tk["dlogits"], dW13=dW13, dW2=dW2, dW_r=dWr,
               dlogit_bias=dlb, **d)
    if c.F_shared:
        out["dW13_s"], out["dW2_s"] = expert_wgrad(c, inp, idx, g, -1)
    return out
