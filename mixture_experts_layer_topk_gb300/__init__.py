"""Python binding of the GB300 MoE layer library (libmoe_gb300.so).

The functions named like the C entry points (moe_router_topk, moe_permute,
moe_grouped_swiglu_mlp, moe_unpermute_combine and their _bwd calls) only
marshal arguments: they pass tensor data pointers and the current CUDA stream
to the C ABI declared in include/moe.h and raise MoeError on a non-OK status.
Every step of the layer runs in the library's CUDA kernels; there is no other
implementation behind these calls, and loading fails loudly when the library
cannot be built or loaded.

MoELayer is a convenience that owns the device buffers of one layer and runs
the calls in order (forward: route, permute, grouped SwiGLU MLP, combine;
backward: the same in reverse).
"""
from __future__ import annotations

import ctypes
import math
import threading
from dataclasses import dataclass

import torch

from . import build as _build

__all__ = ["MoeConfig", "MoeError", "load", "MoELayer", "config_from", "moe_set_wait_limit_ns",
           "moe_get_wait_limit_ns"] + [
    "moe_router_topk", "moe_permute", "moe_grouped_swiglu_mlp", "moe_unpermute_combine",
    "moe_unpermute_combine_bwd", "moe_grouped_swiglu_mlp_bwd", "moe_router_topk_bwd", "moe_permute_bwd",
    "moe_workspace_size", "moe_workspace_init", "moe_read_device_error", "moe_max_rows", "moe_permute_noalloc", "moe_permute_capacity",
    "moe_grouped_swiglu_mlp_gated", "moe_grouped_swiglu_mlp_bwd_gated", "moe_grouped_swiglu_mlp_gather",
    "moe_grouped_swiglu_mlp_bwd_gather"]

EXPORTED = ["moe_status_string", "moe_max_rows", "moe_workspace_size", "moe_workspace_init",
            "moe_read_device_error", "moe_router_topk", "moe_permute", "moe_grouped_swiglu_mlp",
            "moe_unpermute_combine", "moe_unpermute_combine_bwd", "moe_grouped_swiglu_mlp_bwd",
            "moe_router_topk_bwd", "moe_permute_bwd", "moe_permute_noalloc", "moe_fp8_workspace_size",
            "moe_quantize_weights_fp8", "moe_grouped_swiglu_mlp_fp8", "moe_grouped_swiglu_mlp_bwd_fp8",
            "moe_router_replay", "moe_permute_capacity", "moe_grouped_swiglu_mlp_gated",
            "moe_grouped_swiglu_mlp_bwd_gated", "moe_grouped_swiglu_mlp_gather", "moe_grouped_swiglu_mlp_bwd_gather",
            "moe_set_wait_limit_ns", "moe_get_wait_limit_ns"]


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("F", ctypes.c_int32), ("F_shared", ctypes.c_int32), ("score_fn", ctypes.c_int32),
                ("renorm", ctypes.c_int32), ("gate_scale", ctypes.c_float), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("group_score", ctypes.c_int32), ("align", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({_status_text(status)})")


_lock = threading.Lock()
_lib = None


def load(build: bool = True):
    """Load libmoe_gb300.so (building it first when sources are newer).  Raises on failure."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            lib = ctypes.CDLL(path)
            vp = ctypes.c_void_p
            cfgp = ctypes.POINTER(MoeConfig)
            sigs = {
                "moe_max_rows": [cfgp, ctypes.POINTER(ctypes.c_int64)],
                "moe_workspace_size": [cfgp, ctypes.POINTER(ctypes.c_size_t)],
                "moe_workspace_init": [cfgp, vp, vp],
                "moe_read_device_error": [vp, ctypes.POINTER(ctypes.c_int32), vp],
                "moe_router_topk": [cfgp] + [vp] * 11,
                "moe_permute": [cfgp] + [vp] * 10,
                "moe_grouped_swiglu_mlp": [cfgp] + [vp] * 16,
                "moe_unpermute_combine": [cfgp] + [vp] * 6,
                "moe_unpermute_combine_bwd": [cfgp] + [vp] * 9,
                "moe_grouped_swiglu_mlp_bwd": [cfgp] + [vp] * 25,
                "moe_router_topk_bwd": [cfgp] + [vp] * 12,
                "moe_permute_bwd": [cfgp] + [vp] * 6,
                "moe_permute_noalloc": [cfgp] + [vp] * 9,
                "moe_router_replay": [cfgp] + [vp] * 11,
                "moe_permute_capacity": [cfgp, vp, vp, vp, ctypes.c_int32] + [vp] * 9,
                "moe_grouped_swiglu_mlp_gated": [cfgp] + [vp] * 18,
                "moe_grouped_swiglu_mlp_gather": [cfgp] + [vp] * 16,
                "moe_grouped_swiglu_mlp_bwd_gather": [cfgp] + [vp] * 25,
                "moe_grouped_swiglu_mlp_bwd_gated": [cfgp] + [vp] * 29,
                "moe_fp8_workspace_size": [cfgp, ctypes.POINTER(ctypes.c_size_t)],
                "moe_quantize_weights_fp8": [cfgp] + [vp] * 13,
                "moe_grouped_swiglu_mlp_fp8": [cfgp] + [vp] * 20,
                "moe_grouped_swiglu_mlp_bwd_fp8": [cfgp] + [vp] * 29,
            }
            for name, args in sigs.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            lib.moe_status_string.argtypes = [ctypes.c_int]
            lib.moe_status_string.restype = ctypes.c_char_p
            lib.moe_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.moe_set_wait_limit_ns.restype = None
            lib.moe_get_wait_limit_ns.argtypes = []
            lib.moe_get_wait_limit_ns.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def _status_text(s):
    try:
        return load(build=False).moe_status_string(s).decode()
    except Exception:
        return "?"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(*ts):
    for t in ts:
        if t is not None and not isinstance(t, int) and not t.is_cuda:
            raise ValueError("MoE library buffers must be CUDA tensors")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _call(name, cfg, *args):
    rc = getattr(load(), name)(ctypes.byref(cfg), *args)
    if rc != 0:
        raise MoeError(name, rc)


def config_from(w, align: int = 128, group_score: int = 0) -> MoeConfig:
    """MoeConfig from any object with the workload fields (T, H, E, k, F, ...)."""
    return MoeConfig(w.T, w.H, w.E, w.k, w.F, getattr(w, "F_shared", 0), getattr(w, "score_fn", 0),
                     getattr(w, "renorm", 1), float(getattr(w, "gate_scale", 1.0)), getattr(w, "n_group", 1),
                     getattr(w, "topk_group", 1), group_score, align, 0)


def moe_set_wait_limit_ns(ns: int) -> None:
    """Limit of every pipeline wait inside the tensor-core kernels (default 4e9 ns); a wait
    that runs out sets MOE_ERR_TIMEOUT and the kernel unwinds.  0: one test per wait."""
    load().moe_set_wait_limit_ns(int(ns))


def moe_get_wait_limit_ns() -> int:
    return int(load().moe_get_wait_limit_ns())


def moe_max_rows(cfg: MoeConfig) -> int:
    R = ctypes.c_int64()
    _call("moe_max_rows", cfg, ctypes.byref(R))
    return R.value


def moe_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _call("moe_workspace_size", cfg, ctypes.byref(n))
    return n.value


def moe_workspace_init(cfg, ws, stream=None):
    _dev(ws)
    _call("moe_workspace_init", cfg, _ptr(ws), _stream(stream))


def moe_read_device_error(ws, stream=None) -> int:
    v = ctypes.c_int32()
    rc = load().moe_read_device_error(_ptr(ws), ctypes.byref(v), _stream(stream))
    if rc != 0:
        raise MoeError("moe_read_device_error", rc)
    return v.value


def moe_router_topk(cfg, X, W_r, logit_bias, sel_bias, logits, scores, topk_idx, gates, counts, ws, stream=None):
    _dev(X, W_r, logit_bias, sel_bias, logits, scores, topk_idx, gates, counts, ws)
    _call("moe_router_topk", cfg, *map(_ptr, (X, W_r, logit_bias, sel_bias, logits, scores, topk_idx, gates, counts,
                                               ws)), _stream(stream))


def moe_router_replay(cfg, X, W_r, logit_bias, topk_in, logits, scores, topk_idx, gates, counts, ws=None,
                      stream=None):
    _dev(X, W_r, logit_bias, topk_in, logits, scores, topk_idx, gates, counts, ws)
    _call("moe_router_replay", cfg, *map(_ptr, (X, W_r, logit_bias, topk_in, logits, scores, topk_idx, gates, counts,
                                                 ws)), _stream(stream))


def moe_permute(cfg, X, topk_idx, counts, offsets, tile_offsets, row_id_map, slot_src, Xperm, ws, stream=None):
    _dev(X, topk_idx, counts, offsets, tile_offsets, row_id_map, slot_src, Xperm, ws)
    _call("moe_permute", cfg, *map(_ptr, (X, topk_idx, counts, offsets, tile_offsets, row_id_map, slot_src, Xperm,
                                           ws)), _stream(stream))


def moe_permute_capacity(cfg, X, topk_idx, counts, capacity, priority, kept_counts, offsets, tile_offsets,
                         row_id_map, slot_src, Xperm, ws, stream=None):
    """moe_permute with a per-expert capacity.  priority None: each expert keeps its
    first `capacity` assignments in token order; priority [T,k] fp32: the `capacity`
    of largest priority (ties to the earlier assignment).  kept_counts [E] receives
    min(counts, capacity); row_id_map is -1 for a dropped assignment."""
    _dev(X, topk_idx, counts, priority, kept_counts, offsets, tile_offsets, row_id_map, slot_src, Xperm, ws)
    _call("moe_permute_capacity", cfg, _ptr(X), _ptr(topk_idx), _ptr(counts), ctypes.c_int32(int(capacity)),
          *map(_ptr, (priority, kept_counts, offsets, tile_offsets, row_id_map, slot_src, Xperm, ws)),
          _stream(stream))


def moe_permute_noalloc(cfg, X, topk_idx, counts, offsets, tile_offsets, row_id_map, slot_src, Xperm, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device
    memory (the scratch lives in a static device array inside the library; see
    include/moe.h for its size limit and the rule that calls must not overlap)."""
    _dev(X, topk_idx, counts, offsets, tile_offsets, row_id_map, slot_src, Xperm)
    _call("moe_permute_noalloc", cfg, *map(_ptr, (X, topk_idx, counts, offsets, tile_offsets, row_id_map, slot_src,
                                                   Xperm)), _stream(stream))


def moe_grouped_swiglu_mlp(cfg, Xperm, offsets, tile_offsets, W13, W2, GU, A, Yperm, X=None, W13_s=None, W2_s=None,
                           GU_s=None, A_s=None, Yshared=None, ws=None, stream=None):
    _dev(Xperm, offsets, tile_offsets, W13, W2, GU, A, Yperm, X, W13_s, W2_s, GU_s, A_s, Yshared, ws)
    _call("moe_grouped_swiglu_mlp", cfg, *map(_ptr, (Xperm, offsets, tile_offsets, W13, W2, GU, A, Yperm, X, W13_s,
                                                      W2_s, GU_s, A_s, Yshared, ws)), _stream(stream))


def moe_grouped_swiglu_mlp_gated(cfg, Xperm, offsets, tile_offsets, slot_src, gates, W13, W2, GU, A, Yperm, X=None,
                                 W13_s=None, W2_s=None, GU_s=None, A_s=None, Yshared=None, ws=None, stream=None):
    """The expert MLP with each permuted row's gate applied before FC2 (A and Yperm are
    gated); combine with gates=None."""
    ts = (Xperm, offsets, tile_offsets, slot_src, gates, W13, W2, GU, A, Yperm, X, W13_s, W2_s, GU_s, A_s, Yshared,
          ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_gated", cfg, *map(_ptr, ts), _stream(stream))


def moe_grouped_swiglu_mlp_bwd_gated(cfg, Xperm, offsets, tile_offsets, counts, slot_src, row_id_map, gates, W13, W2,
                                     GU, dYperm, dGU, dXperm, A, dW13, dW2, dgates, X=None, dY=None, W13_s=None,
                                     W2_s=None, GU_s=None, A_s=None, dGU_s=None, dX_shared=None, dW13_s=None,
                                     dW2_s=None, ws=None, stream=None):
    """Backward of the gated MLP: recomputes the activations from GU into A and writes dgates."""
    ts = (Xperm, offsets, tile_offsets, counts, slot_src, row_id_map, gates, W13, W2, GU, dYperm, dGU, dXperm, A,
          dW13, dW2, dgates, X, dY, W13_s, W2_s, GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s, ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_bwd_gated", cfg, *map(_ptr, ts), _stream(stream))


def moe_grouped_swiglu_mlp_gather(cfg, X, slot_src, offsets, tile_offsets, W13, W2, GU, A, Yperm, W13_s=None,
                                  W2_s=None, GU_s=None, A_s=None, Yshared=None, ws=None, stream=None):
    """The expert MLP with FC1 gathering the token rows of X through slot_src (no Xperm)."""
    ts = (X, slot_src, offsets, tile_offsets, W13, W2, GU, A, Yperm, W13_s, W2_s, GU_s, A_s, Yshared, ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_gather", cfg, *map(_ptr, ts), _stream(stream))


def moe_grouped_swiglu_mlp_bwd_gather(cfg, X, slot_src, offsets, tile_offsets, counts, W13, W2, GU, A, dYperm, dGU,
                                      dXperm, dW13, dW2, dY=None, W13_s=None, W2_s=None, GU_s=None, A_s=None,
                                      dGU_s=None, dX_shared=None, dW13_s=None, dW2_s=None, ws=None, stream=None):
    """Backward of the gathered-rows MLP (FC1's weight gradient gathers X along K)."""
    ts = (X, slot_src, offsets, tile_offsets, counts, W13, W2, GU, A, dYperm, dGU, dXperm, dW13, dW2, dY, W13_s,
          W2_s, GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s, ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_bwd_gather", cfg, *map(_ptr, ts), _stream(stream))


def moe_unpermute_combine(cfg, Yperm, row_id_map, gates, Yshared, Y, stream=None):
    _dev(Yperm, row_id_map, gates, Yshared, Y)
    _call("moe_unpermute_combine", cfg, *map(_ptr, (Yperm, row_id_map, gates, Yshared, Y)), _stream(stream))


def moe_unpermute_combine_bwd(cfg, dY, Yperm, row_id_map, gates, offsets, counts, dYperm, dgates, stream=None):
    _dev(dY, Yperm, row_id_map, gates, offsets, counts, dYperm, dgates)
    _call("moe_unpermute_combine_bwd", cfg, *map(_ptr, (dY, Yperm, row_id_map, gates, offsets, counts, dYperm,
                                                         dgates)), _stream(stream))


def moe_grouped_swiglu_mlp_bwd(cfg, Xperm, offsets, tile_offsets, counts, W13, W2, GU, A, dYperm, dGU, dXperm, dW13,
                               dW2, X=None, dY=None, W13_s=None, W2_s=None, GU_s=None, A_s=None, dGU_s=None,
                               dX_shared=None, dW13_s=None, dW2_s=None, ws=None, stream=None):
    ts = (Xperm, offsets, tile_offsets, counts, W13, W2, GU, A, dYperm, dGU, dXperm, dW13, dW2, X, dY, W13_s, W2_s,
          GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s, ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_bwd", cfg, *map(_ptr, ts), _stream(stream))


def moe_fp8_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _call("moe_fp8_workspace_size", cfg, ctypes.byref(n))
    return n.value


def moe_quantize_weights_fp8(cfg, W13, W2, W13_s, W2_s, W13q, W13sc, W2q, W2sc, W13q_s=None, W13sc_s=None,
                             W2q_s=None, W2sc_s=None, stream=None):
    ts = (W13, W2, W13_s, W2_s, W13q, W13sc, W2q, W2sc, W13q_s, W13sc_s, W2q_s, W2sc_s)
    _dev(*ts)
    _call("moe_quantize_weights_fp8", cfg, *map(_ptr, ts), _stream(stream))


def moe_grouped_swiglu_mlp_fp8(cfg, Xperm, offsets, tile_offsets, W13q, W13sc, W2q, W2sc, GU, A, Yperm, X=None,
                               W13q_s=None, W13sc_s=None, W2q_s=None, W2sc_s=None, GU_s=None, A_s=None, Yshared=None,
                               fp8_ws=None, ws=None, stream=None):
    ts = (Xperm, offsets, tile_offsets, W13q, W13sc, W2q, W2sc, GU, A, Yperm, X, W13q_s, W13sc_s, W2q_s, W2sc_s,
          GU_s, A_s, Yshared, fp8_ws, ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_fp8", cfg, *map(_ptr, ts), _stream(stream))


def moe_grouped_swiglu_mlp_bwd_fp8(cfg, Xperm, offsets, tile_offsets, counts, W13q, W13sc, W2q, W2sc, GU, A, dYperm,
                                   dGU, dXperm, dW13, dW2, X=None, dY=None, W13q_s=None, W13sc_s=None, W2q_s=None,
                                   W2sc_s=None, GU_s=None, A_s=None, dGU_s=None, dX_shared=None, dW13_s=None,
                                   dW2_s=None, fp8_ws=None, ws=None, stream=None):
    ts = (Xperm, offsets, tile_offsets, counts, W13q, W13sc, W2q, W2sc, GU, A, dYperm, dGU, dXperm, dW13, dW2, X, dY,
          W13q_s, W13sc_s, W2q_s, W2sc_s, GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s, fp8_ws, ws)
    _dev(*ts)
    _call("moe_grouped_swiglu_mlp_bwd_fp8", cfg, *map(_ptr, ts), _stream(stream))


def moe_router_topk_bwd(cfg, X, W_r, logits, scores, topk_idx, gates, dgates, dW_r, dlogit_bias, dX_router, ws,
                        stream=None):
    ts = (X, W_r, logits, scores, topk_idx, gates, dgates, dW_r, dlogit_bias, dX_router, ws)
    _dev(*ts)
    _call("moe_router_topk_bwd", cfg, *map(_ptr, ts), _stream(stream))


def moe_permute_bwd(cfg, dXperm, row_id_map, dX_router, dX_shared, dX, stream=None):
    _dev(dXperm, row_id_map, dX_router, dX_shared, dX)
    _call("moe_permute_bwd", cfg, *map(_ptr, (dXperm, row_id_map, dX_router, dX_shared, dX)), _stream(stream))


@dataclass
class LayerWeights:
    W_r: torch.Tensor                 # [E,H] fp32
    W13: torch.Tensor                 # [E,2F,H] bf16
    W2: torch.Tensor                  # [E,H,F] bf16
    logit_bias: torch.Tensor | None = None
    sel_bias: torch.Tensor | None = None
    W13_s: torch.Tensor | None = None
    W2_s: torch.Tensor | None = None


class MoELayer:
    """Device buffers of one layer plus the forward/backward call sequence.

    All buffers are allocated once here (PyTorch as the allocator); forward()
    and backward() only launch the library's kernels on the current stream, so
    both can be captured in a CUDA graph.
    """

    def __init__(self, cfg: MoeConfig, weights: LayerWeights, device="cuda", fp8: bool = False,
                 capacity: int | None = None, drop_by_gate: bool = False, memory_efficient: bool = False,
                 gather_rows: bool = False):
        if memory_efficient and fp8:
            raise ValueError("the memory-efficient path is built for the bf16 expert GEMMs")
        if gather_rows and (fp8 or memory_efficient):
            raise ValueError("gathered rows are built for the plain bf16 path")
        self.gather_rows = gather_rows
        self.cfg = cfg
        self.w = weights
        self.fp8 = fp8
        self.memory_efficient = memory_efficient
        self.capacity = capacity
        self.drop_by_gate = drop_by_gate
        T, H, E, k, F, Fs = cfg.T, cfg.H, cfg.E, cfg.k, cfg.F, cfg.F_shared
        self.R = R = moe_max_rows(cfg)
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        z = lambda *s, dt=bf: torch.empty(*s, dtype=dt, device=device)
        self.ws = torch.zeros(moe_workspace_size(cfg), dtype=torch.uint8, device=device)
        moe_workspace_init(cfg, self.ws)
        self.logits, self.scores = z(T, E, dt=f32), z(T, E, dt=f32)
        self.topk_idx, self.gates, self.counts = z(T, k, dt=i32), z(T, k, dt=f32), z(E, dt=i32)
        self.offsets, self.tile_offsets = z(E + 1, dt=i32), z(E + 1, dt=i32)
        # with a capacity, the segment sizes every later stage uses are the kept counts
        self.seg_counts = z(E, dt=i32) if capacity is not None else self.counts
        self.row_id_map, self.slot_src = z(T, k, dt=i32), z(R, dt=i32)
        self.Xperm = None if gather_rows else z(R, H)
        self.GU, self.A, self.Yperm = z(R, 2 * F), z(R, F), z(R, H)
        self.Y = z(T, H)
        self.dYperm, self.dgates, self.dGU, self.dXperm = z(R, H), z(T, k, dt=f32), z(R, 2 * F), z(R, H)
        self.dW13, self.dW2 = z(E, 2 * F, H), z(E, H, F)
        self.dW_r, self.dlogit_bias, self.dX_router = z(E, H, dt=f32), z(E, dt=f32), z(T, H, dt=f32)
        self.dX = z(T, H)
        if Fs:
            self.GU_s, self.A_s, self.Yshared = z(T, 2 * Fs), z(T, Fs), z(T, H)
            self.dGU_s, self.dX_shared = z(T, 2 * Fs), z(T, H)
            self.dW13_s, self.dW2_s = z(2 * Fs, H), z(H, Fs)
        else:
            self.GU_s = self.A_s = self.Yshared = self.dGU_s = self.dX_shared = self.dW13_s = self.dW2_s = None
        self.X = None
        self.dY = None
        if fp8:
            u8 = torch.uint8
            q = lambda *s: torch.empty(*s, dtype=u8, device=device)
            self.W13q, self.W13sc = q(E, 2 * F, H), q(E, 2 * F // 128, H // 128)
            self.W2q, self.W2sc = q(E, H, F), q(E, H // 128, F // 128)
            if Fs:
                self.W13q_s, self.W13sc_s = q(2 * Fs, H), q(2 * Fs // 128, H // 128)
                self.W2q_s, self.W2sc_s = q(H, Fs), q(H // 128, Fs // 128)
            else:
                self.W13q_s = self.W13sc_s = self.W2q_s = self.W2sc_s = None
            self.fp8_ws = q(moe_fp8_workspace_size(cfg))

    def quantize_weights(self):
        """FP8 mode: E4M3 copies of the expert weights (128x128 power-of-two block scales)."""
        w = self.w
        moe_quantize_weights_fp8(self.cfg, w.W13, w.W2, w.W13_s, w.W2_s, self.W13q, self.W13sc, self.W2q, self.W2sc,
                                 self.W13q_s, self.W13sc_s, self.W2q_s, self.W2sc_s)

    def forward(self, X: torch.Tensor) -> torch.Tensor:
        c, w = self.cfg, self.w
        self.X = X
        moe_router_topk(c, X, w.W_r, w.logit_bias, w.sel_bias, self.logits, self.scores, self.topk_idx, self.gates,
                        self.counts, self.ws)
        if self.capacity is None:
            moe_permute(c, X, self.topk_idx, self.counts, self.offsets, self.tile_offsets, self.row_id_map,
                        self.slot_src, self.Xperm, self.ws)
        else:
            moe_permute_capacity(c, X, self.topk_idx, self.counts, self.capacity,
                                 self.gates if self.drop_by_gate else None, self.seg_counts, self.offsets,
                                 self.tile_offsets, self.row_id_map, self.slot_src, self.Xperm, self.ws)
        if self.gather_rows:
            moe_grouped_swiglu_mlp_gather(c, X, self.slot_src, self.offsets, self.tile_offsets, w.W13, w.W2, self.GU,
                                          self.A, self.Yperm, w.W13_s, w.W2_s, self.GU_s, self.A_s, self.Yshared,
                                          self.ws)
            moe_unpermute_combine(c, self.Yperm, self.row_id_map, self.gates, self.Yshared, self.Y)
            return self.Y
        if self.memory_efficient:
            moe_grouped_swiglu_mlp_gated(c, self.Xperm, self.offsets, self.tile_offsets, self.slot_src, self.gates,
                                         w.W13, w.W2, self.GU, self.A, self.Yperm, X if c.F_shared else None,
                                         w.W13_s, w.W2_s, self.GU_s, self.A_s, self.Yshared, self.ws)
            moe_unpermute_combine(c, self.Yperm, self.row_id_map, None, self.Yshared, self.Y)
            return self.Y
        if self.fp8:
            self.quantize_weights()
            moe_grouped_swiglu_mlp_fp8(c, self.Xperm, self.offsets, self.tile_offsets, self.W13q, self.W13sc,
                                       self.W2q, self.W2sc, self.GU, self.A, self.Yperm, X if c.F_shared else None,
                                       self.W13q_s, self.W13sc_s, self.W2q_s, self.W2sc_s, self.GU_s, self.A_s,
                                       self.Yshared, self.fp8_ws, self.ws)
        else:
            moe_grouped_swiglu_mlp(c, self.Xperm, self.offsets, self.tile_offsets, w.W13, w.W2, self.GU, self.A,
                                   self.Yperm, X if c.F_shared else None, w.W13_s, w.W2_s, self.GU_s, self.A_s,
                                   self.Yshared, self.ws)
        moe_unpermute_combine(c, self.Yperm, self.row_id_map, self.gates, self.Yshared, self.Y)
        return self.Y

    def backward(self, dY: torch.Tensor) -> torch.Tensor:
        c, w = self.cfg, self.w
        self.dY = dY
        sh = c.F_shared > 0
        if self.gather_rows:
            moe_unpermute_combine_bwd(c, dY, self.Yperm, self.row_id_map, self.gates, self.offsets, self.seg_counts,
                                      self.dYperm, self.dgates)
            moe_grouped_swiglu_mlp_bwd_gather(c, self.X, self.slot_src, self.offsets, self.tile_offsets,
                                              self.seg_counts, w.W13, w.W2, self.GU, self.A, self.dYperm, self.dGU,
                                              self.dXperm, self.dW13, self.dW2, dY if sh else None, w.W13_s, w.W2_s,
                                              self.GU_s, self.A_s, self.dGU_s, self.dX_shared, self.dW13_s,
                                              self.dW2_s, self.ws)
            moe_router_topk_bwd(c, self.X, w.W_r, self.logits, self.scores, self.topk_idx, self.gates, self.dgates,
                                self.dW_r, self.dlogit_bias if w.logit_bias is not None else None, self.dX_router,
                                self.ws)
            moe_permute_bwd(c, self.dXperm, self.row_id_map, self.dX_router, self.dX_shared, self.dX)
            return self.dX
        if self.memory_efficient:
            moe_unpermute_combine_bwd(c, dY, None, self.row_id_map, None, self.offsets, self.seg_counts,
                                      self.dYperm, None)
            moe_grouped_swiglu_mlp_bwd_gated(c, self.Xperm, self.offsets, self.tile_offsets, self.seg_counts,
                                             self.slot_src, self.row_id_map, self.gates, w.W13, w.W2, self.GU,
                                             self.dYperm, self.dGU, self.dXperm, self.A, self.dW13, self.dW2,
                                             self.dgates, self.X if sh else None, dY if sh else None, w.W13_s,
                                             w.W2_s, self.GU_s, self.A_s, self.dGU_s, self.dX_shared, self.dW13_s,
                                             self.dW2_s, self.ws)
            moe_router_topk_bwd(c, self.X, w.W_r, self.logits, self.scores, self.topk_idx, self.gates, self.dgates,
                                self.dW_r, self.dlogit_bias if w.logit_bias is not None else None, self.dX_router,
                                self.ws)
            moe_permute_bwd(c, self.dXperm, self.row_id_map, self.dX_router, self.dX_shared, self.dX)
            return self.dX
        moe_unpermute_combine_bwd(c, dY, self.Yperm, self.row_id_map, self.gates, self.offsets, self.seg_counts,
                                  self.dYperm, self.dgates)
        if self.fp8:
            moe_grouped_swiglu_mlp_bwd_fp8(c, self.Xperm, self.offsets, self.tile_offsets, self.seg_counts, self.W13q,
                                           self.W13sc, self.W2q, self.W2sc, self.GU, self.A, self.dYperm, self.dGU,
                                           self.dXperm, self.dW13, self.dW2, self.X if sh else None,
                                           dY if sh else None, self.W13q_s, self.W13sc_s, self.W2q_s, self.W2sc_s,
                                           self.GU_s, self.A_s, self.dGU_s, self.dX_shared, self.dW13_s, self.dW2_s,
                                           self.fp8_ws, self.ws)
        else:
            moe_grouped_swiglu_mlp_bwd(c, self.Xperm, self.offsets, self.tile_offsets, self.seg_counts, w.W13, w.W2,
                                       self.GU, self.A, self.dYperm, self.dGU, self.dXperm, self.dW13, self.dW2,
                                       self.X if sh else None, dY if sh else None, w.W13_s, w.W2_s, self.GU_s,
                                       self.A_s, self.dGU_s, self.dX_shared, self.dW13_s, self.dW2_s, self.ws)
        moe_router_topk_bwd(c, self.X, w.W_r, self.logits, self.scores, self.topk_idx, self.gates, self.dgates,
                            self.dW_r, self.dlogit_bias if w.logit_bias is not None else None, self.dX_router, self.ws)
        moe_permute_bwd(c, self.dXperm, self.row_id_map, self.dX_router, self.dX_shared, self.dX)
        return self.dX

    def device_error(self) -> int:
        return moe_read_device_error(self.ws)


def gemm_flops(cfg: MoeConfig, fwd_only: bool = False) -> float:
    """Algorithmic grouped-GEMM FLOP of one layer step (padding rows excluded)."""
    per_slot = 6.0 * cfg.H * cfg.F
    shared = 6.0 * cfg.H * cfg.F_shared * cfg.T
    f = per_slot * cfg.T * cfg.k + shared
    return f if fwd_only else 3.0 * f
