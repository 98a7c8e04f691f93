"""Shared test helpers: uploads of the seeded inputs and the error metric."""
from __future__ import annotations

import numpy as np
import torch

import moe_synth as S


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_dev(a, device="cuda"):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return to_dev_bf16(a, device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def slice_rel_err(gpu: np.ndarray, ref: np.ndarray, slice_axes=1) -> float:
    """max over slices of max|gpu-ref| / max|ref|.  A slice is the trailing
    `slice_axes` dimensions (a token row, or one expert's whole gradient).  A
    slice whose reference is all zero must match exactly (error inf otherwise)."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if g.ndim <= slice_axes:
        g = g[None]
        r = r[None]
    lead = int(np.prod(g.shape[: g.ndim - slice_axes]))
    g = g.reshape(lead, -1)
    r = r.reshape(lead, -1)
    num = np.abs(g - r).max(axis=1)
    den = np.abs(r).max(axis=1)
    out = np.where(den > 0, num / np.where(den > 0, den, 1.0), np.where(num > 0, np.inf, 0.0))
    return float(out.max()) if len(out) else 0.0


def logit_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """Router logits: per token, max|gpu-ref| over the experts divided by the
    larger of that token's max|ref| and the RMS of all reference logits.  A
    token whose logits all cancel to near zero (E=1 makes this common) is thus
    measured against the typical logit size instead of its own tiny value."""
    g = np.asarray(gpu, np.float64).reshape(len(gpu), -1)
    r = np.asarray(ref, np.float64).reshape(len(ref), -1)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    den = np.maximum(np.abs(r).max(axis=1), rms)
    return float((np.abs(g - r).max(axis=1) / den).max())


def make_layer(w: S.Workload, inp: dict, device="cuda", capacity=None, drop_by_gate=False,
               memory_efficient=False, gather_rows=False):
    import mixture_experts_layer_topk_gb300 as M
    cfg = M.config_from(w)
    weights = M.LayerWeights(
        W_r=to_dev(inp["W_r"]), W13=to_dev(inp["W13"]), W2=to_dev(inp["W2"]),
        logit_bias=to_dev(inp.get("logit_bias")), sel_bias=to_dev(inp.get("sel_bias")),
        W13_s=to_dev(inp.get("W13_s")), W2_s=to_dev(inp.get("W2_s")))
    return M.MoELayer(cfg, weights, device=device, fp8=getattr(w, "fp8", False), capacity=capacity,
                      drop_by_gate=drop_by_gate, memory_efficient=memory_efficient, gather_rows=gather_rows)
