"""Router projection for E > 32: the tensor-core path (taken when the call has a
workspace) and the FP32 CUDA-core path (no workspace), each against the oracle's
double logits, on shapes that cover both K-split settings of the tensor-core
launch (two K halves when the tiles fill less than half the GPU, else one),
ragged token counts, expert counts that are not a multiple of the 128-expert
tile, and more than one expert tile.  Selections are bit-exact against the
oracle's float32 selection on each path's own logits and scores.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle as O
from helpers import logit_rel_err, slice_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL_ROUTER = 1e-5

CASES = {
    # E not a multiple of 32 (the split's padded rows), two K halves
    "e40-ragged": S.Workload("e40-ragged", T=777, H=512, E=40, k=4, F=128),
    # a long K (H = 4096, as in the Qwen3-style layer), two K halves
    "e128-longk": S.Workload("e128-longk", T=640, H=4096, E=128, k=8, F=128),
    # enough token tiles for one K split, ragged last tile
    "e128-onesplit": S.Workload("e128-onesplit", T=10000, H=256, E=128, k=8, F=128),
    # two expert tiles, sigmoid, groups, selection bias, one K split
    "e256-groups": S.Workload("e256-groups", T=5000, H=384, E=256, k=8, F=128, score_fn=1, gate_scale=2.5,
                              n_group=8, topk_group=4, sel_bias=True),
    # two expert tiles, the longest K of the layers here (H = 7168), two K halves
    "e256-longk": S.Workload("e256-longk", T=300, H=7168, E=256, k=8, F=128, score_fn=1, n_group=8, topk_group=4,
                             sel_bias=True),
    # skewed logit bias (bias enters the logits)
    "e64-skew": S.Workload("e64-skew", T=2000, H=1024, E=64, k=4, F=128, skew=True),
}


def _route(M, cfg, w, X, W_r, lb, sb, ws):
    T, E, k = w.T, w.E, w.k
    f32, i32 = torch.float32, torch.int32
    new = lambda *s, dt=f32: torch.full(s, 7, dtype=dt, device="cuda")  # poisoned outputs
    out = dict(logits=new(T, E), scores=new(T, E), idx=new(T, k, dt=i32), gates=new(T, k), counts=new(E, dt=i32))
    M.moe_router_topk(cfg, X, W_r, lb, sb, out["logits"], out["scores"], out["idx"], out["gates"], out["counts"], ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert M.moe_read_device_error(ws) == 0
    return {k_: v.cpu().numpy() for k_, v in out.items()}


@pytest.mark.parametrize("name", list(CASES))
def test_router_projection_paths(name):
    import mixture_experts_layer_topk_gb300 as M
    w = CASES[name]
    inp = S.host_inputs(w, weights=False)
    cfg = M.config_from(w)
    X, W_r = to_dev(inp["X"]), to_dev(inp["W_r"])
    lb, sb = to_dev(inp.get("logit_bias")), to_dev(inp.get("sel_bias"))
    ws = torch.zeros(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    c = O.cfg(w)
    logits, scores = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    tol_s = TOL_ROUTER * max(1.0, float(np.abs(logits).max()))
    errs = {}
    for path, wsp in (("tensor", ws), ("cuda-core", None)):
        r = _route(M, cfg, w, X, W_r, lb, sb, wsp)
        errs[path] = logit_rel_err(r["logits"], logits)
        assert errs[path] < TOL_ROUTER, (path, errs[path])
        assert slice_rel_err(r["scores"], scores) < tol_s, path
        idx_ora = O.select(c, r["logits"], r["scores"], inp.get("sel_bias"))
        assert np.array_equal(r["idx"], idx_ora), (path, np.argwhere(r["idx"] != idx_ora)[:5])
        assert slice_rel_err(r["gates"], O.gates(c, logits, r["idx"])) < 2 * tol_s, path
        assert np.array_equal(r["counts"], np.bincount(r["idx"].ravel(), minlength=w.E)), path
    print(name, errs)


def test_router_tensor_path_promotes_block_sums():
    """The block sums leave tensor memory every 64 columns of K, so the logit error
    must not grow with K the way a whole-K tensor-memory accumulation does (about
    4e-5 at H = 4096): at H = 7168 it stays well inside the FP32 bound."""
    import mixture_experts_layer_topk_gb300 as M
    w = S.Workload("longk", T=256, H=7168, E=64, k=2, F=128)
    inp = S.host_inputs(w, weights=False)
    cfg = M.config_from(w)
    ws = torch.zeros(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    r = _route(M, cfg, w, to_dev(inp["X"]), to_dev(inp["W_r"]), None, None, ws)
    logits, _ = O.router(O.cfg(w), inp["X"], inp["W_r"], None)
    assert logit_rel_err(r["logits"], logits) < 2e-6


@pytest.mark.parametrize("name", ["e128-longk", "e64-skew"])
def test_router_backward_products(name):
    """dX_router = dlogits W_r and dW_r = dlogits^T X of the layer's backward (tensor-core
    products from bf16 splits for E > 32) against the oracle's dlogits, each on its own.
    The layer's dlogits come from its bf16 expert path, so the bound is the bf16 one."""
    from helpers import make_layer
    w = CASES[name]
    inp = S.host_inputs(w)
    layer = make_layer(w, inp)
    layer.forward(to_dev(inp["X"]))
    layer.backward(to_dev(inp["dY"]))
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    c = O.cfg(w, mirror=True)
    logits, _ = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    idx = layer.topk_idx.cpu().numpy()
    tk = O.tokens(c, inp, idx, logits, O.gates(c, logits, idx))
    dxr = tk["dlogits"] @ np.asarray(inp["W_r"], np.float64)
    assert slice_rel_err(layer.dX_router.cpu().numpy(), dxr) < 2e-2
    dWr, _ = O.router_wgrad(c, inp["X"], tk["dlogits"])
    assert slice_rel_err(layer.dW_r.cpu().numpy(), dWr) < 2e-2
