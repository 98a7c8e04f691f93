"""Router projection: the tensor-core path (taken when the call has a workspace)
and the CUDA-core path (no workspace: one fused launch for E <= 32, an FP32 GEMM
for larger E), each against the oracle's double logits, on shapes that cover
one to eight K splits of the tensor-core launch (partial sums added in a fixed
order), the 32-, 64- and 128-expert tiles, ragged token counts, expert counts
that are not a multiple of the tile, and more than one expert tile.  Selections
are bit-exact against the oracle's float32 selection on each path's own logits
and scores.
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
    # the Mixtral-style router shape: 32 token tiles of 8 experts, several K splits
    "e8-mixtral-shape": S.Workload("e8-mixtral-shape", T=4096, H=4096, E=8, k=2, F=128),
    # few tiles, up to eight K splits; sigmoid with groups
    "e16-groups-splits": S.Workload("e16-groups-splits", T=300, H=1024, E=16, k=3, F=128, score_fn=1, renorm=0,
                                    n_group=4, topk_group=2),
    # one expert, one token tile, two K blocks
    "e1-k1": S.Workload("e1-k1", T=200, H=128, E=1, k=1, F=128),
    # 96 experts: three 32-row blocks per split, K of the dX_router product (3 x 96) not a
    # multiple of 64
    "e96": S.Workload("e96", T=700, H=512, E=96, k=6, F=128),
    # 32 experts (a full 32-expert tile), ragged tokens
    "e32-ragged": S.Workload("e32-ragged", T=1000, H=768, E=32, k=4, F=128),
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


@pytest.mark.parametrize("name", ["e128-longk", "e64-skew", "e96"])
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


@pytest.mark.parametrize("name", ["e8-mixtral-shape", "e40-ragged", "e64-skew", "e96", "e128-longk", "e256-groups"])
def test_router_backward_exact(name):
    """moe_router_topk_bwd on its own, with seeded gate gradients: dX_router = dlogits W_r,
    dW_r = dlogits^T X and dlogit_bias = sum_t dlogits against the oracle's double dlogits
    (its exact gate Jacobian on its own logits and the GPU's selection).  Bounds: dX_router
    2e-4 (three bf16 split products, ~2^-16 each), dW_r 1e-3 (tensor-core FP32 accumulation
    over the token splits), dlogit_bias 1e-5."""
    import mixture_experts_layer_topk_gb300 as M
    w = CASES[name]
    inp = S.host_inputs(w, weights=False)
    cfg = M.config_from(w)
    T, E, k, H = w.T, w.E, w.k, w.H
    X, W_r = to_dev(inp["X"]), to_dev(inp["W_r"])
    lb, sb = to_dev(inp.get("logit_bias")), to_dev(inp.get("sel_bias"))
    ws = torch.zeros(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    f32, i32 = torch.float32, torch.int32
    new = lambda *s, dt=f32: torch.full(s, 7, dtype=dt, device="cuda")
    logits, scores, idx, gates, counts = new(T, E), new(T, E), new(T, k, dt=i32), new(T, k), new(E, dt=i32)
    M.moe_router_topk(cfg, X, W_r, lb, sb, logits, scores, idx, gates, counts, ws)
    dgates_h = S.normal_f32(T * k, 1, 99, 1.0).reshape(T, k)
    dW_r, dlb, dXr = new(E, H), new(E), new(T, H)
    M.moe_router_topk_bwd(cfg, X, W_r, logits, scores, idx, gates, to_dev(dgates_h), dW_r,
                          dlb if lb is not None else None, dXr, ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(ws) == 0
    c = O.cfg(w)
    lg, sc = logits.cpu().numpy(), scores.cpu().numpy()
    sel = idx.cpu().numpy()
    assert np.array_equal(sel, O.select(c, lg, sc, inp.get("sel_bias")))
    lo, _ = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    dl = O.router_dlogits(c, lo, sel, O.gates(c, lo, sel), dgates_h.astype(np.float64))
    dxr = dl @ np.asarray(inp["W_r"], np.float64)
    assert slice_rel_err(dXr.cpu().numpy(), dxr) < 2e-4
    dWr, dlb_o = O.router_wgrad(c, inp["X"], dl)
    assert slice_rel_err(dW_r.cpu().numpy(), dWr) < 1e-3
    if lb is not None:
        assert slice_rel_err(dlb.cpu().numpy(), dlb_o, 1) < 1e-5
