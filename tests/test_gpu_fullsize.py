"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle cannot run the whole layer at these sizes in seconds, so:
  * routing for every token: GPU logits/scores vs the oracle's double values,
    the oracle's float32 selection on the GPU's own scores (bit-exact), and the
    dispatch maps (bit-exact);
  * Y, dX and dgates on a seeded sample of tokens (each token's values depend
    only on that token, so the oracle computes them one by one);
  * the weight gradients of the least-loaded non-empty expert in full, and of the
    most-loaded expert (the long-K and split-tail tiles) and the shared expert at
    a seeded sample of FFN indices f: rows f and F+f of dW13, column f of dW2, each
    entry exactly as the full oracle gradient computes it; every empty expert's
    weight gradient must be 0;
  * the router backward over all T tokens: moe_router_topk_bwd on the layer's own
    routing with seeded gate gradients, dW_r and dlogit_bias against the oracle's
    exact gate Jacobian and its double reduction over every token, dX_router on the
    sampled tokens.
The DeepSeek-V3-style layer also runs with FP8 E4M3 expert GEMMs, held to the FP8
bound against the oracle's FP8 mode.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_topk_gb300 as M
import moe_synth as S
import oracle as O
from helpers import host_f64, logit_rel_err, make_layer, slice_rel_err, to_dev

pytestmark = pytest.mark.gpu

FULL = ["mixtral", "qwen3", "dsv3", "skew", "dsv3-fp8"]
N_TOKENS = 24
N_COLS = 8


def _sampled_wgrad_err(layer, c, inp, idx, g, e, F, rng):
    """Slice error of one expert's weight gradients at N_COLS sampled FFN indices."""
    cols = np.sort(rng.choice(F, size=min(N_COLS, F), replace=False)).astype(np.int32)
    r13, c2 = O.expert_wgrad_cols(c, inp, idx, g, e, cols)
    if e < 0:
        dW13, dW2 = layer.dW13_s, layer.dW2_s
    else:
        dW13, dW2 = layer.dW13[e], layer.dW2[e]
    ci = torch.from_numpy(cols.astype(np.int64)).cuda()
    got13 = torch.cat([dW13[ci], dW13[ci + F]])
    got2 = dW2[:, ci]
    return max(slice_rel_err(host_f64(got13), r13, 2), slice_rel_err(host_f64(got2), c2, 2))


@pytest.mark.parametrize("name", FULL)
def test_fullsize_sampled_parity(name):
    w = S.WORKLOADS[name]
    tol = 6e-2 if w.fp8 else 2e-2
    inp = S.host_inputs(w)
    layer = make_layer(w, inp)
    X, dY = to_dev(inp["X"]), to_dev(inp["dY"])
    layer.forward(X)
    layer.backward(dY)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    c = O.cfg(w)
    lg, sc = layer.logits.cpu().numpy(), layer.scores.cpu().numpy()
    logits, scores = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    assert logit_rel_err(lg, logits) < 1e-5
    tol_s = 1e-5 * max(1.0, float(np.abs(logits).max()))  # exp carries the logit error over
    assert slice_rel_err(sc, scores) < tol_s
    idx = layer.topk_idx.cpu().numpy()
    assert np.array_equal(idx, O.select(c, lg, sc, inp.get("sel_bias")))
    g = O.gates(c, logits, idx)
    assert slice_rel_err(layer.gates.cpu().numpy(), g) < 2 * tol_s
    d = O.dispatch(c, idx, R=layer.R)
    n_used = int(d["offsets"][-1])
    for k in ["counts", "offsets", "tile_offsets", "row_id_map"]:
        assert np.array_equal(getattr(layer, k).cpu().numpy(), d[k]), k
    assert np.array_equal(layer.slot_src.cpu().numpy()[:n_used], d["slot_src"][:n_used])
    counts = d["counts"]
    if w.skew:
        assert (counts == 0).any() and counts.max() > 0.15 * w.T * w.k
    # the oracle's values: FP8 mode computes with the block-quantized weights (replaced in
    # place, one tensor at a time, to bound the host memory of the 22.5 GB layer)
    if w.fp8:
        for key in ("W13", "W2", "W13_s", "W2_s"):
            if inp.get(key) is not None:
                inp[key] = O.qdq_weights(inp[key])
    vinp = inp
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(w.T, size=N_TOKENS, replace=False))
    tk = O.tokens(c, vinp, idx, logits, g, tok_list=toks)
    ti = torch.from_numpy(toks).cuda()
    assert slice_rel_err(host_f64(layer.Y[ti]), tk["Y"]) < tol
    assert slice_rel_err(host_f64(layer.dX[ti]), tk["dX"]) < tol
    assert slice_rel_err(layer.dgates[ti].cpu().numpy(), tk["dgates"]) < tol
    # weight gradients: the least-loaded non-empty expert in full ...
    nz = np.flatnonzero(counts)
    e = int(nz[np.argmin(counts[nz])])
    dW13, dW2 = O.expert_wgrad(c, vinp, idx, g, e)
    assert slice_rel_err(host_f64(layer.dW13[e]), dW13, 2) < tol
    assert slice_rel_err(host_f64(layer.dW2[e]), dW2, 2) < tol
    # ... the most-loaded one and the shared expert at sampled FFN indices
    e_max = int(np.argmax(counts))
    assert _sampled_wgrad_err(layer, c, vinp, idx, g, e_max, w.F, rng) < tol, e_max
    if w.F_shared:
        assert _sampled_wgrad_err(layer, c, vinp, idx, g, -1, w.F_shared, rng) < tol
    for e0 in np.flatnonzero(counts == 0):
        assert layer.dW13[e0].abs().max().item() == 0 and layer.dW2[e0].abs().max().item() == 0

    # router backward over all T tokens, seeded gate gradients (bounds as in the
    # exact router-backward test: the products are FP32-grade)
    T, E, k, H = w.T, w.E, w.k, w.H
    dgates_h = S.normal_f32(T * k, 1, 99, 1.0).reshape(T, k)
    f32 = torch.float32
    dW_r = torch.full((E, H), 7, dtype=f32, device="cuda")
    dlb = torch.full((E,), 7, dtype=f32, device="cuda")
    dXr = torch.full((T, H), 7, dtype=f32, device="cuda")
    has_lb = inp.get("logit_bias") is not None
    M.moe_router_topk_bwd(layer.cfg, X, layer.w.W_r, layer.logits, layer.scores, layer.topk_idx, layer.gates,
                          to_dev(dgates_h), dW_r, dlb if has_lb else None, dXr, layer.ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(layer.ws) == 0
    dl = O.router_dlogits(c, logits, idx, g, dgates_h.astype(np.float64))
    dWr_o, dlb_o = O.router_wgrad(c, inp["X"], dl)
    assert slice_rel_err(dW_r.cpu().numpy(), dWr_o) < 1e-3
    if has_lb:
        assert slice_rel_err(dlb.cpu().numpy(), dlb_o, 1) < 1e-5
    dxr = dl[toks] @ np.asarray(inp["W_r"], np.float64)
    assert slice_rel_err(dXr[ti].cpu().numpy(), dxr) < 2e-4
