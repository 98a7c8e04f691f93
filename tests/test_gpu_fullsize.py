"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle cannot run the whole layer at these sizes in seconds, so:
  * routing for every token: GPU logits/scores vs the oracle's double values,
    the oracle's float32 selection on the GPU's own scores (bit-exact), and the
    dispatch maps (bit-exact);
  * Y, dX and dgates on a seeded sample of tokens (each token's values depend
    only on that token, so the oracle computes them one by one);
  * dW13 and dW2 of the least-loaded non-empty expert (the oracle recomputes
    every token routed to it); every empty expert's weight gradient must be 0.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle as O
from helpers import host_f64, logit_rel_err, make_layer, slice_rel_err, to_dev

pytestmark = pytest.mark.gpu

FULL = ["mixtral", "qwen3", "dsv3", "skew"]


@pytest.mark.parametrize("name", FULL)
def test_fullsize_sampled_parity(name):
    w = S.WORKLOADS[name]
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
    if w.skew:
        counts = d["counts"]
        assert (counts == 0).any() and counts.max() > 0.15 * w.T * w.k
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(w.T, size=24, replace=False))
    tk = O.tokens(c, inp, idx, logits, g, tok_list=toks)
    ti = torch.from_numpy(toks).cuda()
    assert slice_rel_err(host_f64(layer.Y[ti]), tk["Y"]) < 2e-2
    assert slice_rel_err(host_f64(layer.dX[ti]), tk["dX"]) < 2e-2
    assert slice_rel_err(layer.dgates[ti].cpu().numpy(), tk["dgates"]) < 2e-2
    counts = d["counts"]
    nz = np.flatnonzero(counts)
    e = int(nz[np.argmin(counts[nz])])
    dW13, dW2 = O.expert_wgrad(c, inp, idx, g, e)
    assert slice_rel_err(host_f64(layer.dW13[e]), dW13, 2) < 2e-2
    assert slice_rel_err(host_f64(layer.dW2[e]), dW2, 2) < 2e-2
    for e0 in np.flatnonzero(counts == 0):
        assert layer.dW13[e0].abs().max().item() == 0 and layer.dW2[e0].abs().max().item() == 0
