"""Gathered-rows expert MLP (no permuted copy of the tokens): FC1 reads the token rows
of X through the dispatch map with TMA four-row gathers, in the forward and in FC1's
weight gradient.  The GEMMs see exactly the operands of the plain path, so every
output must be bit-identical to it; the gathered path is also held to the oracle
directly, element by element."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle as O
from helpers import host_f64, logit_rel_err, make_layer, slice_rel_err, to_dev

pytestmark = pytest.mark.gpu

GATHER_CASES = {
    # several M tiles per expert and ragged tails
    "ragged-softmax": S.Workload("ragged-softmax", T=1000, H=256, E=8, k=2, F=384),
    # sigmoid, groups, selection bias, shared expert; one M tile per expert
    "dsv3-mini": S.Workload("dsv3-mini", T=520, H=256, E=64, k=6, F=256, F_shared=256, score_fn=1, gate_scale=2.5,
                            n_group=8, topk_group=4, sel_bias=True),
    # 32 experts (fused router), H = 512 (two pair tiles along N in FC1's wgrad)
    "e32-h512": S.Workload("e32-h512", T=700, H=512, E=32, k=4, F=256),
}

OUTPUTS = ("topk_idx", "offsets", "row_id_map", "slot_src", "GU", "A", "Yperm", "Y", "dgates", "dX", "dW13", "dW2",
           "dW_r")


def _run(w, inp, **kw):
    layer = make_layer(w, inp, **kw)
    layer.forward(to_dev(inp["X"]))
    layer.backward(to_dev(inp["dY"]))
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    return layer


def _used(layer, name):
    t = getattr(layer, name)
    if name in ("GU", "A", "Yperm", "slot_src"):  # rows past the used segments are not written
        t = t[: int(layer.offsets[-1].item())]
    return t


@pytest.mark.parametrize("name", list(GATHER_CASES))
def test_gathered_rows_equal_the_permuted_copy(name):
    w = GATHER_CASES[name]
    inp = S.host_inputs(w)
    ref = _run(w, inp)
    got = _run(w, inp, gather_rows=True)
    assert got.Xperm is None
    for n in OUTPUTS:
        assert torch.equal(_used(got, n), _used(ref, n)), n
    if w.F_shared:
        for n in ("Yshared", "dW13_s", "dW2_s"):
            assert torch.equal(getattr(got, n), getattr(ref, n)), n


def test_gathered_rows_with_capacity_dropping():
    w = GATHER_CASES["dsv3-mini"]
    inp = S.host_inputs(w)
    cap = int(np.ceil(0.8 * w.T * w.k / w.E))
    ref = _run(w, inp, capacity=cap, drop_by_gate=True)
    got = _run(w, inp, capacity=cap, drop_by_gate=True, gather_rows=True)
    for n in OUTPUTS:
        assert torch.equal(_used(got, n), _used(ref, n)), n


def test_gathered_rows_without_tokens():
    w = GATHER_CASES["e32-h512"].replace(T=0)
    inp = S.host_inputs(w)
    got = _run(w, inp, gather_rows=True)
    assert int(got.counts.sum().item()) == 0
    assert not got.dW13.any() and not got.dW2.any()


@pytest.mark.parametrize("name", ["ragged-softmax", "dsv3-mini"])
def test_gathered_rows_match_the_oracle(name):
    """The gathered path against the oracle: routing and maps bit-exact (the oracle's
    float32 selection on the GPU's own scores), every value within the bf16 bound."""
    w = GATHER_CASES[name]
    inp = S.host_inputs(w)
    layer = _run(w, inp, gather_rows=True)
    c = O.cfg(w)
    lg, sc = layer.logits.cpu().numpy(), layer.scores.cpu().numpy()
    logits, _ = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    assert logit_rel_err(lg, logits) < 1e-5
    idx = layer.topk_idx.cpu().numpy()
    assert np.array_equal(idx, O.select(c, lg, sc, inp.get("sel_bias")))
    g = O.gates(c, logits, idx)
    d = O.dispatch(c, idx, R=layer.R)
    n_used = int(d["offsets"][-1])
    for k in ["counts", "offsets", "tile_offsets", "row_id_map"]:
        assert np.array_equal(getattr(layer, k).cpu().numpy(), d[k]), k
    assert np.array_equal(layer.slot_src.cpu().numpy()[:n_used], d["slot_src"][:n_used])
    tk = O.tokens(c, inp, idx, logits, g)
    assert slice_rel_err(host_f64(layer.Y), tk["Y"]) < 2e-2
    assert slice_rel_err(layer.dgates.cpu().numpy(), tk["dgates"]) < 2e-2
    assert slice_rel_err(host_f64(layer.dX), tk["dX"]) < 2e-2
    for e in range(w.E):
        dW13, dW2 = O.expert_wgrad(c, inp, idx, g, e)
        assert slice_rel_err(host_f64(layer.dW13[e]), dW13, 2) < 2e-2, e
        assert slice_rel_err(host_f64(layer.dW2[e]), dW2, 2) < 2e-2, e
    if w.F_shared:
        dW13s, dW2s = O.expert_wgrad(c, inp, idx, g, -1)
        assert slice_rel_err(host_f64(layer.dW13_s), dW13s, 2) < 2e-2
        assert slice_rel_err(host_f64(layer.dW2_s), dW2s, 2) < 2e-2
    dWr, _ = O.router_wgrad(c, inp["X"], tk["dlogits"])
    assert slice_rel_err(layer.dW_r.cpu().numpy(), dWr) < 2e-2
