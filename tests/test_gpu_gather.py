"""Gathered-rows expert MLP (no permuted copy of the tokens): FC1 reads the token rows
of X through the dispatch map with TMA four-row gathers, in the forward and in FC1's
weight gradient.  The GEMMs see exactly the operands of the plain path, so every
output must be bit-identical to it (the plain path is held to the oracle in
test_gpu_parity.py)."""
import numpy as np
import pytest
import torch

import moe_synth as S
from helpers import make_layer, to_dev

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
