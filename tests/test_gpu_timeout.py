"""Failure detection inside the tensor-core kernels, without a GPU fault.

Every pipeline wait of the grouped GEMMs and of the router projection is bounded.
Here the bound is set to 0 (moe_set_wait_limit_ns), which makes each pipeline wait
a single non-blocking test: the first wait whose event has not happened yet (the
MMA issuer's first operand stage, the epilogue's first accumulator, a producer's
wait for a free stage) runs out at once.  The kernel must then record
MOE_ERR_TIMEOUT in the workspace's error word and unwind: wait (with its fixed
exit bound) for the copies and MMAs it issued, settle the loads of both CTAs of a
pair, free its tensor memory and exit.  Nothing traps, faults or spins.  The test
reads the error word, restores the bound, and checks that the next calls on the
same workspace run clean and reproduce a clean run's outputs bit for bit.

Cases: CTA-pair and one-CTA bf16 tiles (F = 384 gives 128-wide tiles for FC2's
dgrad and weight gradient), the dense shared-expert segment and the tensor-core
router (E = 64), the FP8 block-scaled one-CTA tiles with their scale-factor warps,
and the one-launch small dispatch's wait for its token rows.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_topk_gb300 as M
import moe_synth as S
from helpers import make_layer, to_dev

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5

CASES = {
    "pairs-and-single": S.Workload("pairs-and-single", T=1000, H=256, E=8, k=2, F=384),
    "shared-router64": S.Workload("shared-router64", T=520, H=256, E=64, k=6, F=256, F_shared=256, score_fn=1,
                                  gate_scale=2.5, n_group=8, topk_group=4, sel_bias=True),
    "fp8": S.Workload("fp8", T=1000, H=256, E=8, k=2, F=384, fp8=True),
}

OUTPUTS = ("topk_idx", "offsets", "row_id_map", "GU", "A", "Yperm", "Y", "dgates", "dX", "dW13", "dW2", "dW_r")


def _step(layer, X, dY):
    layer.forward(X)
    layer.backward(dY)


def _snapshot(layer):
    n = int(layer.offsets[-1].item())
    out = {}
    for name in OUTPUTS:
        t = getattr(layer, name)
        if name in ("GU", "A", "Yperm"):  # rows past the used segments are never written
            t = t[:n]
        out[name] = t.clone()
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_wait_timeout_unwinds_and_the_next_call_is_clean(name):
    w = CASES[name]
    inp = S.host_inputs(w)
    X, dY = to_dev(inp["X"]), to_dev(inp["dY"])
    layer = make_layer(w, inp)
    _step(layer, X, dY)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ref = _snapshot(layer)

    default = M.moe_get_wait_limit_ns()
    assert default > 0
    c = layer.cfg
    try:
        # the expert GEMMs alone, on the valid dispatch maps of the clean run
        M.moe_set_wait_limit_ns(0)
        if layer.fp8:
            M.moe_grouped_swiglu_mlp_fp8(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.W13q, layer.W13sc,
                                         layer.W2q, layer.W2sc, layer.GU, layer.A, layer.Yperm,
                                         X if c.F_shared else None, layer.W13q_s, layer.W13sc_s, layer.W2q_s,
                                         layer.W2sc_s, layer.GU_s, layer.A_s, layer.Yshared, layer.fp8_ws, layer.ws)
        else:
            sh = c.F_shared > 0
            w_ = layer.w
            M.moe_grouped_swiglu_mlp(c, layer.Xperm, layer.offsets, layer.tile_offsets, w_.W13, w_.W2, layer.GU,
                                     layer.A, layer.Yperm, X if sh else None, w_.W13_s, w_.W2_s, layer.GU_s,
                                     layer.A_s, layer.Yshared, layer.ws)
            M.moe_grouped_swiglu_mlp_bwd(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.counts, w_.W13,
                                         w_.W2, layer.GU, layer.A, layer.dYperm, layer.dGU, layer.dXperm, layer.dW13,
                                         layer.dW2, X if sh else None, dY if sh else None, w_.W13_s, w_.W2_s,
                                         layer.GU_s, layer.A_s, layer.dGU_s, layer.dX_shared, layer.dW13_s,
                                         layer.dW2_s, layer.ws)
        M.moe_set_wait_limit_ns(default)
        torch.cuda.synchronize()  # the kernels ended by themselves: the context is usable
        assert layer.device_error() == MOE_ERR_TIMEOUT
        # the router projection on the tensor cores (the routing pass after it reads the
        # partial sums as they are; the layer is re-run below)
        M.moe_set_wait_limit_ns(0)
        w_ = layer.w
        M.moe_router_topk(c, X, w_.W_r, w_.logit_bias, w_.sel_bias, layer.logits, layer.scores, layer.topk_idx,
                          layer.gates, layer.counts, layer.ws)
        M.moe_set_wait_limit_ns(default)
        torch.cuda.synchronize()
        assert layer.device_error() == MOE_ERR_TIMEOUT
    finally:
        M.moe_set_wait_limit_ns(default)

    # the same layer, workspace and buffers: a clean step reproduces the clean run
    _step(layer, X, dY)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    got = _snapshot(layer)
    for n in OUTPUTS:
        assert torch.equal(got[n], ref[n]), n


def test_dispatch_wait_timeout_unwinds():
    """The one-launch small dispatch waits for its token rows within the same limit.  With
    the limit at 0 its single test usually comes before the 33.6 MB of rows of this
    Mixtral-shaped layer have landed: the launch records MOE_ERR_TIMEOUT, waits (bounded)
    for its copies and exits (or, if every CTA found its rows already there, finishes).
    Either way the next dispatch on the same workspace reproduces a clean one bit for bit."""
    w = S.Workload("dispatch-timeout", T=4096, H=4096, E=8, k=2, F=128)
    cfg = M.config_from(w)
    rng = np.random.default_rng(11)
    idx = np.stack([rng.choice(w.E, size=w.k, replace=False) for _ in range(w.T)]).astype(np.int32)
    X = torch.randn(w.T, w.H, device="cuda").to(torch.bfloat16)
    topk = torch.from_numpy(idx).cuda()
    counts = torch.from_numpy(np.bincount(idx.ravel(), minlength=w.E).astype(np.int32)).cuda()
    R = M.moe_max_rows(cfg)
    ws = torch.zeros(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(cfg, ws)

    def outputs():
        i32 = torch.int32
        return [torch.full((w.E + 1,), -7, dtype=i32, device="cuda"),
                torch.full((w.E + 1,), -7, dtype=i32, device="cuda"),
                torch.full((w.T, w.k), -7, dtype=i32, device="cuda"),
                torch.full((R,), -7, dtype=i32, device="cuda"),
                torch.full((R, w.H), 3.0, dtype=torch.bfloat16, device="cuda")]

    ref = outputs()
    M.moe_permute(cfg, X, topk, counts, *ref, ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(ws) == 0
    default = M.moe_get_wait_limit_ns()
    try:
        scratch = outputs()
        M.moe_set_wait_limit_ns(0)
        M.moe_permute(cfg, X, topk, counts, *scratch, ws)
        M.moe_set_wait_limit_ns(default)
        torch.cuda.synchronize()  # the launch ended by itself: the context is usable
        assert M.moe_read_device_error(ws) in (0, MOE_ERR_TIMEOUT)
    finally:
        M.moe_set_wait_limit_ns(default)
    M.moe_workspace_init(cfg, ws)  # clears the error word
    got = outputs()
    M.moe_permute(cfg, X, topk, counts, *got, ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(ws) == 0
    n_used = int(ref[0][-1])
    for a, b in zip(got[:3], ref[:3]):
        assert torch.equal(a, b)
    assert torch.equal(got[3][:n_used], ref[3][:n_used])
    assert torch.equal(got[4][:n_used].view(torch.int16), ref[4][:n_used].view(torch.int16))
