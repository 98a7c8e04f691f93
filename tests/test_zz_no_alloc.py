"""moe_permute_noalloc, the dispatch call for callers that cannot allocate.

Callers such as a serving runtime whose device memory is a fixed arena sized
at start-up, a plugin handed only its inputs and outputs, or code recording a
CUDA graph cannot hand moe_permute a freshly allocated workspace.  The
allocation-free variant keeps its scratch in a static array inside the
library.  This test calls it through the C ABI twice in a row (different
routings, so the second call runs on scratch the first one left behind) and
checks that every output is bit-identical to moe_permute's.  It also checks
that a configuration beyond the built-in scratch is rejected before launch, and
that the maps-only form (no Xperm, as the gathered-rows GEMM uses) matches too.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_layer_topk_gb300 as M
import moe_synth as S
from helpers import to_dev

pytestmark = pytest.mark.gpu


def _routed(w, seed):
    cfg = M.config_from(w)
    inp = S.host_inputs(w, seed=seed, weights=False)
    X = to_dev(inp["X"])
    W_r = to_dev(inp["W_r"])
    T, E, k = w.T, w.E, w.k
    ws = torch.zeros(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(cfg, ws)
    f32, i32 = torch.float32, torch.int32
    logits = torch.empty(T, E, dtype=f32, device="cuda")
    scores = torch.empty_like(logits)
    topk = torch.empty(T, k, dtype=i32, device="cuda")
    gates = torch.empty(T, k, dtype=f32, device="cuda")
    counts = torch.empty(E, dtype=i32, device="cuda")
    M.moe_router_topk(cfg, X, W_r, None, None, logits, scores, topk, gates, counts, ws)
    return cfg, X, topk, counts, ws


def _outputs(cfg, T, H, E, k):
    R = M.moe_max_rows(cfg)
    i32 = torch.int32
    return dict(offsets=torch.full((E + 1,), -7, dtype=i32, device="cuda"),
                tile_offsets=torch.full((E + 1,), -7, dtype=i32, device="cuda"),
                row_id_map=torch.full((T, k), -7, dtype=i32, device="cuda"),
                slot_src=torch.full((R,), -7, dtype=i32, device="cuda"),
                Xperm=torch.full((R, H), 3.0, dtype=torch.bfloat16, device="cuda"))


def _check_against_workspace_call(w, seed):
    cfg, X, topk, counts, ws = _routed(w, seed)
    ref = _outputs(cfg, w.T, w.H, w.E, w.k)
    got = _outputs(cfg, w.T, w.H, w.E, w.k)
    M.moe_permute(cfg, X, topk, counts, ref["offsets"], ref["tile_offsets"], ref["row_id_map"], ref["slot_src"],
                  ref["Xperm"], ws)
    M.moe_permute_noalloc(cfg, X, topk, counts, got["offsets"], got["tile_offsets"], got["row_id_map"],
                          got["slot_src"], got["Xperm"])
    torch.cuda.synchronize()
    n_used = int(ref["offsets"][-1])
    for name in ["offsets", "tile_offsets", "row_id_map"]:
        assert torch.equal(got[name], ref[name]), name
    assert torch.equal(got["slot_src"][:n_used], ref["slot_src"][:n_used])
    a = got["Xperm"][:n_used].view(torch.int16)
    b = ref["Xperm"][:n_used].view(torch.int16)
    assert torch.equal(a, b)
    # the maps only: Xperm (and X) NULL
    maps = _outputs(cfg, w.T, w.H, w.E, w.k)
    M.moe_permute_noalloc(cfg, None, topk, counts, maps["offsets"], maps["tile_offsets"], maps["row_id_map"],
                          maps["slot_src"], None)
    torch.cuda.synchronize()
    for name in ["offsets", "tile_offsets", "row_id_map"]:
        assert torch.equal(maps[name], ref[name]), name
    assert torch.equal(maps["slot_src"][:n_used], ref["slot_src"][:n_used])
    return ref["row_id_map"].clone()


def test_noalloc_permute_matches_workspace_permute_twice():
    w = S.Workload("noalloc", T=1000, H=256, E=16, k=4, F=128)
    first = _check_against_workspace_call(w, seed=1)
    second = _check_against_workspace_call(w, seed=2)
    assert not torch.equal(first, second)  # the two calls routed differently
    # beyond the built-in scratch: ceil(T/128) * E > 65536 is refused before any launch
    big = M.config_from(S.Workload("big", T=32768 + 128, H=128, E=256, k=2, F=128))
    fake = ctypes.c_void_p(0x1000)
    rc = M.load().moe_permute_noalloc(ctypes.byref(big), *([fake] * 8), None)
    assert rc == 3  # MOE_ERR_WORKSPACE
