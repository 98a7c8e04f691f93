"""Dispatch (moe_permute) against the oracle's counting-sort maps, bit for bit, on
every launch form the library picks:

  * a small dropless layer whose token rows fit the copy CTAs' shared memory: maps
    and row copy in one launch (the Mixtral-style token shape among them);
  * a small layer whose rows do not fit: the one-launch maps, then the row copy;
  * a small layer without Xperm (the maps only, as the gathered-rows GEMM uses);
  * more than 32 experts or more than 16K assignments: chunk histogram, scan and
    scatter, then (with Xperm) the row copy.

Routing is drawn directly (distinct experts per token, a skewed mix that leaves
experts empty), so the maps are checked on patterns the router would rarely give.
Xperm starts filled with a non-zero value: every used row must be the token's row
of X or, for padding rows, zero.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_topk_gb300 as M
import oracle as O
import moe_synth as S

pytestmark = pytest.mark.gpu

# name: (T, H, E, k, skewed, with Xperm)
CASES = {
    "mixtral-shape": (4096, 4096, 8, 2, False, True),
    "rows-beyond-shared-memory": (8000, 4096, 8, 2, False, True),
    "max-small-assignments": (8192, 128, 8, 2, True, True),
    "e32-ragged-skewed": (333, 512, 32, 4, True, True),
    "one-token": (1, 256, 8, 2, False, True),
    "e1-k1": (77, 128, 1, 1, False, True),
    "maps-only": (4096, 4096, 8, 2, True, False),
    "chunked-e64": (1000, 256, 64, 6, True, True),
    "chunked-e256-skewed": (700, 128, 256, 8, True, True),
    "chunked-e40-maps-only": (1000, 256, 40, 5, True, False),
    "chunked-e8-many-tokens": (9000, 128, 8, 2, False, True),
}


def _topk(T, E, k, skewed, seed):
    rng = np.random.default_rng(seed)
    p = None
    if skewed:
        # weights 1/(e+1)^2, with a quarter of the experts never chosen (when E > k allows it)
        w = 1.0 / (np.arange(E) + 1.0) ** 2
        if E >= 4 * k:
            w[rng.permutation(E)[: E // 4]] = 0.0
        p = w / w.sum()
    out = np.empty((T, k), np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_maps_and_rows(name):
    T, H, E, k, skewed, with_x = CASES[name]
    w = S.Workload(name, T=T, H=H, E=E, k=k, F=128)
    cfg = M.config_from(w)
    idx = _topk(T, E, k, skewed, seed=sum(name.encode()))
    X_h = np.random.default_rng(7).standard_normal((T, H)).astype(np.float32)
    X = torch.from_numpy(X_h).to(torch.bfloat16).cuda()
    topk = torch.from_numpy(idx).cuda()
    counts = torch.from_numpy(np.bincount(idx.ravel(), minlength=E).astype(np.int32)).cuda()
    R = M.moe_max_rows(cfg)
    i32 = torch.int32
    offsets = torch.full((E + 1,), -7, dtype=i32, device="cuda")
    tile_offsets = torch.full((E + 1,), -7, dtype=i32, device="cuda")
    row_id_map = torch.full((T, k), -7, dtype=i32, device="cuda")
    slot_src = torch.full((R,), -7, dtype=i32, device="cuda")
    Xperm = torch.full((R, H), 3.0, dtype=torch.bfloat16, device="cuda") if with_x else None
    ws = torch.zeros(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(cfg, ws)
    M.moe_permute(cfg, X if with_x else None, topk, counts, offsets, tile_offsets, row_id_map, slot_src, Xperm, ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(ws) == 0

    d = O.dispatch(O.cfg(w, mirror=True), idx, R=R)
    n_used = int(d["offsets"][-1])
    assert np.array_equal(offsets.cpu().numpy(), d["offsets"])
    assert np.array_equal(tile_offsets.cpu().numpy(), d["tile_offsets"])
    assert np.array_equal(row_id_map.cpu().numpy(), d["row_id_map"])
    assert np.array_equal(slot_src.cpu().numpy()[:n_used], d["slot_src"][:n_used])
    if with_x:
        xp = Xperm[:n_used].view(torch.int16).cpu().numpy()
        xs = X.view(torch.int16).cpu().numpy()
        src = d["slot_src"][:n_used]
        real = src >= 0
        assert np.array_equal(xp[real], xs[src[real] // k])
        assert (xp[~real] == 0).all()
