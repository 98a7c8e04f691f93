"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign or index, a swapped gate/up half, a transposed operand) fails:
  * selection: brute force over all k-subsets (and group subsets) on integer
    keys, whose sums are exact and whose ties exercise the lower-index rule;
  * gates: closed forms via scipy's softmax/expit;
  * dispatch maps: bijection and ordering invariants plus a brute-force recount;
  * E=1, k=1 reduces to a dense SwiGLU MLP (numpy matmuls, torch autograd);
  * identical experts give gate_sum * MLP(x) (+ shared);
  * the permuted (grouped) route, computed here with numpy from the maps,
    equals the oracle's per-token route;
  * finite differences of L = <dY, Y> in pure double mode;
  * torch autograd of a float64 re-expression of the forward.
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

import moe_synth as S
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(name="t", **kw):
    base = dict(name=name, T=24, H=16, E=8, k=2, F=8)
    base.update(kw)
    return S.Workload(**base)


def inputs(w, seed=0):
    return S.host_inputs(w, seed=seed)


def f32(bits):
    return S.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- generator


def test_generator_deterministic_and_sliceable():
    a = S.normal_bf16(4096, 3, 7, 1.0)
    b = S.normal_bf16(4096, 3, 7, 1.0)
    assert (a == b).all()
    c = S.normal_bf16(100, 3, 7, 1.0, start=1000)
    assert (c == a[1000:1100]).all()
    d = S.normal_bf16(4096, 3, 8, 1.0)
    assert (a != d).mean() > 0.9  # another tensor id is another stream
    x = S.normal_f32(1 << 20, 1, 2, 0.02)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 1e-4


def test_generator_splitmix_words():
    # splitmix64 of state 0 with the golden-ratio increment: first output is a
    # published constant of the generator (Steele et al. 2014 reference code).
    def mix(z):
        m = (1 << 64) - 1
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9 & m
        z = (z ^ (z >> 27)) * 0x94D049BB133111EB & m
        return z ^ (z >> 31)
    assert mix(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF
    base = mix(0 + 0x9E3779B97F4A7C15) ^ (5 * 0xD1B54A32D192ED03 & ((1 << 64) - 1))
    want = [mix((base + (i + 1) * 0x9E3779B97F4A7C15) & ((1 << 64) - 1)) for i in range(4)]
    assert list(S.words(4, 0, 5)) == want


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(20000).astype(np.float32).astype(np.float64) * 10.0 ** rng.integers(-6, 6, 20000)
    v = v.astype(np.float32).astype(np.float64)  # exactly representable in float32
    ties = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -8 * (1 + 2 ** -8)])
    v = np.concatenate([v, ties])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_bf16(v), ref)


# ---------------------------------------------------------------- selection


def brute_select(key, k, n_group=1, topk_group=1, group_score=0):
    E = len(key)
    allowed = list(range(E))
    if n_group > 1:
        per = E // n_group
        gs = []
        for g in range(n_group):
            vals = np.sort(key[g * per:(g + 1) * per])[::-1]
            gs.append(vals[0] + (vals[1] if group_score == 0 and per > 1 else 0))
        best = max(itertools.combinations(range(n_group), topk_group),
                   key=lambda s: (sum(gs[g] for g in s), [-g for g in s]))
        allowed = [e for e in range(E) if e // per in best]
    best = max(itertools.combinations(allowed, k), key=lambda s: (sum(key[e] for e in s), [-e for e in s]))
    return sorted(best, key=lambda e: (-key[e], e))


@pytest.mark.parametrize("E,k,ng,tg", [(8, 2, 1, 1), (8, 3, 1, 1), (8, 8, 1, 1), (16, 4, 4, 2), (16, 2, 4, 1),
                                       (16, 6, 4, 3), (8, 1, 2, 1)])
@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_select_brute_force(E, k, ng, tg, prec):
    rng = np.random.default_rng(E * 100 + k * 10 + ng)
    T = 200
    keys = rng.integers(-4, 5, size=(T, E)).astype(np.float64)  # exact sums, many ties
    w = small(T=T, E=E, k=k, n_group=ng, topk_group=tg, score_fn=1)
    c = O.cfg(w)
    dt = np.float32 if prec == "f32" else np.float64
    idx = O.select(c, keys.astype(dt), keys.astype(dt))
    for t in range(T):
        assert list(idx[t]) == brute_select(keys[t], k, ng, tg), (t, keys[t], idx[t])


def test_select_softmax_uses_logits_and_bias():
    rng = np.random.default_rng(1)
    T, E, k = 64, 8, 2
    logits = rng.standard_normal((T, E))
    bias = rng.standard_normal(E).astype(np.float32)
    w = small(T=T, E=E, k=k)
    c = O.cfg(w)
    sc = sps.softmax(logits, axis=1)
    idx = O.select(c, logits, sc, bias)
    for t in range(T):
        assert list(idx[t]) == brute_select(logits[t] + bias.astype(np.float64), k)


def test_select_golden_ties():
    with open(os.path.join(GOLDEN, "selection_ties.json")) as fh:
        cases = json.load(fh)["cases"]
    for case in cases:
        keys = np.array([case["keys"]], np.float64)
        w = small(T=1, E=keys.shape[1], k=case["k"], n_group=case.get("n_group", 1),
                  topk_group=case.get("topk_group", 1), score_fn=1)
        idx = O.select(O.cfg(w), keys, keys)
        assert list(idx[0]) == case["expect"], case


# ---------------------------------------------------------------- gates


@pytest.mark.parametrize("score_fn,renorm,scale", [(0, 1, 1.0), (0, 0, 1.0), (1, 1, 2.5), (1, 0, 1.0), (0, 1, 2.5)])
def test_gates_closed_form(score_fn, renorm, scale):
    w = small(T=40, E=8, k=3, score_fn=score_fn, renorm=renorm, gate_scale=scale)
    inp = inputs(w)
    c = O.cfg(w)
    logits, scores = O.router(c, inp["X"], inp["W_r"])
    x = f32(inp["X"])
    assert np.allclose(logits, x @ inp["W_r"].astype(np.float64).T, rtol=0, atol=1e-12)
    if score_fn == 0:
        assert np.allclose(scores, sps.softmax(logits, axis=1), atol=1e-15)
    else:
        assert np.allclose(scores, sps.expit(logits), atol=1e-15)
    idx = O.select(c, logits, scores)
    g = O.gates(c, logits, idx)
    for t in range(w.T):
        sel = idx[t]
        if score_fn == 0 and renorm:
            want = scale * sps.softmax(logits[t, sel])
        elif score_fn == 0:
            want = scale * sps.softmax(logits[t])[sel]
        elif renorm:
            s = sps.expit(logits[t, sel])
            want = scale * s / s.sum()
        else:
            want = scale * sps.expit(logits[t, sel])
        assert np.allclose(g[t], want, rtol=1e-13, atol=1e-15)
        if renorm:
            assert abs(g[t].sum() - scale) < 1e-12


@pytest.mark.parametrize("score_fn,renorm,scale", [(0, 1, 1.0), (0, 0, 1.0), (1, 1, 2.5), (1, 0, 1.0)])
def test_router_dlogits_finite_differences(score_fn, renorm, scale):
    """router_dlogits is the gradient of <dgates, gates(logits)> for a fixed selection:
    central differences of the (closed-form pinned) gates, one logit column at a time."""
    w = small(T=6, E=8, k=3, score_fn=score_fn, renorm=renorm, gate_scale=scale)
    inp = inputs(w)
    c = O.cfg(w)
    logits, scores = O.router(c, inp["X"], inp["W_r"])
    idx = O.select(c, logits, scores)
    g = O.gates(c, logits, idx)
    dg = np.random.default_rng(3).standard_normal((w.T, w.k))
    dl = O.router_dlogits(c, logits, idx, g, dg)
    h = 1e-6
    for e in range(w.E):
        lp, lm = logits.copy(), logits.copy()
        lp[:, e] += h
        lm[:, e] -= h
        fd = ((O.gates(c, lp, idx) - O.gates(c, lm, idx)) * dg).sum(axis=1) / (2 * h)
        assert np.allclose(dl[:, e], fd, rtol=1e-6, atol=1e-8), (e, dl[:, e], fd)


def test_router_logit_bias_enters_logits():
    w = small(T=16, E=8, k=2, skew=True)
    inp = inputs(w)
    b = S.skew_logit_bias(8, n_empty=2)
    c = O.cfg(w)
    l0, _ = O.router(c, inp["X"], inp["W_r"])
    l1, _ = O.router(c, inp["X"], inp["W_r"], b)
    assert np.allclose(l1 - l0, b.astype(np.float64)[None, :], atol=1e-12)


# ---------------------------------------------------------------- dispatch


@pytest.mark.parametrize("align", [1, 4, 128])
def test_dispatch_invariants(align):
    rng = np.random.default_rng(align)
    T, E, k = 300, 16, 4
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[:50, 0] = 3  # skew one expert
    for t in range(50):
        row = idx[t]
        if (row[1:] == 3).any():
            row[1:][row[1:] == 3] = [e for e in range(E) if e not in row][: (row[1:] == 3).sum()]
    idx[:, :][idx == 7] = 8  # make expert 7 empty where possible
    for t in range(T):
        if len(set(idx[t])) < k:
            idx[t] = rng.choice([e for e in range(E) if e != 7], size=k, replace=False)
    w = small(T=T, E=E, k=k)
    c = O.cfg(w, align=align, BM=128)
    d = O.dispatch(c, idx)
    counts, off, rim, src = d["counts"], d["offsets"], d["row_id_map"], d["slot_src"]
    assert counts.sum() == T * k
    assert (counts == np.bincount(idx.ravel(), minlength=E)).all()
    assert counts[7] == 0
    assert off[0] == 0 and (np.diff(off) % align == 0).all() and (np.diff(off) >= counts).all()
    assert (np.diff(off) - counts < align).all()
    assert (d["tile_offsets"] == np.concatenate([[0], np.cumsum((counts + 127) // 128)])).all()
    flat = rim.ravel()
    assert len(np.unique(flat)) == T * k                          # injective
    assert (src[flat] == np.arange(T * k)).all()                  # slot_src o row_id_map = id
    for e in range(E):
        seg = src[off[e]:off[e + 1]]
        real, pad = seg[:counts[e]], seg[counts[e]:]
        assert (pad == -1).all()
        assert (idx.ravel()[real] == e).all()
        assert (np.diff(real // k) > 0).all()                     # stable token order
    # brute-force recount: slot - offset = number of earlier tokens that chose e
    onehot = np.zeros((T, E), np.int64)
    for t in range(T):
        onehot[t, idx[t]] = 1
    before = np.cumsum(onehot, axis=0) - onehot
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            assert rim[t, j] == off[e] + before[t, e]


# ---------------------------------------------------------------- layer values


def dense_swiglu(x, w13, w2):
    F = w13.shape[0] // 2
    g = x @ w13[:F].T
    u = x @ w13[F:].T
    return (g * sps.expit(g) * u) @ w2.T


def test_e1_k1_is_dense_swiglu():
    w = small(T=32, H=16, E=1, k=1, F=24)
    inp = inputs(w)
    out = O.full_layer(w, inp, mirror=False)
    x, w13, w2 = f32(inp["X"]), f32(inp["W13"][0]), f32(inp["W2"][0])
    assert np.allclose(out["Y"], dense_swiglu(x, w13, w2), rtol=1e-12, atol=1e-14)
    assert (out["topk_idx"] == 0).all() and np.allclose(out["gates"], 1.0)
    assert np.abs(out["dW_r"]).max() == 0.0 and np.abs(out["dlogits"]).max() == 0.0
    # backward of the dense MLP by torch autograd
    xt = torch.tensor(x, requires_grad=True)
    a = torch.tensor(w13, requires_grad=True)
    b = torch.tensor(w2, requires_grad=True)
    F = w.F
    g, u = xt @ a[:F].T, xt @ a[F:].T
    y = (torch.nn.functional.silu(g) * u) @ b.T
    (y * torch.tensor(f32(inp["dY"]))).sum().backward()
    assert np.allclose(out["dX"], xt.grad.numpy(), rtol=1e-11, atol=1e-13)
    assert np.allclose(out["dW13"][0], a.grad.numpy(), rtol=1e-11, atol=1e-13)
    assert np.allclose(out["dW2"][0], b.grad.numpy(), rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("score_fn,scale,fs", [(0, 1.0, 0), (1, 2.5, 12)])
def test_identical_experts(score_fn, scale, fs):
    w = small(T=20, H=16, E=4, k=2, F=8, score_fn=score_fn, gate_scale=scale, F_shared=fs)
    inp = inputs(w)
    inp["W13"] = np.repeat(inp["W13"][:1], 4, axis=0)
    inp["W2"] = np.repeat(inp["W2"][:1], 4, axis=0)
    out = O.full_layer(w, inp, mirror=False)
    x = f32(inp["X"])
    want = scale * dense_swiglu(x, f32(inp["W13"][0]), f32(inp["W2"][0]))
    if fs:
        want += dense_swiglu(x, f32(inp["W13_s"]), f32(inp["W2_s"]))
    assert np.allclose(out["Y"], want, rtol=1e-12, atol=1e-14)
    # with renormalised gates the router sees no gradient when experts agree
    assert np.abs(out["dlogits"]).max() < 1e-12


def test_permuted_route_equals_per_token_route():
    w = small(T=40, H=16, E=6, k=3, F=8, score_fn=1, gate_scale=2.5, F_shared=8)
    inp = inputs(w)
    out = O.full_layer(w, inp, mirror=False)
    x = f32(inp["X"])
    off, src, cnt = out["offsets"], out["slot_src"], out["counts"]
    R = off[-1]
    yperm = np.zeros((R, w.H))
    for e in range(w.E):
        rows = src[off[e]:off[e] + cnt[e]] // w.k
        yperm[off[e]:off[e] + cnt[e]] = dense_swiglu(x[rows], f32(inp["W13"][e]), f32(inp["W2"][e]))
    y = np.zeros((w.T, w.H))
    for t in range(w.T):
        for j in range(w.k):
            y[t] += out["gates"][t, j] * yperm[out["row_id_map"][t, j]]
    y += dense_swiglu(x, f32(inp["W13_s"]), f32(inp["W2_s"]))
    assert np.allclose(out["Y"], y, rtol=1e-12, atol=1e-14)


def test_mirror_mode_close_to_pure():
    w = small(T=32, H=64, E=4, k=2, F=64)
    inp = inputs(w)
    a = O.full_layer(w, inp, mirror=True)
    b = O.full_layer(w, inp, mirror=False)
    for key in ["Y", "dX", "dW13", "dW2"]:
        err = np.abs(a[key] - b[key]).max() / np.abs(b[key]).max()
        assert 0 < err < 2e-2, key


# ---------------------------------------------------------------- backward


def loss_pure(w, inp, fixed_idx=None):
    c = O.cfg(w, mirror=False)
    logits, scores = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    idx = O.select(c, logits, scores, inp.get("sel_bias"))
    if fixed_idx is not None and not np.array_equal(idx, fixed_idx):
        return None
    g = O.gates(c, logits, idx)
    Y = O.tokens(c, inp, idx, logits, g, want_bwd=False)["Y"]
    return float((Y * f32(inp["dY"])).sum())


FD_STEP = 2.0 ** -20


def fd_check(w, inp, name, index, analytic, bits):
    """Central difference at an element set to 0, perturbed by +-2^-20 (exact in bf16 and fp32)."""
    base = dict(inp)
    arrs = {}
    for sgn in (+1, -1):
        a = inp[name].copy()
        if bits:
            a[index] = int(np.array([sgn * FD_STEP], np.float32).view(np.uint32)[0] >> 16)
        else:
            a[index] = sgn * FD_STEP
        arrs[sgn] = a
    c = O.cfg(w, mirror=False)
    l0, s0 = O.router(c, inp["X"], inp["W_r"], inp.get("logit_bias"))
    idx0 = O.select(c, l0, s0, inp.get("sel_bias"))
    vals = []
    for sgn in (+1, -1):
        base[name] = arrs[sgn]
        v = loss_pure(w, base, idx0)
        if v is None:
            return None
        vals.append(v)
    fd = (vals[0] - vals[1]) / (2 * FD_STEP)
    return fd, analytic


FD_CASES = [
    small("fd-softmax", T=10, H=8, E=4, k=2, F=6),
    small("fd-softmax-norenorm", T=10, H=8, E=4, k=2, F=6, renorm=0),
    small("fd-sigmoid-groups", T=10, H=8, E=8, k=3, F=6, score_fn=1, gate_scale=2.5, n_group=4,
          topk_group=2, sel_bias=True, F_shared=4),
    small("fd-sigmoid-norenorm", T=10, H=8, E=4, k=2, F=6, score_fn=1, renorm=0, skew=True),
]


@pytest.mark.parametrize("w", FD_CASES, ids=[w.name for w in FD_CASES])
def test_finite_differences(w):
    rng = np.random.default_rng(7)
    inp = inputs(w)
    if w.skew:
        inp["logit_bias"] = rng.standard_normal(w.E).astype(np.float32) * 0.3
    # zero the probed elements so that +-2^-20 is exactly representable
    probes = {
        "X": [tuple(rng.integers(0, s) for s in inp["X"].shape) for _ in range(6)],
        "W13": [tuple(rng.integers(0, s) for s in inp["W13"].shape) for _ in range(6)],
        "W2": [tuple(rng.integers(0, s) for s in inp["W2"].shape) for _ in range(6)],
        "W_r": [tuple(rng.integers(0, s) for s in inp["W_r"].shape) for _ in range(6)],
    }
    if w.F_shared:
        probes["W13_s"] = [tuple(rng.integers(0, s) for s in inp["W13_s"].shape) for _ in range(4)]
        probes["W2_s"] = [tuple(rng.integers(0, s) for s in inp["W2_s"].shape) for _ in range(4)]
    if w.skew:
        probes["logit_bias"] = [(e,) for e in range(w.E)]
    for name, idxs in probes.items():
        for ix in idxs:
            inp[name][ix] = 0
    out = O.full_layer(w, inp, mirror=False)
    grads = {"X": out["dX"], "W13": out["dW13"], "W2": out["dW2"], "W_r": out["dW_r"],
             "W13_s": out.get("dW13_s"), "W2_s": out.get("dW2_s"), "logit_bias": out["dlogit_bias"]}
    checked = 0
    scale = max(np.abs(g).max() for g in grads.values() if g is not None)
    for name, idxs in probes.items():
        bits = inp[name].dtype == np.uint16
        for ix in idxs:
            r = fd_check(w, inp, name, ix, grads[name][ix], bits)
            if r is None:
                continue  # selection changed under the probe
            fd, an = r
            assert abs(fd - an) <= 1e-6 * scale + 1e-7 * abs(an), (name, ix, fd, an)
            checked += 1
    assert checked >= 20


@pytest.mark.parametrize("w", FD_CASES, ids=[w.name for w in FD_CASES])
def test_autograd_matches_backward(w):
    """torch float64 autograd of the same layer, with the oracle's selection held fixed."""
    inp = inputs(w)
    if w.skew:
        inp["logit_bias"] = np.random.default_rng(3).standard_normal(w.E).astype(np.float32) * 0.3
    out = O.full_layer(w, inp, mirror=False)
    idx = torch.tensor(out["topk_idx"], dtype=torch.long)
    X = torch.tensor(f32(inp["X"]), requires_grad=True)
    Wr = torch.tensor(inp["W_r"].astype(np.float64), requires_grad=True)
    lb = torch.tensor((inp["logit_bias"] if inp.get("logit_bias") is not None else np.zeros(w.E)).astype(np.float64),
                      requires_grad=True)
    W13 = torch.tensor(f32(inp["W13"]), requires_grad=True)
    W2 = torch.tensor(f32(inp["W2"]), requires_grad=True)
    logits = X @ Wr.T + lb
    sel_logits = torch.gather(logits, 1, idx)
    if w.score_fn == 0:
        g = torch.softmax(sel_logits, 1) if w.renorm else torch.gather(torch.softmax(logits, 1), 1, idx)
    else:
        s = torch.sigmoid(sel_logits)
        g = s / s.sum(1, keepdim=True) if w.renorm else s
    g = g * w.gate_scale
    Y = torch.zeros(w.T, w.H, dtype=torch.float64)
    F = w.F
    for t in range(w.T):
        for j in range(w.k):
            e = int(idx[t, j])
            h1 = W13[e] @ X[t]
            a = torch.nn.functional.silu(h1[:F]) * h1[F:]
            Y[t] = Y[t] + g[t, j] * (W2[e] @ a)
    extra = []
    if w.F_shared:
        W13s = torch.tensor(f32(inp["W13_s"]), requires_grad=True)
        W2s = torch.tensor(f32(inp["W2_s"]), requires_grad=True)
        h1 = X @ W13s.T
        Fs = w.F_shared
        Y = Y + (torch.nn.functional.silu(h1[:, :Fs]) * h1[:, Fs:]) @ W2s.T
        extra = [(W13s, "dW13_s"), (W2s, "dW2_s")]
    (Y * torch.tensor(f32(inp["dY"]))).sum().backward()
    assert np.allclose(out["Y"], Y.detach().numpy(), rtol=1e-11, atol=1e-13)
    for t, key in [(X, "dX"), (Wr, "dW_r"), (W13, "dW13"), (W2, "dW2"), (lb, "dlogit_bias")] + extra:
        ref = t.grad.numpy()
        assert np.allclose(out[key], ref, rtol=1e-10, atol=1e-12 * max(1.0, np.abs(ref).max())), key


# ---------------------------------------------------------------- FP8 E4M3 (block-scaled)


def torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 1e-2,
                        rng.standard_normal(5000) * 2.0 ** -8])
    grid = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    grid = grid[np.isfinite(grid)]
    mids = (np.sort(grid)[1:] + np.sort(grid)[:-1]) / 2  # exact ties between neighbours
    v = np.concatenate([v, grid, mids[np.abs(mids) <= 448]]).astype(np.float32).astype(np.float64)
    assert np.array_equal(O.e4m3(v), torch_e4m3(v))


def torch_qdq_rows(x, blk=128):
    """Independent block quantize-dequantize: torch's e4m3 cast with power-of-two scales."""
    x = np.asarray(x, np.float64)
    out = np.empty_like(x)
    for b0 in range(0, x.shape[-1], blk):
        blkv = x[..., b0:b0 + blk]
        amax = np.abs(blkv).max(axis=-1, keepdims=True)
        e = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / 448.0)), 0.0)
        s = 2.0 ** e
        out[..., b0:b0 + blk] = torch_e4m3(blkv / s) * s
    return out


def test_block_scales_power_of_two_and_tight():
    rng = np.random.default_rng(12)
    for scale in [1e-3, 1.0, 37.0, 5e3]:
        x = rng.standard_normal(1024) * scale
        q = O.qdq_blocks(x, 128)
        assert np.array_equal(q, torch_qdq_rows(x[None])[0])
        assert np.array_equal(O.qdq_blocks(q, 128), q)  # idempotent
        for b in range(8):
            blk = x[128 * b:128 * b + 128]
            amax = np.abs(blk).max()
            s = 2.0 ** np.ceil(np.log2(amax / 448))
            assert 224 < amax / s <= 448
    assert np.array_equal(O.qdq_blocks(np.zeros(256), 128), np.zeros(256))


def test_weight_blocks_are_128x128():
    rng = np.random.default_rng(13)
    W = (rng.standard_normal((2, 256, 384)) * 0.02).astype(np.float32)
    W[1, :128, 128:256] *= 50  # one block with a larger scale
    bits = torch.from_numpy(W).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q = S.bf16_bits_to_f32(O.qdq_weights(bits)).astype(np.float64)
    wf = S.bf16_bits_to_f32(bits).astype(np.float64)
    for m in range(2):
        for r0 in range(0, 256, 128):
            for c0 in range(0, 384, 128):
                blk = wf[m, r0:r0 + 128, c0:c0 + 128]
                amax = np.abs(blk).max()
                s = 2.0 ** np.ceil(np.log2(amax / 448))
                assert np.array_equal(q[m, r0:r0 + 128, c0:c0 + 128], torch_e4m3(blk / s) * s)


def test_fp8_e1_k1_is_dense_swiglu_on_quantized_operands():
    """E=1, k=1 in FP8 mode: every GEMM operand block-quantized, numpy matmuls in double."""
    w = small(T=200, H=256, E=1, k=1, F=256, fp8=True)
    inp = inputs(w)

    def ramp(bits, axis):
        # alternate 64-entry runs of size 1 and 2^-12 along `axis`: power-of-two scales make
        # E4M3 rounding scale-invariant except in the subnormal range, so a block of the wrong
        # size (sharing a scale across a quiet and a loud run, or not) shows up there
        v = torch.from_numpy(S.bf16_bits_to_f32(bits).copy())
        n = v.shape[axis]
        f = torch.tensor([2.0 ** (-12 * ((i // 64) % 2)) for i in range(n)], dtype=torch.float32)
        v = v * (f if axis == v.dim() - 1 else f[:, None])
        return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    inp["X"] = ramp(ramp(inp["X"], 1), 0)
    inp["dY"] = ramp(ramp(inp["dY"], 1), 0)
    out = O.full_layer(w, inp, mirror=False)
    x = f32(inp["X"])
    W13 = S.bf16_bits_to_f32(O.qdq_weights(inp["W13"]))[0].astype(np.float64)
    W2 = S.bf16_bits_to_f32(O.qdq_weights(inp["W2"]))[0].astype(np.float64)
    F = w.F
    xq = torch_qdq_rows(x)
    g, u = xq @ W13[:F].T, xq @ W13[F:].T
    a = g * sps.expit(g) * u
    y = torch_qdq_rows(a) @ W2.T
    assert np.allclose(out["Y"], y, rtol=1e-12, atol=1e-13)
    dy = f32(inp["dY"])
    dA = torch_qdq_rows(dy) @ W2
    sg = sps.expit(g)
    dG, dU = dA * u * sg * (1 + g * (1 - sg)), dA * g * sg
    dgu = torch_qdq_rows(np.concatenate([dG, dU], axis=1))
    dx = dgu @ W13
    assert np.allclose(out["dX"], dx, rtol=1e-11, atol=1e-12)
    # wgrad operands: 128-token blocks per column
    colq = lambda m: torch_qdq_rows(m.T.copy()).T
    assert np.allclose(out["dW2"][0], colq(dy).T @ colq(a), rtol=1e-11, atol=1e-12)
    assert np.allclose(out["dW13"][0], colq(np.concatenate([dG, dU], axis=1)).T @ colq(x), rtol=1e-11, atol=1e-12)


def test_fp8_layer_close_to_bf16_layer():
    w = small(T=256, H=256, E=4, k=2, F=256)
    inp = inputs(w)
    a = O.full_layer(w, inp, mirror=True)
    b = O.full_layer(w.replace(fp8=True), inp, mirror=True)
    assert np.array_equal(a["topk_idx"], b["topk_idx"])
    # E4M3 keeps 3 mantissa bits: ~2-3% RMS noise per quantized operand, compounded over
    # the two chained GEMMs of an expert; a dropped or wrong term would be O(1)
    for key in ["Y", "dX", "dW13", "dW2"]:
        err = np.sqrt(np.mean((a[key] - b[key]) ** 2) / np.mean(a[key] ** 2))
        assert 1e-3 < err < 0.1, (key, err)


# ---------------------------------------------------------------- capacity-controlled dropping


def test_capacity_dispatch_keeps_first_tokens():
    rng = np.random.default_rng(21)
    T, E, k = 200, 8, 2
    idx = np.stack([rng.choice(E, size=k, replace=False, p=[.4, .2, .1, .1, .05, .05, .05, .05])
                    for _ in range(T)]).astype(np.int32)
    w = small(T=T, E=E, k=k)
    c = O.cfg(w, align=128)
    full = O.dispatch(c, idx)
    same = O.dispatch(c, idx, capacity=int(full["counts"].max()))
    for key in full:
        assert np.array_equal(full[key], same[key]), key
    cap = 30
    d = O.dispatch(c, idx, capacity=cap)
    assert (d["counts"] == np.minimum(np.bincount(idx.ravel(), minlength=E), cap)).all()
    rim = d["row_id_map"]
    for e in range(E):
        pos = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]  # token order
        for n, (t, j) in enumerate(pos):
            if n < cap:
                assert rim[t, j] == d["offsets"][e] + n
            else:
                assert rim[t, j] == -1


def test_capacity_identical_experts_sum_kept_gates():
    w = small(T=60, H=16, E=4, k=2, F=8, score_fn=1, gate_scale=2.0)
    inp = inputs(w)
    inp["W13"] = np.repeat(inp["W13"][:1], 4, axis=0)
    inp["W2"] = np.repeat(inp["W2"][:1], 4, axis=0)
    out = O.full_layer(w, inp, mirror=False, capacity=20)
    kept = out["row_id_map"] >= 0
    assert (~kept).any()
    mlp = dense_swiglu(f32(inp["X"]), f32(inp["W13"][0]), f32(inp["W2"][0]))
    want = (out["gates"] * kept).sum(1, keepdims=True) * mlp
    assert np.allclose(out["Y"], want, rtol=1e-12, atol=1e-14)
    assert (out["dgates"][~kept] == 0).all()


def test_capacity_finite_differences():
    w = small("fd-cap", T=12, H=8, E=4, k=2, F=6, score_fn=0)
    rng = np.random.default_rng(5)
    inp = inputs(w)
    probes = [tuple(rng.integers(0, s) for s in inp["W_r"].shape) for _ in range(6)]
    probes += [("X",) + tuple(rng.integers(0, s) for s in inp["X"].shape) for _ in range(4)]
    for p in probes:
        if p[0] == "X":
            inp["X"][p[1:]] = 0
        else:
            inp["W_r"][p] = 0
    cap = 4
    out = O.full_layer(w, inp, mirror=False, capacity=cap)
    assert (out["row_id_map"] < 0).any()
    c = O.cfg(w, mirror=False)

    def loss(i2):
        lg, sc = O.router(c, i2["X"], i2["W_r"])
        idx = O.select(c, lg, sc)
        if not np.array_equal(idx, out["topk_idx"]):
            return None
        g = O.gates(c, lg, idx)
        d = O.dispatch(c, idx, capacity=cap)
        Y = O.tokens(c, i2, idx, lg, g, want_bwd=False, kept=(d["row_id_map"] >= 0).astype(np.int32))["Y"]
        return float((Y * f32(i2["dY"])).sum())

    checked = 0
    for p in probes:
        vals = []
        for sgn in (1, -1):
            i2 = dict(inp)
            if p[0] == "X":
                a = inp["X"].copy()
                a[p[1:]] = int(np.array([sgn * FD_STEP], np.float32).view(np.uint32)[0] >> 16)
                i2["X"] = a
            else:
                a = inp["W_r"].copy()
                a[p] = sgn * FD_STEP
                i2["W_r"] = a
            vals.append(loss(i2))
        if None in vals:
            continue
        fd = (vals[0] - vals[1]) / (2 * FD_STEP)
        an = out["dX"][p[1:]] if p[0] == "X" else out["dW_r"][p]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (p, fd, an)
        checked += 1
    assert checked >= 6


def test_capacity_priority_policy_brute_force():
    rng = np.random.default_rng(22)
    T, E, k = 150, 6, 3
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    pri = rng.integers(0, 5, size=(T, k)).astype(np.float64)  # many equal priorities
    w = small(T=T, E=E, k=k)
    c = O.cfg(w, align=8)
    cap = 40
    d = O.dispatch(c, idx, capacity=cap, priority=pri)
    flat_e, flat_p = idx.ravel(), pri.ravel()
    keep = np.zeros(T * k, bool)
    for i in range(T * k):
        same = np.flatnonzero(flat_e == flat_e[i])
        better = ((flat_p[same] > flat_p[i]) | ((flat_p[same] == flat_p[i]) & (same < i))).sum()
        keep[i] = better < cap
    assert np.array_equal(d["row_id_map"].ravel() >= 0, keep)
    assert (d["counts"] == np.minimum(np.bincount(flat_e, minlength=E), cap)).all()
    rim = d["row_id_map"].ravel()
    for e in range(E):
        kept_i = [i for i in range(T * k) if flat_e[i] == e and keep[i]]
        assert list(rim[kept_i]) == list(range(d["offsets"][e], d["offsets"][e] + len(kept_i)))
    # constant priority is the position policy
    flat = O.dispatch(c, idx, capacity=cap, priority=np.ones((T, k)))
    pos = O.dispatch(c, idx, capacity=cap)
    for key in pos:
        assert np.array_equal(flat[key], pos[key]), key


def test_capacity_drop_by_gate_keeps_largest_gates():
    w = small(T=80, H=16, E=4, k=2, F=8, score_fn=0)
    inp = inputs(w)
    inp["W13"] = np.repeat(inp["W13"][:1], 4, axis=0)
    inp["W2"] = np.repeat(inp["W2"][:1], 4, axis=0)
    cap = 25
    out = O.full_layer(w, inp, mirror=False, capacity=cap, drop_by_gate=True)
    kept = out["row_id_map"] >= 0
    g, idx = out["gates"], out["topk_idx"]
    for e in range(4):
        sel = idx == e
        if sel.sum() > cap:
            assert kept[sel].sum() == cap
            assert g[sel & kept].min() >= g[sel & ~kept].max()
    mlp = dense_swiglu(f32(inp["X"]), f32(inp["W13"][0]), f32(inp["W2"][0]))
    assert np.allclose(out["Y"], (g * kept).sum(1, keepdims=True) * mlp, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- gated (memory-efficient) form


@pytest.mark.parametrize("wname", ["pins-softmax", "pins-sigmoid-shared"])
def test_gated_form_is_the_same_function(wname):
    """Gate before the down projection vs gate in the combine: identical in exact arithmetic."""
    w = {"pins-softmax": small("g1", T=40, H=32, E=4, k=2, F=16),
         "pins-sigmoid-shared": small("g2", T=40, H=32, E=8, k=3, F=16, F_shared=16, score_fn=1, gate_scale=2.5,
                                      n_group=2, topk_group=1)}[wname]
    inp = inputs(w)
    a = O.full_layer(w, inp, mirror=False)
    b = O.full_layer(w, inp, mirror=False, gated=True)
    for key in ["Y", "dX", "dgates", "dW13", "dW2", "dW_r"]:
        assert np.allclose(a[key], b[key], rtol=1e-12, atol=1e-14), key
    # with bf16 storage the two forms round in different places, within bf16 noise
    am = O.full_layer(w, inp, mirror=True)
    bm = O.full_layer(w, inp, mirror=True, gated=True)
    for key in ["Y", "dX", "dW13", "dW2"]:
        err = np.abs(am[key] - bm[key]).max() / np.abs(am[key]).max()
        assert 0 < err < 2e-2, (key, err)


# ---------------------------------------------------------------- sampled weight gradients
@pytest.mark.parametrize("mode", ["mirror", "pure", "fp8", "gated", "kept"])
def test_expert_wgrad_cols_equals_the_full_gradient(mode):
    """The column-sampled expert weight gradient (used where the full one is out of reach)
    reproduces the entries of the full expert_wgrad bit for bit: the same roundings, the
    same 128-token FP8 blocks (the expert holds more than one 512-token chunk here) and the
    same summation order, for routed experts and the shared one."""
    w = small("wc", T=700, H=256, E=2, k=2, F=256, F_shared=128, score_fn=1, gate_scale=2.5,
              fp8=mode == "fp8")
    inp = inputs(w)
    if mode == "fp8":
        inp = O.fp8_inputs(inp)
    c = O.cfg(w, mirror=mode != "pure", gated=mode == "gated")
    logits, scores = O.router(c, inp["X"], inp["W_r"])
    idx = O.select(c, logits, scores)
    g = O.gates(c, logits, idx)
    kept = None
    if mode == "kept":
        kept = (np.arange(w.T * w.k).reshape(w.T, w.k) % 3 != 0).astype(np.int32)
    counts = np.bincount(idx.ravel(), minlength=w.E)
    assert counts.max() > 512  # more than one chunk
    for e, F in [(int(np.argmax(counts)), w.F), (-1, w.F_shared)]:
        cols = np.array([0, 5, 77, F - 1], np.int32)
        full13, full2 = O.expert_wgrad(c, inp, idx, g, e, kept=kept)
        r13, c2 = O.expert_wgrad_cols(c, inp, idx, g, e, cols, kept=kept)
        assert np.array_equal(r13[:len(cols)], full13[cols])
        assert np.array_equal(r13[len(cols):], full13[F + cols])
        assert np.array_equal(c2, full2[:, cols])
        assert np.abs(c2).max() > 0
