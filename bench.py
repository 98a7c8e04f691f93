"""Benchmark: one MoE layer forward+backward step on GB300, tokens/s.

Workload (default): the DeepSeek-V3-style layer, the largest that fits one GPU:
T=8192 tokens, H=7168, 256 routed experts with top-8 and one always-on shared
expert, sigmoid router with a selection-only bias, group-limited routing (8
groups, top-4 groups), gates renormalised and scaled by 2.5, SwiGLU FFN=2048,
BF16 tokens and expert weights, FP32 router; seeded synthetic inputs.  The other
workloads (Mixtral-, Qwen3-style, skewed, FP8) are selectable with --workload.
A step is one pass of the whole layer: route, permute, grouped SwiGLU MLP,
combine, and their backwards (dX, grouped dgrad and wgrad, router gradient).

Prints one JSON line.  `value` is tokens/s with inputs resident in HBM: T over
the median time of one replay of the step captured as a CUDA graph (K replays
after W warm-up replays, CUDA events between replays).  A second pass gives
the per-stage times, the grouped GEMM's roofline and the HBM stages'
bandwidths: the step captured again with a CUDA event between the stages (the
events become nodes of the graph), replayed K times, so that the stage times
hold no host launch gaps (K eager steps with the same events where the capture
of events is unavailable).  Every eager step carries an NVTX range per stage.
`e2e` is the same metric through the C ABI with the step's inputs copied in
from pinned host memory and its outputs (Y, dX) copied back inside the timed
region (the step on each of two buffer sets replayed as a CUDA graph, the copies
on a second stream).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as S  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "MoE layer fwd+bwd tokens/s and grouped-GEMM TFLOPS (% BF16 peak) on 1 GB300"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity on one process).

    The benchmark reports the slowest rank's time: every rank runs its own replica of
    the layer on its own GPU, and the job is done when the last one finishes."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


# ---------------------------------------------------------------- inputs


def upload_normal_bf16(shape, seed, tid, std, device, chunk_elems=1 << 27):
    import torch
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    stage = torch.empty(min(n, chunk_elems), dtype=torch.bfloat16, pin_memory=True)
    for s in range(0, n, chunk_elems):
        m = min(chunk_elems, n - s)
        S.fill_normal_bf16(stage.data_ptr(), m, seed, tid, std, start=s)
        out[s:s + m].copy_(stage[:m], non_blocking=False)
    return out.view(*shape)


def device_inputs(w, seed, device):
    import torch
    import mixture_experts_layer_topk_gb300 as M
    T, H, E, F = w.T, w.H, w.E, w.F
    W_r = torch.from_numpy(S.normal_f32(E * H, seed, S.TID_WR, w.wr_std)).view(E, H).to(device)
    lb = torch.from_numpy(S.skew_logit_bias(E)).to(device) if w.skew else None
    sb = torch.from_numpy(S.normal_f32(E, seed, S.TID_SEL_BIAS, 0.1)).to(device) if w.sel_bias else None
    W13 = upload_normal_bf16((E, 2 * F, H), seed, S.TID_W13, w.w_std, device)
    W2 = upload_normal_bf16((E, H, F), seed, S.TID_W2, w.w_std, device)
    W13s = W2s = None
    if w.F_shared:
        W13s = upload_normal_bf16((2 * w.F_shared, H), seed, S.TID_W13S, w.w_std, device)
        W2s = upload_normal_bf16((H, w.F_shared), seed, S.TID_W2S, w.w_std, device)
    weights = M.LayerWeights(W_r=W_r, W13=W13, W2=W2, logit_bias=lb, sel_bias=sb, W13_s=W13s, W2_s=W2s)
    X = upload_normal_bf16((T, H), seed, S.TID_X, w.x_std, device)
    dY = upload_normal_bf16((T, H), seed, S.TID_DY, w.dy_std, device)
    return weights, X, dY


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_id)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


# ---------------------------------------------------------------- our arm


STAGES = ["router", "permute", "quant_w", "gemm_fwd", "combine", "combine_bwd", "gemm_bwd", "router_bwd",
          "permute_bwd"]


def run_step(layer, X, dY, ev=None):
    """One forward+backward through the C ABI, with an NVTX range around each stage;
    ev: list of len(STAGES)+1 events recorded between the stages (on the current stream,
    also while it is being captured)."""
    import torch
    import mixture_experts_layer_topk_gb300 as M
    c, w = layer.cfg, layer.w
    nvtx = torch.cuda.nvtx

    def rec(i):
        if i > 0:
            nvtx.range_pop()
        if ev is not None:
            ev[i].record()
        if i < len(STAGES):
            nvtx.range_push(STAGES[i])

    rec(0)
    M.moe_router_topk(c, X, w.W_r, w.logit_bias, w.sel_bias, layer.logits, layer.scores, layer.topk_idx,
                      layer.gates, layer.counts, layer.ws)
    rec(1)
    # gathered rows: the dispatch writes the maps only and FC1 reads X through them
    M.moe_permute(c, None if layer.gather_rows else X, layer.topk_idx, layer.counts, layer.offsets,
                  layer.tile_offsets, layer.row_id_map, layer.slot_src, layer.Xperm, layer.ws)
    rec(2)
    if layer.fp8:
        # the step re-quantizes the weights (as after every optimizer update) inside the timed region
        layer.quantize_weights()
    rec(3)
    if layer.fp8:
        M.moe_grouped_swiglu_mlp_fp8(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.W13q, layer.W13sc,
                                     layer.W2q, layer.W2sc, layer.GU, layer.A, layer.Yperm,
                                     X if c.F_shared else None, layer.W13q_s, layer.W13sc_s, layer.W2q_s,
                                     layer.W2sc_s, layer.GU_s, layer.A_s, layer.Yshared, layer.fp8_ws, layer.ws)
    elif layer.gather_rows:
        M.moe_grouped_swiglu_mlp_gather(c, X, layer.slot_src, layer.offsets, layer.tile_offsets, w.W13, w.W2,
                                        layer.GU, layer.A, layer.Yperm, w.W13_s, w.W2_s, layer.GU_s, layer.A_s,
                                        layer.Yshared, layer.ws)
    elif layer.memory_efficient:
        # gates applied before FC2 (gated rows), so the combine is a plain sum
        M.moe_grouped_swiglu_mlp_gated(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.slot_src,
                                       layer.gates, w.W13, w.W2, layer.GU, layer.A, layer.Yperm,
                                       X if c.F_shared else None, w.W13_s, w.W2_s, layer.GU_s, layer.A_s,
                                       layer.Yshared, layer.ws)
    else:
        M.moe_grouped_swiglu_mlp(c, layer.Xperm, layer.offsets, layer.tile_offsets, w.W13, w.W2, layer.GU, layer.A,
                                 layer.Yperm, X if c.F_shared else None, w.W13_s, w.W2_s, layer.GU_s, layer.A_s,
                                 layer.Yshared, layer.ws)
    rec(4)
    me = layer.memory_efficient
    M.moe_unpermute_combine(c, layer.Yperm, layer.row_id_map, None if me else layer.gates, layer.Yshared, layer.Y)
    rec(5)
    # memory-efficient form: dYperm is a copy of dY's rows, the gate gradient comes from FC2's dgrad
    M.moe_unpermute_combine_bwd(c, dY, None if me else layer.Yperm, layer.row_id_map, None if me else layer.gates,
                                layer.offsets, layer.counts, layer.dYperm, None if me else layer.dgates)
    rec(6)
    sh = c.F_shared > 0
    if me:
        M.moe_grouped_swiglu_mlp_bwd_gated(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.counts,
                                           layer.slot_src, layer.row_id_map, layer.gates, w.W13, w.W2, layer.GU,
                                           layer.dYperm, layer.dGU, layer.dXperm, layer.A, layer.dW13, layer.dW2,
                                           layer.dgates, X if sh else None, dY if sh else None, w.W13_s, w.W2_s,
                                           layer.GU_s, layer.A_s, layer.dGU_s, layer.dX_shared, layer.dW13_s,
                                           layer.dW2_s, layer.ws)
    elif layer.gather_rows:
        M.moe_grouped_swiglu_mlp_bwd_gather(c, X, layer.slot_src, layer.offsets, layer.tile_offsets, layer.counts,
                                            w.W13, w.W2, layer.GU, layer.A, layer.dYperm, layer.dGU, layer.dXperm,
                                            layer.dW13, layer.dW2, dY if sh else None, w.W13_s, w.W2_s, layer.GU_s,
                                            layer.A_s, layer.dGU_s, layer.dX_shared, layer.dW13_s, layer.dW2_s,
                                            layer.ws)
    elif layer.fp8:
        M.moe_grouped_swiglu_mlp_bwd_fp8(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.counts, layer.W13q,
                                         layer.W13sc, layer.W2q, layer.W2sc, layer.GU, layer.A, layer.dYperm,
                                         layer.dGU, layer.dXperm, layer.dW13, layer.dW2, X if sh else None,
                                         dY if sh else None, layer.W13q_s, layer.W13sc_s, layer.W2q_s, layer.W2sc_s,
                                         layer.GU_s, layer.A_s, layer.dGU_s, layer.dX_shared, layer.dW13_s,
                                         layer.dW2_s, layer.fp8_ws, layer.ws)
    else:
        M.moe_grouped_swiglu_mlp_bwd(c, layer.Xperm, layer.offsets, layer.tile_offsets, layer.counts, w.W13, w.W2,
                                     layer.GU, layer.A, layer.dYperm, layer.dGU, layer.dXperm, layer.dW13, layer.dW2,
                                     X if sh else None, dY if sh else None, w.W13_s, w.W2_s, layer.GU_s, layer.A_s,
                                     layer.dGU_s, layer.dX_shared, layer.dW13_s, layer.dW2_s, layer.ws)
    rec(7)
    M.moe_router_topk_bwd(c, X, w.W_r, layer.logits, layer.scores, layer.topk_idx, layer.gates, layer.dgates,
                          layer.dW_r, layer.dlogit_bias if w.logit_bias is not None else None, layer.dX_router,
                          layer.ws)
    rec(8)
    M.moe_permute_bwd(c, layer.dXperm, layer.row_id_map, layer.dX_router, layer.dX_shared, layer.dX)
    rec(9)


def launches_per_step(w, gather=False, memory_efficient=False, nsm=152):
    """Kernels of ours launched by run_step (memsets are not counted)."""
    sh = 1 if w.F_shared else 0
    n = 3                                  # router: W_r split, tensor-core logits, routing
    S_ = w.T * w.k
    if S_ <= 16384 and w.E <= 32 and S_ * w.E <= 131072:
        # small layers: maps and row copy in one launch when each CTA's token rows fit its
        # shared memory (one CTA per SM); otherwise the maps, then (without gather) the copy
        tpc = -(-w.T // min(nsm, w.T))
        fused = not gather and tpc * w.H * 2 <= 219 * 1024 and tpc * w.k <= 1024
        n += 1 if (gather or fused) else 2
    else:
        n += 3 if gather else 4            # chunk histogram, scan, scatter, (row copy)
    n += 1 if memory_efficient else 0      # fixed-order sum of the gate-gradient partials
    n += 2 * (1 + sh)                      # FC1 (+SwiGLU), FC2
    n += 2                                 # combine, combine backward
    n += 4 * (1 + sh)                      # FC2 dgrad, FC2 wgrad, FC1 dgrad, FC1 wgrad
    n += 1 + (1 if w.skew else 0)          # dlogits, (bias column sums)
    n += 3 if w.E > 32 else 1              # W_r split, dW_r, dX_router (E > 32) | dW_r, dX_router
    n += 1 if w.E > 32 or w.T > 64 else 0  # fixed-order reduction of the dW_r partials
    n += 1                                 # permute backward
    if w.fp8:
        n += 2 * (1 + sh)                  # weight quantization
        n += 2 * (1 + sh)                  # forward activations (rows)
        n += 6 * (1 + sh)                  # backward: 2 row-, 4 column-quantizations
    return n


def hbm_bytes(w, gather=False, memory_efficient=False):
    """Algorithmic bytes of the HBM-bound stages (index maps excluded; with gathered rows
    the dispatch writes the maps only and is not an HBM stage; in the memory-efficient
    form the combine backward copies dY's rows and reads no Yperm)."""
    T, H, S_ = w.T, w.H, w.T * w.k
    sh = w.F_shared > 0
    d = {
        "permute": T * H * 2 + S_ * H * 2,
        "combine": S_ * H * 2 + T * H * 2 + (T * H * 2 if sh else 0),
        "combine_bwd": T * H * 2 + 2 * S_ * H * 2,
        "permute_bwd": S_ * H * 2 + T * H * 4 + T * H * 2 + (T * H * 2 if sh else 0),
    }
    # the router streams X once (W_r, logits, scores, selection besides)
    d["router"] = T * H * 2 + w.E * H * 4 + T * w.E * 4 * 2 + T * w.k * 8 + w.E * 4
    if w.fp8:  # bf16 weights read, E4M3 weights written (scales < 0.01%)
        wel = 3 * w.E * w.F * w.H + 3 * w.F_shared * w.H
        d["quant_w"] = wel * 2 + wel
    if gather:
        del d["permute"]
    if memory_efficient:
        d["combine_bwd"] = T * H * 2 + S_ * H * 2
    return d


def kernel_digest(files=("grouped_gemm.cu", "common.cuh")):
    """Digest of the sources that define the grouped GEMM kernel."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mixture_experts_layer_topk_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel, workload):
    """DRAM bytes per step of `kernel` from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as fh:
            d = json.load(fh)
        rec = d.get(f"{kernel}:{workload}")
        if not rec or rec.get("source_digest") != kernel_digest():
            return None
        return rec.get("bytes_per_step")
    except Exception:
        return None


def oracle_inputs(w, seed, tokens):
    """Host inputs for the CPU oracle, for samples drawn from `tokens`.  The routed experts'
    weights are generated only for the experts those tokens reach (the generator is
    counter-based, so an expert's slice is the same as in the full tensor; the other
    experts' pages are never touched); in FP8 mode they are block-quantized once here,
    outside the timed samples."""
    import oracle as O
    inp = S.host_inputs(w, seed=seed, weights=False)
    T, H, E, F, Fs = w.T, w.H, w.E, w.F, w.F_shared
    tokens = np.asarray(tokens, np.int64)
    c = O.cfg(w.replace(T=len(tokens)))
    logits, scores = O.router(c, np.ascontiguousarray(inp["X"][tokens]), inp["W_r"], inp.get("logit_bias"))
    used = sorted(set(int(e) for e in O.select(c, logits, scores, inp.get("sel_bias")).ravel()))
    W13 = np.empty((E, 2 * F, H), np.uint16)
    W2 = np.empty((E, H, F), np.uint16)
    for e in used:
        W13[e] = S.normal_bf16(2 * F * H, seed, S.TID_W13, w.w_std, start=e * 2 * F * H).reshape(2 * F, H)
        W2[e] = S.normal_bf16(H * F, seed, S.TID_W2, w.w_std, start=e * H * F).reshape(H, F)
        if w.fp8:
            W13[e] = O.qdq_weights(W13[e])
            W2[e] = O.qdq_weights(W2[e])
    inp["W13"], inp["W2"] = W13, W2
    if Fs:
        inp["W13_s"] = S.normal_bf16(2 * Fs * H, seed, S.TID_W13S, w.w_std).reshape(2 * Fs, H)
        inp["W2_s"] = S.normal_bf16(H * Fs, seed, S.TID_W2S, w.w_std).reshape(H, Fs)
        if w.fp8:
            inp["W13_s"] = O.qdq_weights(inp["W13_s"])
            inp["W2_s"] = O.qdq_weights(inp["W2_s"])
    return inp


def oracle_sample(w, inp, off, n):
    """The CPU oracle's forward+backward of the layer for the tokens off .. off+n-1: routing
    (logits, selection, gates), the tokens' outputs, input gradients and gate gradients, the
    weight gradients of every expert the tokens are routed to and of the shared expert, and
    the router's weight gradient.  An expert no sampled token reaches has a zero weight
    gradient; it is not computed.  The independent oracle calls of a sample run side by side
    on the host's cores."""
    import oracle as O
    sub = w.replace(T=n)
    si = dict(inp)
    si["X"] = np.ascontiguousarray(inp["X"][off:off + n])
    si["dY"] = np.ascontiguousarray(inp["dY"][off:off + n])
    c = O.cfg(sub)
    logits, scores = O.router(c, si["X"], si["W_r"], si.get("logit_bias"))
    idx = O.select(c, logits, scores, si.get("sel_bias"))
    g = O.gates(c, logits, idx)
    O.dispatch(c, idx)
    experts = sorted(set(int(x) for x in idx.ravel())) + ([-1] if w.F_shared else [])
    # the per-expert weight gradients are independent oracle calls: run them side by side
    # (ctypes releases the GIL) while the tokens' forward+backward runs
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(max_workers=len(experts) + 1) as ex:
        fut_tk = ex.submit(O.tokens, c, si, idx, logits, g)
        futs = [ex.submit(O.expert_wgrad, c, si, idx, g, e) for e in experts]
        tk = fut_tk.result()
        for f in futs:
            f.result()
    O.router_wgrad(c, si["X"], tk["dlogits"])


SAMPLE_TEXT = ("forward+backward of the whole layer for the sampled tokens through the CPU oracle (routing, "
               "outputs, input and gate gradients, the weight gradients of the experts they reach, shared "
               "expert and router weight gradients), double accumulation")


def cpu_baseline(w, seed, budget_s=15.0):
    """The CPU oracle on the first n tokens of the same workload, n sized for about budget_s."""
    inp = oracle_inputs(w, seed, np.arange(min(w.T, 256)))

    def one(n):
        t0 = time.perf_counter()
        oracle_sample(w, inp, 0, n)
        return time.perf_counter() - t0

    # the cost per token falls as the sample grows (fixed costs of the sampled experts'
    # weight gradients), so the size is re-estimated from each run until one takes most of
    # the budget
    n, t = 2, one(2)
    for _ in range(4):
        n_next = max(1, min(w.T, 256, int(n * budget_s / max(t, 1e-3))))
        if n_next <= n or t >= 0.6 * budget_s:
            break
        n, t = n_next, one(n_next)
    return {"value": n / t, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{SAMPLE_TEXT}: the first {n} of {w.T} tokens, {t:.1f} s wall",
            "extrapolated_full_layer_s": round(w.T * t / n, 1)}


def bench_ours(args, w):
    import torch
    import mixture_experts_layer_topk_gb300 as M
    ws_, rank, local = dist_env()
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    weights, X, dY = device_inputs(w, args.seed, dev)
    cfg = M.config_from(w)
    layer = M.MoELayer(cfg, weights, device=dev, fp8=w.fp8, gather_rows=args.gather,
                       memory_efficient=args.memory_efficient)
    stream = torch.cuda.current_stream()

    def barrier():
        if ws_ > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # eager warm-up (sets the kernels' attributes), then the step captured as one CUDA graph
    for _ in range(2):
        run_step(layer, X, dY)
    barrier()
    if layer.device_error() != 0:
        raise RuntimeError("device error during warm-up")
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device=dev)
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        run_step(layer, X, dY)  # one eager step on the capture stream before capturing
        with torch.cuda.graph(graph, stream=cs):
            run_step(layer, X, dY)
    stream.wait_stream(cs)
    for _ in range(args.warmup):
        graph.replay()
    barrier()
    if layer.device_error() != 0:
        raise RuntimeError("device error during the warm-up replays")

    # timed region: K replays, an event between consecutive replays
    sampler = ClockSampler(gpu_id_for_smi(torch, local))
    time.sleep(0.3)
    barrier()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        graph.replay()
        evs[i + 1].record(stream)
    barrier()
    replay_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    total_ms = evs[0].elapsed_time(evs[-1])
    if layer.device_error() != 0:
        raise RuntimeError("device error during the timed replays")

    # stage pass: the step captured with an event between the stages (event nodes of the
    # graph) and replayed K times, each replay's stage times read after it; K eager steps
    # with the same events where events cannot be recorded into a graph
    ns = len(STAGES)
    stage_sum = [0.0] * ns
    pass_ms = 0.0
    stage_timing = "graph"
    try:
        sev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(ns + 1)]
        sgraph = torch.cuda.CUDAGraph()
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            with torch.cuda.graph(sgraph, stream=cs):
                run_step(layer, X, dY, sev)
        stream.wait_stream(cs)
        barrier()
        for i in range(args.steps):
            sgraph.replay()
            torch.cuda.synchronize()
            for j in range(ns):
                stage_sum[j] += sev[j].elapsed_time(sev[j + 1])
            pass_ms += sev[0].elapsed_time(sev[-1])
        del sgraph
    except (TypeError, RuntimeError) as exc:
        stage_timing = "eager (" + type(exc).__name__ + " capturing the stage events)"
        stage_sum = [0.0] * ns
        pass_ms = 0.0
        torch.cuda.synchronize()
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(args.steps)]
        barrier()
        for i in range(args.steps):
            run_step(layer, X, dY, sevs[i])
        barrier()
        for i in range(args.steps):
            for j in range(ns):
                stage_sum[j] += sevs[i][j].elapsed_time(sevs[i][j + 1])
            pass_ms += sevs[i][0].elapsed_time(sevs[i][-1])
    barrier()
    clocks = sampler.stop()
    stage_ms = {s: stage_sum[j] / args.steps for j, s in enumerate(STAGES)}
    stage_pass_ms = pass_ms / args.steps
    if layer.device_error() != 0:
        raise RuntimeError("device error during the stage pass")

    # end to end through the C ABI with host buffers: every step copies its inputs (X, dY)
    # up from pinned host memory and its results (Y, dX) back.  A copy stream moves the
    # next step's inputs and the previous step's results while the current step
    # computes; inputs and outputs alternate between two device buffers each, and the step
    # on each pair of buffers is a CUDA graph of the C-ABI calls, as in the timed replays.
    Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    dYh = torch.empty(dY.shape, dtype=dY.dtype, pin_memory=True)
    Xh.copy_(X)
    dYh.copy_(dY)
    Yh = [torch.empty(X.shape, dtype=X.dtype, pin_memory=True) for _ in range(2)]
    dXh = [torch.empty(X.shape, dtype=X.dtype, pin_memory=True) for _ in range(2)]
    Xd = [torch.empty_like(X) for _ in range(2)]
    dYd = [torch.empty_like(dY) for _ in range(2)]
    Yd = [layer.Y, torch.empty_like(layer.Y)]
    dXd = [layer.dX, torch.empty_like(layer.dX)]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step on buffer b has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of buffer b are on the host
    # the step on each buffer set, captured as a CUDA graph like the headline's step
    egraphs = []
    for b in range(2):
        layer.Y, layer.dX = Yd[b], dXd[b]
        eg = torch.cuda.CUDAGraph()
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            with torch.cuda.graph(eg, stream=cs):
                run_step(layer, Xd[b], dYd[b])
        stream.wait_stream(cs)
        egraphs.append(eg)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        Xd[0].copy_(Xh, non_blocking=True)
        dYd[0].copy_(dYh, non_blocking=True)
        ev_in[0].record(cs)
    for i in range(args.steps):
        b = i % 2
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])
        egraphs[b].replay()
        ev_done[b].record(stream)
        with torch.cuda.stream(cs):
            if i >= 1:  # the previous step's results, then the next step's inputs into its buffers
                cs.wait_event(ev_done[1 - b])
                Yh[1 - b].copy_(Yd[1 - b], non_blocking=True)
                dXh[1 - b].copy_(dXd[1 - b], non_blocking=True)
                ev_out[1 - b].record(cs)
            if i + 1 < args.steps:
                Xd[1 - b].copy_(Xh, non_blocking=True)
                dYd[1 - b].copy_(dYh, non_blocking=True)
                ev_in[1 - b].record(cs)
    last = (args.steps - 1) % 2
    with torch.cuda.stream(cs):
        cs.wait_event(ev_done[last])
        Yh[last].copy_(Yd[last], non_blocking=True)
        dXh[last].copy_(dXd[last], non_blocking=True)
    stream.wait_stream(cs)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    layer.Y, layer.dX = Yd[0], dXd[0]
    del egraphs

    med_ms = statistics.median(replay_ms)
    med_ms, total_ms, e2e_ms = max_over_ranks([med_ms, total_ms, e2e_ms], device=dev)
    if rank != 0:
        return None

    tokens = w.T * ws_
    value = tokens / (med_ms / 1e3)
    pk, pk_kind = peaks()
    gemm_flop = M.gemm_flops(cfg)
    gemm_ms = stage_ms["gemm_fwd"] + stage_ms["gemm_bwd"]
    gemm_tflops = gemm_flop / (gemm_ms / 1e3) / 1e12
    # the GEMMs are timed inside a step of several milliseconds: the sustained peak
    peak_t = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    peak_kind = f"{pk_kind} bf16 sustained"
    if w.fp8:  # dense FP8 runs at twice the BF16 tensor rate (nominal 4.5 vs 2.25 PFLOP/s)
        peak_t *= 2.0
        peak_kind = f"{pk_kind} bf16 sustained x 2 (FP8:BF16 nominal ratio)"
    variant = "-gather" if args.gather else ("-memeff" if args.memory_efficient else "")
    traffic = traffic_record("k_grouped_gemm", w.name + variant)
    hb = hbm_bytes(w, gather=args.gather, memory_efficient=args.memory_efficient)
    hbm = {}
    for s, b in hb.items():
        gbs = b / (stage_ms[s] / 1e3) / 1e9
        hbm[s] = {"achieved": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 3),
                  "ms": round(stage_ms[s], 4)}
    wbytes = (w.E * 3 * w.F * w.H + 3 * w.F_shared * w.H) * 2
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(med_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3" if w.fp8 else "bf16",
        "data": "synthetic (seeded normal inputs)",
        "timing": {"value_from": "median of K CUDA-graph replays of the whole step",
                   "ms_per_step_mean": round(total_ms / args.steps, 4),
                   "ms_per_step_min": round(min(replay_ms), 4), "ms_per_step_max": round(max(replay_ms), 4),
                   "stage_timing": stage_timing, "stage_pass_ms_per_step": round(stage_pass_ms, 4)},
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "F": w.F, "F_shared": w.F_shared,
                   "router": ("softmax" if w.score_fn == 0 else "sigmoid") + (", renorm" if w.renorm else "")
                             + (f", {w.n_group} groups / top-{w.topk_group}" if w.n_group > 1 else "")
                             + (", selection bias" if w.sel_bias else "")
                             + (f", x{w.gate_scale:g}" if w.gate_scale != 1.0 else ""),
                   "dispatch": "gathered rows (no permuted copy)" if args.gather else "permuted copy",
                   "combine": ("gates applied before FC2, unit-weight sum (memory-efficient form)"
                               if args.memory_efficient else "gate-weighted sum"),
                   "l2": "inputs larger than L2 (expert weights %.2f GB re-read every step)" % (wbytes / 1e9),
                   "parallelism": "replicas" if ws_ > 1 else "single GPU"},
        "gemm_tflops": round(gemm_tflops, 1), "gemm_frac_of_peak": round(gemm_tflops / peak_t, 3),
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "roofline": {"kernel": "k_grouped_gemm (FC1+SwiGLU, FC2, FC2 dgrad+dSwiGLU, FC2 wgrad, FC1 dgrad, FC1 wgrad)",
                     "bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": peak_t, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / peak_t, 3), "peak_source": peak_kind,
                     "frac_of_burst": round(gemm_tflops / (pk["bf16_tflops"] * (2.0 if w.fp8 else 1.0)), 3),
                     "traffic": traffic},
        "hbm_stages": hbm,
        "clocks": clocks,
        "gpu_launches": launches_per_step(w, gather=args.gather, memory_efficient=args.memory_efficient,
                                          nsm=torch.cuda.get_device_properties(dev).multi_processor_count) * args.steps,
        "e2e": {"value": round(tokens / (e2e_ms / args.steps / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * X.numel() * 2, "d2h_bytes_per_step": 2 * X.numel() * 2},
    }
    if ws_ == 1 and not args.no_cpu_baseline:
        del graph, layer, weights, X, dY
        torch.cuda.empty_cache()
        line["cpu_baseline"] = cpu_baseline(w, args.seed)
    return line


def bench_reference(args, w):
    """The CPU oracle as the reference arm: each step is the oracle's whole-layer
    forward+backward on a bounded sample of the workload's tokens."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return None
    # each step takes the next n tokens (wrapping); the sample is sized from a 2-token probe
    # on a small input set, then the inputs of every token the steps will touch are made
    inp = oracle_inputs(w, args.seed, np.arange(2))

    def step(n, off):
        oracle_sample(w, inp, off, n)

    t0 = time.perf_counter()
    step(2, 0)
    t_probe = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = max(1, min(w.T, int(2 * budget / max(t_probe, 1e-3))))
    offs = [(i * n) % max(1, w.T - n) for i in range(args.warmup + args.steps)]
    inp = oracle_inputs(w, args.seed, np.unique(np.concatenate([np.arange(o, o + n) for o in offs])))
    for i in range(args.warmup):
        step(n, (i * n) % max(1, w.T - n))
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(n, (i * n) % max(1, w.T - n))
    dt = time.perf_counter() - t0
    v = n * args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normal inputs)",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "F": w.F, "F_shared": w.F_shared},
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{SAMPLE_TEXT}: {n} of {w.T} tokens per step"},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3", choices=sorted(S.WORKLOADS))
    ap.add_argument("--gather", action="store_true",
                    help="gathered-rows dispatch: FC1 reads X through the maps, no permuted copy (bf16 only)")
    ap.add_argument("--memory-efficient", action="store_true",
                    help="gates applied before FC2 and activations recomputed in the backward (bf16 only)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = S.WORKLOADS[args.workload]
    if (args.gather or args.memory_efficient) and w.fp8:
        ap.error("--gather and --memory-efficient are built for the bf16 expert GEMMs")
    if args.gather and args.memory_efficient:
        ap.error("--gather and --memory-efficient are separate forms")
    line = bench_reference(args, w) if args.impl == "reference" else bench_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
