"""Host-side logic of the benchmark (no GPU): the recorded DRAM traffic is reported only
while the grouped GEMM's sources match the ones it was captured on, and the launch counts
and algorithmic HBM bytes cover every stage the benchmark times."""
import json

import pytest

import bench
import moe_synth as S


def _write_traffic(tmp_path, digest, nbytes):
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"k_grouped_gemm:mixtral": {"source_digest": digest, "bytes_per_step": nbytes, "launches": 6}}
    (prof / "traffic.json").write_text(json.dumps(rec))


def test_traffic_record_requires_the_current_kernel_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_digest", lambda files=None: "abc")
    _write_traffic(tmp_path, "abc", 123)
    assert bench.traffic_record("k_grouped_gemm", "mixtral") == 123
    assert bench.traffic_record("k_grouped_gemm", "qwen3") is None  # no capture for that workload
    monkeypatch.setattr(bench, "kernel_digest", lambda files=None: "changed")
    assert bench.traffic_record("k_grouped_gemm", "mixtral") is None  # the kernel changed since


def test_traffic_record_absent_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k_grouped_gemm", "mixtral") is None


def test_kernel_digest_tracks_the_gemm_sources():
    d = bench.kernel_digest()
    assert isinstance(d, str) and len(d) == 16
    assert bench.kernel_digest(("grouped_gemm.cu",)) != d  # common.cuh is part of it


@pytest.mark.parametrize("name", sorted(S.WORKLOADS))
def test_stage_accounting_covers_every_workload(name):
    w = S.WORKLOADS[name]
    n = bench.launches_per_step(w)
    assert isinstance(n, int) and n > 10
    hb = bench.hbm_bytes(w)
    for stage in ("permute", "combine", "combine_bwd", "permute_bwd", "router"):
        assert hb[stage] > 0 and stage in bench.STAGES
    assert ("quant_w" in hb) == w.fp8
    # the permute moves X once and writes it k times; the combine backward reads dY once
    assert hb["permute"] == w.T * w.H * 2 * (1 + w.k)
    assert hb["combine_bwd"] == w.T * w.H * 2 * (1 + 2 * w.k)


def test_gathered_rows_accounting():
    """With gathered rows the dispatch copies nothing: one launch fewer, no permute HBM stage."""
    w = S.WORKLOADS["dsv3"]
    assert bench.launches_per_step(w, gather=True) == bench.launches_per_step(w) - 1
    assert "permute" not in bench.hbm_bytes(w, gather=True)


def test_small_dispatch_accounting():
    """A small dropless layer whose token rows fit one CTA per SM: maps and row copy in one
    launch, so gathered rows save no launch there; with more rows per CTA than shared memory
    holds, the maps and the copy are two launches."""
    w = S.WORKLOADS["mixtral"]
    assert bench.launches_per_step(w, gather=True) == bench.launches_per_step(w)
    big = S.Workload("rows-beyond-shared-memory", T=8000, H=4096, E=8, k=2, F=128)
    assert bench.launches_per_step(big, gather=True) == bench.launches_per_step(big) - 1



@pytest.mark.parametrize("fixed_s,per_token_s", [(0.5, 0.01), (0.0, 0.2), (3.0, 0.001)])
def test_cpu_baseline_sample_fills_its_budget(monkeypatch, fixed_s, per_token_s):
    """The oracle sample is re-sized from each timed run until one takes most of the budget,
    never past 256 tokens or the workload's T, whatever the fixed and per-token costs."""
    clock = [0.0]
    sizes = []

    def fake_sample(w, inp, off, n):
        sizes.append(n)
        clock[0] += fixed_s + per_token_s * n

    monkeypatch.setattr(bench, "oracle_inputs", lambda w, seed, rows: None)
    monkeypatch.setattr(bench, "oracle_sample", fake_sample)
    monkeypatch.setattr(bench.time, "perf_counter", lambda: clock[0])
    w = S.WORKLOADS["dsv3"]
    budget = 15.0
    rec = bench.cpu_baseline(w, 0, budget_s=budget)
    n = sizes[-1]
    assert 1 <= n <= min(w.T, 256)
    t = fixed_s + per_token_s * n
    assert rec["value"] == pytest.approx(n / t)
    assert f"the first {n} of {w.T} tokens" in rec["sample"]
    # the last run takes most of the budget unless the 256-token cap stops it first
    assert t >= 0.6 * budget or n == 256
    assert len(sizes) <= 5
