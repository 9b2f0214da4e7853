"""Host-side pieces of the benchmark, CPU only: the roofline denominator, the
traffic record keyed by the kernel sources, the clock-sample summary, and the
unique-byte count of a batch with shared prefix blocks."""
import json
import time

import numpy as np

import bench
from paged_kv_cache_268_gb300 import workloads as W


def test_measured_peak_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6781.1}))
    assert bench.measured_peak() == (6781.1, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.measured_peak()[1] == "fallback"


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "decode_traffic.json").write_text(json.dumps({
        "llama7b_mha": {"kernel_source_sha": "abc", "dram_bytes_per_full_launch": 123.0}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.recorded_traffic("llama7b_mha") == 123.0
    assert bench.recorded_traffic("cont_batch") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "def")   # sources changed
    assert bench.recorded_traffic("llama7b_mha") is None


def _sampler(rows):
    s = object.__new__(bench.ClockSampler)     # no nvidia-smi process
    s.proc = object()
    s.samples = rows
    return s


def _row(mhz, reasons=("Not Active",) * 4, power="700.0"):
    return ["0", str(mhz), "2070", power, "0x0", *reasons]


def test_clock_summary_window_and_reasons():
    t = time.time()
    rows = [(t - 1.0, _row(1200)),                                   # before the timed region
            (t + 0.1, _row(2070)), (t + 0.2, _row(2055)), (t + 0.3, _row(2070)),
            (t + 0.4, _row(2070, ("Not Active", "Not Active", "Not Active", "Active"), "1390.5")),
            (t + 9.0, _row(900))]                                    # after it
    s = _sampler(rows).summary(t, t + 1.0)
    assert s["window"] == "timed" and s["samples"] == 4
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1390.5
    bad = [(t + 0.1 * i, _row(1800, ("Active", "Not Active", "Active", "Not Active")))
           for i in range(1, 4)]
    assert _sampler(bad).summary(t, t + 1.0)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_short_region_uses_warmup_samples():
    t = time.time()
    rows = [(t - 0.5, _row(2070)), (t - 0.2, _row(2070)), (t + 0.05, _row(2070))]
    s = _sampler(rows).summary(t, t + 0.1)
    assert s["window"] == "warmup+timed" and s["samples"] == 3
    assert _sampler([]).summary(t, t + 1.0)["reasons"] == ["no samples"]


def test_unique_bytes_count_shared_prefix_blocks_once():
    spec = W.scaled(W.WORKLOADS["cont_batch"], 16, 700)
    w = W.make(spec, seed=0)
    row = spec.num_kv_heads * spec.head_dim * 2 * 2
    # brute force: the distinct (physical block, row) pairs the batch reads
    rows = {}
    for i in range(spec.num_seqs):
        L = int(w.context_lens[i])
        for t in range(L):
            p = int(w.block_tables[i, t // spec.block_size])
            rows.setdefault(p, set()).add(t % spec.block_size)
    assert w.unique_kv_bytes() == sum(len(r) for r in rows.values()) * row
    assert w.unique_kv_bytes() < w.kv_bytes()               # the groups share blocks
    plain = W.make(W.scaled(W.WORKLOADS["llama7b_mha"], 4, 300), seed=0)
    assert plain.unique_kv_bytes() == plain.kv_bytes()     # nothing shared
    assert np.all(plain.context_lens >= 1)


def test_host_cpu_description():
    """The CPU baseline states the host it ran on: logical CPUs and a model."""
    h = bench.host_cpu()
    assert h["nproc"] is not None and h["nproc"] >= 1
    assert set(h) == {"nproc", "cpu_model", "machine"}
    assert h["machine"]


def test_committed_traffic_record_is_consistent():
    """profiles/decode_traffic.json, when it was taken on the kernel sources
    as they are (else the benchmark reports no traffic), gives DRAM bytes
    just above each workload's algorithmic bytes (unique bytes for the
    continuous-batching batch, whose shared blocks L2 serves)."""
    import pytest
    for name in ("llama7b_mha", "llama3_8b_gqa", "long_ctx_gqa", "cont_batch"):
        t = bench.recorded_traffic(name)
        if t is None:
            pytest.skip("the traffic record predates the current kernel sources")
        # the seed-0 batch's lengths and tables, without drawing its pools
        spec = W.WORKLOADS[name]
        rng = np.random.default_rng([0, W.ORDER.index(name)])
        lens = W.context_lengths(spec, rng)
        tables, used = W.block_tables(spec, lens, rng)
        w = W.Workload(spec, 0, lens, tables, None, used, None, None, None, None, None)
        ref = w.unique_kv_bytes() if name == "cont_batch" else w.kv_bytes()
        assert 1.0 <= t / ref < 1.05, (name, t / ref)
