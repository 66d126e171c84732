"""Host logic of the benchmark that needs no GPU: the DRAM-traffic records (a record
counts only while the kernel sources it was captured from are unchanged), the
roofline of the unified-span row (taken on DRAM bytes, the logical rate beside it),
the whole-job aggregate, and the oracle's decode CPU baseline."""
import hashlib
import os

import pytest

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "paged_kv_cache_pages_gb300", "csrc")


def _digest(files):
    h = hashlib.sha256()
    for f in files + bench._TRAFFIC_HEADERS:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def test_traffic_record_counts_only_for_the_sources_it_was_taken_from(monkeypatch):
    files = ["k_decode.cu"]
    good = {"bytes": 86.0e6, "files": files, "digest": _digest(files)}
    stale = dict(good, digest="0" * 16)
    monkeypatch.setitem(bench.TRAFFIC, "k_decode", good)
    assert bench.traffic_of("k_decode") == 86.0e6
    monkeypatch.setitem(bench.TRAFFIC, "k_decode", stale)
    assert bench.traffic_of("k_decode") is None


def test_every_traffic_record_names_existing_sources():
    for rec in bench.TRAFFIC.values():
        assert rec["bytes"] > 0 and len(rec["digest"]) == 16
        for f in rec["files"] + bench._TRAFFIC_HEADERS:
            assert os.path.exists(os.path.join(CSRC, f)), f


def test_span_roofline_uses_dram_bytes(monkeypatch):
    monkeypatch.setattr(bench, "traffic_of", lambda k: 116.0e6 if k == "k_decode_span" else None)
    r = bench.span_roofline(10000.0, 0.1, 6784.2)  # 0.1 ms per layer
    assert r["achieved"] == pytest.approx(1160.0)   # 116 MB / 0.1 ms
    assert r["frac"] == pytest.approx(1160.0 / 6784.2, rel=1e-3)
    assert r["logical_gbs"] == 10000.0 and r["peak"] == 6784.2
    monkeypatch.setattr(bench, "traffic_of", lambda k: None)
    r = bench.span_roofline(10000.0, 0.1, 6784.2)
    assert r["achieved"] is None and r["frac"] is None and r["logical_gbs"] == 10000.0


def test_aggregate_is_whole_job_over_slowest_rank():
    assert bench.aggregate(10.0, 2.0, 1) == 5.0
    assert bench.aggregate(10.0, 2.0, 4) == 20.0   # 4 ranks x 10 units in 2 s


def test_decode_cpu_baseline_counts_the_layer_bytes():
    import workloads
    case = workloads.tiny(0)
    r = bench.cpu_baseline_decode(case, reps_budget_s=0.05)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0
    assert r["cores"] >= 1 and "runs in" in r["sample"]


def test_every_traffic_key_the_bench_asks_for_has_a_record():
    """Each `traffic_of(...)` key that bench.py reads names a record (a missing key would
    silently report null traffic)."""
    import re
    with open(bench.__file__) as fh:
        src = fh.read()
    keys = set(re.findall(r'traffic_of\("([a-z0-9_]+)"\)', src))
    keys |= set(re.findall(r'traffic_key="([a-z0-9_]+)"', src))
    assert keys, "no traffic keys found"
    assert keys <= set(bench.TRAFFIC), sorted(keys - set(bench.TRAFFIC))
