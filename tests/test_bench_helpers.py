"""The benchmark's host-side bookkeeping (no GPU): band parity counts, the
walk statistics, and the DRAM-traffic record that is refused once the
captured kernel's source has changed."""
import hashlib
import json

import numpy as np

import bench


def test_band_parity_counts():
    o = {"row_status": np.array([0, 0, 0, 3]), "accepted_len": np.array([1, 2, 0, -1]),
         "out_tokens": np.array([[5, 6, -1], [1, 2, 3], [9, -1, -1], [-1, -1, -1]]),
         "row_margin": np.array([1e-7, 0.3, 0.2, np.inf])}
    g_len = np.array([1, 2, 1, -1])
    g_tok = np.array([[5, 7, -1], [1, 2, 3], [4, 4, -1], [-1, -1, -1]])
    p = bench.band_parity(g_len, g_tok, o)
    # row 0 differs inside the band, row 2 outside it, rows 1 and 3 agree
    assert p == {"rows": 4, "band_mismatches": 1, "outside_band": 1}


def test_walk_stats():
    s = bench.walk_stats(np.array([0, 0, 1, 3, -1]), 3)
    assert s["accepted_len_histogram"] == [2, 1, 0, 1]
    assert s["mean_emitted"] == (1 + 1 + 2 + 4) / 4
    assert s["residual_draws"] == 3 and s["bonus_draws"] == 1


def test_traffic_record_refuses_a_changed_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// v1\n")
    rec = {"k": {"source": str(src), "sha256": hashlib.sha256(b"// v1\n").hexdigest(),
                 "dram_bytes_read": 100, "dram_bytes_write": 5, "capture": "profiles/k.md"}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("k") == (105, "profiles/k.md")
    src.write_text("// v2\n")
    val, why = bench.measured_traffic("k")
    assert val is None and "changed" in why
    assert bench.measured_traffic("other")[0] is None


def test_committed_traffic_record_is_well_formed():
    with open(bench.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    for name, r in rec.items():
        assert {"source", "sha256", "dram_bytes_read", "dram_bytes_write", "capture"} <= set(r), name
        assert r["capture"].startswith("profiles/")


def test_every_traffic_record_the_bench_reads_is_on_file():
    """Each kernel name bench.py looks up has a record whose capture summary
    exists, so a renamed kernel or record cannot turn the figure into a
    silent null."""
    import os
    import re
    with open(bench.__file__) as fh:
        names = set(re.findall(r'measured_traffic\("([^"]+)"\)', fh.read()))
    with open(bench.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    assert names, "bench.py reads no traffic record"
    for name in names:
        assert name in rec, name
        assert os.path.exists(os.path.join(bench.ROOT, rec[name]["capture"])), name

