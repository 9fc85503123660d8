"""Host-side checks of bench.py's measurement bookkeeping (no GPU): the ncu CSV parser behind
roofline.traffic, the source-hash guard on the traffic record, and the step roofline fraction."""
import json

import pytest

import bench

CSV = '''==PROF== Connected to process 1 (/usr/bin/python3)
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python3","h","void gbconv::k_a(int)","1","7","(256, 1, 1)","(2, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","205.55"
"0","1","python3","h","void gbconv::k_a(int)","1","7","(256, 1, 1)","(2, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Kbyte","1,024"
"0","1","python3","h","void gbconv::k_a(int)","1","7","(256, 1, 1)","(2, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","42000"
"1","1","python3","h","void gbconv::k_b(int)","1","7","(256, 1, 1)","(2, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","7"
"2","1","python3","h","void gbconv::k_a(int)","1","7","(256, 1, 1)","(2, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","0.2"
"2","1","python3","h","void gbconv::k_a(int)","1","7","(256, 1, 1)","(2, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","0"
'''


def test_ncu_dram_bytes_sums_read_and_write_per_launch(tmp_path):
    p = tmp_path / "t.csv"
    p.write_text(CSV)
    mean, launches = bench.ncu_dram_bytes(str(p), "k_a")
    assert launches == 2
    assert mean == pytest.approx(((205.55e6 + 1024e3) + 0.2e9) / 2)
    assert bench.ncu_dram_bytes(str(p), "k_b") == (7.0, 1)
    with pytest.raises(ValueError):
        bench.ncu_dram_bytes(str(p), "k_missing")


def test_traffic_record_needs_the_captured_source(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(path))
    assert bench.traffic_record("depthwise.cu", "w")[0] is None
    digest = bench.source_digest("depthwise.cu")
    path.write_text(json.dumps({"w": {"kernel_file": "depthwise.cu", "source_sha16": digest,
                                      "dram_bytes_per_launch": 123}}))
    assert bench.traffic_record("depthwise.cu", "w")[0] == 123.0
    path.write_text(json.dumps({"w": {"kernel_file": "depthwise.cu", "source_sha16": "0" * 16,
                                      "dram_bytes_per_launch": 123}}))
    value, note = bench.traffic_record("depthwise.cu", "w")
    assert value is None and "changed" in note


def test_committed_traffic_records_are_machine_written():
    import os
    if not os.path.exists(bench.TRAFFIC_JSON):
        pytest.skip("no traffic record committed")
    for name, rec in json.load(open(bench.TRAFFIC_JSON)).items():
        assert set(rec) >= {"kernel_file", "source_sha16", "dram_bytes_per_launch", "command", "kernel_regex"}
        assert rec["dram_bytes_per_launch"] > 0
