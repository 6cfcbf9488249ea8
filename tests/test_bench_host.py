"""Host-side pieces of bench.py, without a GPU: the kernel-source hash that
ties a committed ncu summary to the code it was captured on."""
import bench


def test_source_hash_ignores_comments_and_whitespace(tmp_path):
    a = tmp_path / "a.cuh"
    a.write_text("int f(int x) {\n  return x + 1;  // add one\n}\n/* note */\n")
    b = tmp_path / "b.cuh"
    b.write_text("int f(int x){ return x+1; }\n// another comment\n")
    c = tmp_path / "c.cuh"
    c.write_text("int f(int x){ return x+2; }\n")
    ha = bench.kernel_source_hash([str(a)])
    assert ha == bench.kernel_source_hash([str(b)])
    assert ha != bench.kernel_source_hash([str(c)])



def test_traffic_summary_round_trip(tmp_path, monkeypatch):
    """--traffic-from keeps the last captured launch's DRAM bytes, and the
    roofline reads them back only while the kernel sources are unchanged."""
    import json
    csv = tmp_path / "t.csv"
    head = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",' \
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",' \
           '"Metric Value"\n'
    rows = []
    for i, (rd, wr) in enumerate(((100.0, 40.0), (120.0, 60.0))):
        for m, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr),
                     ("lts__t_sectors_op_read.sum", 5.0), ("lts__t_sectors_op_write.sum", 3.0),
                     ("gpu__time_duration.sum", 9.0)):
            rows.append(f'"{i}","1","python","h","k(Params)","1","7","(288,1,1)","(456,1,1)",'
                        f'"0","10.3","Command line profiler metrics","{m}","byte","{v}"\n')
    csv.write_text("==PROF== noise\n" + head + "".join(rows))
    out = tmp_path / "traffic.json"
    monkeypatch.setitem(bench.TRAFFIC_JSON, "prefill", str(out))
    rec = bench.write_traffic_json(str(csv), "prefill")
    assert rec["dram_bytes_read_per_launch"] == 120.0 and rec["dram_bytes_write_per_launch"] == 60.0
    assert rec["lts_write_sector_bytes"] == 96.0 and rec["launches_captured"] == 2
    assert bench.profile_traffic("prefill") == 180.0
    stale = json.loads(out.read_text())
    stale["kernel_source_sha256"] = "0" * 64
    out.write_text(json.dumps(stale))
    assert bench.profile_traffic("prefill") is None


def test_probe_workloads():
    """Every q+k probe that ncu captures use names its own workload (the
    Hadamard probes the plain shapes with the rotation on)."""
    import bench
    for which, T, H, had in [("prefill", 8192, 64, False), ("prefill_h32", 8192, 32, False),
                             ("prefill_h16", 8192, 16, False), ("decode", 64, 64, False),
                             ("prefill_hadamard", 8192, 64, True), ("decode_hadamard", 64, 64, True)]:
        inp, h = bench.probe_workload(which)
        assert (inp.T, inp.H, h) == (T, H, had), which
    import pytest
    with pytest.raises(ValueError):
        bench.probe_workload("prefill_hx")
