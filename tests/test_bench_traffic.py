"""bench.py reports captured DRAM traffic only for the kernel sources it was captured on."""
import bench


def test_traffic_reported_while_sources_match():
    b, k = bench.captured_traffic("scan_bwd")
    assert b is None or (b > 0 and k)


def test_traffic_null_after_a_source_change(monkeypatch):
    cap = dict(bench.TRAFFIC_CAPTURES["scan_bwd"])
    cap["sources"] = {rel: "0" * 64 for rel in cap["sources"]}
    monkeypatch.setitem(bench.TRAFFIC_CAPTURES, "scan_bwd", cap)
    assert bench.captured_traffic("scan_bwd") == (None, None)


def test_traffic_null_for_uncaptured_stage():
    assert bench.captured_traffic("conv_fwd") == (None, None)
