"""Host checks of the benchmark's committed ncu records: the traffic record
parses, is used only while its source hash matches the expert call's code
(the first two checks skip when it does not), and its per-slot DRAM table has one entry per pass size with DRAM reads
between the call's unique and requested expert bytes."""
import pytest

import bench
from moe_expert_layer_warp_gb300 import configs


def test_traffic_record_matches_current_sources():
    rec = bench.load_traffic_record(bench.TRAFFIC_FILE)
    if rec is None:
        pytest.skip("the traffic record was taken on other kernel sources (bench reports null)")
    assert int(rec["dram_bytes_per_launch"]) > 0


def test_perslot_dram_table_is_bounded_by_requested_bytes():
    w = configs.V2_LITE
    sh = w.shape
    e_b = 3 * sh.d * sh.inter * 2
    ps = bench.load_perslot_dram(bench.TRAFFIC_FILE, len(w.pass_sizes))
    if ps is None:
        pytest.skip("the traffic record was taken on other kernel sources (bench reports null)")
    assert len(ps) == len(w.pass_sizes)
    for n, b in zip(w.pass_sizes, ps):
        requested = (n * sh.top_k + sh.n_shared) * e_b
        at_least = (sh.top_k + sh.n_shared) * e_b  # a pass's slots name at least k experts
        assert 0.98 * at_least <= b <= 1.02 * requested, (n, b, requested)
    assert bench.load_perslot_dram(bench.TRAFFIC_FILE, len(w.pass_sizes) + 1) is None


def test_stale_record_is_ignored(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.load_traffic_record(bench.TRAFFIC_FILE) is None
    assert bench.load_traffic(bench.TRAFFIC_FILE) is None
    assert bench.load_perslot_dram(bench.TRAFFIC_FILE, 9) is None
