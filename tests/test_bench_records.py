"""Host checks of the benchmark's committed ncu DRAM records and of the code
that writes and reads them: a record is used only while its source hash
matches the kernels' code, it round-trips from an ncu csv, and every
committed record's DRAM bytes are plausible against the requested bytes (a
dedup call reads each requested byte from DRAM about once; a per-slot call
never reads more than it requests)."""
import json
import os
import types

import pytest

import bench


def _fake_capture(tmp_path, calls, dram):
    """A --calls JSON and an ncu csv in the form ncu writes (two metrics per
    launch, an unrelated kernel in between)."""
    cj = tmp_path / "calls.json"
    cj.write_text(json.dumps({"workload": "v2lite", "rho": 0.9, "calls": calls,
                              "sources_sha256_16": bench.kernel_source_hash()}))
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
            '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
            '"Metric Value"\n')
    lines = ["==PROF== Connected to process 1\n", head]
    for i, (rd, wr) in enumerate(dram):
        kn = "void unnamed>::expert_mma_kernel(unnamed>::Params)"
        for m, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr)):
            lines.append('"%d","1","python3","h","%s","1","7","(384, 1, 1)","(152, 1, 1)","0",'
                         '"10.3","Command line profiler metrics","%s","byte","%s"\n'
                         % (i, kn, m, "{:,}".format(v)))
    cv = tmp_path / "dram.csv"
    cv.write_text("".join(lines))
    return str(cj), str(cv)


def test_dram_record_round_trip(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "dram_record_path",
                        lambda wl: str(tmp_path / ("dram_expert_calls_%s.txt" % wl)))
    calls, dram = [], []
    for n in (1, 2, 3):
        for eng, req, rd in (("perslot", 1000 * n, 700 * n), ("dedup", 900, 901)):
            calls.append({"n": n, "engine": eng, "requested": req})
            dram.append((rd, 3))
    cj, cv = _fake_capture(tmp_path, calls, dram)
    bench.run_dram_record(types.SimpleNamespace(dram_record=(cj, cv)))
    rec = bench.load_dram_record("v2lite")
    assert rec["n"] == [1, 2, 3] and rec["rho"] == 0.9
    assert rec["perslot_requested"] == [1000, 2000, 3000]
    assert rec["perslot_dram"] == [703, 1403, 2103]
    assert rec["dedup_dram"] == [904, 904, 904]
    f = bench.dram_factor("v2lite")
    assert f["perslot"][2] == pytest.approx(1403 / 900)       # over the pass's unique bytes
    assert f["dedup"][3] == pytest.approx(904 / 900)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.load_dram_record("v2lite") is None           # other kernel sources
    assert bench.dram_factor("v2lite") is None


def test_dram_record_refuses_a_launch_count_mismatch(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "dram_record_path", lambda wl: str(tmp_path / "x.txt"))
    calls = [{"n": 1, "engine": "perslot", "requested": 10},
             {"n": 1, "engine": "dedup", "requested": 10}]
    cj, cv = _fake_capture(tmp_path, calls, [(5, 0)])
    with pytest.raises(SystemExit):
        bench.run_dram_record(types.SimpleNamespace(dram_record=(cj, cv)))
    assert not os.path.exists(tmp_path / "x.txt")


@pytest.mark.parametrize("workload", ["v2lite", "mixtral", "v3"])
def test_committed_records_are_plausible(workload):
    rec = bench.load_dram_record(workload, check_hash=False)
    if rec is None:
        pytest.skip("no committed DRAM record for %s" % workload)
    for i, n in enumerate(rec["n"]):
        ps_req, ps_dr = rec["perslot_requested"][i], rec["perslot_dram"][i]
        dd_req, dd_dr = rec["dedup_requested"][i], rec["dedup_dram"][i]
        assert 0.97 * dd_req <= dd_dr <= 1.03 * dd_req, (workload, n, dd_req, dd_dr)
        assert ps_dr <= 1.03 * ps_req, (workload, n, ps_req, ps_dr)
        assert ps_dr >= 0.97 * dd_req, (workload, n)   # the same pass's unique bytes at least
        assert ps_req >= dd_req


def test_crossovers_within_one_pass_size():
    """The stack check's "within one pass size" count: "never" (None) counts
    as one past the largest measured pass size."""
    assert bench._within_one(2, 2, 9) and bench._within_one(2, 3, 9)
    assert not bench._within_one(2, 4, 9)
    assert bench._within_one(None, 9, 9) and bench._within_one(9, None, 9)
    assert not bench._within_one(None, 8, 9)
    assert bench._within_one(None, None, 9)


def test_headline_step_plan_covers_both_engines_at_every_pass_size():
    """One bench step: every pass size once with each engine (18 stack passes,
    90 tokens), the hidden-state variant alternating by step."""
    from moe_expert_layer_warp_gb300 import configs
    w = configs.V2_LITE_STACK
    for step in range(4):
        plan = bench.step_plan(w, step)
        assert sorted((n, e) for n, e, _ in plan) == sorted(
            (n, e) for n in w.pass_sizes for e in ("perslot", "dedup"))
        assert {q for _, _, q in plan} == {step % bench.N_PASSES_PER_N}
    assert sum(n for n, _, _ in bench.step_plan(w, 0)) == 90
    assert bench.kernels_per_pass() * 2 * len(w.pass_sizes) * w.layers == 1872


def test_best_engine_rate_takes_the_faster_engine_at_each_n():
    stack = {"per_rho": [
        {"rho": 0.5, "n": [1, 2], "measured_us": {"perslot": [1.0, 1.0], "dedup": [1.0, 1.0]}},
        {"rho": bench.HEADLINE_RHO, "n": [1, 2, 3],
         "measured_us": {"perslot": [100.0, 300.0, 500.0], "dedup": [110.0, 200.0, 250.0]}}]}
    r = bench.best_engine_rate(stack)
    assert r["engine_by_n"] == ["perslot", "dedup", "dedup"]
    assert r["tokens_per_s"] == pytest.approx(6 / 550e-6, rel=1e-6)
    assert r["per_slot_only_tokens_per_s"] == pytest.approx(6 / 900e-6, rel=1e-6)
    assert bench.best_engine_rate(None) is None
