"""Host-side rules of the benchmark, on CPU: which workloads flush L2 between timed
steps, the algorithmic bytes and FLOPs charged to each stage, and the keys under
which committed profiles record a stage's DRAM traffic."""
import json
import os
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _layer(w, touched, payload="bf16", gather=False):
    counts = torch.zeros(w.E, dtype=torch.int32)
    counts[:touched] = 1
    z = torch.zeros(1)
    return types.SimpleNamespace(counts=counts, payload=payload, gather=gather, fused_fp8=False,
                                 w_gate=z, w_up=z, w_down=z, capacity=-1)


def test_l2_rule_flushes_exactly_the_small_working_sets():
    d1 = workloads.decode(1)
    ws1 = bench.working_set_bytes(d1, _layer(d1, 8))       # 8 experts: 75.6 MB of weights
    assert 75e6 < ws1 < 2 * bench.L2_BYTES
    d8 = workloads.decode(8)
    ws8 = bench.working_set_bytes(d8, _layer(d8, 47))      # about 47 experts touched
    assert ws8 > 2 * bench.L2_BYTES
    d128 = workloads.decode(128)
    assert bench.working_set_bytes(d128, _layer(d128, 123)) > 2 * bench.L2_BYTES
    tiny = workloads.tiny()
    assert bench.working_set_bytes(tiny, _layer(tiny, 8)) < 2 * bench.L2_BYTES
    # the pooled step streams its pools, compact arrays and outputs (GBs), not only the
    # six local experts' weights (170 MB)
    p = workloads.pooled()
    m = dict(dtype=torch.bfloat16, device="meta")
    rows = p.local_per_dest * 33497
    pl = types.SimpleNamespace(w_gate=torch.empty((6, p.d, p.I), **m),
                               w_up=torch.empty((6, p.d, p.I), **m),
                               w_down=torch.empty((6, p.I, p.d), **m),
                               pools=torch.empty((p.n_dest, 3005, p.d), **m),
                               compact=torch.empty((rows, p.d), **m),
                               y=torch.empty((rows, p.d), **m), rows=rows)
    assert bench.working_set_bytes(p, pl) > 5e9


def test_stage_work_follows_the_method_and_the_gather_option():
    w = workloads.prefill()
    acc = w.T * w.k
    counts = torch.full((w.E,), acc // w.E).numpy()
    copy = _layer(w, w.E)
    gath = _layer(w, w.E, gather=True)
    b_copy, _ = bench.stage_work(w, copy, "permute", counts, acc, w.E, w.I, w.d)
    b_gath, _ = bench.stage_work(w, gath, "permute", counts, acc, w.E, w.I, w.d)
    # the copying permute moves every token row once and every accepted row once more
    assert b_copy - b_gath == w.T * w.d * 2 + acc * w.d * 2
    b, f = bench.stage_work(w, copy, "gate_up", counts, acc, w.E, w.I, w.d)
    assert f == 4 * acc * w.d * w.I
    assert b == w.E * 2 * w.d * w.I * 2 + acc * w.d * 2 + acc * w.I * 2
    _, f_down = bench.stage_work(w, copy, "down", counts, acc, w.E, w.I, w.d)
    assert f + f_down == 6 * acc * w.d * w.I  # F = 6 n d d_ff


def test_traffic_keys_name_workload_payload_and_gather():
    w = workloads.v3()
    assert bench.traffic_key(w, _layer(w, 1)) == "v3"
    assert bench.traffic_key(w, _layer(w, 1, payload="fp8_row")) == "v3+fp8_row"
    assert bench.traffic_key(w, _layer(w, 1, gather=True)) == "v3+gather"


def test_committed_traffic_lines_are_read_only_for_the_current_source():
    line, _ = bench.lookup_traffic("gate_up", "decode_T128")
    # the profiles committed with this source carry the gate/up pass's DRAM bytes
    assert line is None or 7e8 < line < 9e8


def test_traffic_lines_with_a_scaling_note(tmp_path, monkeypatch):
    """A capture of a smaller case carries a note saying how it was scaled."""
    sha = bench.kernel_source_sha("combine")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.md").write_text(f"traffic: combine pooled 123 {sha} scaled x4 from T=16384\n"
                               f"traffic: combine v3 77 {sha}\n"
                               f"traffic: combine tiny 5 0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda name: sha)
    assert bench.lookup_traffic("combine", "pooled") == (123, "scaled x4 from T=16384")
    assert bench.lookup_traffic("combine", "v3") == (77, None)
    assert bench.lookup_traffic("combine", "tiny") == (None, None)


def test_nearest_rank_quantiles():
    """Q_q = x_(ceil(q n)): the smallest value with at least q n values at or below it."""
    assert bench.nearest_rank([5, 1, 3, 2, 4], 0.5) == 3
    assert bench.nearest_rank([1, 2, 3, 4], 0.5) == 2
    assert bench.nearest_rank(list(range(1, 11)), 0.9) == 9
    assert bench.nearest_rank([7.0], 0.9) == 7.0


def test_results_log_appends_and_resumes(tmp_path, capsys):
    """--jsonl appends each run's line with its run arguments; --resume finds the last
    line recorded for the same arguments (a torn last line is skipped)."""
    log = str(tmp_path / "runs.jsonl")
    args = types.SimpleNamespace(**{k: None for k in bench.RUN_KEYS})
    args.jsonl, args.config, args.tokens = log, "decode", 8
    bench.emit({"value": 1.0}, args)
    args.tokens = 32
    bench.emit({"value": 2.0}, args)
    args.tokens = 8
    bench.emit({"value": 3.0}, args)
    with open(log, "a") as f:
        f.write('{"value": 4.0, "run": ')  # an interrupted append
    assert bench.logged_line(log, bench.run_key(args))["value"] == 3.0
    args.tokens = 32
    assert bench.logged_line(log, bench.run_key(args))["value"] == 2.0
    args.tokens = 1
    assert bench.logged_line(log, bench.run_key(args)) is None
    assert bench.logged_line(str(tmp_path / "missing.jsonl"), bench.run_key(args)) is None
    out = capsys.readouterr().out.strip().splitlines()
    assert [json.loads(l)["value"] for l in out] == [1.0, 2.0, 3.0]
