"""Host logic of bench.py (no GPU): roofline arithmetic against the pages' worked examples, the
whole-job throughput rule, and the max-over-ranks timing across two gloo ranks."""
import os
import sys

import pytest

import bench


def golden_map(golden, name):
    return {r[0]: float(r[1]) for r in golden(name)}


def test_bytes_per_update_match_page(golden):
    g = golden_map(golden, "bytes_per_update.txt")
    # 19 fp32 populations read and written once per cell update
    assert bench.POP_BYTES == 2 * 19 * 4 == g["in_place"]
    assert bench.algorithmic_bytes(1, "AA") == g["in_place"] + bench.FLAG_BYTES
    assert bench.algorithmic_bytes(1, "AB2") == g["two_buffers"] + bench.FLAG_BYTES
    assert bench.fluid_bytes(10, 7) == 7 * 152 + 10


def test_code_balance_roofline_reproduces_portlbm_example(golden):
    g = golden_map(golden, "portlbm_code_balance.txt")
    assert g["read_bytes"] + g["write_bytes"] == g["code_balance"]
    for bw, glups in (("a30_peak_gbs", "a30_peak_glups"), ("a30_measured_gbs", "a30_measured_glups"),
                      ("mi210_peak_gbs", "mi210_peak_glups")):
        assert abs(bench.roofline_glups(g[bw], g["code_balance"]) - g[glups]) < 0.006


def test_whole_job_throughput_counts_all_ranks():
    # 2 ranks x 100 cells x 10 steps = 2000 updates in 1 ms (the slowest rank) -> 2 MLUPS
    assert bench.whole_job_mlups(100, 10, 2, 1e-3) == pytest.approx(2.0)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.reduce_max(0.5 + rank, world)
    out.put((rank, got))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 1.5, 1: 1.5}


def test_dist_env_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)


def test_recorded_traffic_requires_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.txt").write_text("kernel_source_sha256: deadbeef\naa_odd_dram_bytes_per_cell: 150\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "deadbeef")
    assert bench.recorded_traffic("aa_odd") == 150.0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.recorded_traffic("aa_odd") is None


def test_variant_table_and_unknown_name():
    """The variant workloads of the JSON line come from one table (the --variant entry point
    uses the same names); an unknown name stops before any library or GPU work."""
    specs = bench.variant_specs()
    assert "AA_512^3_periodic_fp16_storage" in specs
    assert specs["AA_128^3_sphere_inlet_outlet"] == (128, "AA", {"sphere": True})
    assert {s for (_, s, _) in specs.values()} == {"AA", "AB"}
    with pytest.raises(SystemExit):
        bench.main(["--variant", "no_such_workload"])


def test_code_tokens_ignore_comments_not_code():
    """The kernel-source hash that guards the recorded DRAM traffic sees code only: comment and
    white-space edits keep it, any code edit changes it (string literals are code)."""
    a = "int a = 1; // one\n/* block\n comment */ float b = 2.0f;"
    b = "int  a = 1;\n\n/* other words */ float b = 2.0f; // trailing"
    assert bench.code_tokens(a) == bench.code_tokens(b) == "int a = 1; float b = 2.0f;"
    assert bench.code_tokens(a) != bench.code_tokens(a.replace("2.0f", "3.0f"))
    s = 'const char* u = "x // y /* z */"; char c = \'"\';'
    assert bench.code_tokens(s) == s


def test_reference_arm_prints_the_contract_line(capsys, monkeypatch):
    """`bench.py --impl reference` times the CPU oracle on a bounded slab of the benchmark's
    porous medium and prints one JSON line with the contract's keys; under torchrun the ranks
    other than 0 print nothing."""
    import json
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == bench.UNIT and line["n_gpus"] == 1
    assert (line["steps"], line["warmup"]) == (1, 3) and line["higher_is_better"] is True
    assert line["vs_baseline"] is None and line["dtype"] == "f64" and line["data"] == "synthetic"
    assert "workload" in line["config"] and "sample" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["sample"] == line["config"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""
