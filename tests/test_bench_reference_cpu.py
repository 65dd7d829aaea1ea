"""The benchmark's reference arm (the CPU oracle) runs on the CPU and prints
one JSON line with the contract's fields."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32_n2_t2_h2", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny_fp32_n2_t2_h2"


def test_non_zero_rank_of_the_reference_arm_does_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32_n2_t2_h2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and not r.stdout.strip()


def test_bench_names_every_variant():
    # the bench line names the kernel of every variant the library can pick
    import bench
    from linear_attention_speculative_gb300 import kda
    for v in kda.VARIANTS.values():
        if v:
            assert v in bench.KERNEL_OF_VARIANT and v in bench.VARIANT_NAME


def test_sweep_report_of_verify_and_decode_rows(tmp_path):
    # the committed report generator: per point the dispatcher's plan, the best
    # explicit plan, and the dispatcher plan's own column against the best
    import bench
    rows = [{"workload": "sweep_T1_N1_H16_HV16_softplus", "op": op, "N": 1, "T": 1, "H": 16, "HV": 16,
             "gate": "softplus", "alg_bytes": 2_000_000, "head_steps": 16, "auto": "item:128",
             "us": {"auto": 10.4, "item:64": 10.2, "item:128": 10.3}, "best": "item:64",
             "best_gbs": 2e6 / 10.2e-6 / 1e9, "auto_over_best": 10.4 / 10.2}
            for op in ("verify", "decode")]
    for op, row in zip(("verify", "decode"), rows):
        path = tmp_path / f"{op}.jsonl"
        path.write_text(json.dumps(row) + "\n")
        text = bench.sweep_report(str(path), 6791.0, "measured")
        assert ("kda_conv_decode" in text) == (op == "decode")
        assert "| 1 | 1 | 16 | 16 | softplus | item:128 | 10.4 | item:64 | 10.2 |" in text
        assert "own column / best: mean 1.0098" in text
    # a grouped point: the dispatcher's q/k roll beside its plan, and the
    # cluster plans' table against the dispatcher
    row = {"workload": "sweep_T2_N8_H32_HV64_softplus", "op": "verify", "N": 8, "T": 2, "H": 32, "HV": 64,
           "gate": "softplus", "alg_bytes": 100_000_000, "head_steps": 1024, "auto": "item:64",
           "auto_roll": "cluster",
           "us": {"auto": 24.8, "item:64": 24.6, "item:64:0:0:counter": 26.6, "item:64:0:0:cluster": 24.6},
           "best": "item:64", "best_gbs": 1e8 / 24.6e-6 / 1e9, "auto_over_best": 24.8 / 24.6}
    path = tmp_path / "grouped.jsonl"
    path.write_text(json.dumps(row) + "\n")
    text = bench.sweep_report(str(path), 6791.0, "measured")
    assert "| 2 | 8 | 32 | 64 | softplus | item:64 (cluster) | 24.8 | item:64 | 24.6 |" in text
    assert "Cluster q/k roll" in text and "| 2 | 0.99 |" in text


def test_committed_ncu_summaries_match_the_kernel_sources():
    # the bench line's DRAM traffic comes from these summaries and is dropped
    # (null) once the kernel sources differ from the ones they were taken on
    import bench
    for wl in ("large_bf16_n256_t4_h32", "gva_bf16_n64_t4_h8_hv32_safe", "decode_bf16_n16_t4_h16"):
        total, rd, wr = bench.ncu_traffic(wl, "kda_tile_kernel")
        assert total is not None and total == rd + wr, wl


def test_back_to_back_rotation_sets_evict_each_set_between_uses():
    # between two uses of one set the other R - 1 sets move more than L2 holds
    # (here at least twice L2), and a call larger than L2 alternates two sets
    import bench
    for nbytes in (34_000_000, 88_800_000, 135_000_000, 268_000_000, 1_070_000_000, 2_840_000_000):
        R = bench.rotation_sets(nbytes)
        assert R >= 2 and (R - 1) * nbytes >= 2 * bench.L2_BYTES or R == 2, (nbytes, R)
        assert R * nbytes >= 3 * bench.L2_BYTES
    assert bench.rotation_sets(88_800_000) == 6
    assert bench.rotation_sets(3 * bench.L2_BYTES) == 2
    # tiny calls would need thousands of sets: no back-to-back figure for them
    assert bench.rotation_sets(1_000_000) > bench.MAX_ROTATION_SETS


def test_decode_and_commit_bytes_equal_the_tensors_they_touch():
    import bench
    from linear_attention_speculative_gb300 import workloads as wk
    for wl in (wk.TINY, wk.DECODE, wk.custom(3, 2, 2, 4, 64, 32, gate="safe", seed=3)):
        s = wl.shape
        inp = wk.make_inputs(wl)
        nb = lambda t: t.numel() * t.element_size()
        # plain decode: every input read once, S and conv_state written in place, o written
        o_bytes = s.N * s.T * s.HV * s.V * s.act_bytes
        dec = sum(nb(v) for v in inp.values() if v is not None) + nb(inp["S0"]) + nb(inp["conv_state"]) + o_bytes
        assert bench.decode_bytes(s, wl.gate) == dec, wl.name
        # commit: one token's state and conv window read, the state and conv_state written, the counts read
        out = wk.empty_outputs(wl)
        one = nb(out["inter_ssm"]) // s.T + nb(out["conv_snapshots"]) // s.T
        assert bench.commit_bytes(s) == 2 * one + 4 * s.N, wl.name


def test_cpu_baseline_reports_the_oracle_on_a_bounded_sample():
    import bench
    from linear_attention_speculative_gb300 import workloads as wk
    d = bench.cpu_baseline(wk.TINY, wk.make_inputs(wk.TINY), cpu_seconds=0.2)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["cores"] >= 1 and d["gb_per_s"] > 0
    assert "oracle" in d["sample"]
