"""The bench's CPU oracle leg: independent single-threaded oracle processes, one per core, combined into the
box's time per layer (the reference arm and the cpu_baseline figure)."""
import math

import bench


def test_rates_of_side_by_side_processes_add():
    a = {"us_per_layer": 100.0, "steps": 3, "warmup": 1, "router_ms": 1.0, "expert_ms": 10.0, "kept": 8.0,
         "ms_per_step": 11.0, "accuracy": {"near_ties": 0}}
    b = {"us_per_layer": 300.0, "steps": 3, "warmup": 1, "router_ms": 3.0, "expert_ms": 30.0, "kept": 6.0,
         "ms_per_step": 33.0}
    r = bench.combine_oracle_results([a, b])
    assert math.isclose(r["us_per_layer"], 75.0)  # 1 / (1/100 + 1/300)
    assert r["single_core_us"] == 200.0
    assert r["procs"] == 2 and r["steps"] == 6
    assert r["accuracy"] == {"near_ties": 0}  # process 0's check is kept
    assert math.isclose(r["kept"], 7.0) and math.isclose(r["router_ms"], 2.0)


def test_one_process_is_its_own_figure():
    a = {"us_per_layer": 123.0, "steps": 2, "warmup": 0, "router_ms": 1.0, "expert_ms": 2.0, "kept": 4.0,
         "ms_per_step": 3.0}
    r = bench.combine_oracle_results([a])
    assert math.isclose(r["us_per_layer"], 123.0) and r["single_core_us"] == 123.0 and r["procs"] == 1


def test_processes_run_the_oracle_on_their_own_tokens():
    r = bench.run_oracle_steps("tiny", 2, 0, procs=2)
    assert r["procs"] == 2 and r["steps"] == 4
    assert r["us_per_layer"] > 0 and r["us_per_layer"] <= r["single_core_us"]
    assert "2 single-threaded oracle processes" in bench.oracle_sample(r, "tiny")
