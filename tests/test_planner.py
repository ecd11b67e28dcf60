"""The packing planner (lora_plan_pack, host code) against its brute-force
oracle, and the oracle against hand-worked cases.

Pins (hand arithmetic, not the oracle's formula retyped): two identical
configurations pack when a step has a fixed overhead; a memory budget that
fits only two of three configurations picks the pair with the best rate; a
short configuration does not ride along with a long one when it would waste
the job's steps; longest-first placement of durations 5, 4, 3 on two GPUs
ends at 7; a four-configuration job is cut in two across two GPUs (41 s ->
21 s), never on one GPU, and a cut into three that ends no sooner is not
taken; one job cut into one part more when no common cap helps (20 s ->
19 s).  Parity: the library's plan equals the exhaustive search on random
instances (partitions and predicted times), including grouped instances on
2-8 GPUs where the cuts decide the plan, which never ends later than the
uncut jobs or one configuration per job.  Invariants at the size of PLoRA's
120-configuration search space: every configuration placed once, memory
budget kept, makespan above the work / GPUs bound."""
import math

import numpy as np
import pytest

import adapter_sgmv_gb300 as lora
from oracle import planner as oplan

GB = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lora.build_library()
    lora.lib()


def cfg(rank, tok, steps, mem):
    return {"rank": rank, "tokens_per_step": tok, "steps": steps, "mem_bytes": mem}


# ---------------------------------------------------------------- pins of the oracle
def test_identical_configs_pack_when_a_step_has_overhead():
    # t0 = 1, each config adds 1 s per step: alone 100 tok / 2 s = 50, together 200 / 3 = 66.7
    cost = {"step_overhead_s": 1.0, "base_s_per_token": 0.01, "gpu_mem_bytes": 10 * GB, "mem_unit_bytes": GB}
    c = [cfg(8, 100, 10, GB), cfg(8, 100, 10, GB)]
    p = oplan.plan(c, cost)
    assert p["sets"] == [[0, 1]]
    assert math.isclose(p["rates"][0], 200 / 3, rel_tol=1e-12)
    assert math.isclose(p["makespan_s"], 10 * 3.0, rel_tol=1e-12)


def test_memory_budget_picks_the_best_fitting_pair():
    # budget 4 units; sizes 2, 2, 3 -> pairs {0,1} only (3 + 2 > 4); a single 2 is worse than the pair
    cost = {"step_overhead_s": 2.0, "base_s_per_token": 0.01, "gpu_mem_bytes": 4 * GB, "mem_unit_bytes": GB}
    c = [cfg(8, 100, 10, 2 * GB), cfg(8, 100, 10, 2 * GB), cfg(8, 300, 10, 3 * GB)]
    p = oplan.plan(c, cost)
    # {2}: 300 / (2 + 3) = 60; {0,1}: 200 / (2 + 2) = 50; {0}: 100 / 3 = 33.3 -> {2} first, then {0,1}
    assert p["sets"] == [[2], [0, 1]]
    assert math.isclose(p["rates"][0], 60.0) and math.isclose(p["rates"][1], 50.0)


def test_short_config_does_not_waste_a_long_job():
    # long: 100 steps, short: 10 steps; together the job runs 100 steps
    cost = {"step_overhead_s": 0.1, "base_s_per_token": 0.01, "gpu_mem_bytes": 10 * GB, "mem_unit_bytes": GB}
    c = [cfg(8, 100, 100, GB), cfg(8, 100, 10, GB)]
    # {0}: 100*100 / (100 * 1.1) = 90.9; {0,1}: (10000 + 1000) / (100 * 2.1) = 52.4; {1}: 1000 / (10 * 1.1) = 90.9
    p = oplan.plan(c, cost)
    assert sorted(map(tuple, p["sets"])) == [(0,), (1,)]
    assert all(math.isclose(r, 10000 / 110) for r in p["rates"])


def test_longest_first_placement_on_two_gpus():
    # three jobs that cannot share memory, durations 5, 4, 3 (one step each, t0 = 0)
    cost = {"base_s_per_token": 1.0, "gpu_mem_bytes": GB, "mem_unit_bytes": GB, "n_gpus": 2}
    c = [cfg(8, 5, 1, GB), cfg(8, 4, 1, GB), cfg(8, 3, 1, GB)]
    p = oplan.plan(c, cost)
    assert p["makespan_s"] == 7.0
    assert [j["gpu"] for j in p["jobs"]] == [0, 1, 1]


def test_a_job_is_cut_across_gpus_when_that_ends_sooner():
    # four identical configs (1 s of tokens per step, 10 steps), t0 = 0.1, two GPUs.
    # The round packs all four: rate 4000 / (10 * 4.1) = 97.6 beats 3000 / 31 = 96.8.
    # Uncut the job takes 41 s; in two parts {0,2} {1,3} each takes 10 * 2.1 = 21 s,
    # one per GPU -> 21; in four parts 11 s each, two per GPU -> 22.  Two parts win.
    cost = {"step_overhead_s": 0.1, "base_s_per_token": 0.01, "gpu_mem_bytes": 10 * GB, "mem_unit_bytes": GB,
            "n_gpus": 2}
    c = [cfg(8, 100, 10, GB)] * 4
    p = oplan.plan(c, cost)
    assert p["sets"] == [[0, 1, 2, 3]]
    assert p["parts"] == [[0, 2], [1, 3]] and p["job_of"] == [0, 1, 0, 1]
    assert math.isclose(p["makespan_s"], 21.0, rel_tol=1e-12)
    assert [j["gpu"] for j in p["jobs"]] == [0, 1]
    got = lora.lora_plan_pack(c, cost)
    assert got["job_of"] == p["job_of"] and math.isclose(got["makespan_s"], 21.0, rel_tol=1e-12)


def test_one_gpu_never_cuts_and_ties_keep_fewer_jobs():
    c = [cfg(8, 100, 10, GB)] * 4
    base = {"step_overhead_s": 0.1, "base_s_per_token": 0.01, "gpu_mem_bytes": 10 * GB, "mem_unit_bytes": GB}
    # one GPU: a cut only adds step overhead -> one job of 41 s
    p = oplan.plan(c, dict(base, n_gpus=1))
    assert p["parts"] == [[0, 1, 2, 3]] and math.isclose(p["makespan_s"], 41.0, rel_tol=1e-12)
    # three GPUs: parts {0,3} {1} {2} (21, 11, 11 s) end at 21 like two parts -> the two parts stay
    p = oplan.plan(c, dict(base, n_gpus=3))
    assert p["parts"] == [[0, 2], [1, 3]] and math.isclose(p["makespan_s"], 21.0, rel_tol=1e-12)
    for n in (1, 3):
        got = lora.lora_plan_pack(c, dict(base, n_gpus=n))
        want = oplan.plan(c, dict(base, n_gpus=n))
        assert got["job_of"] == want["job_of"] and math.isclose(got["makespan_s"], want["makespan_s"])


def test_one_more_part_for_one_job_when_no_common_cap_helps():
    # five configs (steps, step cost): c0 (1, 2), c1 (1, 1), c2 (2, 2), c3 (2, 2), c4 (2, 4); t0 = 3; two GPUs.
    # Rounds: {0,1} rate 2 / (1 * 6) = 0.333, then {2,3} 4 / (2 * 7) = 0.286 (over {2,3,4} 6 / 22), then {4}.
    # Uncut jobs 6, 14, 14 s -> 14 | 14 + 6 = 20.  Caps: 14 is the uncut plan; 10, 6 and 5 cannot hold {4}
    # (14 s); every job cut into singles (5, 4, 10, 10, 14) ends at 23.  One job away: {0,1} in two parts
    # (5 and 4 s) -> 14 + 5 | 14 + 4 = 19; {2,3} in two parts (10, 10) -> 20.  So {0}, {1}, {2,3}, {4}.
    cost = {"step_overhead_s": 3.0, "lora_s_per_token_rank": 1.0, "gpu_mem_bytes": 10 * GB, "mem_unit_bytes": GB,
            "n_gpus": 2}
    c = [cfg(2, 1, 1, GB), cfg(1, 1, 1, GB), cfg(2, 1, 2, GB), cfg(2, 1, 2, GB), cfg(4, 1, 2, GB)]
    p = oplan.plan(c, cost)
    assert p["sets"] == [[0, 1], [2, 3], [4]]
    assert p["parts"] == [[0], [1], [2, 3], [4]] and p["job_of"] == [0, 1, 2, 2, 3]
    assert math.isclose(p["makespan_s"], 19.0, rel_tol=1e-12)
    assert [(j["gpu"], j["start_s"], j["duration_s"]) for j in p["jobs"]] == [(0, 14.0, 5.0), (1, 14.0, 4.0),
                                                                            (0, 0.0, 14.0), (1, 0.0, 14.0)]
    got = lora.lora_plan_pack(c, cost)
    assert got["job_of"] == p["job_of"] and math.isclose(got["makespan_s"], 19.0, rel_tol=1e-12)


# ---------------------------------------------------------------- library vs oracle
def random_instance(rng, m):
    configs = [cfg(int(rng.choice([8, 16, 32, 64, 128])), int(rng.integers(256, 8192)), int(rng.integers(50, 2000)),
                   int(rng.integers(1, 40)) * (GB // 4)) for _ in range(m)]
    cost = {"step_overhead_s": float(rng.uniform(0.0, 0.2)), "base_s_per_token": float(rng.uniform(1e-6, 2e-5)),
            "lora_s_per_token": float(rng.uniform(0.0, 2e-6)), "lora_s_per_token_rank": float(rng.uniform(0.0, 2e-8)),
            "gpu_mem_bytes": 80 * GB, "job_mem_bytes": int(rng.integers(8, 40)) * GB, "mem_unit_bytes": GB // 4,
            "n_gpus": int(rng.integers(1, 5))}
    return configs, cost


@pytest.mark.parametrize("seed", range(12))
def test_library_plan_equals_exhaustive_search(seed):
    rng = np.random.default_rng(seed)
    configs, cost = random_instance(rng, int(rng.integers(1, 11)))
    want = oplan.plan(configs, cost)
    got = lora.lora_plan_pack(configs, cost)
    assert got["job_of"] == want["job_of"]
    assert len(got["jobs"]) == len(want["jobs"])
    for g, w in zip(got["jobs"], want["jobs"]):
        assert g["gpu"] == w["gpu"] and g["n_configs"] == w["n_configs"]
        for k in ("start_s", "duration_s", "step_s"):
            assert math.isclose(g[k], w[k], rel_tol=1e-12, abs_tol=1e-12), k
    assert math.isclose(got["makespan_s"], want["makespan_s"], rel_tol=1e-12)


def grouped_instance(rng, m):
    # configurations in a few groups of equal steps (one dataset, a few batch
    # sizes), a large memory budget and several GPUs: rounds pack whole groups,
    # and cutting them across the GPUs decides the makespan
    toks = [int(t) for t in rng.choice([512, 1024, 2048, 4096], size=int(rng.integers(1, 4)), replace=False)]
    configs = []
    for _ in range(m):
        tok = toks[int(rng.integers(0, len(toks)))]
        configs.append(cfg(int(rng.choice([8, 16, 32, 64, 128])), tok, 4 * (1 << 20) // tok,
                           int(rng.integers(1, 12)) * (GB // 4)))
    cost = {"step_overhead_s": float(rng.uniform(0.005, 0.05)), "base_s_per_token": float(rng.uniform(2e-6, 1e-5)),
            "lora_s_per_token": float(rng.uniform(0.0, 2e-6)), "lora_s_per_token_rank": float(rng.uniform(0.0, 1e-8)),
            "gpu_mem_bytes": 280 * GB, "job_mem_bytes": 24 * GB, "mem_unit_bytes": GB // 4,
            "n_gpus": int(rng.integers(2, 9))}
    return configs, cost


@pytest.mark.parametrize("seed", range(10))
def test_library_plan_equals_exhaustive_search_with_cuts(seed):
    rng = np.random.default_rng(100 + seed)
    configs, cost = grouped_instance(rng, int(rng.integers(2, 11)))
    want = oplan.plan(configs, cost)
    got = lora.lora_plan_pack(configs, cost)
    assert got["job_of"] == want["job_of"]
    assert [(j["gpu"], j["n_configs"]) for j in got["jobs"]] == [(j["gpu"], j["n_configs"]) for j in want["jobs"]]
    for g, w in zip(got["jobs"], want["jobs"]):
        for k in ("start_s", "duration_s", "step_s"):
            assert math.isclose(g[k], w[k], rel_tol=1e-12, abs_tol=1e-12), k
    assert math.isclose(got["makespan_s"], want["makespan_s"], rel_tol=1e-12)
    # never later than the uncut rounds' jobs, nor than one configuration per job
    uncut = oplan.plan(configs, dict(cost))
    uncut_mk = _lpt([max(configs[c]["steps"] for c in s) * (cost["step_overhead_s"] + sum(
        configs[c]["tokens_per_step"] * _w(configs[c], cost) for c in s)) for s in uncut["sets"]], cost["n_gpus"])
    singles_mk = _lpt([c["steps"] * (cost["step_overhead_s"] + c["tokens_per_step"] * _w(c, cost)) for c in configs],
                      cost["n_gpus"])
    assert want["makespan_s"] <= uncut_mk * (1 + 1e-12) and want["makespan_s"] <= singles_mk * (1 + 1e-12)


def _w(c, cost):
    return cost.get("base_s_per_token", 0.0) + cost.get("lora_s_per_token", 0.0) + \
        cost.get("lora_s_per_token_rank", 0.0) * c["rank"]


def _lpt(durs, n_gpus):
    free = [0.0] * n_gpus
    for d in sorted(durs, reverse=True):
        g = min(range(n_gpus), key=lambda q: (free[q], q))
        free[g] += d
    return max(free)


def test_plora_sized_search_space_invariants():
    # 120 configurations: rank x tokens-per-step x learning-rate variants (the rate does not change the cost)
    rng = np.random.default_rng(7)
    configs = []
    for r in (8, 16, 32, 64, 128):
        for tok in (1024, 2048, 4096, 8192):
            for _ in range(6):
                configs.append(cfg(r, tok, int(rng.integers(200, 1200)), (2 + r // 16) * GB + tok * 2 * (1 << 20)))
    cost = {"step_overhead_s": 0.03, "base_s_per_token": 1.2e-5, "lora_s_per_token": 2e-6,
            "lora_s_per_token_rank": 1e-8, "gpu_mem_bytes": 280 * GB, "job_mem_bytes": 24 * GB,
            "mem_unit_bytes": GB // 4, "n_gpus": 8}
    p = lora.lora_plan_pack(configs, cost)
    jobs = p["jobs"]
    assert sorted(set(p["job_of"])) == list(range(len(jobs)))
    assert sum(j["n_configs"] for j in jobs) == len(configs)
    budget = (cost["gpu_mem_bytes"] - cost["job_mem_bytes"]) // cost["mem_unit_bytes"]
    for j in range(len(jobs)):
        members = [c for c, q in enumerate(p["job_of"]) if q == j]
        assert sum(-(-configs[c]["mem_bytes"] // cost["mem_unit_bytes"]) for c in members) <= budget
        steps = max(configs[c]["steps"] for c in members)
        assert math.isclose(jobs[j]["duration_s"], steps * jobs[j]["step_s"], rel_tol=1e-12)
    work = sum(j["duration_s"] for j in jobs)
    assert p["makespan_s"] >= work / cost["n_gpus"] * (1 - 1e-12)
    assert p["makespan_s"] <= work / cost["n_gpus"] + max(j["duration_s"] for j in jobs) + 1e-9
    # packing beats one configuration per job on the same pool under the same cost model
    singles = sorted((c["steps"] * (cost["step_overhead_s"] + c["tokens_per_step"] * (
        cost["base_s_per_token"] + cost["lora_s_per_token"] + cost["lora_s_per_token_rank"] * c["rank"]))
        for c in configs), reverse=True)
    free = [0.0] * cost["n_gpus"]
    for d in singles:
        g = min(range(len(free)), key=lambda q: (free[q], q))
        free[g] += d
    assert p["makespan_s"] < max(free)


def test_planner_rejects_a_config_larger_than_a_gpu():
    cost = {"gpu_mem_bytes": 80 * GB, "job_mem_bytes": 20 * GB, "mem_unit_bytes": GB, "base_s_per_token": 1e-5}
    with pytest.raises(lora.LoraError) as e:
        lora.lora_plan_pack([cfg(8, 1024, 10, 61 * GB)], cost)
    assert e.value.status == 2


def test_planner_rejects_a_knapsack_table_too_large():
    # 4096 configurations over a 2^20-unit budget would need a 4 GB choice table
    cost = {"gpu_mem_bytes": (1 << 20) * 1024, "mem_unit_bytes": 1024, "base_s_per_token": 1e-5}
    with pytest.raises(lora.LoraError) as e:
        lora.lora_plan_pack([cfg(8, 1024, 10, 4096)] * 4096, cost)
    assert e.value.status == 2
