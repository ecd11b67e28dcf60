"""Brute-force oracle of the packing planner (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` import this module; the library's
planner (``lora_plan_pack``) never calls it and shares no code with it.

What it computes, written from the PLoRA technical summary, "1. LoRA Packing
Planner (Offline)" (completion time of a set of LoRA configurations on a fixed
GPU pool, a 0-1 knapsack variant, configurations packed into jobs round after
round with a cost model, then the jobs placed on the hardware), with the
readings stated in the library's header:

  step time    t(S) = t0 + sum_{c in S} tok_c * w_c,
               w_c = base + lora + lora_rank * r_c
  job          runs max_{c in S} steps_c steps of t(S)
  round        the remaining set S that fits one GPU's memory budget (whole
               units, each size rounded up) and maximises
               rate(S) = sum_c steps_c tok_c / (max_c steps_c * t(S)),
               found here by enumerating every subset
  placement    jobs longest first (stable), each on the GPU that frees first
               (lowest index on ties)

Plain Python loops over all 2^M subsets, so only for small M.
"""
from __future__ import annotations

import itertools
import math


def _w(c, cost):
    return cost.get("base_s_per_token", 0.0) + cost.get("lora_s_per_token", 0.0) + \
        cost.get("lora_s_per_token_rank", 0.0) * c["rank"]


def rate(subset, configs, cost):
    """Tokens trained per second by a job packing `subset`."""
    t = cost.get("step_overhead_s", 0.0) + sum(configs[c]["tokens_per_step"] * _w(configs[c], cost) for c in subset)
    steps = max(configs[c]["steps"] for c in subset)
    return sum(configs[c]["steps"] * configs[c]["tokens_per_step"] for c in subset) / (steps * t)


def plan(configs, cost):
    unit = cost.get("mem_unit_bytes", 1 << 20)
    cap = (cost["gpu_mem_bytes"] - cost.get("job_mem_bytes", 0)) // unit
    units = [-(-c["mem_bytes"] // unit) for c in configs]
    left = list(range(len(configs)))
    sets = []
    while left:
        best, best_r = None, -1.0
        for k in range(1, len(left) + 1):
            for sub in itertools.combinations(left, k):
                if sum(units[c] for c in sub) > cap:
                    continue
                r = rate(sub, configs, cost)
                if r > best_r:
                    best, best_r = sub, r
        if best is None:
            raise ValueError("a configuration does not fit one GPU")
        sets.append(sorted(best))
        left = [c for c in left if c not in best]
    t0 = cost.get("step_overhead_s", 0.0)
    step = [t0 + sum(configs[c]["tokens_per_step"] * _w(configs[c], cost) for c in s) for s in sets]
    dur = [max(configs[c]["steps"] for c in s) * st for s, st in zip(sets, step)]
    order = sorted(range(len(sets)), key=lambda j: -dur[j])  # stable: ties keep creation order
    free = [0.0] * cost.get("n_gpus", 1)
    jobs = [None] * len(sets)
    for j in order:
        g = min(range(len(free)), key=lambda q: (free[q], q))
        jobs[j] = {"gpu": g, "n_configs": len(sets[j]), "start_s": free[g], "duration_s": dur[j], "step_s": step[j]}
        free[g] += dur[j]
    job_of = [0] * len(configs)
    for j, s in enumerate(sets):
        for c in s:
            job_of[c] = j
    return {"job_of": job_of, "jobs": jobs, "makespan_s": max(free), "sets": sets,
            "rates": [rate(s, configs, cost) for s in sets], "lower_bound_s": math.fsum(dur) / len(free)}
