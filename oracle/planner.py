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
  makespan     each round's job cut into g = 1 .. |S| parts (configurations
               dealt, largest step cost first, ties by index, to the part
               with the least cost so far, ties to the part with fewer
               configurations, then the lower part); for every cap D among
               the cuts' longest parts, from the largest down, each job takes
               its smallest g whose parts all end within D; last, every job
               cut into single configurations.  The first plan (uncut) and
               then every plan that ends strictly sooner is kept.  Then, while
               one exists, the plan one job away (that job cut into one part
               more or one fewer) that ends soonest, strictly sooner than the
               current one, replaces it.
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
    n_gpus = cost.get("n_gpus", 1)

    def job_cost(c):
        return configs[c]["tokens_per_step"] * _w(configs[c], cost)

    def part(members):
        members = sorted(members)
        c_sum = 0.0
        for c in members:  # ascending order, like the rounds' step time
            c_sum += job_cost(c)
        return {"m": members, "step": t0 + c_sum, "dur": max(configs[c]["steps"] for c in members) * (t0 + c_sum)}

    def cut(s, g):
        bins, load = [[] for _ in range(g)], [0.0] * g
        for c in sorted(s, key=lambda c: -job_cost(c)):  # stable: equal costs keep index order
            p = min(range(g), key=lambda q: (load[q], len(bins[q]), q))
            load[p] += job_cost(c)
            bins[p].append(c)
        return [part(b) for b in bins]

    def place(durs):
        order = sorted(range(len(durs)), key=lambda j: -durs[j])  # stable: ties keep job order
        free = [0.0] * n_gpus
        where = [None] * len(durs)
        for j in order:
            g = min(range(n_gpus), key=lambda q: (free[q], q))
            where[j] = (g, free[g])
            free[g] += durs[j]
        return max(free), where

    cuts = [[cut(s, g) for g in range(1, len(s) + 1)] for s in sets]
    longest = [[max(p["dur"] for p in c) for c in cj] for cj in cuts]
    caps = sorted({d for lj in longest for d in lj}, reverse=True)

    def plan_of(gs):
        return [p for j, g in enumerate(gs) for p in cuts[j][g - 1]]

    best_g = [1] * len(sets)
    best_mk = place([p["dur"] for p in plan_of(best_g)])[0]
    tries = []
    for D in caps:
        gs = []
        for j in range(len(sets)):
            g = next((g for g in range(1, len(sets[j]) + 1) if longest[j][g - 1] <= D), None)
            gs.append(g)
        if None not in gs:
            tries.append(gs)
    tries.append([len(s) for s in sets])
    for gs in tries:
        mk = place([p["dur"] for p in plan_of(gs)])[0]
        if mk < best_mk:
            best_mk, best_g = mk, gs
    # refinement: every plan one job away (one part more or one fewer); the one
    # that ends soonest, if strictly sooner (ties: lower job, then one more part)
    for _ in range(4 * len(configs)):
        cand = None
        for j in range(len(sets)):
            for dg in (1, -1):
                g = best_g[j] + dg
                if 1 <= g <= len(sets[j]):
                    t = list(best_g)
                    t[j] = g
                    mk = place([p["dur"] for p in plan_of(t)])[0]
                    if mk < (best_mk if cand is None else cand[0]):
                        cand = (mk, t)
        if cand is None:
            break
        best_mk, best_g = cand

    parts = plan_of(best_g)
    makespan, where = place([p["dur"] for p in parts])
    jobs = [{"gpu": g, "n_configs": len(p["m"]), "start_s": st, "duration_s": p["dur"], "step_s": p["step"]}
            for p, (g, st) in zip(parts, where)]
    job_of = [0] * len(configs)
    for j, p in enumerate(parts):
        for c in p["m"]:
            job_of[c] = j
    return {"job_of": job_of, "jobs": jobs, "makespan_s": makespan, "sets": sets, "parts": [p["m"] for p in parts],
            "rates": [rate(s, configs, cost) for s in sets],
            "lower_bound_s": math.fsum(p["dur"] for p in parts) / n_gpus}
