// planner.cu -- the packing planner (host code only): group LoRA fine-tuning
// configurations into packed jobs and place the jobs on a pool of GPUs.
//
// PLoRA's offline planner minimises the total completion time of a set of LoRA
// configurations on a fixed hardware pool, a 0-1 knapsack variant; a
// decomposed throughput maximisation picks, round after round, the set of
// configurations to pack into the next job, a cost model estimates memory and
// throughput, and a job planner assigns the jobs to the hardware (PLoRA
// technical summary, "1. LoRA Packing Planner (Offline)").  The pages name a
// commercial ILP solver; this planner solves each round's problem exactly
// with its own method:
//
//   cost model   one job step of the packed set S takes
//                  t(S) = t0 + sum_{c in S} tok_c w_c,
//                  w_c  = base_s_per_token + lora_s_per_token + lora_s_per_token_rank * r_c
//                and the job runs max_{c in S} steps_c steps;
//   round        among the configurations not yet placed, the set S whose
//                memory fits one GPU and that trains the most tokens per
//                second, rate(S) = sum_c steps_c tok_c / (max_c steps_c * t(S));
//   solver       for every choice of the job's longest configuration l (which
//                fixes the denominator's step count), the ratio of two linear
//                functions is maximised by Dinkelbach iterations, each one an
//                exact 0-1 knapsack over the memory budget (dynamic
//                programming in whole memory units);
//   placement    the jobs, longest first, each on the GPU that frees first.
//
// The parallelism degree of a job is one GPU: the library's jobs run on a
// single GPU each (a pool of GPUs runs independent jobs side by side).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "lora_sgmv.h"

namespace {

struct Item {
    double n;        // steps_c * tok_c: tokens the configuration trains
    double cost;     // tok_c * w_c: seconds it adds to every job step
    int64_t steps;
    int32_t units;   // memory, whole units
};

// Best set containing `lead` among `cand` (all with steps <= steps of lead),
// by Dinkelbach's method; returns its rate (0 if lead does not fit).
double best_with_leader(const std::vector<Item> &items, const std::vector<int> &cand, int lead, int32_t cap,
                        double t0, std::vector<int> &best_set)
{
    const Item &L = items[lead];
    const int32_t room = cap - L.units;
    best_set.clear();
    if (room < 0) return 0.0;
    const double sl = (double)L.steps;
    double N = L.n, D = sl * (t0 + L.cost);
    double lambda = N / D;
    std::vector<int> set{lead};
    const int m = (int)cand.size();
    std::vector<double> val(m);
    std::vector<double> dp((size_t)room + 1);
    std::vector<uint8_t> take((size_t)m * (room + 1));
    for (int iter = 0; iter < 64; ++iter) {
        // F(lambda) = max over S containing lead of N(S) - lambda D(S): a 0-1
        // knapsack with values n_c - lambda * steps_l * cost_c (only positive
        // ones can help) on top of the leader's own term
        std::fill(dp.begin(), dp.end(), 0.0);
        for (int i = 0; i < m; ++i) {
            const Item &it = items[cand[i]];
            val[i] = it.n - lambda * sl * it.cost;
            uint8_t *tk = take.data() + (size_t)i * (room + 1);
            std::memset(tk, 0, (size_t)room + 1);
            if (!(val[i] > 0.0) || it.units > room) continue;
            for (int32_t w = room; w >= it.units; --w) {
                const double v = dp[w - it.units] + val[i];
                if (v > dp[w]) {
                    dp[w] = v;
                    tk[w] = 1;
                }
            }
        }
        // reconstruct from the full budget
        std::vector<int> s{lead};
        int32_t w = room;
        for (int i = m - 1; i >= 0; --i) {
            if (take[(size_t)i * (room + 1) + w]) {
                s.push_back(cand[i]);
                w -= items[cand[i]].units;
            }
        }
        double n = 0.0, c = 0.0;
        for (int k : s) {
            n += items[k].n;
            c += items[k].cost;
        }
        const double d = sl * (t0 + c);
        const double F = n - lambda * d;
        if (F <= 1e-12 * n) {  // no set beats the current ratio: lambda is the optimum
            if (n / d > N / D) {
                N = n;
                D = d;
                set = s;
            }
            break;
        }
        N = n;
        D = d;
        set = s;
        lambda = n / d;
    }
    std::sort(set.begin(), set.end());
    best_set = set;
    return N / D;
}

lora_status_t plan_pack(const lora_plan_config *configs, int32_t n_configs, const lora_plan_cost *cost,
                        int32_t *job_of, lora_plan_job *jobs, int32_t *n_jobs, double *makespan_s)
{
    if (configs == nullptr || cost == nullptr || job_of == nullptr || jobs == nullptr || n_jobs == nullptr ||
        makespan_s == nullptr)
        return LORA_ERR_INVALID_ARG;
    if (n_configs < 1 || n_configs > 4096 || cost->n_gpus < 1 || cost->mem_unit_bytes < 1) return LORA_ERR_SHAPE;
    if (!(cost->step_overhead_s >= 0.0) || !(cost->base_s_per_token >= 0.0) || !(cost->lora_s_per_token >= 0.0) ||
        !(cost->lora_s_per_token_rank >= 0.0))
        return LORA_ERR_INVALID_ARG;
    const int64_t budget = cost->gpu_mem_bytes - cost->job_mem_bytes;
    if (budget <= 0) return LORA_ERR_SHAPE;
    const int64_t cap64 = budget / cost->mem_unit_bytes;
    if (cap64 > (1 << 20)) return LORA_ERR_SHAPE;  // the knapsack table would be too large: use a coarser unit
    const int32_t cap = (int32_t)cap64;
    // the knapsack's choice table holds n_configs x (budget + 1) bytes
    if ((int64_t)n_configs * (cap64 + 1) > (int64_t(1) << 28)) return LORA_ERR_SHAPE;
    const double t0 = cost->step_overhead_s;

    std::vector<Item> items(n_configs);
    for (int32_t c = 0; c < n_configs; ++c) {
        const lora_plan_config &k = configs[c];
        if (k.rank < 1 || k.tokens_per_step < 1 || k.steps < 1 || k.mem_bytes < 0) return LORA_ERR_SHAPE;
        const int64_t units = (k.mem_bytes + cost->mem_unit_bytes - 1) / cost->mem_unit_bytes;
        if (units > cap) return LORA_ERR_SHAPE;  // does not fit one GPU even alone
        const double w =
            cost->base_s_per_token + cost->lora_s_per_token + cost->lora_s_per_token_rank * (double)k.rank;
        items[c] = Item{(double)k.steps * k.tokens_per_step, (double)k.tokens_per_step * w, k.steps, (int32_t)units};
        if (!(t0 + items[c].cost > 0.0)) return LORA_ERR_INVALID_ARG;  // a step must take some time
    }

    // rounds: the best remaining set becomes the next job
    std::vector<char> placed(n_configs, 0);
    std::vector<std::vector<int>> sets;
    std::vector<double> dur, step;
    int32_t left = n_configs;
    std::vector<int> cand, s, best;
    while (left > 0) {
        double best_rate = -1.0;
        for (int32_t l = 0; l < n_configs; ++l) {
            if (placed[l]) continue;
            cand.clear();
            for (int32_t c = 0; c < n_configs; ++c)
                if (!placed[c] && c != l && items[c].steps <= items[l].steps) cand.push_back(c);
            const double r = best_with_leader(items, cand, l, cap, t0, s);
            if (r > best_rate) {
                best_rate = r;
                best = s;
            }
        }
        if (best.empty()) return LORA_ERR_SHAPE;
        double c_sum = 0.0;
        int64_t smax = 0;
        for (int k : best) {
            placed[k] = 1;
            job_of[k] = (int32_t)sets.size();
            c_sum += items[k].cost;
            smax = std::max(smax, items[k].steps);
        }
        left -= (int32_t)best.size();
        step.push_back(t0 + c_sum);
        dur.push_back((double)smax * (t0 + c_sum));
        sets.push_back(best);
    }

    // placement: longest job first, on the GPU that frees first (lowest index on ties)
    const int32_t nj = (int32_t)sets.size();
    std::vector<int32_t> order(nj);
    for (int32_t j = 0; j < nj; ++j) order[j] = j;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return dur[a] > dur[b]; });
    std::vector<double> free_at(cost->n_gpus, 0.0);
    double makespan = 0.0;
    for (int32_t j : order) {
        int32_t g = 0;
        for (int32_t q = 1; q < cost->n_gpus; ++q)
            if (free_at[q] < free_at[g]) g = q;
        jobs[j].gpu = g;
        jobs[j].n_configs = (int32_t)sets[j].size();
        jobs[j].start_s = free_at[g];
        jobs[j].duration_s = dur[j];
        jobs[j].step_s = step[j];
        free_at[g] += dur[j];
        makespan = std::max(makespan, free_at[g]);
    }
    *n_jobs = nj;
    *makespan_s = makespan;
    return LORA_OK;
}

}  // namespace

// The planner is host code: any allocation failure is reported as a status,
// never thrown across the C boundary.
extern "C" LORA_API lora_status_t lora_plan_pack(const lora_plan_config *configs, int32_t n_configs,
                                                 const lora_plan_cost *cost, int32_t *job_of, lora_plan_job *jobs,
                                                 int32_t *n_jobs, double *makespan_s)
{
    try {
        return plan_pack(configs, n_configs, cost, job_of, jobs, n_jobs, makespan_s);
    } catch (...) {
        return LORA_ERR_SHAPE;
    }
}
