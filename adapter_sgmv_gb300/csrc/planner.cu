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
//   makespan     a round's job can be long enough to set the pool's
//                completion time alone (a GPU with a large memory budget packs
//                many configurations into it), so jobs are cut into balanced
//                parts where that finishes the pool sooner: for a cap D on a
//                job's duration, every job is cut into the fewest parts that
//                each end within D (configurations dealt, largest step cost
//                first, to the part with the least cost so far); the caps
//                tried are the part durations themselves, plus every job cut
//                into single configurations, and the plan that ends first
//                under the placement below is kept (ties keep fewer jobs);
//                then, while it helps, one job at a time is cut into one part
//                more or one fewer (the change that ends the pool soonest);
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

// One part of a cut job: its configurations (ascending), step time and duration.
struct Part {
    std::vector<int> m;
    double step, dur;
};

// `set` (ascending) cut into g parts: configurations dealt, largest step cost
// first (ties: lower index), each to the part with the least cost so far
// (ties: fewer configurations, then the lower part index).  A part's step
// time adds its costs in ascending configuration order, as a round's job does,
// so one part reproduces the uncut job exactly.
std::vector<Part> cut_job(const std::vector<Item> &items, const std::vector<int> &set, int g, double t0)
{
    std::vector<int> order(set);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return items[a].cost > items[b].cost; });
    std::vector<double> load(g, 0.0);
    std::vector<Part> parts(g);
    for (int c : order) {
        int p = 0;
        for (int q = 1; q < g; ++q)
            if (load[q] < load[p] || (load[q] == load[p] && parts[q].m.size() < parts[p].m.size())) p = q;
        load[p] += items[c].cost;
        parts[p].m.push_back(c);
    }
    for (Part &P : parts) {
        std::sort(P.m.begin(), P.m.end());
        double c_sum = 0.0;
        int64_t smax = 0;
        for (int k : P.m) {
            c_sum += items[k].cost;
            smax = std::max(smax, items[k].steps);
        }
        P.step = t0 + c_sum;
        P.dur = (double)smax * (t0 + c_sum);
    }
    return parts;
}

// Longest job first (stable), each on the GPU that frees first (lowest index
// on ties); returns the completion time of the pool.
double place(const std::vector<double> &dur, int32_t n_gpus, std::vector<int32_t> *gpu, std::vector<double> *start)
{
    const int32_t nj = (int32_t)dur.size();
    std::vector<int32_t> order(nj);
    for (int32_t j = 0; j < nj; ++j) order[j] = j;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return dur[a] > dur[b]; });
    std::vector<double> free_at(n_gpus, 0.0);
    double makespan = 0.0;
    if (gpu) gpu->assign(nj, 0);
    if (start) start->assign(nj, 0.0);
    for (int32_t j : order) {
        int32_t g = 0;
        for (int32_t q = 1; q < n_gpus; ++q)
            if (free_at[q] < free_at[g]) g = q;
        if (gpu) (*gpu)[j] = g;
        if (start) (*start)[j] = free_at[g];
        free_at[g] += dur[j];
        makespan = std::max(makespan, free_at[g]);
    }
    return makespan;
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
        for (int k : best) placed[k] = 1;
        left -= (int32_t)best.size();
        sets.push_back(best);
    }

    // makespan: every job cut into g = 1 .. |S| parts; the longest part of each
    // cut is a cap to try
    const int32_t n_sets = (int32_t)sets.size();
    std::vector<std::vector<std::vector<Part>>> cuts(n_sets);
    std::vector<std::vector<double>> longest(n_sets);
    std::vector<double> caps;
    for (int32_t j = 0; j < n_sets; ++j) {
        for (int g = 1; g <= (int)sets[j].size(); ++g) {
            cuts[j].push_back(cut_job(items, sets[j], g, t0));
            double d = 0.0;
            for (const Part &P : cuts[j].back()) d = std::max(d, P.dur);
            longest[j].push_back(d);
            caps.push_back(d);
        }
    }
    std::sort(caps.begin(), caps.end(), [](double a, double b) { return a > b; });
    caps.erase(std::unique(caps.begin(), caps.end()), caps.end());
    // the plans in the order they are tried: uncut, each cap from the largest
    // down, every job cut into single configurations; a plan is kept only if it
    // ends strictly sooner than the best so far
    std::vector<int> g_of(n_sets, 1), best_g(n_sets, 1);
    auto durations = [&](const std::vector<int> &gs) {
        std::vector<double> d;
        for (int32_t j = 0; j < n_sets; ++j)
            for (const Part &P : cuts[j][gs[j] - 1]) d.push_back(P.dur);
        return d;
    };
    double best_mk = place(durations(best_g), cost->n_gpus, nullptr, nullptr);
    for (size_t k = 0; k <= caps.size(); ++k) {
        bool ok = true;
        for (int32_t j = 0; j < n_sets && ok; ++j) {
            const int n = (int)sets[j].size();
            if (k == caps.size()) {
                g_of[j] = n;
                continue;
            }
            int g = 1;
            while (g <= n && longest[j][g - 1] > caps[k]) ++g;
            if (g > n) ok = false;
            g_of[j] = g;
        }
        if (!ok) continue;
        const double mk = place(durations(g_of), cost->n_gpus, nullptr, nullptr);
        if (mk < best_mk) {
            best_mk = mk;
            best_g = g_of;
        }
    }
    // refinement: one job at a time cut into one part more or one fewer; the
    // change that ends the pool soonest (strictly sooner than now; ties: the
    // lower job, one more before one fewer) is taken, until none helps.  Every
    // step shortens the makespan, so this ends; the bound only caps the work.
    for (int32_t step = 0; step < 4 * n_configs; ++step) {
        double cand_mk = best_mk;
        std::vector<int> cand;
        for (int32_t j = 0; j < n_sets; ++j) {
            for (int dg : {1, -1}) {
                const int g = best_g[j] + dg;
                if (g < 1 || g > (int)sets[j].size()) continue;
                std::vector<int> t = best_g;
                t[j] = g;
                const double mk = place(durations(t), cost->n_gpus, nullptr, nullptr);
                if (mk < cand_mk) {
                    cand_mk = mk;
                    cand = t;
                }
            }
        }
        if (cand.empty()) break;
        best_mk = cand_mk;
        best_g = cand;
    }

    // the kept plan: jobs in round order, a job's parts in part order
    std::vector<double> dur;
    std::vector<const Part *> parts;
    for (int32_t j = 0; j < n_sets; ++j)
        for (const Part &P : cuts[j][best_g[j] - 1]) {
            parts.push_back(&P);
            dur.push_back(P.dur);
        }
    std::vector<int32_t> gpu;
    std::vector<double> start;
    const double makespan = place(dur, cost->n_gpus, &gpu, &start);
    const int32_t nj = (int32_t)parts.size();
    for (int32_t j = 0; j < nj; ++j) {
        for (int c : parts[j]->m) job_of[c] = j;
        jobs[j].gpu = gpu[j];
        jobs[j].n_configs = (int32_t)parts[j]->m.size();
        jobs[j].start_s = start[j];
        jobs[j].duration_s = parts[j]->dur;
        jobs[j].step_s = parts[j]->step;
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
