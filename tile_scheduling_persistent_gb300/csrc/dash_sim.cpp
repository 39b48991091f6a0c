// dash_sim.cpp -- host-side DAG simulator of the DASH tile schedules.
//
// The model of "DASH: Deterministic Attention Scheduling for High-Throughput"
// (gist.science technical summary, section 2.1): every pair (KV tile j,
// Q tile i) is a compute node of cost c followed by a reduce node of cost r;
// the pairs of a task run back to back on one worker (a chain); the reduces
// into one dQ tile follow the accumulation order (a reduce may start only
// when its predecessor in that order has ended).  The critical path of this
// DAG is the makespan.  The visit lists and the worker assignment are the
// kernel's own (dash_schedule.h); the accumulation order is derived here
// independently (a sort by model time) so that it can be compared with the
// device-built rank tables.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <deque>
#include <vector>

#include "../../include/dash.h"
#include "dash_schedule.h"

namespace {

using dash::Shape;

struct Model {
    Shape s{};
    int P = 1;
    int64_t ntasks = 0;
    int64_t tiles = 0;
    std::vector<int64_t> task_off;   // task k -> first pair index
    std::vector<int64_t> tile;       // pair -> dQ tile
    std::vector<int> kv;             // pair -> KV tile
    std::vector<int64_t> entry;      // pair -> tile*n + kv
};

bool build(Model& m, int sched, int causal, int B, int Hq, int Hkv, int n, int P, int band = 0, int nk = 0) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || n <= 0 || P <= 0 || Hq % Hkv || sched < 0 || sched > 4 ||
        (causal != 0 && causal != 1) || band < 0 || (band && !causal) || nk < 0 || (nk && causal))
        return false;
    m.s = Shape{B, Hq, Hkv, n, Hq / Hkv, causal, sched, band, nk == n ? 0 : nk};
    const int nkv = dash::num_kv(m.s);
    m.P = P;
    m.ntasks = dash::num_tasks(m.s);
    m.tiles = (int64_t)B * Hq * n;
    m.task_off.resize(m.ntasks + 1);
    int64_t total = 0;
    for (int64_t k = 0; k < m.ntasks; ++k) {
        m.task_off[k] = total;
        total += dash::task_len(m.s, k);
    }
    m.task_off[m.ntasks] = total;
    m.tile.resize(total);
    m.kv.resize(total);
    m.entry.resize(total);
    for (int64_t k = 0; k < m.ntasks; ++k) {
        const int L = dash::task_len(m.s, k);
        for (int u = 0; u < L; ++u) {
            const dash::Visit v = dash::task_visit(m.s, k, u);
            const int64_t p = m.task_off[k] + u;
            m.tile[p] = ((int64_t)v.b * Hq + v.hq) * n + v.q;
            m.kv[p] = v.kv;
            m.entry[p] = m.tile[p] * nkv + v.kv;
        }
    }
    return true;
}

// Per-worker pair sequences of the static assignment (task k -> worker k % P).
std::vector<std::vector<int64_t>> static_sequences(const Model& m) {
    std::vector<std::vector<int64_t>> seq(m.P);
    for (int64_t k = 0; k < m.ntasks; ++k)
        for (int64_t p = m.task_off[k]; p < m.task_off[k + 1]; ++p) seq[k % m.P].push_back(p);
    return seq;
}

// order[tile] = pair indices in accumulation order.
std::vector<std::vector<int64_t>> accumulation_order(const Model& m) {
    std::vector<std::vector<int64_t>> order(m.tiles);
    const int sched = m.s.sched;
    if (sched == dash::kAtomic) return order;
    const int64_t npairs = (int64_t)m.tile.size();
    if (!dash::is_static(sched)) {
        for (int64_t p = 0; p < npairs; ++p) order[m.tile[p]].push_back(p);
        for (auto& o : order)
            std::sort(o.begin(), o.end(), [&](int64_t a, int64_t b) { return m.kv[a] < m.kv[b]; });
        return order;
    }
    std::vector<int64_t> t(npairs);
    for (auto& seq : static_sequences(m)) {
        int64_t clock = 0;
        for (int64_t p : seq) t[p] = clock++;
    }
    for (int64_t p = 0; p < npairs; ++p) order[m.tile[p]].push_back(p);
    for (auto& o : order)
        std::sort(o.begin(), o.end(), [&](int64_t a, int64_t b) {
            return t[a] != t[b] ? t[a] < t[b] : m.kv[a] < m.kv[b];
        });
    return order;
}

// Longest path over chains + accumulation edges; false on a cycle.
bool static_dag(const Model& m, const std::vector<std::vector<int64_t>>& seq,
                const std::vector<std::vector<int64_t>>& order, double c, double r, std::vector<double>& end) {
    const int64_t npairs = (int64_t)m.tile.size();
    std::vector<int64_t> chain_pred(npairs, -1), turn_pred(npairs, -1), chain_succ(npairs, -1),
        turn_succ(npairs, -1);
    for (const auto& s : seq)
        for (size_t i = 1; i < s.size(); ++i) {
            chain_pred[s[i]] = s[i - 1];
            chain_succ[s[i - 1]] = s[i];
        }
    for (const auto& o : order)
        for (size_t i = 1; i < o.size(); ++i) {
            turn_pred[o[i]] = o[i - 1];
            turn_succ[o[i - 1]] = o[i];
        }
    std::vector<int> indeg(npairs, 0);
    std::deque<int64_t> ready;
    for (int64_t p = 0; p < npairs; ++p) {
        indeg[p] = (chain_pred[p] >= 0) + (turn_pred[p] >= 0);
        if (!indeg[p]) ready.push_back(p);
    }
    end.assign(npairs, 0.0);
    int64_t done = 0;
    while (!ready.empty()) {
        const int64_t p = ready.front();
        ready.pop_front();
        ++done;
        const double cs = chain_pred[p] >= 0 ? end[chain_pred[p]] : 0.0;
        const double rf = turn_pred[p] >= 0 ? end[turn_pred[p]] : 0.0;
        end[p] = std::max(cs + c, rf) + r;
        for (int64_t q : {chain_succ[p], turn_succ[p]})
            if (q >= 0 && --indeg[q] == 0) ready.push_back(q);
    }
    return done == npairs;
}

// Greedy in-order dispatch: task k goes to the worker that is free first
// (lowest id on ties); accumulation predecessors must already be placed.
bool dynamic_sim(const Model& m, const std::vector<std::vector<int64_t>>& order, double c, double r,
                 std::vector<double>& end) {
    const int64_t npairs = (int64_t)m.tile.size();
    std::vector<int64_t> turn_pred(npairs, -1);
    for (const auto& o : order)
        for (size_t i = 1; i < o.size(); ++i) turn_pred[o[i]] = o[i - 1];
    end.assign(npairs, -1.0);
    std::vector<double> free(m.P, 0.0);
    for (int64_t k = 0; k < m.ntasks; ++k) {
        int w = 0;
        for (int x = 1; x < m.P; ++x)
            if (free[x] < free[w]) w = x;
        double t = free[w];
        for (int64_t p = m.task_off[k]; p < m.task_off[k + 1]; ++p) {
            double rs = t + c;
            if (turn_pred[p] >= 0) {
                if (end[turn_pred[p]] < 0) return false;
                rs = std::max(rs, end[turn_pred[p]]);
            }
            t = rs + r;
            end[p] = t;
        }
        free[w] = t;
    }
    return true;
}

}  // namespace

namespace {
int sim_impl(int schedule, int causal, int band, int B, int Hq, int Hkv, int n, int P, double c, double r,
             double* makespan, int32_t* turn_order, int64_t* num_tasks, int nk = 0) {
    Model m;
    try {
        if (!build(m, schedule, causal, B, Hq, Hkv, n, P, band, nk)) return DASH_ERR_ARG;
        const int nkv = dash::num_kv(m.s);
        auto order = accumulation_order(m);
        std::vector<double> end;
        bool ok;
        if (dash::is_static(schedule))
            ok = static_dag(m, static_sequences(m), order, c, r, end);
        else
            ok = dynamic_sim(m, order, c, r, end);
        if (!ok) return DASH_ERR_DEADLOCK;
        if (makespan) *makespan = end.empty() ? 0.0 : *std::max_element(end.begin(), end.end());
        if (num_tasks) *num_tasks = m.ntasks;
        if (turn_order) {
            if (schedule == dash::kAtomic) {
                order.assign(m.tiles, {});
                for (int64_t p = 0; p < (int64_t)m.tile.size(); ++p) order[m.tile[p]].push_back(p);
                for (auto& o : order)
                    std::sort(o.begin(), o.end(), [&](int64_t a, int64_t b) {
                        return end[a] != end[b] ? end[a] < end[b] : m.kv[a] < m.kv[b];
                    });
            }
            for (int64_t t = 0; t < m.tiles; ++t) {
                int32_t* row = turn_order + t * nkv;
                for (int i = 0; i < nkv; ++i) row[i] = -1;
                for (size_t i = 0; i < order[t].size(); ++i) row[i] = m.kv[order[t][i]];
            }
        }
    } catch (...) {
        return DASH_ERR_NOMEM;
    }
    return DASH_OK;
}
}  // namespace

extern "C" int dash_sim_schedule(int schedule, int causal, int B, int Hq, int Hkv, int n, int P, double c, double r,
                                 double* makespan, int32_t* turn_order, int64_t* num_tasks) {
    return sim_impl(schedule, causal, 0, B, Hq, Hkv, n, P, c, r, makespan, turn_order, num_tasks);
}

extern "C" int dash_sim_schedule_band(int schedule, int B, int Hq, int Hkv, int n, int band, int P, double c,
                                      double r, double* makespan, int32_t* turn_order, int64_t* num_tasks) {
    if (band < 1) return DASH_ERR_ARG;
    return sim_impl(schedule, 1, band, B, Hq, Hkv, n, P, c, r, makespan, turn_order, num_tasks);
}

extern "C" int dash_sim_schedule_cross(int schedule, int B, int Hq, int Hkv, int nq, int nkv, int P, double c,
                                       double r, double* makespan, int32_t* turn_order, int64_t* num_tasks) {
    if (nkv < 1) return DASH_ERR_ARG;
    return sim_impl(schedule, 0, 0, B, Hq, Hkv, nq, P, c, r, makespan, turn_order, num_tasks, nkv);
}

extern "C" int dash_sim_check_ranks(int schedule, int causal, int B, int Hq, int Hkv, int n, int P,
                                    const uint16_t* ranks) {
    if (!ranks || !dash::is_static(schedule)) return DASH_ERR_ARG;
    Model m;
    try {
        if (!build(m, schedule, causal, B, Hq, Hkv, n, P)) return DASH_ERR_ARG;
        std::vector<std::vector<int64_t>> order(m.tiles);
        for (int64_t p = 0; p < (int64_t)m.tile.size(); ++p) order[m.tile[p]].push_back(p);
        for (auto& o : order) {
            std::sort(o.begin(), o.end(), [&](int64_t a, int64_t b) { return ranks[m.entry[a]] < ranks[m.entry[b]]; });
            for (size_t i = 0; i < o.size(); ++i)
                if (ranks[m.entry[o[i]]] != i) return DASH_ERR_DEADLOCK;   // missing or repeated rank
        }
        std::vector<double> end;
        if (!static_dag(m, static_sequences(m), order, 1.0, 1.0, end)) return DASH_ERR_DEADLOCK;
    } catch (...) {
        return DASH_ERR_NOMEM;
    }
    return DASH_OK;
}
