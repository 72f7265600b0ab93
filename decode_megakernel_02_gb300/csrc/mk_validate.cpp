// The static validator: the safety gate every lowered schedule passes before
// any launch.
//
// AutoMegaKernel explainer, "Methodology" ("The Safety Gate"): validate()
// certifies deadlock freedom (acyclic DAG, wait thresholds 1 <= t <=
// #producers, valid per-SM queue order), race freedom (joined multi-producer
// counters, happens-before on memory accesses) and correctness (output
// reachability, referential integrity), and a schedule that fails is
// rejected before it can reach the GPU.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <numeric>
#include <string>
#include <vector>

#include "mk_host.h"

namespace mk {

// ------------------------------------------------------------------ validator
namespace {

constexpr int EPOCHS = 3;  // unrolled steps for happens-before and races

struct Fail {
    std::string* why;
    mk_status operator()(const std::string& s) {
        if (why) *why = s;
        return MK_ERR_SCHEDULE_INVALID;
    }
};

}  // namespace

mk_status validate_ir(const mk_ir* ir, std::string* why) {
    Fail fail{why};
    if (!ir) return fail("IR is NULL");
    const int T = ir->n_tasks, NC = ir->n_counters, NB = ir->n_buffers, S = ir->n_sms;
    if (T < 1 || NC < 0 || NB < 1 || S < 1 || ir->n_acc < 0) return fail("empty or negative IR sizes");
    if (!ir->tasks || !ir->queue || !ir->queue_off || (ir->n_acc && !ir->acc)) return fail("NULL IR array");

    // ---- well formed: queues, ids, ranges
    if (ir->queue_off[0] != 0 || ir->queue_off[S] != T) return fail("queues do not hold every task once");
    std::vector<int> qcount(T, 0), seqpos(T, -1), qlen(S);
    for (int s = 0; s < S; ++s) {
        if (ir->queue_off[s + 1] < ir->queue_off[s]) return fail("queue offsets decrease");
        qlen[s] = ir->queue_off[s + 1] - ir->queue_off[s];
        for (int i = ir->queue_off[s]; i < ir->queue_off[s + 1]; ++i) {
            int t = ir->queue[i];
            if (t < 0 || t >= T) return fail("queue of SM " + std::to_string(s) + " names task " + std::to_string(t));
            if (ir->tasks[t].sm != s)
                return fail("task " + std::to_string(t) + " queued on SM " + std::to_string(s) +
                            " but placed on SM " + std::to_string(ir->tasks[t].sm));
            qcount[t]++;
            seqpos[t] = i - ir->queue_off[s];
        }
    }
    for (int t = 0; t < T; ++t)
        if (qcount[t] != 1) return fail("task " + std::to_string(t) + " queued " + std::to_string(qcount[t]) + " times");
    // tagged counters (ctr_buf may be NULL: none)
    std::vector<int> tbuf(NC, -1), tset(NB, -1);  // counter -> buffer; buffer -> clock set
    int n_sets = 1;                                // set 0: happens-before without tagged waits
    for (int c = 0; c < NC && ir->ctr_buf; ++c) {
        const int b = ir->ctr_buf[c];
        if (b < -1 || b >= NB) return fail("counter " + std::to_string(c) + " names missing buffer " + std::to_string(b));
        tbuf[c] = b;
        if (b >= 0 && tset[b] < 0) tset[b] = n_sets++;
    }
    std::vector<int> nprod(NC, 0);
    for (int t = 0; t < T; ++t) {
        const mk_ir_task& k = ir->tasks[t];
        if (k.n_waits < 0 || k.n_waits > MK_IR_MAX_WAITS) return fail("task " + std::to_string(t) + " has bad n_waits");
        for (int w = 0; w < k.n_waits; ++w)
            if (k.wait_ctr[w] < 0 || k.wait_ctr[w] >= NC)
                return fail("task " + std::to_string(t) + " waits on missing counter " + std::to_string(k.wait_ctr[w]));
        if (k.signal_ctr != -1 && (k.signal_ctr < 0 || k.signal_ctr >= NC))
            return fail("task " + std::to_string(t) + " signals missing counter " + std::to_string(k.signal_ctr));
        if (k.signal_ctr >= 0) nprod[k.signal_ctr]++;
        if (k.n_acc < 0 || k.acc_begin < 0 || k.acc_begin + k.n_acc > ir->n_acc)
            return fail("task " + std::to_string(t) + " has a dangling access list");
        for (int a = k.acc_begin; a < k.acc_begin + k.n_acc; ++a) {
            const mk_ir_access& x = ir->acc[a];
            if (x.buf < 0 || x.buf >= NB) return fail("task " + std::to_string(t) + " touches missing buffer");
            if (x.kind < MK_ACC_READ || x.kind > MK_ACC_ATOMIC) return fail("task " + std::to_string(t) + " has a bad access kind");
            if (x.hi < x.lo || x.lo < 0 || x.grow < 0) return fail("task " + std::to_string(t) + " has a bad byte range");
        }
    }

    // ---- deadlock: satisfiable thresholds.  race: joined counters.
    for (int t = 0; t < T; ++t) {
        const mk_ir_task& k = ir->tasks[t];
        for (int w = 0; w < k.n_waits; ++w) {
            int c = k.wait_ctr[w], cnt = k.wait_count[w], off = k.wait_epoch_off[w];
            if (off != 0 && off != -1)
                return fail("task " + std::to_string(t) + " waits with epoch offset " + std::to_string(off));
            if (cnt < 1 || cnt > nprod[c])
                return fail("deadlock: task " + std::to_string(t) + " waits for " + std::to_string(cnt) +
                            " signals on counter " + std::to_string(c) + " which has " +
                            std::to_string(nprod[c]) + " producers (need 1 <= t <= #producers)");
            if (cnt != nprod[c])
                return fail("race: task " + std::to_string(t) + " waits for " + std::to_string(cnt) + " of " +
                            std::to_string(nprod[c]) + " producers of counter " + std::to_string(c) +
                            " (multi-producer counters must be joined)");
        }
    }

    // ---- unrolled happens-before graph: nodes are task instances (t, e) and
    //      counter instances (c, e); edges: queue order, producer -> counter,
    //      counter(e + off) -> waiting task(e).
    const int NT_ = T * EPOCHS, NCN = NC * EPOCHS, N = NT_ + NCN;
    auto tn = [&](int t, int e) { return e * T + t; };
    auto cn = [&](int c, int e) { return NT_ + e * NC + c; };
    std::vector<std::vector<int>> prodlist(NC);
    for (int t = 0; t < T; ++t)
        if (ir->tasks[t].signal_ctr >= 0) prodlist[ir->tasks[t].signal_ctr].push_back(t);
    std::vector<int> indeg(N, 0);
    std::vector<std::vector<int>> out(N);
    // in-edges with the clock sets they count in: -1 all, -2 none, k >= 1 set k only
    std::vector<std::vector<std::pair<int, int>>> in(N);
    auto edge = [&](int a, int b, int set = -1) {
        out[a].push_back(b);
        indeg[b]++;
        in[b].push_back({a, set});
    };
    for (int s = 0; s < S; ++s) {
        int prevn = -1;
        for (int e = 0; e < EPOCHS; ++e)
            for (int i = ir->queue_off[s]; i < ir->queue_off[s + 1]; ++i) {
                int n = tn(ir->queue[i], e);
                if (prevn >= 0) edge(prevn, n);
                prevn = n;
            }
    }
    for (int e = 0; e < EPOCHS; ++e)
        for (int t = 0; t < T; ++t) {
            const mk_ir_task& k = ir->tasks[t];
            if (k.signal_ctr >= 0) edge(tn(t, e), cn(k.signal_ctr, e));
            for (int w = 0; w < k.n_waits; ++w) {
                int ee = e + k.wait_epoch_off[w];
                if (ee >= 0) edge(cn(k.wait_ctr[w], ee), tn(t, e), tbuf[k.wait_ctr[w]] >= 0 ? -2 : -1);
            }
        }
    // Kahn order; a leftover node means a cycle: some wait can never be met.
    std::vector<int> order;
    order.reserve(N);
    {
        std::vector<int> deg = indeg, stack;
        for (int n = 0; n < N; ++n)
            if (!deg[n]) stack.push_back(n);
        while (!stack.empty()) {
            int n = stack.back();
            stack.pop_back();
            order.push_back(n);
            for (int m : out[n])
                if (--deg[m] == 0) stack.push_back(m);
        }
        if ((int)order.size() != N) {
            for (int n = 0; n < NT_; ++n)
                if (deg[n]) {
                    int t = n % T;
                    return fail("deadlock: the dependency graph with per-SM queue order has a cycle "
                                "through task " + std::to_string(t) + " (SM " +
                                std::to_string(ir->tasks[t].sm) + ", queue slot " + std::to_string(seqpos[t]) + ")");
                }
            return fail("deadlock: cycle among counters");
        }
    }
    // A wait on a tagged counter orders the waiting task only after the
    // producers' writes of the tagged buffer that it reads: every byte of the
    // buffer it reads must be written by those producers in the waited step,
    // and it gets a happens-before edge from exactly the producers whose
    // writes overlap its reads (counted only for accesses to that buffer).
    auto range_at = [](const mk_ir_access& x, int e) {
        return std::make_pair(x.lo + e * x.stride, x.hi + e * x.stride + e * x.grow);
    };
    for (int t = 0; t < T; ++t) {
        const mk_ir_task& k = ir->tasks[t];
        for (int w = 0; w < k.n_waits; ++w) {
            const int c = k.wait_ctr[w], b = tbuf[c], off = k.wait_epoch_off[w];
            if (b < 0) continue;
            if (off != 0)  // the poll looks for the running step's tag
                return fail("tagged wait: task " + std::to_string(t) + " waits on counter " + std::to_string(c) +
                            " of an earlier step; tagged values carry only the running step");
            for (int e = 0; e < EPOCHS; ++e) {
                const int ee = e + off;
                if (ee < 0) continue;
                std::vector<std::pair<int64_t, int64_t>> wr;  // producers' writes of b at step ee
                for (int p : prodlist[c]) {
                    const mk_ir_task& pk = ir->tasks[p];
                    bool linked = false;
                    for (int a = pk.acc_begin; a < pk.acc_begin + pk.n_acc; ++a) {
                        const mk_ir_access& y = ir->acc[a];
                        if (y.buf != b || y.kind == MK_ACC_READ) continue;
                        const auto ry = range_at(y, ee);
                        if (ry.second <= ry.first) continue;
                        wr.push_back(ry);
                        for (int a2 = k.acc_begin; a2 < k.acc_begin + k.n_acc && !linked; ++a2) {
                            const mk_ir_access& x = ir->acc[a2];
                            const auto rx = range_at(x, e);
                            if (x.buf == b && rx.first < ry.second && ry.first < rx.second) linked = true;
                        }
                    }
                    if (linked) in[tn(t, e)].push_back({tn(p, ee), tset[b]});
                }
                std::sort(wr.begin(), wr.end());
                for (int a = k.acc_begin; a < k.acc_begin + k.n_acc; ++a) {
                    const mk_ir_access& x = ir->acc[a];
                    if (x.buf != b) continue;
                    const auto rx = range_at(x, e);
                    int64_t at = rx.first;  // first byte not yet covered
                    for (const auto& y : wr)
                        if (y.first <= at) at = std::max(at, y.second);
                    if (at < rx.second)
                        return fail("tagged wait: task " + std::to_string(t) + " reads bytes [" + std::to_string(at) +
                                    ", " + std::to_string(rx.second) + ") of buffer " + std::to_string(b) +
                                    " that no producer of counter " + std::to_string(c) + " writes in that step");
                }
            }
        }
    }
    // Vector clocks: vcs[k][n][s] = last queue index on SM s that happens
    // before n in clock set k.  Set 0 leaves out tagged waits; set tset[b]
    // adds the producer edges of the tagged waits on buffer b.  Those edges
    // run parallel to producer -> counter -> waiter paths of the graph, so
    // Kahn's order is still a topological order.
    auto seq = [&](int t, int e) { return e * qlen[ir->tasks[t].sm] + seqpos[t]; };
    std::vector<std::vector<int32_t>> vcs(n_sets, std::vector<int32_t>((size_t)N * S, -1));
    for (int set = 0; set < n_sets; ++set) {
        std::vector<int32_t>& vc = vcs[set];
        for (int n : order) {
            int32_t* v = &vc[(size_t)n * S];
            for (const auto& pe : in[n]) {
                if (pe.second == -2 || (pe.second >= 0 && pe.second != set)) continue;
                const int32_t* pv = &vc[(size_t)pe.first * S];
                for (int s = 0; s < S; ++s) v[s] = std::max(v[s], pv[s]);
            }
            if (n < NT_) {
                int t = n % T, e = n / T;
                v[ir->tasks[t].sm] = std::max(v[ir->tasks[t].sm], seq(t, e));
            }
        }
    }
    const std::vector<int32_t>& vc0 = vcs[0];
    auto hb = [&](int ta, int ea, int tb, int eb) {  // (ta,ea) happens before (tb,eb) without tagged waits
        return vc0[(size_t)tn(tb, eb) * S + ir->tasks[ta].sm] >= seq(ta, ea);
    };

    // ---- counter reuse across steps: a wait at step e must not be satisfiable
    //      by increments of step e + off + 1, so every producer's next
    //      increment must come after the waiting task.
    for (int t = 0; t < T; ++t) {
        const mk_ir_task& k = ir->tasks[t];
        for (int w = 0; w < k.n_waits; ++w) {
            int c = k.wait_ctr[w], off = k.wait_epoch_off[w];
            if (tbuf[c] >= 0) continue;  // no counter word: reusing a tag is a race on the buffer, checked below
            for (int p : prodlist[c])
                if (!hb(t, 1, p, 2 + off))
                    return fail("race: counter " + std::to_string(c) + " is reused by step e+1 of producer task " +
                                std::to_string(p) + " before waiting task " + std::to_string(t) + " of step e");
        }
    }

    // ---- memory races over the unrolled steps.  For an access X and an SM s,
    //      the accesses on s that X does not order form one run in queue order:
    //      they start after vc[X][s] (everything up to there happens before X)
    //      and end at the first access Y with vc[Y][sm(X)] >= seq(X) (vc is
    //      monotone along a queue, so every later access on s comes after X).
    struct Inst {
        int32_t seq, t, e, kind;
        int64_t lo, hi;
    };
    std::vector<std::vector<std::vector<Inst>>> on(NB, std::vector<std::vector<Inst>>(S));
    for (int e = 0; e < EPOCHS; ++e)
        for (int t = 0; t < T; ++t) {
            const mk_ir_task& k = ir->tasks[t];
            for (int a = k.acc_begin; a < k.acc_begin + k.n_acc; ++a) {
                const mk_ir_access& x = ir->acc[a];
                int64_t lo = x.lo + e * x.stride, hi = x.hi + e * x.stride + e * x.grow;
                if (hi > lo) on[x.buf][k.sm].push_back({seq(t, e), t, e, x.kind, lo, hi});
            }
        }
    for (int b = 0; b < NB; ++b)
        for (int s = 0; s < S; ++s)
            std::stable_sort(on[b][s].begin(), on[b][s].end(), [](const Inst& x, const Inst& y) { return x.seq < y.seq; });
    // Per instance X with a write or atomic access: its non-read ranges, sorted
    // by start with a running maximum of their ends, answer "does range y
    // conflict with X" by binary search.  Atomic ranges are kept apart, since
    // an atomic y conflicts only with X's plain writes.
    struct Rng {
        int64_t lo, hi;
    };
    auto prep = [](std::vector<Rng>& v, std::vector<int64_t>& pm) {
        std::sort(v.begin(), v.end(), [](const Rng& x, const Rng& y) { return x.lo < y.lo; });
        pm.resize(v.size());
        int64_t m = INT64_MIN;
        for (size_t k = 0; k < v.size(); ++k) pm[k] = m = std::max(m, v[k].hi);
    };
    auto hits = [](const std::vector<Rng>& v, const std::vector<int64_t>& pm, int64_t lo, int64_t hi) -> int {
        // index of a range of v overlapping [lo, hi), or -1
        size_t n = std::lower_bound(v.begin(), v.end(), hi, [](const Rng& x, int64_t h) { return x.lo < h; }) - v.begin();
        if (n == 0 || pm[n - 1] <= lo) return -1;
        for (size_t k = n; k-- > 0;)
            if (v[k].hi > lo) return (int)k;
        return -1;
    };
    std::vector<Rng> xw, xa;  // X's plain-write and atomic ranges
    std::vector<int64_t> pw, pa;
    for (int b = 0; b < NB; ++b) {
        const std::vector<int32_t>& vc = vcs[tset[b] > 0 ? tset[b] : 0];
        for (int sx = 0; sx < S; ++sx) {
            const auto& lx = on[b][sx];
            for (size_t i = 0; i < lx.size();) {
                size_t j = i;
                xw.clear();
                xa.clear();
                for (; j < lx.size() && lx[j].seq == lx[i].seq; ++j) {  // one instance: [i, j)
                    if (lx[j].kind == MK_ACC_WRITE) xw.push_back({lx[j].lo, lx[j].hi});
                    if (lx[j].kind == MK_ACC_ATOMIC) xa.push_back({lx[j].lo, lx[j].hi});
                }
                const Inst& x = lx[i];
                i = j;
                if (xw.empty() && xa.empty()) continue;  // every conflicting pair has a write or atomic side
                prep(xw, pw);
                prep(xa, pa);
                const int32_t* vx = &vc[(size_t)tn(x.t, x.e) * S];
                for (int s = 0; s < S; ++s) {
                    const auto& list = on[b][s];
                    auto it = std::upper_bound(list.begin(), list.end(), vx[s],
                                               [](int32_t v, const Inst& y) { return v < y.seq; });
                    int32_t yseq = -1;
                    for (; it != list.end(); ++it) {
                        const Inst& y = *it;
                        if (y.seq != yseq) {  // the ordering test holds for every access of an instance
                            yseq = y.seq;
                            if (vc[(size_t)tn(y.t, y.e) * S + sx] >= x.seq) break;  // y comes after x
                        }
                        if (y.t == x.t && y.e == x.e) continue;
                        int k = hits(xw, pw, y.lo, y.hi);
                        const Rng* r = k >= 0 ? &xw[k] : nullptr;
                        if (!r && y.kind != MK_ACC_ATOMIC) {
                            k = hits(xa, pa, y.lo, y.hi);
                            r = k >= 0 ? &xa[k] : nullptr;
                        }
                        if (!r) continue;
                        return fail("race: task " + std::to_string(x.t) + " (step " + std::to_string(x.e) +
                                    ") and task " + std::to_string(y.t) + " (step " + std::to_string(y.e) +
                                    ") touch buffer " + std::to_string(b) + " bytes [" +
                                    std::to_string(std::max(r->lo, y.lo)) + ", " + std::to_string(std::min(r->hi, y.hi)) +
                                    ") without happens-before");
                    }
                }
            }
        }
    }

    // ---- correctness: every task's writes reach an output (two steps).
    //      Fixpoint over "useful" instances; each round merges the byte ranges
    //      useful instances read and looks writes up by binary search.
    {
        const int E2 = 2;
        std::vector<char> useful((size_t)T * E2, 0);
        bool changed = true;
        while (changed) {
            changed = false;
            std::vector<std::vector<std::pair<int64_t, int64_t>>> rr(NB);
            for (int e = 0; e < E2; ++e)
                for (int t = 0; t < T; ++t) {
                    if (!useful[(size_t)e * T + t]) continue;
                    const mk_ir_task& k = ir->tasks[t];
                    for (int a = k.acc_begin; a < k.acc_begin + k.n_acc; ++a) {
                        const mk_ir_access& x = ir->acc[a];
                        if (x.kind == MK_ACC_WRITE) continue;
                        int64_t lo = x.lo + e * x.stride, hi = x.hi + e * x.stride + e * x.grow;
                        if (hi > lo) rr[x.buf].push_back({lo, hi});
                    }
                }
            for (auto& v : rr) {  // merge into disjoint sorted intervals
                std::sort(v.begin(), v.end());
                std::vector<std::pair<int64_t, int64_t>> m;
                for (auto& r : v) {
                    if (!m.empty() && r.first <= m.back().second) m.back().second = std::max(m.back().second, r.second);
                    else m.push_back(r);
                }
                v.swap(m);
            }
            for (int e = 0; e < E2; ++e)
                for (int t = 0; t < T; ++t) {
                    char& u = useful[(size_t)e * T + t];
                    if (u) continue;
                    const mk_ir_task& k = ir->tasks[t];
                    for (int a = k.acc_begin; a < k.acc_begin + k.n_acc && !u; ++a) {
                        const mk_ir_access& x = ir->acc[a];
                        if (x.kind == MK_ACC_READ) continue;
                        int64_t lo = x.lo + e * x.stride, hi = x.hi + e * x.stride + e * x.grow;
                        if (hi <= lo) continue;
                        if (ir->buf_flags && (ir->buf_flags[x.buf] & MK_BUF_OUTPUT)) {
                            u = 1;
                            break;
                        }
                        const auto& m = rr[x.buf];
                        auto it = std::upper_bound(m.begin(), m.end(), std::make_pair(lo, INT64_MAX));
                        if (it != m.begin() && std::prev(it)->second > lo) u = 1;  // interval starting <= lo
                        if (it != m.end() && it->first < hi) u = 1;                // interval starting in (lo, hi)
                    }
                    if (u) changed = true;
                }
        }
        for (int t = 0; t < T; ++t)
            if (!useful[t] && !useful[(size_t)T + t])
                return fail("dead task " + std::to_string(t) + ": its writes never reach an output");
    }
    return MK_OK;
}

}  // namespace mk

using namespace mk;

extern "C" {

mk_status mk_validate_ir(const mk_ir* ir, char* why, size_t why_len) {
    std::string w;
    mk_status st = validate_ir(ir, &w);
    if (st) set_error("%s", w.c_str());
    if (why && why_len) {
        std::snprintf(why, why_len, "%s", st ? w.c_str() : "ok");
    }
    return st;
}

mk_status mk_validate_schedule(const mk_model_desc* desc, const mk_schedule_config* cfg,
                               int32_t n_sms, char* why, size_t why_len) {
    mk_ir* ir = nullptr;
    mk_status st = mk_build_ir(desc, cfg, n_sms, &ir);
    if (st) {
        if (why && why_len) std::snprintf(why, why_len, "%s", thread_error());
        return st;
    }
    st = mk_validate_ir(ir, why, why_len);
    mk_free_ir(ir);
    return st;
}

}  // extern "C"
