"""Brute-force execution model of a task schedule (ground truth for the validator).

The AutoMegaKernel explainer ("Methodology", Layer 0 and the safety gate)
describes the device as one persistent CTA per SM, each walking its own queue
in order: wait (counter >= threshold) -> run -> signal (counter += 1), with
monotonic counters, and a static validator that must reject a schedule that
can deadlock (cyclic DAG, unsatisfiable threshold 1 <= t <= #producers,
invalid per-SM queue order) or race (un-joined multi-producer counters,
memory accesses without happens-before), or that is incorrect (dangling
references, work that never reaches an output).

This module decides those properties by executing the model, not by the
validator's graph reasoning:

* deadlock: one greedy run over ``epochs`` repetitions of every queue.  Counters
  only grow, so enabling is monotone and any maximal run finishes the same set
  of task instances; the schedule deadlocks iff that set is incomplete.
* races: every reachable state (per SM: queue position and waiting/running) is
  enumerated; two instances race when some reachable state has both running
  while their memory accesses conflict (same buffer, overlapping byte ranges,
  at least one write, not both atomic).
* usefulness: an instance is useful if it writes an output buffer or writes
  bytes that a useful instance reads; a task none of whose instances is useful
  is dead.

Wait semantics at epoch e: (counter c, count t, epoch offset o) passes once
c >= t * (e + 1 + o); a threshold <= 0 passes at once.  Access ranges at epoch
e are [lo + e*stride, hi + e*stride + e*grow).

Tagged counters ("tagged": {counter: buffer}) have no memory word: the
producers' writes of the buffer carry the step's tag and the waiting task
polls the bytes of that buffer it reads.  Such a wait passes once every
producer instance (step e + o) whose writes of the buffer overlap the task's
reads of it has finished, and never if some byte it reads is written by no
producer in that step (the poll would spin forever).  This model keeps
memory sequentially consistent, so it cannot see that such a wait orders
nothing but the tagged buffer; the library's validator checks that part.

IR (plain dicts, the same fields the library exports):
  {"n_sms", "n_counters", "n_buffers", "outputs": [buf ids], "tagged" (optional),
   "tasks": [{"sm", "waits": [(c, t, o)], "signal": c or -1,
              "acc": [(buf, kind, lo, hi, stride, grow)]}],
   "queues": [[task ids of SM 0 in order], ...]}
kind: 1 read, 2 write, 3 atomic.
"""
from collections import deque

READ, WRITE, ATOMIC = 1, 2, 3


def malformed(ir):
    """Referential integrity; returns a reason string or None."""
    n_t, n_c, n_b, n_s = len(ir["tasks"]), ir["n_counters"], ir["n_buffers"], ir["n_sms"]
    if len(ir["queues"]) != n_s:
        return "queue count != n_sms"
    seen = [0] * n_t
    for s, q in enumerate(ir["queues"]):
        for t in q:
            if not (0 <= t < n_t):
                return f"queue {s} names task {t}"
            if ir["tasks"][t]["sm"] != s:
                return f"task {t} queued on SM {s} but placed on {ir['tasks'][t]['sm']}"
            seen[t] += 1
    for t, k in enumerate(seen):
        if k != 1:
            return f"task {t} queued {k} times"
    for c, b in ir.get("tagged", {}).items():
        if not (0 <= c < n_c) or not (0 <= b < n_b):
            return f"tagged counter {c} -> buffer {b}"
    for i, t in enumerate(ir["tasks"]):
        for (c, cnt, o) in t["waits"]:
            if not (0 <= c < n_c):
                return f"task {i} waits on counter {c}"
        if t["signal"] != -1 and not (0 <= t["signal"] < n_c):
            return f"task {i} signals counter {t['signal']}"
        for a in t["acc"]:
            if not (0 <= a[0] < n_b) or a[1] not in (READ, WRITE, ATOMIC) or a[3] < a[2]:
                return f"task {i} bad access {a}"
    return None


def _instances(ir, epochs):
    seqs = []
    for q in ir["queues"]:
        seqs.append([(t, e) for e in range(epochs) for t in q])
    return seqs


def _tag_sources(ir, t, e, c, o, cache):
    """Producer instances a tagged wait of task t at epoch e depends on, or
    None when some byte it reads of the tagged buffer has no producer."""
    key = (t, e, c, o)
    if key not in cache:
        b, ee = ir["tagged"][c], e + o
        reads = [_ranges(x, e)[2:] for x in ir["tasks"][t]["acc"] if x[0] == b]
        writes, srcs = [], []
        for p, task in enumerate(ir["tasks"]):
            if task["signal"] != c or ee < 0:
                continue
            w = [_ranges(y, ee)[2:] for y in task["acc"] if y[0] == b and y[1] != READ]
            w = [r for r in w if r[1] > r[0]]
            writes += w
            if any(lo < hy and ly < hi for (lo, hi) in reads for (ly, hy) in w):
                srcs.append((p, ee))
        covered = all(all(any(ly <= k < hy for (ly, hy) in writes) for k in range(lo, hi)) for (lo, hi) in reads)
        cache[key] = srcs if covered else None
    return cache[key]


def _ready(ir, ctr, t, e, done=None, cache=None):
    tagged = ir.get("tagged", {})
    for (c, cnt, o) in ir["tasks"][t]["waits"]:
        if c in tagged:
            srcs = _tag_sources(ir, t, e, c, o, cache)
            if srcs is None or not all(done(p, ee) for (p, ee) in srcs):
                return False
        elif ctr[c] < cnt * (e + 1 + o):
            return False
    return True


def _index(ir):
    """Task -> (SM, position in its queue, queue length)."""
    where = {}
    for s, q in enumerate(ir["queues"]):
        for i, t in enumerate(q):
            where[t] = (s, i, len(q))
    return where


def deadlocks(ir, epochs=3):
    """True iff a greedy run of ``epochs`` repetitions cannot finish every instance."""
    seqs = _instances(ir, epochs)
    pos = [0] * len(seqs)
    ctr = [0] * ir["n_counters"]
    where, cache = _index(ir), {}

    def done(p, ee):
        s, i, n = where[p]
        return pos[s] > ee * n + i

    progress = True
    while progress:
        progress = False
        for s, seq in enumerate(seqs):
            while pos[s] < len(seq):
                t, e = seq[pos[s]]
                if not _ready(ir, ctr, t, e, done, cache):
                    break
                sig = ir["tasks"][t]["signal"]
                if sig >= 0:
                    ctr[sig] += 1
                pos[s] += 1
                progress = True
    return any(pos[s] < len(seqs[s]) for s in range(len(seqs)))


def _ranges(acc, e):
    buf, kind, lo, hi, stride, grow = acc
    return buf, kind, lo + e * stride, hi + e * stride + e * grow


def conflict(ir, a, b):
    """Do instances a=(t,e) and b=(t2,e2) touch a common byte with a write?"""
    for x in ir["tasks"][a[0]]["acc"]:
        bx, kx, lx, hx = _ranges(x, a[1])
        for y in ir["tasks"][b[0]]["acc"]:
            by, ky, ly, hy = _ranges(y, b[1])
            if bx != by or lx >= hy or ly >= hx or lx == hx or ly == hy:
                continue
            if kx == READ and ky == READ:
                continue
            if kx == ATOMIC and ky == ATOMIC:
                continue
            return True
    return False


def races(ir, epochs=2, max_states=2_000_000):
    """All racing instance pairs found by exhaustive exploration.

    State: per SM (index into its unrolled sequence, running flag).  Counter
    values follow from the finished prefix of every sequence."""
    seqs = _instances(ir, epochs)
    n = len(seqs)
    sig_of = [t["signal"] for t in ir["tasks"]]

    def counters(state):
        ctr = [0] * ir["n_counters"]
        for s in range(n):
            for (t, e) in seqs[s][: state[s][0]]:
                if sig_of[t] >= 0:
                    ctr[sig_of[t]] += 1
        return ctr

    where, cache = _index(ir), {}
    start = tuple((0, 0) for _ in range(n))
    seen = {start}
    dq = deque([start])
    found = set()
    conf_cache = {}
    while dq:
        st = dq.popleft()
        running = [seqs[s][st[s][0]] for s in range(n) if st[s][1] == 1]
        for i in range(len(running)):
            for j in range(i + 1, len(running)):
                key = (running[i], running[j])
                if key not in conf_cache:
                    conf_cache[key] = conflict(ir, running[i], running[j])
                if conf_cache[key]:
                    found.add(tuple(sorted(key)))
        ctr = None
        for s in range(n):
            idx, run = st[s]
            if idx >= len(seqs[s]):
                continue
            if run:
                nxt = list(st)
                nxt[s] = (idx + 1, 0)
            else:
                if ctr is None:
                    ctr = counters(st)
                t, e = seqs[s][idx]

                def done(p, ee, st=st):
                    sp, i, m = where[p]
                    return st[sp][0] > ee * m + i

                if not _ready(ir, ctr, t, e, done, cache):
                    continue
                nxt = list(st)
                nxt[s] = (idx, 1)
            nxt = tuple(nxt)
            if nxt not in seen:
                if len(seen) >= max_states:
                    raise RuntimeError("state space too large for brute force")
                seen.add(nxt)
                dq.append(nxt)
    return sorted(found)


def dead_tasks(ir, epochs=2):
    """Tasks none of whose instances (within ``epochs``) reaches an output."""
    outs = set(ir.get("outputs", []))
    inst = [(t, e) for e in range(epochs) for t in range(len(ir["tasks"]))]
    useful = set()
    changed = True
    while changed:
        changed = False
        for a in inst:
            if a in useful:
                continue
            ok = False
            for x in ir["tasks"][a[0]]["acc"]:
                bx, kx, lx, hx = _ranges(x, a[1])
                if kx == READ or hx <= lx:
                    continue
                if bx in outs:
                    ok = True
                    break
                for b in useful:
                    for y in ir["tasks"][b[0]]["acc"]:
                        by, ky, ly, hy = _ranges(y, b[1])
                        if by == bx and ky in (READ, ATOMIC) and ly < hx and lx < hy:
                            ok = True
                            break
                    if ok:
                        break
                if ok:
                    break
            if ok:
                useful.add(a)
                changed = True
    return sorted({t for t in range(len(ir["tasks"])) if all((t, e) not in useful for e in range(epochs))})


def verdict(ir, epochs=2):
    """Ground truth: (safe: bool, reason: str)."""
    m = malformed(ir)
    if m:
        return False, "malformed: " + m
    if deadlocks(ir, epochs + 1):
        return False, "deadlock"
    r = races(ir, epochs)
    if r:
        return False, f"race: {r[0]}"
    d = dead_tasks(ir, epochs)
    if d:
        return False, f"dead task {d[0]}"
    return True, "ok"
