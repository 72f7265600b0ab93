"""Pins for the brute-force schedule simulator: hand-built schedules whose
safety is known by inspection (classic deadlock, unordered writers, partial
joins, cross-step write-after-read, dead work, atomic accumulation)."""
from oracle import schedule_sim as S

R, W, A = S.READ, S.WRITE, S.ATOMIC


def T(sm, waits=(), signal=-1, acc=()):
    return {"sm": sm, "waits": list(waits), "signal": signal, "acc": list(acc)}


def IR(tasks, queues, n_counters, n_buffers=2, outputs=(1,)):
    return {"n_sms": len(queues), "n_counters": n_counters, "n_buffers": n_buffers,
            "outputs": list(outputs), "tasks": tasks, "queues": queues}


def producer_consumer(count=1, extra_order=False):
    # A writes buf0, signals c0; B waits c0 and reads buf0, writes the output buf1.
    tasks = [T(0, signal=0, acc=[(0, W, 0, 16, 0, 0)]),
             T(1, waits=[(0, count, 0)], signal=1, acc=[(0, R, 0, 16, 0, 0), (1, W, 0, 4, 0, 0)])]
    return IR(tasks, [[0], [1]], 2)


def test_single_step_producer_consumer_safe():
    ir = producer_consumer()
    assert not S.deadlocks(ir, 3)
    assert S.races(ir, epochs=1) == []


def test_cross_step_write_after_read_is_a_race():
    # The schedule repeats every step: A(e+1) rewrites buf0 while B(e) may still read it.
    ir = producer_consumer()
    safe, why = S.verdict(ir, epochs=2)
    assert not safe and why.startswith("race")
    assert ((0, 1), (1, 0)) in S.races(ir, epochs=2)


def test_cross_step_fix_with_back_edge():
    # B signals c1; A waits c1 from the previous step (epoch offset -1).
    tasks = [T(0, waits=[(1, 1, -1)], signal=0, acc=[(0, W, 0, 16, 0, 0)]),
             T(1, waits=[(0, 1, 0)], signal=1, acc=[(0, R, 0, 16, 0, 0), (1, W, 0, 4, 4, 0)])]
    ir = IR(tasks, [[0], [1]], 2)
    assert S.verdict(ir) == (True, "ok")


def test_classic_deadlock():
    tasks = [T(0, waits=[(1, 1, 0)], signal=0, acc=[(1, W, 0, 4, 0, 0)]),
             T(1, waits=[(0, 1, 0)], signal=1, acc=[(1, W, 4, 8, 0, 0)])]
    assert S.verdict(IR(tasks, [[0], [1]], 2)) == (False, "deadlock")


def test_threshold_above_producers_deadlocks():
    assert S.verdict(producer_consumer(count=2))[1] == "deadlock"


def test_queue_order_against_dependency_deadlocks():
    tasks = [T(0, signal=0, acc=[(0, W, 0, 16, 0, 0)]),
             T(0, waits=[(0, 1, 0)], signal=1, acc=[(0, R, 0, 16, 0, 0), (1, W, 0, 4, 0, 0)])]
    assert S.verdict(IR(tasks, [[0, 1]], 2))[0]
    assert S.verdict(IR(tasks, [[1, 0]], 2))[1] == "deadlock"


def test_unordered_writers_race():
    tasks = [T(0, signal=0, acc=[(1, W, 0, 8, 0, 0)]), T(1, signal=1, acc=[(1, W, 4, 12, 0, 0)])]
    safe, why = S.verdict(IR(tasks, [[0], [1]], 2))
    assert not safe and why.startswith("race")


def test_partial_join_races():
    # two producers write halves of buf0; the consumer waits for only one increment
    tasks = [T(0, signal=0, acc=[(0, W, 0, 8, 0, 0)]), T(1, signal=0, acc=[(0, W, 8, 16, 0, 0)]),
             T(2, waits=[(0, 1, 0)], acc=[(0, R, 0, 16, 0, 0), (1, W, 0, 4, 4, 0)])]
    ir = IR(tasks, [[0], [1], [2]], 1)
    safe, why = S.verdict(ir)
    assert not safe and why.startswith("race")
    # joining both producers fixes the step-local race; the next step's producers
    # still rewrite buf0 unordered with the reader, so a back edge is needed too
    tasks[2]["waits"] = [(0, 2, 0)]
    assert S.verdict(ir)[1].startswith("race")
    tasks[2]["signal"] = 1
    tasks[0]["waits"] = [(1, 1, -1)]
    tasks[1]["waits"] = [(1, 1, -1)]
    ir["n_counters"] = 2
    assert S.verdict(ir) == (True, "ok")


def test_dead_task_reported():
    tasks = [T(0, signal=0, acc=[(1, W, 0, 4, 4, 0)]), T(1, acc=[(0, W, 0, 4, 0, 0)])]
    safe, why = S.verdict(IR(tasks, [[0], [1]], 1))
    assert not safe and why == "dead task 1"


def test_atomics_commute_but_conflict_with_reads():
    tasks = [T(0, signal=0, acc=[(0, A, 0, 8, 0, 0)]), T(1, signal=0, acc=[(0, A, 0, 8, 0, 0)]),
             T(2, waits=[(0, 2, 0)], acc=[(0, R, 0, 8, 0, 0), (1, W, 0, 4, 4, 0)])]
    # within one step the two atomics may overlap; the reader is joined
    assert S.races(IR(tasks, [[0], [1], [2]], 1), epochs=1) == []
    # unjoined reader races with an atomic
    tasks[2]["waits"] = [(0, 1, 0)]
    assert S.races(IR(tasks, [[0], [1], [2]], 1), epochs=1) != []


def test_malformed_references():
    ir = producer_consumer()
    ir["tasks"][1]["waits"] = [(5, 1, 0)]
    assert S.verdict(ir)[1].startswith("malformed")
    ir = producer_consumer()
    ir["queues"] = [[0, 1], []]
    assert S.verdict(ir)[1].startswith("malformed")


# ---- tagged counters: the waiter polls the values it reads of the tagged buffer
def tagged_pair(waiter_reads=(0, 8)):
    # P1 writes buf0[0:8), P2 writes buf0[8:16); both "signal" tagged counter c0.
    # W reads buf0[waiter_reads] after a tagged wait on c0 (count 2) and writes
    # the output; P2 first waits for W through the ordinary counter c1.
    lo, hi = waiter_reads
    tasks = [T(0, signal=0, acc=[(0, W, 0, 8, 0, 0)]),
             T(1, waits=[(1, 1, 0)], signal=0, acc=[(0, W, 8, 16, 0, 0), (1, W, 4, 8, 0, 0)]),
             T(2, waits=[(0, 2, 0)], signal=1, acc=[(0, R, lo, hi, 0, 0), (1, W, 0, 4, 0, 0)])]
    ir = IR(tasks, [[0], [1], [2]], 2)
    ir["tagged"] = {0: 0}
    return ir


def test_tagged_wait_needs_only_the_overlapping_producers():
    # As a counter wait this is a cycle W -> P2 -> W; polling buf0[0:8) needs only P1.
    ir = tagged_pair()
    assert not S.deadlocks(ir, 1)
    plain = dict(ir, tagged={})
    assert S.deadlocks(plain, 1)


def test_tagged_wait_on_bytes_nobody_writes_deadlocks():
    # The poll of buf0[16:24) never sees its tag.
    ir = tagged_pair(waiter_reads=(16, 24))
    assert S.deadlocks(ir, 1)


def test_tagged_wait_orders_the_overlapping_producer():
    ir = tagged_pair()
    # W may not run before P1 has written what W reads: no (P1, W) race in one step
    assert ((0, 0), (2, 0)) not in S.races(ir, epochs=1)
