"""Pins for the DAG oracle (oracle/dag.py) against what the pages and the model fix.

* the closed-form makespans of tests/golden/dag_closed_forms.txt (pages' formulas and
  ones derived from the chain recurrence), evaluated here from the formula text;
* the referee's worked counterexample (n = 2, m = 1, causal);
* Lemma 1 by brute force on random parallel isomorphic chains;
* coverage, per-KV contiguity and conflict-freedom of the task orders;
* a textbook longest-path example and cycle detection.
"""

import itertools
import os
import random

import pytest

from oracle.dag import SCHEDULES, chains, longest_path, reduction_order, simulate

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dag_closed_forms.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or line.startswith("EXAMPLE"):
                continue
            mask, sched, _p, m, formula, src = (x.strip() for x in line.split("|"))
            rows.append((mask, sched, m, formula, src))
    return rows


def _valid(mask, sched, n):
    if sched == "shift" and mask != "full":
        return False
    if sched == "symmetric_shift" and (mask != "causal" or n % 2):
        return False
    return True


def test_longest_path_textbook():
    # a -> b (3), a -> c (2), b -> d (4), c -> d (6), d -> e (1): longest to e = 9 via a-c-d-e
    depth = longest_path(5, [(0, 1, 3), (0, 2, 2), (1, 3, 4), (2, 3, 6), (3, 4, 1)])
    assert depth == [0, 3, 2, 8, 9]
    assert longest_path(3, [(0, 1, 1), (1, 2, 1), (2, 0, 1)]) is None


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"{r[0]}-{r[1]}-m{r[2]}")
@pytest.mark.parametrize("c,r", [(3, 1), (5, 2), (1, 4)])
def test_closed_forms(row, c, r):
    mask, sched, m_spec, formula, _src = row
    for n in range(1, 17):
        if not _valid(mask, sched, n):
            continue
        for m in ([1] if m_spec == "1" else [1, 2, 3, 4]):
            got = simulate(mask, sched, n, m, n, c, r)["makespan"]
            want = eval(formula, {}, {"n": n, "m": m, "c": c, "r": r})
            assert got == want, (mask, sched, n, m, c, r, got, want)


@pytest.mark.parametrize("c,r", [(3, 1), (1, 1)])
def test_referee_counterexample(c, r):
    # n = 2, m = 1, causal: every schedule >= 2(c + r) > 1.5(c + r).
    for sched in ("ascending", "descending", "symmetric_shift"):
        for sms in (1, 2):
            t = simulate("causal", sched, 2, 1, sms, c, r)["makespan"]
            assert t >= 2 * (c + r) > 1.5 * (c + r)
    assert simulate("causal", "symmetric_shift", 2, 1, 2, c, r)["makespan"] == 3 * (c + r)


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("mask", ["full", "causal"])
def test_coverage_contiguity_conflicts(mask, sched):
    for n in list(range(1, 17)) + [64, 128]:
        if not _valid(mask, sched, n):
            continue
        ch = chains(mask, sched, n)
        tasks = [t for c in ch for t in c]
        want = {(i, j) for i in range(n) for j in range(n) if mask == "full" or j >= i}
        assert len(tasks) == len(want) and set(tasks) == want
        for c in ch:                       # each KV tile's tasks are contiguous in its chain
            kvs = [i for i, _ in c]
            runs = [k for k, _ in itertools.groupby(kvs)]
            assert len(runs) == len(set(runs))
        assert {i for c in ch for i, _ in c} == set(range(n))
        order = reduction_order(mask, sched, n)
        for j in range(n):
            assert sorted(order[j]) == sorted(i for i, jj in tasks if jj == j)
        if sched in ("shift", "symmetric_shift"):
            for step in range(max(len(c) for c in ch)):
                js = [c[step][1] for c in ch if step < len(c)]
                assert len(js) == len(set(js)), "two SMs reduce into one dQ block at one step"


def test_bounds_hold_everywhere():
    # makespan >= longest chain of one KV tile and >= total work / P
    for mask, sched in itertools.product(["full", "causal"], SCHEDULES):
        for n in (2, 4, 6, 8):
            if not _valid(mask, sched, n):
                continue
            for m, sms in ((1, n), (3, n), (2, 3), (5, 4), (4, 2 * n + 1)):
                c, r = 3, 1
                t = simulate(mask, sched, n, m, sms, c, r)["makespan"]
                slots = len(chains(mask, sched, n))
                if t is None:
                    # a deadlock needs a head whose chains are not all co-resident
                    assert sched in ("shift", "symmetric_shift") and sms < 2 * slots
                    continue
                work = m * sum(len(ch) for ch in chains(mask, sched, n)) * (c + r)
                assert t >= work / sms
                assert t >= n * (c + r)           # KV_0 owns n tasks under both masks


def test_ascending_descending_never_deadlock():
    # Their dQ order is ascending KV index, which is also the dealing order.
    for mask, sched in itertools.product(["full", "causal"], ["ascending", "descending"]):
        for n in (1, 2, 3, 5, 8):
            for m in (1, 2, 3):
                for sms in (1, 2, 3, 7):
                    assert simulate(mask, sched, n, m, sms, 2, 1)["makespan"] is not None


def test_shift_deadlocks_when_a_head_is_split_behind_itself():
    # n = 4 on 3 SMs: KV_3 of head 0 is queued behind KV_0 on SM 0, but KV_0's last task
    # (j = 3, arrival step 3) must wait for KV_3's first reduction into dQ_3 (step 0).
    assert simulate("full", "shift", 4, 1, 3, 3, 1)["makespan"] is None
    assert simulate("full", "shift", 4, 1, 4, 3, 1)["makespan"] == 4 * 4


def _chain_graph(n_chains, weights):
    """n parallel isomorphic chains between one source (0) and one sink (1)."""
    k = len(weights)
    edges = []
    vid = lambda a, p: 2 + a * (k + 1) + p          # vertex p (0..k) of chain a
    for a in range(n_chains):
        edges.append((0, vid(a, 0), 0.0))
        for p, w in enumerate(weights):
            edges.append((vid(a, p), vid(a, p + 1), float(w)))
        edges.append((vid(a, k), 1, 0.0))
    return 2 + n_chains * (k + 1), edges, vid


@pytest.mark.parametrize("seed", range(40))
def test_lemma1_brute_force(seed):
    # Lemma 1: on parallel isomorphic chains with one source and one sink, a zero-weight
    # edge (u, v) keeps the critical path iff depth(u) <= depth(v).
    rng = random.Random(seed)
    n_chains = rng.randint(2, 4)
    weights = [rng.choice([1, 2, 3, 5]) for _ in range(rng.randint(2, 6))]
    nv, edges, vid = _chain_graph(n_chains, weights)
    base = longest_path(nv, edges)
    cp = base[1]
    k = len(weights)
    for _ in range(30):
        a, b = rng.sample(range(n_chains), 2)
        u, v = vid(a, rng.randint(0, k)), vid(b, rng.randint(0, k))
        new = longest_path(nv, edges + [(u, v, 0.0)])
        assert new is not None
        assert (new[1] == cp) == (base[u] <= base[v])


@pytest.mark.parametrize("seed", range(20))
def test_lemma1_sufficient_direction_general_dag(seed):
    # On any DAG, a zero-weight edge with depth(u) <= depth(v) changes no depth at all.
    rng = random.Random(1000 + seed)
    nv = rng.randint(4, 12)
    edges = [(u, v, float(rng.randint(0, 4))) for u in range(nv) for v in range(u + 1, nv)
             if rng.random() < 0.35]
    base = longest_path(nv, edges)
    for u in range(nv):
        for v in range(nv):
            if u != v and base[u] <= base[v] and u < v:
                assert longest_path(nv, edges + [(u, v, 0.0)]) == base


def test_deadlock_detected_when_order_contradicts_program_order():
    # Two KV chains on ONE SM in a fixed order whose dQ order is reversed -> a cycle.
    # Ascending on a single SM works (its dQ order follows the deal order) ...
    assert simulate("full", "ascending", 3, 1, 1, 3, 1)["makespan"] == 9 * 4
    # ... and the explicit graph with a reversed reduction edge has a cycle.
    from oracle.dag import schedule_dag
    nv, edges, tasks, _ = schedule_dag("full", "ascending", 2, 1, 1, 3, 1)
    idx = {t: k for k, t in enumerate(tasks)}
    # force R(1, 0) before R(0, 0): KV_1 runs after KV_0 on the only SM
    edges = edges + [(4 * idx[(0, 1, 0)] + 3, 4 * idx[(0, 0, 0)] + 2, 0.0)]
    assert longest_path(nv, edges) is None


# ---- sync-cost-aware model (simulate_ex) ----------------------------------------------

from oracle.dag import simulate_ex  # noqa: E402

SYNC_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dag_sync_closed_forms.txt")


def _sync_rows():
    rows = []
    with open(SYNC_GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or line.startswith("EXAMPLE"):
                continue
            mode, mask, sched, sms, heads, formula, _src = (x.strip() for x in line.split("|"))
            rows.append((mode, mask, sched, sms, heads, formula))
    return rows


@pytest.mark.parametrize("row", _sync_rows(), ids=lambda r: f"{r[0]}-{r[1]}-{r[2]}-P{r[3]}")
@pytest.mark.parametrize("c,r,h", [(3, 1, 0), (3, 1, 2), (3, 1, 5), (1, 3, 1), (2, 2, 4), (5, 2, 1)])
def test_sync_closed_forms(row, c, r, h):
    mode, mask, sched, sms_spec, heads_spec, formula = row
    for n in range(1, 13):
        if sched == "shift" and n < 2:
            continue
        for m in ([1] if heads_spec == "1" else [1, 2, 3]):
            sms = n if sms_spec == "n" else 1
            got = simulate_ex(mask, sched, n, m, sms, c, r, h, mode == "overlapped")["makespan"]
            want = eval(formula, {"max": max}, {"n": n, "m": m, "c": c, "r": r, "h": h})
            assert got == want, (row, n, m, c, r, h, got, want)


@pytest.mark.parametrize("seed", range(10))
def test_sync_model_reduces_to_the_pages_model(seed):
    rng = random.Random(500 + seed)
    for _ in range(15):
        mask, sched = rng.choice([("full", "ascending"), ("full", "descending"), ("full", "shift"),
                                  ("causal", "ascending"), ("causal", "descending"),
                                  ("causal", "symmetric_shift")])
        n = rng.choice([2, 4, 6, 8])
        m, sms = rng.randint(1, 4), rng.randint(1, 2 * n + 1)
        c, r = rng.choice([(3.0, 1.0), (1.0, 2.0), (2.0, 2.0)])
        a = simulate(mask, sched, n, m, sms, c, r)["makespan"]
        b = simulate_ex(mask, sched, n, m, sms, c, r, 0.0, False)["makespan"]
        assert a == b


@pytest.mark.parametrize("seed", range(10))
def test_overlap_never_slower_and_monotone_in_h(seed):
    rng = random.Random(900 + seed)
    for _ in range(10):
        mask, sched = rng.choice([("full", "ascending"), ("full", "shift"),
                                  ("causal", "descending"), ("causal", "symmetric_shift")])
        n = rng.choice([2, 4, 6])
        m, sms = rng.randint(1, 3), rng.randint(2 * n, 3 * n)   # co-resident: no deadlock
        c, r = rng.choice([(3.0, 1.0), (1.0, 2.0), (2.0, 2.0)])
        prev = None
        for h in (0.0, 0.5, 1.0, 3.0):
            ser = simulate_ex(mask, sched, n, m, sms, c, r, h, False)["makespan"]
            ovl = simulate_ex(mask, sched, n, m, sms, c, r, h, True)["makespan"]
            assert ovl <= ser
            if prev is not None:
                assert ser >= prev[0] and ovl >= prev[1]
            prev = (ser, ovl)


def test_sync_worked_example_accumulator_reuse():
    rows = []
    with open(SYNC_GOLDEN) as f:
        for line in f:
            if line.startswith("EXAMPLE"):
                rows.append([x.strip() for x in line.split("|")[1:]])
    assert rows
    for mode, mask, sched, n, m, sms, c, r, h, want in rows:
        got = simulate_ex(mask, sched, int(n), int(m), int(sms), float(c), float(r), float(h),
                          mode == "overlapped")["makespan"]
        assert got == float(want)



# ---------------------------------------------------------------------------------------
# dQ orders by arrival on a dealt grid (oracle.dag.dealt_reduction_order, dealt=True)
# ---------------------------------------------------------------------------------------
DEALT_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dag_dealt_examples.txt")


def _dealt_rows(kind):
    with open(DEALT_GOLDEN) as f:
        return [[x.strip() for x in line.split("|")[1:]] for line in f
                if line.startswith(kind)]


def test_dealt_worked_examples_orders():
    from oracle.dag import dealt_reduction_order
    rows = _dealt_rows("ORDER")
    assert len(rows) == 14
    for mask, sched, n, m, sms, head, j, want in rows:
        got = dealt_reduction_order(mask, sched, int(n), int(m), int(sms))[(int(head), int(j))]
        assert got == [int(x) for x in want.split()], (mask, sched, j)


def test_dealt_worked_examples_makespans():
    rows = _dealt_rows("MAKESPAN")
    assert len(rows) == 2
    for mask, sched, n, m, sms, c, r, want, ends in rows:
        res = simulate(mask, sched, int(n), int(m), int(sms), float(c), float(r), dealt=True)
        assert res["makespan"] == float(want)
        assert res["sm_end"] == [float(x) for x in ends.split()]
        # the fixed per-schedule order deadlocks on these grids
        assert simulate(mask, sched, int(n), int(m), int(sms), float(c), float(r))["makespan"] is None


def test_balanced_worked_example_deal_and_makespan():
    from oracle.dag import deal
    rows = _dealt_rows("DEAL")
    assert len(rows) == 4
    for mask, sched, n, m, sms, sm, want in rows:
        got = deal(mask, sched, int(n), int(m), int(sms))[int(sm)]
        runs = []
        for piece in want.split(";"):
            h, kv, *qs = (int(x) for x in piece.split())
            runs.append((h, [(kv, q) for q in qs], 0, 0))
        assert got == runs, (sm, got)
    rows = _dealt_rows("BALANCED")
    assert len(rows) == 1
    for mask, sched, n, m, sms, c, r, want, ends in rows:
        res = simulate(mask, sched, int(n), int(m), int(sms), float(c), float(r), dealt=True)
        assert res["makespan"] == float(want)
        assert res["sm_end"] == [float(x) for x in ends.split()]
        # round robin gives two SMs two whole units (10 tasks, makespan 30)
        rr = deal(mask, sched, int(n), int(m), int(sms), balanced=False)
        assert max(sum(len(run) for _, run, _, _ in runs) for runs in rr) == 10


def test_balanced_deal_invariants():
    from oracle.dag import deal
    for mask, sched in [("full", "ascending"), ("full", "shift"), ("causal", "descending"),
                        ("causal", "symmetric_shift")]:
        for n in (2, 4, 6, 8):
            ch = chains(mask, sched, n)
            longest = max(len(c) for c in ch)
            for m, hd in itertools.product((1, 2, 3, 5, 9), (64, 128)):
                for sms in range(1, 3 * n + 2):
                    per_sm = deal(mask, sched, n, m, sms, head_dim=hd)
                    rr = deal(mask, sched, n, m, sms, balanced=False)
                    units = m * len(ch)
                    rest = units % sms
                    halved = sched == "shift" and units > sms and 0 < 2 * rest <= sms
                    if (sched in ("ascending", "descending") or rest == 0
                            or units < sms or (sched == "shift" and not halved)):
                        # fixed-order schedules, whole rounds, a single partial round and
                        # equal-length chains without room to halve: exactly round robin
                        assert per_sm == rr, (mask, sched, n, m, sms)
                        continue
                    if not halved and hd >= 128:
                        # head dim 128: all whole rounds but the last stay round robin
                        lead = units // sms - 1
                        assert all(per_sm[x][:lead] == rr[x][:lead] for x in range(sms))
                    seen = {}
                    halves = {}
                    for sm, runs in enumerate(per_sm):
                        for h, run, part, split in runs:
                            chain = next(c for c in ch if run[0] in c)
                            k = chain.index(run[0])                    # contiguous, in order
                            assert chain[k:k + len(run)] == run
                            if part:
                                assert halved
                                halves.setdefault(split, {})[part] = (sm, h, run)
                                continue
                            kvs = {i for i, _ in run}
                            # a round-robin unit, or one KV tile of a cut chain
                            assert run == chain or len(kvs) == 1
                            for i in kvs:
                                assert (h, i) not in seen              # a KV tile on one SM
                                seen[(h, i)] = sm
                    if halved:
                        # split k: first ceil(len / 2) tasks on SM k, the rest on SM rest + k,
                        # each the last piece of its SM
                        assert sorted(halves) == list(range(rest))
                        for k, pr in halves.items():
                            (sa, ha, ra), (sb, hb, rb) = pr[1], pr[2]
                            assert (sa, sb, ha) == (k, rest + k, hb)
                            assert len(ra) == (len(ra) + len(rb) + 1) // 2
                            assert per_sm[sa][-1][2] == 1 and per_sm[sb][-1][2] == 2
                    tasks = sorted((h, i, j) for runs in per_sm for h, run, _, _ in runs
                                   for (i, j) in run)
                    assert tasks == sorted((h, i, j) for h in range(m) for c in ch
                                           for (i, j) in c)
                    loads = [sum(len(run) for _, run, _, _ in runs) for runs in per_sm]
                    total = sum(loads)
                    if halved:
                        # whole rounds plus at most one half of a unit
                        assert max(loads) == (units // sms) * longest + (longest + 1) // 2
                    else:
                        # greedy list scheduling: the last piece dealt to the busiest SM
                        # started on the least load, at most the mean of the rest
                        assert max(loads) <= total / sms + longest * (1 - 1 / sms) + 1e-9
                    assert max(loads) <= max(sum(len(run) for _, run, _, _ in runs)
                                             for runs in rr)


def test_dealt_equals_the_pages_order_when_heads_start_together():
    # the pages' setting on round-robin SMs (balanced dealing cuts chains only when the
    # units overrun whole rounds, which a head-per-round grid never does)
    from oracle.dag import dealt_reduction_order
    for mask, sched in [("full", "ascending"), ("full", "descending"), ("full", "shift"),
                        ("causal", "ascending"), ("causal", "descending"),
                        ("causal", "symmetric_shift")]:
        for n in (2, 4, 6, 8):
            slots = len(chains(mask, sched, n))
            fixed = reduction_order(mask, sched, n)
            for m in (1, 2, 3):
                sms_list = [slots * k for k in (1, 2, 3)]
                if sched in ("ascending", "descending"):
                    sms_list += [1, 3, 5]          # their order ignores the dealing
                for sms in sms_list:
                    got = dealt_reduction_order(mask, sched, n, m, sms, balanced=False)
                    for h in range(m):
                        for j in range(n):
                            assert got[(h, j)] == fixed[j], (mask, sched, n, m, sms, h, j)


def test_dealt_orders_are_permutations_and_never_deadlock():
    from oracle.dag import dealt_reduction_order
    for mask, sched in [("full", "shift"), ("causal", "symmetric_shift")]:
        for n in (2, 4, 6):
            fixed = reduction_order(mask, sched, n)
            for m in (1, 2, 3):
                for sms in range(1, 2 * n + 2):
                    got = dealt_reduction_order(mask, sched, n, m, sms)
                    for (h, j), kv in got.items():
                        assert sorted(kv) == sorted(fixed[j])
                    assert simulate(mask, sched, n, m, sms, 3, 1, dealt=True)["makespan"] is not None
                    res = simulate_ex(mask, sched, n, m, sms, 3, 1, 2, True, dealt=True)
                    assert res["makespan"] is not None, (mask, sched, n, m, sms)
