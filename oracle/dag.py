"""DASH task orders and the critical path of the compute/reduce DAG (test infrastructure).

Only the test suite may use this module. It shares no code with the C++ schedule
builder and simulator inside the CUDA library; the tests compare the two.

The model (Pith review of "DASH: Deterministic Attention Scheduling for High-throughput
Reproducible LLM Training", sections "Core claim", "What carries the argument" and the
"Axiom & Free-Parameter Ledger"):

* Work is a grid of tasks (KV_i, Q_j). Each task is a chain: a compute phase C(i, j) of
  cost c, then a reduction phase R(i, j) of cost r that adds the task's partial dQ_j into
  the dQ_j accumulator.
* All tasks of one KV tile run back to back on one SM (dK/dV stay resident there).
* The reductions into one dQ_j block run one at a time, in a fixed order; zero-weight
  edges between consecutive reductions encode that order.
* The objective is the critical path (longest path) of the resulting DAG.

Causal masks keep task (i, j) only when j >= i (query tile j sees key tile i); the KV_i
chain then has n - i tasks (referee report, major comment 2).

Schedules (the abstract; the Figure 3, 4, 6 and 7 captions; "What carries the argument"):

* ascending   -- the FlashAttention-3 baseline: KV_i visits Q tiles in increasing order.
* descending  -- Descending Q-Tile Iteration: KV_i visits Q tiles in decreasing order.
* shift       -- Shift Scheduling (full mask): at step t, KV_i works on Q_((i + t) mod n),
                 so no two SMs reduce into the same dQ block at the same step.
* symmetric_shift -- Symmetric Shift (causal mask, n even): one SM slot p < n/2 takes the
                 longest chain KV_p and the shortest chain KV_(n-1-p). Phase 1 covers
                 the dense lower-left rectangle (KV_0..KV_(n/2-1) x Q_(n/2)..Q_(n-1)) by a
                 cyclic shift; phase 2 runs the folded triangles from the diagonal,
                 the upper-left triangle first, then the lower-right one, keeping each
                 KV tile contiguous (Figure 7 caption).

Readings where the pages are silent (listed in the design notes as well):

* The fixed dQ order of ascending and descending is ascending KV index.
* Shift's cyclic index runs over Q tiles for a fixed KV tile (a KV tile must stay on
  one SM); its dQ_j order, like symmetric shift's, is the step at which each
  contribution arrives in the lock-step model.
* Symmetric shift, phase 2: KV_p visits Q_p..Q_(n/2-1) upwards from the diagonal, then
  KV_(n-1-p) visits Q_(n-1) down to Q_(n-1-p).
* m heads are spread over P SMs by dealing the units (head, chain slot) round robin in
  head-major order; each SM runs its units in dealing order.
* With a fixed order per schedule (``dealt=False``), a head whose chains the dealing
  spreads over two rounds of the SMs can wait on itself: a partial of the first round
  may come after one of a chain that only starts in the second round. The pages set
  shift's and symmetric shift's order by arrival and study one head on n SMs, where all
  chains start together. ``dealt=True`` takes "order of arrival" literally on the dealt
  SMs: a partial arrives when its SM has run all the tasks dealt to it before this one
  (the lower KV index first on a tie). Where a head's chains all start together this is
  the fixed order above; ascending and descending keep ascending KV index either way.
* Balanced dealing (``dealt=True`` only; this library's own choice, the pages study one
  head on n SMs): when the units do not fill whole rounds of the SMs (and there are more
  units than SMs), round robin leaves some SMs a whole unit more work than others. Shift
  and symmetric shift then cut every chain where its KV tile changes and deal the pieces
  longest first, each to the SM with the least work dealt so far (the lower SM index on
  a tie; pieces of equal length in head-major chain order); every SM runs its pieces in
  the order dealt. At head dimension 128 the first q - 1 of the q whole rounds stay round
  robin (whole units) and only the units after them are cut and dealt that way (their
  twice larger tiles need the L2 locality a round-robin round keeps; measured on GB300);
  at head dimension 64 every unit is. Each KV tile still runs on one SM, in its chain's order. Equal-length
  pieces (shift) are dealt exactly as round robin deals them, except that when the last
  partial round holds r units with 2 r <= P (and r <= MAX_SPLIT_TILES), each of those r
  KV tiles is split into two halves (the first ceil(len / 2) tasks, then the rest): split
  k's first half goes to SM k and its second half to SM r + k, after their whole units.
  The second half's last reduction ends no earlier than the first half's last one (it
  adds the first half's dK/dV partial before writing dK/dV).
"""

from __future__ import annotations

from collections import deque

__all__ = [
    "SCHEDULES",
    "chains",
    "reduction_order",
    "pieces",
    "deal",
    "dealt_reduction_order",
    "schedule_dag",
    "longest_path",
    "simulate",
    "schedule_dag_ex",
    "simulate_ex",
]

SCHEDULES = ("ascending", "descending", "shift", "symmetric_shift")
MAX_SPLIT_TILES = 256          # most KV tiles one balanced dealing splits in two


def _keys(mask: str, i: int, n: int) -> list[int]:
    """Q tiles that KV tile i contributes to, in increasing order."""
    return list(range(n)) if mask == "full" else list(range(i, n))


def chains(mask: str, sched: str, n: int) -> list[list[tuple[int, int]]]:
    """Task chains, one per SM slot, each a list of (kv_tile, q_tile) in execution order."""
    if mask not in ("full", "causal"):
        raise ValueError(mask)
    if sched == "ascending":
        return [[(i, j) for j in _keys(mask, i, n)] for i in range(n)]
    if sched == "descending":
        return [[(i, j) for j in reversed(_keys(mask, i, n))] for i in range(n)]
    if sched == "shift":
        if mask != "full":
            raise ValueError("shift scheduling is defined for the full mask")
        return [[(i, (i + t) % n) for t in range(n)] for i in range(n)]
    if sched == "symmetric_shift":
        if mask != "causal" or n % 2:
            raise ValueError("symmetric shift is defined for the causal mask with even n")
        half = n // 2
        out = []
        for p in range(half):
            phase1 = [(p, half + (p + t) % half) for t in range(half)]
            upper_left = [(p, p + u) for u in range(half - p)]
            lower_right = [(n - 1 - p, n - 1 - u) for u in range(p + 1)]
            out.append(phase1 + upper_left + lower_right)
        return out
    raise ValueError(sched)


def reduction_order(mask: str, sched: str, n: int) -> dict[int, list[int]]:
    """For each dQ block j, the KV tiles that reduce into it, in the fixed order."""
    ch = chains(mask, sched, n)
    contrib: dict[int, list[tuple[int, int]]] = {j: [] for j in range(n)}
    for chain in ch:
        for step, (i, j) in enumerate(chain):
            contrib[j].append((step, i))
    order = {}
    for j, lst in contrib.items():
        if sched in ("ascending", "descending"):
            order[j] = sorted(i for _, i in lst)
        else:
            steps = [st for st, _ in lst]
            if len(set(steps)) != len(steps):
                raise AssertionError(f"two contributions to dQ_{j} arrive at the same step")
            order[j] = [i for _, i in sorted(lst)]
    return order


def longest_path(n_vertices: int, edges: list[tuple[int, int, float]]):
    """Earliest start time of every vertex (longest path from any source, sources at 0).

    Returns None when the graph has a cycle.
    """
    succ: list[list[tuple[int, float]]] = [[] for _ in range(n_vertices)]
    indeg = [0] * n_vertices
    for u, v, w in edges:
        succ[u].append((v, w))
        indeg[v] += 1
    depth = [0.0] * n_vertices
    ready = deque(v for v in range(n_vertices) if indeg[v] == 0)
    seen = 0
    while ready:
        u = ready.popleft()
        seen += 1
        for v, w in succ[u]:
            depth[v] = max(depth[v], depth[u] + w)
            indeg[v] -= 1
            if indeg[v] == 0:
                ready.append(v)
    return depth if seen == n_vertices else None


def pieces(chain: list[tuple[int, int]]) -> list[list[tuple[int, int]]]:
    """A chain cut where its KV tile changes: its runs of one KV tile, in chain order."""
    out: list[list[tuple[int, int]]] = []
    for task in chain:
        if out and out[-1][-1][0] == task[0]:
            out[-1].append(task)
        else:
            out.append([task])
    return out


def deal(mask: str, sched: str, n: int, m: int, num_sms: int, balanced: bool = True,
         head_dim: int = 128):
    """Per SM, the runs of tasks it executes, in order: lists of (head, [(i, j), ...],
    part, split) -- part 0 for whole KV tiles, 1 and 2 for the first and second half of
    split tile ``split`` (0 where part is 0).

    Round robin deals the units (head, chain slot) head-major, unit u to SM u mod P.
    ``balanced`` deals as the library's kernels do (the module docstring): round robin
    unless the schedule orders dQ by arrival and the units overrun whole rounds of the
    SMs, in which case the chains' KV-tile pieces go longest first to the least-loaded SM
    (shift: its last partial round halved where there is room).
    """
    ch = chains(mask, sched, n)
    units = [(h, slot) for h in range(m) for slot in range(len(ch))]
    per_sm: list[list[tuple[int, list[tuple[int, int]], int, int]]] = [
        [] for _ in range(num_sms)]
    full_rounds, rest = divmod(len(units), num_sms)
    if (not balanced or sched in ("ascending", "descending") or rest == 0
            or full_rounds == 0):
        for u, (h, slot) in enumerate(units):
            per_sm[u % num_sms].append((h, list(ch[slot]), 0, 0))
        return per_sm
    if (sched == "shift" and 2 * rest <= num_sms and rest <= MAX_SPLIT_TILES
            and max(len(c) for c in ch) >= 2):
        whole = len(units) - rest
        for u in range(whole):
            h, slot = units[u]
            per_sm[u % num_sms].append((h, list(ch[slot]), 0, 0))
        for k in range(rest):
            h, slot = units[whole + k]
            cut = (len(ch[slot]) + 1) // 2
            per_sm[k].append((h, list(ch[slot][:cut]), 1, k))
            per_sm[rest + k].append((h, list(ch[slot][cut:]), 2, k))
        return per_sm
    lead = (full_rounds - 1) * num_sms if head_dim >= 128 else 0
    for u in range(lead):
        h, slot = units[u]
        per_sm[u % num_sms].append((h, list(ch[slot]), 0, 0))
    runs = [(h, run) for (h, slot) in units[lead:] for run in pieces(ch[slot])]
    load = [0] * num_sms                     # the round-robin rounds loaded every SM alike
    for k in sorted(range(len(runs)), key=lambda k: (-len(runs[k][1]), k)):
        sm = min(range(num_sms), key=lambda s: (load[s], s))
        per_sm[sm].append((runs[k][0], runs[k][1], 0, 0))
        load[sm] += len(runs[k][1])
    return per_sm


def dealt_reduction_order(mask: str, sched: str, n: int, m: int, num_sms: int,
                          balanced: bool = True, head_dim: int = 128):
    """For each (head, dQ block j), the KV tiles that reduce into it, in the order the
    dealt SMs produce them (the ``dealt=True`` reading in the module docstring); with
    ``balanced`` false, on SMs dealt round robin."""
    if sched in ("ascending", "descending"):
        fixed = reduction_order(mask, sched, n)
        return {(h, j): list(fixed[j]) for h in range(m) for j in range(n)}
    arrivals: dict[tuple[int, int], list[tuple[int, int]]] = {
        (h, j): [] for h in range(m) for j in range(n)}
    for runs in deal(mask, sched, n, m, num_sms, balanced, head_dim):
        place = 0                            # tasks this SM has run so far
        for h, run, _part, _split in runs:
            for (i, j) in run:
                arrivals[(h, j)].append((place, i))
                place += 1
    return {key: [i for _, i in sorted(lst)] for key, lst in arrivals.items()}


def _orders(mask: str, sched: str, n: int, m: int, num_sms: int, dealt: bool,
            head_dim: int = 128):
    """(head, j) -> dQ_j order of that head, fixed per schedule or dealt."""
    if dealt:
        return dealt_reduction_order(mask, sched, n, m, num_sms, head_dim=head_dim)
    fixed = reduction_order(mask, sched, n)
    return {(h, j): fixed[j] for h in range(m) for j in fixed}


def _dealt_tasks(mask: str, sched: str, n: int, m: int, num_sms: int, dealt: bool,
                 head_dim: int = 128):
    """Number the tasks SM by SM in run order: (per_sm task lists, tasks, sm_of_task,
    index, halves). ``dealt`` deals as the kernels do (balanced), else round robin;
    halves lists (last task of a first half, last task of its second half)."""
    per_sm: list[list[int]] = [[] for _ in range(num_sms)]
    tasks: list[tuple[int, int, int]] = []
    sm_of_task: list[int] = []
    index: dict[tuple[int, int, int], int] = {}
    last_of: dict[tuple[int, int], int] = {}
    for sm, runs in enumerate(deal(mask, sched, n, m, num_sms, balanced=dealt,
                                   head_dim=head_dim)):
        for hd, run, part, split in runs:
            for (i, j) in run:
                k = len(tasks)
                tasks.append((hd, i, j))
                sm_of_task.append(sm)
                index[(hd, i, j)] = k
                per_sm[sm].append(k)
            if part:
                last_of[(split, part)] = len(tasks) - 1
    halves = [(last_of[(s, 1)], last_of[(s, 2)]) for (s, p) in sorted(last_of) if p == 1]
    return per_sm, tasks, sm_of_task, index, halves


def schedule_dag(mask: str, sched: str, n: int, m: int, num_sms: int, c: float, r: float,
                 dealt: bool = False, head_dim: int = 128):
    """Build the explicit DAG of m heads' tasks dealt onto ``num_sms`` SMs.

    Every task (head, i, j) owns four vertices: compute start/end and reduce start/end.
    Returns (n_vertices, edges, tasks, sm_of_task) where tasks[k] = (head, i, j) and task k
    owns vertices 4k..4k+3.
    """
    order = _orders(mask, sched, n, m, num_sms, dealt, head_dim)
    per_sm, tasks, sm_of_task, index, halves = _dealt_tasks(mask, sched, n, m, num_sms, dealt,
                                                            head_dim)
    edges: list[tuple[int, int, float]] = []
    for k in range(len(tasks)):
        cs, ce, rs, re = 4 * k, 4 * k + 1, 4 * k + 2, 4 * k + 3
        edges += [(cs, ce, c), (ce, rs, 0.0), (rs, re, r)]
    for lst in per_sm:                               # one SM runs its tasks back to back
        for a, b in zip(lst, lst[1:]):
            edges.append((4 * a + 3, 4 * b, 0.0))
    for (h, j), kv in order.items():                 # fixed dQ reduction order
        for a, b in zip(kv, kv[1:]):
            edges.append((4 * index[(h, a, j)] + 3, 4 * index[(h, b, j)] + 2, 0.0))
    for ka, kb in halves:                            # a second half adds its first's dK/dV
        edges.append((4 * ka + 3, 4 * kb + 3, 0.0))
    return 4 * len(tasks), edges, tasks, sm_of_task


def simulate(mask: str, sched: str, n: int, m: int, num_sms: int, c: float, r: float,
             dealt: bool = False, head_dim: int = 128):
    """Critical path of the schedule DAG.

    Returns a dict with ``makespan`` (None on a cycle, i.e. a deadlock), ``sm_end`` (finish
    time per SM) and ``sm_idle`` (finish time minus busy time per SM).
    """
    nv, edges, tasks, sm_of_task = schedule_dag(mask, sched, n, m, num_sms, c, r, dealt,
                                                head_dim)
    depth = longest_path(nv, edges)
    if depth is None:
        return {"makespan": None, "sm_end": None, "sm_idle": None}
    sm_end = [0.0] * num_sms
    sm_busy = [0.0] * num_sms
    for k, sm in enumerate(sm_of_task):
        sm_end[sm] = max(sm_end[sm], depth[4 * k + 3])       # reduce-end vertex
        sm_busy[sm] += c + r
    makespan = max(sm_end) if tasks else 0.0
    return {"makespan": makespan, "sm_end": sm_end,
            "sm_idle": [e - b for e, b in zip(sm_end, sm_busy)]}


# ---------------------------------------------------------------------------------------
# Sync-cost-aware extension (the Pith review's "Where Pith is reading between the lines"
# proposes nonzero synchronisation edge costs; its Axiom & Free-Parameter Ledger lists the
# zero-cost edge as a domain assumption).
#
# * h: cost of handing a dQ block's turn from one SM to another -- the weight of an order
#   edge between consecutive reductions of one dQ block that run on different SMs (0 when
#   both run on the same SM).
# * overlapped: the SM has two engines instead of running C then R back to back. The
#   compute engine runs the C phases in order, the reduce engine the R phases in order,
#   and C of the k-th task waits for R of the (k-2)-th: the partial of task k needs the
#   accumulator that the read-out of task k-1 frees, and that read-out starts once the
#   reduce engine has finished task k-2.
# With h = 0 and overlapped = False this is exactly schedule_dag / simulate above.
# ---------------------------------------------------------------------------------------
def schedule_dag_ex(mask: str, sched: str, n: int, m: int, num_sms: int, c: float, r: float,
                    h: float, overlapped: bool, dealt: bool = False, head_dim: int = 128):
    """The schedule DAG with hand-off cost ``h`` and, optionally, the two-engine SM.

    Same vertex numbering and return value as schedule_dag.
    """
    order = _orders(mask, sched, n, m, num_sms, dealt, head_dim)
    per_sm, tasks, sm_of_task, index, halves = _dealt_tasks(mask, sched, n, m, num_sms, dealt,
                                                            head_dim)
    edges: list[tuple[int, int, float]] = []
    for k in range(len(tasks)):
        cs, ce, rs, re = 4 * k, 4 * k + 1, 4 * k + 2, 4 * k + 3
        edges += [(cs, ce, c), (ce, rs, 0.0), (rs, re, r)]
    for lst in per_sm:
        for pos in range(1, len(lst)):
            a, b = lst[pos - 1], lst[pos]
            if overlapped:
                edges.append((4 * a + 1, 4 * b, 0.0))          # compute engine in order
                edges.append((4 * a + 3, 4 * b + 2, 0.0))      # reduce engine in order
                if pos >= 2:                                   # accumulator reuse
                    edges.append((4 * lst[pos - 2] + 3, 4 * b, 0.0))
            else:
                edges.append((4 * a + 3, 4 * b, 0.0))          # C then R, task after task
    for (hd, j), kv in order.items():                          # fixed dQ reduction order
        for a, b in zip(kv, kv[1:]):
            ka, kb = index[(hd, a, j)], index[(hd, b, j)]
            w = 0.0 if sm_of_task[ka] == sm_of_task[kb] else h
            edges.append((4 * ka + 3, 4 * kb + 2, w))
    for ka, kb in halves:
        edges.append((4 * ka + 3, 4 * kb + 3, 0.0))
    return 4 * len(tasks), edges, tasks, sm_of_task


def simulate_ex(mask: str, sched: str, n: int, m: int, num_sms: int, c: float, r: float,
                h: float = 0.0, overlapped: bool = False, dealt: bool = False,
                head_dim: int = 128):
    """Critical path of schedule_dag_ex; same return value as simulate."""
    nv, edges, tasks, sm_of_task = schedule_dag_ex(mask, sched, n, m, num_sms, c, r, h,
                                                   overlapped, dealt, head_dim)
    depth = longest_path(nv, edges)
    if depth is None:
        return {"makespan": None, "sm_end": None, "sm_idle": None}
    sm_end = [0.0] * num_sms
    sm_busy = [0.0] * num_sms
    for k, sm in enumerate(sm_of_task):
        sm_end[sm] = max(sm_end[sm], depth[4 * k + 3])
        sm_busy[sm] += c + r
    makespan = max(sm_end) if tasks else 0.0
    return {"makespan": makespan, "sm_end": sm_end,
            "sm_idle": [e - b for e, b in zip(sm_end, sm_busy)]}

