"""The library's schedule tables and DAG simulator (host C++) against the oracle."""
import itertools
import random

import pytest

import reproducible_deterministic_attn_gb300 as da
from oracle import dag
from tests._lib import ensure_built

NAMES = {0: "ascending", 1: "descending", 2: "shift", 3: "symmetric_shift"}
MASKS = {0: "full", 1: "causal"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _valid(mask, sched, n):
    if sched == 2 and mask != 0:
        return False
    if sched == 3 and (mask != 1 or n % 2):
        return False
    return True


@pytest.mark.parametrize("mask,sched", list(itertools.product([0, 1], [0, 1, 2, 3])))
def test_tables_match_oracle(mask, sched):
    for n in list(range(1, 17)) + [64, 128]:
        if not _valid(mask, sched, n):
            assert da.dash_sched_num_slots(mask, sched, n) == -da.DASH_ERR_UNSUPPORTED
            continue
        off, tasks, ords = da.dash_sched_table(mask, sched, n)
        chains = dag.chains(MASKS[mask], NAMES[sched], n)
        assert len(off) == len(chains) + 1
        got = [tasks[off[p]:off[p + 1]] for p in range(len(chains))]
        assert got == [list(c) for c in chains]
        order = dag.reduction_order(MASKS[mask], NAMES[sched], n)
        for j in range(n):
            for pos, i in enumerate(order[j]):
                assert ords[i][j] == pos
        masked = sum(1 for i in range(n) for j in range(n) if ords[i][j] < 0)
        assert masked == (0 if mask == 0 else n * (n - 1) // 2)


@pytest.mark.parametrize("seed", range(8))
def test_dealt_tables_match_oracle(seed):
    rng = random.Random(300 + seed)
    for _ in range(20):
        mask, sched = rng.choice([(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 3)])
        n = rng.choice([1, 2, 3, 4, 6, 8, 12]) if sched != 3 else rng.choice([2, 4, 6, 8, 12])
        m, grid = rng.randint(1, 5), rng.randint(1, 3 * n + 2)
        hd = rng.choice([64, 128])
        got = da.dash_sched_dealt_table(mask, sched, n, m, grid, hd)
        want = dag.dealt_reduction_order(MASKS[mask], NAMES[sched], n, m, grid, head_dim=hd)
        for h in range(m):
            for j in range(n):
                for pos, i in enumerate(want[(h, j)]):
                    assert got[h][i][j] == pos, (mask, sched, n, m, grid, h, i, j)
            masked = sum(1 for i in range(n) for j in range(n) if got[h][i][j] < 0)
            assert masked == (0 if mask == 0 else n * (n - 1) // 2)


@pytest.mark.parametrize("seed", range(6))
def test_deal_matches_oracle(seed):
    rng = random.Random(800 + seed)
    for _ in range(20):
        mask, sched = rng.choice([(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 3)])
        n = rng.choice([1, 2, 3, 4, 6, 8, 12]) if sched != 3 else rng.choice([2, 4, 6, 8, 12])
        m, grid = rng.randint(1, 8), rng.randint(1, 3 * n + 2)
        hd = rng.choice([64, 128])
        got = da.dash_sched_deal(mask, sched, n, m, grid, hd)
        want = dag.deal(MASKS[mask], NAMES[sched], n, m, grid, head_dim=hd)
        assert got == want, (mask, sched, n, m, grid, hd)


def test_deal_at_the_kernel_sizes():
    # 152 CTAs. Causal 4x16 heads of n = 16 at head dim 64 (512 units of 17 tasks): every
    # unit's pieces dealt longest first bring the busiest CTA to the mean (57.3 tasks)
    # instead of a whole unit above it. Causal 1x32 heads of n = 128 at head dim 128 (2048
    # units of 129): 12 round-robin rounds, then the last 224 units' pieces longest first
    # (mean 1738.1; all pieces: 1739). Full 2x16 heads of n = 64 (2048 units of 64, 72 in
    # the last round): those 72 KV tiles are halved over 144 CTAs, so the busiest runs 13.5
    # units (mean 13.47).
    for mask, sched, n, heads, hd, rr_max, max_load, splits in [
            (1, 3, 16, 64, 64, 68, 58, 0), (1, 3, 128, 32, 128, 1806, 1757, 0),
            (1, 3, 128, 32, 64, 1806, 1739, 0), (0, 2, 64, 32, 128, 896, 864, 72)]:
        got = da.dash_sched_deal(mask, sched, n, heads, 152, hd)
        want = dag.deal(MASKS[mask], NAMES[sched], n, heads, 152, head_dim=hd)
        assert got == want
        loads = [sum(len(run) for _, run, _, _ in runs) for runs in got]
        assert max(loads) == max_load
        assert sum(1 for runs in got for pc in runs if pc[2] == 1) == splits
        rr = dag.deal(MASKS[mask], NAMES[sched], n, heads, 152, balanced=False)
        assert max(sum(len(run) for _, run, _, _ in runs) for runs in rr) == rr_max
    with pytest.raises(da.DashError):
        da.dash_sched_deal(1, 3, 8, 0, 4)
    with pytest.raises(da.DashError):
        da.dash_sched_deal(1, 3, 7, 1, 4)             # symmetric shift needs even n


def test_dealt_tables_at_the_kernel_sizes():
    # 152 CTAs: full 2x16 heads of n = 64 and causal 32 heads of n = 128 split heads over
    # two rounds of the grid; the per-head orders still follow the dealing
    for mask, sched, n, heads in [(0, 2, 64, 32), (1, 3, 128, 32)]:
        got = da.dash_sched_dealt_table(mask, sched, n, heads, 152)
        want = dag.dealt_reduction_order(MASKS[mask], NAMES[sched], n, heads, 152)
        _, _, fixed = da.dash_sched_table(mask, sched, n)
        differ = 0
        for h in range(heads):
            for j in range(n):
                assert [i for i in sorted(range(n), key=lambda i: got[h][i][j])
                        if got[h][i][j] >= 0] == want[(h, j)]
            differ += any(got[h][i] != fixed[i] for i in range(n))
        assert differ > 0                      # some head is split by the grid
    with pytest.raises(da.DashError):
        da.dash_sched_dealt_table(0, 2, 8, 0, 4)
    with pytest.raises(da.DashError):
        da.dash_sched_dealt_table(1, 2, 8, 1, 4)      # shift needs the full mask


def test_invalid_n():
    assert da.dash_sched_num_slots(0, 0, 0) == -da.DASH_ERR_INVALID_ARG
    assert da.dash_sched_num_slots(0, 0, 40000) == -da.DASH_ERR_INVALID_ARG


@pytest.mark.parametrize("seed", range(12))
def test_simulator_matches_oracle(seed):
    rng = random.Random(seed)
    for _ in range(25):
        mask, sched = rng.choice([(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 3)])
        n = rng.choice([1, 2, 3, 4, 6, 8, 10]) if sched != 3 else rng.choice([2, 4, 6, 8])
        m = rng.randint(1, 5)
        sms = rng.randint(1, 2 * n + 2)
        c, r = rng.choice([(3.0, 1.0), (1.0, 0.25), (2.0, 2.0), (0.5, 1.5)])
        hd = rng.choice([64, 128])
        want = dag.simulate(MASKS[mask], NAMES[sched], n, m, sms, c, r, dealt=True, head_dim=hd)
        mk, ends = da.dash_sched_simulate(mask, sched, n, m, sms, c, r, hd)
        if want["makespan"] is None:
            assert mk is None, (mask, sched, n, m, sms)
        else:
            assert mk == pytest.approx(want["makespan"], abs=1e-9), (mask, sched, n, m, sms)
            assert ends == pytest.approx(want["sm_end"], abs=1e-9)


def test_simulator_closed_forms_large_n():
    # the pages' full-mask bound (shift) and the symmetric-shift form at the kernel's sizes
    for n in (64, 128):
        for m in (1, 2, 4):
            mk, _ = da.dash_sched_simulate(0, 2, n, m, n, 3.0, 1.0)
            assert mk == m * n * 4.0
            mk, _ = da.dash_sched_simulate(1, 3, n, m, n, 3.0, 1.0)
            assert mk == ((m + 1) // 2) * (n + 1) * 4.0


@pytest.mark.parametrize("seed", range(8))
def test_sync_simulator_matches_oracle(seed):
    rng = random.Random(4000 + seed)
    for _ in range(20):
        mask, sched = rng.choice([(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 3)])
        n = rng.choice([1, 2, 3, 4, 6, 8]) if sched != 3 else rng.choice([2, 4, 6, 8])
        m = rng.randint(1, 4)
        sms = rng.randint(1, 2 * n + 2)
        c, r = rng.choice([(3.0, 1.0), (1.0, 0.25), (2.0, 2.0), (0.5, 1.5)])
        h = rng.choice([0.0, 0.5, 2.0, 5.0])
        ovl = rng.randint(0, 1)
        hd = rng.choice([64, 128])
        want = dag.simulate_ex(MASKS[mask], NAMES[sched], n, m, sms, c, r, h, bool(ovl),
                               dealt=True, head_dim=hd)
        mk, ends = da.dash_sched_simulate_ex(mask, sched, n, m, sms, c, r, h, ovl, hd)
        if want["makespan"] is None:
            assert mk is None
        else:
            assert mk == pytest.approx(want["makespan"], rel=1e-12, abs=1e-9)
            assert ends == pytest.approx(want["sm_end"], rel=1e-12, abs=1e-9)


@pytest.mark.parametrize("seed", range(6))
def test_selector_is_the_oracle_argmin(seed):
    rng = random.Random(7000 + seed)
    for _ in range(12):
        mask = rng.randint(0, 1)
        n = rng.choice([2, 4, 6, 8])
        m, sms = rng.randint(1, 4), rng.randint(1, 3 * n)
        c, r, h = rng.choice([3.0, 1.0]), rng.choice([1.0, 2.5]), rng.choice([0.0, 1.0, 4.0])
        ovl = rng.randint(0, 1)
        hd = rng.choice([64, 128])
        best, best_mk = None, None
        for s in (0, 1, 2, 3):
            if not _valid(mask, s, n):
                continue
            mk = dag.simulate_ex(MASKS[mask], NAMES[s], n, m, sms, c, r, h, bool(ovl),
                                 dealt=True, head_dim=hd)["makespan"]
            if mk is not None and (best is None or mk < best_mk):
                best, best_mk = s, mk
        got, got_mk = da.dash_sched_select(mask, n, m, sms, c, r, h, ovl, hd)
        assert got == best and got_mk == pytest.approx(best_mk)


# Cycles per 128 x 128 task measured on GB300 for the head-dim-128 kernel: compute step
# (non-deterministic), hold of a dQ block's turn (adds + fence + read-out), hand-off.
GB300_COSTS = (6900.0, 5600.0, 3000.0, 1)


@pytest.mark.parametrize("mask,n,heads,hd,measured_best", [
    (0, 64, 32, 128, 2),     # full 2x16x8192x128: shift measured fastest
    (1, 128, 32, 128, 3),    # causal 1x32x16384x128: symmetric shift measured fastest
    (1, 16, 64, 64, 3),      # causal 4x16x2048x64: symmetric shift measured fastest
])
def test_selector_picks_the_measured_best_on_gb300(mask, n, heads, hd, measured_best):
    got, _ = da.dash_sched_select(mask, n, heads, 152, *GB300_COSTS, head_dim=hd)
    assert got == measured_best


def test_selector_and_simulate_ex_argument_errors():
    with pytest.raises(da.DashError):
        da.dash_sched_select(0, 8, 1, 8, -1.0, 1.0, 0.0, 0)
    with pytest.raises(da.DashError):
        da.dash_sched_select(2, 8, 1, 8, 1.0, 1.0, 0.0, 0)
    with pytest.raises(da.DashError):
        da.dash_sched_simulate_ex(0, 0, 8, 1, 8, 1.0, 1.0, -1.0, 0)
    with pytest.raises(da.DashError):
        da.dash_sched_simulate_ex(0, 0, 8, 1, 8, 1.0, 1.0, 0.0, 2)
    for bad_hd in (0, 96):                              # head dims the kernels do not have
        with pytest.raises(da.DashError):
            da.dash_sched_select(0, 8, 1, 8, 1.0, 1.0, 0.0, 0, bad_hd)
        with pytest.raises(da.DashError):
            da.dash_sched_simulate_ex(0, 0, 8, 1, 8, 1.0, 1.0, 0.0, 0, bad_hd)
        with pytest.raises(da.DashError):
            da.dash_sched_dealt_table(0, 2, 8, 1, 4, bad_hd)
        with pytest.raises(da.DashError):
            da.dash_sched_deal(0, 2, 8, 1, 4, bad_hd)
