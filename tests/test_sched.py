"""Schedule tables and the DAG model (CPU only).

Checks the definitions of the schedules (DASH technical summary section 2.2:
Descending Q-Tile Iteration, Shift Scheduling and its symmetric causal form),
the KV-chain constraint (section 2.1), that every dQ tile has one strict
reduction order, that no wait can deadlock, the unit-weight critical paths,
and Lemma 1 (zero-weight edges keep the critical path when depth(u) <=
depth(v)).
"""
import itertools

import pytest

import deterministic_attn_backward_gb300 as dab

SCHEDS = ("serial", "descending_q", "shift", "atomic")
MASKS = ("full", "causal")
NS = list(range(1, 41)) + [64, 96, 128, 160, 256]


def cases():
    for sched, mask, N in itertools.product(SCHEDS, MASKS, NS):
        if sched == "shift" and mask == "causal" and N % 2:
            continue
        yield sched, mask, N


def units(sched, mask, N):
    return [dab.sched_unit(sched, mask, N, u) for u in range(dab.sched_units_per_head(sched, mask, N))]


def visible(mask, i, j):
    return mask == "full" or j >= i


@pytest.mark.parametrize("sched,mask,N", list(cases()))
def test_coverage_chains_and_orders(sched, mask, N):
    U = units(sched, mask, N)
    seen = {}
    for u, steps in enumerate(U):
        for t, (i, j) in enumerate(steps):
            assert 0 <= i < N and 0 <= j < N and visible(mask, i, j)
            assert (i, j) not in seen, "tile visited twice"
            seen[(i, j)] = (u, t)
        # KV-chain constraint: each KV tile's steps are contiguous in its unit
        kvs = [i for i, _ in steps]
        runs = [k for k, _ in itertools.groupby(kvs)]
        assert len(runs) == len(set(runs)), "a KV chain is split"
    assert set(seen) == {(i, j) for i in range(N) for j in range(N) if visible(mask, i, j)}
    # Q-tile order of each chain
    for steps in U:
        for i, grp in itertools.groupby(steps, key=lambda s: s[0]):
            js = [j for _, j in grp]
            if sched in ("serial", "atomic"):
                assert js == sorted(js)
            elif sched == "descending_q":
                assert js == sorted(js, reverse=True)
            elif mask == "full":
                assert js == [(i + t) % N for t in range(N)]
    if sched == "atomic":
        return
    # strict total order per dQ tile: ranks are 0..contributors-1
    for j in range(N):
        ranks = sorted(dab.sched_rank(sched, mask, N, i, j) for i in range(N) if visible(mask, i, j))
        assert ranks == list(range(dab.sched_contributors(mask, N, j)))
    for i in range(N):
        for j in range(N):
            if not visible(mask, i, j):
                assert dab.sched_rank(sched, mask, N, i, j) == -1


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("N", [1, 2, 7, 16, 64, 128])
def test_descending_keeps_serial_reduction_order(mask, N):
    for i in range(N):
        for j in range(N):
            a = dab.sched_rank("serial", mask, N, i, j)
            assert a == dab.sched_rank("descending_q", mask, N, i, j)
            if visible(mask, i, j):
                assert a == i


@pytest.mark.parametrize("mask,N", [("full", n) for n in (2, 5, 16, 64, 128, 256)]
                         + [("causal", n) for n in (2, 4, 16, 64, 128, 256)])
def test_shift_is_conflict_free_and_ranked_by_visit_time(mask, N):
    """In the lockstep model every gang member does one step per time unit:
    no two members of a gang touch one dQ tile at the same step, and dQ_j's
    reduction order is the order of visit (group-major for grouped heads)."""
    U = units("shift", mask, N)
    gang = dab.sched_gang_size("shift", mask, N)
    for g0 in range(0, len(U), gang):
        members = U[g0:g0 + gang]
        for t in range(max(len(s) for s in members)):
            qs = [s[t][1] for s in members if t < len(s)]
            assert len(qs) == len(set(qs)), f"conflict at step {t}"
    for j in range(N):
        contrib = []
        for u, steps in enumerate(U):
            for t, (i, jj) in enumerate(steps):
                if jj == j:
                    contrib.append(((u // gang, t), i))
        order = [i for _, i in sorted(contrib)]
        assert [dab.sched_rank("shift", mask, N, i, j) for i in order] == list(range(len(order)))


@pytest.mark.parametrize("N", [2, 4, 8, 16, 32])
def test_unit_weight_critical_paths(N):
    """Reduction-bound unit model (compute 0, reduction 1, in the chain)."""
    cp = lambda s, m: dab.dag_critical_path(s, m, N, 0.0, 1.0, 0)
    assert cp("serial", "full") == 2 * N - 1
    assert cp("descending_q", "full") == 2 * N - 1
    assert cp("shift", "full") == N
    assert cp("serial", "causal") == 2 * N - 1
    assert cp("descending_q", "causal") == N
    assert cp("shift", "causal") == N + 1
    # compute-bound model: every deterministic schedule's path is its longest chain
    for s in ("serial", "descending_q", "shift"):
        assert dab.dag_critical_path(s, "full", N, 1.0, 0.0, 0) == N


@pytest.mark.parametrize("sched,mask", [("shift", "full"), ("shift", "causal"),
                                        ("serial", "full"), ("descending_q", "full"),
                                        ("descending_q", "causal"), ("serial", "causal")])
@pytest.mark.parametrize("N", [4, 8, 16])
def test_lemma1_depth_condition(sched, mask, N):
    """Lemma 1 on the chain-only DAG (unit weights, every chain starting at 0)
    plus the zero-weight reduction-order edges u -> v (rank(u) = rank(v) - 1
    on one dQ tile).  With depths counted from the sink, the critical path is
    kept exactly when every edge has end(u) <= CP - tail(v); the stronger
    start-depth form end(u) <= start(v) implies it.  The shift schedules meet
    the strong form; serial and descending full masks break both."""
    U = units(sched, mask, N)
    where = {}
    for u, steps in enumerate(U):
        for t, (i, j) in enumerate(steps):
            where[(i, j)] = (u, t)
    by_rank = {(j, dab.sched_rank(sched, mask, N, i, j)): where[(i, j)] for (i, j) in where}
    cp0 = max(len(s) for s in U)
    strong = exact = True
    for (i, j), (uv, tv) in where.items():
        r = dab.sched_rank(sched, mask, N, i, j)
        if r <= 0:
            continue
        uu, tu = by_rank[(j, r - 1)]
        end_u, start_v, tail_v = tu + 1, tv, len(U[uv]) - tv
        strong &= end_u <= start_v
        exact &= end_u <= cp0 - tail_v
    full_cp = dab.dag_critical_path(sched, mask, N, 0.0, 1.0, 0)
    assert exact == (full_cp == cp0), (exact, full_cp, cp0)
    if strong:
        assert exact
    if sched == "shift":
        assert strong
    if sched in ("serial", "descending_q") and mask == "full":
        assert not exact and full_cp > cp0


def test_deadlock_detection_and_progress():
    # full-mask shift needs the whole gang resident
    assert dab.dag_simulate("shift", "full", 16, 4, 16)[0] == 0
    assert dab.dag_simulate("shift", "full", 16, 4, 15)[0] == -2
    assert dab.dag_simulate("shift", "causal", 16, 4, 8)[0] == 0
    assert dab.dag_simulate("shift", "causal", 16, 4, 7)[0] == -2
    # serial / descending / atomic make progress on any number of CTAs
    for s in ("serial", "descending_q", "atomic"):
        for m in MASKS:
            assert dab.dag_simulate(s, m, 16, 3, 1)[0] == 0
            assert dab.dag_simulate(s, m, 16, 3, 5)[0] == 0
    # grouped full-mask shift for long heads: groups of 128 tiles
    assert dab.sched_gang_size("shift", "full", 256) == 128
    assert dab.dag_simulate("shift", "full", 256, 1, 128, 1.0, 0.1, 1)[0] == 0


def test_schedules_recover_utilisation():
    """Many heads on a finite GPU: descending removes the causal stalls of
    serial, and shift keeps full-mask reductions off the critical path."""
    heads, ctas, N = 32, 64, 32
    busy = lambda s, m, wr: dab.dag_simulate(s, m, N, heads, ctas, 1.0, wr, 1)[2]
    assert busy("descending_q", "causal", 0.3) > busy("serial", "causal", 0.3) + 0.1
    assert busy("shift", "full", 1.2) > busy("serial", "full", 1.2) + 0.05
    assert busy("atomic", "full", 0.3) > 0.95


# ---------------------------------------------------------------- palette
def test_interleaved_buffers_in_the_dag_model():
    """ways = 1 is the plain model; with as many buffers as contributors no
    reduction waits on another, so an ordered schedule takes exactly as long
    as the unordered one with the same step order and dispatch."""
    for mask in ("full", "causal"):
        for N in (4, 8):
            a = dab.dag_simulate("serial", mask, N, 3, 5, 1.0, 0.7, 1, ways=1)
            b = dab.dag_simulate("serial", mask, N, 3, 5, 1.0, 0.7, 1)
            assert a == b
            free = dab.dag_simulate("serial", mask, N, 3, 5, 1.0, 0.7, 1, ways=N)
            unordered = dab.dag_simulate("atomic", mask, N, 3, 5, 1.0, 0.7, 1)
            assert free[0] == 0 and abs(free[1] - unordered[1]) < 1e-9
            # more buffers never lengthen the makespan
            m = [dab.dag_simulate("descending_q", mask, N, 3, 5, 1.0, 0.7, 1, ways=w)[1]
                 for w in (1, 2, 4)]
            assert m[0] >= m[1] - 1e-9 >= m[2] - 2e-9


def test_sched_select_picks_a_runnable_deterministic_schedule():
    lib = dab.load_library()
    for mask in ("full", "causal"):
        for B, H, S in ((1, 2, 256), (2, 3, 384), (4, 16, 2048), (2, 16, 8192)):
            for ctas in (4, 37, 152):
                pick = dab.sched_select(mask, B, H, S, ctas)
                assert pick in ("serial", "descending_q", "shift")
                N = S // 128
                if pick == "shift":
                    assert not (mask == "causal" and N % 2)
                    assert dab.sched_gang_size("shift", mask, N) <= ctas
                # deterministic and cached: the same answer again
                assert dab.sched_select(mask, B, H, S, ctas) == pick
    # no SHIFT when its gang cannot be resident, odd causal N never SHIFT
    assert dab.sched_select("full", 1, 1, 128 * 64, 8) != "shift"
    assert dab.sched_select("causal", 1, 4, 384, 152) != "shift"
    # bad arguments
    assert lib.dab_sched_select(2, 1, 1, 256, 152) == -1
    assert lib.dab_sched_select(0, 1, 1, 200, 152) == -1
    assert lib.dab_sched_select(0, 1, 1, 256, 0) == -1




def test_sched_select_follows_the_model():
    """The pick is the model's argmin (ties to descending_q, then serial)."""
    for mask, B, H, S in (("causal", 2, 4, 2048), ("full", 1, 8, 4096), ("full", 2, 16, 8192),
                          ("full", 4, 16, 2048)):
        N = S // 128
        mk = {}
        for s in ("descending_q", "serial", "shift"):
            rc, m, _ = dab.dag_simulate(s, mask, N, B * H, 152, 1.0, 1.0, 1, ways=4)
            if rc == 0 and dab.sched_gang_size(s, mask, N) <= 152:
                mk[s] = m
        best = min(mk.values())
        expect = next(s for s in ("descending_q", "serial", "shift") if s in mk and mk[s] <= best * (1 + 1e-9))
        assert dab.sched_select(mask, B, H, S, 152) == expect


def test_sched_select_matches_the_measured_gb300_winners():
    """At the benchmark workload (B=2, H=16, S=8192, 152 CTAs) the GB300
    measurements have SHIFT fastest under both masks (full: 3.08 ms against
    3.16 for DESCENDING_Q); at B=4, H=16, S=2048 the full mask is a tie
    within 0.3 % and SHIFT is picked."""
    assert dab.sched_select("causal", 2, 16, 8192, 152) == "shift"
    assert dab.sched_select("full", 2, 16, 8192, 152) == "shift"
    assert dab.sched_select("full", 4, 16, 2048, 152) == "shift"
    assert dab.sched_select("causal", 4, 16, 2048, 152) == "shift"


@pytest.mark.parametrize("sched", ["serial", "descending_q", "shift"])
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("N", [1, 2, 5, 8, 16, 64])
def test_final_counts_of_the_accumulation_buffers(sched, mask, N):
    """The main kernel's tail converts dQ tile j once every buffer m < min(c, 4)
    holds (c - 1 - m) // 4 + 1 contributions (c contributors, rank r going to
    buffer r mod 4).  Counted here from the schedule's own ranks."""
    if sched == "shift" and mask == "causal" and N % 2:
        return
    W = 4
    for j in range(N):
        c = dab.sched_contributors(mask, N, j)
        assert c == (N if mask == "full" else j + 1)
        ranks = [dab.sched_rank(sched, mask, N, i, j) for i in range(N)
                 if mask == "full" or i <= j]
        assert sorted(ranks) == list(range(c))
        for m in range(min(c, W)):
            assert sum(1 for r in ranks if r % W == m) == (c - 1 - m) // W + 1
