"""A model of the paired dK/dV kernel's synchronisation, run on the CPU.

In the dense backward (csrc/fa_bwd.cu, bwd_dkdv_kernel with kPair) two CTAs
of a cluster own the adjacent key tiles 2p and 2p+1 and visit the same query
tiles in the same order; tile 2p first visits, in every head, the query tiles
only it sees ("unshared" steps). On a shared step each CTA keeps half of
dQ_i: the group owning the other half stages it over its own Q or dO region
and arrives remotely on the peer's "staged" barrier; the peer's owning group
reads it across the cluster, adds its own partial, stages the sum for its
reducer and arrives remotely on the first CTA's "read" barrier, after which
that CTA's reducer hands the region back to its producer. Unshared steps
reduce both halves locally, as the unpaired kernel does.

Each CTA runs the roles of the unpaired model (tests/test_dkdv_schedule.py)
as coroutines with random latencies over barriers with the hardware's parity
rule. The model checks that
  * every MMA and every warp reads the data of its own step,
  * an owning group reads the peer's staged partial of the same shared step,
    fully written, and no load or later staging overwrites a region that the
    peer has not finished reading,
  * no region is reloaded while its staged dQ is still being reduced,
  * no parity wait (local or cross-CTA) passes on an older phase,
  * nothing deadlocks.
Planted changes show that the reducer's wait for the peer's read, the
owner's wait for the peer's staging, the separate phase count of the
other half's staged barriers, and two exchange barriers per kind (instead
of one) are each needed.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

GROUPS, WARPS_PER_GROUP, BOXES = 2, 4, 2


def step_lists(G, tph1, extra):
    """Per CTA: list of (head, tile, shared index k or None). Tile numbers are
    relative: tile 2p+1 sees tiles extra .. extra + tph1 - 1, tile 2p sees
    0 .. extra + tph1 - 1."""
    s0, s1 = [], []
    for h in range(G):
        for it in range(extra + tph1):
            k = h * tph1 + it - extra if it >= extra else None
            s0.append((h, it, k))
            if k is not None:
                s1.append((h, it, k))
    return [s0, s1]


def simulate(G, tph1, extra, seed, *, reducer_waits_peer_read=True, owner_waits_staged=True,
             other_half_counts=True, xbarriers=2, warp_cycles=(200, 1500), ghost=False):
    rng = random.Random(seed)
    errors = []
    lists = step_lists(G, tph1, extra)
    if ghost:                         # tile 2p+1 does not exist: every step of tile 2p is its own
        lists = [[(h, it, None) for h, it, _ in lists[0]], []]
    pos = [{k: i for i, (_, _, k) in enumerate(lst) if k is not None} for lst in lists]
    pipe = [[], []]
    events = []
    clock = [0.0]

    def later(delay, fn):
        heapq.heappush(events, (clock[0] + delay, rng.random(), ("call", fn)))

    def wait(bar, parity, who, phase=None):
        yield ("wait", lambda: bar.passes(parity))
        if phase is not None and bar.done < phase + 1:
            errors.append(f"{who}: parity wait for phase {phase} passed on an older phase")

    class CTA:
        pass

    ctas = [CTA(), CTA()]
    for c, x in enumerate(ctas):
        x.steps = lists[c]
        x.n = len(x.steps)
        x.kv_full = Barrier(1)
        x.q_full, x.do_full = [Barrier(1), Barrier(1)], [Barrier(1), Barrier(1)]
        x.q_empty, x.do_empty = [Barrier(1), Barrier(1)], [Barrier(1), Barrier(1)]
        x.dq_staged = {(g, st, bx): Barrier(WARPS_PER_GROUP) for g in range(GROUPS) for st in range(2)
                       for bx in range(BOXES)}
        x.s_full, x.dp_full, x.dq_full, x.o_final = Barrier(1), Barrier(1), Barrier(1), Barrier(1)
        nthreads = GROUPS * WARPS_PER_GROUP
        x.p_ready, x.ds_ready = Barrier(nthreads), Barrier(nthreads)
        x.dq_free = Barrier(nthreads + 1)
        x.x_staged = [Barrier(WARPS_PER_GROUP) for _ in range(xbarriers)]
        x.x_read = [Barrier(WARPS_PER_GROUP) for _ in range(xbarriers)]
        # region[(g, st)]: ("Q"/"dO", step) loaded, ("part", step, warps) staged partial,
        # ("sum", step, warps) summed half, None while a load is in flight
        x.region = {(g, st): ("empty", -1) for g in range(GROUPS) for st in range(2)}
        x.vec = [None, None]
        x.reading = {}                 # (g, st) -> outstanding readers (TMA reductions, peer reads)
        x.tmem_s, x.tmem_dp = None, None
        x.p_written, x.ds_buf, x.read_dp, x.read_dq = {}, {}, {}, {}
        x.done = {"dV": -1, "dK": -1, "dQ": -1, "S": -1, "dP": -1}

    def xbar(lst, k):
        return lst[k % xbarriers]

    def xpar(k):
        return (k // xbarriers) & 1

    # ------------------------------------------------------------ per-CTA roles
    def tensor_core(c):
        x = ctas[c]
        while True:
            while not pipe[c]:
                yield ("wait", lambda: bool(pipe[c]))
            op = pipe[c].pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, step = op
            st = step & 1
            if kind in ("S", "dK") and x.region[(0, st)] != ("Q", step):
                errors.append(f"cta {c} {kind}({step}) read Q region {st} holding {x.region[(0, st)]}")
            if kind in ("dP", "dV") and x.region[(1, st)] != ("dO", step):
                errors.append(f"cta {c} {kind}({step}) read dO region {st} holding {x.region[(1, st)]}")
            if kind == "dV" and x.tmem_s != ("P", step):
                errors.append(f"cta {c} dV({step}) read TMEM S holding {x.tmem_s}")
            if kind in ("dK", "dQ") and len(x.ds_buf.get(step, ())) < GROUPS * WARPS_PER_GROUP:
                errors.append(f"cta {c} {kind}({step}) read dS^T before every warp wrote it")
            if kind == "dP" and step > 0 and len(x.read_dq.get(step - 1, ())) < GROUPS * WARPS_PER_GROUP:
                errors.append(f"cta {c} dP({step}) overwrote dQ({step - 1}) before every warp read it")
            yield ("delay", rng.uniform(100, 400))
            x.done[kind] = step
            if kind == "S":
                x.tmem_s = ("S", step)
            elif kind in ("dP", "dQ"):
                x.tmem_dp = (kind, step)

    def producer(c):
        x = ctas[c]

        def land(g, st, step):
            def f():
                x.region[(g, st)] = ("Q" if g == 0 else "dO", step)
                if g == 0:
                    x.vec[st] = step
                (x.q_full if g == 0 else x.do_full)[st].complete_tx(1)
            return f

        x.kv_full.expect_tx(1)
        x.kv_full.arrive()
        later(rng.uniform(300, 3000), lambda: x.kv_full.complete_tx(1))
        for step in range(x.n):
            st, par = step & 1, ((step >> 1) & 1) ^ 1
            for g, empty, full in ((0, x.q_empty, x.q_full), (1, x.do_empty, x.do_full)):
                yield from wait(empty[st], par, f"cta {c} producer empty")
                if x.reading.get((g, st), 0):
                    errors.append(f"cta {c} load of step {step} into region {(g, st)} while it was being read")
                if x.region[(g, st)] is None:
                    errors.append(f"cta {c} load of step {step} into region {(g, st)} over a load in flight")
                full[st].expect_tx(1)
                full[st].arrive()
                x.region[(g, st)] = None
                if g == 0:
                    x.vec[st] = None
                later(rng.uniform(300, 3000), land(g, st, step))

    def issuer(c):
        x = ctas[c]
        n = x.n
        if n == 0:
            pipe[c].append(("commit", x.o_final))
            return
        yield from wait(x.kv_full, 0, f"cta {c} issuer kv")
        yield from wait(x.q_full[0], 0, f"cta {c} issuer q", 0)
        pipe[c].extend([("S", 0), ("commit", x.s_full)])
        yield from wait(x.do_full[0], 0, f"cta {c} issuer do", 0)
        pipe[c].extend([("dP", 0), ("commit", x.dp_full)])
        for step in range(n):
            yield from wait(x.p_ready, step & 1, f"cta {c} issuer p_ready", step)
            pipe[c].append(("dV", step))
            yield from wait(x.ds_ready, step & 1, f"cta {c} issuer ds_ready", step)
            pipe[c].extend([("dK", step), ("dQ", step), ("commit", x.dq_full)])
            if step + 1 < n:
                sn = (step + 1) & 1
                yield from wait(x.q_full[sn], ((step + 1) >> 1) & 1, f"cta {c} issuer q", (step + 1) >> 1)
                pipe[c].extend([("S", step + 1), ("commit", x.s_full)])
                yield from wait(x.dq_free, step & 1, f"cta {c} issuer dq_free", step)
                pipe[c].extend([("dP", step + 1), ("commit", x.dp_full)])
        pipe[c].append(("commit", x.o_final))

    def watcher(c):
        x = ctas[c]
        if x.n > 0:
            yield from wait(x.do_full[0], 0, f"cta {c} watcher", 0)
        for step in range(x.n - 1):
            sn = (step + 1) & 1
            yield from wait(x.do_full[sn], ((step + 1) >> 1) & 1, f"cta {c} watcher do")
            if step > 0:
                yield from wait(x.dq_free, (step - 1) & 1, f"cta {c} watcher gate", step - 1)
            x.dq_free.arrive()

    def reduce_box(c, g, st, step, pending):
        x = ctas[c]
        want = "sum" if x.steps[step][2] is not None else "part"
        r = x.region[(g, st)]
        if r is None or r[0] != want or r[1] != step or len(r[2]) < WARPS_PER_GROUP:
            errors.append(f"cta {c} reducer read half {g} of step {step} from {(g, st)} holding {r}")
        x.reading[(g, st)] = x.reading.get((g, st), 0) + 1
        fin = [False]

        def end():
            x.reading[(g, st)] -= 1
            fin[0] = True
        later(rng.uniform(200, 2000), end)
        pending.append(fin)

    def reducer(c):
        x = ctas[c]
        other_uses = [0, 0]
        for step, (_, _, k) in enumerate(x.steps):
            st = step & 1
            if k is not None:
                go = c
                pend = []
                for bx in range(BOXES):
                    yield from wait(x.dq_staged[(go, st, bx)], (step >> 1) & 1, f"cta {c} reducer staged", step >> 1)
                    reduce_box(c, go, st, step, pend)
                if go == 1:
                    if reducer_waits_peer_read:
                        yield from wait(xbar(x.x_read, k), xpar(k), f"cta {c} reducer x_read", k // xbarriers)
                    x.q_empty[st].arrive()
                yield ("wait", lambda p=pend: all(f[0] for f in p))
                (x.do_empty if go else x.q_empty)[st].arrive()
                if go == 0:
                    if reducer_waits_peer_read:
                        yield from wait(xbar(x.x_read, k), xpar(k), f"cta {c} reducer x_read", k // xbarriers)
                    x.do_empty[st].arrive()
                continue
            pend = {0: [], 1: []}
            for g in range(GROUPS):
                if g != c and other_half_counts:
                    par, ph = other_uses[st] & 1, other_uses[st]
                else:
                    par, ph = (step >> 1) & 1, step >> 1
                for bx in range(BOXES):
                    yield from wait(x.dq_staged[(g, st, bx)], par, f"cta {c} reducer staged ({g})", ph)
                    reduce_box(c, g, st, step, pend[g])
            other_uses[st] += 1
            yield ("wait", lambda p=pend[0]: all(f[0] for f in p))
            x.q_empty[st].arrive()
            yield ("wait", lambda p=pend[1]: all(f[0] for f in p))
            x.do_empty[st].arrive()

    def warp_role(c, g, w):
        x = ctas[c]
        y = ctas[1 - c]
        me = (c, g, w)
        nthreads = GROUPS * WARPS_PER_GROUP
        for step, (_, _, k) in enumerate(x.steps):
            st = step & 1
            yield from wait(x.q_full[st], (step >> 1) & 1, f"warp {me} q", step >> 1)
            yield from wait(x.s_full, step & 1, f"warp {me} s_full", step)
            if x.tmem_s != ("S", step) and not (x.tmem_s == ("P", step) and me not in x.p_written.get(step, ())):
                errors.append(f"warp {me} read S^T({step}) from TMEM holding {x.tmem_s}")
            if x.vec[st] != step:
                errors.append(f"warp {me} read LSE of step {step} from stage {st} holding {x.vec[st]}")
            yield ("delay", rng.uniform(*warp_cycles))
            x.p_written.setdefault(step, set()).add(me)
            if len(x.p_written[step]) == nthreads:
                x.tmem_s = ("P", step)
            x.p_ready.arrive()
            yield from wait(x.dp_full, step & 1, f"warp {me} dp_full", step)
            if x.tmem_dp != ("dP", step):
                errors.append(f"warp {me} read dP^T({step}) from TMEM holding {x.tmem_dp}")
            x.read_dp.setdefault(step, set()).add(me)
            if step > 0 and (x.done["dK"] < step - 1 or x.done["dQ"] < step - 1):
                errors.append(f"warp {me} wrote dS^T({step}) before dK / dQ of step {step - 1} read the last one")
            yield ("delay", rng.uniform(*warp_cycles))
            x.ds_buf.setdefault(step, set()).add(me)
            x.ds_ready.arrive()
            yield from wait(x.dq_full, step & 1, f"warp {me} dq_full", step)
            if x.tmem_dp != ("dQ", step):
                errors.append(f"warp {me} read dQ({step}) from TMEM holding {x.tmem_dp}")
            x.read_dq.setdefault(step, set()).add(me)
            x.dq_free.arrive()
            reg = x.region[(g, st)]
            if reg is None or reg[1] != step or reg[0] not in ("Q", "dO", "part", "sum"):
                errors.append(f"warp {me} staged dQ({step}) over region {(g, st)} holding {reg}")
            if x.done["dK"] < step or x.done["dV"] < step:
                errors.append(f"warp {me} staged dQ({step}) before dK / dV of the step read its region")
            if k is not None and g == c:
                # owner: the peer's partial of this half, then the sum (the
                # warp may be slow to get there: TMEM read-out, scheduling)
                yield ("delay", rng.uniform(0, 20000) if rng.random() < 0.2 else rng.uniform(0, 100))
                if owner_waits_staged:
                    yield from wait(xbar(x.x_staged, k), xpar(k), f"warp {me} x_staged", k // xbarriers)
                sp = pos[1 - c][k] & 1
                pr = y.region[(g, sp)]
                if pr is None or pr[0] != "part" or pr[1] != pos[1 - c][k] or len(pr[2]) < WARPS_PER_GROUP:
                    errors.append(f"warp {me} read the peer's half for shared step {k} from {(g, sp)} holding {pr}")
                y.reading[(g, sp)] = y.reading.get((g, sp), 0) + 1
                yield ("delay", rng.uniform(50, 600))
                y.reading[(g, sp)] -= 1
                pr2 = y.region[(g, sp)]
                if pr2 is None or pr2[0] != "part" or pr2[1] != pos[1 - c][k]:
                    errors.append(f"warp {me}: the peer's half of shared step {k} changed while being read: {pr2}")
                for bx in range(BOXES):
                    yield ("delay", rng.uniform(20, 200))
                    cur = x.region[(g, st)]
                    ws = cur[2] if cur is not None and cur[0] == "sum" and cur[1] == step else set()
                    x.region[(g, st)] = ("sum", step, ws | {me})
                    x.dq_staged[(g, st, bx)].arrive()
                xbar(y.x_read, k).arrive()
                continue
            for bx in range(BOXES):
                yield ("delay", rng.uniform(20, 200))
                cur = x.region[(g, st)]
                ws = cur[2] if cur is not None and cur[0] == "part" and cur[1] == step else set()
                x.region[(g, st)] = ("part", step, ws | {me})
                if k is None:
                    x.dq_staged[(g, st, bx)].arrive()
            if k is not None:
                xbar(y.x_staged, k).arrive()
        yield from wait(x.o_final, 0, f"warp {me} o_final", 0)

    roles = []
    for c in range(2):
        roles += [tensor_core(c), producer(c), issuer(c), watcher(c), reducer(c)]
        roles += [warp_role(c, g, w) for g in range(GROUPS) for w in range(WARPS_PER_GROUP)]
    daemons = {0, 5 + GROUPS * WARPS_PER_GROUP}            # the two tensor cores
    waiting, finished = {}, set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, rng.random(), ("run", i)))
    horizon = 40000.0 * (len(lists[0]) + 4)
    others = set(range(len(roles))) - daemons
    while events and clock[0] < horizon:
        clock[0], _, (what, arg) = heapq.heappop(events)
        if what == "call":
            arg()
            continue
        i = arg
        if i in finished:
            continue
        try:
            y = waiting.pop(i) if i in waiting else next(roles[i])
            while True:
                if y[0] == "delay":
                    heapq.heappush(events, (clock[0] + y[1], rng.random(), ("run", i)))
                    break
                if y[1]():
                    y = next(roles[i])
                    continue
                waiting[i] = y
                heapq.heappush(events, (clock[0] + rng.uniform(20, 200), rng.random(), ("run", i)))
                break
        except StopIteration:
            finished.add(i)
        except AssertionError as e:
            errors.append(str(e))
            return errors
        if others <= finished and not pipe[0] and not pipe[1]:
            break
    if not others <= finished:
        errors.append(f"deadlock: roles {sorted(others - finished)} never finished")
    return errors


CASES = [(1, 1, 1), (1, 3, 1), (2, 4, 1), (3, 2, 1), (2, 5, 0), (2, 3, 2), (1, 6, 0), (4, 1, 1), (2, 0, 2)]


@pytest.mark.parametrize("G,tph1,extra", CASES)
@pytest.mark.parametrize("warp_cycles", [(200, 1500), (50, 5000)])
def test_pair_protocol_holds(G, tph1, extra, warp_cycles):
    for seed in range(12):
        errs = simulate(G, tph1, extra, seed, warp_cycles=warp_cycles)
        assert not errs, (G, tph1, extra, seed, errs[:3])


@pytest.mark.parametrize("G,n", [(1, 3), (2, 4)])
def test_pair_with_missing_second_tile_runs_alone(G, n):
    """An odd number of key tiles: the last CTA's peer has no keys and every
    step is unshared."""
    for seed in range(10):
        errs = simulate(G, n, 1, seed, ghost=True)
        assert not errs, (seed, errs[:3])


def bad_runs(**kw):
    return sum(bool(simulate(G, t, e, seed, warp_cycles=(50, 5000), **kw))
               for G, t, e in ((2, 4, 1), (3, 3, 1), (2, 5, 2)) for seed in range(10))


def test_reducer_must_wait_for_the_peer_read():
    """Handing the staged half back before the peer has read it lets the next
    load overwrite it while the peer reads."""
    assert bad_runs(reducer_waits_peer_read=False) > 0


def test_owner_must_wait_for_the_peer_staging():
    assert bad_runs(owner_waits_staged=False) > 0


def test_other_half_needs_its_own_phase_count():
    """The staged barriers of the half a CTA does not own complete on unshared
    steps only: waiting on them with the step's parity mistakes phases."""
    assert bad_runs(other_half_counts=False) > 0


def test_one_exchange_barrier_per_kind_is_not_enough():
    assert bad_runs(xbarriers=1) > 0
