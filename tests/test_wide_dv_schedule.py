"""A model of the backward's dV pass above d = 128 (csrc/fa_bwd_wide.cu,
wide_dv_kernel), run on the CPU.

Per 128-key tile the pass walks 128-query steps t. Q_t and dO_t each travel
through a ring of four shared-memory slots as two pieces (columns 0-127 and
128-255), in the order the products read them: Q_0, Q_1, then per step dO_t
and Q_{t+2}; a tile's pieces always take slots 0-1 or 2-3. One thread issues
S^T_0 and S^T_1 into two TMEM buffers (each half of the contraction once its
piece has landed), then per step [every warp has written P^T_t over S^T_t]
dV_t (one N = 256 product group over both dO pieces) and S^T_{t+2} into the
buffer dV_t has just read. Each piece's slot
goes back to the producer by a commit after the products that read it; the
step's LSE sits in one of three buffers (t % 3), loaded with Q_t. Eight warps
read S^T_t, write P^T_t and hand the LSE buffer back.

As for the other kernels, the roles run as coroutines with random latencies
over barriers with the hardware's parity rule. The model checks that every
product reads the piece and TMEM buffer of its own step, that no slot, TMEM
buffer or LSE buffer is overwritten while a reader still needs it, that no
parity wait passes on an older phase, that both pieces of dO_t sit in
adjacent slots, and that nothing deadlocks. Planted changes show what the
slot hand-back after the products, the issuer's wait for P^T, the order of
dV_t before S^T_{t+2} and the ring's four slots guard.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

WARPS = 8
SLOTS = 4
NVEC = 3


def piece_order(n):
    """(operand, step, half) in the order the producer loads and the products read."""
    out = []
    for t in range(min(n, 2)):
        out += [("Q", t, 0), ("Q", t, 1)]
    for t in range(n):
        out += [("dO", t, 0), ("dO", t, 1)]
        if t + 2 < n:
            out += [("Q", t + 2, 0), ("Q", t + 2, 1)]
    return out


def simulate(n, seed, *, release_after_products=True, issuer_waits_ready=True, dv_before_next_scores=True,
             warp_cycles=(100, 1500), slots=SLOTS):
    rng = random.Random(seed)
    errors = []
    full = [Barrier(1) for _ in range(slots)]
    empty = [Barrier(1) for _ in range(slots)]
    vec_full = [Barrier(1) for _ in range(NVEC)]
    vec_empty = [Barrier(WARPS) for _ in range(NVEC)]
    s_full = [Barrier(1), Barrier(1)]
    ready = [Barrier(WARPS), Barrier(WARPS)]
    o_final = Barrier(1)
    slot = [None] * slots            # piece held; None while a load is in flight
    inflight = [False] * slots
    vec = [None] * NVEC
    # TMEM buffer b, per warp's region (its 32 lanes, its half of the columns): ("S" | "P", step)
    buf = [[None] * WARPS, [None] * WARPS]
    dv_done = [-1]
    order = piece_order(n)
    pipe, events, clock = [], [], [0.0]

    def wait(bar, parity, who, phase=None):
        yield ("wait", lambda: bar.passes(parity))
        if phase is not None and bar.done < phase + 1:
            errors.append(f"{who}: parity wait for phase {phase} passed on an older phase")

    def later(delay, fn):
        heapq.heappush(events, (clock[0] + delay, rng.random(), ("call", fn)))

    # ------------------------------------------------------------ tensor core
    def tensor_core():
        while True:
            while not pipe:
                yield ("wait", lambda: bool(pipe))
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, t, h, i = op
            # S reads one piece (half h of Q_t); dV reads both pieces of dO_t, from slot i and i + 1
            reads = [(i, ("Q", t, h))] if kind == "S" else [(i, ("dO", t, 0)), (i + 1, ("dO", t, 1))]
            for j, want in reads:
                if j >= slots or slot[j] != want:
                    errors.append(f"{kind}({t}) read slot {j} holding {slot[j] if j < slots else None}, not {want}")
            b = t & 1
            if kind == "S" and h == 0 and t >= 2 and (dv_done[0] < t - 2 or buf[b] != [("P", t - 2)] * WARPS):
                errors.append(f"S({t}) overwrote buffer {b} holding {buf[b]} before dV({t - 2}) read it")
            if kind == "dV" and buf[b] != [("P", t)] * WARPS:
                errors.append(f"dV({t}) read buffer {b} holding {buf[b]}")
            yield ("delay", rng.uniform(100, 600) * len(reads))
            for j, want in reads:
                if j < slots and slot[j] != want:
                    errors.append(f"{kind}({t}): slot {j} changed under the product ({slot[j]})")
            if kind == "S" and h == 1:
                buf[b] = [("S", t)] * WARPS
            if kind == "dV":
                dv_done[0] = t

    # ------------------------------------------------------------ producer
    def producer():
        def land(i, what):
            def f():
                slot[i], inflight[i] = what, False
                full[i].complete_tx(1)
            return f

        def land_vec(x, t):
            def f():
                vec[x] = t
                vec_full[x].complete_tx(1)
            return f

        for k, what in enumerate(order):
            operand, t, h = what
            if operand == "Q" and h == 0:
                x = t % NVEC
                yield from wait(vec_empty[x], ((t // NVEC) & 1) ^ 1, "producer vec_empty")
                vec_full[x].expect_tx(1)
                vec_full[x].arrive()
                vec[x] = None
                later(rng.uniform(200, 2000), land_vec(x, t))
            i = k % slots
            yield from wait(empty[i], ((k // slots) & 1) ^ 1, "producer empty")
            if inflight[i]:
                errors.append(f"{what} loaded into slot {i} while a load was in flight")
            full[i].expect_tx(1)
            full[i].arrive()
            slot[i], inflight[i] = None, True
            later(rng.uniform(300, 4000), land(i, what))

    # ------------------------------------------------------------ issuer
    def issuer():
        k = [0]

        def take():
            i = k[0] % slots
            par = (k[0] // slots) & 1
            k[0] += 1
            yield from wait(full[i], par, "issuer full")
            return i

        def scores(t):
            for h in (0, 1):
                i = yield from take()
                if release_after_products:
                    pipe.extend([("S", t, h, i), ("commit", empty[i])])
                else:
                    pipe.extend([("commit", empty[i]), ("S", t, h, i)])
            pipe.append(("commit", s_full[t & 1]))

        def dv(t):
            i0 = yield from take()
            i1 = yield from take()
            if i1 != i0 + 1:
                errors.append(f"dO({t}) pieces in slots {i0} and {i1}: not adjacent")
            pipe.extend([("dV", t, 0, i0), ("commit", empty[i0]), ("commit", empty[i1])])

        for t in range(min(n, 2)):
            yield from scores(t)
        for t in range(n):
            if issuer_waits_ready:
                yield from wait(ready[t & 1], (t >> 1) & 1, "issuer ready", t >> 1)
            if dv_before_next_scores:
                yield from dv(t)
                if t + 2 < n:
                    yield from scores(t + 2)
            else:
                # the pieces are taken in the same order, the products queued the other way round
                base = len(pipe)
                yield from dv(t)
                dv_ops = pipe[base:]
                del pipe[base:]
                if t + 2 < n:
                    yield from scores(t + 2)
                pipe.extend(dv_ops)
        pipe.append(("commit", o_final))

    # ------------------------------------------------------------ warps
    def warp_role(w):
        for t in range(n):
            b, x = t & 1, t % NVEC
            yield from wait(s_full[b], (t >> 1) & 1, f"warp {w} s_full", t >> 1)
            yield from wait(vec_full[x], (t // NVEC) & 1, f"warp {w} vec_full", t // NVEC)
            if buf[b][w] != ("S", t):
                errors.append(f"warp {w} read S({t}) from buffer {b} holding {buf[b][w]}")
            if vec[x] != t:
                errors.append(f"warp {w} read LSE of step {t} from buffer {x} holding {vec[x]}")
            yield ("delay", rng.uniform(*warp_cycles))          # S read, P^T formed and written
            if buf[b][w] != ("S", t):
                errors.append(f"warp {w} wrote P^T({t}) over buffer {b} holding {buf[b][w]}")
            buf[b] = buf[b][:w] + [("P", t)] + buf[b][w + 1:]
            ready[b].arrive()
            vec_empty[x].arrive()
        yield from wait(o_final, 0, f"warp {w} o_final", 0)

    roles = [tensor_core(), producer(), issuer()] + [warp_role(w) for w in range(WARPS)]
    waiting, finished = {}, set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, rng.random(), ("run", i)))
    horizon = 40000.0 * (n + 4)
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
        if finished == set(range(1, len(roles))) and not pipe:
            break
    if finished != set(range(1, len(roles))):
        errors.append(f"deadlock: roles {sorted(set(range(1, len(roles))) - finished)} never finished")
    return errors


def test_piece_order():
    assert piece_order(0) == []
    assert piece_order(1) == [("Q", 0, 0), ("Q", 0, 1), ("dO", 0, 0), ("dO", 0, 1)]
    order = piece_order(5)
    assert len(order) == 20 and len(set(order)) == 20          # every piece once
    # Q_t always before dO_t, and Q_{t+2} right after dO_t
    for t in range(5):
        assert order.index(("Q", t, 1)) < order.index(("dO", t, 0))
    for t in range(3):
        assert order.index(("Q", t + 2, 0)) == order.index(("dO", t, 1)) + 1


@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 7, 12])
@pytest.mark.parametrize("warp_cycles", [(100, 1500), (20, 6000)])
def test_wide_dv_protocol_holds(n, warp_cycles):
    for seed in range(15):
        errs = simulate(n, seed, warp_cycles=warp_cycles)
        assert not errs, (n, seed, errs[:3])


def bad_runs(**kw):
    return sum(bool(simulate(n, seed, warp_cycles=(20, 6000), **kw)) for n in (3, 7, 12) for seed in range(12))


def test_slot_must_go_back_after_its_products():
    """A commit queued before the products hands the slot back as soon as the
    earlier products complete; the next piece can land under the product."""
    assert bad_runs(release_after_products=False) > 0


def test_dv_must_wait_for_every_warps_p():
    """dV_t reads P^T_t from TMEM; without the ready wait it reads S^T_t or a
    partly written P^T_t."""
    assert bad_runs(issuer_waits_ready=False) > 0


def test_dv_must_precede_the_scores_two_steps_ahead():
    """S^T_{t+2} goes into the buffer that holds P^T_t: dV_t has to be queued
    first."""
    assert bad_runs(dv_before_next_scores=False) > 0


def test_pieces_of_a_tile_share_an_even_slot_pair():
    """One product group reads both pieces of dO_t through one descriptor, so
    they must sit in adjacent slots. Four slots keep every tile's pair in slots
    0-1 or 2-3; five would split some."""
    assert bad_runs() == 0
    assert sum(bool(simulate(n, seed, slots=5)) for n in (3, 7, 12) for seed in range(4)) > 0
