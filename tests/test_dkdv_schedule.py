"""A model of the dK/dV backward kernel's synchronisation, run on the CPU.

The kernel (csrc/fa_bwd.cu, bwd_dkdv_kernel) owns one 128-key tile and walks
the query tiles ("steps") of the heads that read it. Per step the tensor core
computes S^T = K Q^T into TMEM, the softmax-gradient warps turn it into P^T
in place, the tensor core runs dV += P^T dO, computes dP^T = V dO^T into a
second TMEM region, the warps write dS^T to shared memory, the tensor core
runs dQ = dS K into the dP^T columns and then dK += dS^T Q, the warps read dQ
out and stage its two fp32 halves over the step's own Q (once dK, its last
reader, is done) and dO regions (two stages of each), and a reducer warp adds
them into global memory with TMA bulk reductions and hands each region back
to the producer. A watcher folds
"dO of the next step landed" into the dQ-read-out barrier.

As for the forward kernels, the roles run as coroutines with random
latencies over barriers with the hardware's parity rule; the model checks
that every MMA and every warp reads the data of its own step, that no
region, TMEM column group or the dS^T buffer is overwritten while a reader
still needs it, and that no parity wait passes on an older phase. Planted
changes show what the watcher's first wait, the issuer's wait for dQ to be
read out, the reducer's wait for its reads and group 0's wait for dK guard.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

GROUPS, WARPS_PER_GROUP, BOXES = 2, 4, 2


def simulate(n, seed, *, watcher_first_wait=True, issuer_waits_dq_free=True, reducer_waits_reads=True,
             group0_waits_dk=True, warp_cycles=(200, 1500)):
    """Errors seen in one run of n steps (query tiles) for one key tile."""
    rng = random.Random(seed)
    errors = []
    warps = [(g, w) for g in range(GROUPS) for w in range(WARPS_PER_GROUP)]
    nthreads = len(warps)                         # one arrival per warp stands for its 32 threads

    kv_full = Barrier(1)
    q_full = [Barrier(1), Barrier(1)]
    do_full = [Barrier(1), Barrier(1)]
    q_empty = [Barrier(1), Barrier(1)]
    do_empty = [Barrier(1), Barrier(1)]
    dq_staged = {(g, st, bx): Barrier(WARPS_PER_GROUP) for g in range(GROUPS) for st in range(2)
                 for bx in range(BOXES)}
    s_full, dp_full, dq_full, o_final = Barrier(1), Barrier(1), Barrier(1), Barrier(1)
    dk_done = Barrier(1)
    p_ready, ds_ready = Barrier(nthreads), Barrier(nthreads)
    dq_free = Barrier(nthreads + 1)               # + the watcher

    # contents: region[st] = (kind, step) with kind "Q"/"dQ0" or "dO"/"dQ1"; None while a load is in flight
    q_reg, do_reg, vec = [None, None], [None, None], [None, None]
    q_load_inflight, do_load_inflight = [False, False], [False, False]
    reduce_reads = {}                              # (st, g) -> outstanding TMA reduce reads of that region
    staged = {}                                    # (g, st, bx, step) -> warps that wrote the box
    tmem_s = None                                  # ("S" | "P", step)
    p_written = {}
    tmem_dp = None                                 # ("dP" | "dQ", step)
    ds_buf = {}                                    # step -> warps that wrote dS^T
    read_dp = {}                                   # step -> warps that read dP^T
    read_dq = {}                                   # step -> warps that read dQ
    done = {"dV": -1, "dK": -1, "dQ": -1, "S": -1, "dP": -1}
    pipe = []
    clock = [0.0]
    events = []

    def wait(bar, parity, who, phase=None):
        yield ("wait", lambda: bar.passes(parity))
        if phase is not None and bar.done < phase + 1:
            errors.append(f"{who}: parity wait for phase {phase} passed on an older phase")

    def later(delay, fn):
        heapq.heappush(events, (clock[0] + delay, rng.random(), ("call", fn)))

    # ------------------------------------------------------------ tensor core
    def tensor_core():
        nonlocal tmem_s, tmem_dp
        while True:
            while not pipe:
                yield ("wait", lambda: bool(pipe))
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, step = op
            st = step & 1
            if kind == "S":
                if q_reg[st] != ("Q", step):
                    errors.append(f"S({step}) read Q region {st} holding {q_reg[st]}")
                if step > 0 and done["dV"] < step - 1:
                    errors.append(f"S({step}) overwrote P^T({step - 1}) before dV read it")
            elif kind == "dP":
                if do_reg[st] != ("dO", step):
                    errors.append(f"dP({step}) read dO region {st} holding {do_reg[st]}")
                if step > 0 and len(read_dq.get(step - 1, ())) < nthreads:
                    errors.append(f"dP({step}) overwrote dQ({step - 1}) before every warp read it")
            elif kind == "dV":
                if tmem_s != ("P", step):
                    errors.append(f"dV({step}) read TMEM S columns holding {tmem_s}")
                if do_reg[st] != ("dO", step):
                    errors.append(f"dV({step}) read dO region {st} holding {do_reg[st]}")
            elif kind == "dK":
                if len(ds_buf.get(step, ())) < nthreads:
                    errors.append(f"dK({step}) read dS^T before every warp wrote it")
                if q_reg[st] != ("Q", step):
                    errors.append(f"dK({step}) read Q region {st} holding {q_reg[st]}")
            elif kind == "dQ":
                if len(ds_buf.get(step, ())) < nthreads:
                    errors.append(f"dQ({step}) read dS^T before every warp wrote it")
                if len(read_dp.get(step, ())) < nthreads:
                    errors.append(f"dQ({step}) overwrote dP^T({step}) before every warp read it")
            yield ("delay", rng.uniform(100, 400))
            done[kind] = step
            if kind == "S":
                tmem_s = ("S", step)
            elif kind == "dP":
                tmem_dp = ("dP", step)
            elif kind == "dQ":
                tmem_dp = ("dQ", step)

    # ------------------------------------------------------------ producer
    def producer():
        def land_q(st, step):
            def f():
                q_reg[st], vec[st], q_load_inflight[st] = ("Q", step), step, False
                q_full[st].complete_tx(1)
            return f

        def land_do(st, step):
            def f():
                do_reg[st], do_load_inflight[st] = ("dO", step), False
                do_full[st].complete_tx(1)
            return f

        kv_full.expect_tx(1)
        kv_full.arrive()
        later(rng.uniform(300, 3000), lambda: kv_full.complete_tx(1))
        for step in range(n):
            st, par = step & 1, ((step >> 1) & 1) ^ 1
            yield from wait(q_empty[st], par, "producer q_empty")
            if reduce_reads.get((st, 0), 0) or q_load_inflight[st]:
                errors.append(f"Q({step}) loaded into region {st} while it was still being read")
            if step >= 2 and (done["dK"] < step - 2 or done["S"] < step - 2):
                errors.append(f"Q({step}) loaded over Q({step - 2}) before its MMAs ran")
            q_full[st].expect_tx(1)
            q_full[st].arrive()
            q_reg[st], vec[st], q_load_inflight[st] = None, None, True
            later(rng.uniform(300, 3000), land_q(st, step))
            yield from wait(do_empty[st], par, "producer do_empty")
            if reduce_reads.get((st, 1), 0) or do_load_inflight[st]:
                errors.append(f"dO({step}) loaded into region {st} while it was still being read")
            do_full[st].expect_tx(1)
            do_full[st].arrive()
            do_reg[st], do_load_inflight[st] = None, True
            later(rng.uniform(300, 3000), land_do(st, step))

    # ------------------------------------------------------------ issuer
    def issuer():
        if n == 0:
            pipe.append(("commit", o_final))           # no step: dK = dV = 0, still one final commit
            return
        yield from wait(kv_full, 0, "issuer kv")
        yield from wait(q_full[0], 0, "issuer q", 0)
        pipe.extend([("S", 0), ("commit", s_full)])
        yield from wait(do_full[0], 0, "issuer do", 0)
        pipe.extend([("dP", 0), ("commit", dp_full)])
        for step in range(n):
            yield from wait(p_ready, step & 1, "issuer p_ready", step)
            pipe.append(("dV", step))
            yield from wait(ds_ready, step & 1, "issuer ds_ready", step)
            # dQ first (its read-out is on the warps' critical path), then dK
            pipe.extend([("dQ", step), ("commit", dq_full), ("dK", step), ("commit", dk_done)])
            if step + 1 < n:
                sn = (step + 1) & 1
                yield from wait(q_full[sn], ((step + 1) >> 1) & 1, "issuer q", (step + 1) >> 1)
                pipe.extend([("S", step + 1), ("commit", s_full)])
                if issuer_waits_dq_free:
                    yield from wait(dq_free, step & 1, "issuer dq_free", step)
                else:
                    yield from wait(do_full[sn], ((step + 1) >> 1) & 1, "issuer do", (step + 1) >> 1)
                pipe.extend([("dP", step + 1), ("commit", dp_full)])
        pipe.append(("commit", o_final))

    # ------------------------------------------------------------ watcher
    def watcher():
        if n > 0 and watcher_first_wait:
            yield from wait(do_full[0], 0, "watcher", 0)
        for step in range(n - 1):
            sn = (step + 1) & 1
            yield from wait(do_full[sn], ((step + 1) >> 1) & 1, "watcher do")
            if do_reg[sn] != ("dO", step + 1):
                errors.append(f"watcher passed dO({step + 1}) while region {sn} held {do_reg[sn]}")
            if step > 0:
                yield from wait(dq_free, (step - 1) & 1, "watcher gate", step - 1)
            dq_free.arrive()

    # ------------------------------------------------------------ reducer
    def reducer():
        for step in range(n):
            st = step & 1
            pending = {0: [], 1: []}
            for g in range(GROUPS):
                for bx in range(BOXES):
                    yield from wait(dq_staged[(g, st, bx)], (step >> 1) & 1, "reducer staged", step >> 1)
                    if len(staged.get((g, st, bx, step), ())) < WARPS_PER_GROUP:
                        errors.append(f"reducer read dQ half {g} box {bx} of step {step} before it was written")
                    reduce_reads[(st, g)] = reduce_reads.get((st, g), 0) + 1
                    finish = [False]

                    def end(st=st, g=g, finish=finish):
                        reduce_reads[(st, g)] -= 1
                        finish[0] = True
                    later(rng.uniform(200, 2000), end)
                    pending[g].append(finish)
            if reducer_waits_reads:
                yield ("wait", lambda p=pending[0]: all(f[0] for f in p))
            q_empty[st].arrive()
            if reducer_waits_reads:
                yield ("wait", lambda p=pending[1]: all(f[0] for f in p))
            do_empty[st].arrive()

    # ------------------------------------------------------------ softmax-gradient warps
    def warp_role(g, w):
        me = (g, w)
        for step in range(n):
            st = step & 1
            yield from wait(q_full[st], (step >> 1) & 1, f"warp {me} q", step >> 1)
            yield from wait(s_full, step & 1, f"warp {me} s_full", step)
            if tmem_s != ("S", step) and not (tmem_s == ("P", step) and me not in p_written.get(step, ())):
                errors.append(f"warp {me} read S^T({step}) from TMEM holding {tmem_s}")
            if vec[st] != step:
                errors.append(f"warp {me} read LSE of step {step} from stage {st} holding step {vec[st]}")
            yield ("delay", rng.uniform(*warp_cycles))
            p_written.setdefault(step, set()).add(me)
            if len(p_written[step]) == nthreads:
                tmem_s_set(("P", step))
            p_ready.arrive()
            yield from wait(dp_full, step & 1, f"warp {me} dp_full", step)
            if tmem_dp != ("dP", step):
                errors.append(f"warp {me} read dP^T({step}) from TMEM holding {tmem_dp}")
            if vec[st] != step:
                errors.append(f"warp {me} read D of step {step} from stage {st} holding step {vec[st]}")
            read_dp.setdefault(step, set()).add(me)
            if step > 0 and (done["dK"] < step - 1 or done["dQ"] < step - 1):
                errors.append(f"warp {me} wrote dS^T({step}) before dK / dQ of step {step - 1} read the last one")
            yield ("delay", rng.uniform(*warp_cycles))
            ds_buf.setdefault(step, set()).add(me)
            ds_ready.arrive()
            yield from wait(dq_full, step & 1, f"warp {me} dq_full", step)
            # the read-out itself takes time (TMEM loads, scheduling); dQ must
            # still be there at its end
            yield ("delay", rng.uniform(0, 3000) if rng.random() < 0.2 else rng.uniform(0, 200))
            if tmem_dp != ("dQ", step):
                errors.append(f"warp {me} read dQ({step}) from TMEM holding {tmem_dp}")
            read_dq.setdefault(step, set()).add(me)
            dq_free.arrive()
            if g == 0 and group0_waits_dk:
                # Q_i is still read by dK_i, issued after dQ_i
                yield from wait(dk_done, step & 1, f"warp {me} dk_done", step)
            # stage this group's dQ half over the step's own Q (g = 0) or dO (g = 1) region
            reg = q_reg if g == 0 else do_reg
            if reg[st] is None or reg[st][1] != step:
                errors.append(f"warp {me} staged dQ({step}) over region {st} holding {reg[st]}")
            # the region's last MMA readers: S^T and dK read Q_i, dP^T and dV read dO_i
            readers = ("S", "dK") if g == 0 else ("dP", "dV")
            if any(done[k] < step for k in readers):
                errors.append(f"warp {me} staged dQ({step}) before {readers} of the step read its region")
            for bx in range(BOXES):
                yield ("delay", rng.uniform(20, 200))
                staged.setdefault((g, st, bx, step), set()).add(me)
                dq_staged[(g, st, bx)].arrive()
        yield from wait(o_final, 0, f"warp {me} o_final", 0)
        if n == 0:
            # nothing waited for K and V, whose buffers stage dK and dV: let them land
            yield from wait(kv_full, 0, f"warp {me} kv", 0)

    def tmem_s_set(v):
        nonlocal tmem_s
        tmem_s = v

    roles = [tensor_core(), producer(), issuer(), watcher(), reducer()] + [warp_role(g, w) for g, w in warps]
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


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 9])
@pytest.mark.parametrize("warp_cycles", [(200, 1500), (50, 5000)])
def test_dkdv_protocol_holds(n, warp_cycles):
    for seed in range(20):
        errs = simulate(n, seed, warp_cycles=warp_cycles)
        assert not errs, (n, seed, errs[:3])


def bad_runs(**kw):
    return sum(bool(simulate(n, seed, warp_cycles=(50, 5000), **kw)) for n in (3, 5, 9) for seed in range(15))


def test_reducer_must_wait_for_its_reads():
    """Handing a region back before the bulk reductions have read it lets the
    next Q or dO load overwrite the staged dQ."""
    assert bad_runs(reducer_waits_reads=False) > 0


def test_issuer_must_wait_for_dq_read_out():
    """dP^T of the next step goes into the columns dQ occupies."""
    assert bad_runs(issuer_waits_dq_free=False) > 0


def test_group0_must_wait_for_dk_before_staging_over_q():
    """dK_i runs after dQ_i and reads Q_i: staging dQ_i's first half over Q_i
    before dK_i has completed would corrupt dK."""
    assert bad_runs(group0_waits_dk=False) > 0


def test_watcher_must_observe_the_first_do_load():
    """Parity waits only tell phase k from phase k-1: without observing dO_0,
    the watcher can take dO_2's stage for landed while dO_0 is in flight."""
    assert bad_runs(watcher_first_wait=False) > 0
