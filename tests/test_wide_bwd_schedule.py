"""A model of the three-pass backward's dK and dQ passes, run on the CPU.

The kernels (csrc/fa_bwd_wide.cu, wide_dk_kernel and wide_dq_kernel) walk
128-row steps s over two 64 KB shared-memory slots. Each step has an operand
A (Q_s in the dK pass, K_s in the dQ pass), read by the scores S_s and by the
accumulate (dK += dS^T Q_s, dQ += dS K_s), and an operand B (dO_s or V_s),
read only by dP_s. A always lands in slot 0 and B in slot 1. Each pass keeps
one operand in TMEM as the A operand of the scores (K in the dK pass, Q in
the dQ pass): it lands in slot 0, every warp copies its rows, and only then
does slot 0 take A. dP and S share one 128-column TMEM region: one thread
issues dP_0, then per step [every warp has read dP_s, A_s landed] S_s,
[dS_s written] the accumulate, which frees A's slot, and [B_{s+1} landed]
dP_{s+1}; B's slot is free once dP_s completes, early in the step. dS has
one shared-memory buffer; the dK pass double-buffers the step's LSE and D.
Eight warps, two per TMEM lane quarter (one per half of the score columns),
read dP into registers, then read S, form P and write dS.

As for the other kernels, the roles run as coroutines with random latencies
over barriers with the hardware's parity rule. The model checks that every
product and every warp reads the data of its own step, that no slot, TMEM
buffer, dS buffer or vector buffer is overwritten while a reader still needs
it, and that no parity wait passes on an older phase. Planted changes show
what the accumulate's release of A's slot, the warps' wait for dP, the
issuer's wait for every warp's read of dP and the producer's wait for the
TMEM copy guard; the vector buffer's release point turns out to be implied
by the slot order.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

WARPS = 8


def simulate(n, seed, *, dk_pass=True, release_a_after_acc=True, warps_wait_dp=True, vec_release_last=True,
             producer_waits_copy=True, issuer_waits_s_read=True, warp_cycles=(100, 1500)):
    """Errors seen in one run of n steps of one CTA."""
    rng = random.Random(seed)
    errors = []
    full = [Barrier(1), Barrier(1)]
    empty = [Barrier(1), Barrier(1)]
    s_full, s_read, dp_full = Barrier(1), Barrier(WARPS), Barrier(1)
    ready = Barrier(WARPS)
    vec_full = [Barrier(1), Barrier(1)]
    vec_empty = [Barrier(WARPS), Barrier(WARPS)]
    t_full, t_copied = Barrier(1), Barrier(WARPS)
    o_final = Barrier(1)

    slot = [None, None]              # ("A" | "B", step) or ("T",); None while a load is in flight
    inflight = [False, False]
    vec = [None, None]
    sp = [None]                      # the score columns: ("S" | "dP", step)
    read_s, read_dp = {}, {}         # step -> warps that read it
    copied = set()
    ds_buf = [None]                  # (step, set of warps that wrote it)
    done = {"S": -1, "dP": -1, "acc": -1}
    pipe = []
    clock = [0.0]
    events = []

    def a_slot(s):
        return 0

    def b_slot(s):
        return 1

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
            kind, s = op
            if kind == "S":
                if slot[a_slot(s)] != ("A", s):
                    errors.append(f"S({s}) read slot {a_slot(s)} holding {slot[a_slot(s)]}")
                if len(copied) < WARPS:
                    errors.append(f"S({s}) read its TMEM operand before every warp copied its rows")
                if len(read_dp.get(s, ())) < WARPS:
                    errors.append(f"S({s}) overwrote dP({s}) before every warp read it")
            elif kind == "dP":
                if slot[b_slot(s)] != ("B", s):
                    errors.append(f"dP({s}) read slot {b_slot(s)} holding {slot[b_slot(s)]}")
                if s > 0 and len(read_s.get(s - 1, ())) < WARPS:
                    errors.append(f"dP({s}) overwrote S({s - 1}) before every warp read it")
            elif kind == "acc":
                if ds_buf[0] is None or ds_buf[0][0] != s or len(ds_buf[0][1]) < WARPS:
                    errors.append(f"accumulate({s}) read dS holding {ds_buf[0]}")
            yield ("delay", rng.uniform(100, 600))
            if kind == "acc" and slot[a_slot(s)] != ("A", s):
                errors.append(f"accumulate({s}) read slot {a_slot(s)} holding {slot[a_slot(s)]}")
            done[kind] = s
            if kind in ("S", "dP"):
                sp[0] = (kind, s)

    # ------------------------------------------------------------ producer
    def producer():
        uses = [0, 0]

        def land(i, what):
            def f():
                slot[i], inflight[i] = what, False
                full[i].complete_tx(1)
            return f

        def land_vec(x, s):
            def f():
                vec[x] = s
                vec_full[x].complete_tx(1)
            return f

        def land_t():
            slot[0] = ("T",)
            t_full.complete_tx(1)

        if n > 0:
            # the TMEM-bound operand (K in the dK pass, Q in the dQ pass) into
            # slot 0, with the resident one (V or dO)
            t_full.expect_tx(1)
            t_full.arrive()
            later(rng.uniform(300, 4000), land_t)

        def load(i, what):
            if i == 0 and uses[0] == 0 and producer_waits_copy:
                yield from wait(t_copied, 0, "producer copied", 0)
            yield from wait(empty[i], (uses[i] & 1) ^ 1, "producer empty")
            uses[i] += 1
            if inflight[i]:
                errors.append(f"{what} loaded into slot {i} while a load was in flight")
            full[i].expect_tx(1)
            full[i].arrive()
            slot[i], inflight[i] = None, True
            later(rng.uniform(300, 4000), land(i, what))

        for s in range(n):
            yield from load(b_slot(s), ("B", s))
            yield from load(a_slot(s), ("A", s))
            if dk_pass:
                x = s & 1
                yield from wait(vec_empty[x], ((s >> 1) & 1) ^ 1, "producer vec_empty")
                vec_full[x].expect_tx(1)
                vec_full[x].arrive()
                vec[x] = None
                later(rng.uniform(200, 2000), land_vec(x, s))

    # ------------------------------------------------------------ issuer
    def issuer():
        fulls = [0, 0]

        def wait_full(i):
            par = fulls[i] & 1
            fulls[i] += 1
            yield from wait(full[i], par, "issuer full")

        if n == 0:
            pipe.append(("commit", o_final))
            return
        yield from wait(t_full, 0, "issuer t_full", 0)
        yield from wait(t_copied, 0, "issuer copied", 0)
        yield from wait_full(b_slot(0))
        pipe.extend([("dP", 0), ("commit", dp_full), ("commit", empty[b_slot(0)])])
        for s in range(n):
            if issuer_waits_s_read:                                 # every warp read dP_s
                yield from wait(s_read, s & 1, "issuer dp read", s)
            yield from wait_full(a_slot(s))
            pipe.extend([("S", s), ("commit", s_full)])
            if not release_a_after_acc:
                pipe.append(("commit", empty[a_slot(s)]))
            yield from wait(ready, s & 1, "issuer ready", s)
            pipe.append(("acc", s))
            if release_a_after_acc:
                pipe.append(("commit", empty[a_slot(s)]))
            if s + 1 < n:
                yield from wait_full(b_slot(s + 1))
                pipe.extend([("dP", s + 1), ("commit", dp_full), ("commit", empty[b_slot(s + 1)])])
        pipe.append(("commit", o_final))

    # ------------------------------------------------------------ warps
    def warp_role(w):
        if n > 0:
            yield from wait(t_full, 0, f"warp {w} t_full", 0)
            yield ("delay", rng.uniform(50, 600))          # its rows of K or Q into TMEM
            if slot[0] != ("T",):
                errors.append(f"warp {w} copied its TMEM operand from slot 0 holding {slot[0]}")
            copied.add(w)
            t_copied.arrive()
        for s in range(n):
            v = s & 1
            if warps_wait_dp:
                yield from wait(dp_full, s & 1, f"warp {w} dp_full", s)
            if sp[0] != ("dP", s):
                errors.append(f"warp {w} read dP({s}) from score columns holding {sp[0]}")
            yield ("delay", rng.uniform(20, 300))                # dP into registers
            read_dp.setdefault(s, set()).add(w)
            s_read.arrive()
            yield from wait(s_full, s & 1, f"warp {w} s_full", s)
            if dk_pass:
                yield from wait(vec_full[v], (s >> 1) & 1, f"warp {w} vec_full", s >> 1)
                if vec[v] != s:
                    errors.append(f"warp {w} read LSE of step {s} from buffer {v} holding {vec[v]}")
            if sp[0] != ("S", s):
                errors.append(f"warp {w} read S({s}) from score columns holding {sp[0]}")
            yield ("delay", rng.uniform(*warp_cycles))          # S read, P formed
            read_s.setdefault(s, set()).add(w)
            if dk_pass and not vec_release_last:
                vec_empty[v].arrive()
                yield ("delay", rng.uniform(0, 400))
            if dk_pass and vec[v] != s:
                errors.append(f"warp {w} read D of step {s} from buffer {v} holding {vec[v]}")
            # the single dS buffer was last read by the accumulate of step s - 1
            if s >= 1 and done["acc"] < s - 1:
                errors.append(f"warp {w} wrote dS({s}) before the accumulate of step {s - 1} read the buffer")
            yield ("delay", rng.uniform(*warp_cycles))
            if ds_buf[0] is None or ds_buf[0][0] != s:
                ds_buf[0] = (s, set())
            ds_buf[0][1].add(w)
            ready.arrive()
            if dk_pass and vec_release_last:
                vec_empty[v].arrive()
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


@pytest.mark.parametrize("n", [0, 1, 2, 3, 6, 11])
@pytest.mark.parametrize("dk_pass", [True, False])
@pytest.mark.parametrize("warp_cycles", [(100, 1500), (20, 6000)])
def test_wide_bwd_protocol_holds(n, dk_pass, warp_cycles):
    for seed in range(15):
        errs = simulate(n, seed, dk_pass=dk_pass, warp_cycles=warp_cycles)
        assert not errs, (n, seed, dk_pass, errs[:3])


def bad_runs(dk_pass=True, **kw):
    return sum(bool(simulate(n, seed, dk_pass=dk_pass, warp_cycles=(20, 6000), **kw))
               for n in (3, 6, 11) for seed in range(12))


@pytest.mark.parametrize("dk_pass", [True, False])
def test_a_slot_must_wait_for_the_accumulate(dk_pass):
    """A_s is read by S_s and by the accumulate; releasing its slot after S_s
    lets A_{s+1} land over it before the accumulate has read it."""
    assert bad_runs(dk_pass, release_a_after_acc=False) > 0


@pytest.mark.parametrize("dk_pass", [True, False])
def test_warps_must_wait_for_dp(dk_pass):
    """The warps read dP first, into registers; that read needs its own wait."""
    assert bad_runs(dk_pass, warps_wait_dp=False) > 0


@pytest.mark.parametrize("dk_pass", [True, False])
def test_slot_0_must_wait_for_the_tmem_copy(dk_pass):
    """K (dK pass) or Q (dQ pass) lands in slot 0 and each warp copies its
    rows into TMEM; a load into that slot before every warp has copied would
    overwrite the operand under a warp still reading it."""
    assert bad_runs(dk_pass, producer_waits_copy=False) > 0


@pytest.mark.parametrize("dk_pass", [True, False])
def test_scores_must_wait_until_every_warp_read_dp(dk_pass):
    """dP and S share the score columns: S_s may go in only once every warp
    has read dP_s."""
    assert bad_runs(dk_pass, issuer_waits_s_read=False) > 0


def test_vector_release_is_implied_by_the_slot_order():
    """Not load-bearing: the producer loads step s + 2's LSE and D only after
    A_{s+2}, whose slot the accumulate of step s + 1 frees, and that
    accumulate waits for every warp's dS of step s + 1, written after the
    warp finished step s. So handing the vector buffer back early is still
    safe."""
    assert bad_runs(True, vec_release_last=False) == 0
