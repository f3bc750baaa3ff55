"""A model of the three-pass backward's dK and dQ passes, run on the CPU.

The kernels (csrc/fa_bwd_wide.cu, wide_dk_kernel and wide_dq_kernel)
walk 64-row sub-tile steps s over four shared-memory slots. Each step has an
operand A (Q_s in the dK pass, K_s in the dQ pass), read by the scores S_s and
by the accumulate (dK += dS^T Q_s, dQ += dS K_s), and an operand B (dO_s or
V_s), read only by dP_s. One thread issues S_0, dP_0,
then per step: [dS_s written] the accumulate, which frees A_s's slot once it
completes; [A_{s+1} landed] S_{s+1}; [B_{s+1} landed] dP_{s+1}, which frees
B's slot. dS (shared memory) and, in the dK pass, the step's LSE and D are
double-buffered by step parity. Each pass keeps one operand in TMEM as the A
operand of the scores (K in the dK pass, Q in the dQ pass): it lands in slots
0 and 1, every warp copies its rows, and only then do those slots join a ring
of four (A_s and B_s in slots (2s + 2) % 4 and (2s + 3) % 4); S and dP have
one TMEM buffer each. Four warps, one per TMEM lane quarter, form P from S,
wait for dP, and write dS.

As for the other kernels, the roles run as coroutines with random latencies
over barriers with the hardware's parity rule. The model checks that every
product and every warp reads the data of its own step, that no slot, TMEM
buffer, dS buffer or vector buffer is overwritten while a reader still needs
it, and that no parity wait passes on an older phase. Planted changes show
what the accumulate's release of A's slot, the warps' wait for dP and the
producer's wait for the TMEM copy guard; the vector buffer's release point
turns out to be implied by the slot order.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

WARPS = 4


def simulate(n, seed, *, dk_pass=True, release_a_after_acc=True, warps_wait_dp=True, vec_release_last=True,
             producer_waits_q_copy=True, warp_cycles=(100, 1500)):
    """Errors seen in one run of n steps of one CTA. The dQ pass (dk_pass
    False) holds Q in TMEM: four slots, the first two holding the Q tile until
    every warp has copied its row, and one TMEM buffer each for S and dP."""
    rng = random.Random(seed)
    errors = []
    nslots, nbuf = 4, 1                 # slots; TMEM buffers of S and of dP
    full = [Barrier(1) for _ in range(nslots)]
    empty = [Barrier(1) for _ in range(nslots)]
    s_full = [Barrier(1) for _ in range(nbuf)]
    dp_full = [Barrier(1) for _ in range(nbuf)]
    ready = [Barrier(WARPS) for _ in range(nbuf)]
    q_full, q_tmem = Barrier(1), Barrier(WARPS)
    copied = set()
    vec_full = [Barrier(1), Barrier(1)]
    vec_empty = [Barrier(WARPS), Barrier(WARPS)]
    o_final = Barrier(1)

    slot = [None] * nslots           # ("A" | "B", step) or ("Q",); None while a load is in flight
    inflight = [False] * nslots
    vec = [None, None]
    s_buf, dp_buf = [None] * nbuf, [None] * nbuf   # step whose S / dP the buffer holds
    read_s, read_dp = {}, {}                      # step -> warps that read it
    ds_buf = [None, None]                         # (step, set of warps that wrote it)
    done = {"S": -1, "dP": -1, "acc": -1}
    pipe = []
    clock = [0.0]
    events = []

    def a_slot(s):
        return (2 * s + 2) & 3

    def b_slot(s):
        return (2 * s + 3) & 3

    def buf(s):
        return s % nbuf

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
            x = s & 1
            if kind == "S":
                if slot[a_slot(s)] != ("A", s):
                    errors.append(f"S({s}) read slot {a_slot(s)} holding {slot[a_slot(s)]}")
                if len(copied) < WARPS:
                    errors.append(f"S({s}) read its TMEM operand before every warp copied its rows")
                if s >= nbuf and len(read_s.get(s - nbuf, ())) < WARPS:
                    errors.append(f"S({s}) overwrote S({s - nbuf}) before every warp read it")
            elif kind == "dP":
                if slot[b_slot(s)] != ("B", s):
                    errors.append(f"dP({s}) read slot {b_slot(s)} holding {slot[b_slot(s)]}")
                if s >= nbuf and len(read_dp.get(s - nbuf, ())) < WARPS:
                    errors.append(f"dP({s}) overwrote dP({s - nbuf}) before every warp read it")
            elif kind == "acc":
                if ds_buf[x] is None or ds_buf[x][0] != s or len(ds_buf[x][1]) < WARPS:
                    errors.append(f"accumulate({s}) read dS buffer {x} holding {ds_buf[x]}")
            yield ("delay", rng.uniform(100, 600))
            if kind == "acc" and slot[a_slot(s)] != ("A", s):
                errors.append(f"accumulate({s}) read slot {a_slot(s)} holding {slot[a_slot(s)]}")
            done[kind] = s
            if kind == "S":
                s_buf[buf(s)] = s
            elif kind == "dP":
                dp_buf[buf(s)] = s

    # ------------------------------------------------------------ producer
    def producer():
        uses = [0] * nslots

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

        def land_q():
            slot[0] = slot[1] = ("Q",)
            q_full.complete_tx(1)

        if n > 0:
            # the TMEM-bound operand (K in the dK pass, Q in the dQ pass) into
            # slots 0 and 1, with the resident one (V or dO)
            q_full.expect_tx(1)
            q_full.arrive()
            later(rng.uniform(300, 4000), land_q)

        def load(i, what):
            if i < 2 and uses[i] == 0 and producer_waits_q_copy:
                yield from wait(q_tmem, 0, "producer q_tmem", 0)
            yield from wait(empty[i], (uses[i] & 1) ^ 1, "producer empty")
            uses[i] += 1
            if inflight[i]:
                errors.append(f"{what} loaded into slot {i} while a load was in flight")
            full[i].expect_tx(1)
            full[i].arrive()
            slot[i], inflight[i] = None, True
            later(rng.uniform(300, 4000), land(i, what))

        for s in range(n):
            yield from load(a_slot(s), ("A", s))
            if dk_pass:
                x = s & 1
                yield from wait(vec_empty[x], ((s >> 1) & 1) ^ 1, "producer vec_empty")
                vec_full[x].expect_tx(1)
                vec_full[x].arrive()
                vec[x] = None
                later(rng.uniform(200, 2000), land_vec(x, s))
            yield from load(b_slot(s), ("B", s))

    # ------------------------------------------------------------ issuer
    def issuer():
        fulls = [0] * nslots

        def wait_full(i):
            par = fulls[i] & 1
            fulls[i] += 1
            yield from wait(full[i], par, "issuer full")

        if n == 0:
            pipe.append(("commit", o_final))
            return
        yield from wait(q_full, 0, "issuer q_full", 0)
        yield from wait(q_tmem, 0, "issuer q_tmem", 0)
        yield from wait_full(a_slot(0))
        pipe.extend([("S", 0), ("commit", s_full[0])])
        if not release_a_after_acc:
            pipe.append(("commit", empty[a_slot(0)]))
        yield from wait_full(b_slot(0))
        pipe.extend([("dP", 0), ("commit", dp_full[0]), ("commit", empty[b_slot(0)])])
        for s in range(n):
            yield from wait(ready[buf(s)], (s // nbuf) & 1, "issuer ready", s // nbuf)
            pipe.append(("acc", s))
            if release_a_after_acc:
                pipe.append(("commit", empty[a_slot(s)]))
            if s + 1 < n:
                x = buf(s + 1)
                yield from wait_full(a_slot(s + 1))
                pipe.extend([("S", s + 1), ("commit", s_full[x])])
                if not release_a_after_acc:
                    pipe.append(("commit", empty[a_slot(s + 1)]))
                yield from wait_full(b_slot(s + 1))
                pipe.extend([("dP", s + 1), ("commit", dp_full[x]), ("commit", empty[b_slot(s + 1)])])
        pipe.append(("commit", o_final))

    # ------------------------------------------------------------ warps
    def warp_role(w):
        if n > 0:
            yield from wait(q_full, 0, f"warp {w} q_full", 0)
            yield ("delay", rng.uniform(50, 600))          # its rows of K or Q into TMEM
            if slot[0] != ("Q",) or slot[1] != ("Q",):
                errors.append(f"warp {w} copied Q from slots holding {slot[0]}, {slot[1]}")
            copied.add(w)
            q_tmem.arrive()
        for s in range(n):
            x, v = buf(s), s & 1
            yield from wait(s_full[x], (s // nbuf) & 1, f"warp {w} s_full", s // nbuf)
            if dk_pass:
                yield from wait(vec_full[v], (s >> 1) & 1, f"warp {w} vec_full", s >> 1)
                if vec[v] != s:
                    errors.append(f"warp {w} read LSE of step {s} from buffer {v} holding {vec[v]}")
            if s_buf[x] != s:
                errors.append(f"warp {w} read S({s}) from buffer {x} holding {s_buf[x]}")
            read_s.setdefault(s, set()).add(w)
            yield ("delay", rng.uniform(*warp_cycles))          # P from S
            if warps_wait_dp:
                yield from wait(dp_full[x], (s // nbuf) & 1, f"warp {w} dp_full", s // nbuf)
            if dp_buf[x] != s:
                errors.append(f"warp {w} read dP({s}) from buffer {x} holding {dp_buf[x]}")
            read_dp.setdefault(s, set()).add(w)
            if dk_pass and not vec_release_last:
                vec_empty[v].arrive()
                yield ("delay", rng.uniform(0, 400))
            if dk_pass and vec[v] != s:
                errors.append(f"warp {w} read D of step {s} from buffer {v} holding {vec[v]}")
            # dS buffer v was last read by the accumulate of step s - 2
            if s >= 2 and done["acc"] < s - 2:
                errors.append(f"warp {w} wrote dS({s}) before the accumulate of step {s - 2} read the buffer")
            yield ("delay", rng.uniform(*warp_cycles))
            if ds_buf[v] is None or ds_buf[v][0] != s:
                ds_buf[v] = (s, set())
            ds_buf[v][1].add(w)
            ready[x].arrive()
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
    lets B_{s+1} land over it before the accumulate has read it."""
    assert bad_runs(dk_pass, release_a_after_acc=False) > 0


@pytest.mark.parametrize("dk_pass", [True, False])
def test_warps_must_wait_for_dp(dk_pass):
    """P is formed before dP arrives; the dP read still needs its own wait."""
    assert bad_runs(dk_pass, warps_wait_dp=False) > 0


@pytest.mark.parametrize("dk_pass", [True, False])
def test_slots_0_1_must_wait_for_the_tmem_copy(dk_pass):
    """K (dK pass) or Q (dQ pass) lands in slots 0 and 1 and each warp copies
    its rows into TMEM; a load into those slots before every warp has copied
    would overwrite the operand under a warp still reading it."""
    assert bad_runs(dk_pass, producer_waits_q_copy=False) > 0


def test_vector_release_is_implied_by_the_slot_order():
    """Not load-bearing: the producer loads step s + 2's LSE and D only after
    A_{s+2}, whose slot the accumulate of step s frees, and that accumulate
    waits for every warp's dS of step s, written after its D read. So handing
    the vector buffer back early is still safe."""
    assert bad_runs(True, vec_release_last=False) == 0
