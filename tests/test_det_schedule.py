"""Models of the deterministic backward's two kernels (csrc/fa_bwd_det.cu),
run on the CPU, as for the other kernels: every role a coroutine over
barriers with the hardware's parity rule and random latencies.

det_dkdv_kernel (one 128-key tile per CTA): per query step the tensor core
computes S^T, the warps turn it into P^T in place, dP^T = V dO^T goes into a
second TMEM region which the warps overwrite with dS^T, then dV += P^T dO and
dK += dS^T Q; Q, dO, LSE and D come in two stages, each handed back by a
commit after dK.

det_dq_kernel (one 128-row query tile per CTA): K_j and V_j stream through a
five-slot ring, S_j alternates between two TMEM buffers, the warps read S_j
and dP_j, signal "dP read" (so dP_{j+1} may overwrite it), and write dS_j
over S_j, signalling on the dS-ready barrier of tile parity j % 2; dQ +=
dS_j K_j. K_j goes back to the producer after dQ_j, V_j after
dP_j, each by a commit.

The checks: every MMA reads the tile of its own step from a landed slot or
stage, no TMEM region, stage or slot is overwritten while a reader still
needs it, and no parity wait passes on an older phase. Planted changes show
what the second S buffer, the "dP read" wait, the K release after dQ, the
stage release after dK and the second dS-ready barrier guard.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

WARPS = 8                                   # two groups of four; one arrival per warp stands for 32 threads


def run(roles, events, clock, pipe, errors, horizon):
    waiting, finished = {}, set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, random.random(), ("run", i)))
    while events and clock[0] < horizon:
        clock[0], _, (what, arg) = heapq.heappop(events)
        if what == "call":
            arg()
            continue
        r = arg
        if r in finished:
            continue
        try:
            y = waiting.pop(r) if r in waiting else next(roles[r])
            while True:
                if y[0] == "delay":
                    heapq.heappush(events, (clock[0] + y[1], random.random(), ("run", r)))
                    break
                if y[1]():
                    y = next(roles[r])
                    continue
                waiting[r] = y
                heapq.heappush(events, (clock[0] + 50.0, random.random(), ("run", r)))
                break
        except StopIteration:
            finished.add(r)
        if finished == set(range(1, len(roles))) and not pipe:
            break
    if finished != set(range(1, len(roles))):
        errors.append(f"deadlock: roles {sorted(set(range(1, len(roles))) - finished)} never finished")
    return errors


def make_wait(errors):
    def wait(bar, parity, who, phase=None):
        yield ("wait", lambda: bar.passes(parity))
        if phase is not None and bar.done < phase + 1:
            errors.append(f"{who}: parity wait for phase {phase} passed on an older phase")
    return wait


# ---------------------------------------------------------------- dK / dV pass
def simulate_dkdv(n, seed, *, stage_release_after_dk=True, warp_cycles=(200, 1500)):
    rng = random.Random(seed)
    random.seed(seed)
    errors, pipe, clock, events = [], [], [0.0], []
    wait = make_wait(errors)
    kv_full = Barrier(1)
    q_full, q_empty = [Barrier(1), Barrier(1)], [Barrier(1), Barrier(1)]
    s_full, dp_full, o_final = Barrier(1), Barrier(1), Barrier(1)
    p_ready, ds_ready = Barrier(WARPS), Barrier(WARPS)
    stage = [None, None]                       # step whose Q, dO, LSE, D sit in the stage
    tmem_s, tmem_dp = [None], [None]           # ("S" | "P", step), ("dP" | "dS", step)
    wrote = {}
    done = {"S": -1, "dP": -1, "dV": -1, "dK": -1}
    vec_reads = {}                             # step -> warps done reading LSE and D

    def later(dt, fn):
        heapq.heappush(events, (clock[0] + dt, rng.random(), ("call", fn)))

    def tensor_core():
        while True:
            while not pipe:
                yield ("wait", lambda: bool(pipe))
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, step = op
            st = step & 1
            if kind in ("S", "dP", "dV", "dK") and stage[st] != step:
                errors.append(f"{kind}({step}) read stage {st} holding step {stage[st]}")
            if kind == "S" and step > 0 and done["dV"] < step - 1:
                errors.append(f"S({step}) overwrote P^T({step - 1}) before dV read it")
            if kind == "dP" and step > 0 and done["dK"] < step - 1:
                errors.append(f"dP({step}) overwrote dS^T({step - 1}) before dK read it")
            if kind == "dV" and tmem_s[0] != ("P", step):
                errors.append(f"dV({step}) read TMEM S holding {tmem_s[0]}")
            if kind == "dK" and tmem_dp[0] != ("dS", step):
                errors.append(f"dK({step}) read TMEM dP holding {tmem_dp[0]}")
            yield ("delay", rng.uniform(100, 400))
            done[kind] = step
            if kind == "S":
                tmem_s[0] = ("S", step)
            elif kind == "dP":
                tmem_dp[0] = ("dP", step)

    def producer():
        kv_full.expect_tx(1)
        kv_full.arrive()
        later(rng.uniform(300, 3000), lambda: kv_full.complete_tx(1))
        for step in range(n):
            st = step & 1
            yield from wait(q_empty[st], ((step >> 1) & 1) ^ 1, "producer")
            if step >= 2 and (done["dK"] < step - 2 or len(vec_reads.get(step - 2, ())) < WARPS):
                errors.append(f"stage {st} reloaded for step {step} while step {step - 2} was still read")
            q_full[st].expect_tx(1)
            q_full[st].arrive()
            stage[st] = None

            def land(st=st, step=step):
                stage[st] = step
                q_full[st].complete_tx(1)
            later(rng.uniform(300, 3000), land)

    def issuer():
        if n == 0:
            pipe.append(("commit", o_final))
            return
        yield from wait(kv_full, 0, "issuer kv")
        yield from wait(q_full[0], 0, "issuer q", 0)
        pipe.extend([("S", 0), ("commit", s_full)])
        for step in range(n):
            st = step & 1
            pipe.extend([("dP", step), ("commit", dp_full)])
            yield from wait(p_ready, step & 1, "issuer p_ready", step)
            pipe.append(("dV", step))
            if not stage_release_after_dk:
                pipe.append(("commit", q_empty[st]))
            if step + 1 < n:
                yield from wait(q_full[st ^ 1], ((step + 1) >> 1) & 1, "issuer q", (step + 1) >> 1)
                pipe.extend([("S", step + 1), ("commit", s_full)])
            yield from wait(ds_ready, step & 1, "issuer ds_ready", step)
            pipe.append(("dK", step))
            if stage_release_after_dk:
                pipe.append(("commit", q_empty[st]))
        pipe.append(("commit", o_final))

    def warp(w):
        for step in range(n):
            st = step & 1
            yield from wait(q_full[st], (step >> 1) & 1, f"warp {w} q", step >> 1)
            yield from wait(s_full, step & 1, f"warp {w} s_full", step)
            if tmem_s[0] not in (("S", step), ("P", step)) or (tmem_s[0] == ("P", step) and w in wrote.get(("P", step), ())):
                errors.append(f"warp {w} read S^T({step}) from TMEM holding {tmem_s[0]}")
            if stage[st] != step:
                errors.append(f"warp {w} read LSE of step {step} from stage {st} holding {stage[st]}")
            yield ("delay", rng.uniform(*warp_cycles))
            wrote.setdefault(("P", step), set()).add(w)
            if len(wrote[("P", step)]) == WARPS:
                tmem_s[0] = ("P", step)
            p_ready.arrive()
            yield from wait(dp_full, step & 1, f"warp {w} dp_full", step)
            if tmem_dp[0] not in (("dP", step), ("dS", step)) or (tmem_dp[0] == ("dS", step) and w in wrote.get(("dS", step), ())):
                errors.append(f"warp {w} read dP^T({step}) from TMEM holding {tmem_dp[0]}")
            if stage[st] != step:
                errors.append(f"warp {w} read D of step {step} from stage {st} holding {stage[st]}")
            vec_reads.setdefault(step, set()).add(w)
            yield ("delay", rng.uniform(*warp_cycles))
            wrote.setdefault(("dS", step), set()).add(w)
            if len(wrote[("dS", step)]) == WARPS:
                tmem_dp[0] = ("dS", step)
            ds_ready.arrive()
        yield from wait(o_final, 0, f"warp {w} o_final", 0)

    roles = [tensor_core(), producer(), issuer()] + [warp(w) for w in range(WARPS)]
    return run(roles, events, clock, pipe, errors, 40000.0 * (n + 4))


# ---------------------------------------------------------------- dQ pass
def simulate_dq(n, seed, *, slots=5, s_buffers=2, wait_dp_read=True, release_k_after_dq=True,
                split_ds_ready=True, warp_cycles=(200, 1500)):
    rng = random.Random(seed)
    random.seed(seed)
    errors, pipe, clock, events = [], [], [0.0], []
    wait = make_wait(errors)
    q_full = Barrier(1)
    full = [Barrier(1) for _ in range(slots)]
    empty = [Barrier(1) for _ in range(slots)]
    s_full = [Barrier(1) for _ in range(2)]
    dp_full, dq_final = Barrier(1), Barrier(1)
    dp_read = Barrier(WARPS)
    ds_ready = [Barrier(WARPS) for _ in range(2 if split_ds_ready else 1)]

    def dsr(j):                                # dS-ready of tile j: one barrier per tile parity
        return ds_ready[j & 1] if split_ds_ready else ds_ready[0]

    def dsr_phase(j):
        return j >> 1 if split_ds_ready else j
    landed = [None] * slots
    in_flight = [None] * slots
    q_landed = [False]
    tmem_s = [None, None]                      # ("S" | "dS", j) per buffer
    tmem_dp = [None]
    wrote, read_dp = {}, {}
    readers_done, readers_needed = {}, {}
    for j in range(n):
        readers_needed[2 * j] = 2              # K_j: S_j and dQ_j
        readers_needed[2 * j + 1] = 1          # V_j: dP_j
    done = {"dQ": -1, "dP": -1}

    def later(dt, fn):
        heapq.heappush(events, (clock[0] + dt, rng.random(), ("call", fn)))

    def buf(j):
        return j % s_buffers

    def tensor_core():
        while True:
            while not pipe:
                yield ("wait", lambda: bool(pipe))
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, j, load = op
            slot = load % slots
            if landed[slot] != load or in_flight[slot] is not None:
                errors.append(f"{kind}({j}) read slot {slot} holding {landed[slot]}, wanted load {load}")
            if kind in ("S", "dP") and not q_landed[0]:
                errors.append(f"{kind}({j}) read Q / dO before they landed")
            if kind == "S" and j >= s_buffers and done["dQ"] < j - s_buffers:
                errors.append(f"S({j}) overwrote dS({j - s_buffers}) before dQ read it")
            if kind == "dP" and j > 0 and len(read_dp.get(j - 1, ())) < WARPS:
                errors.append(f"dP({j}) overwrote dP({j - 1}) before every warp read it")
            if kind == "dQ" and tmem_s[buf(j)] != ("dS", j):
                errors.append(f"dQ({j}) read S buffer {buf(j)} holding {tmem_s[buf(j)]}")
            yield ("delay", rng.uniform(100, 400))
            readers_done[load] = readers_done.get(load, 0) + 1
            if kind == "S":
                tmem_s[buf(j)] = ("S", j)
            elif kind == "dP":
                tmem_dp[0] = ("dP", j)
                done["dP"] = j
            else:
                done["dQ"] = j

    def producer():
        q_full.expect_tx(1)
        q_full.arrive()

        def land_q():
            q_landed[0] = True
            q_full.complete_tx(1)
        later(rng.uniform(300, 3000), land_q)
        for c in range(2 * n):
            slot = c % slots
            yield from wait(empty[slot], ((c // slots) & 1) ^ 1, "producer")
            prev = c - slots
            if prev >= 0 and readers_done.get(prev, 0) < readers_needed[prev]:
                errors.append(f"load {c} overwrote load {prev} in slot {slot} before its MMAs ran")
            full[slot].expect_tx(1)
            full[slot].arrive()
            in_flight[slot], landed[slot] = c, None

            def land(s=slot, ld=c):
                in_flight[s], landed[s] = None, ld
                full[s].complete_tx(1)
            later(rng.uniform(300, 3000), land)

    def issuer():
        c = [0]

        def take():
            load = c[0]
            c[0] += 1
            yield from wait(full[load % slots], (load // slots) & 1, "issuer", load // slots)
            return load

        if n == 0:
            pipe.append(("commit", dq_final))
            return
        yield from wait(q_full, 0, "issuer q", 0)
        k = yield from take()
        pipe.extend([("S", 0, k), ("commit", s_full[0])])
        v = yield from take()
        pipe.extend([("dP", 0, v), ("commit", dp_full), ("commit", empty[v % slots])])
        for j in range(n):
            k_j = k
            if j + 1 < n:
                k = yield from take()
                pipe.extend([("S", j + 1, k), ("commit", s_full[(j + 1) % 2])])
            if wait_dp_read:
                yield from wait(dp_read, j & 1, "issuer dp_read", j)
            if j + 1 < n:
                v = yield from take()
                pipe.extend([("dP", j + 1, v), ("commit", dp_full), ("commit", empty[v % slots])])
            if not release_k_after_dq:
                pipe.append(("commit", empty[k_j % slots]))
            yield from wait(dsr(j), dsr_phase(j) & 1, "issuer ds_ready", dsr_phase(j))
            pipe.append(("dQ", j, k_j))
            if release_k_after_dq:
                pipe.append(("commit", empty[k_j % slots]))
        pipe.append(("commit", dq_final))

    def warp(w):
        for j in range(n):
            x = j % 2
            yield from wait(s_full[x], (j >> 1) & 1, f"warp {w} s_full", j >> 1)
            yield from wait(dp_full, j & 1, f"warp {w} dp_full", j)
            yield ("delay", rng.uniform(0, 600))      # the TMEM loads of S_j and dP_j
            b = buf(j)
            if tmem_s[b] not in (("S", j), ("dS", j)) or (tmem_s[b] == ("dS", j) and w in wrote.get(j, ())):
                errors.append(f"warp {w} read S({j}) from buffer {b} holding {tmem_s[b]}")
            if tmem_dp[0] != ("dP", j):
                errors.append(f"warp {w} read dP({j}) from TMEM holding {tmem_dp[0]}")
            read_dp.setdefault(j, set()).add(w)
            dp_read.arrive()
            yield ("delay", rng.uniform(*warp_cycles))
            wrote.setdefault(j, set()).add(w)
            if len(wrote[j]) == WARPS:
                tmem_s[b] = ("dS", j)
            dsr(j).arrive()
        yield from wait(dq_final, 0, f"warp {w} dq_final", 0)

    roles = [tensor_core(), producer(), issuer()] + [warp(w) for w in range(WARPS)]
    return run(roles, events, clock, pipe, errors, 40000.0 * (n + 4))


@pytest.mark.parametrize("n", [0, 1, 2, 3, 6, 11])
@pytest.mark.parametrize("warp_cycles", [(200, 1500), (50, 5000)])
def test_det_dkdv_protocol_holds(n, warp_cycles):
    for seed in range(15):
        errs = simulate_dkdv(n, seed, warp_cycles=warp_cycles)
        assert not errs, (n, seed, errs[:3])


@pytest.mark.parametrize("n", [0, 1, 2, 3, 6, 11])
@pytest.mark.parametrize("warp_cycles", [(200, 1500), (50, 5000)])
def test_det_dq_protocol_holds(n, warp_cycles):
    for seed in range(15):
        errs = simulate_dq(n, seed, warp_cycles=warp_cycles)
        assert not errs, (n, seed, errs[:3])


def bad_dkdv(**kw):
    return sum(bool(simulate_dkdv(n, seed, warp_cycles=(50, 5000), **kw)) for n in (3, 6, 11) for seed in range(15))


def bad_dq(**kw):
    return sum(bool(simulate_dq(n, seed, warp_cycles=(50, 5000), **kw)) for n in (3, 6, 11) for seed in range(15))


def test_det_dkdv_stage_goes_back_only_after_dk():
    """Handing a stage back after dV lets the next load overwrite Q while
    dK still reads it."""
    assert bad_dkdv(stage_release_after_dk=False) > 0


def test_det_dq_needs_two_s_buffers():
    assert bad_dq(s_buffers=1) > 0


def test_det_dq_waits_for_dp_to_be_read():
    assert bad_dq(wait_dp_read=False) > 0


def test_det_dq_single_ds_ready_barrier_races():
    """With one dS-ready barrier, a warp that already holds S_{j+1} and
    dP_{j+1} can arrive for tile j+1 while a slower warp is still writing
    dS_j, completing tile j's phase early: dQ_j then reads a partial dS_j.
    (The kernel had this form until this model found it.)"""
    assert bad_dq(split_ds_ready=False) > 0


def test_det_dq_releases_k_after_dq():
    """K_j is read twice, by S_j and by dQ_j; releasing it before dQ_j lets a
    load overwrite it."""
    assert bad_dq(release_k_after_dq=False) > 0
