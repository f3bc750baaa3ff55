"""A model of the bf16 forward kernel's synchronisation (d <= 128), run on the CPU.

The kernel (csrc/fa_fwd.cu, bf16 instantiations) runs two 128-row query
tiles per CTA. Each tile has one S region in TMEM: S_i(j) = Q_i K_j^T, which
its softmax group turns into P_i(j) in place, then P_i(j) V_j accumulates
into O_i and S_i(j+1) is issued right after it, into the same columns. The
issuer waits only for K_0 itself; a ring watcher observes every load in
ring order and folds "V_j and K_{j+1} landed" into each tile's P-ready
barrier (one arrival next to the group's), and hands the ring slots of K_j
and V_{j-1} back once S of the last-issued tile of step j has completed,
which the tensor core runs after every MMA that reads them. A softmax group
rescales its O only once S_i(j) has completed, which follows P_i(j-1) V_{j-1}.

As for the other kernels, the roles run as coroutines with random
latencies over barriers with the hardware's parity rule; every MMA, every
TMEM read and write, every slot reuse and every parity wait is checked, and
planted changes show what the watcher's choice of the last-issued tile,
its wait before handing slots back and its wait for the previous P-ready
phase guard. The watcher's first wait, for K_0, turns out to be implied by
its wait for S before the first hand-back.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

SLOTS = 5
WARPS = 4


def simulate(nkv, seed, *, slots=SLOTS, watcher_first_wait=True, last_tile_rule=True, release_after_s=True,
             watcher_gate=True, softmax_cycles=(300, 1500)):
    """Errors seen in one run of one CTA whose query tiles see nkv[0], nkv[1] key tiles."""
    rng = random.Random(seed)
    errors = []
    nmax = max(nkv)
    full = [Barrier(1) for _ in range(slots)]
    empty = [Barrier(1) for _ in range(slots)]
    q_full = [Barrier(1), Barrier(1)]
    s_full = [Barrier(1), Barrier(1)]
    p_ready = [Barrier(WARPS + 1), Barrier(WARPS + 1)]     # + the watcher
    o_final = [Barrier(1), Barrier(1)]
    landed = [None] * slots
    in_flight = [None] * slots
    q_landed = [False, False]
    tmem_s = [None, None]                          # ("S" | "P", j)
    p_written = {}
    pv_done = [-1, -1]
    s_done = [-1, -1]
    readers_done = {}                              # load -> number of MMAs that read it and completed
    readers_needed = {}
    pipe = []
    clock = [0.0]
    events = []

    for j in range(nmax):
        # K_j read by S_i(j), V_j by P_i(j) V_j, for each tile that reaches step j
        readers_needed[2 * j] = sum(1 for i in range(2) if j < nkv[i])
        readers_needed[2 * j + 1] = sum(1 for i in range(2) if j < nkv[i])

    def wait(bar, parity, who, phase=None):
        yield ("wait", lambda: bar.passes(parity))
        if phase is not None and bar.done < phase + 1:
            errors.append(f"{who}: parity wait for phase {phase} passed on an older phase")

    def tensor_core():
        while True:
            while not pipe:
                yield ("wait", lambda: bool(pipe))
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, i, j, load = op
            slot = load % slots
            if landed[slot] != load or in_flight[slot] is not None:
                errors.append(f"{kind}{i}({j}) read slot {slot} holding {landed[slot]}, wanted load {load}")
            if kind == "S":
                if not q_landed[i]:
                    errors.append(f"S{i}({j}) read Q_{i} before it landed")
                if j > 0 and pv_done[i] < j - 1:
                    errors.append(f"S{i}({j}) overwrote P{i}({j - 1}) before P V read it")
            else:
                if tmem_s[i] != ("P", j):
                    errors.append(f"PV{i}({j}) read TMEM holding {tmem_s[i]}")
            yield ("delay", rng.uniform(200, 300))
            readers_done[load] = readers_done.get(load, 0) + 1
            if kind == "S":
                tmem_s[i] = ("S", j)
                s_done[i] = j
            else:
                pv_done[i] = j

    def producer():
        for i in range(2):
            if nkv[i] == 0:
                continue
            q_full[i].expect_tx(1)
            q_full[i].arrive()

            def land_q(i=i):
                q_landed[i] = True
                q_full[i].complete_tx(1)
            heapq.heappush(events, (clock[0] + rng.uniform(300, 3000), rng.random(), ("call", land_q)))
        for c in range(2 * nmax):
            slot = c % slots
            yield from wait(empty[slot], ((c // slots) & 1) ^ 1, "producer")
            if in_flight[slot] is not None:
                errors.append(f"load {c} issued into slot {slot} with a load in flight")
            prev = c - slots
            if prev >= 0 and readers_done.get(prev, 0) < readers_needed[prev]:
                errors.append(f"load {c} overwrote load {prev} in slot {slot} before its MMAs ran")
            full[slot].expect_tx(1)
            full[slot].arrive()
            in_flight[slot], landed[slot] = c, None

            def land(s=slot, ld=c):
                in_flight[s], landed[s] = None, ld
                full[s].complete_tx(1)
            heapq.heappush(events, (clock[0] + rng.uniform(300, 3000), rng.random(), ("call", land)))

    def issuer():
        for i in range(2):
            if nkv[i] > 0:
                yield from wait(q_full[i], 0, f"issuer q{i}", 0)
        if nmax == 0:
            return
        yield from wait(full[0], 0, "issuer K_0", 0)
        for i in range(2):
            if nkv[i] > 0:
                pipe.extend([("S", i, 0, 0), ("commit", s_full[i])])
        for j in range(nmax):
            for i in range(2):
                if j >= nkv[i]:
                    continue
                yield from wait(p_ready[i], j & 1, f"issuer p_ready{i}", j)
                pipe.append(("PV", i, j, 2 * j + 1))
                if j + 1 < nkv[i]:
                    pipe.extend([("S", i, j + 1, 2 * j + 2), ("commit", s_full[i])])
                else:
                    pipe.append(("commit", o_final[i]))

    def watcher():
        last = 1 if nkv[1] == nmax else 0          # the tile whose S is issued last in each step
        waited = last if last_tile_rule else 0      # the tile whose S the watcher waits for

        def hand_p(i, j):
            if j > 0 and watcher_gate:
                yield from wait(p_ready[i], (j - 1) & 1, f"watcher gate{i}", j - 1)
            elif p_ready[i].done < j:
                errors.append(f"watcher arrived for P-ready{i} phase {j} inside phase {p_ready[i].done}")
            p_ready[i].arrive()

        if nmax > 0 and watcher_first_wait:
            yield from wait(full[0], 0, "watcher K_0", 0)
        for j in range(nmax):
            cv = 2 * j + 1
            yield from wait(full[cv % slots], (cv // slots) & 1, "watcher V", cv // slots)
            if landed[cv % slots] != cv:
                errors.append(f"watcher took V_{j} (load {cv}) for landed while slot held {landed[cv % slots]}")
            if j + 1 < nmax:
                ck = 2 * j + 2
                yield from wait(full[ck % slots], (ck // slots) & 1, "watcher K", ck // slots)
                if landed[ck % slots] != ck:
                    errors.append(f"watcher took K_{j + 1} (load {ck}) for landed while slot held "
                                  f"{landed[ck % slots]}")
            if last == 1 and j < nkv[0]:
                yield from hand_p(0, j)
            if release_after_s and j < nkv[waited]:
                yield from wait(s_full[waited], j & 1, "watcher s_full", j)
            empty[(2 * j) % slots].arrive()
            if j > 0:
                empty[(2 * j - 1) % slots].arrive()
            if j < nkv[last]:
                yield from hand_p(last, j)
            elif last == 0 and j < nkv[0]:
                yield from hand_p(0, j)

    def softmax(i, w):
        for j in range(nkv[i]):
            yield from wait(s_full[i], j & 1, f"softmax{i} s_full", j)
            if tmem_s[i] != ("S", j) and not (tmem_s[i] == ("P", j) and w not in p_written.get((i, j), ())):
                errors.append(f"softmax{i} warp {w} read S{i}({j}) from TMEM holding {tmem_s[i]}")
            yield ("delay", rng.uniform(*softmax_cycles))
            p_written.setdefault((i, j), set()).add(w)
            if len(p_written[(i, j)]) == WARPS:
                tmem_s[i] = ("P", j)
            if j > 0 and rng.random() < 0.3:           # the row max grew: rescale O_i
                if pv_done[i] < j - 1:
                    errors.append(f"softmax{i} rescaled O while P V({j - 1}) was pending")
            p_ready[i].arrive()
        if nkv[i]:
            yield from wait(o_final[i], 0, f"softmax{i} epilogue", 0)

    roles = [tensor_core(), producer(), issuer(), watcher()] + [softmax(i, w) for i in range(2) for w in range(WARPS)]
    waiting, finished = {}, set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, rng.random(), ("run", i)))
    horizon = 20000.0 * (nmax + 4)
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
                    heapq.heappush(events, (clock[0] + y[1], rng.random(), ("run", r)))
                    break
                if y[1]():
                    y = next(roles[r])
                    continue
                waiting[r] = y
                heapq.heappush(events, (clock[0] + rng.uniform(20, 200), rng.random(), ("run", r)))
                break
        except StopIteration:
            finished.add(r)
        except AssertionError as e:
            errors.append(str(e))
            return errors
        if finished == set(range(1, len(roles))) and not pipe:
            break
    if finished != set(range(1, len(roles))):
        errors.append(f"deadlock: roles {sorted(set(range(1, len(roles))) - finished)} never finished")
    return errors


# causal pairs see n or n+1 key tiles per tile; an odd tail has no second tile
CASES = [(1, 1), (1, 2), (2, 3), (3, 3), (4, 5), (7, 7), (11, 12), (6, 0)]


@pytest.mark.parametrize("nkv", CASES)
@pytest.mark.parametrize("softmax_cycles", [(300, 1500), (100, 5000)])
@pytest.mark.parametrize("slots", [SLOTS, 12])
def test_forward_protocol_holds(nkv, softmax_cycles, slots):
    for seed in range(15):
        errs = simulate(nkv, seed, slots=slots, softmax_cycles=softmax_cycles)
        assert not errs, (nkv, seed, errs[:3])


def bad_runs(**kw):
    return sum(bool(simulate(nkv, seed, softmax_cycles=(100, 5000), **kw)) for nkv in [(3, 4), (6, 7), (9, 9)]
               for seed in range(15))


def test_watcher_k0_wait_is_implied_by_the_s_wait():
    """The kernel's watcher observes K_0 (which only the issuer needs) before
    anything else. The model shows that wait is not load-bearing: the next
    load into K_0's slot can only be issued after the watcher hands the slot
    back, which it does after S of step 0 has completed, so K_0 has landed
    before any later parity wait on that slot."""
    assert bad_runs(watcher_first_wait=False) == 0


def test_watcher_gate_needed_with_a_deeper_ring():
    """Arriving for P-ready phase j without waiting for phase j-1 to complete
    can land inside phase j-1 once the ring lets the watcher run ahead."""
    assert sum(bool(simulate(nkv, seed, slots=12, softmax_cycles=(100, 5000), watcher_gate=False))
               for nkv in [(6, 7), (9, 9), (11, 12)] for seed in range(15)) > 0


def test_slots_go_back_after_the_last_issued_s():
    """S of the tile issued first in a step completing says nothing about the
    other tile's S, which still reads K_j."""
    assert bad_runs(last_tile_rule=False) > 0


def test_slots_go_back_only_after_s_completes():
    assert bad_runs(release_after_s=False) > 0
