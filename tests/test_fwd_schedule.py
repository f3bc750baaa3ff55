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


# causal pairs see n or n+1 key tiles per tile; an odd tail has no second tile;
# block-sparse lists give the first tile any prefix of the second's list
# (0 included) and the ring one slot fewer
CASES = [(1, 1), (1, 2), (2, 3), (3, 3), (4, 5), (7, 7), (11, 12), (6, 0), (0, 3), (2, 5), (1, 7), (0, 0)]


@pytest.mark.parametrize("nkv", CASES)
@pytest.mark.parametrize("softmax_cycles", [(300, 1500), (100, 5000)])
@pytest.mark.parametrize("slots", [SLOTS - 1, SLOTS, 12])
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


# ---------------------------------------------------------------- fp32 (tf32) variant
def simulate_tf32(n, seed, *, slots=3, vt_wait_s=True, issuer_waits_p=True, warp_cycles=(300, 1500)):
    """The fp32 instantiation: one query tile, a three-slot ring, no watcher.
    The issuer waits for every load itself; besides the softmax, the four
    warps of the tile split Q and K_0 into tf32 high and low parts (the low
    parts in their own buffers, signalled by Q-K-ready), transpose V_j into a
    V^T buffer (the second Q region) and split K_{j+1}, each warp its own
    rows, before arriving on P-ready. Those buffers are rewritten at step j+1
    only after S_{j+1} has completed, which follows P(j) V^T. With
    vt_wait_s=False the warps write V^T_{j+1} as soon as V_{j+1} lands."""
    rng = random.Random(seed)
    errors = []
    full = [Barrier(1) for _ in range(slots)]
    empty = [Barrier(1) for _ in range(slots)]
    q_full, s_full, o_final = Barrier(1), Barrier(1), Barrier(1)
    p_ready, qk_ready = Barrier(WARPS), Barrier(WARPS)
    landed = [None] * slots
    in_flight = [None] * slots
    split_rows = {}                            # load of a K tile -> warps that split it (hi in place, lo buffer)
    k_lo = [None]                              # (load, warps) whose low part the lo buffer holds
    vt = [None]                                # (j, warps) whose V^T the V^T buffer holds
    q_landed = [False]
    tmem_s = [None]
    p_written = {}
    done = {"S": -1, "PV": -1}
    pipe = []
    clock = [0.0]
    events = []

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
            kind, j, load = op
            if kind == "S":
                if landed[load % slots] != load:
                    errors.append(f"S({j}) read slot {load % slots} holding {landed[load % slots]}")
                if k_lo[0] != (load, WARPS) or len(split_rows.get(load, ())) < WARPS:
                    errors.append(f"S({j}) read K low parts {k_lo[0]}, wanted every row of load {load}")
                if j > 0 and done["PV"] < j - 1:
                    errors.append(f"S({j}) overwrote P({j - 1}) before P V read it")
            else:
                if vt[0] != (j, WARPS):
                    errors.append(f"PV({j}) read V^T buffer holding {vt[0]}")
                if tmem_s[0] != ("P", j):
                    errors.append(f"PV({j}) read TMEM holding {tmem_s[0]}")
            yield ("delay", rng.uniform(200, 300))
            done[kind] = j
            if kind == "S":
                tmem_s[0] = ("S", j)

    def producer():
        q_full.expect_tx(1)
        q_full.arrive()

        def land_q():
            q_landed[0] = True
            q_full.complete_tx(1)
        heapq.heappush(events, (clock[0] + rng.uniform(300, 3000), rng.random(), ("call", land_q)))
        for c in range(2 * n):
            slot = c % slots
            yield from wait(empty[slot], ((c // slots) & 1) ^ 1, "producer")
            if in_flight[slot] is not None:
                errors.append(f"load {c} issued into slot {slot} with a load in flight")
            prev = c - slots
            if prev >= 0 and prev % 2 == 0 and done["S"] < prev // 2:
                errors.append(f"load {c} overwrote K load {prev} before S read it")
            full[slot].expect_tx(1)
            full[slot].arrive()
            in_flight[slot], landed[slot] = c, None

            def land(s=slot, ld=c):
                in_flight[s], landed[s] = None, ld
                full[s].complete_tx(1)
            heapq.heappush(events, (clock[0] + rng.uniform(300, 3000), rng.random(), ("call", land)))

    def issuer():
        if n == 0:
            return
        c = [0]

        def take():
            ld = c[0]
            c[0] += 1
            yield from wait(full[ld % slots], (ld // slots) & 1, "issuer", ld // slots)
            return ld

        yield from wait(q_full, 0, "issuer q", 0)
        k = yield from take()
        yield from wait(qk_ready, 0, "issuer qk", 0)
        pipe.extend([("S", 0, k), ("commit", s_full), ("commit", empty[k % slots])])
        for j in range(n):
            v = yield from take()
            kn = (yield from take()) if j + 1 < n else None
            if issuer_waits_p:
                yield from wait(p_ready, j & 1, "issuer p_ready", j)
            pipe.append(("PV", j, v))
            if kn is not None:
                pipe.extend([("S", j + 1, kn), ("commit", s_full)])
            else:
                pipe.append(("commit", o_final))
            pipe.append(("commit", empty[v % slots]))
            if kn is not None:
                pipe.append(("commit", empty[kn % slots]))

    def split_k(w, load):
        """This warp's rows of K tile `load`: high part in place, low part into the lo buffer."""
        if k_lo[0] is None or k_lo[0][0] != load:
            k_lo[0] = (load, 0)
        split_rows.setdefault(load, set()).add(w)
        k_lo[0] = (load, len(split_rows[load]))

    def warp(w):
        if n == 0:
            return
        yield from wait(q_full, 0, f"warp {w} q", 0)
        yield from wait(full[0], 0, f"warp {w} K_0", 0)
        if landed[0] != 0:
            errors.append(f"warp {w} split K_0 from slot 0 holding {landed[0]}")
        split_k(w, 0)
        qk_ready.arrive()
        for j in range(n):
            yield from wait(s_full, j & 1, f"warp {w} s_full", j)
            if tmem_s[0] != ("S", j) and not (tmem_s[0] == ("P", j) and w not in p_written.get(j, ())):
                errors.append(f"warp {w} read S({j}) from TMEM holding {tmem_s[0]}")
            yield ("delay", rng.uniform(*warp_cycles))
            p_written.setdefault(j, set()).add(w)
            if len(p_written[j]) == WARPS:
                tmem_s[0] = ("P", j)
            # V_j into the V^T buffer, this warp's key rows
            cv = 2 * j + 1
            yield from wait(full[cv % slots], (cv // slots) & 1, f"warp {w} V", cv // slots)
            if landed[cv % slots] != cv:
                errors.append(f"warp {w} transposed V_{j} from slot {cv % slots} holding {landed[cv % slots]}")
            if j > 0 and done["PV"] < j - 1:
                errors.append(f"warp {w} wrote V^T_{j} while P V({j - 1}) still read V^T_{j - 1}")
            if vt[0] is None or vt[0][0] != j:
                vt[0] = (j, 0)
            vt[0] = (j, vt[0][1] + 1)
            if j + 1 < n:
                ck = 2 * j + 2
                yield from wait(full[ck % slots], (ck // slots) & 1, f"warp {w} K", ck // slots)
                if landed[ck % slots] != ck:
                    errors.append(f"warp {w} split K_{j + 1} from slot {ck % slots} holding {landed[ck % slots]}")
                if done["S"] < j:
                    errors.append(f"warp {w} rewrote the K low parts while S({j}) still read them")
                split_k(w, ck)
            if j > 0 and rng.random() < 0.3 and done["PV"] < j - 1:
                errors.append(f"warp {w} rescaled O while P V({j - 1}) was pending")
            p_ready.arrive()
            if not vt_wait_s and j + 1 < n:
                # planted: the next V^T as soon as V_{j+1} lands, without waiting for S_{j+1}
                cv2 = 2 * j + 3
                yield from wait(full[cv2 % slots], (cv2 // slots) & 1, f"warp {w} V early")
                if done["PV"] < j:
                    errors.append(f"warp {w} wrote V^T_{j + 1} while P V({j}) still read V^T_{j}")
        yield from wait(o_final, 0, f"warp {w} epilogue", 0)

    roles = [tensor_core(), producer(), issuer()] + [warp(w) for w in range(WARPS)]
    waiting, finished = {}, set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, rng.random(), ("run", i)))
    horizon = 20000.0 * (n + 4)
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
        if finished == set(range(1, len(roles))) and not pipe:
            break
    if finished != set(range(1, len(roles))):
        errors.append(f"deadlock: roles {sorted(set(range(1, len(roles))) - finished)} never finished")
    return errors


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 10])
@pytest.mark.parametrize("warp_cycles", [(300, 1500), (100, 5000)])
def test_tf32_forward_protocol_holds(n, warp_cycles):
    for seed in range(15):
        errs = simulate_tf32(n, seed, warp_cycles=warp_cycles)
        assert not errs, (n, seed, errs[:3])


def test_tf32_vt_rewrite_must_wait_for_s():
    assert sum(bool(simulate_tf32(n, seed, warp_cycles=(100, 5000), vt_wait_s=False))
               for n in (3, 5, 10) for seed in range(15)) > 0


def test_tf32_issuer_must_wait_for_p_ready():
    assert sum(bool(simulate_tf32(n, seed, warp_cycles=(100, 5000), issuer_waits_p=False))
               for n in (3, 5, 10) for seed in range(15)) > 0
