"""A model of the FP8 forward kernel's synchronisation, run on the CPU.

The kernel (csrc/fa_fwd_fp8.cu) runs two query tiles per CTA. Each softmax
group reads S_j out of TMEM and at once signals "S consumed", so the issuer can
compute S_{j+1} into the same TMEM columns while the group works; the group
writes P_j into one of two shared-memory buffers and signals "P ready". A
watcher folds "K_{j+1} landed" into S-consumed and "V_j landed" into P-ready
(one P-ready barrier per tile and step parity);
ring slots go back by tensor-core commits. A rescale of the accumulator waits
for the previous P V on a per-group barrier.

As for the wide-head kernel, the roles run as coroutines with random
latencies over barriers with the hardware's parity rule, and every MMA, every
P write, every rescale and every parity wait is checked; planted changes show
what the S-consumed signal, the P double buffer and the rescale wait guard.
"""
import heapq
import random

import pytest

from test_wide_schedule import Barrier

SLOTS = 8
WARPS = 4


def simulate(nkv, seed, *, rescale_wait=True, p_buffers=2, early_s=True, split_p_ready=True,
             softmax_cycles=(300, 1500)):
    """One CTA with two query tiles whose key-tile counts are nkv[0], nkv[1]."""
    rng = random.Random(seed)
    errors = []
    nmax = max(nkv)
    full = [Barrier(1) for _ in range(SLOTS)]
    empty = [Barrier(1) for _ in range(SLOTS)]
    s_full = [Barrier(1) for _ in range(2)]
    s_cons = [Barrier(WARPS + 1) for _ in range(2)]
    # P-ready of tile i, step j: barrier [i][j % 2] (or one per tile)
    p_ready = [[Barrier(WARPS + 1) for _ in range(2 if split_p_ready else 1)] for _ in range(2)]

    def pr(i, j):
        return p_ready[i][j & 1] if split_p_ready else p_ready[i][0]

    def pr_parity(j):
        return (j >> 1) & 1 if split_p_ready else j & 1

    def pr_phase(j):
        return j >> 1 if split_p_ready else j

    pv_done = [Barrier(1) for _ in range(2)]
    o_final = [Barrier(1) for _ in range(2)]
    landed = [None] * SLOTS
    in_flight = [None] * SLOTS
    s_buf = [None, None]                       # ("S", j) in the TMEM S columns of tile i
    loaded = [[-1] * WARPS for _ in range(2)]  # last S_j each warp has read out of TMEM
    p_buf = {}                                 # (i, buffer) -> (j, warps written)
    pv_executed = [-1, -1]
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
            kind, i, j, slot, load = op
            if landed[slot] != load or in_flight[slot] is not None:
                errors.append(f"{kind}{i}({j}) read slot {slot} holding {landed[slot]}, wanted load {load}")
            if kind == "S" and j > 0 and min(loaded[i]) < j - 1:
                errors.append(f"S{i}({j}) overwrote S{i}({j - 1}) before every warp read it")
            if kind == "PV":
                buf = p_buf.get((i, j % p_buffers))
                if buf is None or buf[0] != j or buf[1] != set(range(WARPS)):
                    errors.append(f"PV{i}({j}) read P buffer holding {buf}")
            yield ("delay", rng.uniform(200, 300))
            if kind == "S":
                s_buf[i] = ("S", j)
            else:
                pv_executed[i] = j

    def producer():
        for c in range(2 * nmax):
            slot = c % SLOTS
            yield from wait(empty[slot], ((c // SLOTS) & 1) ^ 1, "producer")
            if in_flight[slot] is not None:
                errors.append(f"load {c} issued into slot {slot} with a load in flight")
            full[slot].expect_tx(1)
            full[slot].arrive()
            in_flight[slot], landed[slot] = c, None

            def land(s=slot, ld=c):
                in_flight[s], landed[s] = None, ld
                full[s].complete_tx(1)
            heapq.heappush(events, (clock[0] + rng.uniform(300, 3000), rng.random(), ("call", land)))

    def issuer():
        if nmax > 0:
            yield from wait(full[0], 0, "issuer", 0)
            for i in range(2):
                if nkv[i] > 0:
                    pipe.append(("S", i, 0, 0, 0))
                    pipe.append(("commit", s_full[i]))
            pipe.append(("commit", empty[0]))
        for j in range(nmax):
            slot_k, slot_v = (2 * j + 2) % SLOTS, (2 * j + 1) % SLOTS
            any_s = False
            for i in range(2):
                if j + 1 >= nkv[i]:
                    continue
                if early_s:
                    yield from wait(s_cons[i], j & 1, f"issuer s_cons{i}", j)
                else:
                    yield from wait(pr(i, j), pr_parity(j), f"issuer p_ready{i}", pr_phase(j))
                pipe.append(("S", i, j + 1, slot_k, 2 * j + 2))
                pipe.append(("commit", s_full[i]))
                any_s = True
            if any_s:
                pipe.append(("commit", empty[slot_k]))
            for i in range(2):
                if j >= nkv[i]:
                    continue
                if early_s or j + 1 >= nkv[i]:
                    yield from wait(pr(i, j), pr_parity(j), f"issuer p_ready{i}", pr_phase(j))
                pipe.append(("PV", i, j, slot_v, 2 * j + 1))
                pipe.append(("commit", pv_done[i]))
                if j + 1 == nkv[i]:
                    pipe.append(("commit", o_final[i]))
            pipe.append(("commit", empty[slot_v]))

    def watcher():
        if nmax > 0:
            yield from wait(full[0], 0, "watcher", 0)
        for j in range(nmax):
            cv = 2 * j + 1
            yield from wait(full[cv % SLOTS], (cv // SLOTS) & 1, "watcher", cv // SLOTS)
            for i in range(2):
                if j < nkv[i]:
                    # arrive for step j once the previous phase of the same barrier completed
                    if split_p_ready and j >= 2:
                        yield from wait(pr(i, j), ((j >> 1) - 1) & 1, "watcher gate", (j >> 1) - 1)
                    if not split_p_ready and j >= 1:
                        yield from wait(pr(i, j), (j - 1) & 1, "watcher gate", j - 1)
                    pr(i, j).arrive()
            if j + 1 >= nmax:
                continue
            ck = 2 * j + 2
            yield from wait(full[ck % SLOTS], (ck // SLOTS) & 1, "watcher", ck // SLOTS)
            for i in range(2):
                if j + 1 < nkv[i] and early_s:
                    if j > 0:
                        yield from wait(s_cons[i], (j - 1) & 1, "watcher gate", j - 1)
                    s_cons[i].arrive()

    def softmax(i, w):
        for j in range(nkv[i]):
            yield from wait(s_full[i], j & 1, f"softmax{i}", j)
            if s_buf[i] != ("S", j):
                errors.append(f"softmax{i} warp {w} read {s_buf[i]} at step {j}")
            loaded[i][w] = j
            if j + 1 < nkv[i] and early_s:
                s_cons[i].arrive()
            yield ("delay", rng.uniform(*softmax_cycles))
            b = j % p_buffers
            if j >= p_buffers and pv_executed[i] < j - p_buffers:
                errors.append(f"softmax{i} wrote P({j}) over P({j - p_buffers}) before its P V ran")
            cur = p_buf.get((i, b))
            if cur is None or cur[0] != j:
                p_buf[(i, b)] = (j, set())
            p_buf[(i, b)][1].add(w)
            if j > 0 and rng.random() < 0.3:          # the row max grew: rescale the accumulator
                if rescale_wait:
                    yield from wait(pv_done[i], (j - 1) & 1, f"softmax{i} rescale", j - 1)
                if pv_executed[i] < j - 1:
                    errors.append(f"softmax{i} rescaled O while P V({j - 1}) was pending")
                yield ("delay", rng.uniform(50, 200))
            pr(i, j).arrive()
        if nkv[i]:
            yield from wait(o_final[i], 0, f"softmax{i} epilogue", 0)

    roles = [tensor_core(), producer(), issuer(), watcher()]
    roles += [softmax(i, w) for i in range(2) for w in range(WARPS)]
    waiting, finished = {}, set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, rng.random(), ("run", i)))
    horizon = 20000.0 * (nmax + 4)
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


CASES = [(1, 1), (1, 2), (2, 3), (3, 3), (5, 6), (12, 13), (7, 0), (9, 9)]


@pytest.mark.parametrize("nkv", CASES)
@pytest.mark.parametrize("softmax_cycles", [(300, 1500), (100, 5000)])
def test_fp8_forward_protocol_holds(nkv, softmax_cycles):
    for seed in range(20):
        errs = simulate(nkv, seed, softmax_cycles=softmax_cycles)
        assert not errs, (nkv, seed, errs[:3])


def bad_runs(**kw):
    return sum(bool(simulate(nkv, seed, softmax_cycles=(100, 5000), **kw)) for nkv in [(3, 4), (6, 7), (9, 9)]
               for seed in range(15))


def test_rescale_must_wait_for_previous_p_v():
    assert bad_runs(rescale_wait=False) > 0


def test_one_p_buffer_is_not_enough():
    assert bad_runs(p_buffers=1) > 0


def test_single_p_ready_barrier_per_tile_races():
    """A warp holding S_{j+1} early can arrive for step j+1 before a slow warp
    (or the watcher) arrived for step j."""
    assert bad_runs(split_p_ready=False) > 0
