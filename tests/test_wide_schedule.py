"""A model of the wide-head forward kernel's synchronisation, run on the CPU.

The kernel (csrc/fa_fwd_wide.cu) has a producer that fills a five-slot ring
with the pieces of K_j and V_j, one thread issuing the tensor-core MMAs, a
watcher that folds the V loads into the P-ready barriers, and four softmax
warps. All of them meet only on mbarriers whose waits test one parity bit.
This model runs the same roles as coroutines with random latencies, gives
each barrier the hardware's phase/parity rules and checks at every step that
  * an MMA reads only ring slots holding the load it expects, already landed,
  * P V of step j starts only after all four warps wrote P_j,
  * the S MMA into a buffer starts only after every warp has finished with
    the P it overwrites,
  * a parity wait never passes on a phase older than the one it targets,
  * no slot receives a load while its previous one is in flight,
  * nothing deadlocks.
The same model with a single P-ready barrier for all steps (an earlier form
of the kernel) must fail: a warp that finished step j can already hold
S_{j+1} and arrive for step j+1 before the slowest warp arrived for step j.
"""
import heapq
import random

import pytest

SLOTS = 5
SOFTMAX_WARPS = 4


class Barrier:
    """mbarrier: arrival count, transaction bytes, completed-phase counter."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.done = 0

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise AssertionError("more arrivals than the barrier's count in one phase")
        self._complete()

    def expect_tx(self, nbytes):
        self.tx += nbytes

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def passes(self, parity):
        # try_wait.parity: true once the phase with this parity has completed,
        # i.e. while the current phase has the other parity
        return (self.done & 1) != parity


def item_k(j):
    return 0 if j == 0 else 2 * j - 1


def item_v(j, n):
    return 2 * n - 1 if j == n - 1 else 2 * j + 2


def simulate(n, seed, split=True, softmax_cycles=(300, 1500), slots=SLOTS, watcher_gate=True,
             issuer_waits_k=True, pieces=2, paired=False, xchg_buffers=2):
    """Errors seen in one run of n key tiles. `pieces` is the number of slot
    loads per K or V tile: two in the bf16 kernel, one in the FP8 kernel
    (csrc/fa_fwd_fp8_wide.cu, six slots of 32 KB, whose protocol is
    otherwise the same). `paired` gives each row two softmax warps (one per
    64-key half, as in the FP8 kernel) that exchange their partial row maxima
    every step through a per-quarter barrier and a buffer per step parity
    (`xchg_buffers`). The other keyword switches take parts of the protocol
    out, to show what each one guards against."""
    rng = random.Random(seed)
    SLOTS = slots  # noqa: N806
    errors = []
    full = [Barrier(1) for _ in range(SLOTS)]
    empty = [Barrier(1) for _ in range(SLOTS)]
    warps = 2 * SOFTMAX_WARPS if paired else SOFTMAX_WARPS
    s_full = [Barrier(1), Barrier(1)]
    p_ready = [Barrier(warps + 1) for _ in range(2 if split else 1)]
    # row-max exchange: barrier per (lane quarter, step parity), two warps each;
    # xbuf[(buffer, half, quarter)] = the step whose maximum it holds
    xchg = [[Barrier(2) for _ in range(2)] for _ in range(SOFTMAX_WARPS)]
    xbuf = {}
    pv_done, o_final = Barrier(1), Barrier(1)

    def pr(j):
        return p_ready[j & 1] if split else p_ready[0]

    def pr_parity(j):
        return (j >> 1) & 1 if split else j & 1

    landed = [None] * SLOTS           # load index whose bytes sit in the slot
    in_flight = [None] * SLOTS
    s_buffer = [None, None]           # what a TMEM S buffer holds: ("S", j) or ("P", j)
    p_written = {}
    warp_done = [-1] * warps
    pipe = []
    clock = [0.0]
    events = []

    def wait_full(slot, load, who):
        yield ("wait", lambda: full[slot].passes((load // SLOTS) & 1))
        if full[slot].done < load // SLOTS + 1:
            errors.append(f"{who}: parity wait for load {load} passed on an older phase")

    def tensor_core():
        while True:
            while not pipe:
                yield ("wait", lambda: bool(pipe))
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
                continue
            kind, j, slot, load = op
            if landed[slot] != load or in_flight[slot] is not None:
                errors.append(f"{kind}({j}) read slot {slot} holding {landed[slot]}, wanted load {load}")
            if kind == "PV" and (p_written.get(j) != set(range(warps)) or s_buffer[j & 1] != ("P", j)):
                errors.append(f"PV({j}) started before every warp wrote P_{j}")
            if kind == "S" and j >= 2 and min(warp_done) < j - 2:
                errors.append(f"S({j}) overwrote P_{j - 2} while a warp still worked on it")
            yield ("delay", rng.uniform(400, 600))
            if kind == "S":
                s_buffer[j & 1] = ("S", j)

    def producer():
        for it in range(2 * n):
            for pc in range(pieces):
                load = pieces * it + pc
                slot = load % SLOTS
                yield ("wait", lambda s=slot, p=((load // SLOTS) & 1) ^ 1: empty[s].passes(p))
                if in_flight[slot] is not None:
                    errors.append(f"load {load} issued into slot {slot} with load {in_flight[slot]} in flight")
                full[slot].expect_tx(1)
                full[slot].arrive()
                in_flight[slot], landed[slot] = load, None

                def land(s=slot, ld=load):
                    in_flight[s], landed[s] = None, ld
                    full[s].complete_tx(1)
                heapq.heappush(events, (clock[0] + rng.uniform(300, 3000), rng.random(), ("call", land)))

    def issuer():
        def issue_s(j):
            it = item_k(j)
            for pc in range(pieces):
                load = pieces * it + pc
                if issuer_waits_k:
                    yield from wait_full(load % SLOTS, load, "issuer")
                pipe.append(("S", j, load % SLOTS, load))
                if pc < pieces - 1:
                    pipe.append(("commit", empty[load % SLOTS]))
            pipe.append(("commit", s_full[j & 1]))
            pipe.append(("commit", empty[(pieces * it + pieces - 1) % SLOTS]))

        yield from issue_s(0)
        if n > 1:
            yield from issue_s(1)
        for j in range(n):
            yield ("wait", lambda j=j: pr(j).passes(pr_parity(j)))
            it = item_v(j, n)
            for pc in range(pieces):
                load = pieces * it + pc
                pipe.append(("PV", j, load % SLOTS, load))
                pipe.append(("commit", empty[load % SLOTS]))
            pipe.append(("commit", pv_done))
            if j + 2 < n:
                yield from issue_s(j + 2)
        pipe.append(("commit", o_final))

    def watcher():
        def item(it):
            for pc in range(pieces):
                load = pieces * it + pc
                yield from wait_full(load % SLOTS, load, "watcher")

        yield from item(item_k(0))
        if n > 1:
            yield from item(item_k(1))
        for j in range(n):
            yield from item(item_v(j, n))
            if watcher_gate and split and j >= 2:
                yield ("wait", lambda j=j: pr(j).passes(((j >> 1) - 1) & 1))
            if watcher_gate and not split and j >= 1:
                yield ("wait", lambda j=j: pr(j).passes((j - 1) & 1))
            pr(j).arrive()
            if j + 2 < n:
                yield from item(item_k(j + 2))

    def softmax(w):
        quarter, half = w % SOFTMAX_WARPS, w // SOFTMAX_WARPS
        for j in range(n):
            yield ("wait", lambda j=j: s_full[j & 1].passes((j >> 1) & 1))
            if s_buffer[j & 1] != ("S", j) and s_buffer[j & 1] != ("P", j):
                errors.append(f"warp {w} read {s_buffer[j & 1]} at step {j}")
            if paired:
                yield ("delay", rng.uniform(20, 300))          # S out of TMEM, this half's maximum
                buf = j % xchg_buffers
                xbuf[(buf, half, quarter)] = j
                bar = xchg[quarter][j & 1]
                bar.arrive()
                yield ("wait", lambda b=bar, j=j: b.passes((j >> 1) & 1))
                if bar.done < (j >> 1) + 1:
                    errors.append(f"warp {w}: exchange wait for step {j} passed on an older phase")
                # the read may trail the wait, now and then by a long time
                yield ("delay", rng.uniform(0, 3000) if rng.random() < 0.2 else rng.uniform(0, 200))
                got = xbuf.get((buf, 1 - half, quarter))
                if got != j:
                    errors.append(f"warp {w} read its partner's maximum of step {got} at step {j}")
            yield ("delay", rng.uniform(*softmax_cycles))
            p_written.setdefault(j, set()).add(w)
            if p_written[j] == set(range(warps)):
                s_buffer[j & 1] = ("P", j)
            warp_done[w] = j
            pr(j).arrive()
        yield ("wait", lambda: o_final.passes(0))

    roles = [tensor_core(), producer(), issuer(), watcher()] + [softmax(w) for w in range(warps)]
    waiting = {}
    finished = set()
    for i in range(len(roles)):
        heapq.heappush(events, (0.0, rng.random(), ("run", i)))
    horizon = 20000.0 * (n + 4)      # far beyond any schedule that makes progress
    while events and clock[0] < horizon:
        clock[0], _, (what, arg) = heapq.heappop(events)
        if what == "call":
            arg()
            continue
        i = arg
        try:
            y = waiting.pop(i) if i in waiting else next(roles[i])
            while True:
                if y[0] == "delay":
                    heapq.heappush(events, (clock[0] + y[1], rng.random(), ("run", i)))
                    break
                if y[1]():
                    y = next(roles[i])
                    continue
                waiting[i] = y         # poll again later
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


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 12])
@pytest.mark.parametrize("softmax_cycles", [(300, 1500), (100, 5000)])
@pytest.mark.parametrize("slots,pieces,paired", [(SLOTS, 2, False), (12, 2, False), (6, 1, True), (12, 1, True)])
def test_wide_forward_protocol_holds(n, softmax_cycles, slots, pieces, paired):
    for seed in range(25):
        errs = simulate(n, seed, softmax_cycles=softmax_cycles, slots=slots, pieces=pieces, paired=paired)
        assert not errs, (n, seed, errs[:3])


def count_bad(**kw):
    return sum(bool(simulate(n, seed, softmax_cycles=(100, 5000), **kw)) for n in (2, 3, 4, 7) for seed in range(15))


def test_single_p_ready_barrier_races():
    """The model has teeth: the single-barrier protocol breaks."""
    assert count_bad(split=False) > 0


def test_issuer_must_wait_for_k():
    assert count_bad(issuer_waits_k=False) > 0


def test_fp8_ring_needs_split_p_ready_and_watcher_gate():
    """One load per tile in six slots (the FP8 kernel): the single-barrier
    protocol, an issuer that leaves the K wait to the ring, and a watcher that
    arrives without waiting for the previous phase all break. Unlike the
    five-slot bf16 ring, this ring lets V_{j+2} land before step j completes."""
    assert count_bad(split=False, slots=6, pieces=1) > 0
    assert count_bad(issuer_waits_k=False, slots=6, pieces=1) > 0
    assert count_bad(watcher_gate=False, slots=6, pieces=1) > 0


def test_fp8_row_max_exchange_needs_two_buffers():
    """With one exchange buffer a warp can overwrite its maximum for step
    j+1 before its partner has read the one of step j."""
    assert count_bad(slots=6, pieces=1, paired=True) == 0
    assert count_bad(slots=6, pieces=1, paired=True, xchg_buffers=1) > 0


def test_watcher_gate_needed_with_a_deeper_ring():
    """With five slots the ring itself keeps the watcher from arriving two
    steps ahead (V_{j+2} cannot land before step j completes); with a deeper
    ring only the watcher's wait for the previous phase does."""
    assert count_bad(watcher_gate=False) == 0
    assert count_bad(watcher_gate=False, slots=12) > 0
