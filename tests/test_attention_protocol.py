"""A discrete-event model of one persistent attention block's barrier protocol:
the roles and phase rules of k_attention.cu, namely the TMA lane that publishes
items and feeds the K/V ring, the MMA lane, and the two softmax groups.

Random and skewed timings check four properties:
  * the protocol cannot deadlock;
  * every mbarrier wait finds its barrier at the awaited phase or one past it
    (parity waits cannot tell phases two apart);
  * every reader of the two-entry item ring reads its own item;
  * an item's first PV product, which overwrites O, comes after the softmax
    group has read the previous item's O.

The model mirrors the kernel's barrier order by hand: a change to that order
in the kernel is a change here too.
"""
import heapq
import inspect
import random

import pytest

SLOTS = 3    # K/V ring slots
TILES = 2    # query tiles (softmax groups) per block


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; `done` phases so far."""

    def __init__(self, count=1):
        self.count, self.pending, self.done = count, 0, 0


def run(items, n_ctx, causal, seed, skew=(1, 1, 1, 1)):
    """Simulate one block working through `items` (256-query block indices of
    one head).  skew scales the TMA, softmax-A, softmax-B and epilogue times."""
    rnd = random.Random(seed)
    f_tma, f_sm0, f_sm1, f_epi = skew
    n_all = (n_ctx + 127) // 128

    def tiles(t, mb):  # key tiles of query tile t of block mb
        return (min(2 * mb + 1 + t, n_all) if causal else n_all)

    bars = {}
    now = [0.0]
    events = []          # (time, seq, process or "ARRIVE", payload)
    seq = [0]
    waiting = {}         # barrier name -> [(process, phase)]
    ring = [None, None]  # the item ring: (ordinal, item)
    tensor_free = [0.0]  # the tensor core runs MMAs in issue order
    last_mma_done = [0.0]
    o_read_end = {0: {}, 1: {}}      # item ordinal -> time the group finished reading O
    first_pv_issue = {0: [], 1: []}  # (item ordinal, time)

    def bar(name):
        return bars.setdefault(name, Barrier())

    def push(time, who, payload=None):
        seq[0] += 1
        heapq.heappush(events, (time, seq[0], who, payload))

    def arrive(name):
        b = bar(name)
        b.pending += 1
        if b.pending == b.count:
            b.pending = 0
            b.done += 1
            for proc, _ in waiting.pop(name, []):
                push(now[0], proc)

    def mma(duration=1.0):
        start = max(now[0], tensor_free[0])
        tensor_free[0] = last_mma_done[0] = start + duration

    def commit(name):  # arrives once every MMA issued so far has completed
        push(max(now[0], last_mma_done[0]), "ARRIVE", name)

    def land(name, lo, hi):  # a TMA load completing on `name`
        push(now[0] + f_tma * rnd.uniform(lo, hi), "ARRIVE", name)

    def producer():
        n = 0
        for k in range(len(items) + 1):
            if k > 0:
                yield ("wait", "q_empty", k - 1)
            item = items[k] if k < len(items) else -1
            ring[k & 1] = (k, item)
            arrive("item")
            if item < 0:
                return
            land("q_full", 1, 5)
            for _ in range(2 * tiles(1, item)):
                slot = n % SLOTS
                if n >= SLOTS:
                    yield ("wait", f"empty{slot}", n // SLOTS - 1)
                land(f"full{slot}", 0.5, 4)
                n += 1

    def mma_lane():
        nb, p_seen = 0, [0, 0]
        for k in range(len(items) + 1):
            yield ("wait", "item", k)
            ordinal, item = ring[k & 1]
            assert ordinal == k, ("MMA lane read another item's ring entry", k, ordinal)
            if item < 0:
                return
            n_a, n_b = tiles(0, item), tiles(1, item)
            yield ("wait", "q_full", k)
            yield ("wait", f"full{nb % SLOTS}", nb // SLOTS)
            mma(); commit("s0"); mma(); commit("s1"); commit(f"empty{nb % SLOTS}")
            for j in range(n_b):
                n = nb + 2 * j + 1
                yield ("wait", f"full{n % SLOTS}", n // SLOTS)
                more_a, more_b = j + 1 < n_a, j + 1 < n_b
                if j < n_a:
                    yield ("wait", "p0", p_seen[0]); p_seen[0] += 1
                    if j == 0:
                        first_pv_issue[0].append((k, now[0]))
                    mma()
                    if more_a:
                        n2 = nb + 2 * j + 2
                        yield ("wait", f"full{n2 % SLOTS}", n2 // SLOTS)
                        mma(); commit("s0")
                    else:
                        commit("o0")
                yield ("wait", "p1", p_seen[1]); p_seen[1] += 1
                if j == 0:
                    first_pv_issue[1].append((k, now[0]))
                mma(); commit(f"empty{(nb + 2 * j + 1) % SLOTS}")
                if more_b:
                    if not more_a:
                        n2 = nb + 2 * j + 2
                        yield ("wait", f"full{n2 % SLOTS}", n2 // SLOTS)
                    mma(); commit("s1"); commit(f"empty{(nb + 2 * j + 2) % SLOTS}")
                else:
                    commit("o1")
                if j + 2 == n_b or (n_b == 1 and j == 0):
                    commit("q_empty")
            nb += 2 * n_b

    def softmax(t):
        s_seen = 0
        scale = f_sm1 if t else f_sm0
        for k in range(len(items) + 1):
            yield ("wait", "item", k)
            ordinal, item = ring[k & 1]
            assert ordinal == k, ("softmax group read another item's ring entry", t, k, ordinal)
            if item < 0:
                return
            for _ in range(tiles(t, item)):
                yield ("wait", f"s{t}", s_seen); s_seen += 1
                yield ("delay", scale * rnd.uniform(0.5, 3))
                arrive(f"p{t}")
            yield ("wait", f"o{t}", k)
            yield ("delay", f_epi * rnd.uniform(1, 4))
            o_read_end[t][k] = now[0]

    procs = {"producer": producer(), "mma": mma_lane(), "softmax0": softmax(0), "softmax1": softmax(1)}
    for name in procs:
        push(0.0, name)
    finished = set()
    while events:
        time, _, who, payload = heapq.heappop(events)
        now[0] = time
        if who == "ARRIVE":
            arrive(payload)
            continue
        gen = procs[who]
        try:
            while True:
                cmd = next(gen)
                if cmd[0] == "delay":
                    push(now[0] + cmd[1], who)
                    break
                _, name, phase = cmd
                b = bar(name)
                assert b.done in (phase, phase + 1), (who, cmd, "barrier has completed", b.done)
                if b.done == phase + 1:
                    continue
                waiting.setdefault(name, []).append((who, phase))
                break
        except StopIteration:
            finished.add(who)
    assert finished == set(procs), ("deadlock", set(procs) - finished)
    for t in (0, 1):
        for k, time in first_pv_issue[t]:
            if k > 0:
                assert time >= o_read_end[t][k - 1], ("O overwritten before it was read", t, k)
    return True


SKEWS = [(1, 1, 1, 1), (20, 1, 1, 1), (0.05, 1, 1, 1), (1, 30, 1, 1), (1, 1, 30, 1), (1, 1, 1, 50)]


@pytest.mark.parametrize("n_ctx", [1, 128, 129, 300, 1000, 4096])
@pytest.mark.parametrize("causal", [True, False])
def test_protocol_model(n_ctx, causal):
    blocks = (n_ctx + 255) // 256
    for trial in range(12):
        rnd = random.Random(trial)
        items = [rnd.randrange(blocks) for _ in range(rnd.randint(1, 8))]
        for skew in SKEWS:
            assert run(items, n_ctx, causal, seed=trial * 7 + n_ctx, skew=skew)


def test_model_catches_publishing_before_the_release():
    # publishing an item before the previous item's Q release (the order the
    # model first caught) lets the ring run two entries ahead of the MMA lane
    src = inspect.getsource(run)
    good = ("            if k > 0:\n                yield (\"wait\", \"q_empty\", k - 1)\n"
            "            item = items[k] if k < len(items) else -1\n"
            "            ring[k & 1] = (k, item)\n            arrive(\"item\")\n"
            "            if item < 0:\n                return\n")
    bad = ("            item = items[k] if k < len(items) else -1\n"
           "            ring[k & 1] = (k, item)\n            arrive(\"item\")\n"
           "            if item < 0:\n                return\n"
           "            if k > 0:\n                yield (\"wait\", \"q_empty\", k - 1)\n")
    assert good in src
    ns = dict(globals())
    exec(src.replace(good, bad), ns)
    with pytest.raises(AssertionError):
        for trial in range(20):
            ns["run"]([0, 0, 0, 0], 100, True, seed=trial)


def test_model_catches_releasing_q_before_the_first_p():
    # releasing Q as soon as a one-tile item's S products are issued, before
    # both softmax groups have written the item's first P, lets the producer
    # publish ring entries while a group is still finishing the previous item
    # (the release rule a draft with P in shared memory got wrong)
    src = inspect.getsource(run)
    good = "            mma(); commit(\"s0\"); mma(); commit(\"s1\"); commit(f\"empty{nb % SLOTS}\")\n"
    bad = ("            mma(); commit(\"s0\"); mma(); commit(\"s1\"); commit(f\"empty{nb % SLOTS}\")\n"
           "            if n_b == 1:\n                commit(\"q_empty\")\n")
    rule = "                if j + 2 == n_b or (n_b == 1 and j == 0):\n"
    assert good in src and rule in src
    mutated = src.replace(good, bad).replace(rule, "                if j + 2 == n_b:\n")
    ns = dict(globals())
    exec(mutated, ns)
    with pytest.raises(AssertionError):
        for trial in range(40):
            for skew in SKEWS:
                ns["run"]([0, 0, 0, 0, 0, 0], 100, True, seed=trial, skew=skew)
