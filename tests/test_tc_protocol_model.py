"""CPU model of the synchronisation protocol of the two persistent tcgen05
kernels (csrc/wide.cu, csrc/prefill.cu), checked under random schedules.

The kernel's MMA warp waits on named barriers (bar.sync cannot time out), so
the protocol itself must make every sync complete: each phase of a barrier must
hold exactly one k-step's converter warps plus the MMA warp's sync of that same
k-step, after an abort too.  The model runs the roles of the kernel -- two
loader warps, four converter groups of four warps, the MMA warp -- against
mbarrier rings with phase parity and named barriers with the hardware's
arrival counting, with random delays and an abort injected at random times,
and asserts: no deadlock, every MMA sync phase holds the four converter warps
of its own k-step, and no mbarrier wait can alias a later phase.  A negative
control (one barrier per converter group instead of one per stage, an earlier
draft that hung on the GPU) must fail.  The ring sizes are read from the kernel
sources, so the model follows the kernels' constants.  The two kernels differ
in what frees a ring slot: in wide.cu the MMAs of the slot's previous k-step
(one commit frees slot and stage); in prefill.cu the converter warps that
widened the slot's previous k-step (the raw slot is free once they have read
it).  And in who fills it: in wide.cu the loader warps take turns; in
prefill.cu two loader threads each copy a part of every k-step (activations,
codes) and the slot is full once both copies have landed.
"""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "bitlinear_w1_a8_gb300", "csrc", "wide.cu")
SRC_PREFILL = os.path.join(ROOT, "bitlinear_w1_a8_gb300", "csrc", "prefill.cu")


def _const(text, name):
    m = re.search(r"constexpr\s+(?:int|uint32_t)\s+" + name + r"\s*=\s*([^;]+);", text)
    assert m, name
    return m.group(1).strip()


def kernel_constants():
    text = open(SRC).read()
    ring = int(_const(text, "kRing"))
    done = int(_const(text, "kDoneRing"))
    acc = int(_const(text, "kAccBufs"))
    max_tok = int(_const(text, "kMaxTok"))
    groups = int(_const(text, "kConvGroups"))
    group_warps = int(_const(text, "kGroupWarps"))
    loaders = int(_const(text, "kLoadWarps"))
    assert _const(text, "kWStages").startswith("(512 - kAccBufs * kMaxTok) / 32")
    stages = (512 - acc * max_tok) // 32
    # the barrier of k-step f and the waits, as the kernel writes them
    assert "named_bar_arrive(1 + f % kWStages" in text and "named_bar_sync(1 + stage" in text
    assert "const int prev = f - kWStages;" in text and "const int prev = f - kRing;" in text
    return dict(ring=ring, done=done, stages=stages, groups=groups, gw=group_warps, loaders=loaders, gate="mma")


def prefill_constants():
    """prefill.cu: four stages, converter group g = stage g = named barrier
    1 + g, and the stage's commit barrier empty[g] (phase f / 4 for k-step f)."""
    text = open(SRC_PREFILL).read()
    stages = int(_const(text, "kStages"))
    assert _const(text, "kConvGroups") == "kStages"
    assert "named_bar_arrive(1 + grp, kGroupThreads + 32);" in text and "named_bar_sync(1 + stage" in text
    assert "mbar_wait_lockstep(&ctl.empty[grp], (fill & 1u) ^ 1u" in text and "mma_commit(&ctl.empty[stage]);" in text
    assert "mbar_wait(&ctl.raw_empty[slot]" in text
    # two loader threads (activation tile, codes) each issue every k-step's
    # copy and arm the slot's barrier with it: a slot is full after both
    assert "if ((warp == kLoadWarp0 || warp == kLoadWarp0 + 1) && lane == 0) {" in text
    assert "for (int f = 0; f < total; ++f) {" in text and "mbar_init(&ctl.raw_full[s], 2);" in text
    # empty[g] serves the k-steps f with f % stages == g: a done ring of `stages` barriers
    return dict(ring=int(_const(text, "kRawStages")), done=stages, stages=stages, groups=stages,
                gw=int(_const(text, "kGroupWarps")), loaders=2, gate="conv", fill="all",
                ring_big=int(_const(text, "kRawStagesBig")))


class MBar:
    """Completed-phase counter of one mbarrier; a parity wait for phase k."""

    def __init__(self):
        self.completed = 0

    def done(self, k):
        if self.completed >= k + 2:
            raise AssertionError("mbarrier phase aliasing")
        return self.completed > k


def simulate(c, total, seed, abort_at=None, barrier_of=None):
    rnd = random.Random(seed)
    ring, done_n, stages, groups, gw, loaders = c["ring"], c["done"], c["stages"], c["groups"], c["gw"], c["loaders"]
    barrier_of = barrier_of or (lambda f: 1 + f % stages)
    ring_full = [MBar() for _ in range(ring)]
    done = [MBar() for _ in range(done_n)]
    bars = {}
    pending = []
    st = {"abort": False, "t": 0, "last": 0, "mma_done": -1}
    expect = 32 * gw + 32  # converter group + MMA warp, in threads

    def arrive(b, who, waiter=None):
        B = bars.setdefault(b, {"count": 0, "members": [], "waiters": []})
        B["count"] += 32
        B["members"].append(who)
        if waiter is not None:
            B["waiters"].append(waiter)
        if B["count"] == expect:
            for w in B["waiters"]:
                w["released"] = B["members"]
            B["count"], B["members"], B["waiters"] = 0, [], []

    raw_empty = [MBar() for _ in range(ring)]  # prefill: converter warps of the slot's k-step arrived
    raw_arrivals = {}

    fills = {}  # (slot, use) -> copies landed; "all": every loader fills every k-step

    def loader(li):
        share = range(total) if c.get("fill") == "all" else range(li, total, loaders)
        for f in share:
            if f >= ring:
                prev = f - ring
                if c["gate"] == "mma":
                    freed = lambda: done[prev % done_n].done(prev // done_n)
                else:
                    freed = lambda: raw_empty[prev % ring].done(prev // ring)
                while not freed():
                    if st["abort"]:
                        return
                    yield
            if st["abort"]:
                return
            slot, k = f % ring, f // ring

            def land(slot=slot, k=k):
                assert ring_full[slot].completed == k
                need = loaders if c.get("fill") == "all" else 1
                fills[(slot, k)] = fills.get((slot, k), 0) + 1
                if fills[(slot, k)] == need:
                    ring_full[slot].completed += 1
            pending.append((st["t"] + rnd.randint(1, 40), land))

    def converter(g, w):
        live = True
        for f in range(g, total, groups):
            if live:
                while not ring_full[f % ring].done(f // ring):
                    if st["abort"]:
                        live = False
                        break
                    yield
            prev = f - stages
            if prev >= 0:  # the lockstep wait: taken after an abort too
                while not done[prev % done_n].done(prev // done_n):
                    yield
            for _ in range(rnd.randint(0, 3)):
                yield
            if live and c["gate"] == "conv":  # one arrival per warp once the raw slot has been read
                raw_arrivals[f] = raw_arrivals.get(f, 0) + 1
                if raw_arrivals[f] == gw:
                    assert raw_empty[f % ring].completed == f // ring
                    raw_empty[f % ring].completed += 1
            arrive(barrier_of(f), ("conv", f))

    def mma():
        me = {}
        for f in range(total):
            me["released"] = None
            arrive(barrier_of(f), ("mma", f), waiter=me)
            while me["released"] is None:
                yield
            convs = [m for m in me["released"] if m[0] == "conv"]
            assert len(convs) == gw and all(m[1] == f for m in convs), (f, me["released"])

            def complete(f=f):
                assert st["mma_done"] == f - 1
                st["mma_done"] = f
                assert done[f % done_n].completed == f // done_n
                done[f % done_n].completed += 1
            t0 = max(st["t"], st["last"]) + rnd.randint(1, 30)
            st["last"] = t0
            pending.append((t0, complete))
            yield

    alive = [loader(i) for i in range(loaders)] + [converter(g, w) for g in range(groups) for w in range(gw)] + [mma()]
    steps = 0
    while alive:
        st["t"] += 1
        steps += 1
        if abort_at is not None and st["t"] == abort_at:
            st["abort"] = True
        for e in sorted([e for e in pending if e[0] <= st["t"]], key=lambda e: e[0]):
            pending.remove(e)
            e[1]()
        rnd.shuffle(alive)
        for a in list(alive[: rnd.randint(1, len(alive))]):
            try:
                next(a)
            except StopIteration:
                alive.remove(a)
        if steps > 100000:
            raise AssertionError(f"no progress (deadlock): total={total} seed={seed} abort_at={abort_at}")


@pytest.fixture(scope="module")
def consts():
    return kernel_constants()


@pytest.mark.parametrize("total", list(range(1, 21)) + [48, 83])
@pytest.mark.parametrize("big", [False, True])
def test_prefill_protocol_completes_and_phases_match(total, big):
    """Both raw-ring depths: 192-wide tiles and the 320-wide single-accumulator tiles."""
    c = prefill_constants()
    if big:
        c = dict(c, ring=c["ring_big"])
    for seed in range(6):
        simulate(c, total, seed)
        simulate(c, total, 3000 + seed, abort_at=random.Random(seed).randint(1, 300))


@pytest.mark.parametrize("total", list(range(1, 25)) + [40, 97])
def test_protocol_completes_and_phases_match(consts, total):
    for seed in range(6):
        simulate(consts, total, seed)
        simulate(consts, total, 1000 + seed, abort_at=random.Random(seed).randint(1, 300))


@pytest.mark.parametrize("total", [8, 24, 61])
def test_protocol_with_ten_stages(consts, total):
    """The one-accumulator layout (ten 32-column weight stages) keeps the
    protocol sound as well."""
    c = dict(consts, stages=10, done=16)
    for seed in range(6):
        simulate(c, total, seed)
        simulate(c, total, 2000 + seed, abort_at=random.Random(seed).randint(1, 300))


def test_negative_control_group_barriers_mix_phases(consts):
    """With ten stages, one barrier per converter group lets a group arrive for
    k-step f + 4 before the MMA warp synced k-step f (the draft that hung on the
    GPU): the model must catch it."""
    c = dict(consts, stages=10, done=16)
    groups = c["groups"]
    failed = 0
    for seed in range(20):
        try:
            simulate(c, 24, seed, barrier_of=lambda f: 1 + f % groups)
        except AssertionError:
            failed += 1
    assert failed > 0
