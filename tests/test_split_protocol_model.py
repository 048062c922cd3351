"""CPU model of the K-split protocol of the decode kernel (csrc/decode.cu), checked
under random schedules.

With K split over a thread-block cluster, every CTA (rank) holds the same weight
rows and one K range; ranks 1 .. ks-1 add their row sums into rank 0's shared
memory (`red.shared::cluster.add`) and rank 0 writes the outputs.  Two halves of
the hardware cluster barrier order it: every thread arrives right after its CTA's
row sums are zeroed, waits just before the remote additions, and passes a full
barrier after them; rank 0 reads only after that.  The model runs the ranks with
random interleavings of their steps (zeroing, their own sums, the remote
additions, the barrier halves, rank 0's read and every CTA's exit) against a
barrier with the hardware's phase semantics (a wait returns once every rank has
arrived in the phase it arrived in), and asserts: no deadlock, rank 0 reads the
exact total, and no addition lands in a CTA's shared memory before its zeroing or
after it exited.  A negative control (the additions without the first wait) must
fail.  The protocol's statements are checked against the kernel source.
"""
import os
import random

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "bitlinear_w1_a8_gb300", "csrc", "decode.cu")


def test_kernel_follows_the_modelled_protocol():
    text = open(SRC).read()
    # the early arrive comes right after the row sums are zeroed, before the dependency wait
    zero = text.index("for (int i = t; i < MT * RR; i += kDecThreads) red[i] = 0;")
    early = text.index("if (ks > 1) cluster_arrive();", zero)
    assert early < text.index("pdl_wait_primary();", zero)
    # after the dots: the wait, the remote additions into rank 0, a full barrier, then rank 0 alone writes
    combine = text.index("if (ks > 1) {", early)
    body = text[combine:text.index("if (write_out) {", combine)]
    w, add = body.index("cluster_wait();"), body.index("red_add_cluster(red0")
    last = body.index("cluster_arrive();\n    cluster_wait();")
    assert w < add < last
    assert "rank == 0" in body[last:]
    # the barrier halves are the hardware cluster barrier with release / acquire
    assert '"barrier.cluster.arrive.release.aligned;"' in text
    assert '"barrier.cluster.wait.acquire.aligned;"' in text


class ClusterBarrier:
    """barrier.cluster: a wait returns once all ranks have arrived in the waiter's phase."""

    def __init__(self, n):
        self.n = n
        self.arrived = {}  # phase -> count
        self.phase_of = {}

    def arrive(self, rank):
        ph = self.phase_of.get(rank, 0)
        self.arrived[ph] = self.arrived.get(ph, 0) + 1
        self.phase_of[rank] = ph + 1
        return ph

    def done(self, ph):
        return self.arrived.get(ph, 0) == self.n


def run_protocol(ks, seed, first_wait=True):
    rng = random.Random(seed)
    values = [rng.randrange(-1000, 1000) for _ in range(ks)]
    red = [rng.randrange(1, 10**6) for _ in range(ks)]  # stale shared memory before zeroing
    zeroed = [False] * ks
    alive = [True] * ks
    bar = ClusterBarrier(ks)
    result = {}
    errors = []

    def rank_steps(r):
        red[r] = 0
        zeroed[r] = True
        yield
        ph_a = bar.arrive(r)
        yield
        # the rank's own sums (atomics into its own row sums), possibly split
        half = values[r] // 2
        red[r] += half
        yield
        red[r] += values[r] - half
        yield
        if first_wait:
            while not bar.done(ph_a):
                yield "blocked"
        if r != 0:
            if not zeroed[0] or not alive[0]:
                errors.append(f"rank {r} added into rank 0 before its zeroing or after its exit")
            red[0] += red[r]
            yield
        ph_b = bar.arrive(r)
        yield
        while not bar.done(ph_b):
            yield "blocked"
        if r == 0:
            result["total"] = red[0]
        alive[r] = False

    gens = {r: rank_steps(r) for r in range(ks)}
    steps = 0
    while gens:
        steps += 1
        if steps > 10000:
            raise AssertionError("deadlock")
        r = rng.choice(sorted(gens))
        try:
            next(gens[r])
        except StopIteration:
            del gens[r]
    return result.get("total"), sum(values), errors


@pytest.mark.parametrize("ks", [2, 4, 8])
def test_split_protocol_random_schedules(ks):
    for seed in range(400):
        total, expect, errors = run_protocol(ks, seed)
        assert not errors, errors
        assert total == expect, (seed, total, expect)


def test_split_protocol_negative_control():
    """Without the wait before the remote additions some schedule adds into rank 0's row
    sums before rank 0 zeroes them (the sum is lost) -- the model must notice."""
    failures = 0
    for seed in range(400):
        total, expect, errors = run_protocol(4, seed, first_wait=False)
        failures += bool(errors) or total != expect
    assert failures > 0
