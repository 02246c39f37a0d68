"""A host-side model of bwd_main_kernel's mbarrier protocol (csrc/bwd.cu): the TMA producer,
the MMA thread and the two compute warpgroups, each a sequence of waits and arrivals.

Every barrier keeps its arrival count and completed phases; a wait names the phase it
expects (the kernel waits on its parity).  Over many random interleavings the model checks
that the protocol cannot deadlock, that no waiter is ever two phases behind its barrier
(where a parity wait would take the wrong phase), and that the tile maxima a readout takes
are those of its own query block.  MMAs and TMA copies complete when issued: only ordering
is modelled.  Both loop orders are covered: the plain one and the software-pipelined one
that D = 64 uses (dK, dQ and dP in TMEM columns of their own)."""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.done = name, count, 0, 0

    def arrive(self):
        self.arr += 1
        assert self.arr <= self.count, (self.name, "more arrivals than the count")
        if self.arr == self.count:
            self.arr = 0
            self.done += 1

    def passes(self, k):
        """Wait for completion k (0-based); the kernel's parity wait is only valid while
        the barrier is at most one completion ahead."""
        assert self.done <= k + 1, (self.name, "waiter two phases behind", k, self.done)
        return self.done > k


def model(n_it, pipe, first=False):
    """Actors of one CTA with n_it query blocks.  first=True takes the MMA and producer orders
    of the first pipelined version (everything else as now): its MMA thread waited for
    Q(it + 1) before issuing dV(it), and its producer kept the plain order (dO, dO's codes,
    then Q, one dO buffer)."""
    counts = {"kv": 1, "q_full0": 1, "q_full1": 1, "q_free0": 1 if pipe else 2, "q_free1": 1 if pipe else 2,
              "do_full0": 1, "do_full1": 1, "do_free0": 1, "do_free1": 1, "do8_full": 1, "do8_free": 1,
              "s": 1, "dp": 1, "p": 2, "dk": 1, "part": 1, "dk_read": 2, "dq_read": 2, "free_dp": 2}
    for b in range(2):
        for g in range(2):
            counts[f"ds{b}{g}"] = 1  # one arrival per compute group (128 threads in the kernel)
    B = {n: Bar(n, c) for n, c in counts.items()}
    smax = {}

    def W(name, k):
        return name, k

    def producer():
        B["kv"].arrive()
        if pipe and not first:
            # Q(0), dO(0), its codes; then per block j + 1: Q (after dK(j - 1)), dO into the
            # other of two buffers (after dP(j - 1)), its codes (after dV(j))
            B["q_full0"].arrive()
            B["do_full0"].arrive()
            B["do8_full"].arrive()
            for j in range(n_it - 1):
                q = j + 1
                if q > 1:
                    yield W(f"q_free{q & 1}", (q >> 1) - 1)
                B[f"q_full{q & 1}"].arrive()
                if q > 1:
                    yield W(f"do_free{q & 1}", (q >> 1) - 1)
                B[f"do_full{q & 1}"].arrive()
                yield W("do8_free", j)
                B["do8_full"].arrive()
        else:
            for it in range(n_it):
                if it > 0:
                    yield W("do_free0", it - 1)
                B["do_full0"].arrive()
                if it > 0:
                    yield W("do8_free", it - 1)
                B["do8_full"].arrive()
                if it > 1:
                    yield W(f"q_free{it & 1}", (it >> 1) - 1)
                B[f"q_full{it & 1}"].arrive()

    def issuer():
        yield W("kv", 0)

        def s_(it):
            B["s"].arrive()

        def dp_(it):
            B["dp"].arrive()
            B[f"do_free{it & 1 if pipe and not first else 0}"].arrive()

        def dv_(it):
            B["do8_free"].arrive()

        def dkdq_(it):
            B["dk"].arrive()
            if pipe:
                B[f"q_free{it & 1}"].arrive()  # dK is Q(it)'s last reader
            B["part"].arrive()

        if pipe:
            yield W("q_full0", 0)
            yield W("do_full0", 0)
            s_(0)
            dp_(0)
            # dO(it) of the double buffer, or of the single one of the first version
            do_wait = (lambda i: W("do_full0", i)) if first else (lambda i: W(f"do_full{i & 1}", i >> 1))
            for it in range(n_it):
                more = it + 1 < n_it
                yield W("p", it)
                yield W("do8_full", it)
                if not first:
                    dv_(it)
                    if more:
                        yield W(f"q_full{(it + 1) & 1}", (it + 1) >> 1)
                        s_(it + 1)
                else:
                    if more:
                        yield W(f"q_full{(it + 1) & 1}", (it + 1) >> 1)
                    dv_(it)
                    if more:
                        s_(it + 1)
                yield W(f"ds{it & 1}0", it >> 1)
                yield W(f"ds{it & 1}1", it >> 1)
                if it > 0:
                    yield W("dk_read", it - 1)
                    yield W("dq_read", it - 1)
                dkdq_(it)
                if more:
                    yield do_wait(it + 1)
                    yield W("free_dp", it)
                    dp_(it + 1)
        else:
            for it in range(n_it):
                yield W(f"q_full{it & 1}", it >> 1)
                if it > 0:
                    yield W("dk_read", it - 1)
                s_(it)
                yield W("do_full0", it)
                if it > 0:
                    yield W("free_dp", it - 1)
                dp_(it)
                yield W("p", it)
                yield W("do8_full", it)
                dv_(it)
                yield W(f"ds{it & 1}0", it >> 1)
                yield W(f"ds{it & 1}1", it >> 1)
                dkdq_(it)

    def compute(g):
        pending = [-1]  # Q buffer whose dQ boxes the TMA reduce still reads (plain order)

        def p_phase(it):
            yield W(f"q_full{it & 1}", it >> 1)
            yield W("s", it)
            B["p"].arrive()

        def ds_phase(it):
            yield W("dp", it)
            if pipe:
                B["free_dp"].arrive()
            if not pipe and pending[0] >= 0:
                B[f"q_free{pending[0]}"].arrive()
                pending[0] = -1
            smax[(it & 1, g)] = it
            B[f"ds{it & 1}{g}"].arrive()

        def readout(it):
            yield W("dk", it)
            yield W(f"ds{it & 1}0", it >> 1)
            yield W(f"ds{it & 1}1", it >> 1)
            assert smax[(it & 1, 0)] == it and smax[(it & 1, 1)] == it, ("tile maxima overwritten", it)
            B["dk_read"].arrive()

        def staging(it):
            yield W("part", it)
            B["dq_read" if pipe else "free_dp"].arrive()
            pending[0] = it & 1

        prev = None
        for s in range(n_it + (1 if pipe else 0)):
            if s < n_it:
                yield from p_phase(s)
            if pipe:
                if s > 0:
                    yield from readout(prev)
                    yield from staging(prev)
                if s < n_it:
                    yield from ds_phase(s)
                prev = s
            else:
                yield from ds_phase(s)
                yield from readout(s)
                yield from staging(s)

    return B, {"producer": producer(), "issuer": issuer(), "g0": compute(0), "g1": compute(1)}


def run(n_it, pipe, seed, first=False):
    """Random interleaving; returns None when every actor finishes, else the stuck waits."""
    rng = random.Random(seed)
    B, actors = model(n_it, pipe, first)
    waiting = {k: None for k in actors}
    alive = set(actors)
    while alive:
        ready = [k for k in alive if waiting[k] is None or B[waiting[k][0]].passes(waiting[k][1])]
        if not ready:
            return {k: waiting[k] for k in alive}
        k = rng.choice(ready)
        try:
            waiting[k] = next(actors[k])
        except StopIteration:
            alive.discard(k)
    return None


@pytest.mark.parametrize("pipe", [False, True], ids=["plain", "pipelined"])
def test_protocol_completes_in_every_interleaving(pipe):
    for n_it in range(1, 9):
        for seed in range(120):
            stuck = run(n_it, pipe, seed)
            assert stuck is None, f"n_it={n_it} seed={seed}: stuck at {stuck}"


def test_model_finds_the_first_versions_deadlock():
    """The first pipelined version's MMA thread waited for Q(it + 1) before issuing dV(it),
    while its producer loaded Q(it + 1) only after dV(it) had read dO's codes.  The kernel's
    bounded waits turned that into a timeout status on the GPU; the model reports the cycle."""
    for seed in range(20):
        stuck = run(2, True, seed, first=True)
        assert stuck is not None and stuck["issuer"] == ("q_full1", 0) and stuck["producer"] == ("do8_free", 0)
