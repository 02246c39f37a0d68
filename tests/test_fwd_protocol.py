"""A host-side model of fwd_kernel's mbarrier protocol (csrc/fwd.cu): the TMA producer (Q once,
then K and V tiles through two stages each), the MMA thread and the softmax of query tiles A
and B, each a sequence of waits and arrivals.

Over random interleavings the model checks that the protocol cannot deadlock, that no waiter
is ever two phases behind its barrier (where a parity wait would take the wrong phase), that
an S is only issued from the K tile it needs into columns its softmax has released, that a
softmax reads the S of its own key tile, and that P is only rewritten after the PV that read
it.  MMAs and TMA copies complete when issued: only ordering is modelled.  Covered: the plain
order, NVFP4 (the next S waits for the PV, which reads scale factors from S's columns),
Q-smoothing (the softmax also waits for the value tile, which carries the logit terms) and
ThriftAttention (promoted pairs skipped by both sides); non-causal, causal and a CTA without
tile B."""
import random

import pytest

KS = VS = 2  # K and V stages


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
        assert self.done <= k + 1, (self.name, "waiter two phases behind", k, self.done)
        return self.done > k


def model(lastA, lastB, mode, promoted):
    """lastX: the last key tile of tile X (-1: no tile B); promoted: set of (X, j) pairs that
    ThriftAttention computes elsewhere."""
    n_kv = max(lastA, lastB) + 1
    names = ["q"] + [f"k_full{s}" for s in range(KS)] + [f"k_empty{s}" for s in range(KS)]
    names += [f"v_full{s}" for s in range(VS)] + [f"v_empty{s}" for s in range(VS)]
    names += ["s_full0", "s_full1", "p_full0", "p_full1", "o_done0", "o_done1"]
    B = {n: Bar(n, 1) for n in names}  # each tile's softmax is one actor (its 256 arrivals)
    st = {"k": {}, "s": {0: None, 1: None}, "released": {0: True, 1: True}, "pv_done": {0: -1, 1: -1}}

    def use(X, j):
        return j <= (lastA if X == 0 else lastB) and (X, j) not in promoted

    def W(name, k):
        return name, k

    def producer():
        B["q"].arrive()
        for j in range(n_kv):
            if j >= KS:
                yield W(f"k_empty{j % KS}", j // KS - 1)
            st["k"][j % KS] = j
            B[f"k_full{j % KS}"].arrive()
            if j >= VS:
                yield W(f"v_empty{j % VS}", j // VS - 1)
            B[f"v_full{j % VS}"].arrive()

    def issuer():
        npv = [0, 0]

        def s_(X, j):
            assert st["k"][j % KS] == j, ("K stage holds another tile", X, j)
            assert st["released"][X], ("S columns still being read", X, j)
            st["s"][X], st["released"][X] = j, False
            B[f"s_full{X}"].arrive()

        def pv_(X, j):
            npv[X] += 1
            st["pv_done"][X] = j
            B[f"o_done{X}"].arrive()

        yield W("q", 0)
        yield W("k_full0", 0)
        for X in range(2):
            if use(X, 0):
                s_(X, 0)
        B["k_empty0"].arrive()
        for j in range(n_kv):
            nextk = j + 1 < n_kv
            if nextk:
                yield W(f"k_full{(j + 1) % KS}", (j + 1) // KS)
            yield W(f"v_full{j % VS}", j // VS)
            for X in range(2):
                if mode == "f4":
                    if not use(X, j):
                        continue
                    yield W(f"p_full{X}", npv[X])
                    pv_(X, j)
                    if not use(X, j + 1):
                        continue
                    yield W(f"o_done{X}", npv[X] - 1)
                    s_(X, j + 1)
                else:
                    pv = use(X, j)
                    if pv:
                        yield W(f"p_full{X}", npv[X])
                    if use(X, j + 1):
                        s_(X, j + 1)
                    if pv:
                        pv_(X, j)
            B[f"v_empty{j % VS}"].arrive()
            if nextk:
                B[f"k_empty{(j + 1) % KS}"].arrive()

    def softmax(X):
        last = lastA if X == 0 else lastB
        cnt = 0
        for j in range(last + 1):
            if (X, j) in promoted:
                continue
            yield W(f"s_full{X}", cnt)
            assert st["s"][X] == j, ("softmax reads the S of another key tile", X, j, st["s"][X])
            if mode == "qs":
                yield W(f"v_full{j % VS}", j // VS)
            if cnt > 0:
                yield W(f"o_done{X}", cnt - 1)
            # P(X, j) is written now: the PV of the previous processed tile has read P
            prev = max((i for i in range(j) if use(X, i)), default=-1)
            assert st["pv_done"][X] == prev, ("P rewritten before its PV", X, j)
            st["released"][X] = True
            B[f"p_full{X}"].arrive()
            cnt += 1
        if cnt > 0:
            yield W(f"o_done{X}", cnt - 1)

    actors = {"producer": producer(), "issuer": issuer(), "A": softmax(0)}
    if lastB >= 0:
        actors["B"] = softmax(1)
    return B, actors


def run(lastA, lastB, mode, promoted, seed):
    rng = random.Random(seed)
    B, actors = model(lastA, lastB, mode, promoted)
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


def shapes():
    out = []
    for n in range(1, 7):
        out.append((n - 1, n - 1))  # non-causal pair
        out.append((n - 1, -1))     # no tile B
    for qa in range(0, 8, 2):
        out.append((qa, qa + 1))    # causal pair
    return out


@pytest.mark.parametrize("mode", ["plain", "f4", "qs"])
def test_forward_protocol_completes(mode):
    for la, lb in shapes():
        for seed in range(60):
            stuck = run(la, lb, mode, set(), seed)
            assert stuck is None, f"{mode} lastA={la} lastB={lb} seed={seed}: stuck at {stuck}"


def test_forward_protocol_with_promoted_pairs():
    """ThriftAttention: random promoted pairs, skipped by the MMA thread and the softmax."""
    rng = random.Random(7)
    for la, lb in shapes():
        for seed in range(40):
            tiles = [(0, j) for j in range(la + 1)] + [(1, j) for j in range(lb + 1)]
            promoted = {p for p in tiles if rng.random() < 0.3}
            stuck = run(la, lb, "plain", promoted, seed)
            assert stuck is None, f"lastA={la} lastB={lb} promoted={sorted(promoted)}: stuck at {stuck}"
