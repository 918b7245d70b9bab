"""A host model of the decode kernel's barrier protocol (K/V slot ring, S^T and P^T buffers).

The kernel's arithmetic is restated here: K of the CTA's tile n is ring item 2n and V item
2n + 1, in slot item % SLOTS, loaded on that slot's FULL barrier in phase item / SLOTS; the
producer waits for the slot's EMPTY barrier with parity ((item / SLOTS) & 1) ^ 1 before reusing it;
the MMA thread issues QK(0), then for every n: QK(n + 1), waits for P-full(n), PV(n); the
softmax waits for S-full(n) and, from n = 2, for P-free(n - 2) on the same buffer.

Every barrier is modelled with the hardware's parity semantics (a wait on parity p passes
while the barrier's current phase has the other parity), copies and products complete at random
later times (products in issue order), and the agents run in a random interleaving.  Checked for
every slot count the kernel's configurations use and for short and long shares:
  * every parity wait agrees with the true condition (the completions it needs have happened,
    and no more than one phase beyond): a wait never passes early and never blocks on a phase
    that has already moved on;
  * no buffer is rewritten while its last reader may still run: a K/V slot is reloaded only after
    the product that read it completed, S^T buffer n & 1 is overwritten by QK(n) only after the
    softmax of tile n - 2 released it, and P^T buffer n & 1 only after PV(n - 2) completed;
  * the protocol never deadlocks, and every tile is loaded, multiplied and released in order.
"""
import random

import pytest


class Bar:
    def __init__(self):
        self.done = 0  # completed phases

    def passes(self, parity):
        return (self.done & 1) != parity


def _simulate(slots, n_tiles, seed, empty_flip=1, pfree_back=2):
    """empty_flip / pfree_back restate the kernel's waits; other values plant a mistake."""
    rng = random.Random(seed)
    full = [Bar() for _ in range(slots)]
    empty = [Bar() for _ in range(slots)]
    sfull, pfull, pfree = [Bar(), Bar()], [Bar(), Bar()], [Bar(), Bar()]
    slot_of = lambda item: item % slots
    parity_of = lambda item: (item // slots) & 1

    def check(bar, parity, needed):
        """A parity wait that needs `needed` completions: its answer must be the true condition."""
        ok = bar.passes(parity)
        assert bar.done <= needed + 1, "the barrier ran two phases past a waiter"
        assert ok == (bar.done >= needed), (bar.done, needed, parity)
        return ok

    loads = []       # in-flight copies: FULL barrier indices, complete in any order
    tensor = []      # issued products: lists of barriers to complete, in issue order
    slot_item = [None] * slots  # item held by each slot (for the ordering checks)
    consumed = set()
    pv_done = set()  # tiles whose PV product has completed

    # producer state
    item = 0
    # MMA state: next step
    mma = {"qk": 0, "pv": 0}
    # softmax state
    sm = {"n": 0}

    def producer_step():
        nonlocal item
        if item >= 2 * n_tiles:
            return False
        s = slot_of(item)
        if item >= slots and not check(empty[s], parity_of(item) ^ empty_flip, item // slots):
            return False
        if item >= slots:
            assert slot_item[s] in consumed, "a slot reused before its product read it"
        slot_item[s] = item
        loads.append(s)
        item += 1
        return True

    def mma_step():
        n_qk, n_pv = mma["qk"], mma["pv"]
        # program order: QK(0), then per n: QK(n + 1) (if any), PV(n)
        want_qk = n_qk < n_tiles and n_qk == n_pv + (0 if n_pv == 0 and n_qk == 0 else 1)
        if want_qk:
            it = 2 * n_qk
            if not check(full[slot_of(it)], parity_of(it), it // slots + 1):
                return False
            assert slot_item[slot_of(it)] == it
            # S^T buffer n_qk & 1 held tile n_qk - 2 until its softmax released P-full(n_qk - 2)
            assert n_qk < 2 or sm["n"] >= n_qk - 1, "S^T overwritten before its softmax read it"
            tensor.append([("empty", slot_of(it), it), ("sfull", n_qk & 1, None)])
            mma["qk"] += 1
            return True
        if n_pv < n_tiles:
            n = n_pv
            if not check(pfull[n & 1], (n >> 1) & 1, (n >> 1) + 1):
                return False
            it = 2 * n + 1
            if not check(full[slot_of(it)], parity_of(it), it // slots + 1):
                return False
            assert slot_item[slot_of(it)] == it
            tensor.append([("empty", slot_of(it), it), ("pfree", n & 1, n)])
            mma["pv"] += 1
            return True
        return False

    def softmax_step():
        n = sm["n"]
        if n >= n_tiles:
            return False
        if not check(sfull[n & 1], (n >> 1) & 1, (n >> 1) + 1):
            return False
        if n >= pfree_back:  # P^T buffer n & 1 was last read by PV(n - 2)
            m = n - pfree_back
            if not check(pfree[m & 1], (m >> 1) & 1, (m >> 1) + 1):
                return False
        # P^T buffer n & 1 is written now: its previous reader PV(n - 2) must have completed
        assert n < 2 or (n - 2) in pv_done, "P^T rewritten while PV(n - 2) may still read it"
        pfull[n & 1].done += 1  # the 128 arrivals of tile n
        sm["n"] += 1
        return True

    def copy_lands():
        if not loads:
            return False
        full[loads.pop(rng.randrange(len(loads)))].done += 1
        return True

    def product_completes():
        if not tensor:
            return False
        for kind, idx, it in tensor.pop(0):
            if kind == "empty":
                consumed.add(it)
                empty[idx].done += 1
            elif kind == "sfull":
                sfull[idx].done += 1
            else:
                pv_done.add(it)
                pfree[idx].done += 1
        return True

    agents = [producer_step, mma_step, softmax_step, copy_lands, product_completes]
    for _ in range(200 * (n_tiles + slots)):
        order = agents[:]
        rng.shuffle(order)
        if not any(a() for a in order):
            break
    assert item == 2 * n_tiles and mma["qk"] == n_tiles and mma["pv"] == n_tiles and sm["n"] == n_tiles, \
        ("deadlock", item, mma, sm)
    assert not loads and not tensor
    assert len(consumed) == 2 * n_tiles


@pytest.mark.parametrize("slots", [4, 5, 6, 9, 11, 12])
@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5, 8, 13, 40])
def test_decode_ring_protocol(slots, n_tiles):
    for seed in range(20):
        _simulate(slots, n_tiles, seed * 1000 + slots * 10 + n_tiles)


def test_stricter_waits_are_accepted():
    """Waiting for PV(n - 1) instead of PV(n - 2) is slower but correct: the model accepts it."""
    for seed in range(10):
        _simulate(5, 13, seed, pfree_back=1)


@pytest.mark.parametrize("planted", [dict(empty_flip=0), dict(pfree_back=3)])
def test_model_catches_a_planted_mistake(planted):
    """The model is not vacuous: the producer's EMPTY wait on the slot's own parity (a slot reused
    before its product read it), or a P-free wait one tile too early (P^T rewritten while PV(n - 2)
    may still read it), fails it."""
    failed = 0
    for seed in range(20):
        try:
            _simulate(5, 13, seed, **planted)
        except AssertionError:
            failed += 1
    assert failed > 0, planted
