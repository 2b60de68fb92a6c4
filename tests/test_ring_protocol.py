"""Model check of the kernel's K/V ring protocols (host logic, no GPU).

The forward kernel streams K/V tiles through a shared-memory ring guarded by
mbarriers: the TMA producer waits on an empty barrier before it overwrites
ring space, the MMA issuer waits on a full barrier before it reads a tile, and
tcgen05 commits release tiles when the MMAs that read them complete.  Parity
waits on an mbarrier only tell the two most recent phases apart, so the
bookkeeping must never wait on a phase that the barrier may already have
passed twice.

This module restates the two protocols of `zyfa_fwd_kernel` step by step and
runs them under random interleavings of the producer, the issuer, TMA
completions and commit completions, checking that

- no ring space is overwritten before the tile in it was released,
- no full-barrier wait passes before the tile's bytes have landed,
- no tile is used after its release, and
- every run ends (no wait is left on a phase that never comes).

Slot ring (whole-tile slots, every form but BF16 d_qk = 192): tiles K_0 and
then (V_j, K_j+1) per step; each unit completes on the full barrier of its
first slot, armed with the bytes of both tiles; a slot is released by one
commit per tile at the end of the step.

Piece ring (BF16 d_qk = 192): a FIFO of pieces, a K tile taking three and a
V tile two consecutive pieces, a V tile never wrapping (it skips to piece 0
and keeps the skipped pieces); every tile completes on the full barrier of
its first piece; the producer waits for the release of the owner of a
tile's last piece; the issuer waits for K_j+1 just before its first S and
releases V_j right after its last P V.
"""

import random

import pytest

# (stage-0 tiles n0, stage-1 tiles n1) per work item: stage 1 runs one tile
# more, or is idle when its rows lie past the sequence end.


def _items(rnd, max_items=4, max_n0=6):
    out = []
    for _ in range(rnd.randint(1, max_items)):
        n0 = rnd.randint(1, max_n0)
        out.append((n0, rnd.choice([0, n0 + 1])))
    return out


class _Barrier:
    """An mbarrier reduced to its completed-phase count."""

    def __init__(self):
        self.phase = 0          # completed phases
        self.pending = 0        # tiles still to land on the armed phase

    def passes(self, parity):
        # try_wait.parity(P) returns once the phase with parity P completed:
        # the current (incomplete) phase has parity != P.
        return (self.phase & 1) != parity


class _Run:
    def __init__(self, rnd):
        self.rnd = rnd
        self.loaded = set()
        self.released = set()
        self.waited = set()
        self.tma = []        # (barrier, tile) copies in flight
        self.commits = []    # (barrier, tiles) in issue order

    def land(self, full):
        b, tile = self.tma.pop(self.rnd.randrange(len(self.tma)))
        self.loaded.add(tile)
        full[b].pending -= 1
        if full[b].pending == 0:
            full[b].phase += 1

    def complete_commit(self, empty):
        b, tiles = self.commits.pop(0)     # the tensor pipe completes in order
        empty[b].phase += 1
        self.released.update(tiles)


def _tile_sequence(items):
    seq = []          # (item, kind, j)
    for it, (n0, n1) in enumerate(items):
        for j in range(max(n0, n1)):
            seq.append((it, "K", j))
            seq.append((it, "V", j))
    return seq


def _issuer_ops(items, early_v_release, k_wait_before_s):
    """The issuer's program: waits, uses and commits on tile indices."""
    ops = []
    base = 0
    for n0, n1 in items:
        nload = max(n0, n1)
        K = lambda j: base + 2 * j
        V = lambda j: base + 2 * j + 1
        ops += [("wait", K(0)), ("use", K(0)), ("commit", K(0))]
        for j in range(nload):
            has_next = j + 1 < nload
            ops.append(("wait", V(j)))
            if not k_wait_before_s and has_next:
                ops.append(("wait_same", K(j + 1)))      # covered by V_j's unit barrier
            k_pending = k_wait_before_s and has_next
            s_last_v = 1 if j < n1 else 0
            for s in range(2):
                ns = n0 if s == 0 else n1
                if j >= ns:
                    continue
                ops.append(("use", V(j)))
                if early_v_release and s == s_last_v:
                    ops.append(("commit", V(j)))
                if j + 1 < ns:
                    if k_pending:
                        ops.append(("wait", K(j + 1)))
                        k_pending = False
                    ops.append(("use", K(j + 1)))
            if not early_v_release:
                ops.append(("commit", V(j)))
            if has_next:
                ops.append(("commit", K(j + 1)))
        base += 2 * nload
    return ops


def _simulate_slots(NS, items, seed, mutate=None):
    """Slot ring: returns True when the run ends with every tile used."""
    rnd = random.Random(seed)
    run = _Run(rnd)
    seq = _tile_sequence(items)
    full = [_Barrier() for _ in range(NS)]
    empty = [_Barrier() for _ in range(NS)]
    slot_of = {i: i % NS for i in range(len(seq))}
    occupant = [None] * NS
    unit_bar = None
    unit_first = {}     # tile -> slot whose full barrier completes it
    q = 0               # producer position
    ops = _issuer_ops(items, early_v_release=(mutate == "early_v"), k_wait_before_s=False)
    mi = 0
    fpar = [0] * NS
    while True:
        acts = []
        if q < len(seq):
            slot = slot_of[q]
            if empty[slot].passes(((q // NS) & 1) ^ 1):
                acts.append("P")
        if run.tma:
            acts.append("T")
        if mi < len(ops):
            op, t = ops[mi]
            if op == "wait":
                b = slot_of[t]      # the issuer's own walk: the unit's first slot
                if full[b].passes(fpar[b]):
                    acts.append("M")
            else:
                acts.append("M")
        if run.commits:
            acts.append("C")
        if not acts:
            return q == len(seq) and mi == len(ops) and not run.commits and not run.tma
        a = rnd.choice(acts)
        if a == "P":
            it, kind, j = seq[q]
            slot = slot_of[q]
            if occupant[slot] is not None:
                assert occupant[slot] in run.released, ("overwrite", NS, items, seed, q)
            occupant[slot] = q
            nload = max(items[it])
            if kind == "K" and j == 0:
                full[slot].pending += 1
                unit_first[q] = slot
                run.tma.append((slot, q))
            elif kind == "K":
                unit_first[q] = unit_bar
                run.tma.append((unit_bar, q))
            else:
                full[slot].pending += 1 + (1 if j + 1 < nload else 0)
                unit_first[q] = slot
                unit_bar = slot
                run.tma.append((slot, q))
            q += 1
        elif a == "T":
            run.land(full)
        elif a == "C":
            run.complete_commit(empty)
        else:
            op, t = ops[mi]
            mi += 1
            if op == "wait":
                b = slot_of[t]
                fpar[b] ^= 1
                run.waited.add(t)
                # the unit barrier covers V_j and K_j+1: both have landed
                assert t in run.loaded, ("wait passed before the load", NS, items, seed, t)
                if t + 1 < len(seq) and unit_first.get(t + 1) == b and seq[t][1] == "V":
                    assert t + 1 in run.loaded, ("unit passed before K landed", t)
                    run.waited.add(t + 1)
            elif op == "wait_same":
                assert t in run.waited
            elif op == "use":
                assert t in run.waited and t in run.loaded, ("use before wait", t)
                assert t not in run.released, ("use after release", NS, items, seed, t)
            else:
                run.commits.append((slot_of[t], [t]))


def _place(state, v, NP, nK, nV):
    """The kernel's piece placement: first piece, last piece, pieces taken."""
    n = nV if v else nK
    first = state["pc"]
    base = 0 if (v and first + n > NP) else first
    pc = base + n
    if pc >= NP:
        pc -= NP
    state["pc"] = pc
    last = NP - 1 if pc == 0 else pc - 1
    pieces, p = [], first
    while True:
        pieces.append(p)
        if p == last:
            break
        p = (p + 1) % NP
    return first, last, pieces


def _simulate_pieces(NP, nK, nV, items, seed, mutate=None):
    rnd = random.Random(seed)
    run = _Run(rnd)
    seq = _tile_sequence(items)
    full = [_Barrier() for _ in range(NP)]
    empty = [_Barrier() for _ in range(NP)]
    # both sides walk the same placement
    walk = {"pc": 0}
    placed = [_place(walk, kind == "V", NP, nK, nV) for (_, kind, _) in seq]
    own_b, own_par, own_valid, rel_par = [0] * NP, [0] * NP, [False] * NP, [0] * NP
    occupant = [None] * NP
    q = 0
    ops = _issuer_ops(items, early_v_release=(mutate != "late_v"),
                      k_wait_before_s=(mutate != "unit_wait"))
    if mutate == "v_release_before_use":
        # release V_j before its last P V: must be caught as a use after release
        fixed = []
        for op in ops:
            if op[0] == "commit" and seq[op[1]][1] == "V" and fixed and fixed[-1] == ("use", op[1]):
                fixed.insert(len(fixed) - 1, op)
            else:
                fixed.append(op)
        ops = fixed
    mi = 0
    fpar = [0] * NP
    while True:
        acts = []
        if q < len(seq):
            first, last, pieces = placed[q]
            w = first if mutate == "wait_first_piece" else last
            ok = True
            if own_valid[w]:
                ok = empty[own_b[w]].passes(own_par[w])
            if ok:
                acts.append("P")
        if run.tma:
            acts.append("T")
        if mi < len(ops):
            op, t = ops[mi]
            if op == "wait":
                b = placed[t][0]
                if full[b].passes(fpar[b]):
                    acts.append("M")
            elif op == "wait_same":
                acts.append("M")
            else:
                acts.append("M")
        if run.commits:
            acts.append("C")
        if not acts:
            return q == len(seq) and mi == len(ops) and not run.commits and not run.tma
        a = rnd.choice(acts)
        if a == "P":
            first, last, pieces = placed[q]
            for p in pieces:
                if occupant[p] is not None:
                    assert occupant[p] in run.released, ("overwrite", NP, items, seed, q)
            rp = rel_par[first]
            rel_par[first] ^= 1
            for p in pieces:
                own_b[p], own_par[p], own_valid[p], occupant[p] = first, rp, True, q
            full[first].pending += 1
            run.tma.append((first, q))
            q += 1
        elif a == "T":
            run.land(full)
        elif a == "C":
            run.complete_commit(empty)
        else:
            op, t = ops[mi]
            mi += 1
            if op == "wait":
                b = placed[t][0]
                fpar[b] ^= 1
                run.waited.add(t)
                assert t in run.loaded, ("wait passed before the load", NP, items, seed, t)
            elif op == "wait_same":
                # mutation "unit_wait": K_j+1 read on the strength of V_j's wait
                run.waited.add(t)
            elif op == "use":
                assert t in run.waited and t in run.loaded, ("use before its load", t)
                assert t not in run.released, ("use after release", NP, items, seed, t)
            else:
                run.commits.append((placed[t][0], [t]))


# The kernel's ring shapes: slots for BF16 d128 (5), FP8 d192 (7), FP8 d128
# (8); pieces for BF16 d192 (8 pieces, K 3, V 2).  Smaller shapes stress
# wrap-around and barrier reuse.
SLOT_SHAPES = [2, 3, 4, 5, 7, 8]
PIECE_SHAPES = [(8, 3, 2), (7, 3, 2), (4, 1, 1), (3, 1, 1), (2, 1, 1)]


@pytest.mark.parametrize("NS", SLOT_SHAPES)
def test_slot_ring_protocol(NS):
    for trial in range(300):
        rnd = random.Random(1000 * NS + trial)
        items = _items(rnd)
        assert _simulate_slots(NS, items, trial), ("deadlock", NS, items, trial)


@pytest.mark.parametrize("shape", PIECE_SHAPES)
def test_piece_ring_protocol(shape):
    NP, nK, nV = shape
    for trial in range(300):
        rnd = random.Random(7919 * NP + 31 * nK + trial)
        items = _items(rnd)
        assert _simulate_pieces(NP, nK, nV, items, trial), ("deadlock", shape, items, trial)


def test_piece_ring_late_v_release_also_holds():
    # The end-of-step release (the protocol before V_j was released early)
    # is safe as well; only its timing differs.
    for trial in range(200):
        rnd = random.Random(trial)
        assert _simulate_pieces(8, 3, 2, _items(rnd), trial, mutate="late_v")


def _fails(fn):
    try:
        return not fn()
    except AssertionError:
        return True


def test_model_catches_a_release_before_the_last_use():
    caught = any(_fails(lambda t=t: _simulate_pieces(8, 3, 2, _items(random.Random(t)), t,
                                                     mutate="v_release_before_use"))
                 for t in range(200))
    assert caught


def test_model_catches_reading_k_on_the_v_wait():
    # Without its own wait, K_j+1 can be read before its copy lands.
    caught = any(_fails(lambda t=t: _simulate_pieces(8, 3, 2, _items(random.Random(t)), t,
                                                     mutate="unit_wait"))
                 for t in range(200))
    assert caught


def test_model_catches_waiting_on_the_first_piece():
    # The newest earlier owner of a tile's pieces is the owner of its last
    # piece; waiting on the first piece's owner can let a copy overwrite a
    # piece still in use (or wait on a stale phase).
    caught = any(_fails(lambda t=t: _simulate_pieces(8, 3, 2, _items(random.Random(t)), t,
                                                     mutate="wait_first_piece"))
                 for t in range(300))
    assert caught
