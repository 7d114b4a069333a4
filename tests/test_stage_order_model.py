"""Deadlock freedom of the tensor-core attention kernel's stage order, on a model.

attn_tc_kernel's roles wait only on one another's barrier phases, so whether a
CTA can finish depends on the order in which they fill and free their rings.
This test plays that order out for the ring sizes the kernel instantiates, over
random lists of segments (a CTA's range: one unit after another, some leading
with their special tile), and checks that every role reaches its end:

  producer   loads each segment's Q once the previous segment's last QK
             product has read the old Q, then the segment's stages in load
             order -- K(0), K(x+1) before V(x), V(n-1); a special tile takes
             one stage (its K and V rows), no V part -- each into the next
             ring slot once that slot's previous stage was released.
             bf16: the ring is the NS-stage ring the MMA reads.  FP8: the ring
             is the NR-stage raw ring, and the widening warps move each stage,
             in the same order, into the NS-stage f16 ring (a raw slot is free
             once widened), after rewriting the segment's Q.
  MMA        per segment waits for Q (FP8: for the widened Q), then at step s
             issues QK(s) and PV(s - 1); with NS == KS a leading special tile's
             PV comes at step 0.  A K stage is released by its QK product, a V
             stage by its PV product, a special stage by its PV product.
  softmax    per tile waits for S (QK done) and for the previous tile's PV,
             then publishes P (bf16: first waits for the tile's V stages, whose
             rows without a token it zeroes).
  unit queue (FP8 unit mode, kq slots) the producer publishes each segment's
             unit before its Q and stages, into a slot every other role has
             read kq units before; the MMA thread, the softmax warps and the
             widening warps each take the segment's unit from the queue before
             their first step of it.

The same model with a ring too small for a whole V tile must deadlock, so the
check can see one.  (The model is kept with the kernel's stage order: a change
to one is a change to the other.)
"""
import random

import pytest


def _parts(n, special_first, last=False):
    """Parts of a segment of n tiles in load order: (tile x, is_v, special); the
    special tile is order index 0, or n - 1 with `last`."""
    out = []
    for P in range(2 * n):
        if P == 0:
            x, v = 0, False
        elif P == 2 * n - 1:
            x, v = n - 1, True
        else:
            x = (P - 1) // 2 + (1 if (P - 1) % 2 == 0 else 0)
            v = (P - 1) % 2 == 1
        sp = special_first and x == (n - 1 if last else 0)
        if sp and v:
            continue
        out.append((x, v, sp))
    return out


def runs_to_end(segs, NS, KS, NR=0, kq=None, spec_last=False):
    """True when every role finishes; NR > 0 models the FP8 kernel, kq the
    unit queue's slots (None: no queue)."""
    f8 = NR > 0
    early_special_ok = not spec_last    # a leading special tile's PV may come at step 0
    published = set()                   # units the producer published
    taken = {"mma": -1, "soft": -1, "widen": -1 if f8 else len(segs)}   # last unit taken

    def take(role, si):
        if kq is None or taken[role] >= si:
            return True
        if si not in published:
            return False
        taken[role] = si
        return True
    early_special = NS == KS and early_special_ok
    # stages in load order: (segment, tile, kind) with kind K, V or S (special)
    stages = []
    for si, (n, sp) in enumerate(segs):
        for x, v, s in _parts(n, sp, spec_last):
            kind = "S" if s else ("V" if v else "K")
            stages += [(si, x, kind)] * (1 if s else KS)
    by_part = {}
    for j, (si, x, kind) in enumerate(stages):
        by_part.setdefault((si, x, kind), []).append(j)
    last = {si: n - 1 for si, (n, sp) in enumerate(segs)}
    special = {(si, n - 1 if spec_last else 0) for si, (n, sp) in enumerate(segs) if sp}

    loaded, landed_ring, released = set(), set(), set()   # ring the MMA reads
    raw_free = set()                                       # FP8: raw slots freed
    q_loaded, q_ready = set(), set()
    qk, pv, p_pub = set(), set(), set()
    prod = widen = 0
    mma = []
    for si, (n, sp) in enumerate(segs):
        mma.append(("Q", si, 0))
        for step in range(n + 1):
            if step < n:
                mma.append(("QK", si, step))
            x = (0 if (sp and early_special) else -1) if step == 0 else step - 1
            if step == 1 and sp and early_special:
                x = -1
            if x >= 0:
                mma.append(("PV", si, x))
    soft = [(si, x) for si, (n, sp) in enumerate(segs) for x in range(n)]
    mp = sp_ = 0
    wq = 0   # FP8: segments whose Q the widening warps rewrote
    moved = True
    while moved:
        moved = False
        # producer
        while prod < len(stages):
            si = stages[prod][0]
            if kq is not None and si not in published:
                if si >= kq and min(taken.values()) < si - kq:
                    break
                published.add(si)
                moved = True
            if si not in q_loaded:
                if si > 0 and (si - 1, last[si - 1]) not in qk:
                    break
                q_loaded.add(si)
                moved = True
            ring = NR if f8 else NS
            if prod >= ring and (prod - ring) not in (raw_free if f8 else released):
                break
            loaded.add(prod)
            prod += 1
            moved = True
        if f8:
            # widening warps: Q of each segment, then its stages in order
            while widen < len(stages):
                si = stages[widen][0]
                if not take("widen", si):
                    break
                if wq <= si:
                    if si not in q_loaded:
                        break
                    q_ready.add(si)
                    wq = si + 1
                    moved = True
                if widen not in loaded or (widen >= NS and (widen - NS) not in released):
                    break
                landed_ring.add(widen)
                raw_free.add(widen)
                widen += 1
                moved = True
        else:
            landed_ring = loaded
            q_ready = q_loaded
        # MMA
        while mp < len(mma):
            op, si, x = mma[mp]
            if op == "Q":
                if not take("mma", si) or si not in q_ready:
                    break
            elif op == "QK":
                key = (si, x, "S") if (si, x) in special else (si, x, "K")
                if not all(j in landed_ring for j in by_part[key]):
                    break
                qk.add((si, x))
                if key[2] == "K":
                    released.update(by_part[key])
            else:
                if (si, x) not in p_pub:
                    break
                key = (si, x, "S") if (si, x) in special else (si, x, "V")
                if not all(j in landed_ring for j in by_part[key]):
                    break
                released.update(by_part[key])
                pv.add((si, x))
            mp += 1
            moved = True
        # softmax
        while sp_ < len(soft):
            si, x = soft[sp_]
            if not take("soft", si):
                break
            if (si, x) not in qk:
                break
            if sp_ > 0 and soft[sp_ - 1] not in pv:
                break
            if not f8 and (si, x) not in special:
                if not all(j in landed_ring for j in by_part[(si, x, "V")]):
                    break
            p_pub.add((si, x))
            sp_ += 1
            moved = True
    return prod == len(stages) and mp == len(mma) and sp_ == len(soft)


def _random_segments(rng):
    return [(rng.randint(1, 9), rng.random() < 0.6) for _ in range(rng.randint(1, 4))]


# (NS, KS) of the bf16 instantiations and (NS, KS, NR) of the FP8 ones
BF16 = [(3, 2), (6, 2), (5, 2), (4, 4), (5, 4)]
FP8 = [(5, 2, 3), (3, 2, 6), (3, 2, 4)]


@pytest.mark.parametrize("NS,KS", BF16)
def test_bf16_stage_order_finishes(NS, KS):
    rng = random.Random(1000 * NS + KS)
    for _ in range(1500):
        segs = _random_segments(rng)
        assert runs_to_end(segs, NS, KS), (NS, KS, segs)


@pytest.mark.parametrize("NS,KS,NR", FP8)
def test_fp8_stage_order_finishes(NS, KS, NR):
    rng = random.Random(1000 * NS + 10 * KS + NR)
    for _ in range(1500):
        segs = _random_segments(rng)
        assert runs_to_end(segs, NS, KS, NR), (NS, KS, NR, segs)


@pytest.mark.parametrize("NS,KS,NR", FP8)
def test_fp8_unit_queue_finishes(NS, KS, NR):
    # FP8 unit mode: each segment a whole unit taken through the 4-slot queue
    rng = random.Random(7000 + 1000 * NS + 10 * KS + NR)
    for _ in range(1500):
        segs = [(rng.randint(1, 9), True) for _ in range(rng.randint(1, 8))]
        assert runs_to_end(segs, NS, KS, NR, kq=4), (NS, KS, NR, segs)


@pytest.mark.parametrize("NS,KS", [(3, 2), (6, 2), (5, 2), (5, 4)])
def test_bf16_special_last_finishes(NS, KS):
    # unit mode with a ring deeper than one V tile: the special tile last
    rng = random.Random(9000 + 10 * NS + KS)
    for _ in range(1500):
        segs = [(rng.randint(1, 9), rng.random() < 0.8)]
        assert runs_to_end(segs, NS, KS, spec_last=True), (NS, KS, segs)


@pytest.mark.parametrize("NS,KS,NR", [(5, 2, 3)])
def test_fp8_special_last_with_unit_queue_finishes(NS, KS, NR):
    rng = random.Random(9100 + NS)
    for _ in range(1500):
        segs = [(rng.randint(1, 9), rng.random() < 0.8) for _ in range(rng.randint(1, 8))]
        assert runs_to_end(segs, NS, KS, NR, kq=4, spec_last=True), (NS, KS, NR, segs)


def test_model_sees_a_deadlock():
    # a bf16 ring of one stage cannot hold a 2-stage V tile whose rows the
    # softmax zeroes before the PV product that would free it
    assert not runs_to_end([(3, False)], 1, 2)
    # nor can an FP8 f16 ring of one stage: the PV product needs both V stages
    # widened before it frees either (a one-stage raw ring only serialises:
    # the widening warps free each raw slot as they go)
    assert not runs_to_end([(3, False)], 1, 2, 4)
    assert runs_to_end([(3, False)], 3, 2, 1)
    # the special tile last needs a ring deeper than one V tile: its stage is
    # held to its PV product, after the last V tile's
    assert not runs_to_end([(3, True)], 2, 2, spec_last=True)
    assert runs_to_end([(3, True)], 3, 2, spec_last=True)
    # a unit queue with no slot never publishes a unit
    assert not runs_to_end([(3, True), (2, True)], 5, 2, 3, kq=0)
    assert runs_to_end([(3, True), (2, True)], 5, 2, 3, kq=1)
