"""The FP8 unit mode's work counter, on a model.

attn_tc_kernel's persistent FP8 CTAs take units from a 64-bit word in the
workspace whose high 40 bits hold a launch epoch and low 24 bits a count
(tagged_increment).  A CTA adds one; if the value it added to carried another
epoch (an earlier launch's, or whatever the workspace held), it tries to
replace the word's current value by (epoch, 1) with compare-and-swap and so
takes count 0, re-reading the word while it still carries another epoch, and
adds again once another CTA has installed the epoch.  This model runs that
protocol in threads interleaved at every atomic step in random orders and
checks that the counts handed out are exactly 0, 1, 2, ... (each once), from
any starting word, and that a launch whose last CTA clears the word leaves it
ready for a launch with the same epoch (a replayed graph).
"""
import random

import pytest

MASK = (1 << 64) - 1
CNT = (1 << 24) - 1


def tagged_increment(mem, epoch):
    """Generator: yields before each atomic operation on mem[0]; returns the
    count (or -1 after too many lost races), like the kernel's."""
    for _ in range(64):
        yield
        old = mem[0]
        mem[0] = (old + 1) & MASK                       # atomicAdd
        if old >> 24 == epoch:
            return old & CNT
        cur = (old + 1) & MASK
        for _ in range(65536):
            yield
            seen = mem[0]                               # atomicCAS
            if seen == cur:
                mem[0] = ((epoch << 24) + 1) & MASK
                return 0
            if seen >> 24 == epoch:
                break
            cur = seen
    return -1


def run(threads, per_thread, epoch, start, rng):
    mem = [start]
    gens = []
    for t in range(threads):
        gens.append([tagged_increment(mem, epoch), per_thread])
    results = []
    live = list(range(threads))
    while live:
        i = rng.choice(live)
        g = gens[i]
        try:
            next(g[0])
        except StopIteration as e:
            results.append(e.value)
            g[1] -= 1
            if g[1] == 0:
                live.remove(i)
            else:
                g[0] = tagged_increment(mem, epoch)
    return results, mem[0]


@pytest.mark.parametrize("seed", range(200))
def test_counts_are_handed_out_once_each(seed):
    rng = random.Random(seed)
    threads = rng.choice([1, 2, 3, 8, 32])
    per = rng.choice([1, 2, 5])
    epoch = rng.randrange(1, 1 << 40)
    start = rng.choice([0, rng.randrange(1 << 64), ((epoch - 1) % (1 << 40)) << 24 | rng.randrange(1 << 24),
                        ((epoch ^ 1) << 24) | CNT])
    res, end = run(threads, per, epoch, start, rng)
    assert -1 not in res
    assert sorted(res) == list(range(threads * per)), (res, start)
    assert end == (epoch << 24) | (threads * per)


def test_same_epoch_after_the_clear():
    # a graph replayed with the same epoch: the last CTA cleared the word
    rng = random.Random(7)
    epoch = 12345
    res, end = run(8, 3, epoch, 0, rng)
    assert sorted(res) == list(range(24))
    res, end = run(8, 3, epoch, 0, rng)          # cleared to 0 between launches
    assert sorted(res) == list(range(24))


def test_model_sees_a_stale_same_epoch_word():
    # a word left with this very epoch (not cleared) is taken as current:
    # counts continue from it, which is why the last CTA clears the word
    rng = random.Random(3)
    epoch = 99
    res, _ = run(4, 1, epoch, (epoch << 24) | 10, rng)
    assert sorted(res) == [10, 11, 12, 13]
