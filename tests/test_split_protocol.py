"""Model of the last-wave split's cross-CTA protocol (d = 128 backward,
FP8 forward), run under random schedules on the CPU.

An item split into f parts runs as f CTAs.  Each part stores its partial
result in a slot of its own, publishes it (CTA barrier, release fence) and
adds one to the item's byte counter; four items share a 32-bit word of the
workspace's status block.  The part whose add returns f - 1 is the last: it
clears its byte (an atomic AND, so that the other three items' counts in the
word survive), takes an acquire fence, sums the f slots in part order (its
own values from its registers) and writes the result.

The model checks, over many schedules and several launches on the same
counters:
  * exactly one part of every item finds itself last;
  * the last part reads every other part's slot after that part published it;
  * every counter word is zero after each launch (the next launch needs it);
  * the merged value is the same, bit for bit, whichever part is last;
and that it finds the two mistakes the design avoids: counting before
publishing, and clearing the whole word instead of the item's byte."""
import random

import numpy as np


class Stale(Exception):
    pass


def part_steps(item, part, f, slots_visible, slots_pending, counters, results, own, reset_word=False,
               count_first=False):
    """One part as a sequence of steps (a generator); yields between steps."""
    word, sh = item // 4, 8 * (item % 4)
    # the slot's stores: pending (not yet visible to other CTAs)
    slots_pending[(item, part)] = own[(item, part)]
    yield

    def publish():
        slots_visible[(item, part)] = slots_pending.pop((item, part))

    def count():
        old = counters[word]
        counters[word] = (old + (1 << sh)) & 0xFFFFFFFF
        return (old >> sh) & 0xFF

    if count_first:
        n = count() + 1
        yield
        publish()
    else:
        publish()                           # CTA barrier + release fence
        yield
        n = count() + 1                     # the atomic add
    yield
    if n == f:
        if reset_word:
            counters[word] = 0
        else:
            counters[word] &= ~(0xFF << sh) & 0xFFFFFFFF
        yield
        # acquire; sum the slots in part order, own from registers
        acc = None
        for o in range(f):
            if o == part:
                v = own[(item, part)]
            else:
                if (item, o) not in slots_visible:
                    raise Stale((item, o))
                v = slots_visible[(item, o)]
            acc = v.copy() if acc is None else (acc + v).astype(np.float32)
        results.setdefault(item, []).append((part, acc))


def launch(rng, n_items, f, counters, own, **mut):
    slots_visible, slots_pending, results = {}, {}, {}
    gens = [part_steps(i, j, f, slots_visible, slots_pending, counters, results, own, **mut)
            for i in range(n_items) for j in range(f)]
    live = list(gens)
    while live:
        g = rng.choice(live)
        try:
            next(g)
        except StopIteration:
            live.remove(g)
    return results


def merged_in_order(item, f, own):
    acc = None
    for o in range(f):
        v = own[(item, o)]
        acc = v.copy() if acc is None else (acc + v).astype(np.float32)
    return acc


def make_own(rng, n_items, f):
    g = np.random.default_rng(rng.randrange(1 << 30))
    return {(i, j): (g.standard_normal(8) * 10.0 ** g.integers(-3, 4)).astype(np.float32)
            for i in range(n_items) for j in range(f)}


def test_split_protocol_one_last_part_zeroed_counters_order_free_sum():
    rng = random.Random(7)
    for trial in range(300):
        n_items = rng.randint(1, 11)
        f = rng.randint(2, 4)
        counters = [0] * 56                 # status block words 8..63
        for _ in range(3):                  # launches on the same counters
            own = make_own(rng, n_items, f)
            res = launch(rng, n_items, f, counters, own)
            assert sorted(res) == list(range(n_items)), (trial, res.keys())
            for i, lst in res.items():
                assert len(lst) == 1, (trial, i, lst)
                assert np.array_equal(lst[0][1], merged_in_order(i, f, own)), (trial, i)
            assert all(c == 0 for c in counters), (trial, counters)


def test_split_model_finds_counting_before_publishing():
    rng = random.Random(11)
    found = False
    for _ in range(300):
        n_items, f = rng.randint(1, 6), rng.randint(2, 4)
        try:
            launch(rng, n_items, f, [0] * 56, make_own(rng, n_items, f), count_first=True)
        except Stale:
            found = True
            break
    assert found


def test_split_model_finds_clearing_the_whole_word():
    rng = random.Random(13)
    found = False
    for _ in range(300):
        n_items, f = rng.randint(2, 8), rng.randint(2, 4)
        counters = [0] * 56
        res = launch(rng, n_items, f, counters, make_own(rng, n_items, f), reset_word=True)
        if sorted(res) != list(range(n_items)) or any(len(v) != 1 for v in res.values()) or any(counters):
            found = True
            break
    assert found
