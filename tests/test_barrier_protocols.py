"""A model of the FP8 forward kernel's roles and mbarriers, run under random
schedules, that checks the one rule a parity wait depends on.

`mbarrier.try_wait.parity(P)` answers "has the phase of parity P completed?"
by comparing P with the parity of the phase in progress.  The answer is right
only while the barrier has completed exactly the phases before the awaited one
or one more: two more and the wait sleeps through a completed phase; fewer and
it returns before its phase is done.  Each wait in the model names the phase
it means, and every poll compares the parity answer with the truth.

The roles follow `fa_fwd_fp8_kernel`: a producer fills a ring of K/V stages; an
MMA issuer computes, per key tile, the next tile's S_x for both query tiles,
then O_x += P_x V for both, then releases the stage; two softmax warpgroups
load S_x, release it, write P_x into one of two shared-memory buffers (after
the product that last read that buffer), and sometimes rescale O_x (after the
previous product).  Tensor-core commits and TMA copies complete later, in
order, at random times.  The softmax keeps P in shared memory, so it can run a
tile ahead of the products: the old layout, one P-ready barrier per query
tile, then lets that barrier get two phases ahead of the issuer.  The test
checks that the model finds exactly that, and nothing with one P-ready
barrier per P buffer."""
import random
from collections import deque

STAGES = 3


class Alias(Exception):
    pass


class Deadlock(Exception):
    pass


class Barrier:
    def __init__(self, count=1):
        self.count, self.pending, self.done = count, 0, 0      # done = completed phases

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending, self.done = 0, self.done + 1

    def poll(self, parity, phase):
        """The parity wait's answer; raises if it differs from whether `phase` completed."""
        answer = (self.done & 1) != (parity & 1)
        truth = self.done > phase
        if answer != truth:
            raise Alias(f"waiting for phase {phase} with {self.done} completed")
        return answer


def issuer(n_tiles, per_buffer_pfull):
    """Per key tile u: S of tile u+1 for each query tile that sees it, P.V of
    tile u, then the stage release.  Query tile x sees tiles 0 .. n_tiles[x]-1."""
    total = max(n_tiles)
    ns, nv = [0, 0], [0, 0]
    yield ("wait", "QFULL", 0, 0)
    yield ("wait", ("KFULL", 0), 0, 0)
    for x in range(2):
        if n_tiles[x] > 0:
            yield ("commit", ("SFULL", x))
            ns[x] += 1
    for u in range(total):
        s = u % STAGES
        if u + 1 < total:
            k = (u + 1) // STAGES
            yield ("wait", ("KFULL", (u + 1) % STAGES), k & 1, k)
            for x in range(2):
                if u + 1 >= n_tiles[x]:
                    continue
                yield ("wait", ("SFREE", x), (ns[x] - 1) & 1, ns[x] - 1)
                yield ("commit", ("SFULL", x))
                ns[x] += 1
        vwaited = False
        for x in range(2):
            if u >= n_tiles[x]:
                continue
            if per_buffer_pfull:
                yield ("wait", ("PFULL", x, nv[x] & 1), (nv[x] >> 1) & 1, nv[x] >> 1)
            else:
                yield ("wait", ("PFULL", x), nv[x] & 1, nv[x])
            if not vwaited:
                yield ("wait", ("VFULL", s), (u // STAGES) & 1, u // STAGES)
                vwaited = True
            yield ("commit", ("PFREE", x, nv[x] & 1))
            nv[x] += 1
        yield ("commit", ("KVEMPTY", s))
    yield ("commit", ("OFULL", 0))
    yield ("commit", ("OFULL", 1))


def producer(n_tiles):
    total = max(n_tiles)
    if total:
        yield ("tma", "QFULL")
    for u in range(total):
        s, k = u % STAGES, u // STAGES
        yield ("wait", ("KVEMPTY", s), (k & 1) ^ 1, k - 1)
        yield ("tma", ("KFULL", s))
        yield ("tma", ("VFULL", s))


def softmax(x, n, per_buffer_pfull, rng, p_rescale):
    for it in range(n):
        yield ("wait", ("SFULL", x), it & 1, it)
        yield ("arrive", ("SFREE", x))
        b = it & 1
        if it >= 2:
            yield ("wait", ("PFREE", x, b), ((it >> 1) - 1) & 1, (it >> 1) - 1)
        if it > 0 and rng.random() < p_rescale:
            pb = (it - 1) & 1
            yield ("wait", ("PFREE", x, pb), ((it - 1) >> 1) & 1, (it - 1) >> 1)
        yield ("arrive", ("PFULL", x, b) if per_buffer_pfull else ("PFULL", x))
    if n:
        yield ("wait", ("OFULL", x), 0, 0)


def run(seed, n_tiles, per_buffer_pfull, p_rescale=0.3, max_steps=200000):
    rng = random.Random(seed)
    bars = {}

    def bar(name):
        if name not in bars:
            bars[name] = Barrier()
        return bars[name]

    roles = {"producer": producer(n_tiles), "issuer": issuer(n_tiles, per_buffer_pfull),
             "softmax0": softmax(0, n_tiles[0], per_buffer_pfull, rng, p_rescale),
             "softmax1": softmax(1, n_tiles[1], per_buffer_pfull, rng, p_rescale)}
    nxt = {r: next(g, None) for r, g in roles.items()}
    mma, tma = deque(), deque()
    # skewed speeds: some roles (and the async engines) run much slower than others
    weight = {r: rng.choice([0.05, 0.3, 1.0, 3.0]) for r in list(roles) + ["mma", "tma"]}
    for _ in range(max_steps):
        ready = []
        for r, op in nxt.items():
            if op is None:
                continue
            if op[0] != "wait":
                ready.append(r)
                continue
            try:
                if bar(op[1]).poll(op[2], op[3]):
                    ready.append(r)
            except Alias as e:
                raise Alias(f"{r} on {op[1]}: {e}") from None
        if mma:
            ready.append("mma")
        if tma:
            ready.append("tma")
        if not ready:
            if all(op is None for op in nxt.values()):
                return
            raise Deadlock({r: op for r, op in nxt.items() if op is not None})
        r = rng.choices(ready, weights=[weight[q] for q in ready])[0]
        if r == "mma":
            bar(mma.popleft()).arrive()
        elif r == "tma":
            bar(tma.popleft()).arrive()
        else:
            op = nxt[r]
            if op[0] == "arrive":
                bar(op[1]).arrive()
            elif op[0] == "commit":
                mma.append(op[1])
            elif op[0] == "tma":
                tma.append(op[1])
            nxt[r] = next(roles[r], None)
    raise AssertionError("model did not finish")


TILE_COUNTS = [(1, 1), (2, 2), (3, 3), (7, 7), (12, 12), (3, 5), (5, 6), (0, 4), (8, 1)]


def test_per_buffer_pready_barriers_never_alias():
    for i in range(600):
        run(seed=i, n_tiles=TILE_COUNTS[i % len(TILE_COUNTS)], per_buffer_pfull=True)


def test_model_finds_the_alias_of_one_pready_barrier_per_query_tile():
    found = []
    for i in range(600):
        try:
            run(seed=i, n_tiles=TILE_COUNTS[i % len(TILE_COUNTS)], per_buffer_pfull=False)
        except Alias as e:
            found.append(str(e))
    assert len(found) > 50
    # always the issuer, on a P-ready barrier that has run two phases ahead
    assert all(f.startswith("issuer on ('PFULL'") for f in found), found[:3]
    assert all("with" in f and int(f.split("with ")[1].split()[0]) == int(f.split("phase ")[1].split()[0]) + 2
               for f in found)


def test_model_checker_catches_a_waiter_that_runs_ahead():
    b = Barrier()
    assert not b.poll(0, 0)
    try:
        b.poll(1, 1)            # phase 1 awaited while phase 0 is still open: parity says "done"
    except Alias:
        pass
    else:
        raise AssertionError("alias not reported")
    b.arrive()
    b.arrive()
    try:
        b.poll(0, 0)            # two phases on: parity says "not done"
    except Alias:
        pass
    else:
        raise AssertionError("alias not reported")
