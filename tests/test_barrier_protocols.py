"""Models of the forward (bf16 and FP8), split-KV decode and backward
(d = 64 and d = 128) kernels' roles and mbarriers, run under random schedules, that check
the one rule a parity wait depends on.

`mbarrier.try_wait.parity(P)` answers "has the phase of parity P completed?"
by comparing P with the parity of the phase in progress.  The answer is right
only while the barrier has completed exactly the phases before the awaited one
or one more: two more and the wait sleeps through a completed phase; fewer and
it returns before its phase is done.  Each wait in the model names the phase
it means, and every poll compares the parity answer with the truth.

The roles follow `fa_fwd_fp8_kernel`: a producer fills a ring of K/V stages;
one MMA issuer per query tile x computes, per key tile, the next tile's S_x,
then O_x += P_x V, then releases the stage (a stage is free after both
issuers' releases; an issuer whose query tile skips a key tile releases it
once the stage holds that tile); two softmax warpgroups
load S_x, release it, write P_x into one of two shared-memory buffers (after
the product that last read that buffer), and sometimes rescale O_x (after the
previous product).  Tensor-core commits and TMA copies complete later, in
order, at random times.  The softmax keeps P in shared memory, so it can run a
tile ahead of the products: the old layout, one P-ready barrier per query
tile, then lets that barrier get two phases ahead of the issuer.  The test
checks that the model finds exactly that, and nothing with one P-ready
barrier per P buffer.

The models check barrier phases only: a wait that guards data rather than a
phase (the backward producer's wait before it restages LSE and D, say) shows
up here only if dropping it lets a barrier run two phases ahead."""
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


def issuer(x, n_tiles, per_buffer_pfull):
    """Query tile x's issuer.  It walks the union of the key tiles both query
    tiles see; query tile x sees tiles 0 .. n_tiles[x]-1."""
    total = max(n_tiles)
    ns = nv = 0
    yield ("wait", "QFULL", 0, 0)
    yield ("wait", ("KFULL", 0), 0, 0)
    if n_tiles[x] > 0:
        yield ("commit", ("SFULL", x))
        ns += 1
    for u in range(total):
        s = u % STAGES
        if u + 1 < n_tiles[x]:
            k = (u + 1) // STAGES
            yield ("wait", ("KFULL", (u + 1) % STAGES), k & 1, k)
            yield ("wait", ("SFREE", x), (ns - 1) & 1, ns - 1)
            yield ("commit", ("SFULL", x))
            ns += 1
        if u < n_tiles[x]:
            if per_buffer_pfull:
                yield ("wait", ("PFULL", x, nv & 1), (nv >> 1) & 1, nv >> 1)
            else:
                yield ("wait", ("PFULL", x), nv & 1, nv)
            yield ("wait", ("VFULL", s), (u // STAGES) & 1, u // STAGES)
            yield ("commit", ("PFREE", x, nv & 1))
            nv += 1
            yield ("commit", ("KVEMPTY", s))
        else:
            yield ("wait", ("KFULL", s), (u // STAGES) & 1, u // STAGES)
            yield ("arrive", ("KVEMPTY", s))
    if n_tiles[x] > 0:
        yield ("commit", ("OFULL", x))


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


def schedule(rng, roles, count, max_steps=400000):
    """Run the roles (generators of operations) under a random schedule with
    skewed role speeds.  Commits of one role complete in their issue order;
    bulk copies complete in any order.  `count(name)` is a barrier's arrival
    count per phase."""
    bars = {}

    def bar(name):
        if name not in bars:
            bars[name] = Barrier(count(name))
        return bars[name]

    nxt = {r: next(g, None) for r, g in roles.items()}
    mma = {r: deque() for r in roles}
    tma = []
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
        ready += ["mma " + q for q in mma if mma[q]]
        if tma:
            ready.append("tma")
        if not ready:
            if all(op is None for op in nxt.values()):
                return
            raise Deadlock({r: op for r, op in nxt.items() if op is not None})
        r = rng.choices(ready, weights=[weight[q.split()[0]] for q in ready])[0]
        if r.startswith("mma"):
            bar(mma[r.split()[1]].popleft()).arrive()
        elif r == "tma":
            bar(tma.pop(rng.randrange(len(tma)))).arrive()
        else:
            op = nxt[r]
            if op[0] == "arrive":
                bar(op[1]).arrive()
            elif op[0] == "commit":
                mma[r].append(op[1])
            elif op[0] == "tma":
                tma.append(op[1])
            nxt[r] = next(roles[r], None)
    raise AssertionError("model did not finish")


def run(seed, n_tiles, per_buffer_pfull, p_rescale=0.3):
    rng = random.Random(seed)
    roles = {"producer": producer(n_tiles), "issuer0": issuer(0, n_tiles, per_buffer_pfull),
             "issuer1": issuer(1, n_tiles, per_buffer_pfull),
             "softmax0": softmax(0, n_tiles[0], per_buffer_pfull, rng, p_rescale),
             "softmax1": softmax(1, n_tiles[1], per_buffer_pfull, rng, p_rescale)}
    schedule(rng, roles, lambda name: 2 if name[0] == "KVEMPTY" else 1)   # a stage: both issuers


# ---------------------------------------------------------------- d = 128 backward
# The roles of `fa_bwd128_kernel` for one key tile and n query blocks: a
# producer (K, V once; per block Q into one of two stages, dO into one slot),
# the LSE/D stager (one buffer each, refilled as soon as the P and the dS
# pass have read them; under the causal mask the producer stages both behind
# the previous block's dS pass), the MMA issuer (per block dV, dQ^T, dK,
# then the next block's S^T and dP^T), the compute warpgroups (P^T, dS^T)
# and the dQ drain warpgroup.  The phase each wait means is the block index
# (or half of it for the two Q stages).

def bwd_producer(n, stages_lse=False):
    """stages_lse: the causal mode, where the producer stages LSE and D of
    block i itself once the dS pass has read block i-1's."""
    yield ("tma", "KV")
    for i in range(n):
        s = i & 1
        yield ("wait", ("QEMPTY", s), ((i >> 1) & 1) ^ 1, (i >> 1) - 1)     # dK(i-2) read Q stage s
        yield ("tma", ("QFULL", s))
        yield ("wait", "DVDONE", (i & 1) ^ 1, i - 1)                        # dV(i-1) read dO
        yield ("tma", "DOFULL")
        if stages_lse:
            yield ("wait", "DFREE", (i & 1) ^ 1, i - 1)
            yield ("arrive", "LSE")
            yield ("arrive", "D")


def bwd_stager(n):
    """LSE of block i once the P pass has read block i-1's, D once the dS pass
    has read block i-1's (one buffer each)."""
    for i in range(n):
        if i > 0:
            yield ("wait", "LSEFREE", (i - 1) & 1, i - 1)
        yield ("arrive", "LSE")
        if i > 0:
            yield ("wait", "DFREE", (i - 1) & 1, i - 1)
        yield ("arrive", "D")


def bwd_issuer(n):
    if n:
        yield ("wait", "KV", 0, 0)
        yield ("wait", ("QFULL", 0), 0, 0)
        yield ("wait", "DOFULL", 0, 0)
        yield ("commit", "SFULL")
        yield ("commit", "DPFULL")
    for i in range(n):
        s = i & 1
        yield ("wait", "PFULL", i & 1, i)
        yield ("commit", "DVDONE")                                          # dV(i)
        yield ("wait", "DSFULL", i & 1, i)
        yield ("wait", "DVDONE", i & 1, i)
        yield ("commit", "DQFULL")                                          # dQ^T(i)
        yield ("commit", ("QEMPTY", s))                                     # dK(i)
        if i + 1 < n:
            yield ("wait", ("QFULL", s ^ 1), ((i + 1) >> 1) & 1, (i + 1) >> 1)
            yield ("wait", ("QEMPTY", s), (i >> 1) & 1, i >> 1)
            yield ("commit", "SFULL")                                       # S^T(i+1)
            yield ("wait", "DOFULL", (i + 1) & 1, i + 1)
            yield ("wait", "DQFREE", i & 1, i)
            yield ("commit", "DPFULL")                                      # dP^T(i+1)
    if n:
        yield ("commit", "ACC")


def bwd_compute(n):
    for i in range(n):
        yield ("wait", "LSE", i & 1, i)
        yield ("wait", "SFULL", i & 1, i)
        yield ("arrive", "PFULL")
        yield ("arrive", "LSEFREE")
        yield ("wait", "DPFULL", i & 1, i)
        yield ("wait", "D", i & 1, i)
        yield ("arrive", "DSFULL")
        yield ("arrive", "DFREE")
    if n:
        yield ("wait", "ACC", 0, 0)


def bwd_drain(n):
    for i in range(n):
        yield ("wait", "DQFULL", i & 1, i)
        yield ("arrive", "DQFREE")


def run_bwd128(seed, n, causal=False):
    rng = random.Random(seed)
    roles = {"producer": bwd_producer(n, stages_lse=causal), "issuer": bwd_issuer(n),
             "compute": bwd_compute(n), "drain": bwd_drain(n)}
    if not causal:
        roles["stager"] = bwd_stager(n)
    schedule(rng, roles, lambda name: 1)


# ---------------------------------------------------------------- bf16 forward
# `fa_fwd_kernel`, persistent: the producer takes work items one after
# another and publishes each in one of two slots (ITEM), reusing a slot once
# every consumer has released it (ITEMFREE: the issuer and both softmax
# warpgroups); it loads an item's Q once the previous item's S products are
# done (QEMPTY, committed after the item's last S) and streams the item's key
# tiles through the ring.  An item lists `count` key-tile entries, and query
# tile x sees entry e iff vis[x][e].  P overwrites S in TMEM, so the issuer
# alternates the query tiles: per entry and query tile x, O_x += P_x V once
# P_x is written, then the next entry's S_x once that product has read P_x
# (also across items: the first S_x of an item waits for the previous item's
# last P_x V).  Every counter (ring uses, S, P.V, loaded items) runs on across
# items.

def fwd_producer(items, stages, q_empty_wait=True, slot_free_wait=True):
    m = u = 0
    for k, it in enumerate(list(items) + [None]):
        if k >= 2 and slot_free_wait:
            yield ("wait", ("ITEMFREE", k & 1), ((k >> 1) - 1) & 1, (k >> 1) - 1)
        yield ("arrive", ("ITEM", k & 1))
        if it is None:
            return
        count, _ = it
        if not count:
            continue
        if m > 0 and q_empty_wait:
            yield ("wait", "QEMPTY", (m - 1) & 1, m - 1)
        yield ("tma", "QFULL")
        m += 1
        for _ in range(count):
            s, kk = u % stages, u // stages
            # K once the stage's previous key tile's S products are done, V once
            # its P.V products are
            yield ("wait", ("KEMPTY", s), (kk & 1) ^ 1, kk - 1)
            yield ("tma", ("KFULL", s))
            yield ("wait", ("VEMPTY", s), (kk & 1) ^ 1, kk - 1)
            yield ("tma", ("VFULL", s))
            u += 1


def fwd_issuer(items, stages, sep=False):
    """sep: P in TMEM columns of its own (d = 64): S_x needs only its softmax
    to have loaded the previous S_x (SFREE); per entry both next S first, then
    the P.V products."""
    m = u = 0
    nv = [0, 0]
    ns = [0, 0]

    def s_ready(x):
        if ns[x] == 0:
            return
        if sep:
            yield ("wait", ("SFREE", x), (ns[x] - 1) & 1, ns[x] - 1)
        elif nv[x] > 0:
            yield ("wait", ("PVDONE", x), (nv[x] - 1) & 1, nv[x] - 1)

    for k, it in enumerate(list(items) + [None]):
        yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
        if it is None:
            return
        count, vis = it
        if count:
            yield ("wait", "QFULL", m & 1, m)
            m += 1
            yield ("wait", ("KFULL", u % stages), (u // stages) & 1, u // stages)
            for x in range(2):
                if vis[x][0]:
                    yield from s_ready(x)
                    yield ("commit", ("SFULL", x))
                    ns[x] += 1
            yield ("commit", ("KEMPTY", u % stages))
            if count == 1:
                yield ("commit", "QEMPTY")
            for e in range(count):
                s, s2 = u % stages, (u + 1) % stages
                vwaited = kwaited = False
                if sep:
                    for x in range(2):
                        if e + 1 < count and vis[x][e + 1]:
                            if not kwaited:
                                kk = (u + 1) // stages
                                yield ("wait", ("KFULL", s2), kk & 1, kk)
                                kwaited = True
                            yield from s_ready(x)
                            yield ("commit", ("SFULL", x))
                            ns[x] += 1
                    if e + 1 < count:
                        yield ("commit", ("KEMPTY", s2))
                    if e + 2 == count:
                        yield ("commit", "QEMPTY")
                    for x in range(2):
                        if vis[x][e]:
                            yield ("wait", ("PFULL", x), nv[x] & 1, nv[x])
                            if not vwaited:
                                yield ("wait", ("VFULL", s), (u // stages) & 1, u // stages)
                                vwaited = True
                            yield ("commit", ("PVDONE", x))
                            nv[x] += 1
                    yield ("commit", ("VEMPTY", s))
                    u += 1
                    continue
                for x in range(2):
                    if vis[x][e]:
                        yield ("wait", ("PFULL", x), nv[x] & 1, nv[x])
                        if not vwaited:
                            yield ("wait", ("VFULL", s), (u // stages) & 1, u // stages)
                            vwaited = True
                        yield ("commit", ("PVDONE", x))
                        nv[x] += 1
                    if x == 1:
                        # V's last readers (both P.V) are issued: release it before the
                        # second query tile's next S
                        yield ("commit", ("VEMPTY", s))
                    if e + 1 < count and vis[x][e + 1]:
                        if not kwaited:
                            kk = (u + 1) // stages
                            yield ("wait", ("KFULL", s2), kk & 1, kk)
                            kwaited = True
                        yield from s_ready(x)
                        yield ("commit", ("SFULL", x))
                        ns[x] += 1
                if e + 1 < count:
                    yield ("commit", ("KEMPTY", s2))
                if e + 2 == count:
                    yield ("commit", "QEMPTY")
                u += 1
        yield ("arrive", ("ITEMFREE", k & 1))


def fwd_softmax(x, items, rng, p_rescale, sep=False):
    ns = 0
    for k, it in enumerate(list(items) + [None]):
        yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
        if it is None:
            return
        count, vis = it
        n_item = 0
        for e in range(count):
            if not vis[x][e]:
                continue
            yield ("wait", ("SFULL", x), ns & 1, ns)
            if sep:
                yield ("arrive", ("SFREE", x))
                if ns > 0:                      # the P buffer: the previous P.V has read it
                    yield ("wait", ("PVDONE", x), (ns - 1) & 1, ns - 1)
            elif n_item > 0 and rng.random() < p_rescale:
                yield ("wait", ("PVDONE", x), (ns - 1) & 1, ns - 1)
            yield ("arrive", ("PFULL", x))
            ns += 1
            n_item += 1
        if n_item:
            yield ("wait", ("PVDONE", x), (ns - 1) & 1, ns - 1)
        yield ("arrive", ("ITEMFREE", k & 1))


def fwd_items(rng, n_items):
    """Random work items: without a block mask query tile x sees the first
    n_x key tiles (count = max n_x); under one, an arbitrary subset of the
    listed tiles (each listed tile seen by at least one query tile); the last
    query tile of an odd count has no rows."""
    items = []
    for _ in range(n_items):
        count = rng.choice([0, 1, 1, 2, 3, 4, 7])
        two = rng.random() < 0.8
        if rng.random() < 0.5:
            n = [rng.randint(0, count), rng.randint(0, count) if two else 0]
            n[rng.randrange(2) if two else 0] = count
            vis = [[e < n[x] for e in range(count)] for x in range(2)]
        else:
            vis = [[False] * count, [False] * count]
            for e in range(count):
                b = rng.choice([1, 2, 3]) if two else 1
                vis[0][e], vis[1][e] = bool(b & 1), bool(b & 2)
        items.append((count, vis))
    return items


def run_fwd(seed, stages, n_items=None, p_rescale=0.3, sep=False, **producer_kw):
    rng = random.Random(seed)
    items = fwd_items(rng, n_items if n_items is not None else rng.randint(1, 7))
    roles = {"producer": fwd_producer(items, stages, **producer_kw), "issuer": fwd_issuer(items, stages, sep),
             "softmax0": fwd_softmax(0, items, rng, p_rescale, sep),
             "softmax1": fwd_softmax(1, items, rng, p_rescale, sep)}
    schedule(rng, roles, lambda name: 3 if name[0] == "ITEMFREE" else 1)


# ---------------------------------------------------------------- split-KV decode
# `fa_decode_kernel`: one query tile, S and P in two TMEM buffers (tile i in
# buffer i % 2), so the issuer runs one S ahead of the softmax.

def dec_producer(n, stages):
    if n:
        yield ("tma", "QFULL")
    for it in range(n):
        s, k = it % stages, it // stages
        yield ("wait", ("KVEMPTY", s), (k & 1) ^ 1, k - 1)
        yield ("tma", ("KFULL", s))
        yield ("tma", ("VFULL", s))


def dec_issuer(n, stages):
    if not n:
        return
    yield ("wait", "QFULL", 0, 0)

    def issue_s(i):
        k = i // stages
        yield ("wait", ("KFULL", i % stages), k & 1, k)
        if i >= 2:
            yield ("wait", ("PVDONE", i & 1), ((i - 2) >> 1) & 1, (i - 2) >> 1)
        yield ("commit", ("SFULL", i & 1))

    yield from issue_s(0)
    for it in range(n):
        if it + 1 < n:
            yield from issue_s(it + 1)
        s = it % stages
        yield ("wait", ("PFULL", it & 1), (it >> 1) & 1, it >> 1)
        yield ("wait", ("VFULL", s), (it // stages) & 1, it // stages)
        yield ("commit", ("KVEMPTY", s))
        yield ("commit", ("PVDONE", it & 1))


def dec_softmax(n, rng, p_rescale):
    for it in range(n):
        yield ("wait", ("SFULL", it & 1), (it >> 1) & 1, it >> 1)
        if it > 0 and rng.random() < p_rescale:
            yield ("wait", ("PVDONE", (it - 1) & 1), ((it - 1) >> 1) & 1, (it - 1) >> 1)
        yield ("arrive", ("PFULL", it & 1))
    if n:
        yield ("wait", ("PVDONE", (n - 1) & 1), ((n - 1) >> 1) & 1, (n - 1) >> 1)


def run_decode(seed, n, stages, p_rescale=0.3):
    rng = random.Random(seed)
    roles = {"producer": dec_producer(n, stages), "issuer": dec_issuer(n, stages),
             "softmax": dec_softmax(n, rng, p_rescale)}
    schedule(rng, roles, lambda name: 1)


# ---------------------------------------------------------------- d = 64 backward
# `fa_bwd64_kernel`, persistent: work items (key tiles) published in two
# slots as in the forward (the issuer, the compute warpgroups and the drain
# warpgroup release a slot); K and V double-buffered per item (KVFULL /
# KVFREE, the free commit after the item's products); Q and dO double-buffered
# together, LSE/D per stage, S and dP in their own TMEM columns, dQ into two
# TMEM buffers emptied by the drain warpgroup; an item's dK, dV complete at
# ACC.  Block, stage and item counters run on across items; an item's first
# S and dP wait for the previous block's dV and dK (SFREE, DPFREE).  The
# producer's K/V-free wait guards data only (the issuer has waited for a
# buffer's load before it releases the item slot, so the ready barrier cannot
# run ahead): dropping it shows in the parity tests, not here.

def bwd64_producer(items, kv_free_wait=True):
    i = nkv = 0
    for k, n in enumerate(list(items) + [None]):
        if k >= 2:
            yield ("wait", ("ITEMFREE", k & 1), ((k >> 1) - 1) & 1, (k >> 1) - 1)
        yield ("arrive", ("ITEM", k & 1))
        if n is None:
            return
        if not n:
            continue
        b = nkv & 1
        if nkv >= 2 and kv_free_wait:
            yield ("wait", ("KVFREE", b), ((nkv >> 1) - 1) & 1, (nkv >> 1) - 1)
        yield ("tma", ("KVFULL", b))
        nkv += 1
        for _ in range(n):
            s = i & 1
            yield ("wait", ("QEMPTY", s), ((i >> 1) & 1) ^ 1, (i >> 1) - 1)
            yield ("tma", ("QFULL", s))
            i += 1


LSE_BUFS = 4


def bwd64_stager(items, lse_free_wait=True):
    """Stages every block's LSE and D into a ring of LSE_BUFS buffers, ahead
    of the compute warps and independent of the Q/dO ring."""
    i = 0
    for k, n in enumerate(list(items) + [None]):
        yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
        if n is None:
            return
        for _ in range(n):
            b = i % LSE_BUFS
            if i >= LSE_BUFS and lse_free_wait:
                yield ("wait", ("LSEFREE", b), (i // LSE_BUFS - 1) & 1, i // LSE_BUFS - 1)
            yield ("arrive", ("LSE", b))
            i += 1
        yield ("arrive", ("ITEMFREE", k & 1))


def bwd64_issuer(items):
    i = nkv = 0
    for k, n in enumerate(list(items) + [None]):
        yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
        if n is None:
            return
        if n:
            b = nkv & 1
            yield ("wait", ("KVFULL", b), (nkv >> 1) & 1, nkv >> 1)
            nkv += 1
            yield ("wait", ("QFULL", i & 1), (i >> 1) & 1, i >> 1)
            if i > 0:
                yield ("wait", "SFREE", (i - 1) & 1, i - 1)
            yield ("commit", "SFULL")
            if i > 0:
                yield ("wait", "DPFREE", (i - 1) & 1, i - 1)
            yield ("commit", "DPFULL")
            for e in range(n):
                s, more = i & 1, e + 1 < n
                yield ("wait", "PFULL", i & 1, i)
                yield ("commit", "SFREE")                                       # dV(i) read P
                if more:
                    yield ("wait", ("QFULL", s ^ 1), ((i + 1) >> 1) & 1, (i + 1) >> 1)
                    yield ("wait", "SFREE", i & 1, i)
                    yield ("commit", "SFULL")                                   # S(i+1)
                yield ("wait", "DSFULL", i & 1, i)
                yield ("commit", "DPFREE")                                      # dK(i) read dS
                yield ("commit", ("QEMPTY", s))
                if i >= 2:
                    yield ("wait", ("DQFREE", s), ((i - 2) >> 1) & 1, (i - 2) >> 1)
                yield ("commit", ("DQFULL", s))                                 # dQ(i)
                if more:
                    yield ("wait", "DPFREE", i & 1, i)
                    yield ("commit", "DPFULL")                                  # dP(i+1)
                i += 1
            yield ("commit", "ACC")
            yield ("commit", ("KVFREE", b))
        yield ("arrive", ("ITEMFREE", k & 1))


def bwd64_compute(items):
    i = nacc = 0
    for k, n in enumerate(list(items) + [None]):
        yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
        if n is None:
            return
        for _ in range(n):
            b = i % LSE_BUFS
            yield ("wait", ("LSE", b), (i // LSE_BUFS) & 1, i // LSE_BUFS)
            yield ("wait", "SFULL", i & 1, i)
            yield ("arrive", "PFULL")
            yield ("wait", "DPFULL", i & 1, i)
            if i > 0:
                yield ("wait", ("DQFULL", (i - 1) & 1), ((i - 1) >> 1) & 1, (i - 1) >> 1)
            yield ("arrive", "DSFULL")
            yield ("arrive", ("LSEFREE", b))
            i += 1
        if n:
            yield ("wait", "ACC", nacc & 1, nacc)
            nacc += 1
        yield ("arrive", ("ITEMFREE", k & 1))


def bwd64_drain(items):
    i = 0
    for k, n in enumerate(list(items) + [None]):
        yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
        if n is None:
            return
        for _ in range(n):
            yield ("wait", ("DQFULL", i & 1), (i >> 1) & 1, i >> 1)
            yield ("arrive", ("DQFREE", i & 1))
            i += 1
        yield ("arrive", ("ITEMFREE", k & 1))


def run_bwd64(seed, items=None, lse_free_wait=True, **producer_kw):
    rng = random.Random(seed)
    if items is None:
        items = [rng.choice([0, 1, 1, 2, 3, 4, 5, 9]) for _ in range(rng.randint(1, 7))]
    roles = {"producer": bwd64_producer(items, **producer_kw), "stager": bwd64_stager(items, lse_free_wait),
             "issuer": bwd64_issuer(items), "compute": bwd64_compute(items), "drain": bwd64_drain(items)}
    schedule(rng, roles, lambda name: 4 if name[0] == "ITEMFREE" else 1)


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
    # always an issuer, on a P-ready barrier that has run two phases ahead
    assert all(f.startswith("issuer") and " on ('PFULL'" in f for f in found), found[:3]
    assert all("with" in f and int(f.split("with ")[1].split()[0]) == int(f.split("phase ")[1].split()[0]) + 2
               for f in found)


def test_bf16_forward_protocol_never_aliases():
    for i in range(800):
        run_fwd(seed=i, stages=(2, 4)[i % 2])


def test_bf16_forward_separate_p_protocol_never_aliases():
    """d = 64: P in TMEM columns of its own, the next S after the softmax has
    loaded the current one, the P buffer rewritten after the previous P.V."""
    for i in range(800):
        run_fwd(seed=i, stages=4, sep=True)


def test_separate_p_model_finds_a_dropped_p_buffer_wait():
    """Writing P_x before the previous P_x V has read it lets the softmax run
    ahead of the products: some parity wait then meets a barrier two phases
    away from the one it means."""
    def softmax_no_pv_wait(x, items):
        ns = 0
        for k, it in enumerate(list(items) + [None]):
            yield ("wait", ("ITEM", k & 1), (k >> 1) & 1, k >> 1)
            if it is None:
                return
            count, vis = it
            n_item = 0
            for e in range(count):
                if vis[x][e]:
                    yield ("wait", ("SFULL", x), ns & 1, ns)
                    yield ("arrive", ("SFREE", x))
                    yield ("arrive", ("PFULL", x))
                    ns += 1
                    n_item += 1
            if n_item:
                yield ("wait", ("PVDONE", x), (ns - 1) & 1, ns - 1)
            yield ("arrive", ("ITEMFREE", k & 1))

    found = []
    for i in range(400):
        rng = random.Random(i)
        items = fwd_items(rng, 5)
        roles = {"producer": fwd_producer(items, 4), "issuer": fwd_issuer(items, 4, True),
                 "softmax0": softmax_no_pv_wait(0, items), "softmax1": softmax_no_pv_wait(1, items)}
        try:
            schedule(rng, roles, lambda name: 3 if name[0] == "ITEMFREE" else 1)
        except Alias as e:
            found.append(str(e))
    # the issuer meets a P-ready barrier two phases ahead, or the softmax,
    # run ahead, waits for a P.V product two phases before it completes
    assert found and all("('PFULL'" in f or "('PVDONE'" in f for f in found), found[:3]


def test_forward_model_finds_a_dropped_q_empty_wait():
    """Loading the next item's Q without waiting for the previous item's S
    products lets the Q-ready barrier run two phases ahead of the issuer."""
    found = []
    for i in range(400):
        try:
            run_fwd(seed=i, stages=(2, 4)[i % 2], n_items=6, q_empty_wait=False)
        except Alias as e:
            found.append(str(e))
    assert found and all(" on QFULL" in f for f in found), found[:3]


def test_forward_model_finds_a_dropped_slot_free_wait():
    """Publishing an item into a slot a slow consumer has not yet released
    lets that slot's barrier run two phases ahead of the consumer."""
    found = []
    for i in range(400):
        try:
            run_fwd(seed=i, stages=(2, 4)[i % 2], n_items=7, slot_free_wait=False)
        except Alias as e:
            found.append(str(e))
    assert found and all("('ITEM'" in f for f in found), found[:3]


def test_forward_model_finds_s_issued_before_p_is_awaited():
    """Issuing the next S_x before waiting for P_x (with P kept elsewhere, as
    the FP8 kernel does) lets a softmax warpgroup finish two tiles before
    the issuer's wait: the P-ready barrier runs two phases ahead."""
    def issuer_s_first(n_tiles, stages):
        total = max(n_tiles)
        nv, ns = [0, 0], [0, 0]
        if not total:
            return
        yield ("wait", "QFULL", 0, 0)
        yield ("wait", ("KFULL", 0), 0, 0)
        for x in range(2):
            if n_tiles[x] > 0:
                yield ("commit", ("SFULL", x))
                ns[x] += 1
        yield ("commit", ("KEMPTY", 0))
        for u in range(total):
            s, s2 = u % stages, (u + 1) % stages
            for x in range(2):
                if u + 1 < n_tiles[x]:
                    k = (u + 1) // stages
                    yield ("wait", ("KFULL", s2), k & 1, k)
                    yield ("wait", ("SFREE", x), (ns[x] - 1) & 1, ns[x] - 1)
                    yield ("commit", ("SFULL", x))
                    ns[x] += 1
            if u + 1 < total:
                yield ("commit", ("KEMPTY", s2))
            for x in range(2):
                if u < n_tiles[x]:
                    yield ("wait", ("PFULL", x), nv[x] & 1, nv[x])
                    yield ("wait", ("VFULL", s), (u // stages) & 1, u // stages)
                    yield ("commit", ("PVDONE", x))
                    nv[x] += 1
            yield ("commit", ("VEMPTY", s))

    def softmax_releasing_s(x, n):
        for it in range(n):
            yield ("wait", ("SFULL", x), it & 1, it)
            yield ("arrive", ("SFREE", x))
            yield ("arrive", ("PFULL", x))

    found = []
    for i in range(600):
        n_tiles, stages = TILE_COUNTS[i % len(TILE_COUNTS)], (2, 4)[i % 2]
        one_item = [(max(n_tiles), [[e < n_tiles[x] for e in range(max(n_tiles))] for x in range(2)])]
        roles = {"producer": fwd_producer(one_item, stages), "issuer": issuer_s_first(n_tiles, stages),
                 "softmax0": softmax_releasing_s(0, n_tiles[0]), "softmax1": softmax_releasing_s(1, n_tiles[1])}
        try:
            schedule(random.Random(i), roles, lambda name: 1)
        except Alias as e:
            found.append(str(e))
    assert found and all(f.startswith("issuer on ('PFULL'") for f in found), found[:3]


def test_decode_protocol_never_aliases():
    for i in range(600):
        run_decode(seed=i, n=(1, 2, 3, 4, 7, 13, 40)[i % 7], stages=(3, 6)[i % 2])


def test_bwd64_protocol_never_aliases():
    for i in range(800):
        run_bwd64(seed=i)


def test_bwd64_model_finds_a_dropped_lse_free_wait():
    """Staging LSE and D into a buffer the compute warps have not released
    lets that buffer's ready barrier run two phases ahead of them."""
    found = []
    for i in range(400):
        try:
            run_bwd64(seed=i, items=[9, 5, 9, 7], lse_free_wait=False)
        except Alias as e:
            found.append(str(e))
    assert found and all("('LSE'" in f for f in found), found[:3]



def test_bwd128_protocol_never_aliases():
    for i in range(600):
        run_bwd128(seed=i, n=(1, 2, 3, 4, 5, 9, 16)[i % 7], causal=bool(i & 1))


def test_bwd128_model_finds_a_dropped_drain_wait():
    """Without its wait for the dQ drain, the issuer can complete the next
    block's dQ^T while the drain still waits for the previous one."""
    def issuer_without_dqfree_wait(n):
        return (op for op in bwd_issuer(n) if not (op[0] == "wait" and op[1] == "DQFREE"))
    found = []
    for i in range(300):
        n = (2, 5, 9, 16)[i % 4]
        roles = {"producer": bwd_producer(n), "stager": bwd_stager(n), "issuer": issuer_without_dqfree_wait(n),
                 "compute": bwd_compute(n), "drain": bwd_drain(n)}
        try:
            schedule(random.Random(i), roles, lambda name: 1)
        except Alias as e:
            found.append(str(e))
    assert found and all(f.startswith("drain on DQFULL") for f in found), found[:3]


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
