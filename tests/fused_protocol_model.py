"""A model of the synchronisation protocol of the fused hc=4 kernel
(sinkhorn_mixing_gb300/csrc/hc_fused.cu), run under random interleavings.

Test infrastructure only: it restates the kernel's barriers and roles in
plain Python and shares no code with the kernel.  Each CTA of a cluster runs
the kernel's roles as generators that yield the barrier waits they make:

  producer  per tile, waits for the collapse to be at most `lag` tiles
            behind, then for each stage waits for an empty ring slot, arms
            its full barrier and issues a load that lands later;
  mma       per tile, waits for a free accumulator, consumes every stage in
            order and releases each slot by a commit (commits complete in
            issue order), then commits acc_full; with `post` it waits for
            post_done instead of full, and also stores each rewritten stage
            from its slot by a bulk copy that reads the slot later and writes
            memory later still: it waits until that store has read the slot
            and releases it, and at a tile's last stage waits until the
            tile's stores are written and arrives on its sq_full first;
  sq (x4)   consume every stage in order, release it, publish the tile's sums
            of squares through sq_full / sq_empty (x8 with `norm`); with
            `post` (x8) they
            first rewrite the stage in place (hc_post of the previous
            sublayer) and signal post_done, and leave the release to the MMA
            thread; with `norm` each also waits until the previous tile's
            records were read (recv_free) and sends its rows' Gram entries
            into their owners' records, completing recv_full by bytes;
  epi (x2)  read the accumulator and the squares, wait until the previous
            tile's records were read (recv_free), then send their records to
            the owners, whose recv_full they complete by bytes;
  owner     waits for its records, reads them, stages pre and signals
            pre_ready, re-arms recv_full, then releases the record buffer to
            every sender;
  collapse  (x2) waits for pre, reads the staging slot (with `post`, and
            the tile's new stream as every CTA of the cluster stored it),
            signals col_done.

Up to three randomly chosen roles run a hundred times slower than the rest,
so that single slow roles fall far behind and early-reuse windows are
reached.

mbarrier model: a phase completes when its pending arrivals and its
transaction bytes both reach zero; try_wait(parity) is true iff the current
phase's parity differs from `parity`, so only the current and the previous
phase can be told apart, as on the hardware.

Checks: a load never lands in a slot that is being read; every consumer
finds the stage it expects; an accumulator, a staging slot or a record buffer
is never overwritten while read; no arrival or byte count underflows; and
every role finishes (no deadlock).
"""
import random


class ProtocolError(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.completed = name, count, count, 0, 0

    def arrive(self):
        if self.pending == 0:
            raise ProtocolError("arrival underflow on " + self.name)
        self.pending -= 1
        self._settle()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        if self.tx < 0 and self.pending == 0:
            raise ProtocolError("byte count underflow on " + self.name)
        self._settle()

    def _settle(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def try_wait(self, parity):
        return parity != (self.completed & 1)


def wait(bar, parity):
    return ("wait", bar, parity)


class Cond:
    """A wait on a condition that the hardware guarantees to become true
    (completion of bulk copies already issued)."""

    def __init__(self, fn):
        self.fn = fn

    def try_wait(self, _parity):
        return self.fn()


def until(fn):
    return ("wait", Cond(fn), None)


STEP = ("step",)


def simulate(ctas=4, tiles=5, stages_per_tile=5, slots=3, lag=3, bufs=4, mixes_only=False,
             seed=0, mutation=None, post=False, norm=False):
    """Run one random interleaving; raises ProtocolError on any violation.
    `mutation` plants a known protocol mistake (for the tests that show the
    model can fail): "release_before_read", "empty_parity", and with post
    "mma_waits_full", "release_before_store_read", "visible_before_written", and
    with norm "gram_without_recv_free"."""
    rnd = random.Random(seed)
    events = []

    def later(fn):
        events.append(fn)

    C, T, NS, S = ctas, tiles, stages_per_tile, slots
    NSQ = 8 if (post or norm) else 4  # the wide layout of both variants
    written = set()  # (rank, stage) of x_next stores that reached memory
    cs = []
    for r in range(C):
        cs.append(dict(
            rank=r,
            full=[Barrier("full", 1) for _ in range(S)],
            post_done=[Barrier("post_done", NSQ) for _ in range(S)],
            posted=[set() for _ in range(S)],
            # MMA commit + 4 square warps; with post MMA commit + store read
            empty=[Barrier("empty", 2 if post else 1 + NSQ) for _ in range(S)],
            stores=[],
            slot=[None] * S, holders=[set() for _ in range(S)],
            acc_full=[Barrier("acc_full", 1) for _ in range(2)],
            acc_empty=[Barrier("acc_empty", 2) for _ in range(2)],
            acc=[None, None], acc_readers=[0, 0],
            sq_full=[Barrier("sq_full", NSQ + (1 if post else 0)) for _ in range(2)],
            sq_empty=[Barrier("sq_empty", 2) for _ in range(2)],
            sq=[[None] * NSQ, [None] * NSQ],
            recv_full=Barrier("recv_full", 1), recv_free=Barrier("recv_free", C),
            recv=[None] * C, recv_g={}, reading=[False],
            pre_ready=[Barrier("pre_ready", 1) for _ in range(bufs)],
            col_done=[Barrier("col_done", 2) for _ in range(bufs)],
            stage=[None] * bufs, stage_readers=[0] * bufs))
    # with norm, square warp w holds the rows of tokens TW*w .. TW*w+TW-1 of
    # the 64-token tile and sends each row's Gram entries to the row's owner
    # (TO tokens per owner): every owner hears from every warp that holds one
    # of its rows, in every CTA
    TW, TO = 64 // NSQ, 64 // C
    covers = [sorted({t // TO for t in range(TW * w, TW * w + TW)}) for w in range(NSQ)]
    gram_from = [[w for w in range(NSQ) if o in covers[w]] for o in range(C)]
    per_round = [C + (C * len(gram_from[o]) if norm else 0) for o in range(C)]
    for r, c in enumerate(cs):
        c["recv_full"].expect_tx(per_round[r])

    def producer(c):
        for it in range(T):
            if not mixes_only and it >= lag:
                tw = it - lag
                yield wait(c["col_done"][tw % bufs], (tw // bufs) & 1)
            for st in range(NS):
                q = NS * it + st
                s, use = q % S, q // S
                par = (use & 1) if mutation == "empty_parity" else (use & 1) ^ 1
                yield wait(c["empty"][s], par)
                c["full"][s].expect_tx(1)

                def land(c=c, s=s, q=q):
                    if c["holders"][s]:
                        raise ProtocolError("a load lands in a slot that is being read")
                    c["slot"][s] = q
                    c["posted"][s] = set()
                    c["full"][s].complete_tx(1)
                later(land)

    def mma(c, rank):
        chain = []
        stores = c["stores"]

        def store(s, q):
            rec = dict(q=q, read=False, written=False)
            stores.append(rec)
            c["holders"][s].add(("store", q))

            def read(rec=rec, s=s, q=q):
                rec["read"] = True
                c["holders"][s].discard(("store", q))

                def write(rec=rec, q=q):
                    rec["written"] = True
                    written.add((rank, q))
                later(write)
            later(read)

        def all_done(key):
            return lambda: all(r[key] for r in stores)

        def commit():
            kind, a, b = chain.pop(0)
            if kind == "empty":
                c["holders"][a].discard("mma")
                c["empty"][a].arrive()
            else:
                c["acc"][a] = b
                c["acc_full"][a].arrive()
        for it in range(T):
            b = it & 1
            yield wait(c["acc_empty"][b], ((it >> 1) & 1) ^ 1)
            if c["acc_readers"][b]:
                raise ProtocolError("the MMA overwrites an accumulator being read")
            for st in range(NS):
                q = NS * it + st
                s = q % S
                waits_post = post and mutation != "mma_waits_full"
                yield wait(c["post_done" if waits_post else "full"][s], (q // S) & 1)
                if c["slot"][s] != q:
                    raise ProtocolError("MMA wants stage %d, slot holds %s" % (q, c["slot"][s]))
                if post and len(c["posted"][s]) != NSQ:
                    raise ProtocolError("MMA reads stage %d before it was rewritten" % q)
                c["holders"][s].add("mma")
                chain.append(("empty", s, None))
                later(commit)
                if post:
                    store(s, q)
                    if st + 1 < NS:
                        if mutation != "release_before_store_read":
                            yield until(all_done("read"))
                    else:
                        if mutation != "visible_before_written":
                            yield until(all_done("written"))
                        elif mutation != "release_before_store_read":
                            yield until(all_done("read"))
                        c["sq_full"][b].arrive()
                    c["empty"][s].arrive()
            chain.append(("acc", b, it))
            later(commit)

    def sq(c, w):
        for it in range(T):
            b = it & 1
            for st in range(NS):
                q = NS * it + st
                s = q % S
                yield wait(c["full"][s], (q // S) & 1)
                if c["slot"][s] != q:
                    raise ProtocolError("squares want stage %d, slot holds %s" % (q, c["slot"][s]))
                c["holders"][s].add(w)
                yield STEP
                if post:
                    c["posted"][s].add(w)
                    c["holders"][s].discard(w)
                    c["post_done"][s].arrive()
                else:
                    c["holders"][s].discard(w)
                    c["empty"][s].arrive()
            yield wait(c["sq_empty"][b], ((it >> 1) & 1) ^ 1)
            c["sq"][b][w] = it
            c["sq_full"][b].arrive()
            if norm:
                if mutation != "gram_without_recv_free":
                    yield wait(c["recv_free"], (it & 1) ^ 1)
                for o in covers[w]:
                    def deliver_g(o=o, it=it, rank=c["rank"], w=w):
                        oc = cs[o]
                        if oc["reading"][0]:
                            raise ProtocolError("Gram entries land while their owner reads")
                        if oc["recv_g"].get((rank, w)) is not None:
                            raise ProtocolError("Gram entries overwrite unread ones")
                        oc["recv_g"][(rank, w)] = it
                        oc["recv_full"].complete_tx(1)
                    later(deliver_g)

    def epi(c, rank, half):
        mine = range(half * C // 2, (half + 1) * C // 2) if C > 1 else range(1)
        for it in range(T):
            b = it & 1
            yield wait(c["acc_full"][b], (it >> 1) & 1)
            if c["acc"][b] != it:
                raise ProtocolError("read-out finds the accumulator of %s" % c["acc"][b])
            c["acc_readers"][b] += 1
            yield STEP
            c["acc_readers"][b] -= 1
            c["acc_empty"][b].arrive()
            yield wait(c["sq_full"][b], (it >> 1) & 1)
            if c["sq"][b] != [it] * NSQ:
                raise ProtocolError("read-out finds squares %s" % c["sq"][b])
            if post and any((rank, NS * it + st) not in written for st in range(NS)):
                raise ProtocolError("records of tile %d leave before its new stream is written"
                                    % it)
            c["sq_empty"][b].arrive()
            yield wait(c["recv_free"], (it & 1) ^ 1)
            for o in mine:
                def deliver(o=o, it=it):
                    oc = cs[o]
                    if oc["reading"][0]:
                        raise ProtocolError("a record lands while its owner reads")
                    if oc["recv"][rank] is not None:
                        raise ProtocolError("a record overwrites an unread one")
                    oc["recv"][rank] = it
                    oc["recv_full"].complete_tx(1)
                later(deliver)

    def owner(c):
        for it in range(T):
            yield wait(c["recv_full"], it & 1)
            if c["recv"] != [it] * C:
                raise ProtocolError("owner of tile %d finds records %s" % (it, c["recv"]))
            if norm and any(c["recv_g"].get((r, w)) != it for r in range(C)
                            for w in gram_from[c["rank"]]):
                raise ProtocolError("owner of tile %d finds Gram entries %s" % (it, c["recv_g"]))
            if mutation == "release_before_read":
                for d in cs:
                    later(lambda d=d: d["recv_free"].arrive())
            c["reading"][0] = True
            yield STEP
            c["reading"][0] = False
            if not mixes_only:
                i = it % bufs
                if c["stage_readers"][i]:
                    raise ProtocolError("pre staging overwritten while the collapse reads it")
                c["stage"][i] = it
                c["pre_ready"][i].arrive()
            c["recv"] = [None] * C
            c["recv_g"] = {}
            c["recv_full"].expect_tx(per_round[c["rank"]])
            if mutation != "release_before_read":
                for d in cs:
                    later(lambda d=d: d["recv_free"].arrive())

    def collapse(c):
        for it in range(T):
            i = it % bufs
            yield wait(c["pre_ready"][i], (it // bufs) & 1)
            if c["stage"][i] != it:
                raise ProtocolError("collapse of tile %d reads the pre of %s" % (it, c["stage"][i]))
            if post and any((r, NS * it + st) not in written for r in range(C) for st in range(NS)):
                raise ProtocolError("collapse of tile %d re-reads a stream not yet written" % it)
            c["stage_readers"][i] += 1
            yield STEP
            c["stage_readers"][i] -= 1
            c["col_done"][i].arrive()

    roles = []
    for r, c in enumerate(cs):
        roles += [producer(c), mma(c, r), owner(c)] + [sq(c, w) for w in range(NSQ)]
        roles += [epi(c, r, h) for h in range(2)]
        if not mixes_only:
            roles += [collapse(c), collapse(c)]
    # Adversarial schedule: zero to three roles, chosen at random, run a
    # hundred times slower than the rest, so that one slow consumer or
    # producer falls far behind and the windows in which a buffer could be
    # reused early, or a barrier phase be passed twice, are actually reached.
    speed = [1.0] * len(roles)
    for k in rnd.sample(range(len(roles)), rnd.choice((0, 1, 2, 3))):
        speed[k] = 0.01
    state = [None] * len(roles)
    live = set()
    for k, g in enumerate(roles):
        try:
            state[k] = next(g)
            live.add(k)
        except StopIteration:
            pass
    while live or events:
        ready = [k for k in live if state[k] is STEP or state[k][1].try_wait(state[k][2])]
        if not ready and not events:
            raise ProtocolError("deadlock: %d roles wait forever" % len(live))
        wsum = sum(speed[k] for k in ready) + len(events)
        x = rnd.random() * wsum
        k = None
        for j in ready:
            x -= speed[j]
            if x < 0:
                k = j
                break
        if k is not None:
            try:
                state[k] = next(roles[k])
            except StopIteration:
                live.discard(k)
        else:
            events.pop(rnd.randrange(len(events)))()
