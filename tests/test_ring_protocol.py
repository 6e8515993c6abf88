"""Host model of the kernels' mbarrier protocols, run under random interleavings.

The tcgen05 kernels hand data between a TMA producer warp, MMA-issuing warps
and softmax warps through mbarriers that are waited on by phase parity.  A
parity wait is only exact if the waiter has seen the barrier's previous
phase complete; a waiter two phases behind, or one waiting for a phase whose
predecessor is still pending, misreads the barrier.  Such slips show up on a
GPU as a rare hang or as stale shared memory, so the protocols are modelled
here on the host, step by step, with every agent advanced in random order:

  * producer: fills ring slots in a fixed order, waiting on each slot's
    `empty` barrier (all of the slot's releasers must have arrived);
  * MMA warps: wait with the same parities the kernels use; their MMAs and
    tcgen05.commit arrivals complete in issue order per warp, at random
    later times;
  * softmax warps: wait and arrive as the kernels do.

Each ring slot, TMEM S buffer and shared-memory P buffer carries a tag of
what was last written into it; a read that finds another tag (stale or
overwritten data) is an error, and so is a state in which no agent can move
(a deadlock).  The models follow the kernels in
differential_attention_03_gb300/csrc (onepass.cuh, twopass.cuh, decode.cuh).  Two
variants that were wrong are kept as negative checks: the model must catch
them.
"""

import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        # mbarrier.try_wait.parity: true once the phase of that parity has completed,
        # i.e. when the current phase's parity differs.
        return (self.phase & 1) != parity


class World:
    def __init__(self, seed):
        self.rnd = random.Random(seed)
        self.errors = []
        self.pipes = {}     # MMA warp -> FIFO of ('mma', fn) / ('commit', bar)
        self.tma = []       # (slot, tag, bar)
        self.slot = {}      # ring slot -> tag of the fill it holds
        self.tmem = {}      # TMEM buffer -> tag
        self.pbuf = {}      # P buffer -> tag

    def wait(self, bar, parity):
        while not bar.done(parity):
            yield

    def mma(self, warp, fn):
        self.pipes.setdefault(warp, []).append(("mma", fn))

    def commit(self, warp, bar):
        self.pipes.setdefault(warp, []).append(("commit", bar))

    def expect(self, table, key, tag, what):
        if table.get(key) != tag:
            self.errors.append(f"{what}: {key} holds {table.get(key)}, wanted {tag}")

    def run(self, agents, max_steps=400000):
        live = dict(agents)
        steps = 0
        while live or self.tma or any(self.pipes.values()):
            steps += 1
            if steps > max_steps:  # every agent left is blocked on a wait that never completes
                return "deadlock"
            moves = list(live) + (["tma"] if self.tma else []) + [w for w, q in self.pipes.items() if q]
            c = self.rnd.choice(moves)
            if c == "tma":
                i = 0 if self.rnd.random() < 0.6 else self.rnd.randrange(len(self.tma))
                s, tag, bar = self.tma.pop(i)
                if s != "Q":
                    self.slot[s] = tag
                bar.arrive()
            elif c in live:
                try:
                    next(live[c])
                except StopIteration:
                    del live[c]
            else:
                kind, x = self.pipes[c].pop(0)
                if kind == "commit":
                    x.arrive()
                else:
                    x()
        return "ok" if not self.errors else self.errors[0]


# --------------------------------------------------------------------------- one-pass kernel
def onepass(T, seed, nslot, psm, shared_k, vf=2, npb=1, p_ready_per_buffer=True, items=None):
    """onepass.cuh: persistent; one MMA warp per map, both walk every fill (empty counts 2).

    `items` lists the key-tile counts of the work items one CTA processes in
    turn (default: one item of T tiles); ring, per-tile barriers and their
    phases run on across items, q_free guards Q and o_free the accumulators.
    """
    items = [T] if items is None else items
    W = World(seed)
    full = [Bar(1) for _ in range(nslot)]
    empty = [Bar(2) for _ in range(nslot)]
    s_full = [Bar(1) for _ in range(2)]
    s_free = [Bar(1) for _ in range(2)]
    nbar = npb if p_ready_per_buffer else 1
    p_ready = [[Bar(1) for _ in range(nbar)] for _ in range(2)]
    pv_done = [[Bar(1) for _ in range(npb)] for _ in range(2)]
    q_full, o_full, q_free, o_free = Bar(1), Bar(2), Bar(2), Bar(2)
    W.q = None
    W.oread = {(a, r): -1 for a in range(2) for r in range(2)}  # (softmax agent, O_r) -> last item read
    fills = []
    for it, Ti in enumerate(items):
        fills += [("K1", it, 0)] + ([] if shared_k else [("K2", it, 0)])
        for j in range(Ti):
            if psm and j + 1 < Ti:
                fills += [("K1", it, j + 1)] + ([] if shared_k else [("K2", it, j + 1)])
            fills += [("V", it, j, p) for p in range(vf)]
            if not psm and j + 1 < Ti:
                fills += [("K1", it, j + 1)] + ([] if shared_k else [("K2", it, j + 1)])

    def producer():
        f = 0
        for it, Ti in enumerate(items):
            if it:
                yield from W.wait(q_free, (it - 1) & 1)

            class QLoad:  # lands as a TMA copy: tags the Q buffer, then arrives q_full
                def arrive(self, it=it):
                    W.q = it
                    q_full.arrive()
            W.tma.append(("Q", it, QLoad()))
            n_item = 1 + (0 if shared_k else 1) + Ti * vf + (Ti - 1) * (1 if shared_k else 2)
            for _ in range(n_item):
                s, use = f % nslot, f // nslot
                if use:
                    yield from W.wait(empty[s], (use - 1) & 1)
                W.tma.append((s, fills[f], full[s]))
                f += 1

    def mma(r):
        fill = 0
        mine = "K1" if (r == 0 or shared_k) else "K2"

        def acquire():
            nonlocal fill
            f = fill
            fill += 1
            s = f % nslot
            yield from W.wait(full[s], (f // nslot) & 1)
            W.expect(W.slot, s, fills[f], f"warp {r} acquire")
            return s, fills[f]

        def k_tile(it, g, jj, last):
            while True:
                s, tag = yield from acquire()
                if tag[0] == mine:
                    break
                W.commit(r, empty[s])        # the other map's K: waited on, released
            if psm and g > 0:
                yield from W.wait(s_free[r], (g - 1) & 1)

            def qk(s=s, tag=tag, g=g, it=it):
                W.expect(W.slot, s, tag, f"QK{r + 1}({g}) reads K")
                if W.q != it:
                    W.errors.append(f"QK{r + 1}({g}) read Q of item {W.q}, wanted {it}")
                W.tmem[("S", r)] = g
            W.mma(r, qk)
            W.commit(r, s_full[r])
            W.commit(r, empty[s])
            if last:
                W.commit(r, q_free)
            if not shared_k and r == 0:
                s2, _ = yield from acquire()  # K_2 of the same tile
                W.commit(r, empty[s2])

        gt = 0
        for it, Ti in enumerate(items):
            yield from W.wait(q_full, it & 1)
            yield from k_tile(it, gt, 0, Ti == 1)
            for j in range(Ti):
                g = gt + j
                if psm and j + 1 < Ti:
                    yield from k_tile(it, g + 1, j + 1, j + 2 == Ti)
                sv = []
                for _ in range(vf):
                    sv.append((yield from acquire()))
                b = g % npb
                yield from W.wait(p_ready[r][b if p_ready_per_buffer else 0],
                                  (g // npb if p_ready_per_buffer else g) & 1)
                if j == 0 and it:
                    yield from W.wait(o_free, (it - 1) & 1)
                for i, (s, tag) in enumerate(sv):  # the MMAs of one V part, then its release
                    def pv(s=s, tag=tag, g=g, b=b, it=it, j=j):
                        W.expect(W.slot, s, tag, f"PV{r + 1}({g}) reads V")
                        if psm:
                            W.expect(W.pbuf, (r, b), g, f"PV{r + 1}({g}) reads P")
                        else:
                            W.expect(W.tmem, ("P", r), g, f"PV{r + 1}({g}) reads P in TMEM")
                        if j == 0 and any(W.oread[(a, r)] != it - 1 for a in range(2)):
                            W.errors.append(f"PV{r + 1} of item {it} overwrote O{r + 1} before every epilogue read it")
                        W.tmem[("O", r)] = (it, j)
                    W.mma(r, pv)
                    if i + 1 < len(sv):
                        W.commit(r, empty[s])
                if psm:
                    W.commit(r, pv_done[r][b])
                W.commit(r, empty[sv[-1][0]])
                if not psm and j + 1 < Ti:
                    yield from k_tile(it, g + 1, j + 1, j + 2 == Ti)
            W.commit(r, o_full)
            gt += Ti

    def softmax(r):
        gt = 0
        for it, Ti in enumerate(items):
            for j in range(Ti):
                g = gt + j
                yield from W.wait(s_full[r], g & 1)
                W.expect(W.tmem, ("S", r), g, f"softmax {r + 1} reads S({g})")
                if psm:
                    s_free[r].arrive()
                    b = g % npb
                    if g >= npb:
                        yield from W.wait(pv_done[r][b], ((g - npb) // npb) & 1)
                    W.pbuf[(r, b)] = g
                else:
                    W.tmem[("P", r)] = g      # P over S in TMEM
                yield
                p_ready[r][(g % npb) if p_ready_per_buffer else 0].arrive()
            yield from W.wait(o_full, it & 1)
            # Every epilogue warpgroup reads columns of both accumulators.
            for rr in range(2):
                W.expect(W.tmem, ("O", rr), (it, Ti - 1), f"epilogue {r + 1} reads O{rr + 1} of item {it}")
                W.oread[(r, rr)] = it
                yield
            o_free.arrive()
            gt += Ti

    W.tma_kinds = True
    return W.run({"prod": producer(), "mma0": mma(0), "mma1": mma(1), "sm0": softmax(0), "sm1": softmax(1)})


# --------------------------------------------------------------------------- two-sweep kernel
def twopass(T, seed, nslot=4, vf=2, per_owner_full=True, items=None, wait_o_free=True):
    """twopass.cuh: warp 1 issues map-1 MMAs and P.V, warp 2 map-2 MMAs; each fill has one reader.

    Persistent when `items` lists several items: fills, S-buffer uses and
    sweep-2 tile phases run on across items.  TMEM is modelled by buffer:
    sweep 1 cycles S through buffers 0-3 (O lives in 0 and 1, so an S write
    there clobbers O and the between-sweeps exchange kept in buffer 0), sweep
    2 keeps S_1 in buffer 2 (also the epilogue's exchange) and S_2 in 3.
    """
    items = [T] if items is None else items
    W = World(seed)
    nown = 2 if per_owner_full else 1
    full = [[Bar(1) for _ in range(nslot)] for _ in range(nown)]
    empty = [Bar(1) for _ in range(nslot)]
    s1_full = [Bar(1) for _ in range(4)]
    s1_free = [Bar(1) for _ in range(4)]
    # sweep 2: both softmax agents (all warpgroups in the kernel) load S_1 / S_2
    # and write their part of P: free and ready barriers count both
    a2_full, b2_full, a2_free, b2_free = Bar(1), Bar(1), Bar(2), Bar(2)
    p_ready, pv_done, o_full = Bar(2), Bar(1), Bar(1)
    q_full, q_free, o_free = Bar(1), Bar(2), Bar(2)
    xchg = Bar(2)   # the softmax agents' rendezvous (named barrier)
    W.q = None
    W.tmem = {}

    def tm_write(buf, tag):
        W.tmem[buf] = tag
        if buf in (0, 1):            # O and the exchange columns live in buffers 0 and 1
            W.tmem["O"] = ("clobbered", tag)
            if buf == 0:
                W.tmem["X"] = ("clobbered", tag)
        if buf == 2:
            W.tmem["AX"] = ("clobbered", tag)

    fills = []  # (tag, owner)
    for it, Ti in enumerate(items):
        for j in range(Ti):
            fills += [(("K1", it, j), 0), (("K2", it, j), 1)]
        fills += [(("K2", it, 0), 1), (("K1", it, 0), 0)]
        for j in range(Ti):
            if j + 1 < Ti:
                fills += [(("K2", it, j + 1), 1), (("K1", it, j + 1), 0)]
            fills += [(("V", it, j, p), 0) for p in range(vf)]

    def producer():
        f = 0
        for it, Ti in enumerate(items):
            if it:
                yield from W.wait(q_free, (it - 1) & 1)

            class QLoad:
                def arrive(self, it=it):
                    W.q = it
                    q_full.arrive()
            W.tma.append(("Q", it, QLoad()))
            for _ in range(Ti * (4 + vf)):
                tag, o = fills[f]
                s, use = f % nslot, f // nslot
                if use:
                    yield from W.wait(empty[s], (use - 1) & 1)
                W.tma.append((s, tag, full[o if per_owner_full else 0][s]))
                f += 1

    def mma(mw):
        ph = 0  # per-slot parity bits of this warp's own fills (per-owner barriers)
        it_f = iter([f for f, (_, o) in enumerate(fills) if o == mw])

        def acquire():
            nonlocal ph
            f = next(it_f)
            s = f % nslot
            if per_owner_full:
                par = (ph >> s) & 1
                ph ^= 1 << s
                yield from W.wait(full[mw][s], par)
            else:
                yield from W.wait(full[0][s], (f // nslot) & 1)
            W.expect(W.slot, s, fills[f][0], f"warp {mw + 1} acquire")
            return s, fills[f][0]

        def qk(buf, s, tag, what, it):
            def go():
                W.expect(W.slot, s, tag, what)
                if W.q != it:
                    W.errors.append(f"{what} read Q of item {W.q}, wanted {it}")
                tm_write(buf, what)
            W.mma(mw, go)

        use = {0: 0, 1: 0, 2: 0, 3: 0}
        sfull, sfree = (a2_full, a2_free) if mw == 0 else (b2_full, b2_free)
        g1 = 0
        for it, Ti in enumerate(items):
            yield from W.wait(q_full, it & 1)
            if it and wait_o_free:  # (o_free also follows every sweep-2 read of buffers 2, 3)
                yield from W.wait(o_free, (it - 1) & 1)
            for j in range(Ti):
                k = 2 * (g1 + j) + mw
                bb = k & 3
                s, tag = yield from acquire()
                if use[bb]:
                    yield from W.wait(s1_free[bb], (use[bb] - 1) & 1)
                use[bb] += 1
                qk(bb, s, tag, ("sw1", k), it)
                W.commit(mw, s1_full[bb])
                W.commit(mw, empty[s])
            if use[mw + 2]:
                yield from W.wait(s1_free[mw + 2], (use[mw + 2] - 1) & 1)
            s, tag = yield from acquire()
            qk(mw + 2, s, tag, ("sw2", mw, g1), it)
            W.commit(mw, sfull)
            W.commit(mw, empty[s])
            if Ti == 1:
                W.commit(mw, q_free)
            for j in range(Ti):
                g = g1 + j
                if j + 1 < Ti:
                    s, tag = yield from acquire()
                    yield from W.wait(sfree, g & 1)
                    qk(mw + 2, s, tag, ("sw2", mw, g + 1), it)
                    W.commit(mw, sfull)
                    W.commit(mw, empty[s])
                    if j + 2 == Ti:
                        W.commit(mw, q_free)
                if mw == 0:
                    sv = []
                    for _ in range(vf):
                        sv.append((yield from acquire()))
                    yield from W.wait(p_ready, g & 1)
                    for i, (s_, tag_) in enumerate(sv):  # the MMAs of one V part, then its release
                        def pv(s_=s_, tag_=tag_, g=g, it=it, j=j):
                            W.expect(W.slot, s_, tag_, f"PV({g}) reads V")
                            W.expect(W.pbuf, 0, g, f"PV({g}) reads P of agent 0")
                            W.expect(W.pbuf, 1, g, f"PV({g}) reads P of agent 1")
                            W.tmem[0] = W.tmem[1] = ("O", it, j)
                            W.tmem["O"] = (it, j)
                            W.tmem["X"] = ("clobbered by PV", it)
                        W.mma(mw, pv)
                        if i + 1 < len(sv):
                            W.commit(mw, empty[s_])
                    W.commit(mw, pv_done)
                    W.commit(mw, empty[sv[-1][0]])
            if mw == 0:
                W.commit(mw, o_full)
            g1 += Ti

    def softmax(m):
        g1 = 0
        nx = 0  # rendezvous uses so far
        for it, Ti in enumerate(items):
            for j in range(Ti):
                k = 2 * (g1 + j) + m
                bb = k & 3
                yield from W.wait(s1_full[bb], (k >> 2) & 1)
                W.expect(W.tmem, bb, ("sw1", k), f"sweep-1 softmax {m} reads S")
                s1_free[bb].arrive()
            # exchange through buffer 0's first columns, between two rendezvous
            xchg.arrive()
            yield from W.wait(xchg, nx & 1)
            nx += 1
            W.tmem["X"] = ("x", it)
            xchg.arrive()
            yield from W.wait(xchg, nx & 1)
            nx += 1
            W.expect(W.tmem, "X", ("x", it), f"softmax {m} reads the exchange")
            for j in range(Ti):
                g = g1 + j
                yield from W.wait(b2_full, g & 1)
                W.expect(W.tmem, 3, ("sw2", 1, g), f"sweep-2 softmax {m} reads S2")
                b2_free.arrive()
                yield from W.wait(a2_full, g & 1)
                W.expect(W.tmem, 2, ("sw2", 0, g), f"sweep-2 softmax {m} reads S1")
                a2_free.arrive()
                if g:
                    yield from W.wait(pv_done, (g - 1) & 1)
                W.pbuf[m] = g
                p_ready.arrive()
            yield from W.wait(o_full, it & 1)
            W.expect(W.tmem, "O", (it, Ti - 1), f"epilogue {m} reads O of item {it}")
            W.tmem["AX"] = ("ss", it)         # the sums of squares through buffer 2
            xchg.arrive()
            yield from W.wait(xchg, nx & 1)
            nx += 1
            W.expect(W.tmem, "AX", ("ss", it), f"epilogue {m} reads the exchange in A")
            W.expect(W.tmem, "O", (it, Ti - 1), f"epilogue {m} reads O of item {it} again")
            o_free.arrive()
            g1 += Ti

    return W.run({"prod": producer(), "w1": mma(0), "w2": mma(1), "sm0": softmax(0), "sm1": softmax(1)})


TS = [1, 2, 3, 5, 9]


@pytest.mark.parametrize("T", TS)
def test_onepass_p_in_smem(T):
    for seed in range(25):
        assert onepass(T, seed, nslot=7, psm=True, shared_k=False) == "ok", seed


@pytest.mark.parametrize("T", TS)
def test_onepass_p_in_tmem_shared_k(T):
    for seed in range(25):
        assert onepass(T, seed, nslot=4, psm=False, shared_k=True, vf=1) == "ok", seed


ITEM_LISTS = [[3, 1], [1, 1, 1], [2, 5, 1, 3], [4, 4]]


@pytest.mark.parametrize("items", ITEM_LISTS)
def test_onepass_persistent_p_in_smem(items):
    for seed in range(20):
        assert onepass(0, seed, nslot=7, psm=True, shared_k=False, items=items) == "ok", seed


@pytest.mark.parametrize("items", ITEM_LISTS)
def test_onepass_persistent_p_in_tmem_shared_k(items):
    for seed in range(20):
        assert onepass(0, seed, nslot=4, psm=False, shared_k=True, vf=1, items=items) == "ok", seed


@pytest.mark.parametrize("T", TS)
def test_twopass_per_owner_full_barriers(T):
    for seed in range(25):
        assert twopass(T, seed) == "ok", seed


def test_model_catches_double_buffered_p_with_one_ready_barrier():
    # Two P buffers let a map's softmax finish tiles j and j+1 before its MMA
    # warp waits for tile j: one p_ready barrier then completes two phases unseen.
    bad = [onepass(T, seed, nslot=4, psm=True, shared_k=False, npb=2, p_ready_per_buffer=False)
           for T in (3, 5, 9) for seed in range(25)]
    assert any(r != "ok" for r in bad)
    good = [onepass(T, seed, nslot=4, psm=True, shared_k=False, npb=2, p_ready_per_buffer=True)
            for T in (3, 5, 9) for seed in range(25)]
    assert all(r == "ok" for r in good)


def test_model_catches_missing_q_free_and_o_free():
    import inspect
    src = inspect.getsource(onepass)
    ns = {}
    for cut, what in ((
            """                if j == 0 and it:\n                    yield from W.wait(o_free, (it - 1) & 1)\n""", "o_free"),
            ("""            if it:\n                yield from W.wait(q_free, (it - 1) & 1)\n""", "q_free")):
        assert cut in src, what
        exec(compile(src.replace(cut, ""), __file__, "exec"), globals(), ns)
        bad = [ns["onepass"](0, seed, nslot=7, psm=True, shared_k=False, items=it)
               for it in ([3, 1], [2, 5, 1, 3]) for seed in range(30)]
        assert any(r != "ok" for r in bad), what


@pytest.mark.parametrize("items", ITEM_LISTS)
def test_twopass_persistent(items):
    for seed in range(20):
        assert twopass(0, seed, items=items) == "ok", seed


def test_model_catches_missing_twopass_o_free():
    bad = [twopass(0, seed, items=it, wait_o_free=False) for it in ([3, 1], [1, 2, 1], [2, 5, 1]) for seed in range(40)]
    assert any(r != "ok" for r in bad)


def test_model_catches_shared_full_barriers_with_partial_waiters():
    # One full barrier per slot, but each warp waits only on its own fills: at the
    # switch between the sweeps a warp can take an older phase for its fill.
    bad = [twopass(T, seed, per_owner_full=False) for T in (2, 3, 5) for seed in range(60)]
    assert any(r != "ok" for r in bad)


# --------------------------------------------------------------------------- decode kernel
def decode(nblk, seed, nst=3, nwarp=4, refill_waits_empty=True):
    """decode.cuh: thread 0 issues the first NST stages, then refills stage s once all
    warps have released it (empty, count = warps); every warp waits on every fill in
    order (full, count 1 + the copy's bytes) and reads the stage's keys."""
    W = World(seed)
    full = [Bar(1) for _ in range(nst)]
    empty = [Bar(nwarp) for _ in range(nst)]
    W.stage = {}

    def warp(wi):
        issued = 0
        if wi == 0:  # thread 0 of warp 0 also produces
            while issued < min(nst, nblk):
                W.tma.append((issued % nst, issued, full[issued % nst]))
                issued += 1
        for i in range(nblk):
            s = i % nst
            yield from W.wait(full[s], (i // nst) & 1)
            W.expect(W.slot, s, i, f"warp {wi} reads block {i}")
            yield
            empty[s].arrive()
            if wi == 0 and issued < nblk:
                if refill_waits_empty:
                    yield from W.wait(empty[s], (i // nst) & 1)
                W.tma.append((s, issued, full[s]))
                issued += 1

    return W.run({f"w{w}": warp(w) for w in range(nwarp)})


@pytest.mark.parametrize("nblk", [0, 1, 2, 3, 4, 7, 16])
def test_decode_ring(nblk):
    for seed in range(30):
        assert decode(nblk, seed) == "ok", seed
        assert decode(nblk, seed, nwarp=8) == "ok", seed
        # e4m3 key caches: four stages of 24 KB
        assert decode(nblk, seed, nst=4) == "ok", seed
        assert decode(nblk, seed, nst=4, nwarp=8) == "ok", seed


def test_model_catches_decode_refill_without_empty_wait():
    bad = [decode(nblk, seed, refill_waits_empty=False) for nblk in (5, 9, 16) for seed in range(40)]
    assert any(r != "ok" for r in bad)
